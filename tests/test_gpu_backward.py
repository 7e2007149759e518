"""Parity of the attention backward (sdpa_backward, through the C ABI) with
the fp64 oracle's gradients, on the same seeded q, k, v and output gradient.

The GPU path recomputes the weights from its own forward's log-sum-exp and
bf16 output (sdpa_forward_lse), rounds P and dS to bf16 for the tensor-core
products and the gradients to bf16 at the end.  Tolerance, relative to the
size of each gradient: max-abs <= 2e-2 * max(1, max|ref|) and mean-abs <=
2e-3 * max(1, mean|ref|).
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    import transformer_scaled_dot_softmax_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def dev():
    return torch.device("cuda:0")


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(torch.bfloat16)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_grad(got, ref, what):
    assert np.all(np.isfinite(got)), what + ": non-finite"
    err = np.abs(got - ref)
    big = max(1.0, float(np.abs(ref).max()))
    avg = max(1.0, float(np.abs(ref).mean()))
    assert err.max() <= 2e-2 * big and err.mean() <= 2e-3 * avg, (
        "%s: max %.4g (ref max %.3g) mean %.4g (ref mean %.3g)" % (what, err.max(), np.abs(ref).max(),
                                                                err.mean(), np.abs(ref).mean()))


def run_backward(lib, w, x, dout_bits):
    q, k, v = bf16_dev(x["q_bits"]), bf16_dev(x["k_bits"]), bf16_dev(x["v_bits"])
    lens = None if x["key_lens"] is None else torch.from_numpy(x["key_lens"]).to(dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    o, lse = lib.sdpa_forward_lse(q, k, v, scale=w.scale, mask=w.mask, key_lens=lens, status=status)
    g = bf16_dev(dout_bits)
    dq, dk, dv = lib.sdpa_backward(q, k, v, o, g, lse, scale=w.scale, mask=w.mask, key_lens=lens,
                                   status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return host(dq), host(dk), host(dv)


BWD_SHAPES = [
    (1, 1, 128, 128, si.MASK_NONE),
    (1, 2, 256, 256, si.MASK_CAUSAL),
    (2, 2, 255, 257, si.MASK_NONE),
    (2, 1, 300, 700, si.MASK_KEY_PADDING),
    (1, 2, 384, 384, si.MASK_CAUSAL_KEY_PADDING),
    (1, 1, 130, 1, si.MASK_NONE),
    (1, 1, 1000, 64, si.MASK_CAUSAL),
    (1, 1, 64, 1000, si.MASK_NONE),
    (1, 2, 1024, 1024, si.MASK_CAUSAL),
]


@pytest.mark.parametrize("B,h,T_q,T_k,mask", BWD_SHAPES)
def test_backward_vs_oracle(lib, B, h, T_q, T_k, mask):
    w = si.WORKLOADS[4].replace(B=B, h=h, T_q=T_q, T_k=T_k, mask=mask, len_lo=0, len_hi=T_k,
                                seed=111)
    x = si.make_inputs(w)
    dout = si.round_bf16(si.normal(w.seed, si.TENSOR_IDS["dout"], (B, h, T_q, 64)))
    got = run_backward(lib, w, x, si.f64_to_bf16_bits(dout))
    ref = oracle.sdpa_backward(x["q"], x["k"], x["v"], dout, scale=w.scale, mask=mask,
                               key_lens=x["key_lens"])
    for name, a, r in zip(("dq", "dk", "dv"), got, ref):
        check_grad(a, r, "%s B%d h%d Tq%d Tk%d mask%d" % (name, B, h, T_q, T_k, mask))


def test_backward_key_gradients_sum_to_zero(lib):
    # softmax shift invariance: sum_j dK_j = 0 for every (b, h)
    w = si.WORKLOADS[4].replace(B=1, h=2, T_q=300, T_k=500, mask=si.MASK_NONE, seed=112)
    x = si.make_inputs(w)
    dout = si.round_bf16(si.normal(w.seed, si.TENSOR_IDS["dout"], (1, 2, 300, 64)))
    dq, dk, dv = run_backward(lib, w, x, si.f64_to_bf16_bits(dout))
    col = np.abs(dk).sum(axis=2)
    assert np.all(np.abs(dk.sum(axis=2)) <= 2e-2 * np.maximum(1.0, col))


def test_backward_masked_keys_get_no_gradient(lib):
    w = si.WORKLOADS[4].replace(B=3, h=1, T_q=200, T_k=600, mask=si.MASK_KEY_PADDING, len_lo=0,
                                len_hi=600, seed=113)
    x = si.make_inputs(w)
    x["key_lens"] = np.array([0, 77, 600], dtype=np.int32)
    dout = si.round_bf16(si.normal(w.seed, si.TENSOR_IDS["dout"], (3, 1, 200, 64)))
    dq, dk, dv = run_backward(lib, w, x, si.f64_to_bf16_bits(dout))
    assert np.all(dk[0] == 0) and np.all(dv[0] == 0) and np.all(dq[0] == 0)
    assert np.all(dk[1, :, 77:] == 0) and np.all(dv[1, :, 77:] == 0)


def test_backward_tail_rows_workload_full(lib):
    """The backward at the benchmark's full size (causal, B=2, h=16,
    T=8192, d=64), compared with the fp64 oracle where its tail sums are the
    full gradient: dq of the last 256 query rows (each sums over up to every
    key) and dk, dv of the last 256 keys (two key blocks, each summed over the
    query rows that see it), every head, every element of those rows."""
    w = si.WORKLOADS[4]
    x = si.make_inputs(w)
    dout = si.round_bf16(si.normal(w.seed, si.TENSOR_IDS["dout"], x["q"].shape))
    got = run_backward(lib, w, x, si.f64_to_bf16_bits(dout))
    i0 = w.T_q - 256
    ref = oracle.sdpa_backward_tail(x["q"], x["k"], x["v"], dout, i0, scale=w.scale, mask=w.mask)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check_grad(g[:, :, i0:], r[:, :, i0:], name + " (last 256 rows)")
