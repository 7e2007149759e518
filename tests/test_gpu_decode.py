"""Parity of the decode-step attention (sdpa_decode_forward, through the C ABI)
with the fp64 oracle: the new query rows of each (b, h) against the first
cache_lens[b] rows of the key/value cache, i.e. scaled dot-product attention
with a key-padding mask.

Tolerance: the bf16 bar, max-abs <= 2e-2 and mean-abs <= 2e-3 over every
output element (the kernel keeps q.k, the softmax and the P.V sums in fp32;
only the stored output is rounded to bf16).
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


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


def check_bf16(got, ref, what=""):
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (
        "%s: max %.4g mean %.4g" % (what, err.max(), err.mean()))


def run_decode(lib, w, x, k=None, v=None):
    q = bf16_dev(x["q_bits"])
    k = bf16_dev(x["k_bits"]) if k is None else k
    v = bf16_dev(x["v_bits"]) if v is None else v
    lens = None if x["key_lens"] is None else torch.from_numpy(x["key_lens"]).to(dev())
    out = torch.full((w.B, w.h, w.T_q, w.d_v), float("nan"), dtype=torch.bfloat16, device=dev())
    lib.sdpa_decode_forward(q, k, v, lens, out, scale=w.scale)
    torch.cuda.synchronize()
    return out


def oracle_decode(w, x):
    mask = si.MASK_KEY_PADDING if x["key_lens"] is not None else si.MASK_NONE
    return oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=mask, key_lens=x["key_lens"])


def test_decode_workload_full(lib):
    w = si.WORKLOADS[5]
    x = si.make_inputs(w)
    check_bf16(host(run_decode(lib, w, x)), oracle_decode(w, x), w.name)


@pytest.mark.parametrize("T_q", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("T_k,len_lo,len_hi", [(1, 1, 1), (63, 1, 63), (65, 60, 65),
                                               (1000, 0, 1000), (4097, 4000, 4097)])
def test_decode_rows_and_ragged_caches(lib, T_q, T_k, len_lo, len_hi):
    w = si.WORKLOADS[5].replace(B=3, h=2, T_q=T_q, T_k=T_k, len_lo=len_lo, len_hi=len_hi, seed=51)
    x = si.make_inputs(w)
    check_bf16(host(run_decode(lib, w, x)), oracle_decode(w, x),
               "Tq%d Tk%d lens %s" % (T_q, T_k, list(x["key_lens"])))


def test_decode_without_lengths_uses_whole_cache(lib):
    w = si.WORKLOADS[5].replace(B=2, h=3, T_q=2, T_k=777, mask=si.MASK_NONE, seed=52)
    x = si.make_inputs(w)
    assert x["key_lens"] is None
    check_bf16(host(run_decode(lib, w, x)), oracle_decode(w, x), "no lengths")


def test_decode_empty_cache_outputs_zero(lib):
    w = si.WORKLOADS[5].replace(B=2, h=2, T_q=3, T_k=300, seed=53)
    x = si.make_inputs(w)
    x["key_lens"] = np.array([0, 150], dtype=np.int32)
    out = run_decode(lib, w, x)
    assert torch.all(out[0] == 0)
    check_bf16(host(out), oracle_decode(w, x), "empty cache row")


def test_decode_zero_capacity_outputs_zero(lib):
    q = torch.randn(2, 2, 1, 64, device=dev()).bfloat16()
    kv = torch.empty(2, 2, 0, 64, dtype=torch.bfloat16, device=dev())
    out = lib.sdpa_decode_forward(q, kv, kv)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_decode_rows_bitwise_independent_of_rows_past_length(lib):
    w = si.WORKLOADS[5].replace(B=4, h=2, T_q=2, T_k=2000, len_lo=100, len_hi=1900, seed=54)
    x = si.make_inputs(w)
    a = run_decode(lib, w, x)
    k = bf16_dev(x["k_bits"]).clone()
    v = bf16_dev(x["v_bits"]).clone()
    for b, L in enumerate(x["key_lens"]):
        k[b, :, L:] = torch.randn_like(k[b, :, L:].float()).mul(40).bfloat16()
        v[b, :, L:] = torch.randn_like(v[b, :, L:].float()).mul(40).bfloat16()
    b2 = run_decode(lib, w, x, k=k, v=v)
    assert torch.equal(a.view(torch.int16), b2.view(torch.int16))


def test_decode_single_key_returns_its_value(lib):
    w = si.WORKLOADS[5].replace(B=2, h=2, T_q=4, T_k=500, seed=55)
    x = si.make_inputs(w)
    x["key_lens"] = np.array([1, 1], dtype=np.int32)
    out = run_decode(lib, w, x)
    v0 = bf16_dev(x["v_bits"])[:, :, :1].expand(-1, -1, w.T_q, -1)
    assert torch.equal(out, v0)


def test_decode_constant_values(lib):
    w = si.WORKLOADS[5].replace(B=2, h=2, T_q=3, T_k=3000, len_lo=1000, len_hi=3000, seed=56)
    x = si.make_inputs(w)
    v = torch.full((w.B, w.h, w.T_k, w.d_v), -2.25, dtype=torch.bfloat16, device=dev())
    out = run_decode(lib, w, x, v=v)
    # fp32 softmax weights sum to 1 within rounding; the bf16 result is -2.25
    np.testing.assert_allclose(host(out), -2.25, rtol=0, atol=2.25 * 2 ** -8)


def test_decode_matches_full_kernel_with_padding(lib):
    w = si.WORKLOADS[5].replace(B=3, h=4, T_q=8, T_k=2500, len_lo=500, len_hi=2500, seed=57)
    x = si.make_inputs(w)
    dec = run_decode(lib, w, x)
    q, k, v = bf16_dev(x["q_bits"]), bf16_dev(x["k_bits"]), bf16_dev(x["v_bits"])
    lens = torch.from_numpy(x["key_lens"]).to(dev())
    full = lib.sdpa_forward(q, k, v, scale=w.scale, mask="key_padding", key_lens=lens)
    torch.cuda.synchronize()
    check_bf16(host(dec), host(full), "decode vs full kernel")


# Batch sizes from one entry to more than the 8-CTA clusters fill in one wave,
# with tied and empty caches among the lengths.
@pytest.mark.parametrize("B", [1, 2, 5, 16, 64, 65, 70])
def test_decode_batch_sizes(lib, B):
    w = si.WORKLOADS[5].replace(B=B, h=3, T_q=2, T_k=700, len_lo=0, len_hi=700, seed=60 + B)
    x = si.make_inputs(w)
    lens = x["key_lens"].copy()
    lens[::4] = lens[0]    # ties
    lens[1::7] = 0         # empty caches
    x["key_lens"] = lens
    check_bf16(host(run_decode(lib, w, x)), oracle_decode(w, x), "B%d" % B)


def test_decode_all_lengths_equal(lib):
    w = si.WORKLOADS[5].replace(B=9, h=2, T_q=1, T_k=513, mask=si.MASK_NONE, seed=71)
    x = si.make_inputs(w)
    check_bf16(host(run_decode(lib, w, x)), oracle_decode(w, x), "equal lengths")
