"""Parity of sdpa_forward_host (host buffers in, host buffer out, chunked
copies and launches on two copy streams) with the device path and the fp64
oracle.

The host path runs the same attention kernels on groups of heads, and a
head's output does not depend on the other heads, so its output must equal
the device path's bit for bit; the oracle bounds are those of the device
path (fp32 max-abs 1e-5; bf16 max-abs 2e-2, mean-abs 2e-3).
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MASK_NAMES = {si.MASK_NONE: "none", si.MASK_CAUSAL: "causal",
              si.MASK_KEY_PADDING: "key_padding", si.MASK_CAUSAL_KEY_PADDING: "causal_key_padding"}


@pytest.fixture(scope="module")
def lib():
    import transformer_scaled_dot_softmax_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def bf16_host(bits, pinned):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t.clone()


# (B, h, T_q, T_k, mask): chunks of heads of one batch item (B*h >= 8), whole
# batch items (h small), a head count that does not split evenly, ragged
# lengths that span several tiles, cross attention.
CASES = [(2, 16, 200, 200, si.MASK_CAUSAL), (3, 5, 130, 257, si.MASK_KEY_PADDING),
         (8, 1, 64, 64, si.MASK_NONE), (1, 9, 300, 300, si.MASK_CAUSAL_KEY_PADDING),
         (2, 3, 129, 1000, si.MASK_NONE),
         # longer causal sequences, with and without padding
         (2, 3, 1000, 1000, si.MASK_CAUSAL), (1, 4, 1024, 1024, si.MASK_CAUSAL_KEY_PADDING)]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("B,h,Tq,Tk,mask", CASES)
def test_host_path_bf16(lib, B, h, Tq, Tk, mask, pinned):
    w = si.WORKLOADS[4].replace(B=B, h=h, T_q=Tq, T_k=Tk, mask=mask, len_lo=1, len_hi=Tk, seed=140)
    x = si.make_inputs(w)
    q, k, v = (bf16_host(x[n + "_bits"], pinned) for n in ("q", "k", "v"))
    out = torch.empty((B, h, Tq, 64), dtype=torch.bfloat16)
    out = out.pin_memory() if pinned else out
    lens = None if x["key_lens"] is None else torch.from_numpy(x["key_lens"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.sdpa_forward_host(q, k, v, out, scale=w.scale, mask=MASK_NAMES[mask], key_lens=lens,
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the device path on the same inputs
    dref = lib.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, mask=MASK_NAMES[mask],
                            key_lens=None if lens is None else lens.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out, dref.cpu())
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=mask, key_lens=x["key_lens"])
    err = np.abs(out.float().numpy().astype(np.float64) - ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())


def test_host_path_fp32(lib):
    w = si.WORKLOADS[0].replace(B=2, h=5, T_q=33, T_k=47, mask=si.MASK_CAUSAL, seed=141)
    x = si.make_inputs(w)
    q, k, v = (torch.from_numpy(np.ascontiguousarray(x[n], dtype=np.float32)).pin_memory()
               for n in ("q", "k", "v"))
    out = lib.sdpa_forward_host(q, k, v, scale=w.scale, mask="causal")
    torch.cuda.synchronize()
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=si.MASK_CAUSAL)
    assert np.abs(out.numpy().astype(np.float64) - ref).max() <= 1e-5


def test_host_path_orders_with_the_stream(lib):
    """Work enqueued on the stream after the call sees the output, and a
    second call reusing the workspace and the same host buffers is ordered
    behind the first."""
    w = si.WORKLOADS[4].replace(B=2, h=8, T_q=256, T_k=256, mask=si.MASK_CAUSAL, seed=142)
    x = si.make_inputs(w)
    q, k, v = (bf16_host(x[n + "_bits"], True) for n in ("q", "k", "v"))
    ws = torch.empty(lib.sdpa_forward_host_workspace_bytes(2, 8, 256, 256), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    o1 = torch.empty((2, 8, 256, 64), dtype=torch.bfloat16).pin_memory()
    o2 = torch.empty_like(o1).pin_memory()
    lib.sdpa_forward_host(q, k, v, o1, ws, scale=w.scale, mask="causal", stream=s)
    lib.sdpa_forward_host(q, k, v, o2, ws, scale=w.scale, mask="causal", stream=s)
    s.synchronize()
    assert torch.equal(o1, o2)
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=si.MASK_CAUSAL)
    assert np.abs(o1.float().numpy().astype(np.float64) - ref).max() <= 2e-2
