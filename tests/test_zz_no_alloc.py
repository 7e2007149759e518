"""mha_forward_static_workspace: the MHA forward for callers that cannot
allocate device memory (its scratch lives in a device array inside the
library).  Called through the C ABI and checked against mha_forward, the
entry point that takes a caller-owned workspace: both run the same kernels on
the same inputs, so the outputs must be bit-equal.  The calls come in a row,
each problem smaller than the one before, after a call on NaN inputs has left
NaN in the scratch the later problems reuse -- a read of scratch that the
call itself did not write would show.  This file is collected last on
purpose."""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda:0").view(
        torch.bfloat16)


def _problem(w):
    x = si.make_inputs(w)
    t = {k: _dev(x[k + "_bits"]) for k in ("x_q", "w_q", "w_k", "w_v", "w_o")}
    t["x_kv"] = _dev(x["x_kv_bits"]) if w.cross else t["x_q"]
    t["lens"] = None if x["key_lens"] is None else torch.from_numpy(x["key_lens"]).to("cuda:0")
    return t


def _call_static(nat, w, t, out, status):
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda a: None if a is None else a.data_ptr()  # noqa: E731
    return nat.lib.mha_forward_static_workspace(
        nat.MHA_BF16, p(t["x_q"]), p(t["x_kv"]), p(t["w_q"]), p(t["w_k"]), p(t["w_v"]),
        p(t["w_o"]), p(out), w.B, w.h, w.T_q, w.T_k, w.d_model, w.d_k, w.d_v, w.scale, w.mask,
        p(t["lens"]), p(status), stream)


def _call_workspace(nat, w, t, out):
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda a: None if a is None else a.data_ptr()  # noqa: E731
    need = nat.lib.mha_workspace_bytes(w.B, w.h, w.T_q, w.T_k, w.d_k, w.d_v)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda:0")
    rc = nat.lib.mha_forward(
        nat.MHA_BF16, p(t["x_q"]), p(t["x_kv"]), p(t["w_q"]), p(t["w_k"]), p(t["w_v"]),
        p(t["w_o"]), p(out), p(ws), need, w.B, w.h, w.T_q, w.T_k, w.d_model, w.d_k, w.d_v,
        w.scale, w.mask, p(t["lens"]), None, stream)
    torch.cuda.synchronize()
    return rc


def test_static_workspace_bit_equal_to_caller_workspace_on_shrinking_problems():
    from transformer_scaled_dot_softmax_gb300 import _native as nat
    big = si.WORKLOADS[1]  # self-attention with key padding: 16 MiB of scratch
    problems = [
        big,
        # a smaller problem of another kind: causal cross-attention with
        # key padding over longer keys
        si.WORKLOADS[3].replace(B=2, T_q=200, T_k=700, mask=si.MASK_CAUSAL_KEY_PADDING,
                                len_lo=300, len_hi=700),
        # smaller again, one ragged tile
        si.WORKLOADS[2].replace(B=1, T_q=100, T_k=100),
    ]
    sizes = [nat.lib.mha_workspace_bytes(w.B, w.h, w.T_q, w.T_k, w.d_k, w.d_v) for w in problems]
    assert sizes[0] <= nat.MHA_STATIC_WORKSPACE_BYTES
    assert sizes == sorted(sizes, reverse=True) and len(set(sizes)) == len(sizes)

    # Leave NaN in the scratch: the largest problem on NaN activations.
    t = _problem(big)
    t["x_q"] = torch.full_like(t["x_q"], float("nan"))
    t["x_kv"] = t["x_q"]
    junk = torch.empty((big.B, big.T_q, big.d_model), dtype=torch.bfloat16, device="cuda:0")
    assert _call_static(nat, big, t, junk, None) == nat.MHA_OK
    torch.cuda.synchronize()

    for w in problems:
        t = _problem(w)
        ref = torch.empty((w.B, w.T_q, w.d_model), dtype=torch.bfloat16, device="cuda:0")
        assert _call_workspace(nat, w, t, ref) == nat.MHA_OK
        assert torch.all(torch.isfinite(ref))
        out = torch.full_like(ref, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        assert _call_static(nat, w, t, out, status) == nat.MHA_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            "static-workspace output differs from mha_forward (B%d T_q%d T_k%d)" % (w.B, w.T_q, w.T_k)


def test_static_workspace_rejects_problems_beyond_its_size():
    from transformer_scaled_dot_softmax_gb300 import _native as nat
    w = si.WORKLOADS[3]  # needs 40 MiB of scratch
    assert nat.lib.mha_workspace_bytes(w.B, w.h, w.T_q, w.T_k, w.d_k, w.d_v) > \
        nat.MHA_STATIC_WORKSPACE_BYTES
    t = _problem(w.replace(B=1, T_q=64, T_k=64))  # tensors are never touched
    out = torch.empty(1, dtype=torch.bfloat16, device="cuda:0")
    rc = _call_static(nat, w, t, out, None)
    assert rc == nat.MHA_ERR_WORKSPACE


def test_static_workspace_checks_arguments_first():
    """Argument errors are reported as such (not as a CUDA or workspace
    error), and an empty problem returns MHA_OK, before any device work."""
    from transformer_scaled_dot_softmax_gb300 import _native as nat
    w = si.WORKLOADS[1].replace(B=1, T_q=64, T_k=64)
    t = _problem(w)
    out = torch.empty((w.B, w.T_q, w.d_model), dtype=torch.bfloat16, device="cuda:0")
    bad = dict(t)
    bad["x_q"] = None
    assert _call_static(nat, w, bad, out, None) == nat.MHA_ERR_INVALID_ARG
    assert _call_static(nat, w.replace(d_k=32, d_v=32), t, out, None) == nat.MHA_ERR_UNSUPPORTED
    assert _call_static(nat, w.replace(B=0), t, out, None) == nat.MHA_OK
