"""mha_forward_static_workspace: the MHA forward for callers that cannot
allocate device memory (its scratch lives in a device array inside the
library).  Called through the C ABI and checked against mha_forward, the
entry point that takes a caller-owned workspace, on two calls in a row with
different problems -- the second call reuses the array the first one left
behind.  This file is collected last on purpose."""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


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


def test_static_workspace_matches_caller_workspace_twice():
    from transformer_scaled_dot_softmax_gb300 import _native as nat
    problems = [
        # self-attention with key padding (fits the 32 MiB scratch: 16 MiB)
        si.WORKLOADS[1],
        # then a different shape: causal cross-attention over longer keys
        si.WORKLOADS[3].replace(B=2, T_q=200, T_k=700, mask=si.MASK_CAUSAL_KEY_PADDING,
                                len_lo=300, len_hi=700),
    ]
    for w in problems:
        assert nat.lib.mha_workspace_bytes(w.B, w.h, w.T_q, w.T_k, w.d_k, w.d_v) <= \
            nat.MHA_STATIC_WORKSPACE_BYTES
        t = _problem(w)
        ref = torch.empty((w.B, w.T_q, w.d_model), dtype=torch.bfloat16, device="cuda:0")
        assert _call_workspace(nat, w, t, ref) == nat.MHA_OK
        out = torch.full_like(ref, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        assert _call_static(nat, w, t, out, status) == nat.MHA_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got, exp = out.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        err = np.abs(got - exp)
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (err.max(), err.mean())


def test_static_workspace_rejects_problems_beyond_its_size():
    from transformer_scaled_dot_softmax_gb300 import _native as nat
    w = si.WORKLOADS[3]  # needs 40 MiB of scratch
    assert nat.lib.mha_workspace_bytes(w.B, w.h, w.T_q, w.T_k, w.d_k, w.d_v) > \
        nat.MHA_STATIC_WORKSPACE_BYTES
    t = _problem(w.replace(B=1, T_q=64, T_k=64))  # tensors are never touched
    out = torch.empty(1, dtype=torch.bfloat16, device="cuda:0")
    rc = _call_static(nat, w, t, out, None)
    assert rc == nat.MHA_ERR_WORKSPACE
