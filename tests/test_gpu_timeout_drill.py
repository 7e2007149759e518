"""Failure detection on the GPU without a fault: every wait in the attention
kernel is bounded, and a wait that runs out makes the kernel record
MHA_ERR_TIMEOUT in the caller's status word, drain what it has in flight,
free its tensor memory and return.  The drill entry point makes a wait run
out on purpose -- the loader issues no copy for one key tile, so nothing ever
completes that tile's barrier -- with a 2 ms wait limit.  The kernel must
return (the synchronize comes back), report the timeout, and leave the
context usable: the next ordinary call on the same stream is bit-equal to
one made before the drill."""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LIMIT_NS = 2_000_000  # 2 ms


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda:0").view(
        torch.bfloat16)


def _ordinary(tsds, q, k, v, w):
    out = torch.empty((w.B, w.h, w.T_q, w.d_v), dtype=torch.bfloat16, device="cuda:0")
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    tsds.sdpa_forward(q, k, v, out, scale=w.scale, mask=w.mask, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


# (T_q, T_k, mask, skip_tile): which key split runs, and how far the CTAs get
# before the missing tile -- at the first tile no product has been issued; at
# later tiles score and P.V products of earlier tiles are in flight or done
# and the abort has to drain them.
CASES = [
    (512, 512, si.MASK_CAUSAL, 0),      # key halves, nothing issued yet
    (512, 512, si.MASK_CAUSAL, 2),      # key halves, two tiles' products done
    (128, 2048, si.MASK_NONE, 5),       # alternate tiles, ring wrapped once
]


@pytest.mark.parametrize("T_q,T_k,mask,skip", CASES)
def test_wait_runs_out_and_context_stays_usable(T_q, T_k, mask, skip):
    import transformer_scaled_dot_softmax_gb300 as tsds
    from transformer_scaled_dot_softmax_gb300 import _native as nat
    w = si.WORKLOADS[4].replace(B=1, h=1, T_q=T_q, T_k=T_k, mask=mask, seed=77)
    x = si.make_inputs(w)
    q, k, v = _dev(x["q_bits"]), _dev(x["k_bits"]), _dev(x["v_bits"])
    before = _ordinary(tsds, q, k, v, w)

    o = torch.empty_like(before)
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    rc = nat.lib.sdpa_forward_timeout_drill(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                            w.B, w.h, w.T_q, w.T_k, w.scale, w.mask, None,
                                            LIMIT_NS, skip, status.data_ptr(), stream)
    assert rc == nat.MHA_OK
    torch.cuda.synchronize()  # the kernel gave up and returned
    assert int(status.item()) == nat.MHA_ERR_TIMEOUT

    after = _ordinary(tsds, q, k, v, w)
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
