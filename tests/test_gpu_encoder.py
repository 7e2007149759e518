"""Parity of the encoder-layer path (positional_encoding_add and
encoder_layer_forward, through the C ABI) with the fp64 oracle.

Tolerances (u = 2^-8, the bf16 unit roundoff):
  * positional encoding: one bf16 rounding of x + PE, so
    |got - exact| <= u |exact| + 2e-3 (plus the fp32 angle error, ~1e-7 * pos).
  * encoder layer: its outputs are layer-normalised (unit variance, |y| up to
    ~5), not attention outputs, so the bound scales with them.  The final bf16
    rounding alone is up to u |y|; the sublayer output y1 (LN2's residual and
    the FFN's input), the hidden activations and Q/K/V/O are rounded too, each
    adding a relative ~u that the normalisation (gain 1/sigma ~ 1) passes on.
    Bound: max-abs <= 4u max(1, max|ref|), mean-abs <= u max(1, mean|ref|).
    Measured at D512 / d_ff 2048: max 0.022 (bound ~0.07), mean 1.9e-3
    (bound ~3.9e-3); a missing bias, ReLU or residual errs by 0.1 or more.
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


@pytest.mark.parametrize("B,T,D,pos0", [(2, 7, 8, 0), (3, 130, 512, 0), (1, 64, 1024, 4000)])
def test_positional_encoding_add(lib, B, T, D, pos0):
    x = si.round_bf16(si.normal(131, si.TENSOR_IDS["x_q"], (B, T, D)))
    xd = bf16_dev(si.f64_to_bf16_bits(x))
    out = lib.positional_encoding_add(xd, pos0=pos0)
    inplace = xd.clone()
    lib.positional_encoding_add(inplace, inplace, pos0=pos0)
    torch.cuda.synchronize()
    exact = x + oracle.positional_encoding(T, D, pos0)[None]
    err = np.abs(host(out) - exact)
    assert np.all(err <= 2.0 ** -8 * np.abs(exact) + 2e-3), err.max()
    assert torch.equal(out, inplace)


def encoder_inputs(w):
    x = si.make_inputs(w)
    p = si.encoder_params(w.seed, w.d_model, si.ENCODER_D_FF if w.d_model == 512 else 2 * w.d_model)
    for n in ("w_q", "w_k", "w_v", "w_o"):
        p[n], p[n + "_bits"] = x[n], x[n + "_bits"]
    return x, p


def run_encoder(lib, w, x, p):
    params = {n: bf16_dev(p[n + "_bits"]) for n in lib.ENCODER_PARAMS}
    lens = None if x["key_lens"] is None else torch.from_numpy(x["key_lens"]).to(dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    out = lib.encoder_layer_forward(bf16_dev(x["x_q_bits"]), params, w.h, scale=w.scale,
                                    mask=w.mask, key_lens=lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return host(out)


U = 2.0 ** -8


def check_normalised(got, ref, what):
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    big = 4 * U * max(1.0, float(np.abs(ref).max()))
    avg = U * max(1.0, float(np.abs(ref).mean()))
    assert err.max() <= big and err.mean() <= avg, "%s: max %.4g (bound %.3g) mean %.4g (bound %.3g)" % (
        what, err.max(), big, err.mean(), avg)


@pytest.mark.parametrize("B,T,D,h,mask", [(2, 130, 128, 2, si.MASK_KEY_PADDING),
                                          (1, 300, 512, 8, si.MASK_NONE),
                                          (2, 200, 1024, 16, si.MASK_CAUSAL)])
def test_encoder_layer_vs_oracle(lib, B, T, D, h, mask):
    w = si.WORKLOADS[6].replace(B=B, T_q=T, T_k=T, d_model=D, h=h, mask=mask, len_lo=1, len_hi=T,
                                seed=132)
    x, p = encoder_inputs(w)
    ref = oracle.encoder_layer(x["x_q"], p, h=h, eps=1e-5, scale=w.scale, mask=mask,
                               key_lens=x["key_lens"])
    check_normalised(run_encoder(lib, w, x, p), ref, "encoder B%d T%d D%d" % (B, T, D))


def test_encoder_layer_workload_full(lib):
    w = si.WORKLOADS[6]
    x, p = encoder_inputs(w)
    ref = oracle.encoder_layer(x["x_q"], p, h=w.h, eps=1e-5, scale=w.scale, mask=w.mask,
                               key_lens=x["key_lens"])
    check_normalised(run_encoder(lib, w, x, p), ref, w.name)
