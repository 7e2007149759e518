"""fp64 CPU oracle for scaled dot-product and multi-head attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the benchmark's CPU-baseline leg, never by the product path.  It shares
no code with the CUDA library; the only module both sides use is the seeded
input generator.

The arithmetic lives in ``mha_oracle.c`` (plain C, fp64, libm ``exp``); this
module only marshals numpy arrays through ctypes.  See that file's header for
what is computed and which passage of the pages each step follows.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_CAUSAL_KEY_PADDING = 0, 1, 2, 3

_lib = None


def _load():
    global _lib
    if _lib is None:
        # A test that plants a mistake in a copy of the oracle points this
        # variable at the planted build; nothing else sets it.
        path = os.environ.get("MHA_ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        lp = ctypes.POINTER(ctypes.c_int64)
        ci, cd, cl = ctypes.c_int, ctypes.c_double, ctypes.c_long
        lib.oracle_sdpa.argtypes = [dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, cd, ci, ip]
        lib.oracle_sdpa.restype = ci
        lib.oracle_sdpa_rows.argtypes = [dp, dp, dp, dp, lp, cl, ci, ci, ci, ci, ci, ci, cd,
                                         ci, ip]
        lib.oracle_sdpa_rows.restype = ci
        lib.oracle_mha.argtypes = [dp, dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, ci, cd,
                                   ci, ip, lp, cl]
        lib.oracle_mha.restype = ci
        lib.oracle_sdpa_lse.argtypes = [dp, dp, dp, ci, ci, ci, ci, ci, cd, ci, ip]
        lib.oracle_sdpa_lse.restype = ci
        lib.oracle_sdpa_backward.argtypes = [dp, dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, cd,
                                             ci, ip]
        lib.oracle_sdpa_backward.restype = ci
        lib.oracle_sdpa_backward_tail.argtypes = [dp, dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci,
                                                  cd, ci, ip, ci]
        lib.oracle_sdpa_backward_tail.restype = ci
        lib.oracle_positional_encoding.argtypes = [dp, ci, ci, ci]
        lib.oracle_positional_encoding.restype = ci
        lib.oracle_ffn.argtypes = [dp, dp, dp, dp, dp, dp, cl, ci, ci]
        lib.oracle_ffn.restype = ci
        lib.oracle_add_layernorm.argtypes = [dp, dp, dp, dp, cd, dp, cl, ci]
        lib.oracle_add_layernorm.restype = ci
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ci
        lib.oracle_set_num_threads.argtypes = [ci]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
    return _lib


def _d(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a, t=ctypes.c_double):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(t))


def _lens(key_lens, B):
    if key_lens is None:
        return None
    kl = np.ascontiguousarray(key_lens, dtype=np.int32)
    if kl.shape != (B,):
        raise ValueError("key_lens must have B entries")
    return kl


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the following calls (timing only; results do not depend
    on it)."""
    _load().oracle_set_num_threads(int(n))


def sdpa(q, k, v, scale=None, mask=MASK_NONE, key_lens=None, return_weights=False):
    """softmax(scale * q k^T + mask) v for q (B,H,Tq,dk), k (B,H,Tk,dk),
    v (B,H,Tk,dv).  Returns o (B,H,Tq,dv) [and weights (B,H,Tq,Tk)]."""
    q, k, v = _d(q), _d(k), _d(v)
    B, H, Tq, dk = q.shape
    Tk, dv = k.shape[2], v.shape[3]
    if k.shape != (B, H, Tk, dk) or v.shape != (B, H, Tk, dv):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    kl = _lens(key_lens, B)
    o = np.empty((B, H, Tq, dv))
    w = np.empty((B, H, Tq, Tk)) if return_weights else None
    rc = _load().oracle_sdpa(_p(q), _p(k), _p(v), _p(o), _p(w), B, H, Tq, Tk, dk, dv,
                             float(scale), int(mask), _p(kl, ctypes.c_int32))
    if rc:
        raise RuntimeError("oracle_sdpa failed")
    return (o, w) if return_weights else o


def sdpa_rows(q, k, v, rows, scale=None, mask=MASK_NONE, key_lens=None):
    """Output rows only: rows are flat indices (b*H + h)*Tq + i.  Returns
    (len(rows), dv)."""
    q, k, v = _d(q), _d(k), _d(v)
    B, H, Tq, dk = q.shape
    Tk, dv = k.shape[2], v.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    kl = _lens(key_lens, B)
    o = np.empty((len(r), dv))
    rc = _load().oracle_sdpa_rows(_p(q), _p(k), _p(v), _p(o), _p(r, ctypes.c_int64), len(r),
                                  B, H, Tq, Tk, dk, dv, float(scale), int(mask),
                                  _p(kl, ctypes.c_int32))
    if rc:
        raise RuntimeError("oracle_sdpa_rows failed")
    return o


def mha(x_q, x_kv, w_q, w_k, w_v, w_o, h, scale=None, mask=MASK_NONE, key_lens=None,
        query_rows=None):
    """Concat_i(softmax(scale (x_q W_i^Q)(x_kv W_i^K)^T + mask) x_kv W_i^V) W^O.
    x_q (B,Tq,D), x_kv (B,Tk,D), W^Q/W^K (D,h*dk), W^V (D,h*dv), W^O (h*dv,D).
    Returns (B,Tq,D), or (len(query_rows), D) for flat query rows b*Tq + i."""
    x_q, x_kv = _d(x_q), _d(x_kv)
    w_q, w_k, w_v, w_o = _d(w_q), _d(w_k), _d(w_v), _d(w_o)
    B, Tq, D = x_q.shape
    Tk = x_kv.shape[1]
    dk = w_q.shape[1] // h
    dv = w_v.shape[1] // h
    if (x_kv.shape != (B, Tk, D) or w_q.shape != (D, h * dk) or w_k.shape != (D, h * dk)
            or w_v.shape != (D, h * dv) or w_o.shape != (h * dv, D)):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    kl = _lens(key_lens, B)
    if query_rows is None:
        out = np.empty((B, Tq, D))
        qr, n = None, 0
    else:
        qr = np.ascontiguousarray(query_rows, dtype=np.int64)
        n = len(qr)
        out = np.empty((n, D))
    rc = _load().oracle_mha(_p(x_q), _p(x_kv), _p(w_q), _p(w_k), _p(w_v), _p(w_o), _p(out),
                            B, h, Tq, Tk, D, dk, dv, float(scale), int(mask),
                            _p(kl, ctypes.c_int32), _p(qr, ctypes.c_int64), n)
    if rc:
        raise RuntimeError("oracle_mha failed")
    return out


def add_layernorm(x, s, gamma, beta, eps=1e-5):
    """LayerNorm(x + s) over the last axis with gain gamma and shift beta:
    (v - mean) / sqrt(population variance + eps) * gamma + beta, v = x + s."""
    x, s = _d(x), _d(s)
    gamma, beta = _d(gamma), _d(beta)
    if x.shape != s.shape or gamma.shape != (x.shape[-1],) or beta.shape != gamma.shape:
        raise ValueError("shape mismatch")
    D = x.shape[-1]
    y = np.empty(x.shape)
    rc = _load().oracle_add_layernorm(_p(x), _p(s), _p(gamma), _p(beta), float(eps), _p(y),
                                      x.size // D, D)
    if rc:
        raise RuntimeError("oracle_add_layernorm failed")
    return y


def mha_add_layernorm(x_q, x_kv, w_q, w_k, w_v, w_o, gamma, beta, h, eps=1e-5, scale=None,
                      mask=MASK_NONE, key_lens=None, query_rows=None):
    """The attention sublayer with its residual and normalisation:
    LayerNorm(x_q + MultiHead(x_q, x_kv)).  Shapes as mha(); query_rows
    selects flat rows b*Tq + i."""
    out = mha(x_q, x_kv, w_q, w_k, w_v, w_o, h, scale=scale, mask=mask, key_lens=key_lens,
              query_rows=query_rows)
    xq = _d(x_q).reshape(-1, out.shape[-1])
    res = xq if query_rows is None else xq[np.asarray(query_rows, dtype=np.int64)]
    return add_layernorm(res.reshape(out.shape), out, gamma, beta, eps)


def sdpa_lse(q, k, scale=None, mask=MASK_NONE, key_lens=None):
    """Per query row log sum_{visible j} exp(scale q.k_j), shape (B,H,Tq);
    -inf for a row with no visible key."""
    q, k = _d(q), _d(k)
    B, H, Tq, dk = q.shape
    Tk = k.shape[2]
    if k.shape != (B, H, Tk, dk):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    kl = _lens(key_lens, B)
    lse = np.empty((B, H, Tq))
    rc = _load().oracle_sdpa_lse(_p(q), _p(k), _p(lse), B, H, Tq, Tk, dk, float(scale),
                                 int(mask), _p(kl, ctypes.c_int32))
    if rc:
        raise RuntimeError("oracle_sdpa_lse failed")
    return lse


def sdpa_backward(q, k, v, dout, scale=None, mask=MASK_NONE, key_lens=None):
    """Gradients (dq, dk, dv) of sdpa(q, k, v) for the output gradient dout
    (same shape as the output); d_k == d_v."""
    q, k, v, dout = _d(q), _d(k), _d(v), _d(dout)
    B, H, Tq, d = q.shape
    Tk = k.shape[2]
    if k.shape != (B, H, Tk, d) or v.shape != (B, H, Tk, d) or dout.shape != (B, H, Tq, d):
        raise ValueError("shape mismatch (d_k must equal d_v)")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _lens(key_lens, B)
    dq, dk, dv = np.empty(q.shape), np.empty(k.shape), np.empty(v.shape)
    rc = _load().oracle_sdpa_backward(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv), B, H,
                                      Tq, Tk, d, float(scale), int(mask), _p(kl, ctypes.c_int32))
    if rc:
        raise RuntimeError("oracle_sdpa_backward failed")
    return dq, dk, dv


def sdpa_backward_tail(q, k, v, dout, i0, scale=None, mask=MASK_CAUSAL, key_lens=None):
    """sdpa_backward summed over the query rows i >= i0 only: dq[..., i0:, :]
    is the full gradient, and with a causal mask so are dk[..., i0:, :] and
    dv[..., i0:, :] (no row before i0 sees those keys); dq rows before i0 are
    0, dk and dv rows before i0 partial."""
    q, k, v, dout = _d(q), _d(k), _d(v), _d(dout)
    B, H, Tq, d = q.shape
    Tk = k.shape[2]
    if k.shape != (B, H, Tk, d) or v.shape != (B, H, Tk, d) or dout.shape != (B, H, Tq, d):
        raise ValueError("shape mismatch (d_k must equal d_v)")
    if not 0 <= i0 <= Tq:
        raise ValueError("i0 out of range")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _lens(key_lens, B)
    dq, dk, dv = np.empty(q.shape), np.empty(k.shape), np.empty(v.shape)
    rc = _load().oracle_sdpa_backward_tail(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv),
                                           B, H, Tq, Tk, d, float(scale), int(mask),
                                           _p(kl, ctypes.c_int32), int(i0))
    if rc:
        raise RuntimeError("oracle_sdpa_backward_tail failed")
    return dq, dk, dv


def positional_encoding(T, D, pos0=0):
    """(T, D) table: PE(pos, 2i) = sin(pos / 10000^(2i/D)), PE(pos, 2i+1) =
    cos(pos / 10000^(2i/D)) for pos = pos0 .. pos0+T-1."""
    pe = np.empty((T, D))
    if _load().oracle_positional_encoding(_p(pe), int(T), int(D), int(pos0)):
        raise RuntimeError("oracle_positional_encoding failed")
    return pe


def ffn(x, w1, b1, w2, b2):
    """max(0, x W1 + b1) W2 + b2 over the last axis of x."""
    x, w1, b1, w2, b2 = _d(x), _d(w1), _d(b1), _d(w2), _d(b2)
    D = x.shape[-1]
    F = w1.shape[1]
    if w1.shape != (D, F) or b1.shape != (F,) or w2.shape != (F, D) or b2.shape != (D,):
        raise ValueError("shape mismatch")
    y = np.empty(x.shape)
    if _load().oracle_ffn(_p(x), _p(w1), _p(b1), _p(w2), _p(b2), _p(y), x.size // D, D, F):
        raise RuntimeError("oracle_ffn failed")
    return y


def encoder_layer(x, p, h, eps=1e-5, scale=None, mask=MASK_NONE, key_lens=None):
    """One encoder layer with post-normalisation:
    y = LayerNorm1(x + MultiHead(x, x)), out = LayerNorm2(y + FFN(y)).
    p: dict with w_q, w_k, w_v, w_o, gamma1, beta1, w1, b1, w2, b2, gamma2, beta2."""
    y = mha_add_layernorm(x, x, p["w_q"], p["w_k"], p["w_v"], p["w_o"], p["gamma1"], p["beta1"],
                          h=h, eps=eps, scale=scale, mask=mask, key_lens=key_lens)
    return add_layernorm(y, ffn(y, p["w1"], p["b1"], p["w2"], p["b2"]), p["gamma2"], p["beta2"], eps)
