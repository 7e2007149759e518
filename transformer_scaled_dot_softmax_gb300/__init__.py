"""GB300 (sm_103a) multi-head scaled dot-product attention forward.

A thin binding over the C ABI of libmha.so (include/mha.h): these functions
only marshal arguments -- every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the stream.

    out = sdpa_forward(q, k, v, mask="causal")            # (B, h, T, 64) bf16
    out = sdpa_decode_forward(q, k_cache, v_cache, lens)   # (B, h, T_q <= 8, 64) bf16
    out = mha_forward(x_q, x_kv, w_q, w_k, w_v, w_o, h=8)  # (B, T, d_model) bf16
"""
from __future__ import annotations

import math

from . import _native
from ._native import (MHA_BF16, MHA_F32, MHA_MASK_CAUSAL, MHA_MASK_CAUSAL_KEY_PADDING,
                      MHA_MASK_KEY_PADDING, MHA_MASK_NONE, MHA_OK, lib)

__all__ = ["sdpa_forward", "sdpa_forward_lse", "sdpa_forward_host", "sdpa_forward_host_workspace_bytes",
           "sdpa_bf16_key_split", "sdpa_backward", "positional_encoding_add",
           "encoder_layer_forward", "ENCODER_PARAMS", "sdpa_decode_forward", "mha_forward", "mha_forward_add_layernorm", "mha_workspace_bytes", "status_string", "MhaError",
           "MASKS", "lib"]

MASKS = {"none": MHA_MASK_NONE, "causal": MHA_MASK_CAUSAL, "key_padding": MHA_MASK_KEY_PADDING,
         "causal_key_padding": MHA_MASK_CAUSAL_KEY_PADDING}


class MhaError(RuntimeError):
    def __init__(self, code: int, what: str):
        detail = lib.mha_last_error().decode() if code == _native.MHA_ERR_CUDA else ""
        super().__init__("%s: %s (status %d)%s" % (what, status_string(code), code,
                                                   " -- " + detail if detail else ""))
        self.code = code


def status_string(code: int) -> str:
    return lib.mha_status_string(int(code)).decode()


def _mask_code(mask) -> int:
    if isinstance(mask, str):
        return MASKS[mask]
    return int(mask)


def _torch():
    import torch
    return torch


def _stream_handle(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_dev(name, t, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s" % (name, dtype))


def sdpa_forward(q, k, v, out=None, *, scale=None, mask="none", key_lens=None, status=None,
                 stream=None):
    """softmax(scale * q k^T + mask) v for q (B,h,T_q,d_k), k (B,h,T_k,d_k),
    v (B,h,T_k,d_v); fp32 or bf16 CUDA tensors.  Returns out (B,h,T_q,d_v)."""
    torch = _torch()
    dtype = q.dtype
    if dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_dev(n, t, dtype)
    B, h, T_q, d_k = q.shape
    T_k, d_v = k.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, h, T_q, d_v), dtype=dtype, device=q.device)
    _check_dev("out", out, dtype)
    if key_lens is not None:
        _check_dev("key_lens", key_lens, torch.int32)
    if status is not None:
        _check_dev("status", status, torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    rc = lib.sdpa_forward(MHA_F32 if dtype == torch.float32 else MHA_BF16, _ptr(q), _ptr(k),
                          _ptr(v), _ptr(out), B, h, T_q, T_k, d_k, d_v, float(scale),
                          _mask_code(mask), _ptr(key_lens), _ptr(status), _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "sdpa_forward")
    return out


def sdpa_forward_lse(q, k, v, out=None, lse=None, *, scale=None, mask="none", key_lens=None,
                     status=None, stream=None):
    """sdpa_forward for bf16 tensors that also returns the per-row
    log-sum-exp of the visible scores, lse (B,h,T_q) fp32 (natural log; -inf
    for a row with no visible key).  Returns (out, lse)."""
    torch = _torch()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_dev(n, t, torch.bfloat16)
    B, h, T_q, d_k = q.shape
    T_k, d_v = k.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, h, T_q, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, h, T_q), dtype=torch.float32, device=q.device)
    _check_dev("out", out, torch.bfloat16)
    _check_dev("lse", lse, torch.float32)
    if key_lens is not None:
        _check_dev("key_lens", key_lens, torch.int32)
    if status is not None:
        _check_dev("status", status, torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    rc = lib.sdpa_forward_lse(MHA_BF16, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, h,
                              T_q, T_k, d_k, d_v, float(scale), _mask_code(mask), _ptr(key_lens),
                              _ptr(status), _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "sdpa_forward_lse")
    return out, lse


def _check_host(name, t, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError("%s must be a CPU tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s" % (name, dtype))


def sdpa_bf16_key_split(T_q, T_k, mask="none") -> int:
    """1 if the bf16 attention kernel splits a row's keys between its two
    softmax groups by alternate tiles for this shape, 0 if by key halves."""
    r = int(lib.sdpa_bf16_key_split(T_q, T_k, _mask_code(mask)))
    if r < 0:
        raise ValueError("invalid shape or mask")
    return r


def sdpa_forward_host_workspace_bytes(B, h, T_q, T_k, d_k=64, d_v=64, dtype=None) -> int:
    torch = _torch()
    dt = MHA_F32 if dtype == torch.float32 else MHA_BF16
    return int(lib.sdpa_forward_host_workspace_bytes(dt, B, h, T_q, T_k, d_k, d_v))


def sdpa_forward_host(q, k, v, out=None, workspace=None, *, scale=None, mask="none", key_lens=None,
                      status=None, stream=None):
    """sdpa_forward with q, k, v, out (and key_lens) in host memory (CPU
    tensors, page-locked for overlapped copies) and a device workspace; the
    library copies, computes and copies back in chunks that overlap.  The
    result is in `out` once `stream` has been synchronised.  Returns out."""
    torch = _torch()
    dtype = q.dtype
    if dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_host(n, t, dtype)
    B, h, T_q, d_k = q.shape
    T_k, d_v = k.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, h, T_q, d_v), dtype=dtype, pin_memory=torch.cuda.is_available())
    _check_host("out", out, dtype)
    if key_lens is not None:
        _check_host("key_lens", key_lens, torch.int32)
    if status is not None:
        _check_dev("status", status, torch.int32)
    dt = MHA_F32 if dtype == torch.float32 else MHA_BF16
    need = int(lib.sdpa_forward_host_workspace_bytes(dt, B, h, T_q, T_k, d_k, d_v))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    _check_dev("workspace", workspace)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    rc = lib.sdpa_forward_host(dt, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), B, h, T_q, T_k, d_k,
                               d_v, float(scale), _mask_code(mask), _ptr(key_lens), _ptr(status),
                               _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "sdpa_forward_host")
    return out


def sdpa_backward(q, k, v, o, dout, lse, dq=None, dk=None, dv=None, workspace=None, *,
                  scale=None, mask="none", key_lens=None, status=None, stream=None):
    """Gradients (dq, dk, dv) of sdpa_forward for bf16 tensors, from the
    forward's output o and log-sum-exp lse (sdpa_forward_lse) and the output
    gradient dout."""
    torch = _torch()
    bf = torch.bfloat16
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_dev(n, t, bf)
    _check_dev("lse", lse, torch.float32)
    B, h, T_q, d_k = q.shape
    T_k, d_v = k.shape[2], v.shape[3]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_dev(n, t, bf)
    need = int(lib.sdpa_backward_workspace_bytes(B, h, T_q, T_k, d_k, d_v))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check_dev("workspace", workspace)
    if key_lens is not None:
        _check_dev("key_lens", key_lens, torch.int32)
    if status is not None:
        _check_dev("status", status, torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    rc = lib.sdpa_backward(MHA_BF16, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                           _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), B, h, T_q, T_k, d_k,
                           d_v, float(scale), _mask_code(mask), _ptr(key_lens), _ptr(status),
                           _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "sdpa_backward")
    return dq, dk, dv


def positional_encoding_add(x, out=None, *, pos0=0, stream=None):
    """x + PE(pos0 + t) for bf16 embedding rows x (B, T, d_model); out may be x."""
    torch = _torch()
    _check_dev("x", x, torch.bfloat16)
    B, T, D = x.shape
    out = torch.empty_like(x) if out is None else out
    _check_dev("out", out, torch.bfloat16)
    rc = lib.positional_encoding_add(_ptr(x), _ptr(out), B, T, D, int(pos0), _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "positional_encoding_add")
    return out


ENCODER_PARAMS = ("w_q", "w_k", "w_v", "w_o", "gamma1", "beta1", "w1", "b1", "w2", "b2", "gamma2",
                  "beta2")


def encoder_layer_forward(x, params, h, out=None, workspace=None, *, eps=1e-5, scale=None,
                          mask="none", key_lens=None, status=None, stream=None):
    """One post-LN encoder layer: y = LN1(x + MHA(x, x)), out = LN2(y + FFN(y)).
    params: dict of bf16 CUDA tensors named as ENCODER_PARAMS (W^Q..W^O
    (D, D), gamma/beta (D), w1 (D, F), b1 (F), w2 (F, D), b2 (D))."""
    torch = _torch()
    bf = torch.bfloat16
    _check_dev("x", x, bf)
    for n in ENCODER_PARAMS:
        _check_dev(n, params[n], bf)
    B, T, D = x.shape
    F = params["w1"].shape[1]
    out = torch.empty_like(x) if out is None else out
    _check_dev("out", out, bf)
    need = int(lib.encoder_layer_workspace_bytes(B, T, D, h, F))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check_dev("workspace", workspace)
    if key_lens is not None:
        _check_dev("key_lens", key_lens, torch.int32)
    if status is not None:
        _check_dev("status", status, torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(D // h)
    rc = lib.encoder_layer_forward(_ptr(x), *[_ptr(params[n]) for n in ENCODER_PARAMS], float(eps),
                                   _ptr(out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), B, T, D, h, F,
                                   float(scale), _mask_code(mask), _ptr(key_lens), _ptr(status),
                                   _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "encoder_layer_forward")
    return out


def sdpa_decode_forward(q, k_cache, v_cache, cache_lens=None, out=None, *, scale=None,
                        stream=None):
    """Decoding step: each of the T_q (<= 8) query rows of q (B,h,T_q,64)
    attends to the first cache_lens[b] rows of k_cache / v_cache
    (B,h,T_k,64); bf16 CUDA tensors, cache_lens int32 on the device (None:
    all T_k).  Returns out (B,h,T_q,64)."""
    torch = _torch()
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _check_dev(n, t, torch.bfloat16)
    B, h, T_q, d_k = q.shape
    T_k, d_v = k_cache.shape[2], v_cache.shape[3]
    if out is None:
        out = torch.empty((B, h, T_q, d_v), dtype=torch.bfloat16, device=q.device)
    _check_dev("out", out, torch.bfloat16)
    if cache_lens is not None:
        _check_dev("cache_lens", cache_lens, torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    rc = lib.sdpa_decode_forward(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), B, h, T_q,
                                 T_k, d_k, d_v, float(scale), _ptr(cache_lens),
                                 _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "sdpa_decode_forward")
    return out


def mha_workspace_bytes(B, h, T_q, T_k, d_k=64, d_v=64) -> int:
    return int(lib.mha_workspace_bytes(B, h, T_q, T_k, d_k, d_v))


def _mha_call(x_q, x_kv, w_q, w_k, w_v, w_o, h, out, workspace, scale, mask, key_lens, status,
              stream, ln):
    torch = _torch()
    bf = torch.bfloat16
    for n, t in (("x_q", x_q), ("x_kv", x_kv), ("w_q", w_q), ("w_k", w_k), ("w_v", w_v),
                 ("w_o", w_o)):
        _check_dev(n, t, bf)
    B, T_q, D = x_q.shape
    T_k = x_kv.shape[1]
    d_k = w_q.shape[1] // h
    d_v = w_v.shape[1] // h
    if out is None:
        out = torch.empty((B, T_q, D), dtype=bf, device=x_q.device)
    _check_dev("out", out, bf)
    need = mha_workspace_bytes(B, h, T_q, T_k, d_k, d_v)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x_q.device)
    _check_dev("workspace", workspace)
    if key_lens is not None:
        _check_dev("key_lens", key_lens, torch.int32)
    if status is not None:
        _check_dev("status", status, torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    ws = (_ptr(workspace), workspace.numel() * workspace.element_size())
    tail = (B, h, T_q, T_k, D, d_k, d_v, float(scale), _mask_code(mask), _ptr(key_lens),
            _ptr(status), _stream_handle(stream))
    if ln is None:
        rc = lib.mha_forward(MHA_BF16, _ptr(x_q), _ptr(x_kv), _ptr(w_q), _ptr(w_k), _ptr(w_v),
                             _ptr(w_o), _ptr(out), *ws, *tail)
        what = "mha_forward"
    else:
        gamma, beta, eps = ln
        _check_dev("gamma", gamma, bf)
        _check_dev("beta", beta, bf)
        if gamma.shape != (D,) or beta.shape != (D,):
            raise ValueError("gamma and beta must have d_model entries")
        rc = lib.mha_forward_add_layernorm(MHA_BF16, _ptr(x_q), _ptr(x_kv), _ptr(w_q), _ptr(w_k),
                                           _ptr(w_v), _ptr(w_o), _ptr(gamma), _ptr(beta),
                                           float(eps), _ptr(out), *ws, *tail)
        what = "mha_forward_add_layernorm"
    if rc != MHA_OK:
        raise MhaError(rc, what)
    return out


def mha_forward(x_q, x_kv, w_q, w_k, w_v, w_o, h, out=None, workspace=None, *, scale=None,
                mask="none", key_lens=None, status=None, stream=None):
    """Concat_i(softmax(scale (x_q W_i^Q)(x_kv W_i^K)^T + mask)(x_kv W_i^V)) W^O
    for bf16 CUDA tensors x_q (B,T_q,D), x_kv (B,T_k,D) (may be x_q),
    W^Q/W^K/W^V (D, h*64), W^O (h*64, D).  Returns out (B,T_q,D)."""
    return _mha_call(x_q, x_kv, w_q, w_k, w_v, w_o, h, out, workspace, scale, mask, key_lens,
                     status, stream, None)


def mha_forward_add_layernorm(x_q, x_kv, w_q, w_k, w_v, w_o, gamma, beta, h, eps=1e-5,
                              out=None, workspace=None, *, scale=None, mask="none",
                              key_lens=None, status=None, stream=None):
    """LayerNorm(x_q + mha_forward(...)) with gain gamma and shift beta (bf16,
    d_model entries each): the attention sublayer with its residual
    connection and post-normalisation.  Returns out (B,T_q,D)."""
    return _mha_call(x_q, x_kv, w_q, w_k, w_v, w_o, h, out, workspace, scale, mask, key_lens,
                     status, stream, (gamma, beta, eps))
