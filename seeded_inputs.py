"""Seeded synthetic inputs for the attention workloads.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark.  It holds no attention arithmetic: only random-number
generation, bf16 storage rounding and the table of workloads.

Generator (fixed definition, reproducible on any host):

* one SplitMix64 stream per (seed, tensor id): the stream's starting state is
  ``mix64(seed * 0x9E3779B97F4A7C15 + tensor_id * 0xD1B54A32D192ED03 + 1)``
  and element ``i`` is ``mix64(state + (i + 1) * 0x9E3779B97F4A7C15)``
  (the SplitMix64 output sequence; ``mix64`` is its finaliser);
* uniforms ``u = (x >> 11) * 2**-53`` in [0, 1);
* normals by Box-Muller on consecutive pairs (u1, u2):
  ``r = sqrt(-2 ln(1 - u1))``, ``z0 = r cos(2 pi u2)``, ``z1 = r sin(2 pi u2)``;
* values are rounded to fp32 (round-to-nearest-even) and, for bf16 tensors,
  then to bf16 (round-to-nearest-even on the fp32 bits).  The stored value is
  the input: both sides read the same bits.

Tensor ids: X_q 0, X_kv 1, Q 2, K 3, V 4, W^Q 5, W^K 6, W^V 7, W^O 8,
key lengths 9.  Seed = workload number - 1.

Weights are Xavier-uniform: U(-a, a) with a = sqrt(6 / (fan_in + fan_out))
taken over the full d_model x d_model matrix, i.e. a = sqrt(3 / d_model).
Key lengths are ``lo + floor(u * (hi - lo + 1))``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_TID_MUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TENSOR_IDS = {"x_q": 0, "x_kv": 1, "q": 2, "k": 3, "v": 4,
              "w_q": 5, "w_k": 6, "w_v": 7, "w_o": 8, "key_lens": 9,
              "ln_gamma": 10, "ln_beta": 11, "dout": 12,
              "ffn_w1": 13, "ffn_b1": 14, "ffn_w2": 15, "ffn_b2": 16, "ln2_gamma": 17,
              "ln2_beta": 18}

MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_CAUSAL_KEY_PADDING = 0, 1, 2, 3


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _stream(seed: int, tensor_id: int, n: int) -> np.ndarray:
    base = (np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * _GOLDEN
            + np.uint64(tensor_id) * _TID_MUL + np.uint64(1))
    state = _mix64(np.array([base], dtype=np.uint64))[0]
    idx = np.arange(1, n + 1, dtype=np.uint64)
    return _mix64(state + idx * _GOLDEN)


def uniform01(seed: int, tensor_id: int, n: int) -> np.ndarray:
    """n doubles uniform in [0, 1)."""
    with np.errstate(over="ignore"):
        x = _stream(seed, tensor_id, n)
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tensor_id: int, shape) -> np.ndarray:
    """N(0, 1) doubles of the given shape (Box-Muller), rounded to fp32."""
    n = int(np.prod(shape)) if len(shape) else 1
    m = (n + 1) // 2
    u = uniform01(seed, tensor_id, 2 * m)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n].astype(np.float32).astype(np.float64).reshape(shape)


def xavier_uniform(seed: int, tensor_id: int, shape, fan_in: int, fan_out: int) -> np.ndarray:
    a = math.sqrt(6.0 / (fan_in + fan_out))
    u = uniform01(seed, tensor_id, int(np.prod(shape)))
    return ((2.0 * u - 1.0) * a).astype(np.float32).astype(np.float64).reshape(shape)


def key_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    u = uniform01(seed, TENSOR_IDS["key_lens"], batch)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int32)


def layernorm_params(seed: int, d_model: int) -> dict:
    """Gain and shift of a layer normalisation, bf16: gamma = 1 + N(0,1)/8,
    beta = N(0,1)/8 (learned values near their usual initialisation 1 and 0).
    Returns float64 values and raw bits under 'gamma', 'beta', '*_bits'."""
    out = {}
    for name, base in (("gamma", 1.0), ("beta", 0.0)):
        val = round_bf16(base + normal(seed, TENSOR_IDS["ln_" + name], (d_model,)) / 8.0)
        out[name] = val
        out[name + "_bits"] = f64_to_bf16_bits(val)
    return out


def encoder_params(seed: int, d_model: int, d_ff: int) -> dict:
    """Parameters of one encoder layer beyond the attention projections
    (which make_inputs draws): layer-norm gains and shifts of both sublayers
    (as layernorm_params) and the feed-forward network W1 (d_model, d_ff),
    b1, W2 (d_ff, d_model), b2 -- Xavier-uniform matrices, N(0,1)/8 biases --
    all rounded to bf16.  Float64 values and raw bits under '*_bits'."""
    out = {}
    ln1 = layernorm_params(seed, d_model)
    out.update({"gamma1": ln1["gamma"], "beta1": ln1["beta"]})
    for name, base in (("gamma2", 1.0), ("beta2", 0.0)):
        tid = TENSOR_IDS["ln2_" + name[:-1]]
        out[name] = round_bf16(base + normal(seed, tid, (d_model,)) / 8.0)
    out["w1"] = round_bf16(xavier_uniform(seed, TENSOR_IDS["ffn_w1"], (d_model, d_ff), d_model, d_ff))
    out["w2"] = round_bf16(xavier_uniform(seed, TENSOR_IDS["ffn_w2"], (d_ff, d_model), d_ff, d_model))
    out["b1"] = round_bf16(normal(seed, TENSOR_IDS["ffn_b1"], (d_ff,)) / 8.0)
    out["b2"] = round_bf16(normal(seed, TENSOR_IDS["ffn_b2"], (d_model,)) / 8.0)
    for name in list(out):
        out[name + "_bits"] = f64_to_bf16_bits(out[name])
    return out


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round (via fp32, RNE) to bf16 and return the raw uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f64(f64_to_bf16_bits(x))


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention workload.  kind is 'sdpa' (Q, K, V given) or 'mha'
    (X_q, X_kv and the four projection matrices given)."""
    name: str
    kind: str
    dtype: str              # "f32" or "bf16"
    B: int
    h: int
    T_q: int
    T_k: int
    d_k: int = 64
    d_v: int = 64
    d_model: int = 0
    mask: int = MASK_NONE
    len_lo: int = 0
    len_hi: int = 0
    cross: bool = False     # MHA: X_kv is a separate tensor
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_k)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = [
    Workload("sdpa_f32_B1_h8_T16_d64", "sdpa", "f32", B=1, h=8, T_q=16, T_k=16, seed=0),
    Workload("mha_self_pad_D512_h8_B32_T128", "mha", "bf16", B=32, h=8, T_q=128, T_k=128,
             d_model=512, mask=MASK_KEY_PADDING, len_lo=64, len_hi=128, seed=1),
    Workload("mha_causal_D512_h8_B16_T512", "mha", "bf16", B=16, h=8, T_q=512, T_k=512,
             d_model=512, mask=MASK_CAUSAL, seed=2),
    Workload("mha_cross_pad_D1024_h16_B8_Tq256_Tk1024", "mha", "bf16", B=8, h=16, T_q=256,
             T_k=1024, d_model=1024, mask=MASK_KEY_PADDING, len_lo=512, len_hi=1024,
             cross=True, seed=3),
    Workload("sdpa_causal_bf16_B2_h16_T8192_d64", "sdpa", "bf16", B=2, h=16, T_q=8192,
             T_k=8192, mask=MASK_CAUSAL, seed=4),
    # Decoding: one new query row per sequence against a key/value cache of
    # 8192 slots, of which the first len_b (uniform in [2048, 8192]) hold keys.
    Workload("decode_bf16_B16_h16_Tq1_cache8192", "sdpa", "bf16", B=16, h=16, T_q=1,
             T_k=8192, mask=MASK_KEY_PADDING, len_lo=2048, len_hi=8192, seed=5),
    # One encoder layer of the base model (d_model 512, 8 heads, d_ff 2048):
    # attention sublayer + feed-forward sublayer, each with residual and
    # layer normalisation; inputs as the MHA workloads, d_ff in ENCODER_D_FF.
    Workload("encoder_layer_D512_h8_ff2048_B16_T512", "mha", "bf16", B=16, h=8, T_q=512,
             T_k=512, d_model=512, mask=MASK_KEY_PADDING, len_lo=256, len_hi=512, seed=6),
]
ENCODER_D_FF = 2048


def make_inputs(w: Workload) -> dict:
    """Generate the workload's inputs.  Returns float64 arrays of the stored
    values (exactly representable in the workload's dtype) plus, for bf16
    workloads, the raw uint16 bits under '<name>_bits'."""
    out: dict = {}
    rnd = round_bf16 if w.dtype == "bf16" else (lambda a: a)

    def put(name, val):
        val = rnd(val)
        out[name] = val
        if w.dtype == "bf16":
            out[name + "_bits"] = f64_to_bf16_bits(val)

    if w.kind == "sdpa":
        put("q", normal(w.seed, TENSOR_IDS["q"], (w.B, w.h, w.T_q, w.d_k)))
        put("k", normal(w.seed, TENSOR_IDS["k"], (w.B, w.h, w.T_k, w.d_k)))
        put("v", normal(w.seed, TENSOR_IDS["v"], (w.B, w.h, w.T_k, w.d_v)))
    else:
        D = w.d_model
        put("x_q", normal(w.seed, TENSOR_IDS["x_q"], (w.B, w.T_q, D)))
        if w.cross:
            put("x_kv", normal(w.seed, TENSOR_IDS["x_kv"], (w.B, w.T_k, D)))
        put("w_q", xavier_uniform(w.seed, TENSOR_IDS["w_q"], (D, w.h * w.d_k), D, w.h * w.d_k))
        put("w_k", xavier_uniform(w.seed, TENSOR_IDS["w_k"], (D, w.h * w.d_k), D, w.h * w.d_k))
        put("w_v", xavier_uniform(w.seed, TENSOR_IDS["w_v"], (D, w.h * w.d_v), D, w.h * w.d_v))
        put("w_o", xavier_uniform(w.seed, TENSOR_IDS["w_o"], (w.h * w.d_v, D), w.h * w.d_v, D))
    if w.mask in (MASK_KEY_PADDING, MASK_CAUSAL_KEY_PADDING):
        out["key_lens"] = key_lengths(w.seed, w.B, w.len_lo, w.len_hi)
    else:
        out["key_lens"] = None
    return out
