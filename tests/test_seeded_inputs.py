"""The seeded generator: deterministic, the stated distributions, and bf16
storage rounding that agrees with torch's own fp32 -> bf16 conversion."""
import math

import numpy as np
import pytest

import seeded_inputs as si


def test_streams_are_deterministic_and_distinct():
    a = si.uniform01(3, 2, 1000)
    b = si.uniform01(3, 2, 1000)
    c = si.uniform01(3, 3, 1000)
    d = si.uniform01(4, 2, 1000)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    assert a.min() >= 0.0 and a.max() < 1.0


def test_splitmix64_first_outputs():
    # SplitMix64 finaliser on a known input (published test vector of the
    # finaliser: mix64(0x9E3779B97F4A7C15) from a zero state).
    z = si._mix64(np.array([0x9E3779B97F4A7C15], dtype=np.uint64))[0]
    assert int(z) == 0xE220A8397B1DCDAF


def test_normal_moments():
    z = si.normal(0, 4, (200000,))
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    assert abs((np.abs(z) > 1.96).mean() - 0.05) < 0.003


def test_xavier_bound():
    D = 512
    w = si.xavier_uniform(1, 5, (D, D), D, D)
    a = math.sqrt(6.0 / (2 * D))
    assert abs(a - 0.07655) < 1e-4
    assert np.abs(w).max() <= a
    assert np.abs(w).max() > 0.99 * a
    assert abs(w.var() - a * a / 3) < 0.02 * a * a


def test_key_lengths_range():
    L = si.key_lengths(1, 10000, 64, 128)
    assert L.min() == 64 and L.max() == 128
    assert L.dtype == np.int32


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = si.normal(7, 2, (100000,)) * 37.0
    x = np.concatenate([x, [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65504.0]])
    mine = si.f64_to_bf16_bits(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    np.testing.assert_array_equal(mine, ref.view(np.uint16))
    back = si.bf16_bits_to_f64(mine)
    np.testing.assert_array_equal(back, torch.from_numpy(x.astype(np.float32)).to(
        torch.bfloat16).to(torch.float64).numpy())


def test_workload_table_matches_stated_shapes():
    w = si.WORKLOADS
    assert [x.seed for x in w] == [0, 1, 2, 3, 4, 5, 6]
    assert (w[0].B, w[0].h, w[0].T_q, w[0].dtype, w[0].scale) == (1, 8, 16, "f32", 0.125)
    assert (w[1].d_model, w[1].B, w[1].T_q, w[1].len_lo, w[1].len_hi) == (512, 32, 128, 64, 128)
    assert (w[2].B, w[2].T_q, w[2].mask) == (16, 512, si.MASK_CAUSAL)
    assert (w[3].d_model, w[3].h, w[3].T_q, w[3].T_k, w[3].cross) == (1024, 16, 256, 1024, True)
    assert (w[4].B, w[4].h, w[4].T_q, w[4].mask) == (2, 16, 8192, si.MASK_CAUSAL)
    assert (w[5].B, w[5].h, w[5].T_q, w[5].T_k, w[5].mask, w[5].len_lo, w[5].len_hi) == (
        16, 16, 1, 8192, si.MASK_KEY_PADDING, 2048, 8192)
    assert (w[6].d_model, w[6].h, w[6].B, w[6].T_q, si.ENCODER_D_FF) == (512, 8, 16, 512, 2048)


def test_make_inputs_small():
    w = si.WORKLOADS[3].replace(B=2, T_q=8, T_k=16, d_model=32, h=2, d_k=16, d_v=16,
                                len_lo=8, len_hi=16)
    x = si.make_inputs(w)
    assert x["x_q"].shape == (2, 8, 32) and x["x_kv"].shape == (2, 16, 32)
    assert x["w_o"].shape == (32, 32)
    np.testing.assert_array_equal(si.bf16_bits_to_f64(x["x_q_bits"]), x["x_q"])
    assert x["key_lens"].shape == (2,)
