"""Pins for the fp64 oracle: what the pages and the mathematics fix, checked
without re-typing the oracle's own formula.

Each pin is chosen so that a plausible mistake in the oracle -- a dropped
scale, a transposed operand, a wrong mask index, heads concatenated in the
wrong order -- fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import MASK_CAUSAL, MASK_CAUSAL_KEY_PADDING, MASK_KEY_PADDING, MASK_NONE

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
ALL_MASKS = [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_CAUSAL_KEY_PADDING]


def _rng(seed):
    return np.random.default_rng(seed)


def _weights_for_scores(scores):
    """One query row whose scaled scores are `scores`: q = e_1, k_j = s_j e_1,
    scale 1, V = identity, so the output row is the weight vector."""
    n = len(scores)
    d = max(n, 2)
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, n, d))
    k[0, 0, :, 0] = scores
    v = np.eye(n).reshape(1, 1, n, n)
    o = oracle.sdpa(q, k, v, scale=1.0)
    return o[0, 0, 0]


@pytest.mark.parametrize("case", GOLDEN["softmax"], ids=lambda c: c["source"][:40])
def test_worked_softmax_examples(case):
    w = _weights_for_scores(case["scores"])
    np.testing.assert_allclose(w, case["weights"], atol=case["tol"] + 1e-15, rtol=0)


def test_worked_examples_closed_form():
    # 1/(1+e^-2) for the 12-vs-10 example; the three-score example exactly.
    w = _weights_for_scores([12.0, 10.0])
    assert abs(w[0] - 1.0 / (1.0 + math.exp(-2.0))) < 1e-15
    e = np.exp([2.0, 1.0, 0.5])
    np.testing.assert_allclose(_weights_for_scores([2.0, 1.0, 0.5]), e / e.sum(), rtol=0,
                               atol=1e-15)


def test_gap_of_four_winner_takes_nearly_all():
    g = GOLDEN["gap_winner"]
    w = _weights_for_scores([g["gap"], 0.0])
    assert w[0] >= g["min_winner_weight"]
    assert abs(w[0] - 1.0 / (1.0 + math.exp(-g["gap"]))) < 1e-15


def test_scale_is_division_by_sqrt_dk():
    g = GOLDEN["scale_by_sqrt_dk"]
    d = g["d_k"]
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, 2, d))
    k[0, 0, :, 0] = g["raw_dot_products"]
    v = np.eye(2).reshape(1, 1, 2, 2)
    w = oracle.sdpa(q, k, v)[0, 0, 0]  # default scale 1/sqrt(d_k)
    np.testing.assert_allclose(w, g["weights"], atol=g["tol"], rtol=0)


def test_causal_table_from_pages():
    t = GOLDEN["causal_table"]
    n = len(t["rows"])
    r = _rng(1)
    q = r.standard_normal((1, 1, n, 8))
    k = r.standard_normal((1, 1, n, 8))
    v = r.standard_normal((1, 1, n, 3))
    _, w = oracle.sdpa(q, k, v, mask=MASK_CAUSAL, return_weights=True)
    allowed = np.array(t["allowed"], dtype=bool)
    assert np.all(w[0, 0][~allowed] == 0.0)
    assert np.all(w[0, 0][allowed] > 0.0)


def _random_problem(seed, B=2, H=3, Tq=7, Tk=9, dk=5, dv=4, lens=None):
    r = _rng(seed)
    q = r.standard_normal((B, H, Tq, dk))
    k = r.standard_normal((B, H, Tk, dk))
    v = r.standard_normal((B, H, Tk, dv))
    if lens is None:
        lens = r.integers(1, Tk + 1, size=B).astype(np.int32)
    return q, k, v, lens


def _allowed(mask, lens, B, Tq, Tk):
    a = np.ones((B, Tq, Tk), dtype=bool)
    i = np.arange(Tq)[:, None]
    j = np.arange(Tk)[None, :]
    if mask & MASK_CAUSAL:
        a &= (j <= i)[None]
    if mask & MASK_KEY_PADDING:
        a &= (j[None] < lens[:, None, None])
    return a


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_rows_sum_to_one_and_masked_weights_zero(mask):
    q, k, v, lens = _random_problem(2)
    B, H, Tq, _ = q.shape
    Tk = k.shape[2]
    _, w = oracle.sdpa(q, k, v, mask=mask, key_lens=lens, return_weights=True)
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=0, atol=1e-14)
    allowed = _allowed(mask, lens, B, Tq, Tk)[:, None]
    allowed = np.broadcast_to(allowed, w.shape)
    assert np.all(w[~allowed] == 0.0)
    assert np.all(w[allowed] > 0.0)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_constant_values_give_constant_output(mask):
    q, k, v, lens = _random_problem(3)
    v[:] = 2.5
    o = oracle.sdpa(q, k, v, mask=mask, key_lens=lens)
    np.testing.assert_allclose(o, 2.5, rtol=0, atol=1e-14)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_identical_keys_average_the_visible_values(mask):
    q, k, v, lens = _random_problem(4)
    B, H, Tq, _ = q.shape
    Tk = k.shape[2]
    k[:] = k[:, :, :1, :]
    o = oracle.sdpa(q, k, v, mask=mask, key_lens=lens)
    allowed = _allowed(mask, lens, B, Tq, Tk)
    for b in range(B):
        for h in range(H):
            for i in range(Tq):
                vis = allowed[b, i]
                np.testing.assert_allclose(o[b, h, i], v[b, h, vis].mean(0), rtol=0, atol=1e-14)


def test_zero_query_averages_values():
    q, k, v, _ = _random_problem(5)
    q[:] = 0.0
    o = oracle.sdpa(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(2, keepdims=True), o.shape), rtol=0,
                               atol=1e-14)


def test_dominant_score_selects_its_value():
    q, k, v, _ = _random_problem(6, B=1, H=2, Tq=3, Tk=6, dk=4, dv=3)
    # make key 4 score 50 above every other key for every query
    q[:] = 0.0
    q[..., 0] = 1.0
    k[..., 0] = 0.0
    k[:, :, 4, 0] = 50.0
    o = oracle.sdpa(q, k, v, scale=1.0)
    bound = math.exp(-50.0) * 5 * np.abs(v).max() * 2
    np.testing.assert_allclose(o, np.broadcast_to(v[:, :, 4:5, :], o.shape), rtol=0,
                               atol=bound + 1e-15)


@pytest.mark.parametrize("mask", [MASK_KEY_PADDING, MASK_CAUSAL_KEY_PADDING])
def test_padding_equals_truncated_keys(mask):
    q, k, v, lens = _random_problem(7)
    o = oracle.sdpa(q, k, v, mask=mask, key_lens=lens)
    inner = MASK_CAUSAL if mask & MASK_CAUSAL else MASK_NONE
    for b in range(q.shape[0]):
        L = int(lens[b])
        ob = oracle.sdpa(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], mask=inner)
        np.testing.assert_allclose(o[b:b + 1], ob, rtol=0, atol=1e-14)


def test_causal_row_equals_prefix_problem():
    q, k, v, _ = _random_problem(8, Tq=6, Tk=6)
    o = oracle.sdpa(q, k, v, mask=MASK_CAUSAL)
    for i in range(6):
        oi = oracle.sdpa(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1])
        np.testing.assert_allclose(o[:, :, i:i + 1], oi, rtol=0, atol=1e-14)
    # row 0 sees only key 0
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_masked_keys_do_not_influence_output(mask):
    q, k, v, lens = _random_problem(9, Tq=9, Tk=9)
    o = oracle.sdpa(q, k, v, mask=mask, key_lens=lens)
    k2, v2 = k.copy(), v.copy()
    r = _rng(99)
    B = q.shape[0]
    for b in range(B):
        if mask & MASK_KEY_PADDING:
            L = int(lens[b])
            k2[b, :, L:] = r.standard_normal(k2[b, :, L:].shape) * 100
            v2[b, :, L:] = r.standard_normal(v2[b, :, L:].shape) * 100
    if mask & MASK_CAUSAL:
        # the last query row is the only one that may see the last key
        o_c = oracle.sdpa(q[:, :, :-1], k2, v2, mask=mask, key_lens=lens)
        k2[:, :, -1] = 1e3
        v2[:, :, -1] = -1e3
        o_c2 = oracle.sdpa(q[:, :, :-1], k2, v2, mask=mask, key_lens=lens)
        np.testing.assert_array_equal(o_c, o_c2)
    else:
        o2 = oracle.sdpa(q, k2, v2, mask=mask, key_lens=lens)
        np.testing.assert_array_equal(o, o2)


def test_key_value_permutation_leaves_output_unchanged():
    # notebook chapter, "Positional Encoding": attention is permutation-equivariant
    q, k, v, _ = _random_problem(10)
    perm = _rng(11).permutation(k.shape[2])
    o1 = oracle.sdpa(q, k, v)
    o2 = oracle.sdpa(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)


def test_query_permutation_permutes_output():
    q, k, v, _ = _random_problem(12)
    perm = _rng(13).permutation(q.shape[2])
    o1 = oracle.sdpa(q, k, v)
    o2 = oracle.sdpa(q[:, :, perm], k, v)
    np.testing.assert_allclose(o1[:, :, perm], o2, rtol=0, atol=1e-15)


def test_shift_of_all_keys_leaves_output_unchanged():
    q, k, v, _ = _random_problem(14)
    u = _rng(15).standard_normal(k.shape[-1])
    o1 = oracle.sdpa(q, k, v)
    o2 = oracle.sdpa(q, k + u, v)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_single_key_returns_its_value():
    q, k, v, _ = _random_problem(16, Tk=1)
    np.testing.assert_array_equal(oracle.sdpa(q, k, v), np.broadcast_to(v, (2, 3, 7, 4)))


def test_no_visible_key_gives_zero_row():
    # reading for a case the pages leave open (parity unpinned)
    q, k, v, _ = _random_problem(17, B=2, Tk=5)
    lens = np.array([0, 3], dtype=np.int32)
    o = oracle.sdpa(q, k, v, mask=MASK_KEY_PADDING, key_lens=lens)
    assert np.all(o[0] == 0.0)
    assert np.all(np.isfinite(o))


def _brute_force(q, k, v, scale, allowed):
    """Independent formulation in pure Python: w_j = 1 / sum_l exp(s_l - s_j)
    (no max subtraction), sums with math.fsum."""
    Tq, Tk = allowed.shape
    out = np.zeros((Tq, v.shape[1]))
    for i in range(Tq):
        s = [scale * math.fsum(float(q[i, c]) * float(k[j, c]) for c in range(q.shape[1]))
             for j in range(Tk)]
        vis = [j for j in range(Tk) if allowed[i, j]]
        for j in vis:
            wj = 1.0 / math.fsum(math.exp(s[l] - s[j]) for l in vis)
            for c in range(v.shape[1]):
                out[i, c] += wj * float(v[j, c])
    return out


@pytest.mark.parametrize("Tq,Tk", [(1, 1), (2, 3), (4, 4), (3, 2), (4, 1)])
@pytest.mark.parametrize("mask", ALL_MASKS)
def test_brute_force_tiny(Tq, Tk, mask):
    q, k, v, lens = _random_problem(100 + Tq * 10 + Tk, B=2, H=2, Tq=Tq, Tk=Tk, dk=3, dv=2)
    scale = 0.7
    o = oracle.sdpa(q, k, v, scale=scale, mask=mask, key_lens=lens)
    allowed = _allowed(mask, lens, 2, Tq, Tk)
    for b, h in itertools.product(range(2), range(2)):
        ref = _brute_force(q[b, h], k[b, h], v[b, h], scale, allowed[b])
        rows = allowed[b].any(1)
        np.testing.assert_allclose(o[b, h][rows], ref[rows], rtol=0, atol=1e-14)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_matches_torch_sdpa_library_routine(mask):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    q, k, v, lens = _random_problem(18, B=2, H=3, Tq=11, Tk=13, dk=8, dv=6)
    B, H, Tq, _ = q.shape
    Tk = k.shape[2]
    lens = np.maximum(lens, 1)
    allowed = _allowed(mask, lens, B, Tq, Tk)
    keep = allowed.any(-1)
    o = oracle.sdpa(q, k, v, mask=mask, key_lens=lens)
    am = torch.from_numpy(allowed[:, None])
    ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                         torch.from_numpy(v), attn_mask=am).numpy()
    kk = np.broadcast_to(keep[:, None], o.shape[:3])
    np.testing.assert_allclose(o[kk], ref[kk], rtol=0, atol=1e-13)


def test_mha_with_one_head_and_identity_weights_is_sdpa():
    r = _rng(19)
    B, T, D = 2, 5, 4
    x = r.standard_normal((B, T, D))
    eye = np.eye(D)
    out = oracle.mha(x, x, eye, eye, eye, eye, h=1, scale=0.5)
    ref = oracle.sdpa(x[:, None], x[:, None], x[:, None], scale=0.5)[:, 0]
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-15)


def _torch_mha(x_q, x_kv, w_q, w_k, w_v, w_o, h, mask, lens):
    torch = pytest.importorskip("torch")
    D = x_q.shape[-1]
    m = torch.nn.MultiheadAttention(D, h, bias=False, batch_first=True, dtype=torch.float64)
    with torch.no_grad():
        m.in_proj_weight.copy_(torch.from_numpy(np.concatenate([w_q.T, w_k.T, w_v.T], 0)))
        m.out_proj.weight.copy_(torch.from_numpy(w_o.T))
    B, Tq, _ = x_q.shape
    Tk = x_kv.shape[1]
    kpm = None
    am = None
    if mask & MASK_KEY_PADDING:
        kpm = torch.from_numpy(np.arange(Tk)[None, :] >= lens[:, None])
    if mask & MASK_CAUSAL:
        am = torch.from_numpy(np.arange(Tk)[None, :] > np.arange(Tq)[:, None])
    with torch.no_grad():
        out, _ = m(torch.from_numpy(x_q), torch.from_numpy(x_kv), torch.from_numpy(x_kv),
                   key_padding_mask=kpm, attn_mask=am, need_weights=False)
    return out.numpy()


@pytest.mark.parametrize("mask,cross", [(MASK_NONE, False), (MASK_KEY_PADDING, False),
                                        (MASK_CAUSAL, False), (MASK_CAUSAL_KEY_PADDING, False),
                                        (MASK_KEY_PADDING, True), (MASK_NONE, True)])
def test_mha_matches_torch_multihead_library_routine(mask, cross):
    r = _rng(20)
    B, Tq, D, h = 2, 6, 8, 2
    Tk = 9 if cross else Tq
    x_q = r.standard_normal((B, Tq, D))
    x_kv = r.standard_normal((B, Tk, D)) if cross else x_q
    ws = [r.standard_normal((D, D)) * 0.4 for _ in range(4)]
    lens = np.array([Tk, max(1, Tk - 3)], dtype=np.int32)
    out = oracle.mha(x_q, x_kv, *ws, h=h, mask=mask, key_lens=lens)
    ref = _torch_mha(x_q, x_kv, *ws, h, mask, lens)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_mha_heads_concatenate_in_order():
    # per-head MHA = concat of per-head SDPA on column slices, then W^O
    r = _rng(21)
    B, T, D, h = 1, 4, 6, 3
    d = D // h
    x = r.standard_normal((B, T, D))
    wq, wk, wv = (r.standard_normal((D, D)) for _ in range(3))
    wo = np.eye(D)
    out = oracle.mha(x, x, wq, wk, wv, wo, h=h)
    for i in range(h):
        sl = slice(i * d, (i + 1) * d)
        ref = oracle.sdpa((x @ wq[:, sl])[:, None], (x @ wk[:, sl])[:, None],
                          (x @ wv[:, sl])[:, None])[:, 0]
        np.testing.assert_allclose(out[..., sl], ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_row_subsets_match_full_computation(mask):
    q, k, v, lens = _random_problem(22, B=2, H=2, Tq=10, Tk=12)
    full = oracle.sdpa(q, k, v, mask=mask, key_lens=lens)
    rows = np.array([0, 5, 19, 23, 39])
    sub = oracle.sdpa_rows(q, k, v, rows, mask=mask, key_lens=lens)
    np.testing.assert_array_equal(sub, full.reshape(-1, full.shape[-1])[rows])
    r = _rng(23)
    B, T, D, h = 2, 7, 8, 2
    x = r.standard_normal((B, T, D))
    ws = [r.standard_normal((D, D)) for _ in range(4)]
    full = oracle.mha(x, x, *ws, h=h, mask=mask, key_lens=np.array([7, 4], dtype=np.int32))
    qr = np.array([0, 3, 8, 13])
    sub = oracle.mha(x, x, *ws, h=h, mask=mask, key_lens=np.array([7, 4], dtype=np.int32),
                     query_rows=qr)
    np.testing.assert_allclose(sub, full.reshape(-1, D)[qr], rtol=0, atol=1e-13)


# ----------------------------------------------- residual + layer normalisation
# aiany.app Step 9: LayerNorm(x + Sublayer(x)); notebook chapter "Layer
# Normalization and Residual Connections": (x - mu)/sigma (.) gamma + beta over
# the feature dimension.  Reading: sigma = sqrt(population variance + eps).

def test_add_layernorm_matches_torch_layer_norm():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(61)
    x, s = rng.normal(size=(7, 5, 48)), rng.normal(size=(7, 5, 48)) * 3
    g, b = rng.normal(size=48), rng.normal(size=48)
    for eps in (0.0, 1e-5, 0.3):
        ref = torch.nn.functional.layer_norm(torch.from_numpy(x + s), (48,), torch.from_numpy(g),
                                             torch.from_numpy(b), eps=eps).numpy()
        np.testing.assert_allclose(oracle.add_layernorm(x, s, g, b, eps), ref, rtol=0, atol=1e-12)


def test_add_layernorm_constant_row_gives_shift():
    g, b = np.array([2.0, -1.0, 0.5, 3.0]), np.array([0.25, -4.0, 7.0, 1.0])
    x = np.full((3, 4), 1.75)
    y = oracle.add_layernorm(x, np.full((3, 4), -0.5), g, b, 1e-5)
    np.testing.assert_array_equal(y, np.tile(b, (3, 1)))


def test_add_layernorm_two_features_closed_form():
    # v = (a, c): mean (a+c)/2, population sd |a-c|/2, so v normalises to
    # (-1, +1) when a < c (eps = 0)
    x = np.array([[1.0, 4.0], [10.0, -2.0]])
    s = np.array([[0.5, -0.5], [0.0, 1.0]])  # v = (1.5, 3.5), (10, -1)
    g, b = np.array([3.0, 0.5]), np.array([1.0, -1.0])
    y = oracle.add_layernorm(x, s, g, b, 0.0)
    np.testing.assert_allclose(y, [[-3.0 + 1.0, 0.5 - 1.0], [3.0 + 1.0, -0.5 - 1.0]], atol=1e-15)


def test_add_layernorm_invariant_to_positive_affine_maps():
    rng = np.random.default_rng(62)
    v = rng.normal(size=(4, 32))
    g, b = rng.normal(size=32), rng.normal(size=32)
    zero = np.zeros_like(v)
    ref = oracle.add_layernorm(v, zero, g, b, 0.0)
    np.testing.assert_allclose(oracle.add_layernorm(5.0 * v + 3.0, zero, g, b, 0.0), ref,
                               rtol=0, atol=1e-12)


def test_add_layernorm_adds_the_residual():
    rng = np.random.default_rng(63)
    x, s = rng.normal(size=(3, 16)), rng.normal(size=(3, 16))
    g, b = np.ones(16), np.zeros(16)
    y = oracle.add_layernorm(x, s, g, b, 1e-5)
    np.testing.assert_allclose(y, oracle.add_layernorm(x + s, np.zeros_like(x), g, b, 1e-5),
                               atol=1e-13)
    np.testing.assert_allclose(y, oracle.add_layernorm(s, x, g, b, 1e-5), atol=1e-13)
    assert np.abs(y - oracle.add_layernorm(x, np.zeros_like(x), g, b, 1e-5)).max() > 0.1
    # unit gain, zero shift: every row has mean 0 and variance var/(var+eps)
    v = x + s
    var = v.var(axis=1)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose((y ** 2).mean(axis=1), var / (var + 1e-5), atol=1e-12)


def test_mha_add_layernorm_with_zero_output_projection_normalises_the_input():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(64)
    B, T, D, h = 2, 5, 16, 2
    x = rng.normal(size=(B, T, D))
    w = [rng.normal(size=(D, D)) * 0.3 for _ in range(3)]
    g, b = rng.normal(size=D), rng.normal(size=D)
    y = oracle.mha_add_layernorm(x, x, *w, np.zeros((D, D)), g, b, h=h, eps=1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (D,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)
    # rows selected by index match the full computation
    rows = np.array([0, 3, 7, 9])
    w_o = rng.normal(size=(D, D)) * 0.3
    full = oracle.mha_add_layernorm(x, x, *w, w_o, g, b, h=h, mask=MASK_CAUSAL)
    part = oracle.mha_add_layernorm(x, x, *w, w_o, g, b, h=h, mask=MASK_CAUSAL, query_rows=rows)
    np.testing.assert_allclose(part, full.reshape(-1, D)[rows], rtol=0, atol=1e-13)


# ----------------------------------------------------------- log-sum-exp
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING])
def test_lse_matches_torch_logsumexp(mask):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(81)
    q, k = rng.normal(size=(2, 3, 9, 8)), rng.normal(size=(2, 3, 11, 8))
    lens = np.array([11, 4], dtype=np.int32)
    scale = 0.37
    s = torch.from_numpy(np.einsum("bhqd,bhkd->bhqk", q, k) * scale)
    i = torch.arange(9)[:, None]
    j = torch.arange(11)[None, :]
    vis = torch.ones(2, 1, 9, 11, dtype=torch.bool)
    if mask & MASK_CAUSAL:
        vis = vis & (j <= i)
    if mask & MASK_KEY_PADDING:
        vis = vis & (j[None, None] < torch.from_numpy(lens)[:, None, None, None])
    ref = torch.logsumexp(s.masked_fill(~vis, float("-inf")), dim=-1).numpy()
    got = oracle.sdpa_lse(q, k, scale=scale, mask=mask,
                          key_lens=lens if mask & MASK_KEY_PADDING else None)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_lse_closed_forms_and_consistency_with_weights():
    # equal scores s over n visible keys: lse = s + log n
    q = np.ones((1, 1, 3, 4))
    k = np.full((1, 1, 5, 4), 0.5)  # q.k = 2 for every key
    got = oracle.sdpa_lse(q, k, scale=1.5, mask=MASK_CAUSAL)
    np.testing.assert_allclose(got[0, 0], [3.0 + math.log(1), 3.0 + math.log(2), 3.0 + math.log(3)],
                               atol=1e-14)
    # weights are exp(s - lse)
    rng = np.random.default_rng(82)
    q, k, v = rng.normal(size=(1, 2, 6, 8)), rng.normal(size=(1, 2, 7, 8)), rng.normal(size=(1, 2, 7, 8))
    _, w = oracle.sdpa(q, k, v, scale=0.5, return_weights=True)
    lse = oracle.sdpa_lse(q, k, scale=0.5)
    s = np.einsum("bhqd,bhkd->bhqk", q, k) * 0.5
    np.testing.assert_allclose(w, np.exp(s - lse[..., None]), atol=1e-14)
    # no visible key: -inf
    got = oracle.sdpa_lse(q, k, scale=0.5, mask=MASK_KEY_PADDING, key_lens=np.array([0], np.int32))
    assert np.all(np.isneginf(got))


# ------------------------------------------------------------- backward
def _torch_sdpa_grads(q, k, v, g, scale, mask, lens):
    torch = pytest.importorskip("torch")
    tq, tk, tv = (torch.from_numpy(a).requires_grad_(True) for a in (q, k, v))
    Tq, Tk = q.shape[2], k.shape[2]
    i = torch.arange(Tq)[:, None]
    j = torch.arange(Tk)[None, :]
    vis = torch.ones(q.shape[0], 1, Tq, Tk, dtype=torch.bool)
    if mask & MASK_CAUSAL:
        vis = vis & (j <= i)
    if mask & MASK_KEY_PADDING:
        vis = vis & (j[None, None] < torch.from_numpy(lens)[:, None, None, None])
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=vis, scale=scale)
    o.backward(torch.from_numpy(g))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_CAUSAL_KEY_PADDING])
def test_backward_matches_torch_autograd(mask):
    rng = np.random.default_rng(101)
    B, H, Tq, Tk, d = 2, 2, 7, 9 if not mask & MASK_CAUSAL else 7, 8
    q, g = rng.normal(size=(B, H, Tq, d)), rng.normal(size=(B, H, Tq, d))
    k, v = rng.normal(size=(B, H, Tk, d)), rng.normal(size=(B, H, Tk, d))
    lens = np.array([Tk, 3], dtype=np.int32)
    got = oracle.sdpa_backward(q, k, v, g, scale=0.4, mask=mask,
                               key_lens=lens if mask & MASK_KEY_PADDING else None)
    ref = _torch_sdpa_grads(q, k, v, g, 0.4, mask, lens)
    for a, r in zip(got, ref):
        np.testing.assert_allclose(a, r, rtol=0, atol=1e-12)


def test_backward_matches_finite_differences_of_the_forward():
    rng = np.random.default_rng(102)
    q, g = rng.normal(size=(1, 1, 3, 4)), rng.normal(size=(1, 1, 3, 4))
    k, v = rng.normal(size=(1, 1, 4, 4)), rng.normal(size=(1, 1, 4, 4))
    lens = np.array([3], dtype=np.int32)
    for mask in (MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING):
        kl = lens if mask & MASK_KEY_PADDING else None
        grads = oracle.sdpa_backward(q, k, v, g, scale=0.7, mask=mask, key_lens=kl)
        loss = lambda qq, kk, vv: float(np.sum(g * oracle.sdpa(qq, kk, vv, scale=0.7, mask=mask,
                                                               key_lens=kl)))
        h = 1e-6
        for which, arr in enumerate((q, k, v)):
            num = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                plus, minus = [a.copy() for a in (q, k, v)], [a.copy() for a in (q, k, v)]
                plus[which][idx] += h
                minus[which][idx] -= h
                num[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
            np.testing.assert_allclose(grads[which], num, rtol=0, atol=1e-7)


def test_backward_key_gradients_sum_to_zero_and_masked_keys_get_none():
    # softmax is shift-invariant per row, so sum_j dS_ij = 0 and hence
    # sum_j dK_j = 0 for every (b, h)
    rng = np.random.default_rng(103)
    q, g = rng.normal(size=(2, 2, 6, 8)), rng.normal(size=(2, 2, 6, 8))
    k, v = rng.normal(size=(2, 2, 10, 8)), rng.normal(size=(2, 2, 10, 8))
    lens = np.array([10, 4], dtype=np.int32)
    dq, dk, dv = oracle.sdpa_backward(q, k, v, g, mask=MASK_KEY_PADDING, key_lens=lens)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    assert np.all(dk[1, :, 4:] == 0) and np.all(dv[1, :, 4:] == 0)
    # single visible key: the weight is 1 whatever q and k, so dQ = dK = 0
    # and dV_0 = sum of the output gradients
    dq, dk, dv = oracle.sdpa_backward(q, k, v, g, mask=MASK_KEY_PADDING,
                                      key_lens=np.array([1, 1], dtype=np.int32))
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv[:, :, 0], g.sum(axis=2), atol=1e-13)


@pytest.mark.parametrize("mask", [MASK_CAUSAL, MASK_CAUSAL_KEY_PADDING])
def test_backward_tail_equals_the_full_gradient_where_it_claims_to(mask):
    # Under the causal mask no query row before i0 sees a key at or after i0,
    # so the tail sums give exactly the full dq rows >= i0 and dk, dv rows
    # >= i0 (same terms, same order); the rows it does not claim differ.
    rng = np.random.default_rng(104)
    B, H, T, d = 2, 2, 37, 8
    q, g = rng.normal(size=(B, H, T, d)), rng.normal(size=(B, H, T, d))
    k, v = rng.normal(size=(B, H, T, d)), rng.normal(size=(B, H, T, d))
    lens = np.array([T, 23], dtype=np.int32)
    kl = lens if mask & MASK_KEY_PADDING else None
    full = oracle.sdpa_backward(q, k, v, g, scale=0.3, mask=mask, key_lens=kl)
    for i0 in (0, 1, 17, 36, 37):
        dq, dk, dv = oracle.sdpa_backward_tail(q, k, v, g, i0, scale=0.3, mask=mask, key_lens=kl)
        assert np.array_equal(dq[:, :, i0:], full[0][:, :, i0:])
        assert np.all(dq[:, :, :i0] == 0)
        assert np.array_equal(dk[:, :, i0:], full[1][:, :, i0:])
        assert np.array_equal(dv[:, :, i0:], full[2][:, :, i0:])
    dq, dk, dv = oracle.sdpa_backward_tail(q, k, v, g, 17, scale=0.3, mask=mask, key_lens=kl)
    assert not np.allclose(dv[:, :, :17], full[2][:, :, :17])  # partial there
    with pytest.raises(ValueError):
        oracle.sdpa_backward_tail(q, k, v, g, T + 1, mask=mask, key_lens=kl)


# ------------------------------------------ encoder layer: PE, FFN, composition
def test_positional_encoding_toy_table_from_the_pages():
    g = GOLDEN["positional_encoding_toy"]
    pe = oracle.positional_encoding(len(g["positions"]), g["d_model"])
    np.testing.assert_allclose(pe, g["values"], rtol=0, atol=g["tolerance"])


def test_positional_encoding_offsets_are_rotations():
    # the pages: for a fixed offset k, PE(pos + k) is a linear function of
    # PE(pos) -- per frequency w the pair (sin, cos) turns by the angle k w
    D, k = 16, 5
    pe = oracle.positional_encoding(40, D)
    shifted = oracle.positional_encoding(40, D, pos0=k)
    for i in range(D // 2):
        w = 1.0 / 10000.0 ** (2 * i / D)
        c, s = math.cos(k * w), math.sin(k * w)
        sin_p, cos_p = pe[:, 2 * i], pe[:, 2 * i + 1]
        np.testing.assert_allclose(shifted[:, 2 * i], sin_p * c + cos_p * s, atol=1e-12)
        np.testing.assert_allclose(shifted[:, 2 * i + 1], cos_p * c - sin_p * s, atol=1e-12)
    np.testing.assert_allclose(pe[:, 0::2] ** 2 + pe[:, 1::2] ** 2, 1.0, atol=1e-14)


def test_ffn_matches_torch_linear_relu_linear():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(121)
    x = rng.normal(size=(3, 5, 8))
    w1, b1 = rng.normal(size=(8, 12)), rng.normal(size=12)
    w2, b2 = rng.normal(size=(12, 8)), rng.normal(size=8)
    t = torch.from_numpy
    ref = (torch.relu(t(x) @ t(w1) + t(b1)) @ t(w2) + t(b2)).numpy()
    np.testing.assert_allclose(oracle.ffn(x, w1, b1, w2, b2), ref, rtol=0, atol=1e-12)
    # the ReLU is there: with every pre-activation negative the output is b2
    np.testing.assert_allclose(oracle.ffn(np.abs(x), -np.abs(w1), -np.ones(12), w2, b2),
                               np.broadcast_to(b2, x.shape), atol=1e-15)


def encoder_params(rng, D, F):
    return {"w_q": rng.normal(size=(D, D)) * 0.2, "w_k": rng.normal(size=(D, D)) * 0.2,
            "w_v": rng.normal(size=(D, D)) * 0.2, "w_o": rng.normal(size=(D, D)) * 0.2,
            "gamma1": 1 + rng.normal(size=D) * 0.1, "beta1": rng.normal(size=D) * 0.1,
            "w1": rng.normal(size=(D, F)) * 0.2, "b1": rng.normal(size=F) * 0.1,
            "w2": rng.normal(size=(F, D)) * 0.2, "b2": rng.normal(size=D) * 0.1,
            "gamma2": 1 + rng.normal(size=D) * 0.1, "beta2": rng.normal(size=D) * 0.1}


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_KEY_PADDING])
def test_encoder_layer_matches_torch_transformer_encoder_layer(mask):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(122)
    B, T, D, h, F = 2, 6, 16, 2, 24
    x = rng.normal(size=(B, T, D))
    p = encoder_params(rng, D, F)
    lens = np.array([6, 3], dtype=np.int32)
    layer = torch.nn.TransformerEncoderLayer(D, h, dim_feedforward=F, dropout=0.0,
                                             activation="relu", batch_first=True,
                                             norm_first=False, dtype=torch.float64)
    t = torch.from_numpy
    with torch.no_grad():
        # row-vector weights (y = x W) map to torch's (out, in) matrices
        layer.self_attn.in_proj_weight.copy_(t(np.concatenate([p["w_q"], p["w_k"], p["w_v"]], 1).T))
        layer.self_attn.in_proj_bias.zero_()
        layer.self_attn.out_proj.weight.copy_(t(p["w_o"].T))
        layer.self_attn.out_proj.bias.zero_()
        layer.linear1.weight.copy_(t(p["w1"].T))
        layer.linear1.bias.copy_(t(p["b1"]))
        layer.linear2.weight.copy_(t(p["w2"].T))
        layer.linear2.bias.copy_(t(p["b2"]))
        layer.norm1.weight.copy_(t(p["gamma1"]))
        layer.norm1.bias.copy_(t(p["beta1"]))
        layer.norm2.weight.copy_(t(p["gamma2"]))
        layer.norm2.bias.copy_(t(p["beta2"]))
    layer.norm1.eps = layer.norm2.eps = 1e-5
    layer.eval()
    pad = None
    if mask == MASK_KEY_PADDING:
        pad = torch.arange(T)[None, :] >= t(lens)[:, None]
    with torch.no_grad():
        ref = layer(t(x), src_key_padding_mask=pad).numpy()
    got = oracle.encoder_layer(x, p, h=h, eps=1e-5, mask=mask,
                               key_lens=lens if mask == MASK_KEY_PADDING else None)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)
