"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances: fp32 path max-abs <= 1e-5; bf16 path max-abs <= 2e-2 and
mean-abs <= 2e-3, over every compared output element.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

F32_MAX = 1e-5
BF16_MAX, BF16_MEAN = 2e-2, 2e-3
MASK_NAMES = {si.MASK_NONE: "none", si.MASK_CAUSAL: "causal",
              si.MASK_KEY_PADDING: "key_padding", si.MASK_CAUSAL_KEY_PADDING: "causal_key_padding"}


@pytest.fixture(scope="module")
def lib():
    import transformer_scaled_dot_softmax_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def dev():
    return torch.device("cuda:0")


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(torch.bfloat16)


def f32_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev())


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_bf16(got, ref, what=""):
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (
        "%s: max %.4g mean %.4g" % (what, err.max(), err.mean()))


def lens_dev(x):
    return None if x["key_lens"] is None else torch.from_numpy(x["key_lens"]).to(dev())


# Guard bands: every output buffer below sits between two bands of a canary
# bit pattern (a bf16 NaN payload no kernel produces); a write outside the
# output changes a band and fails the check after the call.
GUARD = 4096          # elements per band (8 KiB: keeps the output 16-byte aligned)
CANARY = 0x7FA5


def guarded_bf16(shape, fill=float("nan")):
    n = int(np.prod(shape))
    buf = torch.full((2 * GUARD + n,), CANARY, dtype=torch.int16, device=dev())
    out = buf[GUARD:GUARD + n].view(torch.bfloat16).view(shape)
    out.fill_(fill)
    return buf, out


def check_guards(buf, what=""):
    assert bool(torch.all(buf[:GUARD] == CANARY)), what + ": write before the output"
    assert bool(torch.all(buf[-GUARD:] == CANARY)), what + ": write past the output"


def run_sdpa_bf16(lib, w, x, q=None, k=None, v=None, poison=True):
    q = bf16_dev(x["q_bits"]) if q is None else q
    k = bf16_dev(x["k_bits"]) if k is None else k
    v = bf16_dev(x["v_bits"]) if v is None else v
    buf, out = guarded_bf16((w.B, w.h, w.T_q, w.d_v), float("nan") if poison else 0.0)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    lib.sdpa_forward(q, k, v, out, scale=w.scale, mask=w.mask, key_lens=lens_dev(x),
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_guards(buf, "sdpa B%d h%d Tq%d Tk%d" % (w.B, w.h, w.T_q, w.T_k))
    return out


# ----------------------------------------------------------------- fp32 path
def test_config1_fp32_full(lib):
    w = si.WORKLOADS[0]
    x = si.make_inputs(w)
    out = lib.sdpa_forward(f32_dev(x["q"]), f32_dev(x["k"]), f32_dev(x["v"]), scale=w.scale)
    torch.cuda.synchronize()
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale)
    assert np.abs(host(out) - ref).max() <= F32_MAX


@pytest.mark.parametrize("mask", list(MASK_NAMES))
# T_k <= 32 with d = 64 runs the short-key (register) kernel, the rest the
# chunked one: (33, 32) and (9, 1) sit at its limits, (40, 33) just past.
@pytest.mark.parametrize("T_q,T_k,d", [(37, 53, 64), (16, 16, 32), (5, 200, 128), (130, 7, 64),
                                       (33, 32, 64), (9, 1, 64), (40, 33, 64)])
def test_fp32_masks_and_ragged(lib, mask, T_q, T_k, d):
    w = si.WORKLOADS[0].replace(B=2, h=3, T_q=T_q, T_k=T_k, d_k=d, d_v=d, mask=mask, len_lo=1,
                                len_hi=T_k, seed=11)
    x = si.make_inputs(w)
    out = lib.sdpa_forward(f32_dev(x["q"]), f32_dev(x["k"]), f32_dev(x["v"]), scale=w.scale,
                           mask=mask, key_lens=lens_dev(x))
    torch.cuda.synchronize()
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=mask, key_lens=x["key_lens"])
    assert np.abs(host(out) - ref).max() <= F32_MAX


@pytest.mark.parametrize("T_k", [20, 50])
def test_fp32_rows_without_visible_keys(lib, T_k):
    """Key lengths of 0 leave whole sequences without a visible key: their
    rows are zeros in both fp32 kernels (short-key and chunked); the other
    sequences match the oracle."""
    w = si.WORKLOADS[0].replace(B=4, h=2, T_q=13, T_k=T_k, mask=si.MASK_CAUSAL_KEY_PADDING,
                                len_lo=1, len_hi=T_k, seed=17)
    x = si.make_inputs(w)
    lens = np.array([0, T_k, 0, 3], dtype=np.int32)
    out = lib.sdpa_forward(f32_dev(x["q"]), f32_dev(x["k"]), f32_dev(x["v"]), scale=w.scale,
                           mask="causal_key_padding", key_lens=torch.from_numpy(lens).to(dev()))
    torch.cuda.synchronize()
    got = host(out)
    assert np.all(got[lens == 0] == 0.0)
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=si.MASK_CAUSAL_KEY_PADDING,
                      key_lens=lens)
    assert np.abs(got[lens > 0] - ref[lens > 0]).max() <= F32_MAX


def test_fp32_unaligned_rows_take_the_chunked_kernel(lib):
    """q and k starting 4 bytes past a 16-byte boundary cannot be read as
    float4: the short-key case then runs the chunked kernel, with the same
    result bit for bit."""
    w = si.WORKLOADS[0].replace(B=1, h=3, T_q=21, T_k=24, mask=si.MASK_CAUSAL, seed=19)
    x = si.make_inputs(w)
    q, k, v = (f32_dev(x[n]) for n in ("q", "k", "v"))
    aligned = lib.sdpa_forward(q, k, v, scale=w.scale, mask="causal")

    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=torch.float32, device=dev())
        view = buf[1:].view(t.shape)
        view.copy_(t)
        return view

    qs, ks = shifted(q), shifted(k)
    assert qs.data_ptr() % 16 != 0 and ks.data_ptr() % 16 != 0
    unaligned = lib.sdpa_forward(qs, ks, v, scale=w.scale, mask="causal")
    torch.cuda.synchronize()
    assert torch.equal(aligned, unaligned)
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=si.MASK_CAUSAL)
    assert np.abs(host(unaligned) - ref).max() <= F32_MAX


# ----------------------------------------------------------------- bf16 SDPA
BF16_SHAPES = [
    (1, 1, 128, 128, si.MASK_NONE),
    (1, 2, 1, 1, si.MASK_NONE),
    (2, 2, 255, 257, si.MASK_NONE),
    (1, 2, 256, 256, si.MASK_CAUSAL),
    (1, 2, 300, 300, si.MASK_CAUSAL),
    (2, 1, 513, 700, si.MASK_KEY_PADDING),
    (2, 2, 384, 384, si.MASK_CAUSAL_KEY_PADDING),
    (1, 1, 64, 1000, si.MASK_NONE),
    (1, 1, 1000, 64, si.MASK_CAUSAL),
    (3, 1, 129, 1025, si.MASK_KEY_PADDING),
    (1, 3, 777, 777, si.MASK_CAUSAL),
]


@pytest.mark.parametrize("B,h,T_q,T_k,mask", BF16_SHAPES)
def test_bf16_sdpa_vs_oracle(lib, B, h, T_q, T_k, mask):
    w = si.WORKLOADS[4].replace(B=B, h=h, T_q=T_q, T_k=T_k, mask=mask, len_lo=1, len_hi=T_k,
                                seed=21)
    x = si.make_inputs(w)
    out = run_sdpa_bf16(lib, w, x)
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=mask, key_lens=x["key_lens"])
    check_bf16(host(out), ref, "B%d h%d Tq%d Tk%d mask%d" % (B, h, T_q, T_k, mask))


def splits_by_tiles(T_q, T_k, causal):
    """The launcher's choice of split between the attention kernel's two
    softmax groups: alternate key tiles when a 128-row query tile has on
    average 8 key tiles or more (key padding ignored), key halves of every
    tile otherwise."""
    nqb = -(-T_q // 128)
    tiles = sum(-(-(min(T_k, (qb + 1) * 128, T_q) if causal else T_k) // 128) for qb in range(nqb))
    return tiles >= 8 * nqb


# Every mask under both splits, with ragged query and key tails.
SPLIT_SHAPES = [
    (1, 2, 2048, 2048, si.MASK_CAUSAL, True),
    (2, 2, 640, 640, si.MASK_CAUSAL, False),
    (1, 2, 1000, 900, si.MASK_NONE, True),
    (2, 1, 300, 896, si.MASK_NONE, False),
    (2, 2, 700, 1100, si.MASK_KEY_PADDING, True),
    (2, 2, 513, 700, si.MASK_KEY_PADDING, False),
    (2, 1, 2100, 2100, si.MASK_CAUSAL_KEY_PADDING, True),
    (2, 2, 384, 384, si.MASK_CAUSAL_KEY_PADDING, False),
    # one partial query tile against long key sequences
    (1, 2, 1, 4096, si.MASK_NONE, True),
    (2, 1, 5, 3000, si.MASK_KEY_PADDING, True),
    (1, 1, 77, 895, si.MASK_NONE, False),
]


@pytest.mark.parametrize("B,h,T_q,T_k,mask,tiles", SPLIT_SHAPES)
def test_bf16_both_key_splits(lib, B, h, T_q, T_k, mask, tiles):
    assert splits_by_tiles(T_q, T_k, bool(mask & si.MASK_CAUSAL)) == tiles
    assert lib.sdpa_bf16_key_split(T_q, T_k, MASK_NAMES[mask]) == int(tiles)
    w = si.WORKLOADS[4].replace(B=B, h=h, T_q=T_q, T_k=T_k, mask=mask, len_lo=1, len_hi=T_k,
                                seed=23)
    x = si.make_inputs(w)
    out = run_sdpa_bf16(lib, w, x)
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=mask, key_lens=x["key_lens"])
    check_bf16(host(out), ref, "B%d h%d Tq%d Tk%d mask%d tiles%d" % (B, h, T_q, T_k, mask, tiles))


def test_config5_every_element(lib):
    """The long-sequence causal workload (B=2, h=16, T=8192, d=64) at full
    size, in the launch the benchmark times, compared with the oracle over
    every output element (aiany.app Step 6: Z = AV for every row)."""
    w = si.WORKLOADS[4]
    x = si.make_inputs(w)
    out = run_sdpa_bf16(lib, w, x)
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=w.mask)
    got = host(out)
    assert got.shape == ref.shape == (2, 16, 8192, 64)
    check_bf16(got, ref, "config 5, every element")


LONG_SHAPES = [
    # one head, a causal sequence 8x longer than the largest workload (131,328 score tiles)
    (1, 1, 65536, 65536, si.MASK_CAUSAL),
    # a short query block against a very long, padded key sequence (1,024 key tiles per item)
    (2, 1, 200, 131072, si.MASK_KEY_PADDING),
]


@pytest.mark.parametrize("B,h,T_q,T_k,mask", LONG_SHAPES)
def test_bf16_long_sequences_sampled_rows(lib, B, h, T_q, T_k, mask):
    """Sequence lengths far past the workloads (the kernel has no length
    limit below 2^31 / 128 query tiles): the rows the oracle can afford --
    the first and last rows, every query-tile boundary region and a seeded
    sample -- are compared element by element."""
    w = si.WORKLOADS[4].replace(B=B, h=h, T_q=T_q, T_k=T_k, mask=mask, len_lo=T_k // 2,
                                len_hi=T_k, seed=37)
    x = si.make_inputs(w)
    got = host(run_sdpa_bf16(lib, w, x))
    rng = np.random.default_rng(37)
    t = np.unique(np.concatenate([[0, 1, 127, 128, 129, T_q // 2, T_q - 2, T_q - 1],
                                  rng.integers(0, T_q, 120)]))
    t = t[t < T_q]
    flat = (np.arange(B * h)[:, None] * T_q + t[None, :]).reshape(-1)
    ref = oracle.sdpa_rows(x["q"], x["k"], x["v"], flat, scale=w.scale, mask=mask,
                           key_lens=x["key_lens"])
    check_bf16(got.reshape(-1, w.d_v)[flat], ref, "long B%d Tq%d Tk%d" % (B, T_q, T_k))


def test_bf16_padding_rows_bitwise_independent_of_masked_keys(lib):
    w = si.WORKLOADS[4].replace(B=3, h=2, T_q=200, T_k=600, mask=si.MASK_KEY_PADDING,
                                len_lo=100, len_hi=500, seed=31)
    x = si.make_inputs(w)
    a = run_sdpa_bf16(lib, w, x)
    k = bf16_dev(x["k_bits"]).clone()
    v = bf16_dev(x["v_bits"]).clone()
    for b, L in enumerate(x["key_lens"]):
        k[b, :, L:] = torch.randn_like(k[b, :, L:].float()).mul(30).bfloat16()
        v[b, :, L:] = torch.randn_like(v[b, :, L:].float()).mul(30).bfloat16()
    b2 = run_sdpa_bf16(lib, w, x, k=k, v=v)
    assert torch.equal(a.view(torch.int16), b2.view(torch.int16))


def test_bf16_causal_rows_bitwise_independent_of_future_keys(lib):
    w = si.WORKLOADS[4].replace(B=1, h=2, T_q=400, T_k=400, mask=si.MASK_CAUSAL, seed=32)
    x = si.make_inputs(w)
    a = run_sdpa_bf16(lib, w, x)
    k = bf16_dev(x["k_bits"]).clone()
    v = bf16_dev(x["v_bits"]).clone()
    cut = 250
    k[:, :, cut:] = 7.0
    v[:, :, cut:] = -9.0
    b2 = run_sdpa_bf16(lib, w, x, k=k, v=v)
    assert torch.equal(a[:, :, :cut].view(torch.int16), b2[:, :, :cut].view(torch.int16))
    # causal row 0 sees key 0 only: output = V_0 (exactly representable)
    assert torch.equal(a[:, :, 0], bf16_dev(x["v_bits"])[:, :, 0])


def test_bf16_constant_values(lib):
    w = si.WORKLOADS[4].replace(B=1, h=2, T_q=300, T_k=900, mask=si.MASK_NONE, seed=33)
    x = si.make_inputs(w)
    v = torch.full((w.B, w.h, w.T_k, w.d_v), 1.5, dtype=torch.bfloat16, device=dev())
    out = run_sdpa_bf16(lib, w, x, v=v)
    # The row sum adds the same bf16-rounded weights the P.V product
    # multiplies, so the normalised weights sum to 1 up to fp32 rounding
    # (~1e-6), far inside half a bf16 ulp of 1.5: the output is 1.5 exactly.
    assert torch.all(out == 1.5)


REF_MAX_PROFILES = ("growing", "jump", "shrinking")


def scaled_keys(x, profile, nt):
    """Key tiles (128 keys) scaled so that a row's maximum score keeps growing
    (every tile by ~20 log2 units: the exact step runs tile after tile),
    jumps far enough that exponentials against the old maximum overflow
    fp32, or only shrinks (the first maximum stays the reference)."""
    f = {"growing": [6 * j + 1 for j in range(nt)],
         "jump": [80 if j in (2, 5) else 1 for j in range(nt)],
         "shrinking": [6 * (nt - j) + 1 for j in range(nt)]}[profile]
    return si.round_bf16(x["k"] * np.repeat(np.array(f, dtype=np.float64), 128)[None, None, :, None])


@pytest.mark.parametrize("T", [1024, 2048])
@pytest.mark.parametrize("mask", [si.MASK_NONE, si.MASK_CAUSAL])
@pytest.mark.parametrize("profile", REF_MAX_PROFILES)
def test_bf16_reference_maximum_updates(lib, profile, mask, T):
    """Scores that move the reference maximum (scaled_keys).  Such scores
    make almost every row select one value row, so the output is that row of
    V, at full range (|v| up to ~4.5 for these N(0,1) values).  Causal
    T = 1024 runs the kernel's key-halves split, the other three its
    alternate-tiles split (see splits_by_tiles)."""
    w = si.WORKLOADS[4].replace(B=1, h=2, T_q=T, T_k=T, mask=mask, seed=36)
    x = si.make_inputs(w)
    k = scaled_keys(x, profile, w.T_k // 128)
    out = run_sdpa_bf16(lib, w, x, k=bf16_dev(si.f64_to_bf16_bits(k)))
    ref = oracle.sdpa(x["q"], k, x["v"], scale=w.scale, mask=mask)
    check_bf16(host(out), ref, "%s mask%d" % (profile, mask))


def dominant_key_inputs(x, profile, seed):
    """One hand-set dominant key per 128-key tile (key 128t + 37): every
    query has feature 0 equal to 1 and the dominant key is g_t e_0, so its
    score g_t/8 beats every other score (~N(0, 1)) by 20 or more; its value
    row is +-[4, 4.5].  "lazy": g_t grows by 80 a tile (scores up by 10, i.e.
    14.4 log2 units: under the kernel's 16-unit trigger, so the new winner's
    weight is taken against the old reference maximum, as 2^14.4, whose
    rounding to bf16 is inexact); "jump": the same, plus a step of 400 at
    tile 3 (50 more, 72 log2 units: the exact step resets the reference)."""
    q, k, v = x["q"].copy(), x["k"].copy(), x["v"].copy()
    q[..., 0] = 1.0
    nt = k.shape[2] // 128
    rng = np.random.default_rng(2000 + seed)
    for t in range(nt):
        j = 128 * t + 37
        g = 200.0 + 80.0 * t + (400.0 if profile == "jump" and t >= 3 else 0.0)
        k[..., j, :] = 0.0
        k[..., j, 0] = g
        mag = 4.0 + 0.5 * rng.random(v[..., j, :].shape)
        v[..., j, :] = np.where(rng.random(mag.shape) < 0.5, -mag, mag)
    return si.round_bf16(q), si.round_bf16(k), si.round_bf16(v)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("T,mask", [(1024, si.MASK_CAUSAL), (1024, si.MASK_NONE)])
@pytest.mark.parametrize("profile", ["lazy", "jump"])
def test_bf16_dominant_key_selects_large_value(lib, profile, T, mask, seed):
    """A dominant score selects its value (aiany.app Step 5: a gap of 4 or
    more and the winner takes nearly all the weight), with the winner's value
    row at +-[4, 4.5], where the bf16 output's half-ulp is already 2^-6.  The
    kernel sums a row's weights after rounding them to bf16 -- the values the
    P.V product multiplies -- so its normalised weights sum to 1 and the
    winner's row comes back up to the output rounding, under the stated
    2e-2 / 2e-3 bounds, however far the winner's score sits above the
    reference maximum.  Causal T = 1024 runs the key-halves split,
    non-causal T = 1024 the alternate-tiles split."""
    assert splits_by_tiles(T, T, mask == si.MASK_CAUSAL) == (mask == si.MASK_NONE)
    w = si.WORKLOADS[4].replace(B=1, h=2, T_q=T, T_k=T, mask=mask, seed=40 + seed)
    q, k, v = dominant_key_inputs(si.make_inputs(w), profile, seed)
    out = run_sdpa_bf16(lib, w, {"key_lens": None}, q=bf16_dev(si.f64_to_bf16_bits(q)),
                        k=bf16_dev(si.f64_to_bf16_bits(k)), v=bf16_dev(si.f64_to_bf16_bits(v)))
    ref = oracle.sdpa(q, k, v, scale=w.scale, mask=mask)
    assert np.mean(np.abs(ref) >= 3.9) > 0.9  # nearly every row selects a +-[4, 4.5] row
    check_bf16(host(out), ref, "%s mask%d seed%d" % (profile, mask, seed))


def test_bf16_zero_length_rows_are_zero(lib):
    w = si.WORKLOADS[4].replace(B=2, h=1, T_q=130, T_k=300, mask=si.MASK_KEY_PADDING, seed=34)
    x = si.make_inputs(w)
    x["key_lens"] = np.array([0, 123], dtype=np.int32)
    out = run_sdpa_bf16(lib, w, x)
    assert torch.all(out[0] == 0)
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=w.mask, key_lens=x["key_lens"])
    check_bf16(host(out), ref, "zero-length rows")


def test_bf16_on_side_stream(lib):
    w = si.WORKLOADS[4].replace(B=1, h=2, T_q=256, T_k=256, mask=si.MASK_CAUSAL, seed=35)
    x = si.make_inputs(w)
    s = torch.cuda.Stream()
    q, k, v = bf16_dev(x["q_bits"]), bf16_dev(x["k_bits"]), bf16_dev(x["v_bits"])
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = lib.sdpa_forward(q, k, v, scale=w.scale, mask="causal")
    s.synchronize()
    ref = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=w.mask)
    check_bf16(host(out), ref, "side stream")


# ------------------------------------------------------------------ bf16 MHA
def run_mha(lib, w, x):
    xq = bf16_dev(x["x_q_bits"])
    xkv = bf16_dev(x["x_kv_bits"]) if w.cross else xq
    buf, out = guarded_bf16((w.B, w.T_q, w.d_model))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    lib.mha_forward(xq, xkv, bf16_dev(x["w_q_bits"]), bf16_dev(x["w_k_bits"]),
                    bf16_dev(x["w_v_bits"]), bf16_dev(x["w_o_bits"]), h=w.h, out=out,
                    scale=w.scale, mask=w.mask, key_lens=lens_dev(x), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_guards(buf, "mha B%d Tq%d Tk%d D%d" % (w.B, w.T_q, w.T_k, w.d_model))
    return host(out)


def oracle_mha(w, x, query_rows=None):
    x_kv = x["x_kv"] if w.cross else x["x_q"]
    return oracle.mha(x["x_q"], x_kv, x["w_q"], x["w_k"], x["w_v"], x["w_o"], h=w.h,
                      scale=w.scale, mask=w.mask, key_lens=x["key_lens"], query_rows=query_rows)


MHA_SMALL = [
    # B, T_q, T_k, D, h, mask, cross
    (2, 130, 130, 128, 2, si.MASK_KEY_PADDING, False),
    (1, 300, 300, 192, 3, si.MASK_CAUSAL, False),
    (2, 70, 333, 128, 2, si.MASK_KEY_PADDING, True),
    (1, 257, 129, 256, 4, si.MASK_NONE, True),
    (2, 64, 64, 64, 1, si.MASK_CAUSAL_KEY_PADDING, False),
    # enough tiles for 128 x 256 projection tiles, with a ragged last row tile
    (3, 1000, 1000, 512, 8, si.MASK_CAUSAL, False),
    # one projection launch whose Q output (T_q a multiple of 128) leaves by
    # TMA tensor stores and whose K, V outputs (T_k not) by row stores; and
    # both by tensor stores
    (2, 128, 300, 256, 4, si.MASK_KEY_PADDING, True),
    (1, 256, 128, 128, 2, si.MASK_NONE, True),
    # 8 key tiles per query tile: the attention takes alternate key tiles
    (2, 700, 900, 512, 8, si.MASK_KEY_PADDING, True),
]


@pytest.mark.parametrize("B,T_q,T_k,D,h,mask,cross", MHA_SMALL)
def test_mha_small_vs_oracle(lib, B, T_q, T_k, D, h, mask, cross):
    w = si.WORKLOADS[3].replace(B=B, T_q=T_q, T_k=T_k, d_model=D, h=h, mask=mask, cross=cross,
                                len_lo=1, len_hi=T_k, seed=41)
    x = si.make_inputs(w)
    check_bf16(run_mha(lib, w, x), oracle_mha(w, x), "mha small")


@pytest.mark.parametrize("idx", [1, 2])
def test_mha_configs_full(lib, idx):
    w = si.WORKLOADS[idx]
    x = si.make_inputs(w)
    check_bf16(run_mha(lib, w, x), oracle_mha(w, x), w.name)


def test_mha_config4_full(lib):
    w = si.WORKLOADS[3]
    x = si.make_inputs(w)
    check_bf16(run_mha(lib, w, x), oracle_mha(w, x), w.name)


# ------------------------------------- attention sublayer: residual + LayerNorm
def run_mha_ln(lib, w, x, ln, eps=1e-5):
    xq = bf16_dev(x["x_q_bits"])
    xkv = bf16_dev(x["x_kv_bits"]) if w.cross else xq
    buf, out = guarded_bf16((w.B, w.T_q, w.d_model))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    lib.mha_forward_add_layernorm(xq, xkv, bf16_dev(x["w_q_bits"]), bf16_dev(x["w_k_bits"]),
                                  bf16_dev(x["w_v_bits"]), bf16_dev(x["w_o_bits"]),
                                  bf16_dev(ln["gamma_bits"]), bf16_dev(ln["beta_bits"]), h=w.h,
                                  eps=eps, out=out, scale=w.scale, mask=w.mask,
                                  key_lens=lens_dev(x), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_guards(buf, "mha+ln B%d Tq%d Tk%d D%d" % (w.B, w.T_q, w.T_k, w.d_model))
    return host(out)


def oracle_mha_ln(w, x, ln, eps=1e-5, query_rows=None):
    x_kv = x["x_kv"] if w.cross else x["x_q"]
    return oracle.mha_add_layernorm(x["x_q"], x_kv, x["w_q"], x["w_k"], x["w_v"], x["w_o"],
                                    ln["gamma"], ln["beta"], h=w.h, eps=eps, scale=w.scale,
                                    mask=w.mask, key_lens=x["key_lens"], query_rows=query_rows)


MHA_LN_SHAPES = [
    # B, T_q, T_k, D, h, mask, cross: D/256 or D/128 CTAs per 128-row block
    (2, 130, 130, 128, 2, si.MASK_KEY_PADDING, False),   # 1 CTA of 128 columns
    (1, 300, 300, 256, 4, si.MASK_CAUSAL, False),        # 2 CTAs of 128
    (2, 70, 333, 384, 6, si.MASK_KEY_PADDING, True),     # 3 CTAs of 128
    (3, 200, 200, 512, 8, si.MASK_CAUSAL, False),        # 4 CTAs of 128
    (1, 257, 129, 1024, 16, si.MASK_NONE, True),         # 4 CTAs of 256
    (1, 130, 130, 2048, 32, si.MASK_CAUSAL, False),      # 8 CTAs of 256
]


@pytest.mark.parametrize("B,T_q,T_k,D,h,mask,cross", MHA_LN_SHAPES)
def test_mha_add_layernorm_vs_oracle(lib, B, T_q, T_k, D, h, mask, cross):
    w = si.WORKLOADS[3].replace(B=B, T_q=T_q, T_k=T_k, d_model=D, h=h, mask=mask, cross=cross,
                                len_lo=1, len_hi=T_k, seed=71)
    x = si.make_inputs(w)
    ln = si.layernorm_params(71, D)
    check_bf16(run_mha_ln(lib, w, x, ln), oracle_mha_ln(w, x, ln), "mha+ln D%d" % D)


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_mha_add_layernorm_configs_full(lib, idx):
    w = si.WORKLOADS[idx]
    x = si.make_inputs(w)
    ln = si.layernorm_params(w.seed, w.d_model)
    check_bf16(run_mha_ln(lib, w, x, ln), oracle_mha_ln(w, x, ln), w.name + " + layer norm")


def test_mha_add_layernorm_rows_are_normalised(lib):
    # unit gain, zero shift: every output row has mean 0 and variance
    # var/(var+eps) (up to bf16 rounding of the stored values)
    w = si.WORKLOADS[2].replace(B=2, T_q=300, T_k=300, seed=72)
    x = si.make_inputs(w)
    D = w.d_model
    ln = {"gamma": np.ones(D), "beta": np.zeros(D),
          "gamma_bits": si.f64_to_bf16_bits(np.ones(D)), "beta_bits": si.f64_to_bf16_bits(np.zeros(D))}
    y = run_mha_ln(lib, w, x, ln, eps=0.0)
    assert np.abs(y.mean(axis=-1)).max() < 5e-3
    assert np.abs((y ** 2).mean(axis=-1) - 1.0).max() < 1e-2


# ------------------------------------------------------- log-sum-exp export
# lse comes from fp32 sums of ex2.approx terms (relative error ~2^-22 each,
# fp32 accumulation over up to 8192 keys): 1e-3 absolute covers it.
# The exported lse is the log of the normaliser the output was divided by,
# the sum of the bf16-rounded weights: each weight's relative rounding is at
# most 2^-8, so the sum, and exp(lse), lie within a factor 1 +- 2^-8 of the
# exact ones, |lse - exact| <= 2^-8; fp32 arithmetic (the scaled maximum, ln,
# ex2.approx) adds ~1e-6 |lse|, well inside the 1e-4 allowed for it.
LSE_TOL = 2.0 ** -8 + 1e-4


def run_sdpa_lse(lib, w, x, k=None):
    q = bf16_dev(x["q_bits"])
    k = bf16_dev(x["k_bits"]) if k is None else k
    v = bf16_dev(x["v_bits"])
    out, lse = lib.sdpa_forward_lse(q, k, v, scale=w.scale, mask=w.mask, key_lens=lens_dev(x))
    torch.cuda.synchronize()
    return out, lse.double().cpu().numpy()


def check_lse(got, ref, what):
    inf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf), what + ": -inf rows differ"
    err = np.abs(got[~inf] - ref[~inf])
    assert err.size == 0 or err.max() <= LSE_TOL, "%s: lse max err %.3g" % (what, err.max())


@pytest.mark.parametrize("B,h,T_q,T_k,mask", BF16_SHAPES + [(1, 2, 2048, 2048, si.MASK_CAUSAL)])
def test_bf16_lse_vs_oracle(lib, B, h, T_q, T_k, mask):
    w = si.WORKLOADS[4].replace(B=B, h=h, T_q=T_q, T_k=T_k, mask=mask, len_lo=0, len_hi=T_k,
                                seed=91)
    x = si.make_inputs(w)
    out, lse = run_sdpa_lse(lib, w, x)
    ref_o = oracle.sdpa(x["q"], x["k"], x["v"], scale=w.scale, mask=mask, key_lens=x["key_lens"])
    check_bf16(host(out), ref_o, "lse call output")
    ref = oracle.sdpa_lse(x["q"], x["k"], scale=w.scale, mask=mask, key_lens=x["key_lens"])
    check_lse(lse, ref, "B%d h%d Tq%d Tk%d mask%d" % (B, h, T_q, T_k, mask))


@pytest.mark.parametrize("profile", ["growing", "jump"])
def test_bf16_lse_across_reference_updates(lib, profile):
    w = si.WORKLOADS[4].replace(B=1, h=2, T_q=1024, T_k=1024, mask=si.MASK_CAUSAL, seed=92)
    x = si.make_inputs(w)
    f = {"growing": [6 * j + 1 for j in range(8)], "jump": [80 if j in (2, 5) else 1 for j in range(8)]}[profile]
    k = si.round_bf16(x["k"] * np.repeat(np.array(f, dtype=np.float64), 128)[None, None, :, None])
    out, lse = run_sdpa_lse(lib, w, x, k=bf16_dev(si.f64_to_bf16_bits(k)))
    ref = oracle.sdpa_lse(x["q"], k, scale=w.scale, mask=w.mask)
    # large scores: compare relative to the row's magnitude
    assert np.all(np.abs(lse - ref) <= LSE_TOL * np.maximum(1.0, np.abs(ref)))
