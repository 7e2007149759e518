"""The C-ABI library loads without a GPU, exports every symbol include/mha.h
declares, and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from transformer_scaled_dot_softmax_gb300 import _native
    return _native


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                                text, flags=re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"sdpa_forward", "mha_forward", "mha_workspace_bytes", "mha_status_string"} <= set(names)
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
        assert n in lib.SIGNATURES, n


def test_status_strings(lib):
    for code in range(8):
        s = lib.lib.mha_status_string(code)
        assert s and s != b"unknown status"
    assert lib.lib.mha_status_string(99) == b"unknown status"


def test_workspace_bytes(lib):
    ws = lib.lib.mha_workspace_bytes
    assert ws(2, 16, 8192, 8192, 64, 64) == 4 * 2 * 16 * 8192 * 64 * 2
    assert ws(1, 1, 3, 5, 64, 64) == 512 + 768 + 768 + 512  # regions rounded to 256 bytes
    assert ws(-1, 1, 1, 1, 64, 64) == 0


FAKE = 1 << 20  # never dereferenced: every case below fails validation first


def sdpa(lib, dt=1, q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, h=1, Tq=8, Tk=8, dk=64, dv=64,
         scale=0.125, mask=0, lens=None):
    return lib.lib.sdpa_forward(dt, q, k, v, o, B, h, Tq, Tk, dk, dv, scale, mask, lens, None, None)


def test_sdpa_rejects_bad_arguments(lib):
    assert sdpa(lib, q=None) == lib.MHA_ERR_INVALID_ARG
    assert sdpa(lib, o=None) == lib.MHA_ERR_INVALID_ARG
    assert sdpa(lib, B=-1) == lib.MHA_ERR_INVALID_ARG
    assert sdpa(lib, dk=0) == lib.MHA_ERR_INVALID_ARG
    assert sdpa(lib, mask=7) == lib.MHA_ERR_INVALID_ARG
    assert sdpa(lib, mask=2, lens=None) == lib.MHA_ERR_INVALID_ARG
    assert sdpa(lib, scale=float("nan")) == lib.MHA_ERR_INVALID_ARG
    assert sdpa(lib, dt=5) == lib.MHA_ERR_INVALID_ARG
    assert sdpa(lib, dk=32, dv=32) == lib.MHA_ERR_UNSUPPORTED
    assert sdpa(lib, dt=0, dk=256) == lib.MHA_ERR_UNSUPPORTED
    assert sdpa(lib, q=FAKE + 8) == lib.MHA_ERR_MISALIGNED
    assert sdpa(lib, o=FAKE + 2) == lib.MHA_ERR_MISALIGNED


def test_empty_problems_are_no_ops(lib):
    assert sdpa(lib, B=0) == lib.MHA_OK
    assert sdpa(lib, Tq=0) == lib.MHA_OK
    assert sdpa(lib, h=0, q=None) == lib.MHA_OK


def mha(lib, dt=1, x=FAKE, ws=FAKE, ws_bytes=1 << 40, B=1, h=2, Tq=8, Tk=8, D=128, dk=64,
        mask=0, lens=None, w=FAKE):
    return lib.lib.mha_forward(dt, x, x, w, w, w, w, FAKE, ws, ws_bytes, B, h, Tq, Tk, D, dk,
                               dk, 0.125, mask, lens, None, None)


def test_mha_rejects_bad_arguments(lib):
    assert mha(lib, x=None) == lib.MHA_ERR_INVALID_ARG
    assert mha(lib, h=0) == lib.MHA_ERR_INVALID_ARG
    assert mha(lib, mask=3, lens=None) == lib.MHA_ERR_INVALID_ARG
    assert mha(lib, dt=0) == lib.MHA_ERR_UNSUPPORTED
    assert mha(lib, dk=128) == lib.MHA_ERR_UNSUPPORTED
    assert mha(lib, D=100) == lib.MHA_ERR_UNSUPPORTED
    assert mha(lib, ws=None) == lib.MHA_ERR_WORKSPACE
    assert mha(lib, ws_bytes=100) == lib.MHA_ERR_WORKSPACE
    assert mha(lib, ws=FAKE + 16) == lib.MHA_ERR_MISALIGNED
    assert mha(lib, w=FAKE + 4) == lib.MHA_ERR_MISALIGNED
    assert mha(lib, B=0) == lib.MHA_OK


def test_python_binding_imports_without_gpu():
    import transformer_scaled_dot_softmax_gb300 as m
    assert m.status_string(6) == "kernel wait timed out"
    assert m.MASKS["causal"] == 1


def decode(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, h=1, Tq=1, Tk=8, dk=64, dv=64, scale=0.125,
           lens=None):
    return lib.lib.sdpa_decode_forward(q, k, v, o, B, h, Tq, Tk, dk, dv, scale, lens, None)


def test_decode_rejects_bad_arguments(lib):
    assert decode(lib, q=None) == lib.MHA_ERR_INVALID_ARG
    assert decode(lib, k=None) == lib.MHA_ERR_INVALID_ARG
    assert decode(lib, o=None) == lib.MHA_ERR_INVALID_ARG
    assert decode(lib, B=-1) == lib.MHA_ERR_INVALID_ARG
    assert decode(lib, scale=float("inf")) == lib.MHA_ERR_INVALID_ARG
    assert decode(lib, Tq=9) == lib.MHA_ERR_UNSUPPORTED
    assert decode(lib, dk=128, dv=128) == lib.MHA_ERR_UNSUPPORTED
    assert decode(lib, q=FAKE + 8) == lib.MHA_ERR_MISALIGNED
    assert decode(lib, v=FAKE + 2) == lib.MHA_ERR_MISALIGNED
    # empty problems are no-ops; T_k == 0 needs no cache pointers
    assert decode(lib, B=0) == lib.MHA_OK
    assert decode(lib, Tq=0) == lib.MHA_OK


def mha_ln(lib, g=FAKE, b=FAKE, eps=1e-5, D=256, **kw):
    x, ws = kw.get("x", FAKE), kw.get("ws", FAKE)
    return lib.lib.mha_forward_add_layernorm(1, x, x, FAKE, FAKE, FAKE, FAKE, g, b, eps, FAKE, ws,
                                             1 << 40, 1, 4, 8, 8, D, 64, 64, 0.125, 0, None, None,
                                             None)


def test_mha_add_layernorm_rejects_bad_arguments(lib):
    assert mha_ln(lib, g=None) == lib.MHA_ERR_INVALID_ARG
    assert mha_ln(lib, b=None) == lib.MHA_ERR_INVALID_ARG
    assert mha_ln(lib, eps=-1.0) == lib.MHA_ERR_INVALID_ARG
    assert mha_ln(lib, eps=float("nan")) == lib.MHA_ERR_INVALID_ARG
    assert mha_ln(lib, g=FAKE + 2) == lib.MHA_ERR_MISALIGNED
    # the normalised row must split into <= 8 blocks of 128 or 256 features
    assert mha_ln(lib, D=192) == lib.MHA_ERR_UNSUPPORTED
    assert mha_ln(lib, D=4096) == lib.MHA_ERR_UNSUPPORTED
    assert mha_ln(lib, x=None) == lib.MHA_ERR_INVALID_ARG


def test_sdpa_lse_rejects_bad_arguments(lib):
    f = lib.lib.sdpa_forward_lse
    args = lambda dt=1, lse=FAKE, B=1: (dt, FAKE, FAKE, FAKE, FAKE, lse, B, 1, 8, 8, 64, 64, 0.125,
                                        0, None, None, None)
    assert f(*args(lse=None)) == lib.MHA_ERR_INVALID_ARG
    assert f(*args(dt=0)) == lib.MHA_ERR_UNSUPPORTED
    assert f(*args(lse=None, B=0)) == lib.MHA_OK


def bwd(lib, dt=1, p=FAKE, ws=FAKE, ws_bytes=1 << 40, B=1, h=1, Tq=8, Tk=8, d=64, mask=0, lens=None,
        lse=FAKE):
    return lib.lib.sdpa_backward(dt, p, p, p, p, p, lse, p, p, p, ws, ws_bytes, B, h, Tq, Tk, d, d,
                                 0.125, mask, lens, None, None)


def test_backward_rejects_bad_arguments(lib):
    assert bwd(lib, p=None) == lib.MHA_ERR_INVALID_ARG
    assert bwd(lib, lse=None) == lib.MHA_ERR_INVALID_ARG
    assert bwd(lib, mask=2, lens=None) == lib.MHA_ERR_INVALID_ARG
    assert bwd(lib, dt=0) == lib.MHA_ERR_UNSUPPORTED
    assert bwd(lib, d=128) == lib.MHA_ERR_UNSUPPORTED
    assert bwd(lib, ws=None) == lib.MHA_ERR_WORKSPACE
    assert bwd(lib, ws_bytes=16) == lib.MHA_ERR_WORKSPACE
    assert bwd(lib, ws=FAKE + 64) == lib.MHA_ERR_MISALIGNED
    assert bwd(lib, p=FAKE + 8) == lib.MHA_ERR_MISALIGNED
    assert bwd(lib, B=0) == lib.MHA_OK
    assert bwd(lib, Tq=0, Tk=0) == lib.MHA_OK
    # fp32 dq accumulator + two per-row vectors over whole 128-row blocks
    assert lib.lib.sdpa_backward_workspace_bytes(2, 3, 130, 7, 64, 64) == (
        2 * 3 * 256 * 64 * 4 + 2 * 2 * 3 * 256 * 4)


def enc(lib, x=FAKE, ws=FAKE, ws_bytes=1 << 40, B=1, T=8, D=128, h=2, F=256, eps=1e-5, w1=FAKE):
    return lib.lib.encoder_layer_forward(x, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, w1, FAKE, FAKE, FAKE,
                                         FAKE, FAKE, eps, FAKE, ws, ws_bytes, B, T, D, h, F, 0.125, 0,
                                         None, None, None)


def test_encoder_layer_rejects_bad_arguments(lib):
    assert enc(lib, x=None) == lib.MHA_ERR_INVALID_ARG
    assert enc(lib, w1=None) == lib.MHA_ERR_INVALID_ARG
    assert enc(lib, eps=-1.0) == lib.MHA_ERR_INVALID_ARG
    assert enc(lib, F=100) == lib.MHA_ERR_UNSUPPORTED          # d_ff % 64
    assert enc(lib, D=192, h=2) == lib.MHA_ERR_UNSUPPORTED     # d_model != 64 h
    assert enc(lib, ws=None) == lib.MHA_ERR_WORKSPACE
    assert enc(lib, ws_bytes=1000) == lib.MHA_ERR_WORKSPACE
    assert enc(lib, w1=FAKE + 2) == lib.MHA_ERR_MISALIGNED
    assert enc(lib, B=0) == lib.MHA_OK
    # attention workspace + the sublayer output + the hidden activations
    assert lib.lib.encoder_layer_workspace_bytes(2, 8, 128, 2, 256) == (
        lib.lib.mha_workspace_bytes(2, 2, 8, 8, 64, 64) + 2 * 8 * 128 * 2 + 2 * 8 * 256 * 2)


def test_positional_encoding_rejects_bad_arguments(lib):
    f = lib.lib.positional_encoding_add
    assert f(None, FAKE, 1, 4, 64, 0, None) == lib.MHA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 1, 4, 60, 0, None) == lib.MHA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, 1, 4, 64, -1, None) == lib.MHA_ERR_INVALID_ARG
    assert f(FAKE + 4, FAKE, 1, 4, 64, 0, None) == lib.MHA_ERR_MISALIGNED
    assert f(FAKE, FAKE, 0, 4, 64, 0, None) == lib.MHA_OK


def host(lib, dt=1, p=FAKE, ws=FAKE, ws_bytes=1 << 40, B=1, h=1, Tq=8, Tk=8, dk=64, dv=64, mask=0,
         lens=None, scale=0.125):
    return lib.lib.sdpa_forward_host(dt, p, p, p, p, ws, ws_bytes, B, h, Tq, Tk, dk, dv, scale, mask,
                                     lens, None, None)


def test_host_path_rejects_bad_arguments(lib):
    # every rejection happens before the library touches CUDA
    assert host(lib, ws=None) == 1
    assert host(lib, ws_bytes=1024) == 1                      # smaller than the device copies
    assert host(lib, ws=FAKE + 16) == 4                       # workspace not 256-byte aligned
    assert host(lib, dk=32, dv=32) == 2                       # bf16 path needs d = 64
    assert host(lib, dt=0, dk=160, dv=160) == 2               # fp32 path: d <= 128
    assert host(lib, dt=7) == 1
    assert host(lib, mask=2, lens=None) == 1                  # key padding needs key_lens
    assert host(lib, mask=9) == 1
    assert host(lib, B=-1) == 1
    assert host(lib, scale=float("nan")) == 1
    assert host(lib, p=None) == 1
    assert host(lib, B=0) == 0 and host(lib, Tq=0) == 0       # empty problems: no-ops


def test_host_workspace_bytes(lib):
    r = lambda x: (x + 255) // 256 * 256
    B, h, Tq, Tk = 2, 3, 130, 7
    bf = lib.lib.sdpa_forward_host_workspace_bytes(1, B, h, Tq, Tk, 64, 64)
    assert bf == r(B * h * Tq * 128) + 2 * r(B * h * Tk * 128) + r(B * h * Tq * 128) + r(B * 4)
    f32 = lib.lib.sdpa_forward_host_workspace_bytes(0, B, h, Tq, Tk, 32, 48)
    assert f32 == r(B * h * Tq * 128) + r(B * h * Tk * 128) + r(B * h * Tk * 192) + r(B * h * Tq * 192) + r(B * 4)
    assert lib.lib.sdpa_forward_host_workspace_bytes(1, -1, h, Tq, Tk, 64, 64) == 0


def test_bf16_key_split_rule(lib):
    """The kernel's choice between its two key splits, a host-side rule: by
    alternate tiles once a 128-row query tile sees 8 key tiles on average."""
    split = lib.lib.sdpa_bf16_key_split
    assert split(8192, 8192, 1) == 1 and split(8192, 8192, 0) == 1   # the causal T=8192 workload
    assert split(128, 128, 0) == 0 and split(512, 512, 1) == 0       # short items: key halves
    assert split(2048, 2048, 1) == 1 and split(1920, 1920, 1) == 1   # causal: 136/16, 120/15 tiles
    assert split(1792, 1792, 1) == 0                                 # 105 tiles over 14 query tiles
    assert split(1000, 1024, 0) == 1 and split(1000, 896, 0) == 0    # non-causal: ceil(T_k/128) >= 8
    assert split(256, 1024, 2) == 1                                  # padding is not counted
    assert split(0, 1024, 0) == 0 and split(64, 0, 0) == 0           # empty problems
    assert split(-1, 8, 0) == -1 and split(8, 8, 7) == -1


def drill(lib, q=FAKE, B=1, h=1, Tq=512, Tk=512, mask=0, lens=None, limit=2_000_000, skip=0,
          status=FAKE):
    return lib.lib.sdpa_forward_timeout_drill(q, FAKE, FAKE, FAKE, B, h, Tq, Tk, 0.125, mask, lens,
                                              limit, skip, status, None)


def test_timeout_drill_rejects_bad_arguments(lib):
    """The failure-detection drill checks its arguments on the host: it needs
    a status word, a wait limit between 0.1 ms and 1 s, a tile index >= 0 and
    a non-empty problem."""
    assert drill(lib, status=None) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, limit=0) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, limit=99_999) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, limit=2_000_000_000) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, skip=-1) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, B=0) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, Tk=0) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, mask=2, lens=None) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, q=None) == lib.MHA_ERR_INVALID_ARG
    assert drill(lib, q=FAKE + 8) == lib.MHA_ERR_MISALIGNED
