"""ctypes view of libmha.so (the C ABI in include/mha.h).

Loading never touches the GPU.  If the library has not been built the import
fails loudly: there is no fallback implementation."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# MHA_LIBRARY may name another build of this same library (the tests load the
# build with device-side bounds checks that way); by default the in-tree build.
LIB_PATH = os.environ.get("MHA_LIBRARY") or os.path.join(_HERE, "_build", "libmha.so")

MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED, MHA_ERR_WORKSPACE = 0, 1, 2, 3
MHA_ERR_MISALIGNED, MHA_ERR_CUDA, MHA_ERR_TIMEOUT, MHA_ERR_BOUNDS = 4, 5, 6, 7
MHA_F32, MHA_BF16 = 0, 1
MHA_STATIC_WORKSPACE_BYTES = 32 << 20
MHA_MASK_NONE, MHA_MASK_CAUSAL, MHA_MASK_KEY_PADDING, MHA_MASK_CAUSAL_KEY_PADDING = 0, 1, 2, 3

# Every symbol include/mha.h declares, with its ctypes signature.
_vp, _ci, _cf, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "sdpa_forward": (_ci, [_ci, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _vp,
                           _vp, _vp]),
    "sdpa_forward_lse": (_ci, [_ci, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _cf,
                               _ci, _vp, _vp, _vp]),
    "sdpa_bf16_key_split": (_ci, [_ci, _ci, _ci]),
    "sdpa_forward_timeout_drill": (_ci, [_vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _cf, _ci, _vp,
                                         ctypes.c_ulonglong, _ci, _vp, _vp]),
    "sdpa_forward_host_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci, _ci]),
    "sdpa_forward_host": (_ci, [_ci, _vp, _vp, _vp, _vp, _vp, _sz, _ci, _ci, _ci, _ci, _ci, _ci,
                                _cf, _ci, _vp, _vp, _vp]),
    "sdpa_backward_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci]),
    "sdpa_backward": (_ci, [_ci, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _ci, _ci,
                            _ci, _ci, _ci, _ci, _cf, _ci, _vp, _vp, _vp]),
    "positional_encoding_add": (_ci, [_vp, _vp, _ci, _ci, _ci, _ci, _vp]),
    "encoder_layer_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci]),
    "encoder_layer_forward": (_ci, [_vp] * 13 + [_cf, _vp, _vp, _sz, _ci, _ci, _ci, _ci, _ci, _cf,
                                                _ci, _vp, _vp, _vp]),
    "sdpa_decode_forward": (_ci, [_vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _cf, _vp,
                                  _vp]),
    "mha_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci]),
    "mha_forward": (_ci, [_ci, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _ci, _ci, _ci, _ci,
                          _ci, _ci, _ci, _cf, _ci, _vp, _vp, _vp]),
    "mha_forward_add_layernorm": (_ci, [_ci, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _cf, _vp, _vp,
                                        _sz, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _vp, _vp,
                                        _vp]),
    "mha_forward_static_workspace": (_ci, [_ci, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci,
                                           _ci, _ci, _ci, _ci, _cf, _ci, _vp, _vp, _vp]),
    "mha_status_string": (ctypes.c_char_p, [_ci]),
    "mha_last_error": (ctypes.c_char_p, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libmha.so is not built (%s); run transformer_scaled_dot_softmax_gb300.build.build() "
            "or __graft_entry__.build() -- there is no CPU fallback" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()
