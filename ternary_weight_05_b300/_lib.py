"""ctypes loader for libbitnet_w2a8.so (the C ABI in include/bitnet_w2a8.h).

There is no fallback: if the shared library is missing or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbitnet_w2a8.so")

# Symbols declared in include/bitnet_w2a8.h, with (restype, argtypes).
_p, _i, _i64, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "bitnet_status_string": (ctypes.c_char_p, [_i]),
    "bitnet_version": (_i, []),
    "bitnet_set_pdl": (None, [_i]),
    "bitnet_pack_workspace_bytes": (_sz, [_i64, _i64]),
    "bitnet_pack_weights": (_i, [_p, _i, _i64, _i64, _f, _f, _p, _p, _p, _p, _sz, _p]),
    "bitnet_quant_act": (_i, [_p, _i, _i64, _i64, _p, _p, _p]),
    "bitnet_gemv_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "bitnet_w2a8_gemv": (_i, [_p, _p, _i64, _p, _p, _i64, _i64, _p, _p, _p, _sz, _p]),
    "bitnet_gemm_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "bitnet_w2a8_gemm": (_i, [_p, _p, _i64, _p, _p, _i64, _i64, _p, _p, _p, _sz, _p]),
    "bitnet_check_device_error": (_i, [_p]),
    "bitnet_w2a8_gemv_static_scratch": (_i, [_p, _p, _i64, _p, _p, _i64, _i64, _p, _p, _p]),
    "bitnet_bitlinear_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "bitnet_bitlinear": (_i, [_p, _i, _i64, _p, _p, _i64, _i64, _p, _p, _p, _p, _p, _sz, _p]),
    "bitnet_bitlinear_swiglu_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "bitnet_pack_weights_grouped": (_i, [_p, _i, _i64, _i64, _i64, _f, _f, _p, _p, _p, _p]),
    "bitnet_w2a8_grouped": (_i, [_p, _p, _i64, _p, _p, _i64, _i64, _i64, _p, _p, _p]),
    "bitnet_bitlinear_grouped_workspace_bytes": (_sz, [_i64, _i64]),
    "bitnet_bitlinear_fake_quant_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "bitnet_selftest_wait_timeout": (_i, [_i64, _p]),
    "bitnet_test_inject_cuda_failures": (_i, [_i]),
    "bitnet_bitlinear_fake_quant": (_i, [_p, _i, _p, _i, _i64, _i64, _i64, _f, _f, _p, _p, _p, _p, _p, _p, _p, _p,
                                         _sz, _p]),
    "bitnet_bitlinear_grouped": (_i, [_p, _i, _i64, _p, _p, _i64, _i64, _i64, _p, _p, _p, _p, _p, _sz, _p]),
    "bitnet_bitlinear_swiglu": (_i, [_p, _i, _i64, _p, _p, _p, _p, _i64, _i64, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "bitnet_rmsnorm_quant_act": (_i, [_p, _i, _i64, _i64, _p, _f, _p, _p, _p, _p, _p]),
    "bitnet_grouped_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "bitnet_w2a8_grouped_ws": (_i, [_p, _p, _i64, _p, _p, _i64, _i64, _i64, _p, _p, _p, _sz, _p]),
    "bitnet_bitlinear_rmsnorm": (_i, [_p, _i, _i64, _p, _f, _p, _p, _i64, _i64, _p, _p, _p, _p, _p, _p, _sz, _p]),
}

STATUS = {
    0: "BITNET_OK", 1: "BITNET_ERR_INVALID_ARG", 2: "BITNET_ERR_SHAPE", 3: "BITNET_ERR_ALIGNMENT",
    4: "BITNET_ERR_UNSUPPORTED", 5: "BITNET_ERR_CUDA", 6: "BITNET_ERR_TIMEOUT", 7: "BITNET_ERR_WORKSPACE",
    8: "BITNET_ERR_TOO_LARGE",
}

_lib = None


class BitnetError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(fn: str, status: int) -> None:
    if status != 0:
        raise BitnetError(fn, status)
