"""ctypes loader for ``liblora_linear.so``: declares every exported C function's signature.

Raises if the library has not been built; there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liblora_linear.so")

_lib = None

P = C.c_void_p
I32P = C.POINTER(C.c_int32)
IP = C.POINTER(C.c_int)

SIGNATURES = {
    "lora_linear_create": (C.c_int, [C.POINTER(P), C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]),
    "lora_linear_forward": (C.c_int, [P, P, C.c_int, I32P, I32P, C.c_int, P, C.POINTER(P), C.POINTER(P),
                                      C.POINTER(C.c_float), C.c_int, P, P]),
    "lora_linear_forward_host": (C.c_int, [P, P, C.c_int, I32P, I32P, C.c_int, P, C.POINTER(P), C.POINTER(P),
                                           C.POINTER(C.c_float), C.c_int, P, P]),
    "lora_linear_w4_repack": (C.c_int, [P, P, C.c_longlong, P]),
    "lora_linear_forward_w4": (C.c_int, [P, P, C.c_int, I32P, I32P, C.c_int, P, P, C.POINTER(P), C.POINTER(P),
                                         C.POINTER(C.c_float), C.c_int, P, P]),
    "lora_linear_forward_host_w4": (C.c_int, [P, P, C.c_int, I32P, I32P, C.c_int, P, P, C.POINTER(P),
                                              C.POINTER(P), C.POINTER(C.c_float), C.c_int, P, P]),
    "lora_linear_destroy": (C.c_int, [P]),
    "lora_linear_status": (C.c_int, [P, C.c_int]),
    "lora_linear_plan": (C.c_int, [I32P, I32P, C.c_int, C.c_int, I32P, IP, I32P, IP]),
    "lora_linear_validate": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, P, C.c_int, I32P, I32P,
                                       C.c_int, P, C.POINTER(P), C.POINTER(P), C.POINTER(C.c_float), C.c_int, P]),
    "lora_linear_set_option": (C.c_int, [P, C.c_int, C.c_longlong]),
    "lora_linear_timing": (C.c_int, [P, C.c_int, C.POINTER(C.c_double), C.POINTER(C.c_longlong),
                                     C.POINTER(C.c_longlong)]),
    "lora_linear_describe": (C.c_int, [P, C.c_int, I32P, I32P, C.c_int, IP, IP, IP, IP, IP, IP, IP]),
    "lora_linear_error_string": (C.c_char_p, [C.c_int]),
    "lora_linear_shape": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, I32P, I32P, C.c_int, C.c_int,
                                    IP, IP, IP, IP, IP, IP, IP]),
    "lora_linear_host_chunks": (C.c_int, [C.c_int, I32P, IP]),
    "lora_linear_k_split": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, IP]),
    "lora_linear_forward_noalloc": (C.c_int, [P, C.c_int, I32P, I32P, C.c_int, C.c_int, C.c_int, C.c_int, P,
                                              C.POINTER(P), C.POINTER(P), C.POINTER(C.c_float), C.c_int, P, P]),
}

# return codes and options, as in include/lora_linear.h
LORA_OK, LORA_EINVAL, LORA_ENOMEM, LORA_ECUDA, LORA_ETIMEOUT, LORA_EUNSUPPORTED, LORA_ENODEV = 0, -1, -2, -3, -4, -5, -6
(OPT_TILE_N, OPT_WAIT_LIMIT_US, OPT_DEBUG_STALL, OPT_TIMING, OPT_RASTER, OPT_TWO_LAUNCH, OPT_CLUSTER,
 OPT_RASTER_GROUP, _OPT_RETIRED_9, OPT_TILE_K, OPT_INLINE_WORK_LIST, OPT_MMA_GROUP,
 OPT_DEBUG_PUBLISH_DELAY_US, OPT_K_SPLIT, OPT_MAX_CTAS, OPT_PDL,
 OPT_TOKEN_COLUMNS, OPT_W4_K_SPLIT, OPT_WIDE_TILES) = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16, 17, 18, 19


def load():
    """The loaded library (once per process)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                           "(or python -m mixed_lora_projection_gb300.build)")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
