"""ctypes declarations of the C ABI in ``include/pa.h``.

Loading fails loudly (``ImportError``) when ``libpa.so`` has not been built:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_CUDA = 4

PA_KV_BF16 = 0
PA_KV_FP8_E4M3 = 1

PA_STATIC_WORKSPACE_BYTES = 32 << 20

PA_DEVERR_BAD_BLOCK = 0x1
PA_DEVERR_BAD_CONTEXT = 0x2
PA_DEVERR_TIMEOUT = 0x4
PA_DEVERR_BAD_SLOT = 0x8
PA_DEVERR_OUT_OF_BLOCKS = 0x10

# name -> (restype, argtypes); the order matches include/pa.h
_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "pa_slot_mapping": (_I, [_P, _I, _P, _I, _I, _P, _P]),
    "pa_cache_append": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "pa_decode_max_partitions": (_I, [_I, _I, _I]),
    "pa_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "pa_decode_partitions": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _I,
                                  _P, _SZ, _P]),
    "pa_decode_reduce": (_I, [_P, _SZ, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "pa_decode": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _I, _P, _SZ,
                       _P, _P]),
    "pa_decode_step": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F,
                            _I, _P, _SZ, _P, _P, _P]),
    "pa_cache_append_scaled": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "pa_decode_step_scaled": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P,
                                   _P, _F, _I, _P, _SZ, _P, _P, _P]),
    "pa_decode_step_fp8_qk": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P,
                                   _P, _F, _F, _I, _P, _SZ, _P, _P, _P]),
    "pa_block_alloc": (_I, [_P, _I, _P, _I, _I, _I, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P]),
    "pa_block_alloc_chunk": (_I, [_P, _I, _P, _P, _I, _I, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P]),
    "pa_chunk_slot_mapping": (_I, [_P, _I, _P, _P, _I, _I, _P, _P]),
    "pa_prefill": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _P,
                        _P]),
    "pa_prefill_scaled": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _F, _P,
                               _P]),
    "pa_prefill_mma": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F,
                            _P, _P]),
    "pa_decode_static_workspace": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                        _F, _I, _P, _P]),
    "pa_test_set_wait": (_I, [ctypes.c_uint64, _I]),
    "pa_device_errors": (_I, [ctypes.POINTER(ctypes.c_uint), _I]),
    "pa_status_string": (ctypes.c_char_p, [_I]),
    "pa_last_error": (ctypes.c_char_p, []),
}

_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libpa.so (``PA_LIBRARY`` in the environment selects another build
    of the same library, e.g. a launch-shape variant)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or os.environ.get("PA_LIBRARY") or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(
            f"{p} not found: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib
