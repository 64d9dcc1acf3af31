"""ctypes loader for libmp.so.  Loading fails loudly: there is no fallback."""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I32, I64, SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t

# name -> (restype, argtypes), exactly the prototypes of include/mp.h
SIGNATURES = {
    "mp_status_string": (ctypes.c_char_p, [I32]),
    "mp_last_cuda_error": (I32, []),
    "mp_build_map_workspace_size": (SZ, [I64, I32, I32]),
    "mp_build_map": (I32, [P, I64, I32, I32, P, P, P, P, P, SZ, P, P]),
    "mp_build_map_capacity": (I32, [P, I64, I32, I32, I32, P, P, P, P, P, SZ, P, P]),
    "mp_build_map_noalloc": (I32, [P, I64, I32, I32, P, P, P, P, P, P]),
    "mp_topk_softmax": (I32, [P, I64, I32, I32, I32, I32, P, P, P]),
    "mp_topk_softmax_bwd": (I32, [P, P, P, I64, I32, I32, P, P]),
    "mp_permute": (I32, [P, P, P, I64, I32, I32, P, P, P]),
    "mp_unpermute": (I32, [P, P, P, I64, I32, I32, P, P]),
    "mp_unpermute_ep": (I32, [P, P, P, P, I64, I32, I32, I32, I32, I32, P, P]),
    "mp_permute_bwd": (I32, [P, P, P, I64, I32, I32, P, P, P]),
    "mp_unpermute_bwd": (I32, [P, P, P, P, I64, I32, I32, P, P, P]),
    "mp_zero_rows_from": (I32, [P, I64, I64, P, P]),
    "mp_sort_chunks_pad": (I32, [P, P, P, P, I32, I32, I32, I64, I64, I32, P, P, P, P, P, P]),
    "mp_unpad_restore": (I32, [P, P, P, I64, I64, I32, P, P, P, P]),
    "mp_sort_chunks_pad_bwd": (I32, [P, P, P, I64, I64, I32, P, P, P, P]),
    "mp_unpad_restore_bwd": (I32, [P, P, P, I64, I64, I32, P, P, P, P]),
    "mp_sort_chunks_pad_ex": (I32, [P, I32, P, P, P, P, I32, I32, I32, I64, I64, I32, P, P, P, P,
                                    P, P]),
    "mp_unpad_restore_ex": (I32, [P, I32, P, P, I64, I64, I32, P, P, P, P]),
    "mp_sort_chunks_pad_bwd_ex": (I32, [P, I32, P, P, I64, I64, I32, P, P, P, P]),
    "mp_unpad_restore_bwd_ex": (I32, [P, I32, P, P, I64, I64, I32, P, P, P, P]),
}


def path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libmp.so.  Raises if it is absent (run ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            if not build_if_missing:
                raise RuntimeError(
                    f"libmp.so is not built ({_build.LIB}); build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            _build.build()
        lib = ctypes.CDLL(_build.LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
