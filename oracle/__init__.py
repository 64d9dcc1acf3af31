"""Oracle for the MoE token permute / unpermute path: plain C on the CPU.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never imports it.

Every function here marshals numpy arrays into ``oracle.c`` (built with
``gcc -O2 -ffp-contract=off``) and returns numpy arrays.  bf16 tensors are
carried as ``uint16`` bit patterns.  What each function computes, and the
page it follows, is documented in ``oracle.c``.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (in place) if it is stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Flags(ctypes.Structure):
    _fields_ = [("bad_split", ctypes.c_int32), ("bad_order", ctypes.c_int32),
                ("split_overflow", ctypes.c_int32), ("rows_overflow", ctypes.c_int32),
                ("bad_padded", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Routes every oracle call to another build of oracle.c for the duration
    (the tests that plant a mistake in a copy of the oracle use this)."""
    global _lib
    with _lock:
        saved = _lib
        _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _configure(lib):
    P = ctypes.c_void_p
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    lib.orc_f32_from_bf16.argtypes = [ctypes.c_uint16]
    lib.orc_f32_from_bf16.restype = ctypes.c_float
    lib.orc_bf16_from_f32.argtypes = [ctypes.c_float]
    lib.orc_bf16_from_f32.restype = ctypes.c_uint16
    lib.orc_build_map.argtypes = [P, i64, i32, i32, P, P, P, P]
    lib.orc_build_map.restype = i64
    lib.orc_build_map_capacity.argtypes = [P, i64, i32, i32, i32, P, P, P, P]
    lib.orc_build_map_capacity.restype = i64
    lib.orc_bf16_from_f64.argtypes = [ctypes.c_double]
    lib.orc_bf16_from_f64.restype = ctypes.c_uint16
    lib.orc_unpermute_ep.argtypes = [P, P, P, P, i64, i32, i32, i32, i32, i32, i32, P]
    lib.orc_unpermute_ep.restype = None
    lib.orc_topk_softmax.argtypes = [P, i64, i32, i32, i32, i32, P, P]
    lib.orc_topk_softmax.restype = None
    lib.orc_topk_softmax_bwd.argtypes = [P, P, P, i64, i32, i32, P]
    lib.orc_topk_softmax_bwd.restype = None
    lib.orc_permute.argtypes = [P, P, P, i64, i32, i32, P, P]
    lib.orc_permute.restype = None
    lib.orc_unpermute.argtypes = [P, P, P, i64, i32, i32, P]
    lib.orc_unpermute.restype = None
    lib.orc_permute_bwd.argtypes = [P, P, P, i64, i32, i32, P, P]
    lib.orc_permute_bwd.restype = None
    lib.orc_unpermute_bwd.argtypes = [P, P, P, P, i64, i32, i32, P, P]
    lib.orc_unpermute_bwd.restype = None
    lib.orc_sort_chunks_pad.argtypes = [P, P, P, P, P, i32, i32, i32, i64, i64, i32,
                                        P, P, P, P, ctypes.POINTER(_Flags)]
    lib.orc_sort_chunks_pad.restype = None
    for name in ("orc_unpad_restore", "orc_sort_chunks_pad_bwd",
                 "orc_unpad_restore_bwd"):
        fn = getattr(lib, name)
        fn.argtypes = [P, P, P, i64, i64, i32, P, P]
        fn.restype = None
    return lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# scalar conversions
# --------------------------------------------------------------------------

def bf16_from_f32(values) -> np.ndarray:
    """float32 array -> uint16 bf16 bits, round to nearest even."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    out = np.fromiter((lib.orc_bf16_from_f32(float(f)) for f in v), dtype=np.uint16,
                      count=v.size)
    return out.reshape(np.shape(values))


def bf16_from_f64(values) -> np.ndarray:
    """float64 array -> uint16 bf16 bits, one round-to-nearest-even."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64).ravel()
    out = np.fromiter((lib.orc_bf16_from_f64(float(f)) for f in v), dtype=np.uint16,
                      count=v.size)
    return out.reshape(np.shape(values))


def f32_from_bf16(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.fromiter((lib.orc_f32_from_bf16(int(x)) for x in b), dtype=np.float32,
                      count=b.size)
    return out.reshape(np.shape(bits))


# --------------------------------------------------------------------------
# routing map, permute, unpermute and their backwards
# --------------------------------------------------------------------------

def build_map(idx: np.ndarray, E: int):
    """Returns (row_id_map[T,K], sorted_to_flat[T*K], counts[E], offsets[E+1], n_bad)."""
    lib = _load()
    idx = _c(idx, np.int32)
    T, K = idx.shape
    row_id_map = np.empty((T, K), np.int32)
    s2f = np.empty(T * K, np.int32)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    bad = lib.orc_build_map(_p(idx), T, K, E, _p(row_id_map), _p(s2f), _p(counts),
                            _p(offsets))
    return row_id_map, s2f, counts, offsets, int(bad)


def build_map_capacity(idx: np.ndarray, E: int, capacity: int):
    """build_map keeping at most `capacity` routes per expert (earliest first)."""
    lib = _load()
    idx = _c(idx, np.int32)
    T, K = idx.shape
    row_id_map = np.empty((T, K), np.int32)
    s2f = np.empty(T * K, np.int32)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    bad = lib.orc_build_map_capacity(_p(idx), T, K, E, capacity, _p(row_id_map), _p(s2f),
                                     _p(counts), _p(offsets))
    return row_id_map, s2f, counts, offsets, int(bad)


def _out(a, shape, dtype):
    """A caller-supplied output array, checked to be a C-contiguous array the
    C code may write through."""
    if a.dtype != dtype or a.shape[1:] != shape[1:] or not a.flags.c_contiguous \
            or not a.flags.writeable:
        raise ValueError("output array of the wrong type, shape or layout")
    return a


def permute(x, probs, row_id_map, out_rows=None, out=None, out_probs=None):
    """x[T,H] uint16, probs[T,K] f32 or None -> (out[out_rows,H], out_probs or None).

    Rows no slot maps to are left at zero here (the CUDA path leaves them
    unwritten; the tests compare only mapped rows).  With `out` (and
    `out_probs`) given, only the mapped rows of those arrays are written, so
    calls on disjoint token ranges can share them."""
    lib = _load()
    x = _c(x, np.uint16)
    row_id_map = _c(row_id_map, np.int32)
    probs = _c(probs, np.float32)
    T, H = x.shape
    K = row_id_map.shape[1]
    if out_rows is None:
        out_rows = T * K if out is None else out.shape[0]
    if out is None:
        out = np.zeros((out_rows, H), np.uint16)
    out = _out(out, (out_rows, H), np.uint16)
    if probs is not None and out_probs is None:
        out_probs = np.zeros(out_rows, np.float32)
    if probs is None:
        out_probs = None
    elif out_probs.shape != (out.shape[0],):
        raise ValueError("out_probs must have one entry per row of out")
    lib.orc_permute(_p(x), _p(probs), _p(row_id_map), T, K, H, _p(out), _p(out_probs))
    return out, out_probs


def unpermute(rows, probs, row_id_map, T, H):
    lib = _load()
    rows = _c(rows, np.uint16)
    probs = _c(probs, np.float32)
    row_id_map = _c(row_id_map, np.int32)
    K = row_id_map.shape[1]
    out = np.empty((T, H), np.uint16)
    lib.orc_unpermute(_p(rows), _p(probs), _p(row_id_map), T, K, H, _p(out))
    return out


def unpermute_ep(rows, probs, row_id_map, idx, T, H, E, ep_size, bf16_partials=False,
                 fp64_cross_rank=False):
    """Rank-ordered combine over ep_size ranks of E/ep_size experts each."""
    lib = _load()
    rows = _c(rows, np.uint16)
    probs = _c(probs, np.float32)
    row_id_map = _c(row_id_map, np.int32)
    idx = _c(idx, np.int32)
    K = row_id_map.shape[1]
    out = np.empty((T, H), np.uint16)
    lib.orc_unpermute_ep(_p(rows), _p(probs), _p(row_id_map), _p(idx), T, K, H, E, ep_size,
                         int(bool(bf16_partials)), int(bool(fp64_cross_rank)), _p(out))
    return out


def permute_bwd(g_out, g_out_probs, row_id_map, T, H):
    lib = _load()
    g_out = _c(g_out, np.uint16)
    g_out_probs = _c(g_out_probs, np.float32)
    row_id_map = _c(row_id_map, np.int32)
    K = row_id_map.shape[1]
    g_x = np.empty((T, H), np.uint16)
    g_probs = np.empty((T, K), np.float32) if g_out_probs is not None else None
    lib.orc_permute_bwd(_p(g_out), _p(g_out_probs), _p(row_id_map), T, K, H, _p(g_x),
                        _p(g_probs))
    return g_x, g_probs


def unpermute_bwd(g_y, rows, probs, row_id_map, out_rows=None, g_rows=None):
    """Returns (g_rows[out_rows,H] uint16, g_probs[T,K] float64 or None).

    With `g_rows` given, only the rows the map names are written into it."""
    lib = _load()
    g_y = _c(g_y, np.uint16)
    rows = _c(rows, np.uint16)
    probs = _c(probs, np.float32)
    row_id_map = _c(row_id_map, np.int32)
    T, H = g_y.shape
    K = row_id_map.shape[1]
    if out_rows is None:
        out_rows = T * K if g_rows is None else g_rows.shape[0]
    if g_rows is None:
        g_rows = np.zeros((out_rows, H), np.uint16)
    g_rows = _out(g_rows, (out_rows, H), np.uint16)
    g_probs = np.empty((T, K), np.float64) if probs is not None else None
    lib.orc_unpermute_bwd(_p(g_y), _p(rows), _p(probs), _p(row_id_map), T, K, H,
                          _p(g_rows), _p(g_probs))
    return g_rows, g_probs


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------

def topk_softmax(logits, K, n_groups=1, topk_groups=1):
    """logits f32 [T,E] -> (idx int32 [T,K], probs f32 [T,K])."""
    lib = _load()
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, K), np.int32)
    probs = np.empty((T, K), np.float32)
    lib.orc_topk_softmax(_p(logits), T, E, K, n_groups, topk_groups, _p(idx), _p(probs))
    return idx, probs


def topk_softmax_bwd(g_probs, probs, idx, E):
    lib = _load()
    g_probs = _c(g_probs, np.float32)
    probs = _c(probs, np.float32)
    idx = _c(idx, np.int32)
    T, K = idx.shape
    g_logits = np.empty((T, E), np.float32)
    lib.orc_topk_softmax_bwd(_p(g_probs), _p(probs), _p(idx), T, E, K, _p(g_logits))
    return g_logits


# --------------------------------------------------------------------------
# chunk sort + pad, unpad + restore
# --------------------------------------------------------------------------

def as_units(rows: np.ndarray) -> np.ndarray:
    """A [N, ...] array of 2- or 4-byte elements as [N, W] uint16 units (the
    chunk functions only move bits)."""
    a = np.ascontiguousarray(rows)
    return a.reshape(a.shape[0], -1).view(np.uint16)


def sort_chunks_pad(x, probs, split_sizes, chunk_order, G, align, out_rows, padded_sizes=None):
    """Returns (out, out_probs, row_map, group_off[G+1] int64, flags dict).
    x may be bf16 / fp16 bits (uint16) or float32 rows; out has x's dtype."""
    lib = _load()
    dtype = np.asarray(x).dtype
    xu = as_units(x)
    probs = _c(probs, np.float32)
    split_sizes = _c(split_sizes, np.int32)
    chunk_order = _c(chunk_order, np.int32)
    padded_sizes = _c(padded_sizes, np.int32)
    N, W = xu.shape
    C = split_sizes.shape[0]
    out = np.empty((out_rows, W), np.uint16)
    out_probs = np.empty(out_rows, np.float32) if probs is not None else None
    row_map = np.empty(out_rows, np.int32)
    group_off = np.empty(G + 1, np.int64)
    flags = _Flags()
    lib.orc_sort_chunks_pad(_p(xu), _p(probs), _p(split_sizes), _p(chunk_order),
                            _p(padded_sizes), C, G, align, N, out_rows, W, _p(out),
                            _p(out_probs), _p(row_map), _p(group_off), ctypes.byref(flags))
    fl = {name: int(getattr(flags, name)) for name, _ in _Flags._fields_}
    return out.view(dtype).reshape((out_rows,) + np.asarray(x).shape[1:]), out_probs, \
        row_map, group_off, fl


def _rowmap_call(name, src, src_probs, row_map, N, out_shape_rows, init):
    lib = _load()
    dtype = np.asarray(src).dtype
    su = as_units(src)
    src_probs = _c(src_probs, np.float32)
    row_map = _c(row_map, np.int32)
    W = su.shape[1]
    out = as_units(np.array(init[0], copy=True)).copy() if init is not None else \
        np.zeros((out_shape_rows, W), np.uint16)
    out_probs = None
    if src_probs is not None:
        out_probs = np.array(init[1], dtype=np.float32, copy=True) if init is not None \
            else np.zeros(out_shape_rows, np.float32)
    getattr(lib, name)(_p(su), _p(src_probs), _p(row_map), row_map.shape[0], N, W,
                       _p(out), _p(out_probs))
    return out.view(dtype).reshape((out_shape_rows,) + np.asarray(src).shape[1:]), out_probs


def unpad_restore(padded, padded_probs, row_map, N, init=None):
    """y[N,H]: rows no output row maps to keep ``init`` (zeros by default)."""
    return _rowmap_call("orc_unpad_restore", padded, padded_probs, row_map, N, N, init)


def sort_chunks_pad_bwd(g_out, g_out_probs, row_map, N, init=None):
    return _rowmap_call("orc_sort_chunks_pad_bwd", g_out, g_out_probs, row_map, N, N,
                        init)


def unpad_restore_bwd(g_y, g_y_probs, row_map, N):
    lib = _load()
    dtype = np.asarray(g_y).dtype
    gu = as_units(g_y)
    g_y_probs = _c(g_y_probs, np.float32)
    row_map = _c(row_map, np.int32)
    out_rows = row_map.shape[0]
    W = gu.shape[1]
    g_padded = np.empty((out_rows, W), np.uint16)
    g_padded_probs = np.empty(out_rows, np.float32) if g_y_probs is not None else None
    lib.orc_unpad_restore_bwd(_p(gu), _p(g_y_probs), _p(row_map), out_rows, N, W,
                              _p(g_padded), _p(g_padded_probs))
    return g_padded.view(dtype).reshape((out_rows,) + np.asarray(g_y).shape[1:]), \
        g_padded_probs
