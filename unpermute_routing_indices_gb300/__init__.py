"""MoE token permute / unpermute for one GB300 GPU.

A thin binding over the C ABI of ``libmp.so`` (declared in ``include/mp.h``):
every function here has the name of the C entry point it calls, checks and
marshals torch tensors (device, dtype, contiguity, shapes), allocates the
outputs it is not given, and launches on the current torch CUDA stream.  All
arithmetic and data movement happens in the library's CUDA kernels; there is
no CPU or PyTorch fallback, and a missing library raises.

Tensors: bf16 hidden rows, fp32 probabilities, int32 indices and maps.
"""
from __future__ import annotations

import contextlib
import ctypes

import torch

from . import _lib

__all__ = [
    "MPError", "mp_build_map", "mp_build_map_capacity", "mp_build_map_workspace_size",
    "mp_topk_softmax", "mp_topk_softmax_bwd", "mp_permute", "mp_unpermute", "mp_unpermute_ep", "EP_BF16_PARTIALS", "EP_FP64_CROSS_RANK",
    "mp_permute_bwd", "mp_unpermute_bwd", "mp_sort_chunks_pad", "mp_unpad_restore",
    "mp_sort_chunks_pad_bwd", "mp_unpad_restore_bwd", "status_bits", "library_path",
]

STATUS_BITS = {
    "bad_expert": 0x1, "bad_split": 0x2, "bad_order": 0x4, "split_overflow": 0x8,
    "rows_overflow": 0x10, "bad_row": 0x20, "bad_padded": 0x40,
}


DTYPES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}   # MP_DTYPE_*
EP_BF16_PARTIALS = 0x1
EP_FP64_CROSS_RANK = 0x2


class MPError(RuntimeError):
    def __init__(self, fn: str, code: int):
        lib = _lib.load()
        msg = lib.mp_status_string(code).decode()
        if code == -4:
            msg += f" (cudaError {lib.mp_last_cuda_error()})"
        super().__init__(f"{fn}: {msg} [{code}]")
        self.code = code


def library_path() -> str:
    return _lib.path()


def status_bits(word: int) -> set[str]:
    """Names of the MP_STATUS_* bits set in a device status word."""
    return {name for name, bit in STATUS_BITS.items() if word & bit}


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise MPError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device):
    """The current CUDA stream of `device` as a raw handle."""
    if _raw_stream is not None and device.index is not None:
        return ctypes.c_void_p(_raw_stream(device.index))
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _on(device):
    """Context that makes `device` current for the call (free when it is)."""
    if device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _need(t, name, dtype, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _opt(t, *a, **k):
    return None if t is None else _need(t, *a, **k)


def _shape(t, name, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# --------------------------------------------------------------------------
# routing map
# --------------------------------------------------------------------------

def mp_build_map_workspace_size(num_tokens: int, topk: int, num_experts: int) -> int:
    n = _lib.load().mp_build_map_workspace_size(num_tokens, topk, num_experts)
    if n == 0:
        raise ValueError("invalid sizes for mp_build_map")
    return int(n)


def mp_build_map(idx, num_experts: int, *, with_sorted_to_flat: bool = True,
                 row_id_map=None, sorted_to_flat=None, counts=None, offsets=None,
                 workspace=None, status=None):
    """idx int32 [T,K] (-1 = empty slot) -> (row_id_map [T,K], sorted_to_flat [T*K]
    or None, counts [E], offsets [E+1]), all int32 on idx's device."""
    return _build_map("mp_build_map", idx, num_experts, None, with_sorted_to_flat, row_id_map,
                      sorted_to_flat, counts, offsets, workspace, status)


def mp_build_map_capacity(idx, num_experts: int, capacity: int, *,
                          with_sorted_to_flat: bool = True, row_id_map=None,
                          sorted_to_flat=None, counts=None, offsets=None, workspace=None,
                          status=None):
    """mp_build_map keeping at most `capacity` routes per expert (the earliest in
    token, slot order); dropped routes get row -1 and offsets[E] is the row count."""
    return _build_map("mp_build_map_capacity", idx, num_experts, int(capacity),
                      with_sorted_to_flat, row_id_map, sorted_to_flat, counts, offsets,
                      workspace, status)


def _build_map(fn, idx, num_experts, capacity, with_sorted_to_flat, row_id_map, sorted_to_flat,
               counts, offsets, workspace, status):
    lib = _lib.load()
    _need(idx, "idx", torch.int32, 2)
    dev = idx.device
    T, K = idx.shape
    E = int(num_experts)
    row_id_map = torch.empty((T, K), dtype=torch.int32, device=dev) if row_id_map is None \
        else _need(row_id_map, "row_id_map", torch.int32, 2, dev)
    if sorted_to_flat is None and with_sorted_to_flat:
        sorted_to_flat = torch.empty(T * K, dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev) if counts is None \
        else _need(counts, "counts", torch.int32, 1, dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None \
        else _need(offsets, "offsets", torch.int32, 1, dev)
    _shape(row_id_map, "row_id_map", (T, K))
    _shape(counts, "counts", (E,))
    _shape(offsets, "offsets", (E + 1,))
    if sorted_to_flat is not None:
        _need(sorted_to_flat, "sorted_to_flat", torch.int32, 1, dev)
        _shape(sorted_to_flat, "sorted_to_flat", (T * K,))
    ws_bytes = mp_build_map_workspace_size(T, K, E)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    else:
        _need(workspace, "workspace", torch.uint8, 1, dev)
    _opt(status, "status", torch.int32, 1, dev)
    with _on(dev):
        if capacity is None:
            code = lib.mp_build_map(
                _ptr(idx), T, K, E, _ptr(row_id_map), _ptr(sorted_to_flat), _ptr(counts),
                _ptr(offsets), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev))
        else:
            code = lib.mp_build_map_capacity(
                _ptr(idx), T, K, E, capacity, _ptr(row_id_map), _ptr(sorted_to_flat),
                _ptr(counts), _ptr(offsets), _ptr(workspace), workspace.numel(), _ptr(status),
                _stream(dev))
        _check(fn, code)
    return row_id_map, sorted_to_flat, counts, offsets


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------

def mp_topk_softmax(logits, topk: int, *, n_groups: int = 1, topk_groups: int = 1, idx=None,
                    probs=None):
    """logits fp32 [T,E] -> (idx int32 [T,K], probs fp32 [T,K]): top-K experts
    (optionally within the best `topk_groups` of `n_groups` expert groups) and
    the fp32 softmax over the K picked logits."""
    lib = _lib.load()
    _need(logits, "logits", torch.float32, 2)
    dev = logits.device
    T, E = logits.shape
    K = int(topk)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev) if idx is None \
        else _need(idx, "idx", torch.int32, 2, dev)
    probs = torch.empty((T, K), dtype=torch.float32, device=dev) if probs is None \
        else _need(probs, "probs", torch.float32, 2, dev)
    _shape(idx, "idx", (T, K))
    _shape(probs, "probs", (T, K))
    with _on(dev):
        _check("mp_topk_softmax", lib.mp_topk_softmax(
            _ptr(logits), T, E, K, int(n_groups), int(topk_groups), _ptr(idx), _ptr(probs),
            _stream(dev)))
    return idx, probs


def mp_topk_softmax_bwd(g_probs, probs, idx, num_experts: int, *, g_logits=None):
    """Gradient of mp_topk_softmax w.r.t. the logits: fp32 [T,E]."""
    lib = _lib.load()
    _need(g_probs, "g_probs", torch.float32, 2)
    dev = g_probs.device
    T, K = g_probs.shape
    _need(probs, "probs", torch.float32, 2, dev)
    _need(idx, "idx", torch.int32, 2, dev)
    _shape(probs, "probs", (T, K))
    _shape(idx, "idx", (T, K))
    E = int(num_experts)
    g_logits = torch.empty((T, E), dtype=torch.float32, device=dev) if g_logits is None \
        else _need(g_logits, "g_logits", torch.float32, 2, dev)
    _shape(g_logits, "g_logits", (T, E))
    with _on(dev):
        _check("mp_topk_softmax_bwd", lib.mp_topk_softmax_bwd(
            _ptr(g_probs), _ptr(probs), _ptr(idx), T, E, K, _ptr(g_logits), _stream(dev)))
    return g_logits


# --------------------------------------------------------------------------
# permute / unpermute and backwards
# --------------------------------------------------------------------------

def mp_permute(x, row_id_map, probs=None, *, num_out_rows: int | None = None, out=None,
               out_probs=None):
    """x bf16 [T,H] -> (out bf16 [R,H], out_probs fp32 [R] or None), R = T*K by default."""
    lib = _lib.load()
    _need(x, "x", torch.bfloat16, 2)
    dev = x.device
    _need(row_id_map, "row_id_map", torch.int32, 2, dev)
    T, H = x.shape
    K = row_id_map.shape[1]
    _shape(row_id_map, "row_id_map", (T, K))
    R = T * K if num_out_rows is None else int(num_out_rows)
    if probs is not None:
        _need(probs, "probs", torch.float32, 2, dev)
        _shape(probs, "probs", (T, K))
    out = torch.empty((R, H), dtype=torch.bfloat16, device=dev) if out is None \
        else _need(out, "out", torch.bfloat16, 2, dev)
    if probs is not None and out_probs is None:
        out_probs = torch.empty(out.shape[0], dtype=torch.float32, device=dev)
    _opt(out_probs, "out_probs", torch.float32, 1, dev)
    with _on(dev):
        _check("mp_permute", lib.mp_permute(
            _ptr(x), _ptr(probs), _ptr(row_id_map), T, K, H, _ptr(out),
            _ptr(out_probs if probs is not None else None), _stream(dev)))
    return out, (out_probs if probs is not None else None)


def mp_unpermute(rows, row_id_map, probs=None, *, out=None):
    """rows bf16 [R,H] -> out bf16 [T,H] (slot-order fp32 FMA, one bf16 rounding)."""
    lib = _lib.load()
    _need(rows, "rows", torch.bfloat16, 2)
    dev = rows.device
    _need(row_id_map, "row_id_map", torch.int32, 2, dev)
    T, K = row_id_map.shape
    H = rows.shape[1]
    if probs is not None:
        _need(probs, "probs", torch.float32, 2, dev)
        _shape(probs, "probs", (T, K))
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if out is None \
        else _need(out, "out", torch.bfloat16, 2, dev)
    _shape(out, "out", (T, H))
    with _on(dev):
        _check("mp_unpermute", lib.mp_unpermute(
            _ptr(rows), _ptr(probs), _ptr(row_id_map), T, K, H, _ptr(out), _stream(dev)))
    return out


def mp_unpermute_ep(rows, row_id_map, idx, num_experts: int, ep_size: int, probs=None, *,
                    bf16_partials: bool = False, fp64_cross_rank: bool = False, out=None):
    """Rank-ordered combine over `ep_size` expert-parallel ranks: per-rank
    slot-order FMA partials (optionally rounded to bf16), added in rank order
    (fp32, or fp64), one bf16 rounding.  idx int32 [T,K] holds each slot's expert."""
    lib = _lib.load()
    _need(rows, "rows", torch.bfloat16, 2)
    dev = rows.device
    _need(row_id_map, "row_id_map", torch.int32, 2, dev)
    T, K = row_id_map.shape
    _need(idx, "idx", torch.int32, 2, dev)
    _shape(idx, "idx", (T, K))
    H = rows.shape[1]
    if probs is not None:
        _need(probs, "probs", torch.float32, 2, dev)
        _shape(probs, "probs", (T, K))
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if out is None \
        else _need(out, "out", torch.bfloat16, 2, dev)
    _shape(out, "out", (T, H))
    flags = (EP_BF16_PARTIALS if bf16_partials else 0) | \
        (EP_FP64_CROSS_RANK if fp64_cross_rank else 0)
    with _on(dev):
        _check("mp_unpermute_ep", lib.mp_unpermute_ep(
            _ptr(rows), _ptr(probs), _ptr(row_id_map), _ptr(idx), T, K, H, int(num_experts),
            int(ep_size), flags, _ptr(out), _stream(dev)))
    return out


def mp_permute_bwd(g_out, row_id_map, g_out_probs=None, *, g_x=None, g_probs=None):
    """Gradient of mp_permute: (g_x bf16 [T,H], g_probs fp32 [T,K] or None)."""
    lib = _lib.load()
    _need(g_out, "g_out", torch.bfloat16, 2)
    dev = g_out.device
    _need(row_id_map, "row_id_map", torch.int32, 2, dev)
    T, K = row_id_map.shape
    H = g_out.shape[1]
    _opt(g_out_probs, "g_out_probs", torch.float32, 1, dev)
    g_x = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if g_x is None \
        else _need(g_x, "g_x", torch.bfloat16, 2, dev)
    _shape(g_x, "g_x", (T, H))
    if g_out_probs is not None and g_probs is None:
        g_probs = torch.empty((T, K), dtype=torch.float32, device=dev)
    if g_out_probs is None:
        g_probs = None
    _opt(g_probs, "g_probs", torch.float32, 2, dev)
    with _on(dev):
        _check("mp_permute_bwd", lib.mp_permute_bwd(
            _ptr(g_out), _ptr(g_out_probs), _ptr(row_id_map), T, K, H, _ptr(g_x),
            _ptr(g_probs), _stream(dev)))
    return g_x, g_probs


def mp_unpermute_bwd(g_y, row_id_map, rows=None, probs=None, *, num_out_rows=None,
                     g_rows=None, g_probs=None):
    """Gradient of mp_unpermute: (g_rows bf16 [R,H], g_probs fp32 [T,K] or None).
    With probs, `rows` (the forward input) is required."""
    lib = _lib.load()
    _need(g_y, "g_y", torch.bfloat16, 2)
    dev = g_y.device
    _need(row_id_map, "row_id_map", torch.int32, 2, dev)
    T, K = row_id_map.shape
    H = g_y.shape[1]
    _shape(g_y, "g_y", (T, H))
    if probs is not None:
        _need(probs, "probs", torch.float32, 2, dev)
        _shape(probs, "probs", (T, K))
        if rows is None:
            raise ValueError("mp_unpermute_bwd with probs needs the forward rows")
    _opt(rows, "rows", torch.bfloat16, 2, dev)
    R = (rows.shape[0] if rows is not None else T * K) if num_out_rows is None \
        else int(num_out_rows)
    g_rows = torch.empty((R, H), dtype=torch.bfloat16, device=dev) if g_rows is None \
        else _need(g_rows, "g_rows", torch.bfloat16, 2, dev)
    if probs is not None and g_probs is None:
        g_probs = torch.empty((T, K), dtype=torch.float32, device=dev)
    if probs is None:
        g_probs = None
    _opt(g_probs, "g_probs", torch.float32, 2, dev)
    with _on(dev):
        _check("mp_unpermute_bwd", lib.mp_unpermute_bwd(
            _ptr(g_y), _ptr(rows), _ptr(probs), _ptr(row_id_map), T, K, H, _ptr(g_rows),
            _ptr(g_probs), _stream(dev)))
    return g_rows, g_probs


def mp_zero_rows_from(buf, first_row):
    """Zeroes rows [first_row[0], buf.shape[0]) of a contiguous device tensor,
    the start read on the device (e.g. offsets[-1:] of mp_build_map: the
    rows of a permuted buffer no slot maps to).  Returns buf."""
    lib = _lib.load()
    if not isinstance(buf, torch.Tensor) or not buf.is_cuda or not buf.is_contiguous():
        raise TypeError("buf must be a contiguous CUDA tensor")
    dev = buf.device
    _need(first_row, "first_row", torch.int32, 1, dev)
    if first_row.numel() < 1:
        raise ValueError("first_row must hold at least one element")
    rows = buf.shape[0] if buf.dim() > 0 else 1
    row_bytes = (buf.numel() // rows if rows else 0) * buf.element_size()
    with _on(dev):
        _check("mp_zero_rows_from", lib.mp_zero_rows_from(
            _ptr(buf), rows, row_bytes, _ptr(first_row), _stream(dev)))
    return buf


# --------------------------------------------------------------------------
# chunk sort + pad, unpad + restore
# --------------------------------------------------------------------------

def _token_dtype(t, name):
    if not isinstance(t, torch.Tensor) or t.dtype not in DTYPES:
        raise TypeError(f"{name} must be a bf16, fp16 or fp32 tensor")
    return DTYPES[t.dtype]


def mp_sort_chunks_pad(x, split_sizes, chunk_order, num_groups: int, align: int,
                       out_rows: int, probs=None, *, padded_sizes=None, out=None,
                       out_probs=None, row_map=None, group_off=None, status=None):
    """x [N,H] (bf16, fp16 or fp32) -> (out [out_rows,H], out_probs or None,
    row_map int32 [out_rows], group_off int64 [G+1]).  padded_sizes (int32 [G])
    fixes each group's row count instead of rounding up to `align`."""
    lib = _lib.load()
    dt = _token_dtype(x, "x")
    _need(x, "x", x.dtype, 2)
    dev = x.device
    N, H = x.shape
    _need(split_sizes, "split_sizes", torch.int32, 1, dev)
    _need(chunk_order, "chunk_order", torch.int32, 1, dev)
    C, G = split_sizes.shape[0], int(num_groups)
    _shape(chunk_order, "chunk_order", (C,))
    if padded_sizes is not None:
        _need(padded_sizes, "padded_sizes", torch.int32, 1, dev)
        _shape(padded_sizes, "padded_sizes", (G,))
    _opt(probs, "probs", torch.float32, 1, dev)
    out = torch.empty((out_rows, H), dtype=x.dtype, device=dev) if out is None \
        else _need(out, "out", x.dtype, 2, dev)
    if probs is not None and out_probs is None:
        out_probs = torch.empty(out_rows, dtype=torch.float32, device=dev)
    if probs is None:
        out_probs = None
    row_map = torch.empty(out_rows, dtype=torch.int32, device=dev) if row_map is None \
        else _need(row_map, "row_map", torch.int32, 1, dev)
    group_off = torch.empty(G + 1, dtype=torch.int64, device=dev) if group_off is None \
        else _need(group_off, "group_off", torch.int64, 1, dev)
    _opt(status, "status", torch.int32, 1, dev)
    with _on(dev):
        if dt == 0 and padded_sizes is None:
            code = lib.mp_sort_chunks_pad(
                _ptr(x), _ptr(probs), _ptr(split_sizes), _ptr(chunk_order), C, G, int(align), N,
                int(out_rows), H, _ptr(out), _ptr(out_probs), _ptr(row_map), _ptr(group_off),
                _ptr(status), _stream(dev))
        else:
            code = lib.mp_sort_chunks_pad_ex(
                _ptr(x), dt, _ptr(probs), _ptr(split_sizes), _ptr(chunk_order),
                _ptr(padded_sizes), C, G, int(align), N, int(out_rows), H, _ptr(out),
                _ptr(out_probs), _ptr(row_map), _ptr(group_off), _ptr(status), _stream(dev))
        _check("mp_sort_chunks_pad", code)
    return out, out_probs, row_map, group_off


def _remap(name, src, row_map, n_rows, src_probs, out, out_probs, status, gather):
    lib = _lib.load()
    dt = _token_dtype(src, "input")
    _need(src, "input", src.dtype, 2)
    dev = src.device
    _need(row_map, "row_map", torch.int32, 1, dev)
    H = src.shape[1]
    rows_out = row_map.shape[0] if gather else n_rows
    out = torch.empty((rows_out, H), dtype=src.dtype, device=dev) if out is None \
        else _need(out, "out", src.dtype, 2, dev)
    _opt(src_probs, "probs", torch.float32, 1, dev)
    if src_probs is not None and out_probs is None:
        out_probs = torch.empty(rows_out, dtype=torch.float32, device=dev)
    if src_probs is None:
        out_probs = None
    _opt(status, "status", torch.int32, 1, dev)
    with _on(dev):
        if dt == 0:
            code = getattr(lib, name)(
                _ptr(src), _ptr(src_probs), _ptr(row_map), row_map.shape[0], int(n_rows), H,
                _ptr(out), _ptr(out_probs), _ptr(status), _stream(dev))
        else:
            code = getattr(lib, name + "_ex")(
                _ptr(src), dt, _ptr(src_probs), _ptr(row_map), row_map.shape[0], int(n_rows), H,
                _ptr(out), _ptr(out_probs), _ptr(status), _stream(dev))
        _check(name, code)
    return out, out_probs


def mp_unpad_restore(padded, row_map, num_rows: int, padded_probs=None, *, y=None,
                     y_probs=None, status=None):
    """padded [out_rows,H] -> (y [num_rows,H], y_probs or None).  Rows of y that
    row_map never names are not written (pass `y` to keep their contents)."""
    return _remap("mp_unpad_restore", padded, row_map, num_rows, padded_probs, y, y_probs,
                  status, gather=False)


def mp_sort_chunks_pad_bwd(g_out, row_map, num_rows: int, g_out_probs=None, *, g_x=None,
                           g_probs=None, status=None):
    return _remap("mp_sort_chunks_pad_bwd", g_out, row_map, num_rows, g_out_probs, g_x,
                  g_probs, status, gather=False)


def mp_unpad_restore_bwd(g_y, row_map, g_y_probs=None, *, g_padded=None, g_padded_probs=None,
                         status=None):
    return _remap("mp_unpad_restore_bwd", g_y, row_map, g_y.shape[0], g_y_probs, g_padded,
                  g_padded_probs, status, gather=True)
