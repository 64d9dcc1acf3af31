"""Differentiable forms of the dispatch / combine path for a training step.

Each function is a ``torch.autograd.Function`` whose forward and backward are
calls of the C-ABI binding (every value is computed by the library's CUDA
kernels).  The operations and their gradients are those of the pages:
``moe_permute_with_probs`` / ``moe_unpermute_mask`` ("d9d 0.1.0 —
d9d/kernel/moe/permute_with_probs.py"), the batch-invariant ``unpermute`` and
its rank-partial form ("core.transformer.moe.batch_invariant"), the fused
chunk sort + pad and its restore ("[PyTorch] Fuse MoE chunk sorting and
padding"), and the top-K softmax router ("moe-ops 0.1.0", Operators).

    idx, probs = topk_softmax(logits, 8)
    rows, rows_probs, d = permute(x, idx, num_experts, probs)
    ...  expert computation on rows (d.routed_rows() rows are routed)  ...
    y = unpermute(expert_out, d, probs)

Rows of the permuted buffer past the routed count (empty slots, routes
dropped by a capacity) are zero in the forward output and get zero gradient,
so a computation over the whole buffer stays finite.  Rows of a restored
tensor that no chunk names (past the sum of the split sizes) are zero too.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (mp_build_map, mp_build_map_capacity, mp_permute, mp_permute_bwd,
               mp_sort_chunks_pad, mp_sort_chunks_pad_bwd, mp_topk_softmax,
               mp_topk_softmax_bwd, mp_unpad_restore, mp_unpad_restore_bwd, mp_unpermute,
               mp_unpermute_bwd, mp_unpermute_ep, mp_zero_rows_from)

__all__ = ["Dispatch", "topk_softmax", "permute", "unpermute", "unpermute_ep",
           "sort_chunks_pad", "unpad_restore"]


@dataclass
class Dispatch:
    """The routing map of one batch.

    row_id_map [T,K]: the permuted row of slot (t,k), -1 if none;
    sorted_to_flat [rows]: the slot t*K+k of each routed row;
    counts [E] / offsets [E+1]: rows per expert and where each expert's rows
    start (offsets[E] = routed rows); idx [T,K]: the experts; num_rows: rows
    of the permuted buffer."""

    row_id_map: torch.Tensor
    sorted_to_flat: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    idx: torch.Tensor
    num_experts: int
    num_rows: int

    def routed_rows(self) -> torch.Tensor:
        """The routed row count, a one-element device tensor."""
        return self.offsets[-1:]


class _Permute(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, probs, row_id_map, routed, num_rows):
        out, out_probs = mp_permute(x, row_id_map, probs, num_out_rows=num_rows)
        mp_zero_rows_from(out, routed)
        if out_probs is not None:
            mp_zero_rows_from(out_probs, routed)
        ctx.save_for_backward(row_id_map)
        ctx.has_probs = probs is not None
        return out, out_probs

    @staticmethod
    def backward(ctx, g_out, g_out_probs):
        (row_id_map,) = ctx.saved_tensors
        gp = None
        if ctx.has_probs and ctx.needs_input_grad[1]:
            gp = torch.zeros(g_out.shape[0], dtype=torch.float32, device=g_out.device) \
                if g_out_probs is None else g_out_probs.contiguous()
        g_x, g_probs = mp_permute_bwd(g_out.contiguous(), row_id_map, gp)
        return g_x, g_probs, None, None, None


class _Unpermute(torch.autograd.Function):
    @staticmethod
    def forward(ctx, rows, probs, row_id_map, routed, ep):
        if ep is None:
            y = mp_unpermute(rows, row_id_map, probs)
        else:
            idx, E, ep_size, bf16p, fp64 = ep
            y = mp_unpermute_ep(rows, row_id_map, idx, E, ep_size, probs, bf16_partials=bf16p,
                                fp64_cross_rank=fp64)
        ctx.save_for_backward(rows if probs is not None else None, probs, row_id_map, routed)
        ctx.num_rows = rows.shape[0]
        return y

    @staticmethod
    def backward(ctx, g_y):
        rows, probs, row_id_map, routed = ctx.saved_tensors
        g_rows, g_probs = mp_unpermute_bwd(g_y.contiguous(), row_id_map, rows, probs,
                                           num_out_rows=ctx.num_rows)
        mp_zero_rows_from(g_rows, routed)
        return g_rows, g_probs, None, None, None


class _TopkSoftmax(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, topk, n_groups, topk_groups):
        idx, probs = mp_topk_softmax(logits, topk, n_groups=n_groups, topk_groups=topk_groups)
        ctx.mark_non_differentiable(idx)
        ctx.save_for_backward(probs, idx)
        ctx.num_experts = logits.shape[1]
        return idx, probs

    @staticmethod
    def backward(ctx, g_idx, g_probs):
        probs, idx = ctx.saved_tensors
        g = mp_topk_softmax_bwd(g_probs.contiguous(), probs, idx, ctx.num_experts)
        return g, None, None, None


class _SortChunksPad(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, probs, split_sizes, chunk_order, num_groups, align, out_rows,
                padded_sizes):
        out, out_probs, row_map, group_off = mp_sort_chunks_pad(
            x, split_sizes, chunk_order, num_groups, align, out_rows, probs,
            padded_sizes=padded_sizes)
        ctx.mark_non_differentiable(row_map, group_off)
        ctx.save_for_backward(row_map)
        ctx.num_rows = x.shape[0]
        ctx.has_probs = probs is not None
        return out, out_probs, row_map, group_off

    @staticmethod
    def backward(ctx, g_out, g_out_probs, g_row_map, g_group_off):
        (row_map,) = ctx.saved_tensors
        g_x = torch.zeros((ctx.num_rows, g_out.shape[1]), dtype=g_out.dtype,
                          device=g_out.device)
        gp = g_pr = None
        if ctx.has_probs and ctx.needs_input_grad[1]:
            gp = torch.zeros(g_out.shape[0], dtype=torch.float32, device=g_out.device) \
                if g_out_probs is None else g_out_probs.contiguous()
            g_pr = torch.zeros(ctx.num_rows, dtype=torch.float32, device=g_out.device)
        mp_sort_chunks_pad_bwd(g_out.contiguous(), row_map, ctx.num_rows, gp, g_x=g_x,
                               g_probs=g_pr)
        return g_x, g_pr, None, None, None, None, None, None


class _UnpadRestore(torch.autograd.Function):
    @staticmethod
    def forward(ctx, padded, padded_probs, row_map, num_rows):
        y = torch.zeros((num_rows, padded.shape[1]), dtype=padded.dtype, device=padded.device)
        y_probs = None if padded_probs is None else \
            torch.zeros(num_rows, dtype=torch.float32, device=padded.device)
        mp_unpad_restore(padded, row_map, num_rows, padded_probs, y=y, y_probs=y_probs)
        ctx.save_for_backward(row_map)
        ctx.has_probs = padded_probs is not None
        return y, y_probs

    @staticmethod
    def backward(ctx, g_y, g_y_probs):
        (row_map,) = ctx.saved_tensors
        gp = None
        if ctx.has_probs and ctx.needs_input_grad[1]:
            gp = torch.zeros(g_y.shape[0], dtype=torch.float32, device=g_y.device) \
                if g_y_probs is None else g_y_probs.contiguous()
        g_padded, g_padded_probs = mp_unpad_restore_bwd(g_y.contiguous(), row_map, gp)
        return g_padded, g_padded_probs, None, None


def topk_softmax(logits: torch.Tensor, topk: int, n_groups: int = 1, topk_groups: int = 1):
    """fp32 logits [T,E] -> (idx int32 [T,K], probs fp32 [T,K]); probs is
    differentiable w.r.t. the logits (softmax over the K picks)."""
    return _TopkSoftmax.apply(logits, int(topk), int(n_groups), int(topk_groups))


def permute(x: torch.Tensor, idx: torch.Tensor, num_experts: int, probs=None, *,
            capacity: int | None = None):
    """bf16 x [T,H], int32 idx [T,K] (-1 = empty slot) -> (rows bf16 [R,H],
    rows_probs fp32 [R] or None, Dispatch).  R = T*K, or min(T*K, E*capacity)
    when each expert keeps at most `capacity` routes (the earliest)."""
    T, K = idx.shape
    if capacity is None:
        rim, s2f, counts, offsets = mp_build_map(idx, num_experts)
        R = T * K
    else:
        rim, s2f, counts, offsets = mp_build_map_capacity(idx, num_experts, capacity)
        R = min(T * K, num_experts * int(capacity))
    d = Dispatch(rim, s2f, counts, offsets, idx, int(num_experts), R)
    rows, rows_probs = _Permute.apply(x, probs, rim, d.routed_rows(), R)
    return rows, rows_probs, d


def unpermute(rows: torch.Tensor, dispatch: Dispatch, probs=None) -> torch.Tensor:
    """bf16 rows [R,H] -> y bf16 [T,H]: slot-order fp32 fused multiply-adds
    (plain adds without probs), one bf16 rounding."""
    return _Unpermute.apply(rows, probs, dispatch.row_id_map, dispatch.routed_rows(), None)


def unpermute_ep(rows: torch.Tensor, dispatch: Dispatch, ep_size: int, probs=None, *,
                 bf16_partials: bool = False, fp64_cross_rank: bool = False) -> torch.Tensor:
    """unpermute as a rank-ordered sum over `ep_size` expert-parallel ranks
    (per-rank partials, optionally bf16; cross-rank sum in fp32 or fp64).  The
    gradient is that of the plain combine: the summation tree changes the
    rounding, not the derivative."""
    ep = (dispatch.idx, dispatch.num_experts, int(ep_size), bool(bf16_partials),
          bool(fp64_cross_rank))
    return _Unpermute.apply(rows, probs, dispatch.row_id_map, dispatch.routed_rows(), ep)


def sort_chunks_pad(x: torch.Tensor, split_sizes: torch.Tensor, chunk_order: torch.Tensor,
                    num_groups: int, align: int, out_rows: int, probs=None, *,
                    padded_sizes=None):
    """Fused chunk sort + zero pad: (out [out_rows,H], out_probs or None,
    row_map int32 [out_rows], group_off int64 [G+1]).  The gradient of a
    padding row is dropped; rows of x that no chunk names get zero gradient."""
    return _SortChunksPad.apply(x, probs, split_sizes, chunk_order, int(num_groups), int(align),
                                int(out_rows), padded_sizes)


def unpad_restore(padded: torch.Tensor, row_map: torch.Tensor, num_rows: int,
                  padded_probs=None):
    """Inverse of sort_chunks_pad: (y [num_rows,H], y_probs or None); rows no
    chunk names are zero; padding rows get zero gradient."""
    return _UnpadRestore.apply(padded, padded_probs, row_map, int(num_rows))
