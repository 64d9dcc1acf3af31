"""The library allocates no device memory: the boundary's ownership rule.

Every entry point is called with every output, workspace and status word
supplied by the caller, first once (which loads the library's kernels and its
static device data), then again on the same buffers.  Across the second round
neither the driver's free device memory nor torch's allocated bytes may
change: a cudaMalloc inside the library would take at least one 2 MiB page
from the free memory, and the binding is not allowed to allocate an output it
was given.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import workloads as wl
from tests.gpu_util import DEV, d, status_word

pytestmark = pytest.mark.gpu


def _all_calls():
    w = wl.routed("mid", T=1500)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    R = T * K
    idx, probs, x, gy = d(w["idx"]), d(w["probs"]), d(w["x"]), d(w["g_y"])
    st = status_word()
    rim = torch.empty((T, K), dtype=torch.int32, device=DEV)
    s2f = torch.empty(R, dtype=torch.int32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(mp.mp_build_map_workspace_size(T, K, E), dtype=torch.uint8, device=DEV)
    rows = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    rows_p = torch.empty(R, dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    g_rows = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    g_probs = torch.empty((T, K), dtype=torch.float32, device=DEV)
    g_x = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    g_xp = torch.empty((T, K), dtype=torch.float32, device=DEV)
    logits = d(wl.router_logits("mid", T=T))
    r_idx = torch.empty_like(idx)
    r_probs = torch.empty_like(probs)
    g_logits = torch.empty_like(logits)
    start = torch.tensor([R // 2], dtype=torch.int32, device=DEV)

    c = wl.chunks(3000, H=512)
    G, align = c["G"], c["align"]
    N = c["N"]
    out_rows = wl.padded_rows_bound(N, G, align)
    cx, cp = d(c["x"]), d(c["probs"])
    sz, od = d(c["split_sizes"]), d(c["chunk_order"])
    cout = torch.empty((out_rows, 512), dtype=torch.bfloat16, device=DEV)
    cout_p = torch.empty(out_rows, dtype=torch.float32, device=DEV)
    row_map = torch.empty(out_rows, dtype=torch.int32, device=DEV)
    goff = torch.empty(G + 1, dtype=torch.int64, device=DEV)
    cy = torch.empty((N, 512), dtype=torch.bfloat16, device=DEV)
    cy_p = torch.empty(N, dtype=torch.float32, device=DEV)
    cgx = torch.empty((N, 512), dtype=torch.bfloat16, device=DEV)
    cgx_p = torch.empty(N, dtype=torch.float32, device=DEV)
    cgp = torch.empty((out_rows, 512), dtype=torch.bfloat16, device=DEV)
    cgp_p = torch.empty(out_rows, dtype=torch.float32, device=DEV)

    def run():
        mp.mp_topk_softmax(logits, K, idx=r_idx, probs=r_probs)
        mp.mp_topk_softmax_bwd(probs, r_probs, r_idx, E, g_logits=g_logits)
        mp.mp_build_map(idx, E, row_id_map=rim, sorted_to_flat=s2f, counts=counts,
                        offsets=offsets, workspace=ws, status=st)
        mp.mp_build_map_capacity(idx, E, R // E, row_id_map=rim, sorted_to_flat=s2f,
                                 counts=counts, offsets=offsets, workspace=ws, status=st)
        mp.mp_build_map(idx, E, row_id_map=rim, sorted_to_flat=s2f, counts=counts,
                        offsets=offsets, workspace=ws, status=st)
        mp.mp_permute(x, rim, probs, out=rows, out_probs=rows_p)
        mp.mp_zero_rows_from(rows, start)
        mp.mp_unpermute(rows, rim, probs, out=y)
        mp.mp_unpermute_ep(rows, rim, idx, E, 8, probs, bf16_partials=True,
                           fp64_cross_rank=True, out=y)
        mp.mp_unpermute_bwd(gy, rim, rows, probs, g_rows=g_rows, g_probs=g_probs)
        mp.mp_permute_bwd(g_rows, rim, rows_p, g_x=g_x, g_probs=g_xp)
        mp.mp_sort_chunks_pad(cx, sz, od, G, align, out_rows, cp, out=cout, out_probs=cout_p,
                              row_map=row_map, group_off=goff, status=st)
        mp.mp_unpad_restore(cout, row_map, N, cout_p, y=cy, y_probs=cy_p, status=st)
        mp.mp_sort_chunks_pad_bwd(cout, row_map, N, cout_p, g_x=cgx, g_probs=cgx_p, status=st)
        mp.mp_unpad_restore_bwd(cy, row_map, cy_p, g_padded=cgp, g_padded_probs=cgp_p,
                                status=st)
    return run


def test_entry_points_allocate_no_device_memory():
    run = _all_calls()
    run()                                   # loads the kernels and the static data
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(DEV)
    used0 = torch.cuda.memory_allocated(DEV)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(DEV)
    used1 = torch.cuda.memory_allocated(DEV)
    assert used1 == used0
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
