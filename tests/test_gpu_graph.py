"""CUDA-graph replay with changing routing at fixed buffer sizes: the grids
depend on shapes only and all metadata stays on the device."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import workloads as wl
from tests.gpu_util import DEV, d, h

pytestmark = pytest.mark.gpu


def test_routed_path_graph_replay():
    T, H, E, K = 2048, 256, 64, 6
    ws = [wl.routed("mid", T=T, H=H, seed=s) for s in (1, 2, 3)]
    idx = d(ws[0]["idx"]); probs = d(ws[0]["probs"]); x = d(ws[0]["x"]); gy = d(ws[0]["g_y"])
    rim = torch.empty((T, K), dtype=torch.int32, device=DEV)
    s2f = torch.empty(T * K, dtype=torch.int32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    wsp = torch.empty(mp.mp_build_map_workspace_size(T, K, E), dtype=torch.uint8, device=DEV)
    rows = torch.empty((T * K, H), dtype=torch.bfloat16, device=DEV)
    rows_p = torch.empty(T * K, dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    g_rows = torch.empty((T * K, H), dtype=torch.bfloat16, device=DEV)
    g_probs = torch.empty((T, K), dtype=torch.float32, device=DEV)
    g_x = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)

    def step():
        mp.mp_build_map(idx, E, row_id_map=rim, sorted_to_flat=s2f, counts=counts,
                        offsets=offsets, workspace=wsp)
        mp.mp_permute(x, rim, probs, out=rows, out_probs=rows_p)
        mp.mp_unpermute(rows, rim, probs, out=y)
        mp.mp_unpermute_bwd(gy, rim, rows, probs, g_rows=g_rows, g_probs=g_probs)
        mp.mp_permute_bwd(g_rows, rim, g_x=g_x)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                       # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()

    for w in ws[1:] + ws[:1]:
        idx.copy_(d(w["idx"])); probs.copy_(d(w["probs"]))
        x.copy_(d(w["x"])); gy.copy_(d(w["g_y"]))
        g.replay()
        torch.cuda.synchronize()
        o_rim, o_s2f, o_counts, o_offsets, _ = oracle.build_map(w["idx"], E)
        o_rows, _ = oracle.permute(w["x"], w["probs"], o_rim)
        np.testing.assert_array_equal(h(rim), o_rim)
        np.testing.assert_array_equal(h(offsets), o_offsets)
        np.testing.assert_array_equal(h(rows), o_rows)
        np.testing.assert_array_equal(h(y), oracle.unpermute(o_rows, w["probs"], o_rim, T, H))
        o_grows, _ = oracle.unpermute_bwd(w["g_y"], o_rows, w["probs"], o_rim)
        np.testing.assert_array_equal(h(g_rows), o_grows)
        o_gx, _ = oracle.permute_bwd(o_grows, None, o_rim, T, H)
        np.testing.assert_array_equal(h(g_x), o_gx)


@pytest.mark.parametrize("H", [128, 1024])      # flat copy (16 vectors) and warp per row
def test_sort_pad_graph_replay_with_new_sizes(H):
    N, G, align = 4096, 16, 128
    out_rows = wl.padded_rows_bound(N, G, align)
    layouts = [wl.chunk_layout(N, seed=s) for s in (10, 11, 12)]
    x_np = wl.random_rows(N, H, 4)
    x = d(x_np)
    sizes = d(layouts[0][0]); order = d(layouts[0][1])
    out = torch.empty((out_rows, H), dtype=torch.bfloat16, device=DEV)
    row_map = torch.empty(out_rows, dtype=torch.int32, device=DEV)
    goff = torch.empty(G + 1, dtype=torch.int64, device=DEV)
    y = torch.empty((N, H), dtype=torch.bfloat16, device=DEV)

    def step():
        mp.mp_sort_chunks_pad(x, sizes, order, G, align, out_rows, out=out, row_map=row_map,
                              group_off=goff)
        mp.mp_unpad_restore(out, row_map, N, y=y)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for sz, od in layouts[1:]:
        sizes.copy_(d(sz)); order.copy_(d(od))
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        o_out, _, o_map, o_goff, _ = oracle.sort_chunks_pad(x_np, None, sz, od, G, align,
                                                            out_rows)
        np.testing.assert_array_equal(h(row_map), o_map)
        np.testing.assert_array_equal(h(goff), o_goff)
        np.testing.assert_array_equal(h(out), o_out)
        np.testing.assert_array_equal(h(y), x_np)
