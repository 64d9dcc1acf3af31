"""Back-to-back library calls on one stream with no synchronisation between
them, against the oracle.

Every kernel of the library is a programmatic dependent launch: it may be
scheduled while the kernel before it is still running and waits on the
device before its first read.  The map's rank kernel reads idx even before
that wait (the count kernel in front of it waited for idx's writer).  These
tests run whole chains with every buffer reused across iterations, so a read
that overtook its writer (router -> map -> permute -> unpermute -> backward),
or a write that overtook the previous iteration's reader, changes a result.
Each map form runs: one launch (<= 4,096 routes), count + rank, and count +
scan + rank (E = 1,024 over 64 tiles).  Only the per-iteration outputs are
distinct buffers; everything is checked after one synchronisation at the end."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import workloads as wl
from tests.gpu_util import DEV, d, gprobs_bound, h

pytestmark = pytest.mark.gpu


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("T,E,K,H", [(256, 64, 8, 128),       # single-launch map
                                     (2048, 128, 8, 256),     # count + rank
                                     (16384, 1024, 8, 64)])   # count + scan + rank
def test_routed_chain_without_sync(T, E, K, H):
    iters = 4
    rng = np.random.default_rng(T + E)
    logits = [(rng.standard_normal((T, E)) * 2).astype(np.float32) for _ in range(iters)]
    x = [wl.random_rows(T, H, 100 + i) for i in range(iters)]
    gy = [wl.random_rows(T, H, 200 + i) for i in range(iters)]
    d_logits, d_x, d_gy = [d(a) for a in logits], [d(a) for a in x], [d(a) for a in gy]

    # shared buffers, reused by every iteration
    rim = torch.empty((T, K), dtype=torch.int32, device=DEV)
    s2f = torch.empty(T * K, dtype=torch.int32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(mp.mp_build_map_workspace_size(T, K, E), dtype=torch.uint8, device=DEV)
    rows = torch.empty((T * K, H), dtype=torch.bfloat16, device=DEV)
    rows_p = torch.empty(T * K, dtype=torch.float32, device=DEV)
    g_rows = torch.empty((T * K, H), dtype=torch.bfloat16, device=DEV)
    # per-iteration results
    idx = [torch.empty((T, K), dtype=torch.int32, device=DEV) for _ in range(iters)]
    probs = [torch.empty((T, K), dtype=torch.float32, device=DEV) for _ in range(iters)]
    y = [torch.empty((T, H), dtype=torch.bfloat16, device=DEV) for _ in range(iters)]
    y_ep = [torch.empty((T, H), dtype=torch.bfloat16, device=DEV) for _ in range(iters)]
    g_probs = [torch.empty((T, K), dtype=torch.float32, device=DEV) for _ in range(iters)]
    g_x = [torch.empty((T, H), dtype=torch.bfloat16, device=DEV) for _ in range(iters)]

    torch.cuda.synchronize()
    for i in range(iters):
        mp.mp_topk_softmax(d_logits[i], K, idx=idx[i], probs=probs[i])
        mp.mp_build_map(idx[i], E, row_id_map=rim, sorted_to_flat=s2f, counts=counts,
                        offsets=offsets, workspace=ws)
        mp.mp_permute(d_x[i], rim, probs[i], out=rows, out_probs=rows_p)
        mp.mp_unpermute(rows, rim, probs[i], out=y[i])
        mp.mp_unpermute_ep(rows, rim, idx[i], E, 8, probs[i], out=y_ep[i])
        mp.mp_unpermute_bwd(d_gy[i], rim, rows, probs[i], g_rows=g_rows, g_probs=g_probs[i])
        mp.mp_permute_bwd(g_rows, rim, g_x=g_x[i])
        # every route is kept, so nothing is zeroed; the rows stay for the check
        mp.mp_zero_rows_from(rows, offsets[-1:])
    torch.cuda.synchronize()

    for i in range(iters):
        o_idx, _ = oracle.topk_softmax(logits[i], K)
        np.testing.assert_array_equal(h(idx[i]), o_idx)
        p = h(probs[i])
        o_rim, *_ = oracle.build_map(o_idx, E)
        o_rows, _ = oracle.permute(x[i], p, o_rim)
        np.testing.assert_array_equal(h(y[i]), oracle.unpermute(o_rows, p, o_rim, T, H))
        np.testing.assert_array_equal(
            h(y_ep[i]), oracle.unpermute_ep(o_rows, p, o_rim, o_idx, T, H, E, 8, False, False))
        o_grows, o_gprobs = oracle.unpermute_bwd(gy[i], o_rows, p, o_rim)
        o_gx, _ = oracle.permute_bwd(o_grows, None, o_rim, T, H)
        np.testing.assert_array_equal(h(g_x[i]), o_gx)
        gp = h(g_probs[i]).astype(np.float64)
        bound = gprobs_bound(_f32(o_rows)[o_rim], _f32(gy[i])[:, None, :], o_gprobs)
        assert np.all(np.abs(gp - o_gprobs) <= bound)
    # the last iteration's permuted rows are still in the shared buffer
    o_rim, *_ = oracle.build_map(h(idx[-1]), E)
    o_rows, _ = oracle.permute(x[-1], h(probs[-1]), o_rim)
    np.testing.assert_array_equal(h(rows), o_rows)


def test_chunk_chain_without_sync():
    """sort+pad -> unpad+restore -> the same pair again on the restored rows,
    four times over shared padded buffers, with new split sizes each time."""
    iters, G, R, H, align = 4, 8, 4, 512, 16
    C = G * R
    rng = np.random.default_rng(77)
    cases = []
    for i in range(iters):
        sizes = rng.integers(0, 300, size=C).astype(np.int32)
        order = rng.permutation(C).astype(np.int32)
        N = int(sizes.sum())
        x = wl.random_rows(N, H, 300 + i)
        pr = rng.random(N).astype(np.float32)
        cases.append((sizes, order, N, x, pr))
    out_rows = max(c[2] for c in cases) + G * (align - 1)
    out = torch.empty((out_rows, H), dtype=torch.bfloat16, device=DEV)
    out_p = torch.empty(out_rows, dtype=torch.float32, device=DEV)
    row_map = torch.empty(out_rows, dtype=torch.int32, device=DEV)
    goff = torch.empty(G + 1, dtype=torch.int64, device=DEV)
    mid = torch.empty((max(c[2] for c in cases), H), dtype=torch.bfloat16, device=DEV)
    mid_p = torch.empty(mid.shape[0], dtype=torch.float32, device=DEV)
    dev_in = [(d(c[0]), d(c[1]), d(c[3]), d(c[4])) for c in cases]
    ys = [torch.empty((c[2], H), dtype=torch.bfloat16, device=DEV) for c in cases]
    yps = [torch.empty(c[2], dtype=torch.float32, device=DEV) for c in cases]
    outs = [torch.empty((out_rows, H), dtype=torch.bfloat16, device=DEV) for _ in cases]
    torch.cuda.synchronize()
    for i, (sizes, order, N, x, pr) in enumerate(cases):
        ds, do, dx, dp = dev_in[i]
        mp.mp_sort_chunks_pad(dx, ds, do, G, align, out_rows, dp, out=out, out_probs=out_p,
                              row_map=row_map, group_off=goff)
        mp.mp_unpad_restore(out, row_map, N, out_p, y=mid[:N], y_probs=mid_p[:N])
        mp.mp_sort_chunks_pad(mid[:N], ds, do, G, align, out_rows, mid_p[:N], out=outs[i],
                              out_probs=out_p, row_map=row_map, group_off=goff)
        mp.mp_unpad_restore(outs[i], row_map, N, out_p, y=ys[i], y_probs=yps[i])
    torch.cuda.synchronize()
    for i, (sizes, order, N, x, pr) in enumerate(cases):
        o_out, _, _, _, _ = oracle.sort_chunks_pad(x, pr, sizes, order, G, align, out_rows)
        np.testing.assert_array_equal(h(outs[i]), o_out)
        np.testing.assert_array_equal(h(ys[i]), x)
        np.testing.assert_array_equal(h(yps[i]), pr)
