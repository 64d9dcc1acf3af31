"""Seeded random shapes through every op, against the oracle.

Each case draws T, K, E, H, the fraction of empty slots, duplicate experts
per token and a pointer offset (so both the 16-byte vector path and the
element path run), then checks the map, permute, unpermute (with and
without probs), both backwards, the EP combine (every mode, K <= 16), the
router and the chunk sort+pad roundtrip: bit-exact, except the probability
gradient (fp32 summation bound against the oracle's fp64 sum) and the router
probabilities (a few ulps: two expf implementations)."""
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


def _offset(a, elems):
    """A CUDA copy of a that starts `elems` elements past a 16-byte boundary."""
    t = d(a)
    if elems == 0:
        return t
    base = torch.empty(t.numel() + elems, dtype=t.dtype, device=DEV)
    v = base[elems:].view(t.shape)
    v.copy_(t)
    return v


def _routed_case(rng):
    T = int(rng.integers(1, 700))
    K = int(rng.choice([1, 2, 3, 4, 6, 8, 16]))
    E = int(rng.choice([1, 3, 8, 64, 257, 1024]))
    H = int(rng.choice([8, 24, 40, 64, 128, 136, 1000, 1023, 2048]))
    idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    idx[rng.random((T, K)) < rng.choice([0.0, 0.1, 0.5])] = -1
    probs = rng.random((T, K)).astype(np.float32) + np.float32(1e-3)
    x = wl.random_rows(T, H, int(rng.integers(1 << 30)))
    rows = wl.random_rows(T * K, H, int(rng.integers(1 << 30)))
    gy = wl.random_rows(T, H, int(rng.integers(1 << 30)))
    off = int(rng.choice([0, 0, 1, 3])) if H % 8 == 0 else 0
    return T, K, E, H, idx, probs, x, rows, gy, off


@pytest.mark.parametrize("seed", range(24))
def test_routed_ops_fuzz(seed):
    rng = np.random.default_rng(9000 + seed)
    _check_routed(rng, *_routed_case(rng))


# K across the slot batches of the register row kernels (2, 4, 6 and 8
# slots, two batches past 8), on rows that take one pass per CTA (2,048), a
# ragged second pass (1,032) and the element path (1,001)
@pytest.mark.parametrize("K", [2, 3, 5, 6, 7, 9, 14])
@pytest.mark.parametrize("H", [2048, 1032, 1001])
def test_routed_ops_across_slot_batches(K, H):
    rng = np.random.default_rng(K * 10007 + H)
    T, E = 300, 64
    idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    idx[rng.random((T, K)) < 0.1] = -1
    probs = rng.random((T, K)).astype(np.float32) + np.float32(1e-3)
    x = wl.random_rows(T, H, K + 1)
    rows = wl.random_rows(T * K, H, K + 2)
    gy = wl.random_rows(T, H, K + 3)
    _check_routed(rng, T, K, E, H, idx, probs, x, rows, gy, 0)


# The permute's vector widths on wide rows: 32-byte vectors (H = 4,096 from a
# 32-byte aligned base), 16-byte ones when the base is only 16-byte aligned
# (offset by 8 elements) or the vector count is odd (H = 4,104)
@pytest.mark.parametrize("H,off", [(4096, 0), (4096, 8), (4104, 0), (7168, 0)])
def test_routed_ops_wide_rows_vector_widths(H, off):
    rng = np.random.default_rng(H + off)
    T, K, E = 200, 8, 128
    idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    idx[rng.random((T, K)) < 0.1] = -1
    probs = rng.random((T, K)).astype(np.float32) + np.float32(1e-3)
    x = wl.random_rows(T, H, 11)
    rows = wl.random_rows(T * K, H, 12)
    gy = wl.random_rows(T, H, 13)
    _check_routed(rng, T, K, E, H, idx, probs, x, rows, gy, off)


def _check_routed(rng, T, K, E, H, idx, probs, x, rows, gy, off):
    o_rim, o_s2f, o_counts, o_offsets, _ = oracle.build_map(idx, E)
    rim, s2f, counts, offsets = mp.mp_build_map(d(idx), E)
    for got, want in ((rim, o_rim), (s2f, o_s2f), (counts, o_counts), (offsets, o_offsets)):
        np.testing.assert_array_equal(h(got), want)
    mapped = np.sort(o_rim[o_rim >= 0])
    dp = d(probs)

    out, out_p = mp.mp_permute(_offset(x, off), rim, dp)
    o_out, o_out_p = oracle.permute(x, probs, o_rim)
    np.testing.assert_array_equal(h(out)[mapped], o_out[mapped])
    np.testing.assert_array_equal(h(out_p)[mapped], o_out_p[mapped])

    drows = _offset(rows, off)
    for p in (probs, None):
        y = mp.mp_unpermute(drows, rim, None if p is None else d(p))
        np.testing.assert_array_equal(h(y), oracle.unpermute(rows, p, o_rim, T, H))

    g_out_p = rng.standard_normal(T * K).astype(np.float32)
    g_x, g_p = mp.mp_permute_bwd(drows, rim, d(g_out_p))
    o_gx, o_gp = oracle.permute_bwd(rows, g_out_p, o_rim, T, H)
    np.testing.assert_array_equal(h(g_x), o_gx)
    np.testing.assert_array_equal(h(g_p), o_gp)

    g_rows, g_probs = mp.mp_unpermute_bwd(_offset(gy, off), rim, drows, dp)
    o_grows, o_gprobs = oracle.unpermute_bwd(gy, rows, probs, o_rim)
    np.testing.assert_array_equal(h(g_rows)[mapped], o_grows[mapped])
    gp = h(g_probs).astype(np.float64)
    bound = gprobs_bound(_f32(rows)[np.maximum(o_rim, 0)], _f32(gy)[:, None, :], o_gprobs)
    assert np.all(np.abs(gp - o_gprobs) <= bound)

    if K <= 16:
        ep = int(rng.choice([r for r in (1, 2, 4, 8) if E % r == 0]))
        for bf16p, fp64 in ((False, False), (True, False), (False, True), (True, True)):
            got = mp.mp_unpermute_ep(drows, rim, d(idx), E, ep, dp, bf16_partials=bf16p,
                                     fp64_cross_rank=fp64)
            want = oracle.unpermute_ep(rows, probs, o_rim, idx, T, H, E, ep, bf16p, fp64)
            np.testing.assert_array_equal(h(got), want)


@pytest.mark.parametrize("seed", range(12))
def test_router_fuzz(seed):
    rng = np.random.default_rng(9500 + seed)
    T = int(rng.integers(1, 3000))
    G = int(rng.choice([1, 2, 4, 8, 16, 32]))
    per = int(rng.choice([1, 2, 3, 8, 32]))
    E = G * per
    if E > 1024:
        E, per = G * (1024 // G), 1024 // G
    TG = int(rng.integers(1, G + 1))
    K = int(rng.integers(1, min(32, TG * per) + 1))
    logits = (rng.standard_normal((T, E)) * rng.choice([0.1, 1.0, 30.0])).astype(np.float32)
    if rng.random() < 0.3:
        logits = np.round(logits).astype(np.float32)        # ties
    idx, probs = mp.mp_topk_softmax(d(logits), K, n_groups=G, topk_groups=TG)
    o_idx, o_probs = oracle.topk_softmax(logits, K, G, TG)
    np.testing.assert_array_equal(h(idx), o_idx)
    got = h(probs)
    assert np.all(np.abs(got - o_probs) <= 8 * np.spacing(np.abs(o_probs).astype(np.float32)))
    g = rng.standard_normal((T, K)).astype(np.float32)
    gl = mp.mp_topk_softmax_bwd(d(g), probs, idx, E)
    np.testing.assert_array_equal(h(gl), oracle.topk_softmax_bwd(g, got, o_idx, E))


@pytest.mark.parametrize("seed", range(12))
def test_sort_pad_fuzz(seed):
    rng = np.random.default_rng(9800 + seed)
    G = int(rng.choice([1, 2, 4, 16, 32]))
    R = int(rng.choice([1, 2, 5, 8, 16]))
    C = G * R
    H = int(rng.choice([8, 24, 37, 256, 2048]))
    align = int(rng.choice([1, 2, 8, 64, 128]))
    sizes = rng.integers(0, int(rng.choice([3, 40, 300])), size=C).astype(np.int32)
    sizes[rng.random(C) < 0.3] = 0
    order = rng.permutation(C).astype(np.int32)
    N = int(sizes.sum())
    extra = int(rng.integers(0, 50))
    out_rows = N + G * (align - 1) + extra
    x = wl.random_rows(max(N, 1), H, seed)[:N]
    probs = rng.random(N).astype(np.float32)
    dx = d(x) if N else torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    dpr = d(probs) if N else torch.empty(0, dtype=torch.float32, device=DEV)
    out, out_p, row_map, goff = mp.mp_sort_chunks_pad(dx, d(sizes), d(order), G, align,
                                                      out_rows, dpr)
    o_out, o_out_p, o_map, o_goff, _ = oracle.sort_chunks_pad(x, probs, sizes, order, G,
                                                              align, out_rows)
    np.testing.assert_array_equal(h(out), o_out)
    np.testing.assert_array_equal(h(out_p), o_out_p)
    np.testing.assert_array_equal(h(row_map), o_map)
    np.testing.assert_array_equal(h(goff), o_goff)
    if N:
        y, y_p = mp.mp_unpad_restore(out, row_map, N, out_p)
        np.testing.assert_array_equal(h(y), x)
        np.testing.assert_array_equal(h(y_p), probs)
