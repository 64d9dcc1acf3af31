"""Parity of the fused chunk sort+pad, unpad+restore and their backwards
(through the C ABI) with the oracle: bit-exact layouts, maps, offsets and
copies, status bits for bad metadata."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import workloads as wl
from tests.gpu_util import DEV, d, h, status_word

pytestmark = pytest.mark.gpu


def run_case(x, probs, sizes, order, G, align, out_rows, expect_flags=()):
    N = x.shape[0]
    st = status_word()
    out, out_p, row_map, goff = mp.mp_sort_chunks_pad(
        d(x), d(sizes), d(order), G, align, out_rows, d(probs) if probs is not None else None,
        status=st)
    o_out, o_out_p, o_map, o_goff, fl = oracle.sort_chunks_pad(x, probs, sizes, order, G,
                                                               align, out_rows)
    np.testing.assert_array_equal(h(row_map), o_map)
    np.testing.assert_array_equal(h(goff), o_goff)
    np.testing.assert_array_equal(h(out), o_out)
    if probs is not None:
        np.testing.assert_array_equal(h(out_p), o_out_p)
    want = {k for k, v in fl.items() if v}
    assert mp.status_bits(int(h(st)[0])) == want
    assert want == set(expect_flags)
    return out, out_p, row_map, o_map


@pytest.mark.parametrize("N", [8192, 32768])
@pytest.mark.parametrize("capacity", [False, True])
def test_sort_pad_roundtrip_workload(N, capacity):
    c = wl.chunks(N)
    G, align = c["G"], c["align"]
    exact_rows = int(sum(-(-int(s) // align) * align for s in
                         c["split_sizes"][c["chunk_order"]].reshape(G, -1).sum(1)))
    out_rows = wl.padded_rows_bound(N, G, align) if capacity else exact_rows
    out, out_p, row_map, o_map = run_case(c["x"], c["probs"], c["split_sizes"],
                                          c["chunk_order"], G, align, out_rows)
    # restore
    y, y_p = mp.mp_unpad_restore(out, row_map, N, out_p)
    np.testing.assert_array_equal(h(y), c["x"])
    np.testing.assert_array_equal(h(y_p), c["probs"])
    # backwards
    g_out = wl.random_rows(out_rows, c["H"], c["g_seed"])
    g_out_p = np.random.default_rng(c["g_seed"]).standard_normal(out_rows).astype(np.float32)
    g_x, g_xp = mp.mp_sort_chunks_pad_bwd(d(g_out), row_map, N, d(g_out_p))
    o_gx, o_gxp = oracle.sort_chunks_pad_bwd(g_out, g_out_p, o_map, N)
    np.testing.assert_array_equal(h(g_x), o_gx)
    np.testing.assert_array_equal(h(g_xp), o_gxp)
    g_y = wl.random_rows(N, c["H"], c["g_seed"] + 1)
    g_yp = np.random.default_rng(c["g_seed"] + 1).standard_normal(N).astype(np.float32)
    g_pad, g_padp = mp.mp_unpad_restore_bwd(d(g_y), row_map, d(g_yp))
    o_gpad, o_gpadp = oracle.unpad_restore_bwd(g_y, g_yp, o_map, N)
    np.testing.assert_array_equal(h(g_pad), o_gpad)
    np.testing.assert_array_equal(h(g_padp), o_gpadp)
    assert np.all(h(g_pad)[o_map < 0] == 0)


def _meta(seed, G, R, max_size=40, empty_group=False):
    rng = np.random.default_rng(seed)
    C = G * R
    sizes = rng.integers(0, max_size, size=C).astype(np.int32)
    sizes[rng.random(C) < 0.25] = 0
    order = rng.permutation(C).astype(np.int32)
    if empty_group:
        sizes[order[:R]] = 0
    return sizes, order


@pytest.mark.parametrize("G,R,align,H,empty_group,extra", [
    (16, 8, 128, 2048, True, 0),    # one warp per row, one unrolled pass
    (4, 3, 8, 37, False, 5),        # element path (37 units, warp per row), capacity tail
    (1, 1, 1, 64, False, 0),        # one chunk, no padding; rows of 8 vectors (flat copy)
    (32, 32, 16, 128, True, 100),   # C = MP_MAX_CHUNKS: metadata built by the whole CTA
    (32, 8, 16, 256, False, 0),     # C = 256: the largest metadata built by one warp
    (2, 129, 8, 256, True, 0),      # C = 258: the smallest built by the whole CTA
    (5, 2, 3, 24, False, 0),        # rows of 3 vectors (flat copy)
    (8, 4, 64, 512, True, 7),       # 64 vectors per row, a partial unrolled pass
    (4, 4, 16, 7168, False, 3),     # 896 vectors per row, several passes
    (2, 2, 4, 24576, True, 0),      # 3072 vectors per row
    (64, 2, 4, 2048, True, 9),      # G = 64 > 32 groups with C = 128: metadata by the whole CTA
    (48, 2, 8, 256, False, 3),      # the same for rows of 32 vectors (the per-CTA-rows kernel)
])
def test_sort_pad_edges(G, R, align, H, empty_group, extra):
    sizes, order = _meta(G * 100 + R, G, R, empty_group=empty_group)
    N = int(sizes.sum())
    x = wl.random_rows(N, H, 3)
    probs = np.random.default_rng(1).random(N).astype(np.float32)
    out_rows = N + G * (align - 1) + extra
    out, out_p, row_map, _ = run_case(x, probs, sizes, order, G, align, out_rows)
    y, y_p = mp.mp_unpad_restore(out, row_map, N, out_p)
    np.testing.assert_array_equal(h(y), x)
    np.testing.assert_array_equal(h(y_p), probs)
    # without probs
    out2, none, _, _ = mp.mp_sort_chunks_pad(d(x), d(sizes), d(order), G, align, out_rows)
    assert none is None
    np.testing.assert_array_equal(h(out2), h(out))


def test_sort_pad_many_chunks_large_output():
    """512 chunks (metadata built by the whole CTA) and more than 16,384 output
    rows (one row per warp in flight): the remaining kernel variant."""
    G, R, align, H = 16, 32, 8, 512
    sizes, order = _meta(512, G, R, max_size=120)
    N = int(sizes.sum())
    out_rows = N + G * (align - 1) + 11
    assert out_rows > 16384 and G * R > 256
    x = wl.random_rows(N, H, 4)
    probs = np.random.default_rng(5).random(N).astype(np.float32)
    out, out_p, row_map, _ = run_case(x, probs, sizes, order, G, align, out_rows)
    y, y_p = mp.mp_unpad_restore(out, row_map, N, out_p)
    np.testing.assert_array_equal(h(y), x)
    np.testing.assert_array_equal(h(y_p), probs)


@pytest.mark.parametrize("H,shift", [(512, 0), (512, 8), (520, 0)])
def test_sort_pad_large_output_vector_widths(H, shift):
    """Outputs of more than 16,384 rows copy 32-byte vectors when the tensors
    start on 32-byte boundaries and a row is an even number of 16-byte
    vectors (H = 512), else 16-byte ones: a base 8 elements (16 bytes) past
    the boundary, or rows of 65 16-byte vectors (H = 520)."""
    G, R, align = 16, 8, 8
    sizes, order = _meta(77 + H + shift, G, R, max_size=400)
    N = int(sizes.sum())
    out_rows = N + G * (align - 1) + 5
    assert out_rows > 16384
    x = wl.random_rows(N, H, 6)
    probs = np.random.default_rng(7).random(N).astype(np.float32)
    xb = torch.empty(N * H + shift, dtype=torch.bfloat16, device=DEV)
    dx = xb[shift:].view(N, H)
    dx.copy_(d(x))
    ob = torch.empty(out_rows * H + shift, dtype=torch.bfloat16, device=DEV)
    dout = ob[shift:].view(out_rows, H)
    out, out_p, row_map, _ = mp.mp_sort_chunks_pad(dx, d(sizes), d(order), G, align, out_rows,
                                                   d(probs), out=dout)
    o_out, o_out_p, o_map, _, _ = oracle.sort_chunks_pad(x, probs, sizes, order, G, align,
                                                         out_rows)
    np.testing.assert_array_equal(h(row_map), o_map)
    np.testing.assert_array_equal(h(out), o_out)
    np.testing.assert_array_equal(h(out_p), o_out_p)


def test_sort_pad_status_bits():
    x = wl.random_rows(64, 16, 5)
    p = np.arange(64, dtype=np.float32)
    run_case(x, p, np.array([10, -3, 12, 5], np.int32), np.array([0, 1, 2, 3], np.int32),
             2, 4, 48, expect_flags=("bad_split",))
    run_case(x, p, np.array([40, 40], np.int32), np.array([1, 0], np.int32), 1, 1, 90,
             expect_flags=("split_overflow",))
    run_case(x, p, np.array([30, 30], np.int32), np.array([0, 1], np.int32), 2, 8, 50,
             expect_flags=("rows_overflow",))
    run_case(x, p, np.array([3, 3, 3, 3], np.int32), np.array([0, 7, 2, 3], np.int32), 2, 2,
             16, expect_flags=("bad_order",))


@pytest.mark.parametrize("H", [2048, 64])
def test_sort_pad_order_naming_a_chunk_twice(H):
    """chunk_order need not be a permutation: a chunk named at two positions is
    copied to both, a chunk named nowhere is not copied, and an entry out of
    range names nothing (status bit).  Rows of 256 vectors go through the
    kernel that scatters input rows; rows of 8 through the one that gathers."""
    G, R, align = 4, 4, 8
    sizes, order = _meta(71, G, R, max_size=50)
    order = order.copy()
    order[5] = order[2]                 # named twice; the old order[5] named nowhere
    order[9] = 99                       # out of range
    N = int(sizes.sum()) + 7            # rows past the named ones are never read
    x = wl.random_rows(N, H, 8)
    probs = np.random.default_rng(3).random(N).astype(np.float32)
    out_rows = N + int(sizes[order[5]]) + G * (align - 1) + 4
    run_case(x, probs, sizes, order, G, align, out_rows, expect_flags=("bad_order",))


def test_restore_bad_row_sets_status():
    padded = d(wl.random_rows(8, 16, 1))
    row_map = d(np.array([0, 1, -1, 9, 2, -5, 3, 4], np.int32))
    st = status_word()
    y = torch.zeros((5, 16), dtype=torch.bfloat16, device=DEV)
    mp.mp_unpad_restore(padded, row_map, 5, y=y, status=st)
    assert mp.status_bits(int(h(st)[0])) == {"bad_row"}
    want = np.zeros((5, 16), np.uint16)
    src = h(padded)
    for dd, s in enumerate([0, 1, -1, 9, 2, -5, 3, 4]):
        if 0 <= s < 5:
            want[s] = src[dd]
    np.testing.assert_array_equal(h(y), want)


def test_sort_pad_many_rows():
    """More than 155,000 rows of 64 vectors: thousands of CTAs, every row
    position in a CTA and every warp's share of rows used."""
    G, R, align, H = 16, 8, 128, 512
    sizes, order = _meta(99, G, R, max_size=3600)
    N = int(sizes.sum())
    assert N > 2 * 2 * 152 * 256
    x = wl.random_rows(N, H, 12)
    probs = np.random.default_rng(2).random(N).astype(np.float32)
    out_rows = N + G * (align - 1)
    out, out_p, row_map, o_map = run_case(x, probs, sizes, order, G, align, out_rows)
    y, y_p = mp.mp_unpad_restore(out, row_map, N, out_p)
    np.testing.assert_array_equal(h(y), x)
    np.testing.assert_array_equal(h(y_p), probs)
    g_pad, _ = mp.mp_unpad_restore_bwd(d(x), row_map)
    np.testing.assert_array_equal(h(g_pad), h(out))


# --------------------------------------------------------------------------
# fp16 / fp32 tokens and caller-supplied padded sizes
# --------------------------------------------------------------------------

def _dev_tokens(x_np):
    t = torch.from_numpy(np.ascontiguousarray(x_np))
    return t.to(DEV)


@pytest.mark.parametrize("dtype,H", [(np.float32, 2048), (np.float16, 2048), (np.float32, 5),
                                     (np.float16, 37)])
def test_sort_pad_roundtrip_other_token_types(dtype, H):
    N = 8192 if H > 64 else 3000
    c = wl.chunks(N, H=8)                               # sizes and order only
    rng = np.random.default_rng(17)
    x = rng.standard_normal((N, H)).astype(dtype)
    G, align = c["G"], c["align"]
    out_rows = wl.padded_rows_bound(N, G, align)
    st = status_word()
    out, out_p, row_map, goff = mp.mp_sort_chunks_pad(
        _dev_tokens(x), d(c["split_sizes"]), d(c["chunk_order"]), G, align, out_rows,
        d(c["probs"]), status=st)
    o_out, o_p, o_map, o_goff, _ = oracle.sort_chunks_pad(x, c["probs"], c["split_sizes"],
                                                          c["chunk_order"], G, align, out_rows)
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got.view(np.uint16), o_out.view(np.uint16))
    np.testing.assert_array_equal(h(row_map), o_map)
    np.testing.assert_array_equal(h(goff), o_goff)
    assert int(h(st)[0]) == 0
    y, _ = mp.mp_unpad_restore(out, row_map, N, out_p)
    np.testing.assert_array_equal(y.cpu().numpy().view(np.uint16), x.view(np.uint16))
    # both backwards on independent gradients, against the oracle's backwards
    g_y = rng.standard_normal((N, H)).astype(dtype)
    g_y_p = rng.standard_normal(N).astype(np.float32)
    g_pad, g_pad_p = mp.mp_unpad_restore_bwd(_dev_tokens(g_y), row_map, d(g_y_p))
    o_gpad, o_gpad_p = oracle.unpad_restore_bwd(g_y, g_y_p, o_map, N)
    np.testing.assert_array_equal(g_pad.cpu().numpy().view(np.uint16), o_gpad.view(np.uint16))
    np.testing.assert_array_equal(h(g_pad_p), o_gpad_p)
    g_out = rng.standard_normal((out_rows, H)).astype(dtype)
    g_out_p = rng.standard_normal(out_rows).astype(np.float32)
    g_x, g_x_p = mp.mp_sort_chunks_pad_bwd(_dev_tokens(g_out), row_map, N, d(g_out_p))
    o_gx, o_gx_p = oracle.sort_chunks_pad_bwd(g_out, g_out_p, o_map, N)
    got_gx = g_x.cpu().numpy()
    np.testing.assert_array_equal(got_gx.view(np.uint16), o_gx.view(np.uint16))
    np.testing.assert_array_equal(h(g_x_p), o_gx_p)


@pytest.mark.parametrize("slack", ["exact", "larger", "smaller"])
def test_sort_pad_explicit_padded_sizes(slack):
    N, H = 8192, 2048
    c = wl.chunks(N)
    G, R = c["G"], c["C"] // c["G"]
    sizes, order = c["split_sizes"], c["chunk_order"]
    grows = np.array([sizes[order[g * R:(g + 1) * R]].sum() for g in range(G)])
    rng = np.random.default_rng(23)
    if slack == "exact":
        padded = grows
    elif slack == "larger":
        padded = grows + rng.integers(0, 300, size=G)
    else:
        padded = grows - rng.integers(0, 40, size=G)
        padded[3] = -5                                   # negative: an empty group
    padded = padded.astype(np.int32)
    out_rows = int(np.maximum(padded, 0).sum()) + 10
    st = status_word()
    out, out_p, row_map, goff = mp.mp_sort_chunks_pad(
        d(c["x"]), d(sizes), d(order), G, 1, out_rows, d(c["probs"]), padded_sizes=d(padded),
        status=st)
    o_out, o_p, o_map, o_goff, fl = oracle.sort_chunks_pad(c["x"], c["probs"], sizes, order, G,
                                                           1, out_rows, padded_sizes=padded)
    np.testing.assert_array_equal(h(out), o_out)
    np.testing.assert_array_equal(h(out_p), o_p)
    np.testing.assert_array_equal(h(row_map), o_map)
    np.testing.assert_array_equal(h(goff), o_goff)
    assert mp.status_bits(int(h(st)[0])) == {k for k, v in fl.items() if v}
    assert (slack == "smaller") == bool(fl["bad_padded"])


def test_sort_pad_past_int32_element_offsets():
    """540,000 rows of H = 4,096 (2.2e9 elements, past 2^31) through sort+pad
    and unpad+restore: row offsets must be formed in 64 bits.  The rows are
    counter-based, so any row can be rebuilt on the host; the layout (row_map,
    group_off) is checked in full against the oracle, whose layout does not
    depend on H, and the copied rows on a sample that includes the last ones."""
    N, H = 540000, 4096
    sizes, order = wl.chunk_layout(N)
    G, align = wl.CHUNKS["experts"], wl.CHUNKS["align"]
    out_rows = wl.padded_rows_bound(N, G, align)
    assert out_rows * H > 2**31
    x = wl.hashed_rows_torch(N, H, 41, DEV)
    out, _, row_map, goff = mp.mp_sort_chunks_pad(x, d(sizes), d(order), G, align, out_rows)
    _, _, o_map, o_goff, _ = oracle.sort_chunks_pad(np.zeros((N, 8), np.uint16), None, sizes,
                                                    order, G, align, out_rows)
    np.testing.assert_array_equal(h(row_map), o_map)
    np.testing.assert_array_equal(h(goff), o_goff)
    rng = np.random.default_rng(8)
    dsample = np.unique(np.concatenate([rng.choice(out_rows, 96, replace=False),
                                        np.arange(out_rows - 32, out_rows),
                                        np.nonzero(o_map >= N - 16)[0]]))
    got = h(out.index_select(0, torch.from_numpy(dsample.astype(np.int64)).to(DEV)))
    src = o_map[dsample]
    want = np.zeros((dsample.size, H), np.uint16)
    want[src >= 0] = wl.hashed_rows(src[src >= 0], H, 41)
    np.testing.assert_array_equal(got, want)
    del x
    y, _ = mp.mp_unpad_restore(out, row_map, N)
    ysample = np.unique(np.concatenate([rng.choice(N, 96, replace=False),
                                        np.arange(N - 32, N)]))
    np.testing.assert_array_equal(
        h(y.index_select(0, torch.from_numpy(ysample.astype(np.int64)).to(DEV))),
        wl.hashed_rows(ysample, H, 41))
