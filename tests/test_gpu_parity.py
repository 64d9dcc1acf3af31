"""Parity of the CUDA path (through the C ABI) with the oracle.

Bar: bit-exact for every integer, layout and copied output and for the bf16
outputs of unpermute / permute_bwd / unpermute_bwd (both sides run the same
slot-order fp32 FMA chain and one round-to-nearest-even); g_probs of
unpermute_bwd within the fp32 summation bound against the oracle's fp64 sum
(gpu_util.gprobs_bound).  Small and mid workloads are compared element by
element; the full-size skewed and large workloads are compared element by
element in tests/test_gpu_fullsize.py.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import workloads as wl
from tests.gpu_util import DEV, bf16_ulp_distance, d, gprobs_bound, h, status_word

pytestmark = pytest.mark.gpu


def f32(bits):
    return oracle.f32_from_bf16(bits) if bits.size < 4096 else \
        (bits.astype(np.uint32) << 16).view(np.float32)


def check_map(idx, E, expect_status=0):
    st = status_word()
    rim, s2f, counts, offsets = mp.mp_build_map(d(idx), E, status=st)
    o_rim, o_s2f, o_counts, o_offsets, bad = oracle.build_map(idx, E)
    np.testing.assert_array_equal(h(rim), o_rim)
    np.testing.assert_array_equal(h(s2f), o_s2f)
    np.testing.assert_array_equal(h(counts), o_counts)
    np.testing.assert_array_equal(h(offsets), o_offsets)
    assert int(h(st)[0]) == expect_status
    assert (bad > 0) == bool(expect_status & 1)
    return rim, o_rim


# --------------------------------------------------------------------------
# routing map
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "mid", "skewed", "large"])
def test_build_map_workloads(name):
    idx, _, E = wl.routing(name)
    check_map(idx, E)


def _edge_idx(case):
    rng = np.random.default_rng(sum(map(ord, case)))
    if case == "one":
        return np.zeros((1, 1), np.int32), 1
    if case == "ragged_dups_empty":
        idx = rng.integers(-1, 37, size=(3001, 3)).astype(np.int32)
        return idx, 37
    if case == "max_experts":
        return rng.integers(0, 1024, size=(5000, 2)).astype(np.int32), 1024
    if case == "one_hot_expert":
        return np.full((4099, 4), 5, np.int32), 8
    if case == "e1":
        return np.zeros((2049, 3), np.int32), 1
    if case == "k16":
        return rng.integers(0, 64, size=(777, 16)).astype(np.int32), 64
    if case == "all_empty":
        return -np.ones((300, 4), np.int32), 16
    if case == "three_launch":       # count matrix too large for the fused rank
        return rng.integers(-1, 1024, size=(25600, 8)).astype(np.int32), 1024
    if case == "tile_x8":            # 1M routes: 8 sub-tiles per tile
        return rng.integers(0, 16, size=(131072, 8)).astype(np.int32), 16
    raise KeyError(case)


@pytest.mark.parametrize("case", ["one", "ragged_dups_empty", "max_experts", "one_hot_expert",
                                  "e1", "k16", "all_empty", "three_launch", "tile_x8"])
def test_build_map_edges(case):
    idx, E = _edge_idx(case)
    check_map(idx, E)


@pytest.mark.parametrize("T,K,E,empty", [
    (4097, 1, 7, 0.0),        # one route past the one-CTA form: a cluster of 3
    (513, 8, 64, 0.1),        # 4,104 routes
    (2048, 16, 1024, 0.0),    # 32,768 routes: 16 CTAs, the largest cluster, E at its limit
    (2047, 16, 1, 0.3),       # one expert, many empty slots
    (4000, 8, 257, 0.05),     # 32,000 routes, ragged last tile
    (1500, 6, 1024, 0.5),     # half the slots empty
])
def test_build_map_cluster_sizes(T, K, E, empty):
    """The map built by one thread-block cluster (4,097 to 32,768 routes)."""
    rng = np.random.default_rng(T * K + E)
    idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    idx[rng.random((T, K)) < empty] = -1
    check_map(idx, E)
    cap = max(1, T * K // (2 * E))
    got = mp.mp_build_map_capacity(d(idx), E, cap)
    want = oracle.build_map_capacity(idx, E, cap)
    for a, b in zip(got, want[:4]):
        np.testing.assert_array_equal(h(a), b)


@pytest.mark.parametrize("T", [500, 2500, 12000])   # one CTA, one cluster, two kernels
def test_build_map_bad_index_sets_status(T):
    rng = np.random.default_rng(5)
    idx = rng.integers(0, 20, size=(T, 4)).astype(np.int32)
    idx[7, 1] = 20
    idx[T - 3, 3] = -7
    check_map(idx, 20, expect_status=mp.STATUS_BITS["bad_expert"])


def test_build_map_empty_batch():
    rim, s2f, counts, offsets = mp.mp_build_map(torch.zeros((0, 4), dtype=torch.int32,
                                                            device=DEV), 9)
    assert h(counts).sum() == 0 and np.all(h(offsets) == 0)


def test_build_map_is_deterministic():
    idx, _, E = wl.routing("skewed")
    a = mp.mp_build_map(d(idx), E)
    for _ in range(3):
        b = mp.mp_build_map(d(idx), E)
        for x, y in zip(a, b):
            assert torch.equal(x, y)


# --------------------------------------------------------------------------
# permute / unpermute / backwards, element by element
# --------------------------------------------------------------------------

def _full_case(name, H=None, T=None, empty=False, rows_seed=7):
    w = wl.routed(name, T=T, H=H)
    if empty:
        rng = np.random.default_rng(3)
        w["idx"][rng.random(w["idx"].shape) < 0.15] = -1
    T, H, K = w["T"], w["H"], w["K"]
    w["rows_in"] = wl.random_rows(T * K, H, seed=rows_seed)
    w["g_rows_in"] = wl.random_rows(T * K, H, seed=rows_seed + 1)
    return w


@pytest.mark.parametrize("name,H,T,empty", [
    ("tiny", None, None, False),
    ("mid", None, None, False),
    ("mid", None, 1234, True),          # ragged T, empty slots
    ("mid", 40, 3000, False),           # H % 8 == 0 but short rows
    ("mid", 37, 999, True),             # element path (H % 8 != 0)
    ("skewed", 264, 3000, False),       # skewed routing, odd vector count
])
def test_forward_and_backward_elementwise(name, H, T, empty):
    w = _full_case(name, H=H, T=T, empty=empty)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    idx, probs = d(w["idx"]), d(w["probs"])
    rim, _, _, _ = mp.mp_build_map(idx, E)
    o_rim, *_ = oracle.build_map(w["idx"], E)
    np.testing.assert_array_equal(h(rim), o_rim)
    mapped = np.sort(o_rim[o_rim >= 0])

    # permute
    out, out_p = mp.mp_permute(d(w["x"]), rim, probs)
    o_out, o_out_p = oracle.permute(w["x"], w["probs"], o_rim)
    np.testing.assert_array_equal(h(out)[mapped], o_out[mapped])
    np.testing.assert_array_equal(h(out_p)[mapped], o_out_p[mapped])
    out2, _ = mp.mp_permute(d(w["x"]), rim)
    np.testing.assert_array_equal(h(out2)[mapped], o_out[mapped])

    # unpermute of independent rows, with and without probs
    rows = d(w["rows_in"])
    y = mp.mp_unpermute(rows, rim, probs)
    np.testing.assert_array_equal(h(y), oracle.unpermute(w["rows_in"], w["probs"], o_rim, T, H))
    y0 = mp.mp_unpermute(rows, rim)
    np.testing.assert_array_equal(h(y0), oracle.unpermute(w["rows_in"], None, o_rim, T, H))

    # permute backward
    g_out = d(w["g_rows_in"])
    g_op = d(w["g_out_probs"])
    g_x, g_p = mp.mp_permute_bwd(g_out, rim, g_op)
    o_gx, o_gp = oracle.permute_bwd(w["g_rows_in"], w["g_out_probs"], o_rim, T, H)
    np.testing.assert_array_equal(h(g_x), o_gx)
    np.testing.assert_array_equal(h(g_p), o_gp)

    # unpermute backward with probs
    g_rows, g_probs = mp.mp_unpermute_bwd(d(w["g_y"]), rim, rows, probs)
    o_grows, o_gprobs = oracle.unpermute_bwd(w["g_y"], w["rows_in"], w["probs"], o_rim)
    np.testing.assert_array_equal(h(g_rows)[mapped], o_grows[mapped])
    gp = h(g_probs).astype(np.float64)
    rf = f32(w["rows_in"])[np.maximum(o_rim, 0)]           # [T,K,H]
    gyf = f32(w["g_y"])[:, None, :]
    bound = gprobs_bound(rf, gyf, o_gprobs)
    assert np.all(np.abs(gp - o_gprobs) <= bound)
    assert np.all(gp[o_rim < 0] == 0)
    # ... and without probs: a plain copy of g_y to every row
    g_rows0, none = mp.mp_unpermute_bwd(d(w["g_y"]), rim)
    assert none is None
    o_grows0, _ = oracle.unpermute_bwd(w["g_y"], None, None, o_rim)
    np.testing.assert_array_equal(h(g_rows0)[mapped], o_grows0[mapped])


def test_misaligned_rows_take_the_element_path():
    w = _full_case("mid", H=64, T=500)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    rim, *_ = mp.mp_build_map(d(w["idx"]), E)
    o_rim, *_ = oracle.build_map(w["idx"], E)
    base = torch.empty(T * H + 1, dtype=torch.bfloat16, device=DEV)
    x = base[1:].view(T, H)                              # 2-byte offset: not 16-B aligned
    x.copy_(d(w["x"]))
    out, _ = mp.mp_permute(x, rim)
    o_out, _ = oracle.permute(w["x"], None, o_rim)
    np.testing.assert_array_equal(h(out), o_out)
    rbase = torch.empty(T * K * H + 1, dtype=torch.bfloat16, device=DEV)
    rows = rbase[1:].view(T * K, H)
    rows.copy_(d(w["rows_in"]))
    y = mp.mp_unpermute(rows, rim, d(w["probs"]))
    np.testing.assert_array_equal(h(y), oracle.unpermute(w["rows_in"], w["probs"], o_rim, T, H))


def test_unpermute_k1_unit_probs_is_identity():
    rng = np.random.default_rng(2)
    T, H, E = 3000, 512, 16
    idx = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    x = wl.random_rows(T, H, 9)
    rim, *_ = mp.mp_build_map(d(idx), E)
    rows, _ = mp.mp_permute(d(x), rim)
    ones = torch.ones((T, 1), dtype=torch.float32, device=DEV)
    np.testing.assert_array_equal(h(mp.mp_unpermute(rows, rim, ones)), x)
    np.testing.assert_array_equal(h(mp.mp_unpermute(rows, rim)), x)


def test_unpermute_is_batch_invariant():
    """A token's output bits do not change with the rest of the batch."""
    w = _full_case("mid", T=2048)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    rim, *_ = mp.mp_build_map(d(w["idx"]), E)
    rows, _ = mp.mp_permute(d(w["rows_in"][:T]), rim)
    y_full = h(mp.mp_unpermute(rows, rim, d(w["probs"])))
    rng = np.random.default_rng(4)
    sel = np.sort(rng.choice(T, 300, replace=False))
    for trial in range(2):
        perm = rng.permutation(300)
        idx_s = w["idx"][sel][perm]
        rim_s, *_ = mp.mp_build_map(d(idx_s), E)
        rows_s, _ = mp.mp_permute(d(w["rows_in"][:T][sel][perm]), rim_s)
        y_s = h(mp.mp_unpermute(rows_s, rim_s, d(w["probs"][sel][perm])))
        np.testing.assert_array_equal(y_s, y_full[sel][perm])


def test_unpermute_bwd_is_deterministic():
    w = _full_case("mid", T=2048)
    rim, *_ = mp.mp_build_map(d(w["idx"]), w["E"])
    rows, gy, probs = d(w["rows_in"]), d(w["g_y"]), d(w["probs"])
    a = mp.mp_unpermute_bwd(gy, rim, rows, probs)
    for _ in range(3):
        b = mp.mp_unpermute_bwd(gy, rim, rows, probs)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_unpermute_ulp_fallback_not_needed():
    """The fallback tolerance (1 bf16 ulp) is stated but unused: distance 0."""
    w = _full_case("tiny")
    rim, *_ = mp.mp_build_map(d(w["idx"]), w["E"])
    o_rim, *_ = oracle.build_map(w["idx"], w["E"])
    y = h(mp.mp_unpermute(d(w["rows_in"]), rim, d(w["probs"])))
    o = oracle.unpermute(w["rows_in"], w["probs"], o_rim, w["T"], w["H"])
    assert bf16_ulp_distance(y, o).max() <= 1
    assert bf16_ulp_distance(y, o).max() == 0


@pytest.mark.parametrize("K", [8, 5, 3, 2])   # the 8-, 6-, 4- and 2-slot batches
def test_staged_row_kernels_full_compare(K):
    """16,385 tokens, one per CTA (H = 1,032: 129 vectors, so a second pass
    with one lane busy), make grids past 16,384 CTAs, which run the forms that
    stage their rows in shared memory: unpermute, its backward and the permute
    backward.  A tenth of the slots are unrouted.  Every output is compared
    with the oracle in full."""
    T, H = 16385, 1032
    idx, probs, E = wl.routing("skewed", T=T)
    idx, probs = idx[:, :K].copy(), np.ascontiguousarray(probs[:, :K])
    rng = np.random.default_rng(5)
    idx = idx.copy()
    idx[rng.random(idx.shape) < 0.1] = -1
    rows = wl.random_rows(T * K, H, 21)
    gy = wl.random_rows(T, H, 22)
    rim, *_ = mp.mp_build_map(d(idx), E)
    o_rim, _, _, o_offsets, _ = oracle.build_map(idx, E)
    np.testing.assert_array_equal(h(rim), o_rim)
    routed = int(o_offsets[-1])
    dr, dp = d(rows), d(probs)

    y = mp.mp_unpermute(dr, rim, dp)
    np.testing.assert_array_equal(h(y), oracle.unpermute(rows, probs, o_rim, T, H))

    g_rows, g_probs = mp.mp_unpermute_bwd(d(gy), rim, dr, dp)
    o_grows, o_gp = oracle.unpermute_bwd(gy, rows, probs, o_rim)
    np.testing.assert_array_equal(h(g_rows)[:routed], o_grows[:routed])
    gp = h(g_probs).astype(np.float64)
    for k in range(K):
        bound = gprobs_bound(f32(rows)[np.maximum(o_rim[:, k], 0)], f32(gy), o_gp[:, k])
        assert np.all(np.abs(gp[:, k] - o_gp[:, k]) <= bound)
    assert np.all(gp[o_rim < 0] == 0)

    g_x, _ = mp.mp_permute_bwd(dr, rim)
    np.testing.assert_array_equal(h(g_x), oracle.permute_bwd(rows, None, o_rim, T, H)[0])


def test_rows_past_int32_element_offsets():
    """T = 66,000 tokens, K = 8, H = 4,096: the permuted tensors hold 2.16e9
    elements, past 2^31, so row offsets must be formed in 64 bits.  All the
    row tensors are counter-based (rebuilt on the host for any row); sampled
    tokens include those holding the last rows of the permuted tensor."""
    T, H, K = 66000, 4096, 8
    idx_h, probs_h, E = wl.routing("skewed", T=T, seed=5)
    R = T * K
    assert R * H > 2**31
    rim = mp.mp_build_map(d(idx_h), E)[0]
    o_rim, *_ = oracle.build_map(idx_h, E)
    np.testing.assert_array_equal(h(rim), o_rim)
    rng = np.random.default_rng(12)
    high = np.unique(np.nonzero(o_rim >= (2**31) // H)[0])           # rows past 2^31 elements
    sample = np.unique(np.concatenate([rng.choice(T, 64, replace=False),
                                       rng.choice(high, 64, replace=False), [0, T - 1]]))
    assert (o_rim[sample] >= (2**31) // H).any()
    rs = torch.from_numpy(o_rim[sample].ravel().astype(np.int64)).to(DEV)
    ts = torch.from_numpy(sample.astype(np.int64)).to(DEV)
    probs = d(probs_h)

    x = wl.hashed_rows_torch(T, H, 31, DEV)
    out, _ = mp.mp_permute(x, rim)
    got = h(out.index_select(0, rs)).reshape(len(sample), K, H)
    np.testing.assert_array_equal(got, np.repeat(wl.hashed_rows(sample, H, 31)[:, None, :], K,
                                                 axis=1))
    del out, x

    rows = wl.hashed_rows_torch(R, H, 32, DEV)
    rim_s = o_rim[sample]
    rows_s = wl.hashed_rows(rim_s.ravel(), H, 32)
    local = np.arange(rim_s.size, dtype=np.int32).reshape(rim_s.shape)
    y = h(mp.mp_unpermute(rows, rim, probs).index_select(0, ts))
    np.testing.assert_array_equal(y, oracle.unpermute(rows_s, probs_h[sample], local,
                                                      len(sample), H))
    y_ep = h(mp.mp_unpermute_ep(rows, rim, d(idx_h), E, 8, probs).index_select(0, ts))
    np.testing.assert_array_equal(y_ep, oracle.unpermute_ep(rows_s, probs_h[sample], local,
                                                            idx_h[sample], len(sample), H, E, 8))
    g_x, _ = mp.mp_permute_bwd(rows, rim)
    o_gx, _ = oracle.permute_bwd(rows_s, None, local, len(sample), H)
    np.testing.assert_array_equal(h(g_x.index_select(0, ts)), o_gx)
    del g_x

    gy = wl.hashed_rows_torch(T, H, 33, DEV)
    gy_s = wl.hashed_rows(sample, H, 33)
    g_rows, g_probs = mp.mp_unpermute_bwd(gy, rim, rows, probs)
    o_grows, o_gp = oracle.unpermute_bwd(gy_s, rows_s, probs_h[sample], local)
    np.testing.assert_array_equal(h(g_rows.index_select(0, rs)), o_grows)
    gp = h(g_probs)[sample].astype(np.float64)
    bound = gprobs_bound(f32(rows_s).reshape(len(sample), K, H), f32(gy_s)[:, None, :], o_gp)
    assert np.all(np.abs(gp - o_gp) <= bound)


# --------------------------------------------------------------------------
# expert capacity (token dropping)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name,T,cap", [
    ("skewed", None, 1024),       # hot experts overflow, cold ones keep all
    ("skewed", 3000, 0),          # everything dropped
    ("mid", None, 300),
    ("large", None, 700),         # 2 sub-tiles per tile
    ("mid", 2000, -1),            # no limit: the plain map
    ("skewed", 300, 10),          # one CTA (2,400 routes)
    ("skewed", 4000, 150),        # one thread-block cluster (32,000 routes)
])
def test_build_map_capacity(name, T, cap):
    idx, probs, E = wl.routing(name, T=T)
    st = status_word()
    got = mp.mp_build_map_capacity(d(idx), E, cap, status=st)
    want = oracle.build_map_capacity(idx, E, cap)
    for a, b in zip(got, want[:4]):
        np.testing.assert_array_equal(h(a), b)
    assert int(h(st)[0]) == 0
    if cap >= 0:
        assert h(got[2]).max(initial=0) <= cap


def test_build_map_capacity_three_launch_path_and_dropped_rows_downstream():
    rng = np.random.default_rng(12)
    T, K, E, H = 25600, 8, 1024, 64               # count matrix above the fused limit
    idx = rng.integers(-1, E, size=(T, K)).astype(np.int32)
    idx[:, 0] = 3                                   # one very hot expert
    got = mp.mp_build_map_capacity(d(idx), E, 5000)
    want = oracle.build_map_capacity(idx, E, 5000)
    for a, b in zip(got, want[:4]):
        np.testing.assert_array_equal(h(a), b)
    # dropped slots behave as empty slots in the row ops
    x = wl.random_rows(T, H, 3)
    probs = rng.random((T, K)).astype(np.float32)
    R = int(want[3][-1])
    out, _ = mp.mp_permute(d(x), got[0], d(probs), num_out_rows=R)
    o_out, _ = oracle.permute(x, probs, want[0], out_rows=R)
    np.testing.assert_array_equal(h(out), o_out)
    y = mp.mp_unpermute(out, got[0], d(probs))
    np.testing.assert_array_equal(h(y), oracle.unpermute(o_out, probs, want[0], T, H))


# --------------------------------------------------------------------------
# rank-ordered combine over EP ranks
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name,T,H,ep", [("mid", 2000, None, 8), ("skewed", 3000, 264, 16),
                                          ("tiny", None, None, 4), ("mid", 1500, 37, 2),
                                          # one token per CTA, a ragged last pass
                                          ("mid", 700, 1032, 8), ("skewed", 400, 1160, 4)])
@pytest.mark.parametrize("bf16p,fp64", [(False, False), (True, False), (False, True),
                                         (True, True)])
def test_unpermute_ep(name, T, H, ep, bf16p, fp64):
    w = _full_case(name, T=T, H=H, empty=(name == "mid"))
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    rim, *_ = mp.mp_build_map(d(w["idx"]), E)
    o_rim, *_ = oracle.build_map(w["idx"], E)
    rows = d(w["rows_in"])
    for probs in (w["probs"], None):
        got = mp.mp_unpermute_ep(rows, rim, d(w["idx"]), E, ep,
                                 None if probs is None else d(probs),
                                 bf16_partials=bf16p, fp64_cross_rank=fp64)
        want = oracle.unpermute_ep(w["rows_in"], probs, o_rim, w["idx"], T, H, E, ep, bf16p, fp64)
        np.testing.assert_array_equal(h(got), want)


@pytest.mark.parametrize("K,H,ep", [(12, 136, 8), (16, 64, 4), (9, 37, 16), (16, 40, 64),
                                    (8, 72, 3), (6, 48, 6)])    # ranks not a power of two
@pytest.mark.parametrize("bf16p,fp64", [(False, False), (True, False), (False, True),
                                         (True, True)])
def test_unpermute_ep_wide_slots_and_odd_ranks(K, H, ep, bf16p, fp64):
    """9 to 16 slots per token (the second kernel form), and rank counts that
    are not powers of two, with empty slots and repeated experts, on the
    vector and element paths."""
    rng = np.random.default_rng(K * H + ep)
    T, E = 777, (64 if 64 % ep == 0 else 96)
    idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    idx[rng.random((T, K)) < 0.15] = -1
    probs = rng.random((T, K)).astype(np.float32)
    rows = wl.random_rows(T * K, H, K + H)
    rim, *_ = mp.mp_build_map(d(idx), E)
    o_rim, *_ = oracle.build_map(idx, E)
    for p in (probs, None):
        got = mp.mp_unpermute_ep(d(rows), rim, d(idx), E, ep, None if p is None else d(p),
                                 bf16_partials=bf16p, fp64_cross_rank=fp64)
        want = oracle.unpermute_ep(rows, p, o_rim, idx, T, H, E, ep, bf16p, fp64)
        np.testing.assert_array_equal(h(got), want)


def test_unpermute_ep_one_rank_is_unpermute():
    w = _full_case("mid", T=1000)
    rim, *_ = mp.mp_build_map(d(w["idx"]), w["E"])
    rows, probs = d(w["rows_in"]), d(w["probs"])
    a = mp.mp_unpermute_ep(rows, rim, d(w["idx"]), w["E"], 1, probs)
    assert torch.equal(a, mp.mp_unpermute(rows, rim, probs))


@pytest.mark.parametrize("T,H", [(700, 64), (300, 1024)])   # token groups; a token per CTA
def test_unpermute_ep_wide_ranging_partials(T, H):
    """Rows whose values span ~130 binades, so the per-element rank partials
    often range past what an fp32 sum holds exactly: the fp64 cross-rank sum
    must still match the oracle bit for bit."""
    rng = np.random.default_rng(31)
    K, E, ep = 8, 64, 8
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    probs = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
    ex = rng.integers(60, 191, size=(T * K, H)).astype(np.uint16)
    rows = ((rng.integers(0, 2, size=(T * K, H)) << 15) | (ex << 7) |
            rng.integers(0, 128, size=(T * K, H))).astype(np.uint16)
    rim, *_ = mp.mp_build_map(d(idx), E)
    o_rim, *_ = oracle.build_map(idx, E)
    for bf16p, fp64 in ((True, True), (False, True), (True, False)):
        got = mp.mp_unpermute_ep(d(rows), rim, d(idx), E, ep, d(probs), bf16_partials=bf16p,
                                 fp64_cross_rank=fp64)
        want = oracle.unpermute_ep(rows, probs, o_rim, idx, T, H, E, ep, bf16p, fp64)
        np.testing.assert_array_equal(h(got), want)


@pytest.mark.parametrize("H", [8, 1032])   # token groups; a token per CTA, ragged last pass
@pytest.mark.parametrize("bf16p", [True, False])
def test_unpermute_ep_fp64_sum_on_bf16_ties(bf16p, H):
    """Rank partials 1, 2^-8 (together exactly halfway between two bf16 values)
    and a small third partial on a third rank that decides the rounding, from
    2^-12 to 2^-40 of the first, either sign, or zero.  A third partial
    below an fp32 ulp of the sum puts the midpoint at one end of the kernel's
    directed-rounding bracket: where the other end rounds the other way, the
    kernel takes its fp64 path for that element; elsewhere the bracket
    decides alone.  The oracle's rounding of some rows is pinned below.  The last
    rows cancel exactly: a sum rounded toward -inf gives -0 there, where the
    fp64 sum is +0."""
    E, ep, K = 8, 4, 3
    vals = [(1.0, 2.0**-8, 2.0**-30), (1.0, 2.0**-8, -2.0**-30), (1.0, 2.0**-8, 2.0**-40),
            (1.0, 2.0**-8, -2.0**-40), (1.0, 2.0**-8, 0.0), (-1.0, -(2.0**-8), -(2.0**-30)),
            (3.0, 2.0**-7, 2.0**-33), (2.0**-30, 1.0, 2.0**-8),
            (1.0, 2.0**-8, 2.0**-12), (1.0, 2.0**-8, -2.0**-12), (1.0, 2.0**-8, 2.0**-14),
            (1.0, 2.0**-8, -2.0**-15), (1.0, 2.0**-8, 2.0**-15), (1.0, 2.0**-8, 2.0**-19),
            (1.0, 2.0**-8, -2.0**-21), (-(2.0**-14), -1.0, -(2.0**-8)),
            (1.0, 2.0**-8, 2.0**-33), (1.0, 2.0**-8, -2.0**-34), (1.0, 2.0**-8, 2.0**-20),
            (1.0, -1.0, 0.0), (1.0, -1.0, 2.0**-30), (-(2.0**-8), 1.0, -1.0)]
    T = len(vals)
    idx = np.tile(np.array([[0, 2, 4]], np.int32), (T, 1))      # ranks 0, 1, 2
    rows_f = np.zeros((T * K, H), np.float32)
    rim, *_ = oracle.build_map(idx, E)
    for t, v in enumerate(vals):
        for k in range(K):
            rows_f[rim[t, k]] = v[k]
    rows = torch.from_numpy(rows_f).to(torch.bfloat16)
    assert torch.equal(rows.float(), torch.from_numpy(rows_f))   # all bf16 values
    rows_bits = rows.view(torch.int16).numpy().view(np.uint16)
    g_rim, *_ = mp.mp_build_map(d(idx), E)
    got = mp.mp_unpermute_ep(d(rows_bits), g_rim, d(idx), E, ep, None, bf16_partials=bf16p,
                             fp64_cross_rank=True)
    want = oracle.unpermute_ep(rows_bits, None, rim, idx, T, H, E, ep, bf16p, True)
    np.testing.assert_array_equal(h(got), want)
    up = oracle.bf16_from_f32(np.float32(1.0078125))
    one = oracle.bf16_from_f32(np.float32(1.0))
    assert want[0, 0] == up and want[1, 0] == one
    assert want[8, 0] == up and want[9, 0] == one and want[11, 0] == one
