"""Element-complete parity at full size: the skewed dispatch (T=16,384,
H=4,096, E=128, K=8, Zipf-biased router) and the large-hidden step
(T=32,768, H=7,168, E=256, K=8, group-limited router), in the launch
configuration the benchmark times.

One chain per workload, as the benchmark's step runs it:

    build_map -> permute(x, probs) -> unpermute(rows_in, probs)
              -> unpermute_bwd(g_y, rows_in, probs) -> permute_bwd(g_rows)

`rows_in` are independent expert rows (the counter-based bf16 tensor of the
input generator), so the combine sums K different rows per token.  The map
is compared in full.  Every element of every other output is then compared
with the oracle, walking the tokens in blocks: the block's rows are gathered
on the device (by the oracle's map, which equals the device map), copied to
the host, and the oracle runs on the same block with the routes renumbered
locally, on a thread pool over token sub-ranges (each token's outputs depend
on that token alone).  The permute backward's oracle input is the oracle's
own row gradient, which the device's was just checked equal to.

Bar: bit-exact everywhere except g_probs of the unpermute backward, which is
within the fp32 summation bound against the oracle's fp64 sum (the same bound
the other parity tests use).  Combine arithmetic: "core.transformer.moe.
batch_invariant", `_rank_tree_unpermute_kernel` (slot-order FP32 FMA from
zero, one BF16 rounding); row placement: "d9d 0.1.0 -- permute_with_probs.py",
`_permute_kernel`.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import workloads as wl
from tests.gpu_util import DEV, d, gprobs_bound, h

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROWS_SEED = 77
BLOCK = {"skewed": 2048, "large": 1024}     # tokens per host block


def _f32(bits):
    """bf16 bit patterns -> float32 (exact widening)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _check_subrange(a, b, blk, w):
    """Oracle on tokens [a, b) of a block and element-wise comparison with the
    device results gathered for that block.  Returns a list of failures."""
    K, H = w["K"], w["H"]
    rim = blk["rim"][a:b]
    n = b - a
    local = np.where(rim >= 0, np.arange(n * K, dtype=np.int32).reshape(n, K), -1)
    routed = (rim >= 0).ravel()
    r0, r1 = a * K, b * K                      # this sub-range's slice of the gathered rows
    rows_in = blk["rows_in"][r0:r1]
    x, probs, g_y = w["x"][blk["t0"] + a:blk["t0"] + b], blk["probs"][a:b], \
        w["g_y"][blk["t0"] + a:blk["t0"] + b]
    bad = []

    o_out, o_out_p = oracle.permute(x, probs, local)
    if not np.array_equal(blk["out"][r0:r1][routed], o_out[routed]):
        bad.append(("permute rows", a, b))
    if not np.array_equal(blk["out_p"][r0:r1][routed], o_out_p[routed]):
        bad.append(("permute probs", a, b))

    o_y = oracle.unpermute(rows_in, probs, local, n, H)
    if not np.array_equal(blk["y"][a:b], o_y):
        bad.append(("unpermute", a, b))

    o_grows, o_gp = oracle.unpermute_bwd(g_y, rows_in, probs, local)
    if not np.array_equal(blk["g_rows"][r0:r1][routed], o_grows[routed]):
        bad.append(("unpermute_bwd g_rows", a, b))
    gp = blk["g_probs"][a:b].astype(np.float64)
    rf = _f32(rows_in).reshape(n, K, H)
    bound = gprobs_bound(rf, _f32(g_y)[:, None, :], o_gp)
    if not np.all(np.abs(gp - o_gp) <= bound):
        bad.append(("unpermute_bwd g_probs", a, b))

    o_gx, _ = oracle.permute_bwd(o_grows, None, local, n, H)
    if not np.array_equal(blk["g_x"][a:b], o_gx):
        bad.append(("permute_bwd", a, b))
    return bad


@pytest.mark.parametrize("name", ["skewed", "large"])
def test_full_size_every_element(name):
    w = wl.routed(name)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    R = T * K

    idx, probs = d(w["idx"]), d(w["probs"])
    rim, s2f, counts, offsets = mp.mp_build_map(idx, E)
    o_rim, o_s2f, o_counts, o_offsets, n_bad = oracle.build_map(w["idx"], E)
    assert n_bad == 0
    np.testing.assert_array_equal(h(rim), o_rim)
    np.testing.assert_array_equal(h(s2f), o_s2f)
    np.testing.assert_array_equal(h(counts), o_counts)
    np.testing.assert_array_equal(h(offsets), o_offsets)

    out, out_p = mp.mp_permute(d(w["x"]), rim, probs)
    rows_in = wl.hashed_rows_torch(R, H, ROWS_SEED, DEV)
    y = mp.mp_unpermute(rows_in, rim, probs)
    g_rows, g_probs = mp.mp_unpermute_bwd(d(w["g_y"]), rim, rows_in, probs)
    g_x, _ = mp.mp_permute_bwd(g_rows, rim)
    torch.cuda.synchronize()

    threads = max(1, min(32, os.cpu_count() or 1))
    bt = BLOCK[name]
    failures = []
    with ThreadPoolExecutor(max_workers=threads) as pool:
        for t0 in range(0, T, bt):
            t1 = min(T, t0 + bt)
            rim_b = o_rim[t0:t1]
            sel = torch.from_numpy(np.maximum(rim_b, 0).ravel().astype(np.int64)).to(DEV)
            blk = {"t0": t0, "rim": rim_b, "probs": w["probs"][t0:t1],
                   "out": h(out.index_select(0, sel)), "out_p": h(out_p.index_select(0, sel)),
                   "rows_in": h(rows_in.index_select(0, sel)),
                   "g_rows": h(g_rows.index_select(0, sel)),
                   "y": h(y[t0:t1]), "g_probs": h(g_probs[t0:t1]), "g_x": h(g_x[t0:t1])}
            # the gathered expert rows are the generator's rows (first and last routes)
            ends = np.concatenate([rim_b.ravel()[:4], rim_b.ravel()[-4:]])
            np.testing.assert_array_equal(
                np.concatenate([blk["rows_in"][:4], blk["rows_in"][-4:]]),
                wl.hashed_rows(ends, H, ROWS_SEED))
            n = t1 - t0
            edges = [n * i // threads for i in range(threads + 1)]
            parts = [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]
            for bad in pool.map(lambda ab: _check_subrange(ab[0], ab[1], blk, w), parts):
                failures.extend((what, t0 + a, t0 + b) for what, a, b in bad)
            if len(failures) > 20:
                break
    assert not failures, f"mismatches (op, first token, end token): {failures[:20]}"


def _check_ep_subrange(a, b, blk, w, modes):
    """Oracle's rank-ordered combine (ep = 8) on tokens [a, b) of a block, in
    every mode, against the device outputs of the block."""
    K, H, E = w["K"], w["H"], w["E"]
    rim = blk["rim"][a:b]
    n = b - a
    local = np.where(rim >= 0, np.arange(n * K, dtype=np.int32).reshape(n, K), -1)
    rows_in = blk["rows_in"][a * K:b * K]
    t0 = blk["t0"]
    bad = []
    for m, (bf16p, fp64) in enumerate(modes):
        want = oracle.unpermute_ep(rows_in, w["probs"][t0 + a:t0 + b], local,
                                   w["idx"][t0 + a:t0 + b], n, H, E, 8, bf16p, fp64)
        if not np.array_equal(blk["y"][m][a:b], want):
            bad.append((f"unpermute_ep(bf16_partials={bf16p}, fp64_cross_rank={fp64})", a, b))
    return bad


@pytest.mark.parametrize("name", ["skewed", "large"])
def test_full_size_ep_every_element(name):
    """The rank-ordered combine over 8 simulated EP ranks ("core.transformer.
    moe.batch_invariant", `_rank_tree_unpermute_kernel`: per-rank slot-order
    FMA partials, optionally rounded to bf16, added in rank order in fp32 or
    fp64, one bf16 rounding) at full size, every element of every mode."""
    w = wl.routed(name, grads=False)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    R = T * K
    idx, probs = d(w["idx"]), d(w["probs"])
    rim, *_ = mp.mp_build_map(idx, E)
    o_rim, *_ = oracle.build_map(w["idx"], E)
    np.testing.assert_array_equal(h(rim), o_rim)
    rows_in = wl.hashed_rows_torch(R, H, ROWS_SEED + 1, DEV)
    modes = [(False, False), (True, False), (False, True), (True, True)]
    ys = [mp.mp_unpermute_ep(rows_in, rim, idx, E, 8, probs, bf16_partials=b16,
                             fp64_cross_rank=f64) for b16, f64 in modes]
    torch.cuda.synchronize()

    threads = max(1, min(32, os.cpu_count() or 1))
    bt = BLOCK[name]
    failures = []
    with ThreadPoolExecutor(max_workers=threads) as pool:
        for t0 in range(0, T, bt):
            t1 = min(T, t0 + bt)
            rim_b = o_rim[t0:t1]
            sel = torch.from_numpy(np.maximum(rim_b, 0).ravel().astype(np.int64)).to(DEV)
            blk = {"t0": t0, "rim": rim_b, "rows_in": h(rows_in.index_select(0, sel)),
                   "y": [h(y[t0:t1]) for y in ys]}
            ends = np.concatenate([rim_b.ravel()[:4], rim_b.ravel()[-4:]])
            np.testing.assert_array_equal(
                np.concatenate([blk["rows_in"][:4], blk["rows_in"][-4:]]),
                wl.hashed_rows(ends, H, ROWS_SEED + 1))
            n = t1 - t0
            edges = [n * i // threads for i in range(threads + 1)]
            parts = [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]
            for bad in pool.map(lambda ab: _check_ep_subrange(ab[0], ab[1], blk, w, modes),
                                parts):
                failures.extend((what, t0 + a, t0 + b) for what, a, b in bad)
            if len(failures) > 20:
                break
    assert not failures, f"mismatches (mode, first token, end token): {failures[:20]}"
