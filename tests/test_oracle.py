"""Pins of the oracle against what the pages and the mathematics fix.

Each check is independent of the oracle's own code: the worked example printed
on the d9d/TransformerEngine page, brute-force sorting of (expert, token,
slot) keys, exact rational arithmetic for every floating-point step, adjoint
identities that a transposed or mis-indexed gradient breaks, and invariants.
No GPU is needed.
"""
from __future__ import annotations

import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_sections(path):
    sec, out = None, {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            sec = line.strip("[]")
            out[sec] = []
            continue
        out[sec].append([int(v) for v in line.split()])
    return {k: np.array(v, dtype=np.int32) for k, v in out.items()}


def _brute_map(idx, E):
    T, K = idx.shape
    keys = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K)
                  if 0 <= idx[t, k] < E)
    rim = -np.ones((T, K), np.int32)
    s2f = -np.ones(T * K, np.int32)
    for row, (e, t, k) in enumerate(keys):
        rim[t, k] = row
        s2f[row] = t * K + k
    counts = np.array([sum(1 for key in keys if key[0] == e) for e in range(E)], np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return rim, s2f, counts, offsets


def _rand_bf16(rng, shape, lo=-3.0, hi=3.0):
    f = rng.uniform(lo, hi, size=shape).astype(np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf(b):
    return float(exact.frac_of_bf16(int(b)))


# --------------------------------------------------------------------------
# routing map
# --------------------------------------------------------------------------

def test_worked_example_from_page():
    """make_row_id_map's worked example: 5 tokens, 3 experts."""
    g = _read_sections(os.path.join(GOLDEN, "worked_example_row_id_map.txt"))
    mask, pass2 = g["routing_map"], g["pass2"]
    T, E = mask.shape
    K = int(mask.sum(1).max())
    idx = -np.ones((T, K), np.int32)          # experts of each token, ascending
    for t in range(T):
        ex = np.nonzero(mask[t])[0]
        idx[t, :len(ex)] = ex
    rim, s2f, counts, offsets, bad = oracle.build_map(idx, E)
    expect = np.where(idx >= 0, pass2[np.arange(T)[:, None], np.maximum(idx, 0)], -1)
    assert bad == 0
    np.testing.assert_array_equal(rim, expect)
    np.testing.assert_array_equal(rim, [[0, 3], [1, 5], [6, -1], [2, 4], [-1, -1]])
    np.testing.assert_array_equal(counts, mask.sum(0))
    np.testing.assert_array_equal(offsets, [0, 3, 5, 7])
    np.testing.assert_array_equal(s2f[:7], [0, 2, 6, 1, 7, 3, 4])
    np.testing.assert_array_equal(s2f[7:], [-1, -1, -1])


@pytest.mark.parametrize("seed", range(40))
def test_build_map_brute_force(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(0, 13))
    K = int(rng.integers(1, 5))
    E = int(rng.integers(1, 6))
    idx = rng.integers(-1, E, size=(T, K)).astype(np.int32)   # dups and empties
    rim, s2f, counts, offsets, bad = oracle.build_map(idx, E)
    b_rim, b_s2f, b_counts, b_offsets = _brute_map(idx, E)
    assert bad == 0
    np.testing.assert_array_equal(rim, b_rim)
    np.testing.assert_array_equal(s2f, b_s2f)
    np.testing.assert_array_equal(counts, b_counts)
    np.testing.assert_array_equal(offsets, b_offsets)


def test_build_map_bad_indices_count_as_empty():
    idx = np.array([[0, 7], [-5, 1], [1, -1]], np.int32)
    rim, s2f, counts, offsets, bad = oracle.build_map(idx, 3)
    assert bad == 2
    np.testing.assert_array_equal(rim, [[0, -1], [-1, 1], [2, -1]])
    np.testing.assert_array_equal(offsets, [0, 1, 3, 3])


def test_build_map_invariants():
    rng = np.random.default_rng(7)
    T, K, E = 300, 6, 17
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    rim, s2f, counts, offsets, _ = oracle.build_map(idx, E)
    R = T * K
    assert sorted(rim.ravel().tolist()) == list(range(R))         # bijection onto [0,R)
    assert counts.sum() == R and offsets[E] == R
    assert np.all(np.diff(offsets) >= 0)
    flat = rim.ravel()
    np.testing.assert_array_equal(s2f[flat], np.arange(R))        # inverse
    exp_of_row = idx.ravel()[s2f]
    tok_of_row = s2f // K
    for e in range(E):
        seg = slice(offsets[e], offsets[e + 1])
        assert np.all(exp_of_row[seg] == e)
        assert np.all(np.diff(tok_of_row[seg]) > 0)               # tokens ascending


def test_build_map_empty_and_degenerate():
    rim, s2f, counts, offsets, _ = oracle.build_map(np.zeros((0, 4), np.int32), 5)
    assert rim.shape == (0, 4) and counts.sum() == 0 and np.all(offsets == 0)
    rim, _, counts, offsets, _ = oracle.build_map(np.zeros((6, 2), np.int32), 1)
    np.testing.assert_array_equal(rim.ravel(), np.arange(12))   # E=1: identity order
    idx = np.full((4, 3), 2, np.int32)                          # one hot expert, dup slots
    rim, _, counts, offsets, _ = oracle.build_map(idx, 4)
    np.testing.assert_array_equal(rim.ravel(), np.arange(12))
    np.testing.assert_array_equal(offsets, [0, 0, 0, 12, 12])


# --------------------------------------------------------------------------
# bf16 conversion
# --------------------------------------------------------------------------

SPECIAL_F32 = [0x00000000, 0x80000000, 0x3F800000, 0x3F808000, 0x3F818000, 0x3F80FFFF,
               0x3F808001, 0xBF808000, 0x7F7FFFFF, 0x7F7F7FFF, 0x7F7F8000, 0xFF7FFFFF,
               0x00000001, 0x00008000, 0x00018000, 0x0000FFFF, 0x807FFFFF, 0x00800000,
               0x7F800000, 0xFF800000, 0x477FE000, 0x33800000]


def test_bf16_rne_against_exact_rounding():
    rng = random.Random(3)
    bits = SPECIAL_F32 + [rng.getrandbits(32) for _ in range(3000)]
    bits = [b for b in bits if (b & 0x7F800000) != 0x7F800000 or (b & 0x7FFFFF) == 0]
    vals = np.array(bits, np.uint32).view(np.float32)
    got = oracle.bf16_from_f32(vals)
    for b, g in zip(bits, got):
        assert int(g) == exact.bf16_of_f32(exact.f32_from_bits(b)), hex(b)


def test_bf16_rne_matches_torch_and_widening_is_exact():
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    u = u[(u & 0x7F800000) != 0x7F800000]
    f = u.view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_from_f32(f), ref)
    b = rng.integers(0, 2**16, size=5000).astype(np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]
    np.testing.assert_array_equal(oracle.f32_from_bf16(b).view(np.uint32),
                                  b.astype(np.uint32) << 16)


def test_bf16_nan_stays_nan():
    assert (int(oracle.bf16_from_f32(np.float32(np.nan))) & 0x7FFF) > 0x7F80


# --------------------------------------------------------------------------
# permute / unpermute
# --------------------------------------------------------------------------

def _case(seed, T, K, E, H, empty=False, dup=False):
    rng = np.random.default_rng(seed)
    if dup:
        idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    else:
        idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    if empty:
        idx[rng.random((T, K)) < 0.2] = -1
    probs = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
    x = _rand_bf16(rng, (T, H))
    return idx, probs, x


@pytest.mark.parametrize("empty,dup", [(False, False), (True, False), (False, True)])
def test_permute_places_rows_and_probs(empty, dup):
    idx, probs, x = _case(1, 37, 4, 9, 24, empty, dup)
    rim, *_ = oracle.build_map(idx, 9)
    out, out_probs = oracle.permute(x, probs, rim)
    t, k = np.nonzero(rim >= 0)
    np.testing.assert_array_equal(out[rim[t, k]], x[t])
    np.testing.assert_array_equal(out_probs[rim[t, k]], probs[t, k])


def _unpermute_exact(rows, probs, rim, T, H):
    """Slot-order chain of fused multiply-adds, every rounding done exactly."""
    K = rim.shape[1]
    out = np.zeros((T, H), np.uint16)
    for t in range(T):
        for h in range(H):
            acc = 0.0
            for k in range(K):
                r = rim[t, k]
                if r < 0:
                    continue
                rv = _bf(rows[r, h])
                p = 1.0 if probs is None else float(probs[t, k])
                acc = exact.fma_f32(p, rv, acc)        # 1*r is exact: acc + r
            out[t, h] = exact.bf16_of_f32(acc)
    return out


@pytest.mark.parametrize("with_probs", [True, False])
@pytest.mark.parametrize("seed", range(3))
def test_unpermute_exact_fma_chain(with_probs, seed):
    T, K, E, H = 6, 4, 5, 9
    idx, probs, x = _case(seed, T, K, E, H, empty=(seed == 2))
    rng = np.random.default_rng(100 + seed)
    rim, *_ = oracle.build_map(idx, E)
    rows = _rand_bf16(rng, (T * K, H))
    p = probs if with_probs else None
    got = oracle.unpermute(rows, p, rim, T, H)
    np.testing.assert_array_equal(got, _unpermute_exact(rows, p, rim, T, H))


def test_unpermute_fma_differs_from_mul_add():
    """p=1+2^-23, r=1.5, then r=-1.5 with p=1: the exact FMA keeps 1.5*2^-23."""
    p0 = exact.f32_from_bits(0x3F800001)
    rows = np.array([[0x3FC0], [0xBFC0]], np.uint16)      # 1.5, -1.5
    rim = np.array([[1, 0]], np.int32)                      # slot 0 -> row 1 (-1.5)
    probs = np.array([[1.0, p0]], np.float32)
    got = oracle.unpermute(rows, probs, rim, 1, 1)
    want = exact.bf16_of_f32(exact.fma_f32(p0, 1.5, -1.5))
    assert int(got[0, 0]) == want
    assert _bf(want) == pytest.approx(1.5 * 2.0**-23, rel=2**-7)


def test_unpermute_k1_unit_probs_is_identity():
    T, H, E = 50, 33, 7
    idx, _, x = _case(5, T, 1, E, H)
    rim, *_ = oracle.build_map(idx, E)
    rows, _ = oracle.permute(x, None, rim)
    np.testing.assert_array_equal(oracle.unpermute(rows, None, rim, T, H), x)
    ones = np.ones((T, 1), np.float32)
    np.testing.assert_array_equal(oracle.unpermute(rows, ones, rim, T, H), x)
    g_x, _ = oracle.permute_bwd(rows, None, rim, T, H)
    np.testing.assert_array_equal(g_x, x)


def test_unpermute_within_fp64_bound():
    T, K, E, H = 64, 8, 16, 96
    idx, probs, x = _case(9, T, K, E, H, empty=True)
    rng = np.random.default_rng(19)
    rim, *_ = oracle.build_map(idx, E)
    rows = _rand_bf16(rng, (T * K, H))
    got = oracle.f32_from_bf16(oracle.unpermute(rows, probs, rim, T, H)).astype(np.float64)
    rf = oracle.f32_from_bf16(rows).astype(np.float64)
    ex = np.zeros((T, H))
    absum = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            if rim[t, k] >= 0:
                term = float(probs[t, k]) * rf[rim[t, k]]
                ex[t] += term
                absum[t] += np.abs(term)
    bound = np.abs(ex) * 2.0**-8 + K * 2.0**-24 * absum * (1 + 2.0**-8) + 1e-40
    assert np.all(np.abs(got - ex) <= bound)


def test_unpermute_is_batch_invariant():
    """A token's output bits do not depend on the other tokens in the batch."""
    T, K, E, H = 40, 4, 6, 16
    idx, probs, x = _case(21, T, K, E, H)
    rim, *_ = oracle.build_map(idx, E)
    rows, _ = oracle.permute(x, None, rim)
    full = oracle.unpermute(rows, probs, rim, T, H)
    sel = np.array([3, 17, 29])
    rim_s, *_ = oracle.build_map(idx[sel], E)
    rows_s, _ = oracle.permute(x[sel], None, rim_s)
    np.testing.assert_array_equal(oracle.unpermute(rows_s, probs[sel], rim_s, 3, H),
                                  full[sel])


# --------------------------------------------------------------------------
# backwards: exact adjoint identities on exactly representable data
# --------------------------------------------------------------------------

def _small_int_bf16(rng, shape, lim=4):
    return oracle.bf16_from_f32(rng.integers(-lim, lim + 1, size=shape).astype(np.float32))


def test_permute_bwd_is_adjoint_of_permute():
    T, K, E, H = 30, 4, 7, 12
    rng = np.random.default_rng(31)
    idx, probs, _ = _case(31, T, K, E, H, empty=True)
    rim, *_ = oracle.build_map(idx, E)
    x = _small_int_bf16(rng, (T, H))
    G = _small_int_bf16(rng, (T * K, H))
    Gp = rng.integers(-3, 4, size=T * K).astype(np.float32)
    Px, Pp = oracle.permute(x, probs, rim)
    g_x, g_p = oracle.permute_bwd(G, Gp, rim, T, H)
    xf, Gf = oracle.f32_from_bf16(x).astype(np.float64), oracle.f32_from_bf16(G).astype(np.float64)
    mapped = np.sort(rim[rim >= 0])
    lhs = np.sum(oracle.f32_from_bf16(Px[mapped]).astype(np.float64) * Gf[mapped])
    rhs = np.sum(xf * oracle.f32_from_bf16(g_x).astype(np.float64))
    assert lhs == rhs
    lhs_p = np.sum(Pp[mapped].astype(np.float64) * Gp[mapped])
    assert lhs_p == np.sum(probs.astype(np.float64) * g_p)
    assert np.all(g_p[rim < 0] == 0)


def test_permute_bwd_of_permute_with_one_slot_is_identity():
    """K = 1, no probs: each token has one row, and the backward's slot sum
    of a single bf16 value (widened to fp32 and rounded back) is that value,
    except -0, which comes back as +0 because the sum starts from +0."""
    rng = np.random.default_rng(33)
    T, E, H = 57, 5, 9
    idx = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    rim, *_ = oracle.build_map(idx, E)
    x = rng.integers(0, 1 << 16, size=(T, H)).astype(np.uint16)
    x[(x & 0x7F80) == 0x7F80] = 0x3F80          # no inf / NaN patterns
    x[::7, 2] = 0x8000                           # -0
    x[::5, 3] = 0x0001                           # the smallest subnormal
    out, _ = oracle.permute(x, None, rim)
    g_x, _ = oracle.permute_bwd(out, None, rim, T, H)
    want = np.where(x == 0x8000, np.uint16(0), x)
    np.testing.assert_array_equal(g_x, want)


def test_unpermute_bwd_is_adjoint_of_unpermute():
    T, K, E, H = 24, 4, 6, 10
    rng = np.random.default_rng(41)
    idx, _, _ = _case(41, T, K, E, H, empty=True)
    rim, *_ = oracle.build_map(idx, E)
    probs = (2.0 ** -rng.integers(0, 3, size=(T, K))).astype(np.float32)
    rows = _small_int_bf16(rng, (T * K, H), lim=3)
    gy = _small_int_bf16(rng, (T, H), lim=3)
    y = oracle.unpermute(rows, probs, rim, T, H)
    g_rows, g_probs = oracle.unpermute_bwd(gy, rows, probs, rim)
    yf = oracle.f32_from_bf16(y).astype(np.float64)
    gyf = oracle.f32_from_bf16(gy).astype(np.float64)
    rf = oracle.f32_from_bf16(rows).astype(np.float64)
    inner = np.sum(yf * gyf)
    assert inner == np.sum(probs.astype(np.float64) * g_probs)     # d/dprobs
    mapped = rim[rim >= 0]
    assert inner == np.sum(oracle.f32_from_bf16(g_rows[mapped]).astype(np.float64) * rf[mapped])
    assert np.all(g_probs[rim < 0] == 0)
    # without probs the gradient is a plain copy to every row
    g_rows0, g0 = oracle.unpermute_bwd(gy, None, None, rim)
    assert g0 is None
    t, k = np.nonzero(rim >= 0)
    np.testing.assert_array_equal(g_rows0[rim[t, k]], gy[t])


def test_unpermute_bwd_rows_grad_is_one_rounded_product():
    T, K, E, H = 5, 3, 4, 7
    rng = np.random.default_rng(51)
    idx, probs, _ = _case(51, T, K, E, H)
    rim, *_ = oracle.build_map(idx, E)
    rows = _rand_bf16(rng, (T * K, H))
    gy = _rand_bf16(rng, (T, H))
    g_rows, g_probs = oracle.unpermute_bwd(gy, rows, probs, rim)
    for t in range(T):
        for k in range(K):
            r = rim[t, k]
            for h in range(H):
                prod = exact.round_f32(exact.Fraction(float(probs[t, k])) *
                                       exact.frac_of_bf16(int(gy[t, h])))
                assert int(g_rows[r, h]) == exact.bf16_of_f32(prod)
            dot = sum(exact.frac_of_bf16(int(rows[r, h])) * exact.frac_of_bf16(int(gy[t, h]))
                      for h in range(H))
            assert g_probs[t, k] == pytest.approx(float(dot), rel=1e-15, abs=1e-300)


# --------------------------------------------------------------------------
# chunk sort + pad
# --------------------------------------------------------------------------

def _brute_sort_pad(x, probs, sizes, order, G, align, out_rows):
    N, H = x.shape
    C = len(sizes)
    starts = np.concatenate([[0], np.cumsum(np.maximum(sizes, 0))])
    rows, offs = [], []
    for g in range(G):
        offs.append(len(rows))
        grp = []
        for c in order[g * (C // G):(g + 1) * (C // G)]:
            grp += list(range(starts[c], starts[c] + max(sizes[c], 0)))
        pad = (-len(grp)) % align
        rows += grp + [-1] * pad
    offs.append(len(rows))
    rows = [r if r < N else -1 for r in rows]
    rows = (rows + [-1] * out_rows)[:out_rows]
    row_map = np.array(rows, np.int32)
    out = np.zeros((out_rows, H), np.uint16)
    outp = np.zeros(out_rows, np.float32)
    ok = row_map >= 0
    out[ok] = x[row_map[ok]]
    outp[ok] = probs[row_map[ok]]
    return out, outp, row_map, np.array(offs, np.int64)


@pytest.mark.parametrize("seed", range(12))
def test_sort_chunks_pad_brute_force(seed):
    rng = np.random.default_rng(seed)
    G = int(rng.integers(1, 5))
    R = int(rng.integers(1, 4))
    C = G * R
    align = int(rng.choice([1, 2, 4, 8]))
    sizes = rng.integers(0, 6, size=C).astype(np.int32)
    sizes[rng.random(C) < 0.3] = 0
    if seed % 4 == 0:
        sizes[:R] = 0                                      # an all-empty group
    N = int(sizes.sum())
    H = 5
    order = rng.permutation(C).astype(np.int32)
    x = _rand_bf16(rng, (N, H))
    probs = rng.random(N).astype(np.float32)
    out_rows = int(N + G * (align - 1) + rng.integers(0, 4))
    got = oracle.sort_chunks_pad(x, probs, sizes, order, G, align, out_rows)
    want = _brute_sort_pad(x, probs, sizes, order, G, align, out_rows)
    for a, b in zip(got[:4], want):
        np.testing.assert_array_equal(a, b)
    assert not any(got[4].values())
    off = got[3]
    assert np.all(np.diff(off) % align == 0)
    # restore inverts sort+pad on the valid rows; pad rows are zero
    y, yp = oracle.unpad_restore(got[0], got[1], got[2], N)
    np.testing.assert_array_equal(y, x)
    np.testing.assert_array_equal(yp, probs)
    pad = got[2] < 0
    assert np.all(got[0][pad] == 0) and np.all(got[1][pad] == 0)


def test_sort_pad_backwards_are_adjoints():
    rng = np.random.default_rng(77)
    G, R, align, H = 3, 4, 4, 6
    C = G * R
    sizes = rng.integers(0, 7, size=C).astype(np.int32)
    N = int(sizes.sum())
    order = rng.permutation(C).astype(np.int32)
    out_rows = N + G * (align - 1)
    x = _small_int_bf16(rng, (N, H))
    probs = rng.integers(-3, 4, size=N).astype(np.float32)
    out, outp, row_map, _, _ = oracle.sort_chunks_pad(x, probs, sizes, order, G, align,
                                                      out_rows)
    Gd = _small_int_bf16(rng, (out_rows, H))
    Gp = rng.integers(-3, 4, size=out_rows).astype(np.float32)
    g_x, g_p = oracle.sort_chunks_pad_bwd(Gd, Gp, row_map, N)
    f = lambda a: oracle.f32_from_bf16(a).astype(np.float64)
    assert np.sum(f(out) * f(Gd)) == np.sum(f(x) * f(g_x))
    assert np.sum(outp.astype(np.float64) * Gp) == np.sum(probs.astype(np.float64) * g_p)
    # unpad+restore backward: pad rows get zero gradient, the rest is a gather
    gy = _small_int_bf16(rng, (N, H))
    gyp = rng.integers(-3, 4, size=N).astype(np.float32)
    g_pad, g_padp = oracle.unpad_restore_bwd(gy, gyp, row_map, N)
    y, yp = oracle.unpad_restore(out, outp, row_map, N)
    assert np.sum(f(y) * f(gy)) == np.sum(f(out) * f(g_pad))
    assert np.all(g_pad[row_map < 0] == 0) and np.all(g_padp[row_map < 0] == 0)
    assert np.sum(yp.astype(np.float64) * gyp) == np.sum(outp.astype(np.float64) * g_padp)


def test_sort_pad_flags():
    x = np.arange(10, dtype=np.uint16).reshape(10, 1)
    p = np.arange(10, dtype=np.float32)
    # negative split size counts as 0
    *_, fl = oracle.sort_chunks_pad(x, p, np.array([2, -1, 3, 1], np.int32),
                                    np.array([0, 1, 2, 3], np.int32), 2, 2, 12)
    assert fl["bad_split"] == 1 and fl["split_overflow"] == 0
    # sum of sizes above N: rows past N are padding
    out, _, rm, off, fl = oracle.sort_chunks_pad(x, p, np.array([6, 6], np.int32),
                                                 np.array([0, 1], np.int32), 1, 1, 12)
    assert fl["split_overflow"] == 1
    np.testing.assert_array_equal(rm, list(range(10)) + [-1, -1])
    # padded total above out_rows: dropped rows, offsets unclamped
    out, _, rm, off, fl = oracle.sort_chunks_pad(x, p, np.array([3, 3], np.int32),
                                                 np.array([0, 1], np.int32), 2, 4, 6)
    assert fl["rows_overflow"] == 1
    np.testing.assert_array_equal(off, [0, 4, 8])
    np.testing.assert_array_equal(rm, [0, 1, 2, -1, 3, 4])
    # chunk order out of range
    *_, fl = oracle.sort_chunks_pad(x, p, np.array([3, 3], np.int32),
                                    np.array([0, 9], np.int32), 1, 1, 6)
    assert fl["bad_order"] == 1


# --------------------------------------------------------------------------
# expert capacity (token dropping)
# --------------------------------------------------------------------------

def _brute_capacity(idx, E, cap):
    T, K = idx.shape
    keys = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K)
                  if 0 <= idx[t, k] < E)
    kept, seen = [], {}
    for e, t, k in keys:
        seen[e] = seen.get(e, 0) + 1
        if cap < 0 or seen[e] <= cap:
            kept.append((e, t, k))
    rim = -np.ones((T, K), np.int32)
    s2f = -np.ones(T * K, np.int32)
    for row, (e, t, k) in enumerate(kept):
        rim[t, k] = row
        s2f[row] = t * K + k
    counts = np.array([sum(1 for key in kept if key[0] == e) for e in range(E)], np.int32)
    return rim, s2f, counts, np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


@pytest.mark.parametrize("seed", range(30))
def test_build_map_capacity_brute_force(seed):
    rng = np.random.default_rng(500 + seed)
    T, K, E = int(rng.integers(0, 14)), int(rng.integers(1, 5)), int(rng.integers(1, 6))
    cap = int(rng.integers(-1, 6))
    idx = rng.integers(-1, E, size=(T, K)).astype(np.int32)
    got = oracle.build_map_capacity(idx, E, cap)
    for a, b in zip(got[:4], _brute_capacity(idx, E, cap)):
        np.testing.assert_array_equal(a, b)


def test_build_map_capacity_limits_reduce_to_plain_map():
    idx, _, _ = _case(3, 40, 4, 7, 1)
    plain = oracle.build_map(idx, 7)
    for cap in (-1, 160, 10**6):
        for a, b in zip(oracle.build_map_capacity(idx, 7, cap)[:4], plain[:4]):
            np.testing.assert_array_equal(a, b)
    rim, s2f, counts, offsets, _ = oracle.build_map_capacity(idx, 7, 0)
    assert np.all(rim == -1) and np.all(s2f == -1) and offsets[-1] == 0


def test_build_map_capacity_keeps_the_earliest_tokens():
    idx = np.array([[0, 1], [0, 2], [0, 1], [1, 0]], np.int32)
    rim, s2f, counts, offsets, _ = oracle.build_map_capacity(idx, 3, 2)
    np.testing.assert_array_equal(counts, [2, 2, 1])
    np.testing.assert_array_equal(rim, [[0, 2], [1, 4], [-1, 3], [-1, -1]])
    np.testing.assert_array_equal(s2f, [0, 2, 1, 5, 3, -1, -1, -1])


# --------------------------------------------------------------------------
# rank-ordered combine over EP ranks
# --------------------------------------------------------------------------

def test_bf16_from_f64_against_exact_rounding():
    rng = random.Random(8)
    vals = [0.0, -0.0, 1.0, 1.00390625, 1.01171875, -1.00390625, 2.0**-133, 2.0**-134,
            3 * 2.0**-134, 2.0**-126 * (1 - 2.0**-9), 3.3895313892515355e38,
            3.3961775292304e38, 3.4e38, 1e300, -1e300, 1e-300, 1.0 + 2.0**-8 + 2.0**-40]
    vals += [rng.uniform(-1, 1) * 2.0 ** rng.randint(-140, 130) for _ in range(3000)]
    got = oracle.bf16_from_f64(np.array(vals))
    for v, g in zip(vals, got):
        if v == 0:
            want = 0x8000 if math.copysign(1, v) < 0 else 0
        else:
            want = exact.round_bf16_bits(exact.Fraction(v))
        assert int(g) == want, (v, hex(int(g)), hex(want))


def _ep_exact(rows, probs, rim, idx, T, H, E, ep, bf16p, fp64):
    """The same tree with every rounding done exactly (fp32 via exact rounding,
    fp64 sums via exact rational then round to binary64)."""
    K = rim.shape[1]
    per = E // ep
    out = np.zeros((T, H), np.uint16)
    for t in range(T):
        for h in range(H):
            acc = exact.Fraction(0)
            accf = 0.0
            for r in range(ep):
                part = 0.0
                for k in range(K):
                    if rim[t, k] < 0 or idx[t, k] // per != r:
                        continue
                    x = _bf(rows[rim[t, k], h])
                    p = 1.0 if probs is None else float(probs[t, k])
                    part = exact.fma_f32(p, x, part)
                if bf16p:
                    part = float(exact.frac_of_bf16(exact.bf16_of_f32(part)))
                if fp64:
                    acc = exact.Fraction(float(acc + exact.Fraction(part)))  # binary64 add
                else:
                    accf = exact.fma_f32(1.0, part, accf)
            if fp64:
                out[t, h] = 0 if acc == 0 else exact.round_bf16_bits(acc)
            else:
                out[t, h] = exact.bf16_of_f32(accf)
    return out


@pytest.mark.parametrize("ep,bf16p,fp64", [(1, False, False), (2, True, False),
                                            (4, False, True), (4, True, True), (8, True, False)])
def test_unpermute_ep_exact_tree(ep, bf16p, fp64):
    T, K, E, H = 6, 4, 8, 7
    idx, probs, _ = _case(70 + ep, T, K, E, H, empty=True)
    rng = np.random.default_rng(90 + ep)
    rim, *_ = oracle.build_map(idx, E)
    rows = _rand_bf16(rng, (T * K, H))
    for p in (probs, None):
        got = oracle.unpermute_ep(rows, p, rim, idx, T, H, E, ep, bf16p, fp64)
        np.testing.assert_array_equal(got, _ep_exact(rows, p, rim, idx, T, H, E, ep, bf16p, fp64))


def test_unpermute_ep_fp64_sum_decides_a_bf16_tie():
    """Three ranks with partials 1, 2^-8 and +-2^-30 (one slot each, no probs):
    1 + 2^-8 lies exactly halfway between the bf16 values 1 and 1 + 2^-7.  The
    binary64 sum keeps the 2^-30 and rounds away from the tie; an fp32 sum
    drops it (half an fp32 ulp of 1 is 2^-24) and ties to even, giving 1."""
    bits = {1.0: 0x3F80, 2.0**-8: 0x3B80, 2.0**-30: 0x3080, -(2.0**-30): 0xB080,
            -1.0: 0xBF80, -(2.0**-8): 0xBB80}
    cases = [((1.0, 2.0**-8, 2.0**-30), 0x3F81, 0x3F80),
             ((1.0, 2.0**-8, -(2.0**-30)), 0x3F80, 0x3F80),
             ((-1.0, -(2.0**-8), -(2.0**-30)), 0xBF81, 0xBF80)]
    T, K, E, H = len(cases), 3, 3, 1
    idx = np.tile(np.arange(3, dtype=np.int32), (T, 1))          # slot k on rank k
    rim, *_ = oracle.build_map(idx, E)
    rows = np.zeros((T * K, H), np.uint16)
    for t, (vals, _, _) in enumerate(cases):
        for k in range(K):
            rows[rim[t, k], 0] = bits[vals[k]]
    y64 = oracle.unpermute_ep(rows, None, rim, idx, T, H, E, 3, False, True)
    y32 = oracle.unpermute_ep(rows, None, rim, idx, T, H, E, 3, False, False)
    assert [int(v) for v in y64[:, 0]] == [c[1] for c in cases]
    assert [int(v) for v in y32[:, 0]] == [c[2] for c in cases]


def test_unpermute_ep_with_one_rank_is_unpermute():
    T, K, E, H = 30, 4, 8, 16
    idx, probs, _ = _case(77, T, K, E, H, empty=True)
    rng = np.random.default_rng(78)
    rim, *_ = oracle.build_map(idx, E)
    rows = _rand_bf16(rng, (T * K, H))
    np.testing.assert_array_equal(oracle.unpermute_ep(rows, probs, rim, idx, T, H, E, 1),
                                  oracle.unpermute(rows, probs, rim, T, H))
    # bf16 partials with one rank: bf16(bf16(x)) == bf16(x)
    np.testing.assert_array_equal(oracle.unpermute_ep(rows, probs, rim, idx, T, H, E, 1, True),
                                  oracle.unpermute(rows, probs, rim, T, H))


# --------------------------------------------------------------------------
# router: fused top-k softmax
# --------------------------------------------------------------------------

def test_topk_softmax_selection_matches_stable_argsort():
    rng = np.random.default_rng(4)
    logits = rng.integers(-3, 4, size=(200, 24)).astype(np.float32)   # many ties
    idx, probs = oracle.topk_softmax(logits, 5)
    want = np.argsort(-logits, axis=1, kind="stable")[:, :5]
    np.testing.assert_array_equal(idx, want)


def test_topk_softmax_probs_within_fp32_bound_of_fp64():
    rng = np.random.default_rng(5)
    T, E, K = 300, 64, 8
    logits = (3 * rng.standard_normal((T, E))).astype(np.float32)
    idx, probs = oracle.topk_softmax(logits, K)
    sel = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    z = sel - sel[:, :1]
    p64 = np.exp(z) / np.exp(z).sum(1, keepdims=True)
    # each term: z rounding (|z| ulp/2), expf (<= 1 ulp), sum (K ulp), divide
    bound = (np.abs(z).max(1, keepdims=True) * 2.0**-24 + (K + 4) * 2.0**-24) * p64 * 2
    assert np.all(np.abs(probs - p64) <= bound)
    np.testing.assert_allclose(probs.sum(1), 1.0, rtol=K * 2.0**-23)


def test_topk_softmax_group_limited_brute_force():
    rng = np.random.default_rng(6)
    T, E, K, G, TG = 120, 32, 4, 8, 3
    logits = rng.integers(-4, 5, size=(T, E)).astype(np.float32)
    idx, _ = oracle.topk_softmax(logits, K, G, TG)
    per = E // G
    for t in range(T):
        score = [max(logits[t, g * per:(g + 1) * per]) for g in range(G)]
        groups = sorted(range(G), key=lambda g: (-score[g], g))[:TG]
        cand = [e for e in range(E) if e // per in groups]
        best = sorted(cand, key=lambda e: (-logits[t, e], e))[:K]
        assert list(idx[t]) == best


def test_topk_softmax_bwd_is_the_softmax_jacobian():
    rng = np.random.default_rng(7)
    T, E, K = 50, 16, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, probs = oracle.topk_softmax(logits, K)
    g = rng.standard_normal((T, K)).astype(np.float32)
    gl = oracle.topk_softmax_bwd(g, probs, idx, E)
    p = probs.astype(np.float64)
    for t in range(T):
        J = np.diag(p[t]) - np.outer(p[t], p[t])          # d p / d z, symmetric
        want = J @ g[t].astype(np.float64)
        got = gl[t, idx[t]].astype(np.float64)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-6)
        mask = np.ones(E, bool)
        mask[idx[t]] = False
        assert np.all(gl[t, mask] == 0)
        assert abs(got.sum()) < 1e-6


# --------------------------------------------------------------------------
# chunk sort + pad: explicit padded sizes, other token types
# --------------------------------------------------------------------------

def _brute_sort_pad_sizes(x, probs, sizes, order, G, padded_sizes, out_rows):
    N = x.shape[0]
    C = len(sizes)
    starts = np.concatenate([[0], np.cumsum(np.maximum(sizes, 0))])
    rows, offs = [], []
    for g in range(G):
        offs.append(len(rows))
        grp = []
        for c in order[g * (C // G):(g + 1) * (C // G)]:
            grp += list(range(starts[c], starts[c] + max(sizes[c], 0)))
        ps = max(int(padded_sizes[g]), 0)
        grp = grp[:ps]
        rows += grp + [-1] * (ps - len(grp))
    offs.append(len(rows))
    rows = [r if r < N else -1 for r in rows]
    row_map = np.array((rows + [-1] * out_rows)[:out_rows], np.int32)
    out = np.zeros((out_rows,) + x.shape[1:], x.dtype)
    ok = row_map >= 0
    out[ok] = x[row_map[ok]]
    return out, row_map, np.array(offs, np.int64)


@pytest.mark.parametrize("seed", range(10))
def test_sort_chunks_pad_explicit_sizes_brute_force(seed):
    rng = np.random.default_rng(200 + seed)
    G, R = int(rng.integers(1, 5)), int(rng.integers(1, 4))
    C = G * R
    sizes = rng.integers(0, 6, size=C).astype(np.int32)
    order = rng.permutation(C).astype(np.int32)
    N = int(sizes.sum())
    x = rng.standard_normal((N, 3)).astype(np.float32)          # fp32 tokens
    probs = rng.random(N).astype(np.float32)
    grows = np.array([sizes[order[g * R:(g + 1) * R]].sum() for g in range(G)])
    padded = (grows + rng.integers(-2, 5, size=G)).astype(np.int32)   # some too small
    out_rows = int(np.maximum(padded, 0).sum() + rng.integers(0, 3))
    out, out_p, rm, off, fl = oracle.sort_chunks_pad(x, probs, sizes, order, G, 1, out_rows,
                                                     padded_sizes=padded)
    want_out, want_rm, want_off = _brute_sort_pad_sizes(x, probs, sizes, order, G, padded,
                                                        out_rows)
    np.testing.assert_array_equal(out.view(np.uint32), want_out.view(np.uint32))
    np.testing.assert_array_equal(rm, want_rm)
    np.testing.assert_array_equal(off, want_off)
    assert fl["bad_padded"] == int(np.any(padded < grows))


def test_sort_chunks_pad_is_dtype_agnostic():
    rng = np.random.default_rng(9)
    sizes = np.array([3, 0, 4, 2], np.int32)
    order = np.array([2, 0, 3, 1], np.int32)
    x32 = rng.standard_normal((9, 5)).astype(np.float32)
    x16 = x32.view(np.uint16)                                   # same bits, 2x wider
    a = oracle.sort_chunks_pad(x32, None, sizes, order, 2, 4, 16)
    b = oracle.sort_chunks_pad(x16, None, sizes, order, 2, 4, 16)
    np.testing.assert_array_equal(a[0].view(np.uint16), b[0])
    y, _ = oracle.unpad_restore(a[0], None, a[2], 9)
    np.testing.assert_array_equal(y.view(np.uint32), x32.view(np.uint32))
