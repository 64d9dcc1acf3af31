"""Row ops on special bf16 values, bit-exact against the oracle: +-0 (a sum
from +0 turns a lone -0 into +0), subnormals (fp32 holds every bf16
subnormal exactly, and no flush to zero is allowed), and values near the
bf16 maximum whose slot sums overflow to +-inf.  Inputs are finite, so a
single slot-order chain never makes a NaN (products of a probability in
(0,1] and a finite row cannot overflow, and an infinite running sum never
meets an infinity of the other sign); the rank-ordered combine can, when two
ranks' partials overflow with opposite signs."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import unpermute_routing_indices_gb300 as mp
from tests.gpu_util import d, h

pytestmark = pytest.mark.gpu

SPECIAL = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x7F7F, 0xFF7F, 0x7F00,
                    0xFF00, 0x3F80, 0xBF80], np.uint16)


def _case(seed, T=600, K=6, E=24, H=64):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < 0.1] = -1
    probs = rng.random((T, K)).astype(np.float32)
    probs[rng.random((T, K)) < 0.3] = 1.0
    probs[probs == 0] = 0.5
    rows = SPECIAL[rng.integers(0, SPECIAL.size, size=(T * K, H))]
    x = SPECIAL[rng.integers(0, SPECIAL.size, size=(T, H))]
    g = SPECIAL[rng.integers(0, SPECIAL.size, size=(T, H))]
    return idx, probs, rows, x, g, E


@pytest.mark.parametrize("seed", [1, 2])
def test_row_ops_on_special_values(seed):
    idx, probs, rows, x, g, E = _case(seed)
    T, H = x.shape
    rim, *_ = mp.mp_build_map(d(idx), E)
    o_rim, *_ = oracle.build_map(idx, E)
    mapped = np.sort(o_rim[o_rim >= 0])
    # combine, with and without probs
    for p in (probs, None):
        y = mp.mp_unpermute(d(rows), rim, None if p is None else d(p))
        np.testing.assert_array_equal(h(y), oracle.unpermute(rows, p, o_rim, T, H))
    # permute and its backward (a plain slot sum)
    out, _ = mp.mp_permute(d(x), rim)
    o_out, _ = oracle.permute(x, None, o_rim)
    np.testing.assert_array_equal(h(out)[mapped], o_out[mapped])
    g_x, _ = mp.mp_permute_bwd(d(rows), rim)
    np.testing.assert_array_equal(h(g_x), oracle.permute_bwd(rows, None, o_rim, T, H)[0])
    # unpermute backward: each row gradient is one rounded fp32 product
    g_rows, _ = mp.mp_unpermute_bwd(d(g), rim, d(rows), d(probs))
    o_grows, _ = oracle.unpermute_bwd(g, rows, probs, o_rim)
    np.testing.assert_array_equal(h(g_rows)[mapped], o_grows[mapped])
    # the outputs do hold the special cases
    y = oracle.unpermute(rows, probs, o_rim, T, H)
    assert np.any(y == 0x7F80) and np.any(y == 0xFF80)           # overflow to +-inf
    assert np.any((y & 0x7F80) == 0) and np.any(y == 0x0000)     # subnormal / zero results


# the 8-slot and 16-slot forms on token groups, and one token per CTA
@pytest.mark.parametrize("K,H", [(6, 64), (12, 64), (6, 1032)])
@pytest.mark.parametrize("bf16p,fp64", [(False, False), (True, False), (False, True),
                                         (True, True)])
def test_ep_combine_on_special_values(bf16p, fp64, K, H):
    idx, probs, rows, _, _, E = _case(7, K=K, E=24, H=H)
    T, H = idx.shape[0], rows.shape[1]
    rim, *_ = mp.mp_build_map(d(idx), E)
    o_rim, *_ = oracle.build_map(idx, E)
    for p in (probs, None):
        got = h(mp.mp_unpermute_ep(d(rows), rim, d(idx), E, 4, None if p is None else d(p),
                                   bf16_partials=bf16p, fp64_cross_rank=fp64))
        want = oracle.unpermute_ep(rows, p, o_rim, idx, T, H, E, 4, bf16p, fp64)
        # two ranks' partials may overflow to opposite infinities: their sum is a
        # NaN, whose payload is not specified; every other element is bit-exact
        nan = _is_nan(want)
        assert np.array_equal(_is_nan(got), nan)
        np.testing.assert_array_equal(got[~nan], want[~nan])


def _is_nan(bits):
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)
