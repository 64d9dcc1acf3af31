"""No op writes outside its outputs, or into the parts it promises to leave.

Every output tensor is a view into the middle of a larger buffer whose guard
regions before and after hold a sentinel pattern; after the call the guards
must be unchanged.  Where the API leaves part of an output unwritten (the
permuted rows that no slot maps to, the rows of y that unpad+restore does not
name), that part must still hold the sentinel.  Sizes have ragged tails and
cover every map form (one CTA, one cluster, two kernels), the 16-byte vector
path and the element path (odd H)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import workloads as wl
from tests.gpu_util import DEV, d

pytestmark = pytest.mark.gpu

GUARD = 256            # elements of guard on each side (a multiple of 16 bytes for every dtype)
SENT = {torch.bfloat16: -12288.0, torch.float32: -7.5e33, torch.int32: -0x5A5A5A5B,
        torch.int64: -0x5A5A5A5A5A5A5A5B}


class Guarded:
    """A tensor of `shape` inside a sentinel-filled buffer."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) if len(shape) else 1
        self.base = torch.full((n + 2 * GUARD,), SENT[dtype], dtype=dtype, device=DEV)
        self.t = self.base[GUARD:GUARD + n].view(shape)
        self.n = n

    def guards_intact(self):
        s = SENT[self.base.dtype]
        before, after = self.base[:GUARD], self.base[GUARD + self.n:]
        return bool((before == s).all()) and bool((after == s).all())

    def sentinel(self):
        return self.t == SENT[self.t.dtype]


def _routing(T, K, E, empty, seed):
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    idx[rng.random((T, K)) < empty] = -1
    probs = rng.random((T, K)).astype(np.float32)
    return idx, probs


@pytest.mark.parametrize("T,K,E,H", [(301, 8, 64, 136),       # one-CTA map
                                     (2501, 6, 64, 40),       # cluster map
                                     (9001, 8, 128, 264),     # two-kernel map
                                     (777, 4, 16, 37)])       # element path
def test_routed_ops_stay_inside_their_outputs(T, K, E, H):
    idx, probs = _routing(T, K, E, 0.15, T + H)
    R = T * K
    di, dp = d(idx), d(probs)
    rim, s2f = Guarded((T, K), torch.int32), Guarded((R,), torch.int32)
    counts, offsets = Guarded((E,), torch.int32), Guarded((E + 1,), torch.int32)
    mp.mp_build_map(di, E, row_id_map=rim.t, sorted_to_flat=s2f.t, counts=counts.t,
                    offsets=offsets.t)
    for g in (rim, s2f, counts, offsets):
        assert g.guards_intact()
    routed = int(offsets.t[-1].item())

    x = d(wl.random_rows(T, H, 1))
    out, out_p = Guarded((R, H), torch.bfloat16), Guarded((R,), torch.float32)
    mp.mp_permute(x, rim.t, dp, out=out.t, out_probs=out_p.t)
    assert out.guards_intact() and out_p.guards_intact()
    # rows past the routed ones are no slot's: left as they were
    assert bool(out.sentinel()[routed:].all()) and bool(out_p.sentinel()[routed:].all())
    assert not bool(out.sentinel()[:routed].any())

    rows = d(wl.random_rows(R, H, 2))
    y = Guarded((T, H), torch.bfloat16)
    mp.mp_unpermute(rows, rim.t, dp, out=y.t)
    assert y.guards_intact()
    y_ep = Guarded((T, H), torch.bfloat16)
    if E % 8 == 0:
        mp.mp_unpermute_ep(rows, rim.t, di, E, 8, dp, fp64_cross_rank=True, out=y_ep.t)
        assert y_ep.guards_intact()

    gy = d(wl.random_rows(T, H, 3))
    g_rows, g_probs = Guarded((R, H), torch.bfloat16), Guarded((T, K), torch.float32)
    mp.mp_unpermute_bwd(gy, rim.t, rows, dp, g_rows=g_rows.t, g_probs=g_probs.t)
    assert g_rows.guards_intact() and g_probs.guards_intact()
    assert bool(g_rows.sentinel()[routed:].all())

    g_x, g_xp = Guarded((T, H), torch.bfloat16), Guarded((T, K), torch.float32)
    mp.mp_permute_bwd(rows, rim.t, d(np.ones(R, np.float32)), g_x=g_x.t, g_probs=g_xp.t)
    assert g_x.guards_intact() and g_xp.guards_intact()

    z = Guarded((R, H), torch.bfloat16)
    z.t.copy_(rows)
    mp.mp_zero_rows_from(z.t, offsets.t[-1:])
    assert z.guards_intact()
    assert bool((z.t[routed:] == 0).all()) and torch.equal(z.t[:routed], rows[:routed])


@pytest.mark.parametrize("T,E,K,G,TG", [(333, 128, 8, 1, 1), (257, 256, 8, 8, 4),
                                        (99, 40, 5, 1, 1)])
def test_router_stays_inside_its_outputs(T, E, K, G, TG):
    logits = d(np.random.default_rng(T).standard_normal((T, E)).astype(np.float32))
    idx, probs = Guarded((T, K), torch.int32), Guarded((T, K), torch.float32)
    mp.mp_topk_softmax(logits, K, n_groups=G, topk_groups=TG, idx=idx.t, probs=probs.t)
    assert idx.guards_intact() and probs.guards_intact()
    g = d(np.ones((T, K), np.float32))
    gl = Guarded((T, E), torch.float32)
    mp.mp_topk_softmax_bwd(g, probs.t, idx.t, E, g_logits=gl.t)
    assert gl.guards_intact()


@pytest.mark.parametrize("N,H,G,R,align", [(5000, 264, 16, 8, 128), (999, 37, 4, 3, 8)])
def test_chunk_ops_stay_inside_their_outputs(N, H, G, R, align):
    C = G * R
    rng = np.random.default_rng(N)
    sizes = rng.multinomial(N, np.ones(C) / C).astype(np.int32)
    order = rng.permutation(C).astype(np.int32)
    out_rows = wl.padded_rows_bound(N, G, align) + 5
    x = d(wl.random_rows(N, H, 4))
    pr = d(rng.random(N).astype(np.float32))
    out, out_p = Guarded((out_rows, H), torch.bfloat16), Guarded((out_rows,), torch.float32)
    row_map, goff = Guarded((out_rows,), torch.int32), Guarded((G + 1,), torch.int64)
    mp.mp_sort_chunks_pad(x, d(sizes), d(order), G, align, out_rows, pr, out=out.t,
                          out_probs=out_p.t, row_map=row_map.t, group_off=goff.t)
    for g_ in (out, out_p, row_map, goff):
        assert g_.guards_intact()
    # y holds N + 7 rows: the restore names only the first N
    y, y_p = Guarded((N + 7, H), torch.bfloat16), Guarded((N + 7,), torch.float32)
    mp.mp_unpad_restore(out.t, row_map.t, N, out_p.t, y=y.t[:N], y_probs=y_p.t[:N])
    assert y.guards_intact() and y_p.guards_intact()
    assert torch.equal(y.t[:N], x) and bool(y.sentinel()[N:].all())
    g_pad, g_padp = Guarded((out_rows, H), torch.bfloat16), Guarded((out_rows,), torch.float32)
    mp.mp_unpad_restore_bwd(x, row_map.t, pr, g_padded=g_pad.t, g_padded_probs=g_padp.t)
    assert g_pad.guards_intact() and g_padp.guards_intact()
