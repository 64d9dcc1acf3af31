"""The autograd layer and the zero fill, through the C ABI, against the oracle.

Forward values and gradients are bit-exact against the oracle (rows, combine,
g_x, g_rows, router gradient, chunk sort / restore) and the probability
gradient of the combine is within the fp32 summation bound of the oracle's
fp64 sum.  Rows past the routed count are zero in the permuted output and in
its gradient.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import autograd as ag
from unpermute_routing_indices_gb300 import workloads as wl
from tests.gpu_util import DEV, d, gprobs_bound, h

pytestmark = pytest.mark.gpu


def f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# zero fill from a device-held start row
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape,dtype,offset", [
    ((300, 64), torch.bfloat16, 0),     # 16-byte stores
    ((300, 6), torch.bfloat16, 0),      # 12-byte rows: 4-byte stores
    ((301, 3), torch.bfloat16, 0),      # 6-byte rows: byte stores
    ((777,), torch.float32, 0),         # probs: 4-byte rows
    ((129, 64), torch.bfloat16, 1),     # 2-byte offset: not 16-byte aligned
    ((5003, 24), torch.bfloat16, 0),    # 3 vectors a row: a ragged last chunk
    ((20000, 1024), torch.bfloat16, 0), # more units than one pass of the grid
])
@pytest.mark.parametrize("start", [-5, 0, 7, "last", "rows", "past"])
def test_zero_rows_from(shape, dtype, offset, start):
    n = int(np.prod(shape))
    base = torch.empty(n + offset, dtype=dtype, device=DEV)
    buf = base[offset:].view(shape)
    ref = torch.arange(1, n + 1, device=DEV).to(dtype).view(shape)
    buf.copy_(ref)
    rows = shape[0]
    s = {"last": rows - 1, "rows": rows, "past": rows + 10}.get(start, start)
    mp.mp_zero_rows_from(buf, torch.tensor([s], dtype=torch.int32, device=DEV))
    c = min(max(s, 0), rows)
    assert torch.equal(buf[:c], ref[:c])
    assert bool((buf[c:] == 0).all())


# --------------------------------------------------------------------------
# dispatch -> expert rows -> combine, forward and backward
# --------------------------------------------------------------------------

def _case(T, empty, seed=3):
    w = wl.routed("mid", T=T)
    if empty:
        rng = np.random.default_rng(seed)
        w["idx"][rng.random(w["idx"].shape) < 0.15] = -1
    w["rows_in"] = wl.random_rows(T * w["K"], w["H"], seed=7)
    w["g_rows_in"] = wl.random_rows(T * w["K"], w["H"], seed=8)
    return w


@pytest.mark.parametrize("T,empty,capacity", [(1234, True, None), (2000, False, 150),
                                              (999, True, 60), (512, False, None)])
def test_permute_unpermute_autograd(T, empty, capacity):
    w = _case(T, empty)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    if capacity is None:
        o_rim, _, _, o_off, _ = oracle.build_map(w["idx"], E)
        R = T * K
    else:
        o_rim, _, _, o_off, _ = oracle.build_map_capacity(w["idx"], E, capacity)
        R = min(T * K, E * capacity)
    routed = int(o_off[-1])

    # dispatch forward and backward
    x = d(w["x"]).requires_grad_()
    probs = d(w["probs"]).requires_grad_()
    rows, rows_p, dsp = ag.permute(x, d(w["idx"]), E, probs, capacity=capacity)
    assert rows.shape == (R, H) and dsp.num_rows == R
    np.testing.assert_array_equal(h(dsp.row_id_map), o_rim)
    o_rows, o_rows_p = oracle.permute(w["x"], w["probs"], o_rim, out_rows=R)
    np.testing.assert_array_equal(h(rows), o_rows)          # tail rows are zero on both
    np.testing.assert_array_equal(h(rows_p), o_rows_p)
    g_rows_in = w["g_rows_in"][:R]
    g_rp = w["g_out_probs"].ravel()[:R].copy() if w["g_out_probs"].size >= R else \
        np.random.default_rng(5).random(R).astype(np.float32)
    torch.autograd.backward([rows, rows_p], [d(g_rows_in), d(g_rp)])
    o_gx, o_gp = oracle.permute_bwd(g_rows_in, g_rp, o_rim, T, H)
    np.testing.assert_array_equal(h(x.grad), o_gx)
    np.testing.assert_array_equal(h(probs.grad), o_gp)

    # combine forward and backward over independent expert rows, whose tail
    # rows hold nonzero values that must not reach y and must get zero grad
    ex = d(w["rows_in"][:R]).requires_grad_()
    probs2 = d(w["probs"]).requires_grad_()
    y = ag.unpermute(ex, dsp, probs2)
    np.testing.assert_array_equal(h(y), oracle.unpermute(w["rows_in"][:R], w["probs"], o_rim,
                                                         T, H))
    y.backward(d(w["g_y"]))
    o_grows, o_gprobs = oracle.unpermute_bwd(w["g_y"], w["rows_in"][:R], w["probs"], o_rim,
                                             out_rows=R)
    np.testing.assert_array_equal(h(ex.grad), o_grows)      # zero past the routed rows
    assert not h(ex.grad)[routed:].any()
    gp = h(probs2.grad).astype(np.float64)
    rf = f32(w["rows_in"][:R])[np.maximum(o_rim, 0)]
    bound = gprobs_bound(rf, f32(w["g_y"])[:, None, :], o_gprobs)
    assert np.all(np.abs(gp - o_gprobs) <= bound)
    assert np.all(gp[o_rim < 0] == 0)


def test_unpermute_without_probs_and_ep_form():
    w = _case(1500, True)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    o_rim, *_ = oracle.build_map(w["idx"], E)
    _, _, dsp = ag.permute(d(w["x"]), d(w["idx"]), E)
    ex = d(w["rows_in"]).requires_grad_()
    y = ag.unpermute(ex, dsp)
    np.testing.assert_array_equal(h(y), oracle.unpermute(w["rows_in"], None, o_rim, T, H))
    y.backward(d(w["g_y"]))
    o_grows, _ = oracle.unpermute_bwd(w["g_y"], None, None, o_rim)
    np.testing.assert_array_equal(h(ex.grad), o_grows)
    # rank-ordered form: its own forward, the combine's gradient
    ex2 = d(w["rows_in"]).requires_grad_()
    probs = d(w["probs"]).requires_grad_()
    y2 = ag.unpermute_ep(ex2, dsp, 8, probs, bf16_partials=True, fp64_cross_rank=True)
    want = oracle.unpermute_ep(w["rows_in"], w["probs"], o_rim, w["idx"], T, H, E, 8, True, True)
    np.testing.assert_array_equal(h(y2), want)
    y2.backward(d(w["g_y"]))
    o_grows, _ = oracle.unpermute_bwd(w["g_y"], w["rows_in"], w["probs"], o_rim)
    np.testing.assert_array_equal(h(ex2.grad), o_grows)


def test_router_autograd():
    rng = np.random.default_rng(4)
    T, E, K = 3000, 64, 6
    logits_np = rng.standard_normal((T, E)).astype(np.float32)
    logits = d(logits_np).requires_grad_()
    idx, probs = ag.topk_softmax(logits, K)
    o_idx, o_probs = oracle.topk_softmax(logits_np, K)
    np.testing.assert_array_equal(h(idx), o_idx)
    g = rng.standard_normal((T, K)).astype(np.float32)
    probs.backward(d(g))
    np.testing.assert_array_equal(h(logits.grad), oracle.topk_softmax_bwd(g, h(probs), o_idx, E))
    assert not idx.requires_grad


# --------------------------------------------------------------------------
# chunk sort + pad and its restore
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,short", [(8192, 0), (4096, 300)])
def test_sort_pad_restore_autograd(N, short):
    c = wl.chunks(N)
    G, align, H = c["G"], c["align"], c["H"]
    sizes = c["split_sizes"].copy()
    if short:                                   # the last rows of x belong to no chunk
        nz = np.flatnonzero(sizes)
        for i in nz[::-1]:
            take = min(short, sizes[i])
            sizes[i] -= take
            short -= take
            if short == 0:
                break
    out_rows = wl.padded_rows_bound(N, G, align)
    x = d(c["x"]).requires_grad_()
    p = d(c["probs"]).requires_grad_()
    out, out_p, row_map, goff = ag.sort_chunks_pad(x, d(sizes), d(c["chunk_order"]), G, align,
                                                   out_rows, p)
    o_out, o_out_p, o_map, o_goff, _ = oracle.sort_chunks_pad(
        c["x"], c["probs"], sizes, c["chunk_order"], G, align, out_rows)
    np.testing.assert_array_equal(h(out), o_out)
    np.testing.assert_array_equal(h(out_p), o_out_p)
    np.testing.assert_array_equal(h(row_map), o_map)
    np.testing.assert_array_equal(h(goff), o_goff)
    y, y_p = ag.unpad_restore(out, row_map, N, out_p)
    named = int(sizes.sum())
    np.testing.assert_array_equal(h(y)[:named], c["x"][:named])
    assert not h(y)[named:].any() and not h(y_p)[named:].any()
    g = wl.random_rows(N, H, seed=11)
    gpr = np.random.default_rng(12).random(N).astype(np.float32)
    torch.autograd.backward([y, y_p], [d(g), d(gpr)])
    # restore o sort is the identity on named rows, so is its gradient
    np.testing.assert_array_equal(h(x.grad)[:named], g[:named])
    np.testing.assert_array_equal(h(p.grad)[:named], gpr[:named])
    assert not h(x.grad)[named:].any() and not h(p.grad)[named:].any()
