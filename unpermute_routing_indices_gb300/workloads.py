"""Seeded synthetic inputs for the permute / unpermute path.

This module only draws inputs: router indices and probabilities, hidden rows,
gradients and chunk sizes.  It holds none of the path's arithmetic (no map,
no permutation, no combine) and imports neither the CUDA library nor the
oracle, so both sides can be fed the same arrays.

Everything is numpy with ``default_rng(seed)`` (PCG64, stable across numpy
versions and machines).  bf16 tensors are returned as ``uint16`` bit patterns;
the float32 -> bf16 rounding of the normal draws is delegated to
``torch.Tensor.to(torch.bfloat16)``.

Workloads (sizes from the routing problem statements on the pages):
  tiny     T=16,    H=64,   E=32,  K=4   logits ~N(0,1), distinct top-4
  mid      T=4096,  H=2048, E=64,  K=6   logits ~N(0,1)
  skewed   T=16384, H=4096, E=128, K=8   logits ~N(0,1) + 2*ln(Zipf(1.2) weight)
  chunks   N=8192 / 32768, H=2048, 16 experts x 8 rank chunks, align 128
  large    T=32768, H=7168, E=256, K=8   8 groups, top-4 groups, top-8 in them
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 1000


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) draws rounded to bf16; returns the uint16 bit patterns."""
    import torch

    f = rng.standard_normal(size=shape, dtype=np.float32)
    t = torch.from_numpy(f).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def topk_softmax(logits: np.ndarray, K: int):
    """Top-K experts per token (larger logit first, lower index on ties) and the
    fp32 softmax over the K selected logits."""
    order = np.argsort(-logits, axis=1, kind="stable")[:, :K]
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float32)
    m = sel.max(axis=1, keepdims=True)
    e = np.exp(sel - m, dtype=np.float32)
    probs = (e / e.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    return order.astype(np.int32), probs


def zipf_bias(rng: np.random.Generator, E: int, s: float = 1.2) -> np.ndarray:
    """bias_e = 2 ln w_pi(e), w_i = i^-s / sum_j j^-s, pi a seeded permutation."""
    i = np.arange(1, E + 1, dtype=np.float64)
    w = i ** (-s)
    w /= w.sum()
    perm = rng.permutation(E)
    return (2.0 * np.log(w[perm])).astype(np.float32)


def group_limited_topk(logits: np.ndarray, K: int, n_groups: int, topk_groups: int):
    """Keep the top `topk_groups` expert groups by their largest logit, then the
    top-K experts inside them; softmax over the K selected logits."""
    T, E = logits.shape
    gmax = logits.reshape(T, n_groups, E // n_groups).max(axis=2)
    keep = np.argsort(-gmax, axis=1, kind="stable")[:, :topk_groups]
    mask = np.zeros((T, n_groups), dtype=bool)
    np.put_along_axis(mask, keep, True, axis=1)
    masked = np.where(np.repeat(mask, E // n_groups, axis=1), logits, -np.inf)
    return topk_softmax(masked.astype(np.float32), K)


# --------------------------------------------------------------------------
# routed permute / unpermute workloads
# --------------------------------------------------------------------------

ROUTED = {
    "tiny": dict(T=16, H=64, E=32, K=4, kind="uniform", seed=SEED_BASE + 1),
    "mid": dict(T=4096, H=2048, E=64, K=6, kind="uniform", seed=SEED_BASE + 2),
    "skewed": dict(T=16384, H=4096, E=128, K=8, kind="zipf", seed=SEED_BASE + 3),
    "large": dict(T=32768, H=7168, E=256, K=8, kind="grouped", seed=SEED_BASE + 5,
                  n_groups=8, topk_groups=4),
}


def router_logits(name: str, T: int | None = None, seed: int | None = None) -> np.ndarray:
    """The fp32 router logits [T,E] a named routed workload draws its routing from."""
    cfg = ROUTED[name]
    T = cfg["T"] if T is None else T
    rng = _rng(cfg["seed"] if seed is None else seed)
    E = cfg["E"]
    if cfg["kind"] == "zipf":
        bias = zipf_bias(rng, E)
        return (rng.standard_normal((T, E), dtype=np.float32) + bias[None, :]).astype(np.float32)
    return rng.standard_normal((T, E), dtype=np.float32)


def routing(name: str, T: int | None = None, seed: int | None = None):
    """(idx[T,K] int32, probs[T,K] f32, E) for a named routed workload.
    T may be overridden (a leading slice of the same distribution)."""
    cfg = ROUTED[name]
    E, K = cfg["E"], cfg["K"]
    logits = router_logits(name, T=T, seed=seed)
    if cfg["kind"] == "grouped":
        idx, probs = group_limited_topk(logits, K, cfg["n_groups"], cfg["topk_groups"])
    else:
        idx, probs = topk_softmax(logits, K)
    return idx, probs, E


def routed(name: str, T: int | None = None, H: int | None = None,
           grads: bool = True, seed: int | None = None) -> dict:
    """Full inputs of a routed workload: idx, probs, x, and (if grads) the
    upstream gradients g_y[T,H] (bf16) and g_rows_probs[T*K] (f32)."""
    cfg = ROUTED[name]
    T = cfg["T"] if T is None else T
    H = cfg["H"] if H is None else H
    base = cfg["seed"] if seed is None else seed
    idx, probs, E = routing(name, T=T, seed=base)
    rng = _rng(base + 100)
    out = dict(name=name, T=T, H=H, E=E, K=cfg["K"], idx=idx, probs=probs,
               x=bf16_normal(rng, (T, H)))
    if grads:
        out["g_y"] = bf16_normal(rng, (T, H))
        out["g_out_probs"] = rng.standard_normal(T * cfg["K"], dtype=np.float32)
    return out


def random_rows(rows: int, H: int, seed: int) -> np.ndarray:
    """Independent bf16 rows (e.g. an expert output to unpermute)."""
    return bf16_normal(_rng(seed), (rows, H))


# --------------------------------------------------------------------------
# chunk sort + pad workload
# --------------------------------------------------------------------------

CHUNKS = dict(H=2048, experts=16, ranks=8, align=128, empty_frac=1 / 8,
              seed=SEED_BASE + 4)


def chunk_layout(N: int, experts: int = 16, ranks: int = 8, empty_frac: float = 1 / 8,
                 seed: int = SEED_BASE + 4):
    """Chunk sizes and order for N dispatched rows.

    Input chunks arrive rank-major (chunk c = r*experts + e, as after an
    all-to-all); the order groups them expert-major, chunk_order[e*ranks + r]
    = r*experts + e.  Sizes are Multinomial(N, w) with a seeded fraction of
    chunks at weight 0 (empty) and the rest equal."""
    rng = _rng(seed)
    C = experts * ranks
    w = np.ones(C, dtype=np.float64)
    n_empty = int(round(C * empty_frac))
    w[rng.choice(C, size=n_empty, replace=False)] = 0.0
    w /= w.sum()
    sizes = rng.multinomial(N, w).astype(np.int32)
    e = np.arange(experts)[:, None]
    r = np.arange(ranks)[None, :]
    order = (r * experts + e).reshape(-1).astype(np.int32)
    return sizes, order


def chunks(N: int, H: int = CHUNKS["H"], seed: int = CHUNKS["seed"], grads: bool = True
           ) -> dict:
    sizes, order = chunk_layout(N, CHUNKS["experts"], CHUNKS["ranks"],
                                CHUNKS["empty_frac"], seed)
    rng = _rng(seed + 100)
    out = dict(N=N, H=H, C=sizes.shape[0], G=CHUNKS["experts"], align=CHUNKS["align"],
               split_sizes=sizes, chunk_order=order, x=bf16_normal(rng, (N, H)),
               probs=rng.random(N, dtype=np.float32))
    if grads:
        out["g_seed"] = seed + 200
    return out


def padded_rows_bound(N: int, G: int, align: int) -> int:
    """Capacity that fits any split of N rows into G groups padded to align."""
    return N + G * (align - 1)


# --------------------------------------------------------------------------
# counter-based rows: any row can be drawn alone, on either side
# --------------------------------------------------------------------------
#
# bits(i, h) = fmix32((seed * 0x9E3779B1 + i * H + h) mod 2^32), the 32-bit
# finaliser of MurmurHash3 (x ^= x>>16; x *= 0x85EBCA6B; x ^= x>>13;
# x *= 0xC2B2AE35; x ^= x>>16).  The bf16 value keeps the hash's sign bit and
# its 7 low mantissa bits, with an exponent in [120, 127]: magnitudes in
# [2^-7, 2).  numpy and torch evaluate the same integer recipe, so a test can
# fill a full-size tensor on the GPU and rebuild just the rows it samples on
# the host.

_M32 = 0xFFFFFFFF


def _fmix32_np(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint64) & _M32
    x ^= x >> np.uint64(16)
    x = (x * np.uint64(0x85EBCA6B)) & np.uint64(_M32)
    x ^= x >> np.uint64(13)
    x = (x * np.uint64(0xC2B2AE35)) & np.uint64(_M32)
    x ^= x >> np.uint64(16)
    return x


def _hash_to_bf16_np(hv: np.ndarray) -> np.ndarray:
    sign = (hv >> np.uint64(16)) & np.uint64(0x8000)
    exp = (np.uint64(120) + ((hv >> np.uint64(7)) & np.uint64(7))) << np.uint64(7)
    return (sign | exp | (hv & np.uint64(0x7F))).astype(np.uint16)


def hashed_rows(row_ids, H: int, seed: int) -> np.ndarray:
    """Rows `row_ids` (any order) of the counter-based bf16 tensor, as uint16."""
    r = np.asarray(row_ids, dtype=np.uint64).reshape(-1, 1)
    ctr = (np.uint64(seed) * np.uint64(0x9E3779B1) + r * np.uint64(H)
           + np.arange(H, dtype=np.uint64)[None, :])
    return _hash_to_bf16_np(_fmix32_np(ctr))


def hashed_rows_torch(n_rows: int, H: int, seed: int, device, chunk_rows: int = 8192):
    """The whole [n_rows, H] counter-based tensor as torch.bfloat16 on `device`
    (integer work in int64 with explicit 32-bit masks)."""
    import torch

    out = torch.empty((n_rows, H), dtype=torch.int16, device=device)
    cols = torch.arange(H, dtype=torch.int64, device=device)
    base = (seed * 0x9E3779B1) & _M32
    for r0 in range(0, n_rows, chunk_rows):
        r1 = min(n_rows, r0 + chunk_rows)
        rows = torch.arange(r0, r1, dtype=torch.int64, device=device)
        x = (base + rows[:, None] * H + cols[None, :]) & _M32
        x = x ^ (x >> 16)
        x = (x * 0x85EBCA6B) & _M32
        x = x ^ (x >> 13)
        x = (x * 0xC2B2AE35) & _M32
        x = x ^ (x >> 16)
        sign = (x >> 16) & 0x8000
        exp = (120 + ((x >> 7) & 7)) << 7
        bits = sign | exp | (x & 0x7F)
        out[r0:r1] = (bits - ((bits >> 15) << 16)).to(torch.int16)
    return out.view(torch.bfloat16)
