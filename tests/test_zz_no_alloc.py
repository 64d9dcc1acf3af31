"""The allocation-free routing map, called through the C ABI.

mp_build_map_noalloc is for callers that cannot call cudaMalloc: an inference
runtime or plugin that fixes all device memory at start-up, a framework whose
allocator owns the device memory, or a path that must not risk cudaMalloc's
implicit device synchronisation.  Its scratch is a static device array inside
libmp, shared by every call.  These tests call it directly through ctypes and
require its outputs to equal, bit for bit, those of mp_build_map (which takes
a caller-provided workspace) on consecutive calls with different routing, so a
stale array from the previous call would show.  This file is collected last
and does not depend on any other test having run.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import _lib
from unpermute_routing_indices_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, idx, E):
    T, K = idx.shape
    fill = -7                      # anything the call fails to write shows up
    rim = torch.full((T, K), fill, dtype=torch.int32, device=DEV)
    s2f = torch.full((T * K,), fill, dtype=torch.int32, device=DEV)
    counts = torch.full((E,), fill, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1,), fill, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    code = lib.mp_build_map_noalloc(_p(idx), T, K, E, _p(rim), _p(s2f), _p(counts),
                                    _p(offsets), _p(status), stream)
    assert code == 0, lib.mp_status_string(code)
    return rim, s2f, counts, offsets, status


def test_noalloc_map_matches_the_workspace_map_on_consecutive_calls():
    lib = _lib.load()
    torch.cuda.init()
    cases = [wl.routing("skewed"), wl.routing("mid"), wl.routing("skewed", seed=4242)]
    rng = np.random.default_rng(8)
    # more than 32,768 routes, so the count and rank kernels (which keep their
    # tile counts in the static array) see the bad expert
    idx_bad = rng.integers(0, 40, size=(20000, 3)).astype(np.int32)
    idx_bad[5, 1] = 99                                  # bad expert: status bit
    idx_bad[19997, 2] = -3
    cases.append((idx_bad, None, 40))
    for idx_np, _, E in cases:
        idx = torch.from_numpy(idx_np).to(DEV)
        st_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
        ref = mp.mp_build_map(idx, E, status=st_ref)      # caller-provided workspace
        got = _noalloc(lib, idx, E)
        torch.cuda.synchronize()
        for a, b in zip(got[:4], ref):
            assert torch.equal(a, b)
        assert torch.equal(got[4], st_ref)


def _tiles(routes):
    """Tile count of the map, as include/mp.h states it."""
    f = 1
    while f < 8 and -(-routes // (2048 * f)) > 64:
        f *= 2
    return -(-routes // (2048 * f))


def test_noalloc_map_rejects_sizes_beyond_its_scratch():
    lib = _lib.load()
    E, K = 1024, 8
    limit_words = (1 << 20) // 4
    T = 4096
    while (E + 1) * _tiles(T * K) <= limit_words:
        T += 4096
    # Real, correctly sized buffers: were the size accepted, the call would
    # still be valid and in bounds.
    idx = torch.zeros((T, K), dtype=torch.int32, device=DEV)
    rim = torch.empty((T, K), dtype=torch.int32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    code = lib.mp_build_map_noalloc(_p(idx), T, K, E, _p(rim), None, _p(counts), _p(offsets),
                                    None, stream)
    torch.cuda.synchronize()
    assert code == -3                                     # MP_ERR_UNSUPPORTED
    assert b"limit" in lib.mp_status_string(code)
    # one tile fewer is accepted and matches the workspace entry point
    T_ok = T - 4096
    ok = _noalloc(lib, idx[:T_ok], E)
    ref = mp.mp_build_map(idx[:T_ok].contiguous(), E)
    torch.cuda.synchronize()
    for a, b in zip(ok[:4], ref):
        assert torch.equal(a, b)
