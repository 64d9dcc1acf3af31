"""The double-buffered host pipeline gives every step the results of running
that step alone: distinct inputs per step, each step's outputs compared bit
for bit with the same calls made serially (a wrong wait between the streams
would let a step read another step's inputs or overwrite results before they
were copied out)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import unpermute_routing_indices_gb300 as mp
from unpermute_routing_indices_gb300 import workloads as wl
from unpermute_routing_indices_gb300.pipeline import HostPipeline
from tests.gpu_util import DEV

pytestmark = pytest.mark.gpu


def _pinned(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.pin_memory()


def _step_fn(E, T, K, H):
    R = T * K
    rows = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    rows_p = torch.empty(R, dtype=torch.float32, device=DEV)
    g_rows = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)

    def step(din, dout):
        rim, _, _, _ = mp.mp_build_map(din["idx"], E)
        mp.mp_permute(din["x"], rim, din["probs"], out=rows, out_probs=rows_p)
        mp.mp_unpermute(rows, rim, din["probs"], out=dout["y"])
        mp.mp_unpermute_bwd(din["g_y"], rim, rows, din["probs"], g_rows=g_rows,
                            g_probs=dout["g_probs"])
        mp.mp_permute_bwd(g_rows, rim, g_x=dout["g_x"])
    return step


@pytest.mark.parametrize("n_steps,graph", [(1, False), (2, False), (7, False), (1, True),
                                           (7, True)])
def test_pipeline_matches_serial_steps(n_steps, graph):
    T, H = 2048, 1024
    sets = []
    for s in range(3):
        w = wl.routed("mid", T=T, H=H, seed=100 + s)
        sets.append({"idx": _pinned(w["idx"]), "probs": _pinned(w["probs"]),
                     "x": _pinned(w["x"]), "g_y": _pinned(w["g_y"])})
    E, K = w["E"], w["K"]
    in_spec = {k: (tuple(t.shape), t.dtype) for k, t in sets[0].items()}
    out_spec = {"y": ((T, H), torch.bfloat16), "g_x": ((T, H), torch.bfloat16),
                "g_probs": ((T, K), torch.float32)}
    step = _step_fn(E, T, K, H)
    pipe = HostPipeline(DEV, in_spec, out_spec, step, graph=graph)
    host_in = [sets[i % 3] for i in range(n_steps)]
    host_out = [{k: torch.empty(s, dtype=t).pin_memory() for k, (s, t) in out_spec.items()}
                for _ in range(n_steps)]
    pipe.run(host_in, host_out)
    for i in range(n_steps):
        din = {k: v.to(DEV) for k, v in host_in[i].items()}
        dout = {k: torch.empty(s, dtype=t, device=DEV) for k, (s, t) in out_spec.items()}
        step(din, dout)
        for k in out_spec:
            assert torch.equal(host_out[i][k], dout[k].cpu()), (i, k)


def test_pipeline_rejects_unpinned_or_misshapen_host_tensors():
    spec = {"a": ((4, 8), torch.float32)}
    pipe = HostPipeline(DEV, spec, spec, lambda din, dout: dout["a"].copy_(din["a"]))
    good = {"a": torch.zeros(4, 8).pin_memory()}
    with pytest.raises(ValueError):
        pipe.submit(0, {"a": torch.zeros(4, 8)}, good)               # not pinned
    with pytest.raises(ValueError):
        pipe.submit(0, good, {"a": torch.zeros(4, 9).pin_memory()})   # wrong shape
    out = {"a": torch.empty(4, 8).pin_memory()}
    src = {"a": torch.arange(32, dtype=torch.float32).view(4, 8).pin_memory()}
    pipe.submit(0, src, out).synchronize()
    assert torch.equal(out["a"], src["a"])
