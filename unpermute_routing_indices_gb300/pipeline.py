"""Double-buffered host <-> device step pipeline.

A step whose inputs come from host memory and whose results go back to it is
bound by the host link (on GB300 about 200 GB/s each way over NVLink-C2C,
340 GB/s both ways at once) well before the HBM-bound kernels.  This runs the
three phases of consecutive steps at the same time, on three streams:

    copy-in  (stream 1):  host inputs of step i    -> device input set i % 2
    compute  (stream 2):  the step on input set i % 2 -> device output set i % 2
    copy-out (stream 3):  device output set i % 2  -> host outputs of step i

Events order the reuse of each buffer set: step i's copy-in waits until the
compute of step i-2 has finished reading that input set, and its compute
waits until the copy-out of step i-2 has finished reading that output set.
The step function launches library calls on the current stream; it must not
allocate buffers that outlive the call on another stream.

With graph=True the step is captured once per buffer set, as a CUDA graph on
the compute stream, the first time that set is used; later steps replay the
graph, so issuing a step costs one replay instead of one Python call per
kernel.  The step must then be capturable: no host synchronisation and no
data-dependent host logic.  Every library call is.
"""
from __future__ import annotations

from typing import Callable, Dict, Sequence, Tuple

import torch

Spec = Dict[str, Tuple[Tuple[int, ...], torch.dtype]]


class HostPipeline:
    """Runs `step(dev_in, dev_out)` for a sequence of host input sets.

    in_spec / out_spec: name -> (shape, dtype) of each input / output tensor.
    Host tensors passed to run() must be pinned (page-locked) and match the
    specs; device buffers (two sets each) are allocated here."""

    def __init__(self, device, in_spec: Spec, out_spec: Spec,
                 step: Callable[[Dict[str, torch.Tensor], Dict[str, torch.Tensor]], None],
                 graph: bool = False):
        self.device = torch.device(device)
        self.graph = graph
        self._graphs = [None, None]     # the captured step of each buffer set
        self.in_spec, self.out_spec, self.step = in_spec, out_spec, step
        self.dev_in = [{k: torch.empty(s, dtype=t, device=self.device)
                        for k, (s, t) in in_spec.items()} for _ in range(2)]
        self.dev_out = [{k: torch.empty(s, dtype=t, device=self.device)
                         for k, (s, t) in out_spec.items()} for _ in range(2)]
        self.s_in = torch.cuda.Stream(self.device)
        self.s_comp = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        self._in_free = [None, None]    # compute of the set's last step done
        self._out_free = [None, None]   # copy-out of the set's last step done

    def h2d_bytes(self) -> int:
        return sum(torch.empty(0, dtype=t).element_size() * _numel(s)
                   for s, t in self.in_spec.values())

    def d2h_bytes(self) -> int:
        return sum(torch.empty(0, dtype=t).element_size() * _numel(s)
                   for s, t in self.out_spec.values())

    def _check_host(self, tensors: Dict[str, torch.Tensor], spec: Spec, what: str):
        for k, (s, t) in spec.items():
            h = tensors[k]
            if h.is_cuda or not h.is_pinned() or h.dtype != t or tuple(h.shape) != tuple(s) \
                    or not h.is_contiguous():
                raise ValueError(f"{what} '{k}' must be a pinned contiguous host tensor "
                                 f"{tuple(s)} {t}")

    def submit(self, i: int, host_in: Dict[str, torch.Tensor],
               host_out: Dict[str, torch.Tensor]) -> torch.cuda.Event:
        """Enqueues step i (copy-in, compute, copy-out) without waiting; returns
        the event that marks its results in host_out.  Steps must be submitted
        in order; host_in must stay unchanged and host_out unread until the
        step's event has completed."""
        self._check_host(host_in, self.in_spec, "input")
        self._check_host(host_out, self.out_spec, "output")
        b = i % 2
        din, dout = self.dev_in[b], self.dev_out[b]
        if self.graph and self._graphs[b] is None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.s_comp):
                self.step(din, dout)
            self._graphs[b] = g
        with torch.cuda.stream(self.s_in):
            if self._in_free[b] is not None:
                self.s_in.wait_event(self._in_free[b])
            for k in self.in_spec:
                din[k].copy_(host_in[k], non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(self.s_in)
        with torch.cuda.stream(self.s_comp):
            self.s_comp.wait_event(ready)
            if self._out_free[b] is not None:
                self.s_comp.wait_event(self._out_free[b])
            if self.graph:
                self._graphs[b].replay()
            else:
                self.step(din, dout)
            done = torch.cuda.Event()
            done.record(self.s_comp)
        self._in_free[b] = done
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(done)
            for k in self.out_spec:
                host_out[k].copy_(dout[k], non_blocking=True)
            out_done = torch.cuda.Event()
            out_done.record(self.s_out)
        self._out_free[b] = out_done
        return out_done

    def run(self, host_in: Sequence[Dict[str, torch.Tensor]],
            host_out: Sequence[Dict[str, torch.Tensor]]) -> None:
        """Runs one step per (host_in[i], host_out[i]) and waits for the last."""
        last = None
        for i, (hi, ho) in enumerate(zip(host_in, host_out)):
            last = self.submit(i, hi, ho)
        if last is not None:
            last.synchronize()


def _numel(shape) -> int:
    n = 1
    for d in shape:
        n *= int(d)
    return n
