"""Benchmark of the MoE permute / unpermute path on GB300.

One step = the whole routed path on one batch of the skewed dispatch workload
(T=16384 tokens, H=4096 bf16, E=128 experts, K=8, Zipf(1.2)-biased router):

    mp_build_map -> mp_permute (+probs) -> mp_unpermute (probs)      forward
    mp_unpermute_bwd (probs, grad probs) -> mp_permute_bwd           backward

with the identity as the expert in between (the unpermute reads the permuted
rows; the permute backward reads the unpermute backward's row gradients).

`value` is algorithmic bytes per step / device time per step, in GB/s
(1 GB = 1e9 B), inputs resident in HBM, L2 flushed between steps.  Each step
is timed with events at its two ends only, so consecutive kernels overlap as
programmatic dependent launches; the per-op times come from the same steps
run again with an event after every op.  Byte
accounting: every input row read once, every output row written once, maps
and probabilities once.  `e2e` is the same metric through the same calls with
the inputs copied from pinned host memory and the results copied back inside
the timed region.  The JSON line also carries the per-op times, the roofline
of the dominant kernel, the chunk sort+pad roundtrip (8,192 and 32,768 rows,
H=2048, 16 experts x 8 rank chunks, align 128) and the oracle timed on the
host cores (`cpu_baseline`).

`--impl reference` times the oracle (plain C on the CPU) on a bounded sample
of the same workload instead.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "skewed"
METRIC = ("permute+unpermute GB/s and % of GB300 HBM peak; tokens/s at "
          "T=16K,H=4096,K=8")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of one launch of that kernel alone, keyed by (op, workload,
# T); a figure counts only while the profiled kernel code is unchanged
# (sha256 prefix of its .cu file and common.cuh, comments left out).  No
# matching capture: null.
NCU_TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
    #     -k regex:"^<kernel>$" -s <n> -c 1 python bench.py --workload <w> --steps 3
    #     --warmup 3 --no-cpu --no-chunks --no-extras   (one pass per launch)
    ("permute", "mid", 4096): {"bytes": 16990976 + 39353088, "src": "4de68a6e1acd2556"},
    ("unpermute", "mid", 4096): {"bytes": 100872960 + 4466432, "src": "4de68a6e1acd2556"},
    ("unpermute_bwd", "mid", 4096): {"bytes": 117673984 + 43074560, "src": "4de68a6e1acd2556"},
    ("permute_bwd", "mid", 4096): {"bytes": 100771840 + 3934720, "src": "4de68a6e1acd2556"},
    ("permute", "skewed", 16384): {"bytes": 135397888 + 1012604928, "src": "4de68a6e1acd2556"},
    ("unpermute", "skewed", 16384): {"bytes": 1074866944 + 124409344, "src": "4de68a6e1acd2556"},
    ("unpermute_bwd", "skewed", 16384): {"bytes": 1209062400 + 1021680640, "src": "4de68a6e1acd2556"},
    ("permute_bwd", "skewed", 16384): {"bytes": 1074287360 + 124515328, "src": "4de68a6e1acd2556"},
    ("permute", "large", 32768): {"bytes": 472453632 + 3697769216, "src": "4de68a6e1acd2556"},
    ("unpermute", "large", 32768): {"bytes": 3760299008 + 459797760, "src": "4de68a6e1acd2556"},
    ("unpermute_bwd", "large", 32768): {"bytes": 4230063616 + 3708089600, "src": "4de68a6e1acd2556"},
    ("permute_bwd", "large", 32768): {"bytes": 3759203328 + 459230720, "src": "4de68a6e1acd2556"},
}


# --------------------------------------------------------------------------
# byte accounting (per call)
# --------------------------------------------------------------------------

def routed_bytes(T, H, K, E, routed):
    """Algorithmic bytes of each op for T tokens, K slots, `routed` routed slots."""
    R, row = routed, 2 * H
    tok = T * row
    return {
        "build_map": 4 * T * K + 4 * T * K + 4 * T * K + 4 * E + 4 * (E + 1),
        "permute": tok + 4 * T * K + 4 * T * K + R * row + 4 * R,
        "unpermute": R * row + 4 * T * K + 4 * T * K + tok,
        "unpermute_bwd": tok + R * row + 4 * T * K + 4 * T * K + R * row + 4 * T * K,
        "permute_bwd": R * row + 4 * T * K + tok,
    }


def chunk_bytes(N, H, padded_total, out_rows):
    row = 2 * H + 4                      # bf16 row + fp32 prob
    return {
        "sort_chunks_pad": N * row + out_rows * row + out_rows * 4 + 8 * 17,
        "unpad_restore": out_rows * 4 + N * row + N * row,
    }


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def map_launches(routes: int, E: int) -> int:
    """Kernels mp_build_map launches for this many routes: one CTA (up to
    4,096 routes) or one thread-block cluster (up to 32,768) in one launch;
    beyond, the count and rank kernels, with a scan kernel in between when
    the count matrix ((E+1) x tiles of 2048*f routes, f doubling up to 8 until
    there are at most 64 tiles) exceeds 32,768 entries."""
    if routes <= 32768:
        return 1
    f = 1
    while f < 8 and -(-routes // (2048 * f)) > 64:
        f *= 2
    tiles = -(-routes // (2048 * f))
    return 2 if (E + 1) * tiles <= 32768 else 3


def ncu_traffic(op, workload, T):
    """DRAM bytes of one launch of op's kernel from its ncu capture at this
    workload and size, or None (no capture, or the kernel source changed)."""
    tr = NCU_TRAFFIC.get((op, workload, T))
    src = {"build_map": "map.cu"}.get(op, "rows.cu")
    return tr["bytes"] if tr is not None and tr["src"] == src_hash(src) else None


def code_only(text):
    """C++ source without its comments and blank lines (a comment-only edit
    leaves the compiled kernels, and so their profiled traffic, unchanged)."""
    import re

    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def src_hash(name):
    """Hash of the code of a kernel's source file and of the device helpers
    it includes, comments left out."""
    h = hashlib.sha256()
    for part in (name, "common.cuh"):
        with open(os.path.join(ROOT, "unpermute_routing_indices_gb300", "csrc", part)) as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self, t0, t1):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------------------
# data-parallel bookkeeping (one rank per GPU; every rank runs the whole path
# on its own token batch, so the only cross-rank traffic is timing)
# --------------------------------------------------------------------------

def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s token batch: independent batches, same distribution."""
    return base_seed + 7919 * rank


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time (a MAX all-reduce); the value itself at world 1."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: int, world: int, ms: float) -> float:
    """Whole-job GB/s: the bytes every rank moved per step over the slowest
    rank's step time (weak scaling)."""
    return world * bytes_per_rank_step / (ms * 1e-3) / 1e9


# --------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------

def oracle_step_rate(seconds: float, sample_tokens: int = 256):
    """Runs the oracle's version of one step on the first `sample_tokens`
    tokens of the workload until `seconds` have passed; returns GB/s."""
    import oracle
    from unpermute_routing_indices_gb300 import workloads as wl

    w = wl.routed(WORKLOAD, T=sample_tokens)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    it, t0 = 0, time.perf_counter()
    nbytes = 0
    while True:
        rim, s2f, counts, offsets, _ = oracle.build_map(w["idx"], E)
        routed = int(offsets[-1])
        rows, rows_p = oracle.permute(w["x"], w["probs"], rim)
        y = oracle.unpermute(rows, w["probs"], rim, T, H)
        g_rows, g_probs = oracle.unpermute_bwd(w["g_y"], rows, w["probs"], rim)
        g_x, _ = oracle.permute_bwd(g_rows, None, rim, T, H)
        nbytes += sum(routed_bytes(T, H, K, E, routed).values())
        it += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    sample = (f"{sample_tokens} tokens of the skewed workload (T={sample_tokens}, H={H}, "
              f"E={E}, K={K}), whole fwd+bwd step, {it} steps in {dt:.1f} s")
    return nbytes / dt / 1e9, it, dt, sample


def cpu_model() -> str:
    """A one-line description of the host CPU (model name where the kernel
    reports one, else the architecture)."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_step_sharded(w, rim, routed, pool, n_shards):
    """One fwd+bwd step of the oracle with the row work split over token
    ranges on a thread pool: the map is built once for the whole batch (its
    scan is global), then permute, unpermute, unpermute_bwd and permute_bwd
    each run on disjoint token ranges (the oracle's C calls release the GIL).
    Every token's outputs depend on that token alone, so the result is
    bit-identical to the single-thread oracle."""
    import oracle

    T, H, K = w["T"], w["H"], w["K"]
    edges = [T * i // n_shards for i in range(n_shards + 1)]
    shards = [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]
    R = T * K
    rows = np.zeros((R, H), np.uint16)
    rows_p = np.zeros(R, np.float32)
    g_rows = np.zeros((R, H), np.uint16)
    y = np.empty((T, H), np.uint16)
    g_x = np.empty((T, H), np.uint16)
    g_probs = np.empty((T, K), np.float64)
    x, probs, g_y = w["x"], w["probs"], w["g_y"]

    def fwd_perm(s):
        a, b = s
        oracle.permute(x[a:b], probs[a:b], rim[a:b], out=rows, out_probs=rows_p)

    def fwd_unperm(s):
        a, b = s
        y[a:b] = oracle.unpermute(rows, probs[a:b], rim[a:b], b - a, H)

    def bwd_unperm(s):
        a, b = s
        _, gp = oracle.unpermute_bwd(g_y[a:b], rows, probs[a:b], rim[a:b], g_rows=g_rows)
        g_probs[a:b] = gp

    def bwd_perm(s):
        a, b = s
        g_x[a:b] = oracle.permute_bwd(g_rows, None, rim[a:b], b - a, H)[0]

    for phase in (fwd_perm, fwd_unperm, bwd_unperm, bwd_perm):
        list(pool.map(phase, shards))
    return {"rows": rows[:routed], "rows_probs": rows_p[:routed], "y": y,
            "g_rows": g_rows[:routed], "g_probs": g_probs, "g_x": g_x}


class ShardedOracle:
    """The oracle's fwd+bwd step on n_threads * tokens_per_thread tokens of the
    workload, its row work over token ranges on a pool of n_threads threads.
    The first step is checked bit-identical to the single-thread oracle."""

    def __init__(self, n_threads: int, tokens_per_thread: int):
        from concurrent.futures import ThreadPoolExecutor

        import oracle
        from unpermute_routing_indices_gb300 import workloads as wl

        self.n = n_threads
        self.w = w = wl.routed(WORKLOAD, T=n_threads * tokens_per_thread)
        T, H, E, K = w["T"], w["H"], w["E"], w["K"]
        self.rim, _, _, offsets, _ = oracle.build_map(w["idx"], E)
        self.routed = int(offsets[-1])
        self.step_bytes = sum(routed_bytes(T, H, K, E, self.routed).values())
        self.pool = ThreadPoolExecutor(max_workers=n_threads)
        got = oracle_step_sharded(w, self.rim, self.routed, self.pool, n_threads)
        want = oracle_step_sharded(w, self.rim, self.routed, _Serial(), 1)
        if not all(np.array_equal(got[k], want[k]) for k in got):
            raise RuntimeError("threaded oracle differs from the single-thread oracle")

    def step(self) -> float:
        """One whole step (map + row work); returns its wall time in seconds."""
        import oracle

        t0 = time.perf_counter()
        oracle.build_map(self.w["idx"], self.w["E"])
        oracle_step_sharded(self.w, self.rim, self.routed, self.pool, self.n)
        return time.perf_counter() - t0

    def describe(self, steps: int, seconds: float) -> str:
        w = self.w
        return (f"{w['T']} tokens of the skewed workload (T={w['T']}, H={w['H']}, E={w['E']}, "
                f"K={w['K']}), whole fwd+bwd step, row work over {self.n} token ranges on "
                f"{self.n} threads ({cpu_model()}), bit-identical to one thread; "
                f"{steps} steps in {seconds:.1f} s")

    def close(self):
        self.pool.shutdown()


def oracle_threads_rate(seconds: float, n_threads: int, tokens_per_thread: int = 256):
    """ShardedOracle steps until `seconds` have passed; returns
    (GB/s, steps, seconds, sample description)."""
    so = ShardedOracle(n_threads, tokens_per_thread)
    it, dt = 0, 0.0
    while dt < seconds:
        dt += so.step()
        it += 1
    so.close()
    return it * so.step_bytes / dt / 1e9, it, dt, so.describe(it, dt)


class _Serial:
    """The map() of a pool, run on the calling thread."""

    @staticmethod
    def map(fn, items):
        return [fn(i) for i in items]


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_gpu(args):
    import torch
    import torch.distributed as dist

    import unpermute_routing_indices_gb300 as mp
    from unpermute_routing_indices_gb300 import workloads as wl

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- routed workload: per-rank batch (weak scaling), seeded per rank
    base_seed = rank_seed(wl.ROUTED[WORKLOAD]["seed"], rank)
    w = wl.routed(WORKLOAD, T=args.tokens, seed=base_seed)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    R = T * K

    def dev_t(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.to(dev)

    idx, probs, x, gy = dev_t(w["idx"]), dev_t(w["probs"]), dev_t(w["x"]), dev_t(w["g_y"])
    rim = torch.empty((T, K), dtype=torch.int32, device=dev)
    s2f = torch.empty(R, dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ws = torch.empty(mp.mp_build_map_workspace_size(T, K, E), dtype=torch.uint8, device=dev)
    rows = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    rows_p = torch.empty(R, dtype=torch.float32, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    g_rows = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    g_probs = torch.empty((T, K), dtype=torch.float32, device=dev)
    g_x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)

    ops = ["build_map", "permute", "unpermute", "unpermute_bwd", "permute_bwd"]
    # kernels each op launches
    launches = {"build_map": map_launches(R, E), "permute": 1, "unpermute": 1,
                "unpermute_bwd": 1, "permute_bwd": 1}

    def call(op):
        if op == "build_map":
            mp.mp_build_map(idx, E, row_id_map=rim, sorted_to_flat=s2f, counts=counts,
                            offsets=offsets, workspace=ws)
        elif op == "permute":
            mp.mp_permute(x, rim, probs, out=rows, out_probs=rows_p)
        elif op == "unpermute":
            mp.mp_unpermute(rows, rim, probs, out=y)
        elif op == "unpermute_bwd":
            mp.mp_unpermute_bwd(gy, rim, rows, probs, g_rows=g_rows, g_probs=g_probs)
        elif op == "permute_bwd":
            mp.mp_permute_bwd(g_rows, rim, g_x=g_x)

    stream = torch.cuda.current_stream(dev)
    nev = len(ops) + 1

    def timed_steps(n, per_op, flushed=True):
        """n steps.  per_op=False: events at the ends of each step only, so each
        kernel's launch overlaps the tail of the one before it (programmatic
        dependent launch); per_op=True: an event after every op as well, which
        serialises the ops and times each one alone."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev if per_op else 2)]
               for _ in range(n)]
        for i in range(n):
            if flushed:
                flush(i)                                # L2 flush between steps
            evs[i][0].record(stream)
            for j, op in enumerate(ops):
                call(op)
                if per_op:
                    evs[i][j + 1].record(stream)
            if not per_op:
                evs[i][1].record(stream)
        return evs

    for _ in range(args.warmup):
        timed_steps(1, False)
        timed_steps(1, True)
    torch.cuda.synchronize()
    routed = int(offsets[-1].item())
    nbytes = routed_bytes(T, H, K, E, routed)
    step_bytes = sum(nbytes.values())

    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier()
        t0 = time.time()
        evs = timed_steps(args.steps, False)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier()
        # the same steps again with an event after every op: per-kernel times
        op_evs = timed_steps(args.steps, True)
        torch.cuda.synchronize()
        barrier()
    clocks = clk.summary(t0, t1)

    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    samples = {op: [] for op in ops}
    op_step_ms = []
    for e in op_evs:
        op_step_ms.append(e[0].elapsed_time(e[-1]))
        for j, op in enumerate(ops):
            samples[op].append(e[j].elapsed_time(e[j + 1]))
    ms_serialised = sum(op_step_ms) / len(op_step_ms)
    per_op = {op: statistics.mean(v) for op, v in samples.items()}
    med_op = {op: statistics.median(v) for op, v in samples.items()}

    # warm numbers: the same steps back to back, no L2 flush in between
    warm_n = max(3, min(args.steps, 100))
    torch.cuda.synchronize()
    wev = timed_steps(warm_n, True, flushed=False)
    torch.cuda.synchronize()
    warm_op = {op: statistics.median(wev[i][j].elapsed_time(wev[i][j + 1]) for i in range(warm_n))
               for j, op in enumerate(ops)}

    # the cost of any launch under the same timing: a one-element torch kernel
    # between two events after the same L2 flush
    tiny = torch.zeros(1, device=dev)
    floor_us = time_op(lambda: tiny.fill_(1.0), flush, stream, 50)

    peak, peak_kind = measured_peaks()
    gbs = job_throughput(step_bytes, world, ms)
    dom = max(ops, key=lambda o: per_op[o])
    traffic = ncu_traffic(dom, WORKLOAD, T)
    achieved = nbytes[dom] / (per_op[dom] * 1e-3) / 1e9

    # ---- e2e through host buffers (pinned), same calls.  Serial: every copy
    # and kernel in order on one stream.  Pipelined (the reported e2e): the
    # library's HostPipeline overlaps step i+1's copy-in, step i's kernels and
    # step i-1's copy-out on three streams with double-buffered device sets.
    from unpermute_routing_indices_gb300.pipeline import HostPipeline

    def pinned(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.pin_memory()

    h_in = {"idx": pinned(w["idx"]), "probs": pinned(w["probs"]), "x": pinned(w["x"]),
            "g_y": pinned(w["g_y"])}
    out_spec = {"y": ((T, H), torch.bfloat16), "g_x": ((T, H), torch.bfloat16),
                "g_probs": ((T, K), torch.float32)}
    h_outs = [{k: torch.empty(sh, dtype=dt_).pin_memory() for k, (sh, dt_) in out_spec.items()}
              for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_outs[0].values())

    def e2e_step():
        idx.copy_(h_in["idx"], non_blocking=True)
        probs.copy_(h_in["probs"], non_blocking=True)
        x.copy_(h_in["x"], non_blocking=True)
        gy.copy_(h_in["g_y"], non_blocking=True)
        for op in ops:
            call(op)
        h_outs[0]["y"].copy_(y, non_blocking=True)
        h_outs[0]["g_x"].copy_(g_x, non_blocking=True)
        h_outs[0]["g_probs"].copy_(g_probs, non_blocking=True)

    e2e_steps = max(50, min(args.steps, 200))   # its own count: the pipeline fills and drains once
    for _ in range(max(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    barrier()

    def pipe_step(din, dout):
        mp.mp_build_map(din["idx"], E, row_id_map=rim, sorted_to_flat=s2f, counts=counts,
                        offsets=offsets, workspace=ws)
        mp.mp_permute(din["x"], rim, din["probs"], out=rows, out_probs=rows_p)
        mp.mp_unpermute(rows, rim, din["probs"], out=dout["y"])
        mp.mp_unpermute_bwd(din["g_y"], rim, rows, din["probs"], g_rows=g_rows,
                            g_probs=dout["g_probs"])
        mp.mp_permute_bwd(g_rows, rim, g_x=dout["g_x"])

    in_spec = {k: (tuple(t.shape), t.dtype) for k, t in h_in.items()}
    pipe = HostPipeline(dev, in_spec, out_spec, pipe_step, graph=True)
    pipe.run([h_in] * max(args.warmup, 3), [h_outs[i % 2] for i in range(max(args.warmup, 3))])
    torch.cuda.synchronize()
    barrier()
    p0 = torch.cuda.Event(enable_timing=True)
    p0.record(pipe.s_in)
    last = None
    for i in range(e2e_steps):
        last = pipe.submit(i, h_in, h_outs[i % 2])
    p1 = torch.cuda.Event(enable_timing=True)
    p1.record(pipe.s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(p0.elapsed_time(p1) / e2e_steps, world, dev)
    # the pipelined results are the serial ones
    if not (torch.equal(h_outs[(e2e_steps - 1) % 2]["y"], y.cpu())
            and torch.equal(h_outs[(e2e_steps - 1) % 2]["g_x"], g_x.cpu())):
        raise RuntimeError("pipelined step differs from the serial step")
    barrier()

    # ---- chunk sort+pad roundtrip (context: the pages' only published timing)
    sort_pad = {}
    if rank == 0 and not args.no_chunks:
        sort_pad = bench_chunks(mp, wl, dev, flush, args)

    # ---- the widened rows, on the same batch: capacity map, EP-rank combine
    extras = {}
    if rank == 0 and not args.no_extras:
        cap = -(-5 * routed // (4 * E))                   # capacity factor 1.25
        ep = 8
        ep_bytes = nbytes["unpermute"] + 4 * T * K        # + the slot experts
        logits = dev_t(wl.router_logits(WORKLOAD, T=T, seed=base_seed))
        r_idx, r_probs = torch.empty_like(idx), torch.empty_like(probs)
        n_groups = wl.ROUTED[WORKLOAD].get("n_groups", 1)
        topk_groups = wl.ROUTED[WORKLOAD].get("topk_groups", 1)
        g_rp = torch.ones_like(probs)
        g_logits = torch.empty_like(logits)
        quarter = torch.tensor([R * 3 // 4], dtype=torch.int32, device=dev)
        rim_c, s2f_c = torch.empty_like(rim), torch.empty_like(s2f)
        counts_c, offsets_c = torch.empty_like(counts), torch.empty_like(offsets)
        extra_ops = {
            f"build_map_capacity(cap={cap})": (
                lambda: mp.mp_build_map_capacity(idx, E, cap, row_id_map=rim_c,
                                                 sorted_to_flat=s2f_c, counts=counts_c,
                                                 offsets=offsets_c, workspace=ws),
                nbytes["build_map"]),
            "topk_softmax(router)": (
                lambda: mp.mp_topk_softmax(logits, K, n_groups=n_groups, topk_groups=topk_groups,
                                           idx=r_idx, probs=r_probs),
                4 * T * E + 8 * T * K),
            "topk_softmax_bwd(router)": (
                lambda: mp.mp_topk_softmax_bwd(g_rp, r_probs, r_idx, E, g_logits=g_logits),
                12 * T * K + 4 * T * E),
            "zero_rows_from(last quarter of the rows)": (
                lambda: mp.mp_zero_rows_from(g_rows, quarter), (R - R * 3 // 4) * 2 * H),
            "zero_rows_from(all rows routed: no store)": (
                lambda: mp.mp_zero_rows_from(g_rows, offsets[-1:]), 0),
            f"unpermute_ep(ep={ep})": (
                lambda: mp.mp_unpermute_ep(rows, rim, idx, E, ep, probs, out=y), ep_bytes),
            f"unpermute_ep(ep={ep},bf16_partials)": (
                lambda: mp.mp_unpermute_ep(rows, rim, idx, E, ep, probs, bf16_partials=True,
                                           out=y), ep_bytes),
            f"unpermute_ep(ep={ep},fp64_cross_rank)": (
                lambda: mp.mp_unpermute_ep(rows, rim, idx, E, ep, probs, fp64_cross_rank=True,
                                           out=y), ep_bytes),
            f"unpermute_ep(ep={ep},bf16_partials,fp64_cross_rank)": (
                lambda: mp.mp_unpermute_ep(rows, rim, idx, E, ep, probs, bf16_partials=True,
                                           fp64_cross_rank=True, out=y), ep_bytes),
        }
        call("build_map")
        call("permute")
        mp.mp_topk_softmax(logits, K, n_groups=n_groups, topk_groups=topk_groups, idx=r_idx,
                           probs=r_probs)
        for name, (fn, b) in extra_ops.items():
            us = time_op(fn, flush, stream, max(30, min(args.steps, 100)))
            extras[name] = {"us": round(us, 2), "GB/s": round(b / (us * 1e-6) / 1e9, 1),
                            "frac_of_measured": round(b / (us * 1e-6) / 1e9 / peak, 4)}
        call("build_map")
        call("permute")

    # ---- the other routed workloads at full size (mid: T=4096, H=2048, E=64,
    # K=6; large: T=32768, H=7168, E=256, K=8; whichever is not the headline)
    workloads = {}
    if rank == 0 and not args.no_extras:
        for name in ("mid", "skewed", "large"):
            if name != WORKLOAD:
                workloads[name] = bench_routed(mp, wl, name, dev, flush,
                                               max(20, min(args.steps, 100)), peak)
                torch.cuda.empty_cache()

    out = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy; router logits N(0,1) + 2 ln Zipf(1.2) bias)",
        "config": {"workload": f"{WORKLOAD} dispatch T={T} H={H} E={E} K={K}, fwd+bwd step",
                   "T": T, "H": H, "E": E, "K": K, "routed_rows": routed,
                   "bytes_per_step": step_bytes,
                   "l2": "flushed between steps, outside the events: a 2xL2 buffer written, "
                         "then another 2xL2 buffer read (L2 cold and clean)",
                   "parallelism": f"dp{world} (independent token batches, no collective)"},
        "pct_of_nominal_peak": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_peak": round(100 * gbs / world / peak, 2),
        "tokens_per_s": round(world * T / (ms * 1e-3), 1),
        "ms_per_step_serialised": round(ms_serialised, 4),
        "ops_timing": "each op alone: the same steps again with an event after every op",
        "launch_floor_us": {"value": round(floor_us, 2),
                            "how": "a one-element torch kernel timed the same way (events "
                                   "around it after an L2 flush): the part of every short "
                                   "op's time that is launch and event overhead"},
        "ops": {op: {"us": round(per_op[op] * 1e3, 2), "us_median": round(med_op[op] * 1e3, 2),
                     "us_warm_median": round(warm_op[op] * 1e3, 2), "bytes": nbytes[op],
                     "GB/s": round(nbytes[op] / (per_op[op] * 1e-3) / 1e9, 1),
                     "frac_of_measured": round(nbytes[op] / (per_op[op] * 1e-3) / 1e9 / peak, 4),
                     "dram_traffic": ncu_traffic(op, WORKLOAD, T)}
                for op in ops},
        "permute_incl_map": {
            "us": round((per_op["build_map"] + per_op["permute"]) * 1e3, 2),
            "GB/s": round((nbytes["build_map"] + nbytes["permute"])
                          / ((per_op["build_map"] + per_op["permute"]) * 1e-3) / 1e9, 1),
            "tokens_per_s": round(T / ((per_op["build_map"] + per_op["permute"]) * 1e-3), 1)},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": nbytes[dom]},
        "e2e": {"value": round(job_throughput(step_bytes, world, e2e_ms), 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "HostPipeline: copy-in, kernels and copy-out of consecutive steps "
                       "overlapped on three streams, double-buffered device sets, the "
                       "step's kernels replayed from a CUDA graph per set; "
                       f"{e2e_steps} steps between events"},
        "e2e_serial": {"value": round(job_throughput(step_bytes, world, e2e_serial_ms), 1),
                       "unit": "GB/s", "ms_per_step": round(e2e_serial_ms, 4),
                       "how": "copies and kernels in order on one stream"},
        "gpu_launches": sum(launches.values()) * args.steps,
        "clocks": clocks,
    }
    if sort_pad:
        out["sort_pad_roundtrip"] = sort_pad
    if extras:
        out["extras"] = extras
    if workloads:
        out["extras"]["workloads"] = workloads
    if rank == 0 and not args.no_cpu:
        v, it, dt, sample = oracle_step_rate(args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": 1,
                               "kind": "oracle", "sample": sample}
        n = host_threads()
        v, it, dt, sample = oracle_threads_rate(args.cpu_seconds * 2 / 3, n)
        out["cpu_baseline_threads"] = {"value": round(v, 4), "unit": "GB/s", "cores": n,
                                       "kind": "oracle", "sample": sample}
    if world > 1:
        barrier()   # rank 0 ran the chunk, extra and other-workload timings alone
        dist.destroy_process_group()
    return out if rank == 0 else None


class L2Flush:
    """Leaves L2 cold and clean between timed steps: a write of a buffer twice
    the size of L2 evicts every line the last step left, then a read of a
    second such buffer evicts the written (dirty) lines, so their write-back
    happens here rather than inside the next timed region."""

    def __init__(self, dev):
        import torch

        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.zeros(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self, i=0):
        import torch

        self.w.fill_(float(i))
        torch.amax(self.r, dim=0, keepdim=True, out=self.sink)


def time_op(fn, flush, stream, n):
    """Mean device time (us) of fn over n launches, L2 flushed before each."""
    import torch

    for _ in range(3):
        fn()
    evs = []
    for i in range(n):
        flush(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return 1e3 * statistics.mean(a.elapsed_time(b) for a, b in evs)


def bench_routed(mp, wl, name, dev, flush, n, peak):
    """The whole fwd+bwd step on another routed workload (its full size, as
    the headline step runs it): per-op device times with an event after every
    op (L2 flushed before each step), and the step with events at its ends
    only.  Returns per-op us, GB/s and fraction of the measured peak."""
    import torch

    w = wl.routed(name)
    T, H, E, K = w["T"], w["H"], w["E"], w["K"]
    R = T * K

    def dev_t(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.to(dev)

    idx, probs, x, gy = dev_t(w["idx"]), dev_t(w["probs"]), dev_t(w["x"]), dev_t(w["g_y"])
    del w
    rim = torch.empty((T, K), dtype=torch.int32, device=dev)
    s2f = torch.empty(R, dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ws = torch.empty(mp.mp_build_map_workspace_size(T, K, E), dtype=torch.uint8, device=dev)
    rows = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    rows_p = torch.empty(R, dtype=torch.float32, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    g_rows = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    g_probs = torch.empty((T, K), dtype=torch.float32, device=dev)
    g_x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ops = {
        "build_map": lambda: mp.mp_build_map(idx, E, row_id_map=rim, sorted_to_flat=s2f,
                                             counts=counts, offsets=offsets, workspace=ws),
        "permute": lambda: mp.mp_permute(x, rim, probs, out=rows, out_probs=rows_p),
        "unpermute": lambda: mp.mp_unpermute(rows, rim, probs, out=y),
        "unpermute_bwd": lambda: mp.mp_unpermute_bwd(gy, rim, rows, probs, g_rows=g_rows,
                                                     g_probs=g_probs),
        "permute_bwd": lambda: mp.mp_permute_bwd(g_rows, rim, g_x=g_x),
    }
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        for fn in ops.values():
            fn()
    torch.cuda.synchronize()
    routed = int(offsets[-1].item())
    nbytes = routed_bytes(T, H, K, E, routed)
    ev = lambda: torch.cuda.Event(enable_timing=True)       # noqa: E731
    per_op = [[ev() for _ in range(len(ops) + 1)] for _ in range(n)]
    for i, es in enumerate(per_op):
        flush(i)
        es[0].record(stream)
        for j, fn in enumerate(ops.values()):
            fn()
            es[j + 1].record(stream)
    chained = [(ev(), ev()) for _ in range(n)]
    for i, (a, z) in enumerate(chained):
        flush(i)
        a.record(stream)
        for fn in ops.values():
            fn()
        z.record(stream)
    torch.cuda.synchronize()
    step_ms = statistics.mean(a.elapsed_time(z) for a, z in chained)
    res = {"workload": f"{name} dispatch T={T} H={H} E={E} K={K}, fwd+bwd step",
           "routed_rows": routed, "ms_per_step": round(step_ms, 4),
           "GB/s": round(sum(nbytes.values()) / (step_ms * 1e-3) / 1e9, 1),
           "frac_of_measured": round(sum(nbytes.values()) / (step_ms * 1e-3) / 1e9 / peak, 4),
           "ops": {}}
    for j, op in enumerate(ops):
        us = 1e3 * statistics.mean(es[j].elapsed_time(es[j + 1]) for es in per_op)
        gbs = nbytes[op] / (us * 1e-6) / 1e9
        res["ops"][op] = {"us": round(us, 2), "bytes": nbytes[op], "GB/s": round(gbs, 1),
                          "frac_of_measured": round(gbs / peak, 4),
                          "dram_traffic": ncu_traffic(op, name, T)}
    return res


def bench_chunks(mp, wl, dev, flush, args):
    import torch

    res = {}
    stream = torch.cuda.current_stream(dev)
    for N, tdt in ((8192, torch.bfloat16), (32768, torch.bfloat16), (32768, torch.float32)):
        c = wl.chunks(N)
        G, align, H = c["G"], c["align"], c["H"]
        out_rows = wl.padded_rows_bound(N, G, align)

        def t(a):
            tt = torch.from_numpy(np.ascontiguousarray(a))
            if a.dtype == np.uint16:
                tt = tt.view(torch.int16).view(torch.bfloat16)
            return tt.to(dev)

        x, p, sz, od = t(c["x"]), t(c["probs"]), t(c["split_sizes"]), t(c["chunk_order"])
        x = x.to(tdt)
        esize = x.element_size()
        out = torch.empty((out_rows, H), dtype=tdt, device=dev)
        out_p = torch.empty(out_rows, dtype=torch.float32, device=dev)
        row_map = torch.empty(out_rows, dtype=torch.int32, device=dev)
        goff = torch.empty(G + 1, dtype=torch.int64, device=dev)
        y = torch.empty((N, H), dtype=tdt, device=dev)
        y_p = torch.empty(N, dtype=torch.float32, device=dev)

        def roundtrip():
            mp.mp_sort_chunks_pad(x, sz, od, G, align, out_rows, p, out=out, out_probs=out_p,
                                  row_map=row_map, group_off=goff)
            mp.mp_unpad_restore(out, row_map, N, out_p, y=y, y_probs=y_p)

        for _ in range(5):
            roundtrip()
        n = max(50, min(args.steps, 200))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for e in evs:
            flush(1)
            e[0].record(stream)
            mp.mp_sort_chunks_pad(x, sz, od, G, align, out_rows, p, out=out, out_probs=out_p,
                                  row_map=row_map, group_off=goff)
            e[1].record(stream)
            mp.mp_unpad_restore(out, row_map, N, out_p, y=y, y_probs=y_p)
            e[2].record(stream)
        torch.cuda.synchronize()
        # Means: the event timer ticks in steps of about 1 us here, so the
        # median of short ops sits on a tick while the mean of many samples
        # resolves below it.
        sp = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
        ur = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
        rt = statistics.mean(e[0].elapsed_time(e[2]) for e in evs)
        # the same roundtrip with events at its ends only: the restore's launch
        # then overlaps the tail of sort+pad (programmatic dependent launch)
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, z in cev:
            flush(1)
            a.record(stream)
            roundtrip()
            z.record(stream)
        torch.cuda.synchronize()
        rt_chained = statistics.mean(a.elapsed_time(z) for a, z in cev)
        padded = int(goff[-1].item())
        b = chunk_bytes(N, H * esize // 2, padded, out_rows)
        key = str(N) if tdt == torch.bfloat16 else f"{N} fp32"

        # each op alone after its own flush, and a plain device copy of the
        # same N rows (torch copy_) timed the same way, for scale
        def alone(fn):
            ev = []
            for i in range(n):
                flush(i)
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                z.record(stream)
                ev.append((a, z))
            torch.cuda.synchronize()
            v = [a.elapsed_time(z) * 1e3 for a, z in ev]
            return statistics.mean(v), statistics.median(v)

        sp_alone, sp_alone_med = alone(lambda: mp.mp_sort_chunks_pad(
            x, sz, od, G, align, out_rows, p, out=out, out_probs=out_p, row_map=row_map,
            group_off=goff))
        ur_alone, ur_alone_med = alone(lambda: mp.mp_unpad_restore(out, row_map, N, out_p, y=y,
                                                                   y_probs=y_p))
        copy_us, copy_us_med = alone(lambda: y.copy_(x))
        res[key] = {"roundtrip_ms": round(rt, 4), "sort_pad_us": round(sp * 1e3, 2),
                    "unpad_restore_us": round(ur * 1e3, 2),
                    "roundtrip_GB/s": round((b["sort_chunks_pad"] + b["unpad_restore"])
                                            / (rt * 1e-3) / 1e9, 1),
                    "roundtrip_chained_ms": round(rt_chained, 4),
                    "sort_pad_alone_us": round(sp_alone, 2),
                    "unpad_restore_alone_us": round(ur_alone, 2),
                    "sort_pad_alone_GB/s": round(b["sort_chunks_pad"] / sp_alone / 1e3, 1),
                    "unpad_restore_alone_GB/s": round(b["unpad_restore"] / ur_alone / 1e3, 1),
                    "plain_copy_us": round(copy_us, 2),
                    "medians_us": {"sort_pad_alone": round(sp_alone_med, 2),
                                   "unpad_restore_alone": round(ur_alone_med, 2),
                                   "plain_copy": round(copy_us_med, 2)},
                    "timing": f"means of {n} samples, each after an L2 flush",
                    "out_rows": out_rows, "padded_rows": padded}
        if tdt == torch.bfloat16:
            res[key]["published_b200_fused_ms"] = {8192: 0.1717, 32768: 0.2029}[N]
    return res


def run_reference(args):
    """The oracle as it stands, on the host cores: each step is one whole
    fwd+bwd step over a bounded sample of the workload (64 tokens per host
    thread), the row work split over token ranges on all host threads."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    n = host_threads()
    so = ShardedOracle(n, 64)
    for _ in range(args.warmup):
        so.step()
    secs = [so.step() for _ in range(args.steps)]
    so.close()
    mean_s = statistics.mean(secs)
    v = so.step_bytes / mean_s / 1e9
    from unpermute_routing_indices_gb300 import workloads as wl

    full = wl.ROUTED[WORKLOAD]
    T, H, E, K = full["T"], full["H"], full["E"], full["K"]
    cfg = {"workload": f"{WORKLOAD} dispatch T={T} H={H} E={E} K={K}, fwd+bwd step",
           "T": T, "H": H, "E": E, "K": K,
           "sample": f"{so.w['T']} tokens per step ({so.routed} routed rows, "
                     f"{so.step_bytes} bytes)"}
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * mean_s, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded numpy)", "config": cfg,
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
                             "sample": so.describe(args.steps, sum(secs))},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-chunks", action="store_true", help="skip the sort+pad roundtrip")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the capacity-map and EP-combine timings")
    ap.add_argument("--tokens", type=int, default=None,
                    help="smaller T of the same workload (profiling captures only)")
    ap.add_argument("--workload", choices=["skewed", "large", "mid"], default="skewed",
                    help="routed workload of the step (the metric is quoted on 'skewed')")
    args = ap.parse_args()
    global WORKLOAD
    WORKLOAD = args.workload
    if args.warmup < 3:
        args.warmup = 3
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
