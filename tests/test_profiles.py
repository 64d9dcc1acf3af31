"""The committed ncu summaries stay in step with the sources (CPU only).

Every summary under profiles/ that is named for a kernel must name a kernel
that csrc/ still defines, and must carry the ncu command that made it, with
`--clock-control none`.  The index in profiles/README.md must list every
summary, and nothing else."""
from __future__ import annotations

import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "unpermute_routing_indices_gb300", "csrc")


def _summaries():
    return sorted(p for p in glob.glob(os.path.join(PROFILES, "*.md"))
                  if os.path.basename(p) != "README.md")


def _kernels():
    """Names of the __global__ functions in csrc/: the first k_* name called
    after each __global__ (launch bounds come between)."""
    src = "".join(open(p).read() for p in glob.glob(os.path.join(CSRC, "*.cu")))
    names = set()
    for chunk in src.split("__global__")[1:]:
        m = re.search(r"\b(k_\w+)\s*\(", chunk)
        if m:
            names.add(m.group(1))
    return names


def test_kernel_summaries_name_existing_kernels():
    kernels = _kernels()
    assert "k_unpermute_bwd_staged" in kernels and "k_permute" in kernels
    for p in _summaries():
        title = open(p).readline()
        m = re.match(r"# `(k_\w+)", title)
        if m is None:
            continue   # launch list, traffic table: named for the workload
        assert m.group(1) in kernels, (os.path.basename(p), m.group(1))
        assert os.path.basename(p).startswith(m.group(1)), os.path.basename(p)


def test_summaries_carry_their_ncu_command():
    for p in _summaries():
        text = open(p).read()
        cmds = [ln for ln in text.splitlines() if re.match(r"\s*ncu\s+-", ln)]
        assert cmds, os.path.basename(p)
        for c in cmds:
            assert "--clock-control none" in c, (os.path.basename(p), c)


def test_index_lists_every_summary():
    index = open(os.path.join(PROFILES, "README.md")).read()
    listed = set(re.findall(r"`([\w.]+\.md)`", index))
    present = {os.path.basename(p) for p in _summaries()}
    assert listed == present, (sorted(listed - present), sorted(present - listed))


def test_traffic_figure_matches_its_summary():
    """bench.py's recorded DRAM traffic of the dominant kernel is the figure
    the traffic summary states."""
    import importlib.util
    import sys
    spec = importlib.util.spec_from_file_location("bench_for_profiles",
                                                  os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    argv, sys.argv = sys.argv, ["bench.py"]
    try:
        spec.loader.exec_module(bench)
    finally:
        sys.argv = argv
    summary = open(os.path.join(PROFILES, "traffic_skewed_T16384_row_kernels.md")).read()
    for rec in bench.NCU_TRAFFIC.values():
        assert f"{rec['bytes']:,}" in summary
