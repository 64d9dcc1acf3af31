"""The host-side legs of bench.py: the oracle split over token ranges on a
thread pool gives the single-thread oracle's bits, and the oracle wrappers'
caller-owned outputs take only the rows the map names."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import bench
import oracle
from unpermute_routing_indices_gb300 import workloads as wl


def _small(T=37):
    w = wl.routed("mid", T=T)
    rim, _, _, offsets, _ = oracle.build_map(w["idx"], w["E"])
    return w, rim, int(offsets[-1])


@pytest.mark.parametrize("n_shards", [2, 3, 5])
def test_sharded_step_is_bit_identical_to_one_thread(n_shards):
    w, rim, routed = _small()
    want = bench.oracle_step_sharded(w, rim, routed, bench._Serial(), 1)
    with ThreadPoolExecutor(max_workers=n_shards) as pool:
        got = bench.oracle_step_sharded(w, rim, routed, pool, n_shards)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


def test_sharded_step_matches_the_whole_batch_calls():
    w, rim, routed = _small(T=19)
    T, H = w["T"], w["H"]
    got = bench.oracle_step_sharded(w, rim, routed, bench._Serial(), 4)
    rows, rows_p = oracle.permute(w["x"], w["probs"], rim)
    y = oracle.unpermute(rows, w["probs"], rim, T, H)
    g_rows, g_probs = oracle.unpermute_bwd(w["g_y"], rows, w["probs"], rim)
    g_x, _ = oracle.permute_bwd(g_rows, None, rim, T, H)
    assert np.array_equal(got["rows"], rows[:routed])
    assert np.array_equal(got["rows_probs"], rows_p[:routed])
    assert np.array_equal(got["y"], y)
    assert np.array_equal(got["g_rows"], g_rows[:routed])
    assert np.array_equal(got["g_probs"], g_probs)
    assert np.array_equal(got["g_x"], g_x)


def test_caller_outputs_take_only_mapped_rows():
    w, rim, routed = _small(T=11)
    R, H = rim.size, w["H"]
    out = np.full((R + 3, H), 0xBEEF, np.uint16)
    out_p = np.full(R + 3, -7.0, np.float32)
    oracle.permute(w["x"][:5], w["probs"][:5], rim[:5], out=out, out_probs=out_p)
    named = set(int(r) for r in rim[:5].ravel() if r >= 0)
    for r in range(R + 3):
        if r in named:
            t, k = map(int, np.argwhere(rim == r)[0])
            assert np.array_equal(out[r], w["x"][t]) and out_p[r] == w["probs"][t, k]
        else:
            assert np.all(out[r] == 0xBEEF) and out_p[r] == -7.0
    g_rows = np.full((R, H), 0xBEEF, np.uint16)
    oracle.unpermute_bwd(w["g_y"][5:], out, w["probs"][5:], rim[5:], g_rows=g_rows)
    named = set(int(r) for r in rim[5:].ravel() if r >= 0)
    untouched = [r for r in range(R) if r not in named]
    assert np.all(g_rows[untouched] == 0xBEEF)


def test_caller_outputs_are_checked():
    w, rim, _ = _small(T=4)
    with pytest.raises(ValueError):
        oracle.permute(w["x"], w["probs"], rim, out=np.zeros((rim.size, w["H"]), np.int32))
    with pytest.raises(ValueError):
        oracle.permute(w["x"], w["probs"], rim,
                       out=np.zeros((rim.size, w["H"] + 1), np.uint16))
    with pytest.raises(ValueError):
        oracle.unpermute_bwd(w["g_y"], w["x"], w["probs"], rim,
                             g_rows=np.zeros((w["H"], rim.size), np.uint16)[:, ::2])


def test_sharded_oracle_reports_its_sample():
    so = bench.ShardedOracle(2, 8)
    try:
        assert so.w["T"] == 16 and so.step() > 0
        d = so.describe(1, 0.5)
        assert "2 threads" in d and "bit-identical" in d
    finally:
        so.close()


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the keys the driver reads, on the GPU arm's metric."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"], capture_output=True, text=True,
                         timeout=600, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_traffic_source_check_ignores_comments_only():
    """The DRAM-traffic figures are keyed to the kernel code: a comment or
    blank-line edit keeps the key, a code edit changes it."""
    src = "int a = 1;  // one\n/* block\n   comment */\n\nint b = a + 2;\n"
    assert bench.code_only(src) == "int a = 1;\nint b = a + 2;"
    assert bench.code_only(src.replace("// one", "// two")) == bench.code_only(src)
    assert bench.code_only(src.replace("a + 2", "a + 3")) != bench.code_only(src)
