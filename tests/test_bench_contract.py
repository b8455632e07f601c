"""The benchmark's accounting and its CPU (reference) arm, on the CPU.

The masked-FLOP count is pinned to a brute-force count of the mask
inequalities; the algorithmic bytes to a hand count on a tiny batch; and the
`--impl reference` line (the oracle timed on the host) to the keys the
benchmark contract names.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _brute_counts(lq, lk, causal, wl):
    out = []
    for i in range(lq):
        n = 0
        for j in range(lk):
            ok = True
            if causal and not (j <= i + lk - lq):
                ok = False
            if wl >= 0 and not (j + lq + wl >= lk + i):
                ok = False
            n += ok
        out.append(n)
    return np.array(out)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("wl", [-1, 0, 3, 40])
def test_valid_counts_match_the_mask(causal, wl):
    rng = np.random.default_rng(11)
    for _ in range(20):
        lk = int(rng.integers(1, 60))
        lq = int(rng.integers(1, lk + 1)) if causal else int(rng.integers(1, 60))
        assert np.array_equal(bench.valid_counts(lq, lk, causal, wl),
                              _brute_counts(lq, lk, causal, wl))


def test_accounting_by_hand():
    # one decode row over 33 keys in pages of 16: 3 pages, every key live
    pb = workloads.make_paged_batch([1], [33], 4, 2, 8, 16, "bf16", 1)
    flops, byts = bench.accounting(pb, False, -1)
    assert flops == 4 * 8 * 4 * 33
    assert byts == 33 * 2 * 8 * 2 * 2 + 1 * 4 * 8 * 2 * 2 + 1 * 4 * 4 + 4 * 3
    # window 4 keeps keys 28..32 of the single row: 5 keys in pages 1 and 2
    flops, byts = bench.accounting(pb, True, 4)
    assert flops == 4 * 8 * 4 * 5
    assert byts == 5 * 2 * 8 * 2 * 2 + 4 * 8 * 2 * 2 + 4 * 4 + 4 * 2


def test_reference_arm_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert set(cb) >= {"value", "unit", "cores", "kind", "sample"}
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("batch decode")
    # every core of the affinity, and a measured step: steps x ms_per_step is
    # the time the timed steps took (nothing scaled up from a sample)
    assert cb["cores"] == len(os.sched_getaffinity(0))
    assert abs(line["ms_per_step"] * line["steps"] / 1e3 - line["timed_wall_s"]) <= \
        0.1 * line["timed_wall_s"] + 0.05
