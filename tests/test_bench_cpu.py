"""bench.py's contract and host-side helpers, without a GPU.

- the reference arm (`--impl reference`, the CPU oracle) prints one JSON line with the
  keys the driver reads;
- the workloads are the metric's five configurations with their sizes;
- the algorithmic bytes and flops follow their definitions;
- every candidate plan the sweep would time passes the library's plan check;
- the committed DRAM-traffic table still matches the router kernel's source (else the
  bench line's `traffic` turns null).
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--cpu-budget", "0.5"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] >= 3
    assert d["unit"] == "us/call" and d["higher_is_better"] is False and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"] and "model" not in d["config"]


def test_workloads_are_the_metric_configs():
    pts = {name: bench.workload_points(name) for name in ("smallest", "router", "decode", "mlp", "prefill")}
    assert [(p["M"], p["N"], p["K"], p["bias"]) for p in pts["smallest"]] == [(4, 256, 2048, False)]
    kn = {(p["K"], p["N"]) for p in pts["router"]}
    assert kn == {(4096, 256), (6144, 256), (7168, 256), (7168, 384), (2880, 128)}
    assert sorted({p["M"] for p in pts["router"]}) == list(range(1, 17)) and len(pts["router"]) == 80
    assert [(p["M"], p["N"], p["K"]) for p in pts["decode"]] == [(m, 2112, 7168) for m in (1, 2, 4, 8, 16, 32, 64)]
    assert [(p["M"], p["N"], p["K"], p["bias"]) for p in pts["mlp"]] == [(m, 14336, 4096, True) for m in (1, 8, 64, 256)]
    assert len(pts["prefill"]) == 12
    assert {(p["M"], p["K"], p["N"], p["bias"]) for p in pts["prefill"]} == {
        (m, k, n, b) for m in (2048, 8192) for (k, n) in ((7168, 2112), (4096, 14336), (7168, 7168))
        for b in (False, True)}


def test_algorithmic_work():
    assert bench.algo_bytes(4, 256, 2048, False) == 2 * 256 * 2048 + 2 * 4 * 2048 + 2 * 4 * 256
    assert bench.algo_bytes(4, 256, 2048, True) == bench.algo_bytes(4, 256, 2048, False) + 2 * 256
    assert bench.algo_flops(2048, 7168, 7168, False) == 2 * 2048 * 7168 * 7168


@pytest.mark.parametrize("shape", [(4, 256, 2048), (16, 384, 7168), (8, 2112, 7168), (64, 2112, 7168),
                                   (64, 14336, 4096), (256, 14336, 4096), (2048, 7168, 7168)])
def test_sweep_candidates_pass_the_plan_check(lib, shape):
    M, N, K = shape
    cands = bench.candidate_plans(lib, M, N, K)
    assert cands
    bad = []
    for p in cands:
        try:
            lib.plan_check(M, N, K, p)
        except lib.BF16LinearError:
            bad.append(p.as_dict())
    assert not bad, bad[:3]
    assert lib.plan_check(M, N, K, lib.plan(M, N, K)).grid > 0


def test_kernel_source_hash_covers_every_kernel(lib):
    for name in lib.KERNEL_NAMES.values():
        h = bench.kernel_source_hash(name)
        assert isinstance(h, str) and len(h) == 12, name


def test_committed_traffic_matches_the_router_kernel():
    """profiles/dram_traffic.txt holds the ncu DRAM bytes of the router kernels at the source they were
    captured from; the dominant router kernel's lines must still match its source."""
    shapes = [(m, n, k) for (k, n) in ((7168, 256), (7168, 384)) for m in range(5, 17)]
    lines = [l.split() for l in open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) if l.startswith("dotmma ")]
    listed = {(int(f[1]), int(f[2]), int(f[3])) for f in lines}
    some = [s for s in shapes if s in listed]
    assert some, "no dotmma shape in the traffic table"
    t = bench.ncu_traffic("dotmma", some)
    assert t is not None and t > 0
    algo = sum(bench.algo_bytes(m, n, k, False) for (m, n, k) in some) / len(some)
    assert 0.95 < t / algo < 1.2


class _FakeSmi:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_and_slowdown_retime_rule():
    """The nvidia-smi lines become the clocks record; hardware and thermal slowdowns call for a
    second timed region, a power cap alone does not."""
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi()
    s.lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1980, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    c = s.stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"] and bench.slowdowns(c) == []
    s.lines.append("0, 1500, 2070, 1400.0, 0x88, Active, Not Active, Active, Not Active")
    c = s.stop()
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert bench.slowdowns(c) == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.slowdowns({"sm_mhz": None, "reasons": ["nvidia-smi unavailable"]}) == []
