"""Host-side logic of bench.py, on the CPU: the FLOP convention, the count of
visible score pairs under a window band, the clock-sample summary, the
source-digest check that guards the committed ncu traffic figures, and the
reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

import bench
from seeded_inputs import CONFIGS, PACKED_CONFIGS, Workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def brute_pairs(n, causal, window):
    left, right = window if window is not None else (-1, -1)
    count = 0
    for i in range(n):
        for j in range(n):
            if causal and j > i:
                continue
            if left >= 0 and j < i - left:
                continue
            if right >= 0 and j > i + right:
                continue
            count += 1
    return count


@pytest.mark.parametrize("n", [1, 2, 7, 33])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (0, 0), (3, -1), (-1, 2), (4, 5)])
def test_band_pairs_matches_brute_force(n, causal, window):
    assert bench.band_pairs(n, causal, window) == brute_pairs(n, causal, window)


def test_flop_convention_at_the_causal_drill_size():
    # 4 * B * H * S^2 * D / 2 forward (causal halves it), backward 2.5x.
    f, b = bench.conv_flops(CONFIGS["c2"])
    assert f == 4 * 4 * 16 * 4096 ** 2 * 64 / 2 == 137_438_953_472
    assert b == 2.5 * f
    f4, _ = bench.conv_flops(CONFIGS["c4"])
    assert f4 == 4 * 2 * 32 * 8192 ** 2 * 128


def test_window_flops_count_visible_pairs():
    w = Workload("w", 1, 2, 50, 16, "fp16", True, window=(7, -1))
    f, _ = bench.conv_flops(w)
    assert f == 4 * 16 * 2 * brute_pairs(50, True, (7, -1))


def test_kernel_work_names_the_launched_forward():
    assert "fa_fwd4p_kernel" in bench.kernel_work(CONFIGS["c2"])           # fixed length, S <= 6144
    assert "fa_fwd4_kernel" in bench.kernel_work(CONFIGS["leaderboard"])   # S = 16384
    assert "fa_fwd4_kernel" in bench.kernel_work(CONFIGS["window"])        # a window band
    assert "fa_fwd4_kernel" in bench.kernel_work(CONFIGS["c2"], general=True)  # split-KV
    assert "fa_fwd_kernel" in bench.kernel_work(CONFIGS["c4"])
    kind, amount = bench.kernel_work(CONFIGS["c2"])["fa_bwd_dkdv_kernel"]
    assert kind == "tensor" and amount == 2 * bench.conv_flops(CONFIGS["c2"])[0]


def test_backward_intervals_follow_the_launch_order():
    """At D <= 64 with fixed lengths and no window the dQ pass computes Delta and runs first;
    otherwise the Delta kernel, the dK/dV pass and the dQ pass run in that order."""
    fused = ["fa_bwd_dq_kernel", "fa_bwd_dkdv_kernel", None]
    split = ["fa_bwd_preprocess_kernel", "fa_bwd_dkdv_kernel", "fa_bwd_dq_kernel"]
    assert bench.bwd_intervals(CONFIGS["c2"]) == fused
    assert bench.bwd_intervals(CONFIGS["c4"]) == split            # D = 128
    assert bench.bwd_intervals(CONFIGS["window"]) == split        # a window band
    assert bench.bwd_intervals(PACKED_CONFIGS["varlen"]) == split
    assert "fa_bwd_preprocess_kernel" not in bench.kernel_work(CONFIGS["c2"])
    assert "fa_bwd_preprocess_kernel" in bench.kernel_work(CONFIGS["c4"])


def test_traffic_is_dropped_when_the_kernel_sources_change(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        table = json.load(f)["bytes_per_launch"]["c2"]
    monkeypatch.setattr(bench, "sources_digest", lambda k: table[k]["sources_digest"])
    assert bench.load_traffic("c2") == {k: r["bytes"] for k, r in table.items()}
    assert bench.load_traffic("no-such-workload") == {}
    # A change to one kernel's sources drops that kernel's figure only.
    fwd = next(k for k in table if k.startswith("fa_fwd"))
    monkeypatch.setattr(bench, "sources_digest",
                        lambda k: "0000000000000000" if k == fwd else table[k]["sources_digest"])
    got = bench.load_traffic("c2")
    assert fwd not in got and got["fa_bwd_dkdv_kernel"] == table["fa_bwd_dkdv_kernel"]["bytes"]


def test_every_kernel_lists_existing_sources():
    for kernel, files in bench.KERNEL_SOURCES.items():
        for rel in files:
            assert os.path.exists(os.path.join(ROOT, rel)), (kernel, rel)
        assert len(bench.sources_digest(kernel)) == 16


def test_clock_summary_reports_throttle_reasons():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [(1.0, ["0", "1900", "2070", "800", "0x0", "Not Active", "Not Active", "Not Active", "Active"]),
                 (1.1, ["0", "2000", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]),
                 (9.0, ["0", "100", "2070", "90", "0x0", "Active", "Not Active", "Not Active", "Not Active"])]
    out = s.summary(0.9, 1.2)
    assert out["samples"] == 2 and out["sm_mhz"] == 1950 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"] and out["power_w_max"] == 900


def test_reference_arm_prints_one_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["dtype"] == "f64"
