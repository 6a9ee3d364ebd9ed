"""Host-side checks of the benchmark's accounting (no GPU).

* the algorithmic bytes and FLOPs of one forward (the roofline numerator) on a hand-worked routing:
  active experts, routes under both dispatch schemes (a repeated expert in a row shares its fixed
  slot), MXFP4 weight bytes of 17/32 byte per element (codes and E8M0 scales), x read and out
  written in BF16;
* on the decode workload, the same figures from the definition: every active expert streams its
  W13 (2I x H) and W2 (H x I) once;
* the traffic record is used only for a kernel whose sources still hash to the recorded value;
* the reference arm prints one JSON line with the contract's keys.
"""

import json
import os
import subprocess
import sys
import types

import numpy as np

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _w(**kw):
    return types.SimpleNamespace(**kw)


def test_bytes_and_flops_on_a_hand_worked_routing():
    ids = np.array([[0, 1], [1, -1], [3, 3]], dtype=np.int32)
    H = I = 128
    for dispatch, routes in (("compact", 5), ("fixed", 4)):  # fixed: (2, 3) twice is one slot
        w = _w(nvr=3, T=3, E=4, H=H, I=I, dispatch=dispatch)
        r = bench.workload_bytes_flops(w, ids)
        assert r["active"] == 3 and r["routes"] == routes
        assert r["w13"] == 3 * 17408      # 2*128*128 elements * 17/32 byte
        assert r["w2"] == 3 * 8704        # 128*128 elements * 17/32 byte
        assert r["step"] == 3 * 17408 + 3 * 8704 + 3 * 128 * 2 * 2
        assert r["flops"] == 6 * H * I * routes
    # rows at or past num_valid_rows and ids >= E route nowhere
    w = _w(nvr=1, T=3, E=4, H=H, I=I, dispatch="compact")
    r = bench.workload_bytes_flops(w, np.array([[0, 9], [1, 2], [3, 3]], dtype=np.int32))
    assert r["active"] == 1 and r["routes"] == 1
    assert r["step"] == 17408 + 8704 + 1 * 128 * 2 + 3 * 128 * 2


def test_decode_workload_bytes_follow_the_definition():
    w = synth.get("decode_flash")
    ids, _ = synth.make_routing(w)
    r = bench.workload_bytes_flops(w, ids)
    active = len(set(int(e) for e in ids[: w.nvr].reshape(-1) if 0 <= e < w.E))
    assert r["active"] == active
    per_expert = (2 * w.I * w.H + w.H * w.I) * 17 / 32  # 12.53 MB of W13 + 6.27 MB of W2
    assert abs(r["w13"] + r["w2"] - active * per_expert) <= 2 * active
    assert 6.0e9 < r["step"] < 6.5e9


def test_traffic_record_needs_matching_sources():
    assert bench.traffic_for("fused", "no_such_workload") is None
    t = bench.traffic_for("fused", "decode_flash")
    rec = json.load(open(os.path.join(ROOT, "profiles", "fused_traffic.json")))["decode_flash"]
    if rec["source_sha"] == bench.source_sha("fused"):
        assert t == float(rec["dram_bytes_per_launch"])
    else:
        assert t is None


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny"


def test_per_config_record_fractions():
    """A per-workload record from hand-set timings: HBM and FP8 fractions follow from the algorithmic
    bytes and FLOPs over the median step time and the stated peaks."""
    w = synth.get("largem_pro")
    ids, _ = synth.make_routing(w)
    r = {"w": w, "ids": ids, "step_ms": [3.0, 2.0, 4.0], "launches": 21, "stage_ms": [0.1, 0.1, 1.5, 1.0, 0.1],
         "path": "multi", "scheme": "compact", "clocks": {}}
    rec = bench.config_record(r, 6000.0, 2000.0, 1800.0, "measured", cpu={"value": 1.0})
    wb = bench.workload_bytes_flops(w, ids)
    assert rec["ms_median"] == 3.0 and rec["tokens_per_s"] == w.nvr / 3e-3
    assert abs(rec["roofline"]["hbm"]["frac"] - wb["step"] / 3e-3 / 6000e9) < 1e-12
    assert rec["roofline"]["fp8"]["peak_tflops"] == 4000.0
    assert abs(rec["roofline"]["fp8"]["frac"] - wb["flops"] / 3e-3 / 4000e12) < 1e-12
    assert rec["roofline"]["bound"] == "hbm"          # AI ~ 464 F/B below the ridge of 4000/6 ~ 667
    k = rec["dominant_kernel"]
    assert k["name"] == "GEMM1" and abs(k["fp8_frac"] - 4 * w.H * w.I * wb["routes"] / 1.5e-3 / 4000e12) < 1e-12
    assert rec["gpu_launches_per_step"] == 7 and rec["cpu_baseline"] == {"value": 1.0}
