"""Benchmark of the fused block-scaled MoE layer on GB300.

One step = one forward of the whole layer (dispatch, MXFP8 quantisation,
GEMM1 + SwiGLU + re-quantisation, GEMM2, combine) over one batch of synthetic
rows.  Default workload: decode, fixed-slot, DeepSeek-V4-Flash shape (T=128,
H=5120, I=2304, 384 experts, top-6, MTPR 128, clamp-10 SwiGLU).

Prints one JSON line.  `value` is MoE-layer tokens/s with inputs resident in
HBM; `e2e` is the same metric through the public API with host buffers (H2D of
the step's inputs and D2H of its output inside the timed region); `roofline`
reports the dominant kernel against the measured HBM copy bandwidth: the
single-launch fused kernel (the whole layer) when the forward takes that path,
as decode does, else GEMM1 (it streams 2/3 of the active-expert weight bytes);
`cpu_baseline` times the CPU oracle on a bounded sample of the same workload.

`per_config` (one GPU) adds one record per other workload (small-M, large-M and
skewed prefill by default): median step time, tokens/s, the layer's fraction of
the measured HBM copy rate and of the dense FP8 tensor peak (2 x the measured
BF16 rate), the dominant kernel's, and the CPU oracle (all cores and one core).
Stage times come from a separate profiled pass, so the timed steps carry no
events but their own.

--impl reference times the CPU oracle itself on the same workload (bounded
row sample per step) and prints the same line with "impl": "reference".
Multi-GPU (torchrun): every rank runs an independent replica (the layer does
not shard on one GPU per box); value = tokens of all ranks / max rank time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Fused MoE tokens/s per T; decode % of HBM BW, prefill % of FP8 MMA peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decode_flash")
    p.add_argument("--cpu-rows", type=int, default=16, help="oracle sample rows for the CPU baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--path", default="auto", choices=["auto", "fused", "multi"],
                   help="layer path (auto: the fused kernel where the handle allows it)")
    p.add_argument("--per-config", default="smallm_pro,largem_pro,skewed_flash",
                   help="other workloads measured after the headline one (comma list, '' for none; one GPU only)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [ln for ln in out.splitlines() if ln.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_bytes_flops(w, ids):
    """Algorithmic HBM bytes and FLOPs of one forward from the actual routing."""
    import numpy as np
    v = ids[: w.nvr].reshape(-1)
    v = v[(v >= 0) & (v < w.E)]
    if w.dispatch == "fixed":
        rows = len({(int(t), int(e)) for t, row in enumerate(ids[: w.nvr]) for e in row if 0 <= e < w.E})
    else:
        rows = int(v.size)
    active = int(np.unique(v).size)
    H, I = w.H, w.I
    w13 = active * 2 * I * H * 17 // 32          # codes (1/2 B) + scales (1/32 B) per element
    w2 = active * H * I * 17 // 32
    x_bytes = w.nvr * H * 2 + w.T * H * 2         # read x, write out (bf16)
    gemm1_act = rows * (H + H // 32) + rows * (I + I // 32)  # read packed rows, write h
    flops = 6 * H * I * rows
    return {"active": active, "routes": rows, "w13": w13, "w2": w2, "step": w13 + w2 + x_bytes,
            "gemm1": w13 + gemm1_act, "flops": flops}


# source files of each kernel whose ncu traffic figure is committed under profiles/
KERNEL_SOURCES = {  # the kernels' sources and the launcher that builds their tensor maps
    "gemm1": ("moe_gemm.cu", "gemm_common.cuh", "ptx.cuh", "moe_api.cu"),
    "fused": ("moe_fused.cu", "gemm_common.cuh", "layer_rows.cuh", "ptx.cuh", "moe_api.cu"),
}


def source_sha(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_scaled_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, workload):
    """dram bytes per launch of `kernel` from a committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_sha") == source_sha(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def max_over_ranks(v: float, world: int, device=None) -> float:
    """The largest of every rank's `v` (the slowest rank's time); `v` itself on one rank."""
    if world <= 1:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(valid_rows_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s: the valid rows of every rank's steps over the slowest rank's time."""
    return valid_rows_per_step * steps * world / (max_ms / 1e3)


def cpu_baseline(w, x, ids, wts, Wh, rows_n, rows_1core=2):
    """The oracle as it stands on the host cores: a seeded sample of `rows_n` valid rows on every core of
    the affinity mask, and `rows_1core` rows on one core."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(np.arange(w.nvr), size=min(rows_n, w.nvr), replace=False)).astype(np.int32)
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    t0 = time.perf_counter()
    oracle.moe_forward(x, ids, wts, Wh, num_valid_rows=w.nvr, swiglu_limit=w.swiglu_limit, rows=rows,
                       nthreads=threads)
    dt = time.perf_counter() - t0
    r1 = rows[:rows_1core]
    t0 = time.perf_counter()
    oracle.moe_forward(x, ids, wts, Wh, num_valid_rows=w.nvr, swiglu_limit=w.swiglu_limit, rows=r1, nthreads=1)
    dt1 = time.perf_counter() - t0
    return {"value": len(rows) / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} of {w.nvr} valid rows of the {w.name} workload (seeded), "
                      f"{dt:.2f} s wall on {threads} threads",
            "value_1core": len(r1) / dt1, "sample_1core": f"{len(r1)} of those rows on 1 thread, {dt1:.2f} s wall"}


def fp8_peaks(bf16_tf, bf16_tf_sus):
    """Dense FP8 tensor peak: the measured cuBLAS BF16 rate times the nominal FP8 / BF16 ratio (4.5 / 2.25)."""
    return 2.0 * bf16_tf, 2.0 * bf16_tf_sus


def measure(w, dev, args, path, stream, flush, world=1, e2e=False):
    """One workload on this rank's GPU: warm-up, `args.steps` timed forwards (CUDA events on the forward's
    stream, L2 flushed before each outside the events, no profiling events inside), then a separate
    profiled pass for the per-stage times.  Inputs are device-resident; `e2e` adds the end-to-end pass."""
    import numpy as np
    import torch

    import block_scaled_moe_gb300 as bm
    import synth
    x = synth.make_x(w)
    ids, wts = synth.make_routing(w)
    W = synth.make_weights(w, dev)
    layer = bm.BlockScaledMoE(w.H, w.I, w.E, w.K, w.capacity, dispatch=w.dispatch, swiglu_limit=w.swiglu_limit,
                              path=path)
    layer.bind_weights(*W)
    xd = x.to(dev)
    idsd = torch.from_numpy(ids).to(dev)
    wtsd = torch.from_numpy(wts).to(dev)
    nvrd = torch.tensor([w.nvr], dtype=torch.int32, device=dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)

    def step():
        layer.forward(xd, idsd, wtsd, nvrd, out=out, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    status = layer.read_status()
    if status:
        raise RuntimeError(f"device status {status:#x} after warm-up ({w.name})")

    # ---- timed region: device-resident inputs, L2 flushed between steps (outside the events)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = layer.launches
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        for i in range(args.steps):
            flush.fill_(1.0)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    launches = layer.launches - launches0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # ---- per-stage times in a separate profiled pass (CUDA events between the stages)
    layer.set_profile(True)
    stage_ms = []
    for _ in range(max(3, min(args.steps, 10))):
        flush.fill_(1.0)
        step()
        stage_ms.append(layer.profile_ms())
    layer.set_profile(False)
    torch.cuda.synchronize()

    r = {"w": w, "ids": ids, "x": x, "wts": wts, "W": W, "step_ms": step_ms, "launches": launches,
         "stage_ms": [statistics.mean(s[i] for s in stage_ms) for i in range(5)], "path": layer.last_path,
         "scheme": layer.scheme, "clocks": clk.summary()}
    if e2e:
        # ---- end to end: pinned host buffers, H2D inputs + forward + D2H output per step.  The step's
        # inputs (x, top-k ids and weights, the row count) sit in one pinned host buffer and one device
        # buffer at 256-byte aligned offsets, so that each step is one H2D copy (a copy's fixed cost on
        # the GPU timeline is a few microseconds, more than the transfer of these sizes)
        parts = [x.contiguous().view(torch.uint8).reshape(-1), torch.from_numpy(ids).view(torch.uint8).reshape(-1),
                 torch.from_numpy(wts).view(torch.uint8).reshape(-1),
                 torch.tensor([w.nvr], dtype=torch.int32).view(torch.uint8)]
        offs, total = [], 0
        for t in parts:
            offs.append(total)
            total += (t.numel() + 255) // 256 * 256
        inh = torch.empty(total, dtype=torch.uint8).pin_memory()
        for o, t in zip(offs, parts):
            inh[o:o + t.numel()].copy_(t)
        ind = torch.empty(total, dtype=torch.uint8, device=dev)
        xe = ind[offs[0]:offs[0] + parts[0].numel()].view(torch.bfloat16).view(w.T, w.H)
        ie = ind[offs[1]:offs[1] + parts[1].numel()].view(torch.int32).view(w.T, w.K)
        we = ind[offs[2]:offs[2] + parts[2].numel()].view(torch.float32).view(w.T, w.K)
        ne = ind[offs[3]:offs[3] + 4].view(torch.int32)
        outh = torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory()

        def e2e_step():
            ind.copy_(inh, non_blocking=True)
            layer.forward(xe, ie, we, ne, out=out, stream=stream)
            outh.copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(1.0)
            es[i].record(stream)
            e2e_step()
            ee[i].record(stream)
        torch.cuda.synchronize()
        r["e2e_ms"] = [s.elapsed_time(e) for s, e in zip(es, ee)]
        r["h2d"] = total  # the inputs' bytes plus their alignment padding (< 1 KB)
        r["d2h"] = outh.numel() * 2
    layer.close()
    return r


def config_record(r, hbm_gbs, bf16_tf, bf16_tf_sus, peak_src, cpu=None):
    """One workload's record: median step time, tokens/s, the layer's HBM and FP8 tensor fractions, the
    dominant kernel's, and the CPU oracle next to it."""
    w = r["w"]
    wb = workload_bytes_flops(w, r["ids"])
    med = statistics.median(r["step_ms"])
    fp8, fp8_sus = fp8_peaks(bf16_tf, bf16_tf_sus)
    gbs = wb["step"] / (med / 1e3) / 1e9
    tf = wb["flops"] / (med / 1e3) / 1e12
    fused = r["path"] == "fused"
    k_ms = r["stage_ms"][2]
    k_bytes = wb["step"] if fused else wb["gemm1"]
    k_flops = wb["flops"] if fused else 4 * w.H * w.I * wb["routes"]
    ridge = fp8 * 1e12 / (hbm_gbs * 1e9)
    rec = {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "topk": w.K, "num_valid_rows": w.nvr,
           "dispatch": r["scheme"], "path": r["path"], "swiglu_limit": w.swiglu_limit, "routes": wb["routes"],
           "active_experts": wb["active"], "steps": len(r["step_ms"]), "ms_median": med,
           "ms_mean": statistics.mean(r["step_ms"]), "tokens_per_s": w.nvr / (med / 1e3),
           "roofline": {"bytes_per_step": wb["step"], "flops_per_step": wb["flops"],
                        "arithmetic_intensity": wb["flops"] / wb["step"], "ridge_flop_per_byte": ridge,
                        "bound": "hbm" if wb["flops"] / wb["step"] < ridge else "tensor",
                        "hbm": {"achieved_gbs": gbs, "peak_gbs": hbm_gbs, "frac": gbs / hbm_gbs},
                        "fp8": {"achieved_tflops": tf, "peak_tflops": fp8, "frac": tf / fp8,
                                "peak_tflops_sustained": fp8_sus, "frac_of_sustained": tf / fp8_sus},
                        "peak_source": peak_src,
                        "fp8_peak_derivation": "2 x the measured cuBLAS BF16 rate (nominal dense FP8 / BF16 = "
                                               "4.5 / 2.25 PFLOP/s); burst figure for a step timed alone"},
           "dominant_kernel": {"name": "fused layer kernel" if fused else "GEMM1", "ms_mean": k_ms,
                               "hbm_frac": k_bytes / (k_ms / 1e3) / 1e9 / hbm_gbs,
                               "fp8_frac": k_flops / (k_ms / 1e3) / 1e12 / fp8},
           "stage_ms_mean": r["stage_ms"],
           "stages": ["-", "-", "fused kernel", "-", "-"] if fused else
                     ["dispatch", "quant+scatter", "gemm1", "gemm2", "combine"],
           "gpu_launches_per_step": r["launches"] / max(1, len(r["step_ms"])), "clocks": r["clocks"]}
    if cpu is not None:
        rec["cpu_baseline"] = cpu
    return rec


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import numpy as np
    import torch

    import synth
    w = synth.get(args.workload)

    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle
        oracle.build()
        x, ids, wts = synth.make_x(w), *synth.make_routing(w)
        Wh = [t.cpu() for t in synth.make_weights(w, "cuda" if torch.cuda.is_available() else "cpu")]
        threads = len(os.sched_getaffinity(0))
        rng = np.random.default_rng(2)
        times, ntok = [], 0
        for i in range(args.warmup + args.steps):
            rows = np.sort(rng.choice(np.arange(w.nvr), size=min(4, w.nvr), replace=False)).astype(np.int32)
            t0 = time.perf_counter()
            oracle.moe_forward(x, ids, wts, Wh, num_valid_rows=w.nvr, swiglu_limit=w.swiglu_limit, rows=rows,
                               nthreads=threads)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                times.append(dt)
                ntok += len(rows)
        total = sum(times)
        val = ntok / total
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "topk": w.K,
                           "num_valid_rows": w.nvr, "dispatch": w.dispatch, "step_sample_rows": 4},
                "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                 "sample": f"4 seeded rows of {w.nvr} per step, {args.steps} steps"},
                "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import __graft_entry__
    __graft_entry__.build()

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)  # before the process group, so that NCCL binds this rank's GPU
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # 512 MiB > 129 MB L2
    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = peaks()

    r = measure(w, dev, args, args.path, stream, flush, world=world, e2e=True)
    step_ms = r["step_ms"]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = job_throughput(w.nvr, args.steps, world, total_ms)
    e2e_ms = max_over_ranks(sum(r["e2e_ms"]), world, dev)
    e2e_value = job_throughput(w.nvr, args.steps, world, e2e_ms)

    # ---- roofline of the dominant kernel from its CUDA-event durations (stage slot 2 holds GEMM1, or the
    # whole fused kernel on the single-launch path), measured in the profiled pass
    wb = workload_bytes_flops(w, r["ids"])
    fused = r["path"] == "fused"
    kern = "fused" if fused else "gemm1"
    k_ms = r["stage_ms"][2]
    k_bytes = wb["step"] if fused else wb["gemm1"]
    achieved = k_bytes / (k_ms / 1e3) / 1e9
    traffic = traffic_for(kern, w.name)
    step_gbs = wb["step"] / (total_ms / args.steps / world / 1e3) / 1e9

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8 x mxfp4 (e4m3 x e2m1, fp32 accumulate)",
            "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "topk": w.K,
                       "num_valid_rows": w.nvr, "dispatch": r["scheme"], "capacity": w.capacity,
                       "path": r["path"],
                       "swiglu_limit": w.swiglu_limit, "routes": wb["routes"], "active_experts": wb["active"],
                       "l2": "512 MiB buffer written between timed steps (outside the events)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"kernel": ("fused layer (one cooperative launch: dispatch, MXFP8 quant, tcgen05 GEMM1 + "
                                    "SwiGLU/MXFP8, tcgen05 GEMM2, combine)") if fused else
                                   "GEMM1 (tcgen05 block-scaled, W13 stream + SwiGLU/MXFP8 epilogue)",
                         "bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "traffic": traffic, "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": k_bytes, "launch_ms": k_ms,
                         "launch_ms_from": "separate profiled pass (CUDA events on the forward's stream)"},
            "step_roofline": {"bytes_per_step": wb["step"], "achieved_gbs": step_gbs,
                              "frac_of_hbm": step_gbs / hbm_gbs,
                              "tflops": wb["flops"] / (total_ms / args.steps / world / 1e3) / 1e12,
                              "ms_median": statistics.median(step_ms),
                              "stage_ms_mean": r["stage_ms"],
                              "stages": (["-", "-", "fused kernel", "-", "-"] if fused else
                                         ["dispatch", "quant+scatter", "gemm1", "gemm2", "combine"])},
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": r["launches"] * world,
            "clocks": r["clocks"]}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, r["x"], r["ids"], r["wts"], [t.cpu() for t in r["W"]], args.cpu_rows)
        line["cpu_baseline"] = cpu
    del r["W"]
    # ---- the other workloads on this GPU, one record each (one GPU only: the scaling runs keep to the
    # headline workload)
    names = [n for n in args.per_config.split(",") if n and n != w.name] if world == 1 else []
    if names:
        per = {w.name: config_record(r, hbm_gbs, bf16_tf, bf16_tf_sus, peak_src, cpu)}
        del r
        torch.cuda.empty_cache()
        for n in names:
            wn = synth.get(n)
            rn = measure(wn, dev, args, "auto", stream, flush)
            cn = None
            if not args.no_cpu_baseline:
                cn = cpu_baseline(wn, rn["x"], rn["ids"], rn["wts"], [t.cpu() for t in rn["W"]], 8)
            del rn["W"]
            torch.cuda.empty_cache()
            per[n] = config_record(rn, hbm_gbs, bf16_tf, bf16_tf_sus, peak_src, cn)
            del rn
            torch.cuda.empty_cache()
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
