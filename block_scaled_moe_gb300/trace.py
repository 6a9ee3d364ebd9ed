"""Pipeline traces of the tracing build (libblockmoe_trace.so, -DBMOE_TRACE).

    BMOE_LIB_VARIANT=trace python -m block_scaled_moe_gb300.trace WORKLOAD [--path multi|fused]

runs one seeded workload (three warm-up forwards, then one forward after a 512 MiB write that
evicts the weights from L2) and prints what the kernels stamped:

* multi-kernel path, per stand-alone GEMM: every CTA's start and end (globaltimer), so the spread of
  finishing times (the balance of the unit list over the CTAs), and, for CTAs 0 and 1, per K stage
  the producer's wait for a free stage, the load latency from issue to a full stage, the MMA warp's
  wait and issue times and the stage period (clock64 cycles);
* fused path: per CTA the phase boundaries and wait totals of the single-launch kernel (ns).

The tracing build only adds stores of clock stamps; it is a separate library, never the one
`__graft_entry__.build()` makes for the product path.
"""

from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np

GEMM_STAGE_EVENTS = 8      # per CTA: stage stamps of 8 events x 512 stages (CTAs 0 and 1)
GEMM_JOBS = 512
GEMM_PER = 2 * GEMM_STAGE_EVENTS * GEMM_JOBS + 2 * 1024   # int64 per GEMM: stage stamps, then CTA start/end


def gemm_trace(lib, n_sms: int) -> dict:
    """The stand-alone GEMMs' stamps of the last multi-kernel forward: per GEMM, `stages` [2 CTAs][8][512]
    (0 producer got a free stage, 1 producer issued it, 2 MMA warp saw it full, 3 MMA warp issued;
    4 / 5 epilogue saw / released each unit's accumulator; 6 / 7 weight-scale warp got / filled the
    stage) and `cta` [n_sms][2] start / end ns."""
    buf = np.zeros(2 * GEMM_PER, np.int64)
    lib.bmoe_gemm_trace_copy.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    rc = lib.bmoe_gemm_trace_copy(buf.ctypes.data, buf.nbytes)
    if rc:
        raise RuntimeError(f"bmoe_gemm_trace_copy failed ({rc}): is this the tracing build?")
    out = {}
    for gi, name in enumerate(("gemm1", "gemm2")):
        b = buf[gi * GEMM_PER:(gi + 1) * GEMM_PER]
        out[name] = {"stages": b[:2 * GEMM_STAGE_EVENTS * GEMM_JOBS].reshape(2, GEMM_STAGE_EVENTS, GEMM_JOBS),
                     "cta": b[2 * GEMM_STAGE_EVENTS * GEMM_JOBS:].reshape(1024, 2)[:n_sms]}
    return out


def summarize_gemm(name: str, t: dict) -> list:
    lines = []
    se = t["cta"].astype(np.float64)
    ok = se[:, 1] > 0
    t0 = se[ok, 0].min()
    en = (se[ok, 1] - t0) / 1e3
    lines.append(f"{name}: {int(ok.sum())} CTAs; end min {en.min():.1f} med {np.median(en):.1f} "
                 f"p90 {np.percentile(en, 90):.1f} max {en.max():.1f} us; spread max-min {en.max() - en.min():.1f} us "
                 f"({100 * (en.max() - en.min()) / en.max():.1f}% of the kernel)")
    for cta in range(2):
        s = t["stages"][cta].astype(np.float64)
        n = int((s[1] > 0).sum())
        if n < 4:
            continue
        P0, P1, M0, M1 = s[0, :n], s[1, :n], s[2, :n], s[3, :n]
        lines.append(f"  CTA {cta}, first {n} stages (cycles, median): producer wait for a free stage "
                     f"{np.median(P0[1:] - P1[:-1]):.0f}, load latency issue->full {np.median(M0 - P1):.0f}, "
                     f"MMA wait {np.median(M0[1:] - M1[:-1]):.0f}, MMA issue {np.median(M1 - M0):.0f}, "
                     f"stage period {np.median(np.diff(M0)):.0f} (mean {np.mean(np.diff(M0)):.0f})")
    return lines


FUSED_FIELDS = [(0, "start"), (1, "phase 1 (GEMMs) start"), (2, "first GEMM2 wait begin"), (5, "producer done"),
                (6, "MMA done"), (7, "epilogue done"), (9, "after the last grid barrier"), (10, "end")]


def fused_trace(lib, n_sms: int) -> np.ndarray:
    buf = np.zeros(1024 * 32, np.int64)
    lib.bmoe_fused_trace_copy.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    rc = lib.bmoe_fused_trace_copy(buf.ctypes.data, buf.nbytes)
    if rc:
        raise RuntimeError(f"bmoe_fused_trace_copy failed ({rc}): is this the tracing build?")
    return buf.reshape(1024, 32)[:n_sms]


FUSED_STAGES = 4096


FUSED_STAGE_EVENTS = 16


def fused_stage_trace(lib) -> np.ndarray:
    """[2 CTAs][16][4096] clock64 per K stage: 0 producer got a free stage, 1 issued it, 2 MMA chain 0 saw it
    full, 3 chain 0 issued, 4 weight-scale warp got it, 5 that warp filled it, 6 producer began waiting for
    it, 7 / 8 / 9 chains 1 / 2 / 3 (those there are) issued, 10 chain 0 began waiting for it, 11 the last
    chain saw it full; per unit
    of the CTA: 12 producer entered it, 13 decoded it, 14 issued its prefetch, 15 chain 0 decoded it."""
    buf = np.zeros(2 * FUSED_STAGE_EVENTS * FUSED_STAGES, np.int64)
    lib.bmoe_fused_stage_trace_copy.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    rc = lib.bmoe_fused_stage_trace_copy(buf.ctypes.data, buf.nbytes)
    if rc:
        raise RuntimeError(f"bmoe_fused_stage_trace_copy failed ({rc})")
    return buf.reshape(2, FUSED_STAGE_EVENTS, FUSED_STAGES)


def summarize_fused_stages(st: np.ndarray, n_g1: int) -> list:
    """Per-stage medians of CTA 0, GEMM1 stages [0, n_g1) and GEMM2 stages after them (cycles)."""
    lines = []
    s = st[0].astype(np.float64)
    n = int((s[3] > 0).sum())
    for name, lo, hi in (("GEMM1", 1, min(n_g1, n)), ("GEMM2", n_g1 + 1, n)):
        if hi - lo < 4:
            continue
        sl = slice(lo, hi)
        P0, P1, M0, M1, S0, S1 = (s[i] for i in range(6))
        lines.append(f"  CTA 0 {name} stages {lo}..{hi} (cycles, median): producer wait for a free stage "
                     f"{np.median(P0[sl] - P1[lo - 1:hi - 1]):.0f}, load latency issue->full "
                     f"{np.median(M0[sl] - P1[sl]):.0f}, scale warp fills {np.median(S1[sl] - P1[sl]):.0f} after the "
                     f"issue, MMA chain 0 wait {np.median(M0[sl] - M1[lo - 1:hi - 1]):.0f}, issue "
                     f"{np.median(M1[sl] - M0[sl]):.0f}, stage period {np.median(np.diff(M0[lo - 1:hi])):.0f} "
                     f"(mean {np.mean(np.diff(M0[lo - 1:hi])):.0f})")
    return lines


def transition_costs(st: np.ndarray, cta: int, n1: int, n_units: int, kt1: int, kt2: int) -> dict:
    """Unit transitions of one traced CTA (cycles, medians over its units after the first), per GEMM:
    the producer from its last issue of a unit to entering the next (`enter`), decoding it (`decode`),
    issuing the prefetch of the unit after it (`prefetch`), and from there to starting the wait for the
    new unit's first stage (`to_wait`, which holds the GEMM2 readiness wait); the MMA warp from its last
    issue to having decoded the next unit (`mma_decode`) and then to starting its first wait
    (`mma_to_wait`); and the period of chain 0 at the unit's first stage against the median period
    (`first_period`, `period`).  Unit u of the CTA starts at stage sum(kt of units < u); its first n1
    units are GEMM1 units of kt1 stages, the rest GEMM2 units of kt2."""
    s = st[cta].astype(np.int64)
    P1, M0, M1, PW, MW0 = s[1], s[2], s[3], s[6], s[10]
    U0, U1, U2, UM = s[12], s[13], s[14], s[15]
    starts = np.cumsum([0] + [kt1 if u < n1 else kt2 for u in range(n_units - 1)])
    n_stages = int((M1 > 0).sum())
    out = {}
    for name, units in (("GEMM1", np.arange(1, n1)), ("GEMM2", np.arange(n1 + 1, n_units))):
        units = units[starts[units] < n_stages]
        if len(units) == 0:
            continue
        b = starts[units]
        med = lambda a: float(np.median(a))
        periods = np.diff(M0[:n_stages])
        out[name] = {"units": int(len(units)), "enter": med(U0[units] - P1[b - 1]),
                     "decode": med(U1[units] - U0[units]), "prefetch": med(U2[units] - U1[units]),
                     "to_wait": med(PW[b] - U2[units]), "mma_decode": med(UM[units] - M1[b - 1]),
                     "mma_to_wait": med(MW0[b] - UM[units]), "first_period": med(M0[b] - M0[b - 1]),
                     "period": med(periods)}
    return out


def summarize_fused(t: np.ndarray) -> list:
    t = t.astype(np.float64)
    base = t[:, 0].min()
    lines = ["fused kernel, per CTA (us from the first CTA's start): min / median / max"]
    for c, name in FUSED_FIELDS:
        v = (t[:, c] - base) / 1e3
        lines.append(f"  {name:32s} {v.min():8.1f} {np.median(v):8.1f} {v.max():8.1f}")
    for c, name in ((4, "GEMM1->GEMM2 readiness waits"), (16, "producer wait, GEMM1"), (17, "producer wait, GEMM2"),
                    (18, "MMA wait for data, GEMM1"), (19, "MMA wait for data, GEMM2")):
        v = t[:, c] / 1e3
        lines.append(f"  {name:32s} {v.min():8.1f} {np.median(v):8.1f} {v.max():8.1f}  (total us)")
    return lines


def main(argv=None) -> int:
    p = argparse.ArgumentParser()
    p.add_argument("workload")
    p.add_argument("--path", default="auto", choices=["auto", "fused", "multi"])
    p.add_argument("--save", default="", help="also write the raw stamps to this .npz file")
    args = p.parse_args(argv)
    if os.environ.get("BMOE_LIB_VARIANT") != "trace":
        print("run with BMOE_LIB_VARIANT=trace (the tracing build)", file=sys.stderr)
        return 2
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch

    import synth
    from block_scaled_moe_gb300 import BlockScaledMoE, _build, load
    _build.build(variant="trace")
    lib = load()
    w = synth.get(args.workload)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    x = synth.make_x(w).to(dev)
    ids, wts = synth.make_routing(w)
    L = BlockScaledMoE(w.H, w.I, w.E, w.K, w.capacity, dispatch=w.dispatch, swiglu_limit=w.swiglu_limit,
                       path=args.path)
    L.bind_weights(*synth.make_weights(w, dev))
    idsd, wtsd = torch.from_numpy(ids).to(dev), torch.from_numpy(wts).to(dev)
    nvr = torch.tensor([w.nvr], dtype=torch.int32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(4):
        flush.fill_(1.0)
        L.forward(x, idsd, wtsd, nvr)
    torch.cuda.synchronize()
    status = L.read_status()
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    print(f"{w.name}: T={w.T} H={w.H} I={w.I} E={w.E} top-{w.K} nvr={w.nvr}, path {L.last_path}, status {status:#x}")
    if L.last_path == "fused":
        ft = fused_trace(lib, n_sms)
        fs = fused_stage_trace(lib)
        n1 = int(ft[0, 11])
        lines = summarize_fused(ft) + summarize_fused_stages(fs, n1 * (w.H // 128))
        kt2 = w.I // 128 if w.H % 256 == 0 else w.I // (256 if w.I % 256 == 0 else 128)
        for name, c in transition_costs(fs, 0, n1, n1 + int(ft[0, 12]), w.H // 128, kt2).items():
            lines.append(f"  CTA 0 {name} unit transitions (cycles, median over {c['units']} units): producer "
                         f"enter {c['enter']:.0f}, decode {c['decode']:.0f}, prefetch {c['prefetch']:.0f}, to the "
                         f"first wait {c['to_wait']:.0f}; MMA decode {c['mma_decode']:.0f}, to the first wait "
                         f"{c['mma_to_wait']:.0f}; first-stage period {c['first_period']:.0f} against "
                         f"{c['period']:.0f}")
        raw = {"fused_phases": ft, "fused_stages": fs}
    else:
        t = gemm_trace(lib, n_sms)
        lines = summarize_gemm("GEMM1", t["gemm1"]) + summarize_gemm("GEMM2", t["gemm2"])
        raw = {f"{g}_{k}": v for g, d in t.items() for k, v in d.items()}
    if args.save:
        np.savez(args.save, **raw)
    print("\n".join(lines))
    L.close()
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
