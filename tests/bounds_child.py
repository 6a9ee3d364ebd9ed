"""Child process of test_gpu_bounds.py: runs the layer through the bounds-checking build.

The parent starts it with BMOE_LIB_VARIANT=bounds, so the binding loads libblockmoe_bounds.so.  For
every case of CASES it records the output bits, the status word and the first-miss record; then it
plants misses (a packed-row limit of 8 through MOE_OPT_DEBUG_BOUNDS_ROWS on the multi-kernel path),
records what the kernels reported, restores the limit and records one more forward.  Results go to
the .npz file named on the command line.
"""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

import synth  # noqa: E402

# (name, synth.micro arguments, layer options): both paths, both dispatch schemes, decode and
# prefill route tiles, ragged valid-row counts, MXFP8 GEMM2 rows, the debug capture
CASES = [
    ("tiny_fused", dict(T=64, H=256, I=128, E=8, K=2, nvr=60, invalid_frac=0.1, seed=3),
     dict(route_tile=32, path="fused")),
    ("fixed_fused_clamp", dict(T=100, H=256, I=256, E=8, K=3, nvr=77, dispatch="fixed", swiglu_limit=10.0, seed=4),
     dict(route_tile=32, path="fused")),
    ("compact_multi_nt144", dict(T=300, H=256, I=256, E=6, K=4, nvr=290, invalid_frac=0.05, seed=5),
     dict(route_tile=144, path="multi")),
    ("fixed_multi_nt128_debug", dict(T=200, H=512, I=256, E=5, K=2, nvr=200, dispatch="fixed", seed=6),
     dict(route_tile=128, path="multi", debug=True)),
    ("mxfp8_rows_multi", dict(T=96, H=512, I=256, E=12, K=4, nvr=90, seed=7),
     dict(route_tile=32, path="multi", y_format="mxfp8")),
    ("wide_fused", dict(T=256, H=1024, I=512, E=16, K=4, nvr=256, invalid_frac=0.02, swiglu_limit=10.0, seed=8),
     dict(route_tile=32, path="fused")),
]


def case_inputs(args):
    from parity_util import Case
    a = dict(args)
    w = synth.micro(a.pop("T"), a.pop("H"), a.pop("I"), a.pop("E"), a.pop("K"), **a)
    return Case(w)


def run_case(c, opts):
    import torch
    from parity_util import torch_bf16_bits
    L = c.layer(**opts)
    out = L.forward(c.xd, c.idsd, c.wtsd, c.nvrd)
    torch.cuda.synchronize()
    return L, torch_bf16_bits(out), L.debug_array("bounds"), L.read_status()


def main(path):
    import torch
    import block_scaled_moe_gb300 as bm
    torch.cuda.set_device(0)
    res = {}
    for name, args, opts in CASES:
        c = case_inputs(args)
        L, bits, rec, st = run_case(c, opts)
        res[name + "_build"] = np.array(int(bm.moe_get_option(L.h, bm.MOE_OPT_BOUNDS_BUILD)))
        res[name + "_out"], res[name + "_rec"], res[name + "_status"] = bits, rec, np.array(st)
        L.close()
    # planted misses: legitimate rows beyond 8 count as out of range, are skipped and recorded
    name, args, _ = CASES[0]
    c = case_inputs(args)
    L, _, _, _ = run_case(c, dict(route_tile=32, path="multi"))
    rows = L.debug_array("y").size // args["H"]  # the workspace's packed rows
    bm.moe_set_option(L.h, bm.MOE_OPT_DEBUG_BOUNDS_ROWS, 8)
    L.forward(c.xd, c.idsd, c.wtsd, c.nvrd)
    torch.cuda.synchronize()
    res["shrink_rec"] = L.debug_array("bounds")
    res["shrink_status"] = np.array(L.read_status())
    res["shrink_rec_after_read"] = L.debug_array("bounds")
    bm.moe_set_option(L.h, bm.MOE_OPT_DEBUG_BOUNDS_ROWS, rows)
    out = L.forward(c.xd, c.idsd, c.wtsd, c.nvrd)
    torch.cuda.synchronize()
    from parity_util import torch_bf16_bits
    res["restored_out"] = torch_bf16_bits(out)
    res["restored_status"] = np.array(L.read_status())
    L.close()
    np.savez(path, **res)


if __name__ == "__main__":
    main(sys.argv[1])
