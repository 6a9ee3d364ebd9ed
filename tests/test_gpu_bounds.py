"""GPU tests of the bounds-checking build (the pages' plan for memory errors without a sanitizer:
a build that checks indices and records the first one out of range, nothing trapping).

libblockmoe_bounds.so is the library compiled with -DMOE_DEBUG_BOUNDS: every index the kernels
compute into a workspace region or an output row is checked before use, a miss sets MOE_ST_BOUNDS,
the first one is recorded (MOE_DBG_BOUNDS: site and index) and the access is skipped.  A child
process loads it (BMOE_LIB_VARIANT=bounds) and runs the cases of bounds_child.CASES; here:

* every case reports no miss and no other status bit, and its output is bitwise the normal build's;
* planted misses (a packed-row limit of 8 on the multi-kernel path) are reported with a row site and
  an index of at least 8, nothing times out, reading the status clears the record, and with the
  limit restored the next forward is bitwise the normal build's again;
* the normal build says it is not the checking build and refuses the row-limit option.
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import bounds_child

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def child_results(tmp_path_factory):
    from block_scaled_moe_gb300 import _build
    _build.build(variant="bounds")
    out = tmp_path_factory.mktemp("bounds") / "results.npz"
    env = dict(os.environ, BMOE_LIB_VARIANT="bounds")
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_child.py"), str(out)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return dict(np.load(out))


def _normal_bits(args, opts):
    import block_scaled_moe_gb300 as bm
    c = bounds_child.case_inputs(args)
    L, bits, rec, st = bounds_child.run_case(c, opts)
    assert st == 0 and not rec.any()
    assert int(bm.moe_get_option(L.h, bm.MOE_OPT_BOUNDS_BUILD)) == 0
    L.close()
    return bits


@pytest.mark.parametrize("case", bounds_child.CASES, ids=[c[0] for c in bounds_child.CASES])
def test_checked_build_is_clean_and_bitwise_equal(child_results, case):
    name, args, opts = case
    res = child_results
    assert int(res[name + "_build"]) == 1  # the child ran the checking build
    assert int(res[name + "_status"]) == 0, hex(int(res[name + "_status"]))
    assert not res[name + "_rec"].any(), res[name + "_rec"]
    assert np.array_equal(res[name + "_out"], _normal_bits(args, opts)), name


def test_planted_misses_are_reported_and_recovered(child_results):
    import block_scaled_moe_gb300 as bm
    res = child_results
    st = int(res["shrink_status"])
    assert st & bm.MOE_ST_BOUNDS, hex(st)
    assert not st & bm.MOE_ST_TIMEOUT, hex(st)
    site, index = (int(v) for v in res["shrink_rec"])
    assert site in (5, 6, 7, 8), site  # a scattered row, scale atom, combined row or GEMM unit
    assert index >= 8 or site == 6, (site, index)
    assert not res["shrink_rec_after_read"].any()
    assert int(res["restored_status"]) == 0
    name, args, _ = bounds_child.CASES[0]
    assert np.array_equal(res["restored_out"], _normal_bits(args, dict(route_tile=32, path="multi")))


def test_normal_build_refuses_the_row_limit():
    import block_scaled_moe_gb300 as bm
    name, args, opts = bounds_child.CASES[0]
    c = bounds_child.case_inputs(args)
    L = c.layer(**opts)
    assert int(bm.moe_get_option(L.h, bm.MOE_OPT_BOUNDS_BUILD)) == 0
    with pytest.raises(bm.MoeError):
        bm.moe_set_option(L.h, bm.MOE_OPT_DEBUG_BOUNDS_ROWS, 8)
    L.close()
