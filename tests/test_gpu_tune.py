"""GPU tests of the T-bucketed path table.

* moe_autotune times the paths a handle allows for each bucket T and records one per bucket; the
  table round-trips through get/set, and refused tables change nothing;
* a forward under MOE_PATH_AUTO takes the path of the nearest bucket (ties: the larger bucket), the
  explicit MOE_PATH_* options override the table, and every path still gives the oracle's result;
* a handle that cannot run the fused kernel (128-row route tiles) records the multi-kernel path only.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import Case, assert_close, torch_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    torch.cuda.set_device(0)


def _case():
    w = synth.micro(64, 256, 256, 8, 2, nvr=64, invalid_frac=0.05, dispatch="compact", seed=31)
    return Case(w)


def _fwd(c, L, T):
    out = L.forward(c.xd[:T], c.idsd[:T], c.wtsd[:T], None)
    torch.cuda.synchronize()
    return torch_bf16_bits(out)


def _ref(c, T):
    return oracle.moe_forward(c.x[:T], c.ids[:T], c.wts[:T], c.Wh)


def test_autotune_records_a_path_per_bucket():
    c = _case()
    L = c.layer(route_tile=32)
    table = L.autotune([1, 16, 64], reps=2)
    assert sorted(table) == [1, 16, 64]
    assert set(table.values()) <= {"fused", "multi"}
    for T, bucket in [(1, 1), (10, 16), (40, 64), (64, 64)]:
        got = _fwd(c, L, T)
        assert L.last_path == table[bucket], (T, table)
        assert_close(got, _ref(c, T), f"T={T}")
    assert L.read_status() == 0


def test_nearest_bucket_and_overrides():
    import block_scaled_moe_gb300 as bm
    c = _case()
    L = c.layer(route_tile=32)
    L.set_path_table({8: "multi", 32: "fused"})
    assert L.path_table == {8: "multi", 32: "fused"}
    seen = {}
    for T, want in [(5, "multi"), (8, "multi"), (19, "multi"), (20, "fused"), (40, "fused")]:  # 20: tie -> 32
        seen[T] = _fwd(c, L, T)
        assert L.last_path == want, (T, L.last_path)
    bm.moe_set_option(L.h, bm.MOE_OPT_PATH, bm.MOE_PATH_MULTI)
    m = _fwd(c, L, 40)
    assert L.last_path == "multi"
    assert np.array_equal(m, seen[40])  # both paths give the same bits
    bm.moe_set_option(L.h, bm.MOE_OPT_PATH, bm.MOE_PATH_FUSED)
    _fwd(c, L, 5)
    assert L.last_path == "fused"
    bm.moe_set_option(L.h, bm.MOE_OPT_PATH, bm.MOE_PATH_AUTO)
    L.set_path_table({})
    assert L.path_table == {}
    _fwd(c, L, 40)
    assert L.last_path == "fused"  # default rule: fused for T <= 512 where allowed
    assert_close(seen[19], _ref(c, 19), "T=19")


def test_refused_tables_change_nothing():
    import block_scaled_moe_gb300 as bm
    c = _case()
    L = c.layer(route_tile=32)
    L.set_path_table({4: "fused", 64: "multi"})
    for bad_t, bad_p in [([8, 4], [bm.MOE_PATH_FUSED, bm.MOE_PATH_MULTI]),     # not ascending
                         ([0], [bm.MOE_PATH_MULTI]),                             # T < 1
                         ([65], [bm.MOE_PATH_MULTI]),                            # T > capacity
                         ([8], [bm.MOE_PATH_AUTO])]:                             # not a concrete path
        with pytest.raises(bm.MoeError):
            bm.moe_set_path_table(L.h, bad_t, bad_p)
        assert L.path_table == {4: "fused", 64: "multi"}
    Lw = c.layer(route_tile=128)  # 128-row route tiles: no fused kernel
    with pytest.raises(bm.MoeError):
        Lw.set_path_table({16: "fused"})
    assert Lw.path_table == {}
    with pytest.raises(bm.MoeError):
        bm.moe_autotune(Lw.h, [16, 8])


def test_autotune_multi_only_handle():
    c = _case()
    Lw = c.layer(route_tile=128)
    assert Lw.autotune([64], reps=1) == {64: "multi"}
    got = _fwd(c, Lw, 64)
    assert Lw.last_path == "multi"
    assert_close(got, _ref(c, 64), "T=64 multi")
