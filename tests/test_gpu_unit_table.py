"""GPU parity where a CTA holds more units than its decoded-unit table.

Each CTA of the stand-alone GEMMs decodes its first 384 units into shared memory before its
pipeline starts and decodes any later ones with the role's cursor over the tile plan.  The
workloads of the other tests stay well below 384 units per CTA, so this case makes many route
tiles with a short weight tile stride: 28,672 rows, top-8, 512 experts, H = 256, I = 2048,
32-row route tiles on the multi-kernel path (the GEMM1 unit list is ~7,700 route tiles x 16
weight tiles, ~800 units per CTA).  Rows covering every expert's first and last route tile are
compared with the oracle at the usual tolerance, and the unit count is checked to exceed the
table so that the cursor path really runs.
"""

import numpy as np
import pytest
import torch

import synth
from parity_util import Case, assert_close, cover_rows, torch_bf16_bits

pytestmark = pytest.mark.gpu

TABLE = 384  # decoded units per CTA in the stand-alone GEMMs


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    torch.cuda.set_device(0)


def _route_tiles(ids, E, nvr, NT):
    counts = np.zeros(E, np.int64)
    v = ids[:nvr].reshape(-1)
    v = v[(v >= 0) & (v < E)]
    np.add.at(counts, v, 1)
    return int(np.sum((counts + NT - 1) // NT))


def test_units_past_the_table_match_oracle():
    T, H, I, E, K, NT = 28672, 256, 2048, 512, 8, 32
    w = synth.micro(T, H, I, E, K, nvr=T - 37, invalid_frac=0.02, swiglu_limit=10.0, dispatch="compact", seed=91)
    c = Case(w, weights_on_device=True)
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = _route_tiles(c.ids, E, w.nvr, NT) * (I // 128)
    assert (units + n_sms - 1) // n_sms > TABLE, (units, n_sms)
    L = c.layer(route_tile=NT, path="multi")
    out = c.run(L)
    torch.cuda.synchronize()
    assert L.last_path == "multi"
    got = torch_bf16_bits(out)
    rows = cover_rows(c.ids, E, w.nvr, NT, L.scheme, extra=24, seed=5)
    ref = c.oracle(rows=rows)
    assert_close(got[rows], ref, "units past the decoded-unit table")
    assert np.all(got[w.nvr:] == 0)
    assert L.read_status() == 0
