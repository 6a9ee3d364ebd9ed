"""GPU tests of a caller-owned workspace (moe_set_workspace; the layer's own allocation otherwise).

* a 256-byte aligned torch buffer of moe_workspace_bytes bytes, handed over before the first
  forward, gives the same bits as the handle's own workspace, on both paths;
* a misaligned pointer and a buffer one region too small are refused and change nothing: the handle
  keeps its own workspace and still gives the same bits; after the first forward the call is refused.
"""

import numpy as np
import pytest
import torch

import synth
from parity_util import Case, torch_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    torch.cuda.set_device(0)


def _aligned(nbytes):
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    return buf, buf[off:off + nbytes]


@pytest.mark.parametrize("path", ["fused", "multi"])
def test_caller_workspace_gives_the_same_bits(path):
    c = Case(synth.get("tiny"))
    own = c.layer(route_tile=32, path=path)
    ref = torch_bf16_bits(c.run(own))
    nbytes = own.workspace_bytes
    assert nbytes > 0
    keep, ws = _aligned(nbytes)
    L = c.layer(route_tile=32, path=path, workspace=ws)
    got = torch_bf16_bits(c.run(L))
    torch.cuda.synchronize()
    assert L.last_path == path
    assert np.array_equal(got, ref)
    assert L.read_status() == 0
    L.close()
    del keep


def test_refused_workspaces_change_nothing():
    import block_scaled_moe_gb300 as bm
    c = Case(synth.get("tiny"))
    L = c.layer(route_tile=32)
    nbytes = L.workspace_bytes
    keep, ws = _aligned(nbytes + 512)
    with pytest.raises(bm.MoeError):
        bm.moe_set_workspace(L.h, ws.data_ptr() + 16, nbytes)      # not 256-byte aligned
    with pytest.raises(bm.MoeError):
        bm.moe_set_workspace(L.h, ws.data_ptr(), nbytes - 256)     # too small
    ref_layer = c.layer(route_tile=32)
    ref = torch_bf16_bits(c.run(ref_layer))
    assert np.array_equal(torch_bf16_bits(c.run(L)), ref)          # its own workspace, unchanged
    with pytest.raises(bm.MoeError):
        bm.moe_set_workspace(L.h, ws.data_ptr(), nbytes)           # after the first forward
    assert np.array_equal(torch_bf16_bits(c.run(L)), ref)
    torch.cuda.synchronize()
    del keep
