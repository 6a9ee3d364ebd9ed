"""GPU tests of the W13 row-order flag and the layer binding slots.

* gate-up-interleaved W13 (row 2j gate j, row 2j+1 up j) bound with MOE_OPT_W13_LAYOUT gives the
  same bits as the concatenated layout on both paths and both route tiles, and matches the
  oracle run on the interleaved bytes;
* layer slots: two layers bound in two slots of one handle, selected in turn (also inside one
  CUDA graph), each give the bits of a handle bound to that layer alone; a refused bind_layer
  (bad slot, strided weights) changes neither the slot nor the current slot.
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


def _interleave(t):
    """[E, 2I, n] concatenated -> interleaved rows (a fresh contiguous tensor)."""
    E, I2, n = t.shape
    I = I2 // 2
    return torch.stack([t[:, :I, :], t[:, I:, :]], dim=2).reshape(E, I2, n).contiguous()


def _fwd(c, L):
    out = c.run(L)
    torch.cuda.synchronize()
    return torch_bf16_bits(out)


LAYOUT_CFGS = [
    # T, H, I, E, K, dispatch, route_tile, path
    (40, 256, 256, 6, 3, "compact", 32, "fused"),
    (40, 256, 256, 6, 3, "compact", 32, "multi"),
    (64, 512, 384, 5, 2, "fixed", 32, "fused"),     # H % 512 == 0: 16-byte GEMM1 scale loads
    (200, 384, 256, 4, 4, "compact", 128, "multi"),
    # H, I multiples of 512: prefill tiles read the weight scales as 16-byte vectors (4 K stages);
    # several vector groups per unit, several units per CTA
    (1200, 1024, 1024, 16, 2, "compact", 144, "multi"),
    (600, 2048, 512, 8, 2, "compact", 128, "multi"),
]


@pytest.mark.parametrize("cfg", LAYOUT_CFGS, ids=[f"T{c[0]}H{c[1]}I{c[2]}{c[5]}NT{c[6]}{c[7]}" for c in LAYOUT_CFGS])
def test_interleaved_w13_equals_concat(cfg):
    T, H, I, E, K, disp, nt, path = cfg
    w = synth.micro(T, H, I, E, K, nvr=T - 3, invalid_frac=0.05, dispatch=disp, seed=T + I, swiglu_limit=10.0)
    c = Case(w)
    Lc = c.layer(route_tile=nt, path=path)
    Li = c.layer(route_tile=nt, path=path, w13_layout="interleaved")
    wi = [_interleave(c.Wd[0]), _interleave(c.Wd[1]), c.Wd[2], c.Wd[3]]
    Li.bind_weights(*wi)
    a, b = _fwd(c, Lc), _fwd(c, Li)
    assert Li.last_path == path
    assert np.array_equal(a, b)
    ref = oracle.moe_forward(c.x, c.ids, c.wts, [t.cpu() for t in wi], num_valid_rows=w.nvr,
                             swiglu_limit=w.swiglu_limit, w13_layout="interleaved")
    assert_close(b, ref, str(cfg))
    assert Li.read_status() == 0


def test_interleaved_w13_full_decode():
    w = synth.get("decode_flash")
    c = Case(w, weights_on_device=True)
    Lc = c.layer()
    Li = c.layer(w13_layout="interleaved")
    Li.bind_weights(_interleave(c.Wd[0]), _interleave(c.Wd[1]), c.Wd[2], c.Wd[3])
    assert np.array_equal(_fwd(c, Lc), _fwd(c, Li))


def test_layer_slots_select_and_graph():
    import block_scaled_moe_gb300 as bm
    w = synth.micro(48, 256, 256, 6, 2, nvr=45, invalid_frac=0.05, dispatch="compact", seed=11)
    c = Case(w)
    W1 = c.Wd
    W2 = [t.cpu() for t in synth.make_weights(synth.micro(48, 256, 256, 6, 2, seed=12), "cpu")]
    W2 = [t.cuda() for t in W2]
    L = c.layer(route_tile=32, layer_slots=3)
    L.bind_layer(0, *W1)
    L.bind_layer(2, *W2)
    assert L.layer == 2
    ref1 = c.layer(route_tile=32)
    ref2 = c.layer(route_tile=32)
    ref2.bind_weights(*W2)
    r1, r2 = _fwd(c, ref1), _fwd(c, ref2)
    assert not np.array_equal(r1, r2)
    assert np.array_equal(_fwd(c, L), r2)
    L.select_layer(0)
    assert np.array_equal(_fwd(c, L), r1)
    with pytest.raises(bm.MoeError):
        L.select_layer(1)                     # never bound
    with pytest.raises(bm.MoeError):
        L.bind_layer(3, *W2)                  # no such slot
    with pytest.raises(ValueError):
        L.bind_layer(2, W1[0][:, ::2], W1[1], W1[2], W1[3])  # strided view refused
    assert L.layer == 0
    L.select_layer(2)
    assert np.array_equal(_fwd(c, L), r2)    # slot 2 kept its weights after the refusals
    # one graph with both layers, each captured with its slot
    s = torch.cuda.Stream()
    o1, o2 = torch.empty_like(c.xd), torch.empty_like(c.xd)
    with torch.cuda.stream(s):
        L.select_layer(0)
        L.forward(c.xd, c.idsd, c.wtsd, c.nvrd, out=o1, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.select_layer(0)
        L.forward(c.xd, c.idsd, c.wtsd, c.nvrd, out=o1, stream=s)
        L.select_layer(2)
        L.forward(c.xd, c.idsd, c.wtsd, c.nvrd, out=o2, stream=s)
    o1.zero_()
    o2.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(torch_bf16_bits(o1), r1)
    assert np.array_equal(torch_bf16_bits(o2), r2)
    assert L.read_status() == 0
