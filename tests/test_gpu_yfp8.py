"""GPU tests of GEMM2 rows handed to the combine as MXFP8 (MOE_OPT_Y_FORMAT).

* the fused and multi-kernel paths give the same bits;
* against the oracle's MXFP8-row mode (y_format="mxfp8"): relative L2 <= 1e-2, no NaN, and at most
  2e-4 of the elements outside the usual elementwise bound.  The extra allowance: a y element whose
  float value sits within the FP32-vs-double accumulation difference (~1e-6 relative) of an E4M3
  rounding boundary may take the neighbouring code on the two sides (one E4M3 step, up to 2^-3 of
  the element, times its top-k weight), which the elementwise bound does not cover where the
  output cancels;
* paired W2 tiles (128-row route tiles) and single tiles, both dispatch schemes, graph replay.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import ELEM_REL, ELEM_RMS, Case, bits_to_f64, torch_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    torch.cuda.set_device(0)


def _close_fp8(got, ref, what):
    g, r = bits_to_f64(got), bits_to_f64(ref)
    assert np.all(np.isfinite(g)), what
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
    bad = np.count_nonzero(np.abs(g - r) > ELEM_REL * np.abs(r) + ELEM_RMS * rms)
    assert rel <= 1e-2, (what, rel)
    assert bad <= max(2, 2e-4 * r.size), (what, bad, r.size)


def _fwd(c, L):
    out = c.run(L)
    torch.cuda.synchronize()
    return torch_bf16_bits(out)


CFGS = [
    # T, H, I, E, K, dispatch, route_tile
    (64, 256, 256, 8, 4, "compact", 32),
    (48, 512, 384, 6, 2, "fixed", 32),
    (300, 512, 256, 4, 4, "compact", 128),   # H % 256 == 0: paired W2 tiles
    (200, 384, 256, 4, 3, "compact", 128),   # H % 256 != 0: single W2 tiles
]


@pytest.mark.parametrize("cfg", CFGS, ids=[f"T{c[0]}H{c[1]}I{c[2]}{c[5]}NT{c[6]}" for c in CFGS])
def test_mxfp8_rows_match_oracle(cfg):
    T, H, I, E, K, disp, nt = cfg
    w = synth.micro(T, H, I, E, K, nvr=T - 2, invalid_frac=0.05, dispatch=disp, seed=T * 3 + H, swiglu_limit=10.0)
    c = Case(w)
    ref = oracle.moe_forward(c.x, c.ids, c.wts, c.Wh, num_valid_rows=w.nvr, swiglu_limit=10.0, y_format="mxfp8")
    paths = ["fused", "multi"] if nt == 32 else ["multi"]
    outs = []
    for path in paths:
        L = c.layer(route_tile=nt, path=path, y_format="mxfp8")
        got = _fwd(c, L)
        assert L.last_path == path
        _close_fp8(got, ref, f"{cfg} {path}")
        assert np.all(got[w.nvr:] == 0)
        assert L.read_status() == 0
        outs.append(got)
    if len(outs) == 2:
        assert np.array_equal(outs[0], outs[1])
    bf = _fwd(c, c.layer(route_tile=nt))
    assert not np.array_equal(bf, outs[0])  # the format does change the result


def test_mxfp8_rows_full_decode_and_graph():
    w = synth.get("decode_flash")
    c = Case(w, weights_on_device=True)
    L = c.layer(y_format="mxfp8")
    eager = _fwd(c, L)
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(np.arange(w.nvr), size=12, replace=False))
    ref = oracle.moe_forward(c.x, c.ids, c.wts, c.Wh, num_valid_rows=w.nvr, swiglu_limit=w.swiglu_limit,
                             rows=rows, y_format="mxfp8")
    _close_fp8(eager[rows], ref, "decode_flash")
    s = torch.cuda.Stream()
    out = torch.empty_like(c.xd)
    with torch.cuda.stream(s):
        c.run(L, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.run(L, out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(torch_bf16_bits(out), eager)
    assert L.read_status() == 0
