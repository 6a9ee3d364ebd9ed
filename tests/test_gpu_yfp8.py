"""GPU tests of GEMM2 rows handed to the combine as MXFP8 (MOE_OPT_Y_FORMAT).

* the fused and multi-kernel paths give the same bits;
* each route layer by layer, code by code: the GPU's h codes against the oracle's float h, then the
  GPU's MXFP8 y row against the oracle's GEMM2 (double sums) of the GPU's own h codes, both
  re-quantised by the OCP MX rule.  Every E8M0 scale and E4M3 code must be equal, except where the
  float value lies within 1e-4 of its block's largest magnitude of an E4M3 rounding midpoint (or
  the block maximum that close to a power of two, for a scale): there the tensor cores' FP32 sums
  and the oracle's double sums may round to the two neighbours of that midpoint, and the GPU value
  must be one of the two;
* the combine, bit for bit, against a CPU float sum (ascending k, one BF16 rounding) of the GPU's own
  MXFP8 rows;
* the outputs against the oracle's MXFP8-row mode: relative L2 <= 1e-2 and, for every element,
  |d| <= 0.08*|ref| + 1e-2*rms(ref), widened only for elements whose route's y row changed through a
  flip of the kind above, by that change times the route's weight;
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


E4M3 = None


def _e4m3_table():
    global E4M3
    if E4M3 is None:
        from independent_ref import e4m3_decode
        E4M3 = e4m3_decode(np.arange(256, dtype=np.uint8))
    return E4M3


EPS = 1e-4   # window around a rounding midpoint / power of two, relative to the block's largest magnitude


def _gpu_rows(L, w):
    """(y8 codes [rows, H], ys scales [rows, H/32], yrow [T, K]) of the last forward."""
    raw = L.debug_array("y").view(np.uint8)
    rows = raw.size // (2 * w.H)
    y8 = raw[: rows * w.H].reshape(rows, w.H)
    ys = raw[rows * w.H: rows * w.H + rows * (w.H // 32)].reshape(rows, w.H // 32)
    return y8, ys, L.debug_array("yrow").reshape(w.T, w.K)


def _codes_at(y, scales):
    """E4M3 codes (round to nearest even, saturating at 448) of float y over the given block scales."""
    sc = np.ldexp(1.0, 127 - np.repeat(scales.astype(np.int64), 32))
    v = np.clip(y.astype(np.float64) * sc, -448.0, 448.0).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _check_codes(v_ref, codes, scales, what):
    """GPU E4M3 codes of float v_ref over `scales`: equal to round-to-nearest-even, except the two
    neighbours of a rounding midpoint that v_ref lies within EPS of its block's largest magnitude."""
    tab = _e4m3_table()
    blk = np.abs(v_ref.astype(np.float64)).reshape(-1, 32).max(axis=1)
    want = _codes_at(v_ref, scales)
    unit = np.ldexp(1.0, np.repeat(scales.astype(np.int64), 32) - 127)
    win = np.repeat(EPS * blk, 32)
    for i in np.nonzero(codes != want)[0]:
        g, r = tab[codes[i]] * unit[i], tab[want[i]] * unit[i]
        lo, hi = min(g, r), max(g, r)
        assert not np.any((tab * unit[i] > lo) & (tab * unit[i] < hi)), (what, "not neighbours", i, int(codes[i]),
                                                                         int(want[i]))
        assert abs(float(v_ref[i]) - 0.5 * (g + r)) <= win[i], (what, "flip away from a midpoint", i,
                                                               int(codes[i]), int(want[i]), float(v_ref[i]), win[i])
    return int(np.count_nonzero(codes != want))


def _check_scales(v_ref, scales, what):
    """GPU E8M0 scales of float v_ref: the OCP rule's, except blocks whose largest magnitude lies within
    EPS (relative) of a power of two."""
    from independent_ref import q8
    _, rs = q8(v_ref[None, :])
    blk = np.abs(v_ref.astype(np.float64)).reshape(-1, 32).max(axis=1)
    for b in np.nonzero(scales != rs[0])[0]:
        m, _ = np.frexp(blk[b])
        assert abs(m - 0.5) <= EPS or abs(m - 1.0) <= EPS, (what, "scale", b, int(scales[b]), int(rs[0][b]), blk[b])


def _check_route(c, t, e, hq_gpu, y8, ys, w2deq):
    """One route, layer by layer.  h: the GPU's E4M3 codes against the oracle's float h (its scales, which
    the library does not expose, taken as the oracle's); y: the GPU's MXFP8 row against the oracle's
    GEMM2 of the GPU's own h codes.  Returns the GPU's dequantised y row."""
    from independent_ref import q8_dequant, swiglu
    w = c.w
    ri = oracle.route_intermediates(c.x[t], e, c.Wh, w.swiglu_limit)
    h_ref = swiglu(ri["g"][None, :], w.I, w.swiglu_limit)[0]
    _check_codes(h_ref, hq_gpu, ri["hs"], ("h", t, e))
    y_exp = (q8_dequant(hq_gpu[None, :], ri["hs"][None, :]) @ w2deq.T)[0].astype(np.float32)
    _check_scales(y_exp, ys, ("y", t, e))
    _check_codes(y_exp, y8, ys, ("y", t, e))
    tab = _e4m3_table()
    return tab[y8] * np.ldexp(1.0, np.repeat(ys.astype(np.int64), 32) - 127)


def _cpu_combine(y8, ys, yrow, wts, nvr):
    """out = BF16(sum over valid k ascending of fp32(w * fp32(deq(y)))), +0 for rows without a slot."""
    from independent_ref import bf16_bits
    tab = _e4m3_table().astype(np.float32)
    T, K = yrow.shape
    H = y8.shape[1]
    acc = np.zeros((T, H), np.float32)
    anyv = np.zeros(T, bool)
    for k in range(K):
        r = yrow[:, k]
        ok = r >= 0
        if not ok.any():
            continue
        rr = np.where(ok, r, 0)
        sc = np.ldexp(np.float32(1.0), ys[rr].astype(np.int32) - 127).astype(np.float32)
        yv = (tab[y8[rr]] * np.repeat(sc, 32, axis=1)).astype(np.float32)
        contrib = (wts[:, k:k + 1].astype(np.float32) * yv).astype(np.float32)
        acc = np.where(ok[:, None], (acc + contrib).astype(np.float32), acc)
        anyv |= ok
    out = bf16_bits(acc)
    out[~anyv] = 0
    return out


def _check_fp8_rows(L, c, got, rows, what):
    """Layer by layer on `rows`: h and y codes (_check_route), the combine bit for bit, then the outputs
    against the oracle, widened where a code flip (of h or y) changed a route's dequantised y row."""
    from independent_ref import fp4_dequant
    w = c.w
    y8, ys, yrow = _gpu_rows(L, w)
    hq = L.debug_array("hq").reshape(-1, w.I)
    assert np.array_equal(got, _cpu_combine(y8, ys, yrow, c.wts, w.nvr)), (what, "combine")
    ref = oracle.moe_forward(c.x, c.ids, c.wts, c.Wh, num_valid_rows=w.nvr, swiglu_limit=w.swiglu_limit,
                             rows=rows, y_format="mxfp8")
    w2, w2s = c.Wh[2].numpy(), c.Wh[3].numpy()
    w2deq = {}
    tab = _e4m3_table()
    widen = np.zeros((len(rows), w.H))
    for j, t in enumerate(rows):
        for k in range(w.K):
            e = int(c.ids[t, k])
            if t >= w.nvr or e < 0 or e >= w.E:
                continue
            if e not in w2deq:
                w2deq[e] = fp4_dequant(w2[e], w2s[e])
            r = yrow[t, k]
            y_gpu = _check_route(c, t, e, hq[r], y8[r], ys[r], w2deq[e])
            ri = oracle.route_intermediates(c.x[t], e, c.Wh, w.swiglu_limit)
            from independent_ref import q8
            oq, os_ = q8(ri["y"][None, :])
            y_orc = tab[oq[0]] * np.ldexp(1.0, np.repeat(os_[0].astype(np.int64), 32) - 127)
            widen[j] += abs(float(c.wts[t, k])) * np.abs(y_gpu - y_orc)
    g, r = bits_to_f64(got[rows]), bits_to_f64(ref)
    assert np.all(np.isfinite(g)), what
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
    bound = ELEM_REL * np.abs(r) + ELEM_RMS * rms
    # where a flip changed a route's y: its exact weighted size, plus one BF16 rounding of the sum
    bound = np.where(widen > 0, bound + widen + np.abs(r) * 2.0 ** -8, bound)
    bad = np.count_nonzero(np.abs(g - r) > bound)
    assert rel <= 1e-2, (what, rel)
    assert bad == 0, (what, bad)


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
    paths = ["fused", "multi"] if nt == 32 else ["multi"]
    outs = []
    for path in paths:
        L = c.layer(route_tile=nt, path=path, y_format="mxfp8")
        got = _fwd(c, L)
        assert L.last_path == path
        _check_fp8_rows(L, c, got, np.arange(w.T), f"{cfg} {path}")
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
    _check_fp8_rows(L, c, eager, rows, "decode_flash")
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
