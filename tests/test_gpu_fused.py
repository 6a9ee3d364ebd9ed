"""GPU parity of the single-launch fused path.

The fused kernel (dispatch, quantisation, GEMM1, GEMM2 and combine in one
cooperative launch) must give the same bits as the multi-kernel path on the
same inputs, and stay within the output tolerance of the oracle: decode-width
configurations of both dispatch schemes, ragged and empty inputs, invalid
slots, ids >= E, CUDA-graph replay, repeated forwards with changing T, and the
full-size decode and small-input workloads.
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


def _pair(c: Case, **kw):
    """The same layer twice: fused and multi-kernel."""
    return c.layer(route_tile=32, path="fused", **kw), c.layer(route_tile=32, path="multi", **kw)


def _fwd(c, L, **kw):
    out = c.run(L, **kw)
    torch.cuda.synchronize()
    return torch_bf16_bits(out)


FUSED_CFGS = [
    # T, H, I, E, K, nvr, routing, invalid, limit, dispatch
    (1, 128, 128, 1, 1, 1, "uniform", 0.0, 0.0, "compact"),
    (5, 256, 128, 3, 2, 5, "uniform", 0.0, 0.0, "fixed"),
    (37, 128, 256, 4, 3, 30, "uniform", 0.3, 10.0, "compact"),
    (37, 128, 256, 4, 3, 30, "uniform", 0.3, 10.0, "fixed"),
    (200, 256, 128, 6, 4, 190, "hot_zipf", 0.0, 0.0, "compact"),   # repeated experts, multi-tile experts
    (200, 256, 384, 6, 4, 190, "hot_zipf", 0.0, 0.0, "fixed"),     # I % 256 != 0: one K chunk per GEMM2 stage
    (512, 256, 256, 16, 6, 500, "uniform", 0.05, 0.0, "compact"),  # the largest capacity the fused path takes
    (64, 128, 256, 512, 16, 64, "uniform", 0.1, 10.0, "compact"),  # E = 512 and top-16: the table limits
    (96, 384, 512, 40, 8, 90, "hot_zipf", 0.1, 0.0, "fixed"),
    # GEMM1 units not a multiple of the grid, several rounds of GEMM2 units per CTA, H = 1024
    (256, 1024, 512, 128, 8, 250, "uniform", 0.02, 10.0, "compact"),
]


@pytest.mark.parametrize("cfg", FUSED_CFGS, ids=[f"T{m[0]}H{m[1]}I{m[2]}E{m[3]}K{m[4]}{m[9]}" for m in FUSED_CFGS])
def test_fused_equals_multi_and_matches_oracle(cfg):
    T, H, I, E, K, nvr, routing, inv, lim, disp = cfg
    w = synth.micro(T, H, I, E, K, nvr=nvr, routing=routing, invalid_frac=inv, swiglu_limit=lim, dispatch=disp,
                    seed=T * 11 + E, hot_frac=0.5)
    c = Case(w)
    Lf, Lm = _pair(c)
    f = _fwd(c, Lf)
    m = _fwd(c, Lm)
    assert Lf.last_path == "fused" and Lm.last_path == "multi"
    assert np.array_equal(f, m), str(cfg)
    assert_close(f, c.oracle(), str(cfg))
    assert Lf.read_status() == 0 and Lm.read_status() == 0


@pytest.mark.parametrize("dispatch", ["compact", "fixed"])
def test_fused_tiny_both_schemes_and_launch_count(dispatch):
    c = Case(synth.get("tiny"))
    Lf, Lm = _pair(c, dispatch=dispatch)
    n0 = Lf.launches
    f = _fwd(c, Lf)
    assert Lf.launches - n0 == 1
    assert np.array_equal(f, _fwd(c, Lm))
    assert_close(f, c.oracle(), dispatch)


def test_auto_path_selection_and_refusal():
    import block_scaled_moe_gb300 as bm
    c = Case(synth.get("tiny"))
    La = c.layer(route_tile=32)
    _fwd(c, La)
    assert La.last_path == "fused"
    Lw = c.layer(route_tile=128)
    _fwd(c, Lw)
    assert Lw.last_path == "multi"
    with pytest.raises(bm.MoeError):
        bm.moe_set_option(Lw.h, bm.MOE_OPT_PATH, bm.MOE_PATH_FUSED)
    with pytest.raises(bm.MoeError):
        bm.moe_set_option(La.h, bm.MOE_OPT_PATH, 3)


def test_fused_num_valid_rows_variants():
    w = synth.micro(40, 256, 256, 5, 3, nvr=40, invalid_frac=0.1, dispatch="compact", seed=3)
    c = Case(w)
    Lf, Lm = _pair(c)
    for nv in [0, 1, 17, 40, 1000]:
        c.nvrd.fill_(nv)
        f = _fwd(c, Lf)
        assert np.array_equal(f, _fwd(c, Lm)), nv
        assert np.all(f[min(nv, w.T):] == 0)
        if nv > 0:
            ref = oracle.moe_forward(c.x, c.ids, c.wts, c.Wh, num_valid_rows=nv)
            assert_close(f, ref, f"nvr={nv}")
    f = torch_bf16_bits(Lf.forward(c.xd, c.idsd, c.wtsd, None))
    torch.cuda.synchronize()
    assert np.array_equal(f, torch_bf16_bits(Lm.forward(c.xd, c.idsd, c.wtsd, None)))


def test_fused_all_invalid_and_bad_ids():
    w = synth.micro(33, 128, 128, 4, 2, nvr=33, invalid_frac=0.0, dispatch="fixed", seed=5)
    c = Case(w)
    Lf, Lm = _pair(c)
    c.idsd.fill_(-1)
    assert np.all(_fwd(c, Lf) == 0)
    assert Lf.read_status() == 0
    ids = c.ids.copy()
    ids[3, 1] = w.E + 2
    ids[7, 0] = 1 << 20
    c.idsd.copy_(torch.from_numpy(ids))
    f = _fwd(c, Lf)
    assert np.array_equal(f, _fwd(c, Lm))
    import block_scaled_moe_gb300 as bm
    assert Lf.read_status() & bm.MOE_ST_BAD_ID
    ids[ids >= w.E] = -1
    ref = oracle.moe_forward(c.x, ids, c.wts, c.Wh, num_valid_rows=w.nvr)
    assert_close(f, ref, "ids >= E skipped")
    assert Lf.read_status() == 0


def test_fused_repeated_forwards_with_changing_T():
    """The grid-barrier words persist between launches: many forwards of varying
    size on one handle must each be right."""
    w = synth.micro(128, 256, 256, 8, 4, nvr=128, invalid_frac=0.05, dispatch="compact", seed=9)
    c = Case(w)
    Lf, Lm = _pair(c)
    for T in [128, 1, 77, 128, 32, 5, 128]:
        xs, ids, wts = c.xd[:T], c.idsd[:T], c.wtsd[:T]
        f = torch_bf16_bits(Lf.forward(xs, ids, wts, None))
        m = torch_bf16_bits(Lm.forward(xs, ids, wts, None))
        torch.cuda.synchronize()
        assert np.array_equal(f, m), T
    assert Lf.read_status() == 0


def test_fused_graph_replay_equals_eager():
    c = Case(synth.get("tiny"))
    L = c.layer(route_tile=32, path="fused")
    eager = _fwd(c, L)
    s = torch.cuda.Stream()
    out = torch.empty_like(c.xd)
    with torch.cuda.stream(s):
        c.run(L, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.run(L, out=out, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(torch_bf16_bits(out), eager)
    c.nvrd.fill_(10)
    g.replay()
    torch.cuda.synchronize()
    got = torch_bf16_bits(out)
    assert np.array_equal(got[:10], eager[:10]) and np.all(got[10:] == 0)
    assert L.read_status() == 0


def test_fused_debug_capture_dispatch_bit_exact():
    w = synth.micro(200, 256, 128, 6, 4, nvr=190, routing="hot_zipf", invalid_frac=0.05, dispatch="compact",
                    seed=21, hot_frac=0.5)
    c = Case(w)
    L = c.layer(route_tile=32, path="fused", debug=True)
    _fwd(c, L)
    d = oracle.dispatch_compact(c.ids, w.E, w.nvr)
    assert np.array_equal(L.debug_array("counts"), d["counts"])
    assert np.array_equal(L.debug_array("offsets"), d["offsets"])
    R = int(d["offsets"][-1])
    assert np.array_equal(L.debug_array("perm")[:R], d["perm"])
    assert np.array_equal(L.debug_array("route_row"), d["route_row"].reshape(-1))
    codes, scales = oracle.quant_mxfp8_rows(c.x)
    # rows at or beyond num_valid_rows are not quantised
    assert np.array_equal(L.debug_array("xq").reshape(w.T, -1)[:w.nvr], codes[:w.nvr])
    assert np.array_equal(L.debug_array("xs").reshape(w.T, -1)[:w.nvr], scales[:w.nvr])


@pytest.mark.parametrize("name,rows", [("decode_flash", 16), ("smallm_pro", 8)])
def test_full_size_fused_equals_multi(name, rows):
    w = synth.get(name)
    c = Case(w, weights_on_device=True)
    Lf = c.layer(path="fused")
    Lm = c.layer(path="multi")
    f = _fwd(c, Lf)
    m = _fwd(c, Lm)
    assert Lf.last_path == "fused"
    assert np.array_equal(f, m), name
    rng = np.random.default_rng(1)
    sel = np.sort(rng.choice(np.arange(min(w.nvr, w.T)), size=rows, replace=False))
    assert_close(f[sel], c.oracle(rows=sel), name)
    assert np.all(f[w.nvr:] == 0)
    assert Lf.read_status() == 0
