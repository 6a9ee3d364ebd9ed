"""GPU parity of the router top-k softmax and of the routed forward.

* ids bit-exact against the oracle (the picks compare the logits themselves), weights within
  2e-6 relative (float32 exp against the oracle's double), on float32 and bf16 logits, with ties,
  rows that run out of finite logits, expert counts that are not multiples of 32, E = 1 and 4096,
  top-16, rows past num_valid_rows and the non-renormalised weights;
* moe_forward_routed gives the bits of moe_topk_softmax followed by moe_forward, matches the
  oracle, and in a CUDA graph follows num_valid_rows at replay.
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


def _logits(T, E, seed, ties=True, neg_inf_rows=0):
    g = torch.Generator().manual_seed(seed)
    lg = torch.randn((T, E), generator=g, dtype=torch.float32) * 2.0
    if ties:
        lg[:, ::7] = torch.round(lg[:, ::7])
    for r in range(min(neg_inf_rows, T)):
        keep = r % 3  # rows with 0, 1 or 2 finite logits
        lg[r, :] = float("-inf")
        lg[r, :keep] = torch.arange(keep, dtype=torch.float32)
    return lg


def _check(got_ids, got_w, ref, what):
    ids = got_ids.cpu().numpy()
    w = got_w.cpu().numpy()
    assert np.array_equal(ids, ref["ids"]), what
    fin = np.isfinite(ref["weights"])
    assert np.array_equal(fin, np.isfinite(w)), what
    np.testing.assert_allclose(w[fin], ref["weights"][fin], rtol=2e-6, atol=1e-30, err_msg=what)


@pytest.mark.parametrize("T,E,K", [(300, 384, 6), (64, 37, 5), (40, 4096, 16), (16, 1, 1), (129, 512, 8)])
@pytest.mark.parametrize("renorm", [True, False])
def test_topk_softmax_matches_oracle(T, E, K, renorm):
    import block_scaled_moe_gb300 as bm
    lg = _logits(T, E, seed=T + E, neg_inf_rows=4 if E > 2 else 0)
    ids, w = bm.topk_softmax(lg.cuda(), K, renormalize=renorm)
    torch.cuda.synchronize()
    _check(ids, w, oracle.topk_softmax(lg.numpy(), K, renormalize=renorm), f"T{T} E{E} K{K}")


def test_topk_softmax_bf16_and_row_count():
    import block_scaled_moe_gb300 as bm
    lg = _logits(200, 384, seed=3).to(torch.bfloat16)
    wide = lg.float().numpy()   # bf16 -> float32 is exact
    for nv in [0, 1, 77, 200, 1000, -3]:
        nvr = torch.tensor([nv], dtype=torch.int32, device="cuda")
        ids, w = bm.topk_softmax(lg.cuda(), 6, num_valid_rows=nvr)
        torch.cuda.synchronize()
        _check(ids, w, oracle.topk_softmax(wide, 6, num_valid_rows=nv), f"nvr={nv}")


def test_forward_routed_equals_topk_then_forward():
    import block_scaled_moe_gb300 as bm
    w = synth.micro(96, 256, 256, 40, 6, nvr=90, invalid_frac=0.0, dispatch="compact", seed=31)
    c = Case(w)
    lg = _logits(w.T, w.E, seed=5, ties=False).cuda()
    for path in ["fused", "multi"]:
        L = c.layer(route_tile=32, path=path, debug=True)
        a = torch_bf16_bits(L.forward_routed(c.xd, lg, c.nvrd))
        torch.cuda.synchronize()
        ids, wts = bm.topk_softmax(lg, w.K, num_valid_rows=c.nvrd)
        b = torch_bf16_bits(L.forward(c.xd, ids, wts, c.nvrd))
        torch.cuda.synchronize()
        assert np.array_equal(a, b), path
        assert np.array_equal(L.debug_array("topk_ids").reshape(w.T, w.K), ids.cpu().numpy())
        r = oracle.topk_softmax(lg.cpu().numpy(), w.K, num_valid_rows=w.nvr)
        ref = oracle.moe_forward(c.x, r["ids"], r["weights"], c.Wh, num_valid_rows=w.nvr)
        assert_close(a, ref, path)
        assert L.read_status() == 0


def test_forward_routed_graph_follows_row_count():
    w = synth.micro(64, 256, 128, 8, 2, nvr=64, invalid_frac=0.0, dispatch="fixed", seed=41)
    c = Case(w)
    lg = _logits(w.T, w.E, seed=6, ties=False).cuda()
    L = c.layer(route_tile=32)
    eager = torch_bf16_bits(L.forward_routed(c.xd, lg, c.nvrd))
    s = torch.cuda.Stream()
    out = torch.empty_like(c.xd)
    with torch.cuda.stream(s):
        L.forward_routed(c.xd, lg, c.nvrd, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.forward_routed(c.xd, lg, c.nvrd, out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(torch_bf16_bits(out), eager)
    c.nvrd.fill_(9)
    g.replay()
    torch.cuda.synchronize()
    got = torch_bf16_bits(out)
    assert np.array_equal(got[:9], eager[:9]) and np.all(got[9:] == 0)
