"""GPU stress and boundary tests (the pages' test list: epoch words preset a few counts short of 2^31 and 2^32,
interleaved calls of the two paths, eager and graph forwards over many shape transitions, no writes
past `out`, every route on one expert).

* the single-launch kernel's grid-barrier generation word preset a few counts short of 2^32 and 2^31 wraps
  during the next forwards without changing a bit;
* two handles on the same weights (fused and multi-kernel path) alternate eager forwards and CUDA
  graph replays over changing T; every output equals the reference of its T bitwise;
* guard rows after `out` stay untouched on both paths, with num_valid_rows below T;
* every row routes its first slot to the same expert (one expert holds several route tiles);
* failure detection without a fault: a grid barrier that can never complete (its arrival count
  preset out of reach through the test-only MOE_OPT_DEBUG_STALL_GRID) makes every CTA give up after
  the bounded wait; the status word reports the timeout and the grid-barrier site, and the next
  forward, after the status was read, is bitwise the earlier result.
"""

import time

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


def _case(T=128, seed=41):
    w = synth.micro(T, 256, 256, 12, 4, nvr=T, invalid_frac=0.05, dispatch="compact", seed=seed, swiglu_limit=10.0)
    return Case(w)


def _fwd(c, L, T, nv=None):
    nvr = None if nv is None else torch.tensor([nv], dtype=torch.int32, device="cuda")
    out = L.forward(c.xd[:T], c.idsd[:T], c.wtsd[:T], nvr)
    torch.cuda.synchronize()
    return torch_bf16_bits(out)


@pytest.mark.parametrize("preset", [(1 << 32) - 3, (1 << 31) - 3])
def test_grid_barrier_generation_word_wraps(preset):
    import block_scaled_moe_gb300 as bm
    c = _case()
    Lf = c.layer(route_tile=32, path="fused")
    Lm = c.layer(route_tile=32, path="multi")
    ref = _fwd(c, Lm, 128)
    bm.moe_set_option(Lf.h, bm.MOE_OPT_DEBUG_GRID_GEN, float(preset))
    for _ in range(3):  # each forward passes several grid barriers: the word wraps during these
        got = _fwd(c, Lf, 128)
        assert Lf.last_path == "fused"
        assert np.array_equal(got, ref)
    assert Lf.read_status() == 0
    with pytest.raises(bm.MoeError):
        bm.moe_set_option(Lf.h, bm.MOE_OPT_DEBUG_GRID_GEN, float(1 << 32))


def test_alternating_paths_eager_and_graphs():
    c = _case()
    Lf = c.layer(route_tile=32, path="fused")
    Lm = c.layer(route_tile=32, path="multi")
    Ts = [1, 5, 17, 32, 64, 100, 128]
    ref = {T: _fwd(c, Lm, T) for T in Ts}
    # one captured graph per (handle, T) for three sizes, each with its own output buffer
    s = torch.cuda.Stream()
    graphs = {}
    for L in (Lf, Lm):
        for T in (5, 64, 128):
            out = torch.empty((T, c.w.H), dtype=torch.bfloat16, device="cuda")
            with torch.cuda.stream(s):
                L.forward(c.xd[:T], c.idsd[:T], c.wtsd[:T], None, out=out, stream=s)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                L.forward(c.xd[:T], c.idsd[:T], c.wtsd[:T], None, out=out, stream=s)
            graphs[(id(L), T)] = (g, out)
    rng = np.random.default_rng(7)
    prev, transitions = None, 0
    for it in range(160):
        L = Lf if it % 2 == 0 else Lm
        if it % 3 == 0:
            T = int(rng.choice([5, 64, 128]))
            g, out = graphs[(id(L), T)]
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            got = torch_bf16_bits(out)
        else:
            T = int(rng.choice(Ts))
            got = _fwd(c, L, T)
        transitions += int(T != prev)
        prev = T
        assert np.array_equal(got, ref[T]), (it, T, L.last_path)
    assert transitions > 60
    assert Lf.read_status() == 0 and Lm.read_status() == 0


@pytest.mark.parametrize("path", ["fused", "multi"])
def test_no_writes_past_out(path):
    c = _case(T=100)
    L = c.layer(route_tile=32, path=path)
    T, guard = 100, 8
    buf = torch.empty((T + guard, c.w.H), dtype=torch.bfloat16, device="cuda")
    buf.view(torch.int16).fill_(0x5A5A)
    nvr = torch.tensor([77], dtype=torch.int32, device="cuda")
    L.forward(c.xd[:T], c.idsd[:T], c.wtsd[:T], nvr, out=buf[:T])
    torch.cuda.synchronize()
    tail = buf[T:].view(torch.int16).cpu().numpy()
    assert np.all(tail == 0x5A5A)
    got = torch_bf16_bits(buf[:T])
    assert np.all(got[77:] == 0)
    ref = oracle.moe_forward(c.x[:T], c.ids[:T], c.wts[:T], c.Wh, num_valid_rows=77,
                             swiglu_limit=c.w.swiglu_limit)
    assert_close(got, ref, path)


@pytest.mark.parametrize("route_tile", [32, 144])
def test_every_row_on_one_expert(route_tile):
    w = synth.micro(300, 256, 256, 8, 3, nvr=300, invalid_frac=0.0, dispatch="compact", seed=13, capacity=300)
    c = Case(w)
    t = np.arange(w.T)
    others = np.array([0, 1, 2, 3, 4, 6, 7], dtype=np.int32)
    ids = np.stack([np.full(w.T, 5, np.int32), others[t % 7], others[(t + 3) % 7]], axis=1)  # distinct per row
    c.ids = ids
    c.idsd.copy_(torch.from_numpy(ids))
    L = c.layer(route_tile=route_tile)
    got = torch_bf16_bits(c.run(L))
    torch.cuda.synchronize()
    assert_close(got, c.oracle(), f"NT={route_tile}")
    assert L.read_status() == 0


def test_stalled_grid_barrier_times_out_and_recovers():
    import block_scaled_moe_gb300 as bm
    c = _case()
    Lf = c.layer(route_tile=32, path="fused")
    ref = _fwd(c, Lf, 128)
    assert Lf.read_status() == 0
    with pytest.raises(bm.MoeError):
        bm.moe_set_option(Lf.h, bm.MOE_OPT_DEBUG_STALL_GRID, 2.0)
    bm.moe_set_option(Lf.h, bm.MOE_OPT_DEBUG_STALL_GRID, 1.0)
    t0 = time.monotonic()
    Lf.forward(c.xd, c.idsd, c.wtsd, None)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert Lf.last_path == "fused"
    assert 1.5 < waited < 60, waited  # every CTA's wait is bounded at 2 s
    st = Lf.read_status()
    assert st & bm.MOE_ST_TIMEOUT, hex(st)
    assert st & (1 << 14), hex(st)  # site: the fused path's grid barrier
    for _ in range(2):  # reading the timeout reset the barrier words
        assert np.array_equal(_fwd(c, Lf, 128), ref)
    assert Lf.read_status() == 0
