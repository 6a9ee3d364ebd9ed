"""Expert-parallel host logic on two gloo ranks (CPU processes, no GPU).

Each rank owns half of the experts and a shard of the tokens.  Dispatch sends MXFP8 rows (codes and
1x32 scales), each rank runs the layer (the CPU oracle stands in for the GPU layer) on one row per
valid local slot with weight 1 and MXFP8 GEMM2 rows, the GEMM2 rows travel back as MXFP8 and the owner
combines them with its own top-k weights.  For every token the result must equal the single-process
oracle with MXFP8 GEMM2 rows bit for bit (both formats are exact for what they carry), and the bytes
per row on the wire are the MXFP8 ones.  The runtime choice follows the largest token count over the
ranks.

Failure detection (host side, no GPU): a rank that leaves between steps, with none of its exchanges in
flight, makes the other rank's next exchange end with an error within the process group's short
timeout instead of waiting for ever.
"""

import datetime
import os
import socket
import time

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_q, cut=17):
    import torch.distributed as dist
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        from block_scaled_moe_gb300 import ep
        from parity_util import compare

        w = synth.micro(40, 256, 128, 8, 3, nvr=38, routing="uniform", invalid_frac=0.1, seed=77)
        x, ids, wts, W = synth.make_all(w)
        Wh = [t.cpu() for t in W]
        per = ep.experts_per_rank(w.E, world)
        # this rank's token shard (uneven on purpose, or empty) and its experts' weights
        lo, hi = (0, cut) if rank == 0 else (cut, w.T)
        nv_local = max(0, min(hi, w.nvr) - lo)
        xl, idsl, wtsl = x[lo:hi], torch.from_numpy(ids[lo:hi]), torch.from_numpy(wts[lo:hi])
        plan = ep.make_plan(idsl, wtsl, w.E, world, rank, num_valid_rows=nv_local)
        rcv = ep.dispatch(plan, xl)
        rt = ep.routes(rcv)
        mine = [t[rank * per:(rank + 1) * per].contiguous() for t in Wh]
        if rt.x.shape[0]:
            part = oracle.moe_forward(rt.x, rt.ids.numpy(), rt.weights.numpy(), mine, y_format="mxfp8")
            y_rows = torch.from_numpy(part.view(np.int16)).view(torch.bfloat16)
        else:
            y_rows = torch.zeros((0, w.H), dtype=torch.bfloat16)
        out, back_bytes = ep.combine(plan, rcv, rt, y_rows, wtsl, hi - lo)
        ref = oracle.moe_forward(x, ids, wts, Wh, num_valid_rows=w.nvr, y_format="mxfp8")[lo:hi]
        got = out.view(torch.int16).numpy().view(np.uint16)
        c = compare(got, ref)
        c["exact"] = bool(np.array_equal(got, ref))
        c["wire"] = (rcv.wire_bytes_per_row, back_bytes)
        zero_rows_ok = bool(np.all(got[nv_local:] == 0))
        # runtime choice: the same answer on every rank, from the largest local count
        biggest = max(cut, w.T - cut)
        choice_small = ep.select_runtime(hi - lo, small_max=biggest)      # the largest shard fits
        choice_large = ep.select_runtime(hi - lo, small_max=biggest - 1)  # it does not
        result_q.put((rank, c, zero_rows_ok, choice_small, choice_large, plan.send_counts, rcv.recv_counts))
        dist.destroy_process_group()
    except Exception as exc:  # pragma: no cover - reported to the parent
        result_q.put((rank, repr(exc), None, None, None, None, None))


@pytest.mark.parametrize("cut", [17, 0, 40], ids=["uneven", "rank0_idle", "rank1_idle"])
def test_ep_dispatch_combine_two_gloo_ranks(cut):
    """Token shards [0, cut) and [cut, 40): uneven, or one rank holding no tokens (it still computes
    the rows the other rank sends to its experts)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q, cut)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r = q.get(timeout=300)
        res[r[0]] = r
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    H, K = 256, 3
    for rank in range(2):
        _, c, zero_ok, small, large, sent, recv = res[rank]
        assert isinstance(c, dict), c
        assert c["nan"] == 0 and c["rel_l2"] <= 1e-2 and c["bad"] == 0, (rank, c)
        assert c["exact"], (rank, c)
        # dispatch: H E4M3 codes + H/32 E8M0 scales + K int32 slot ids per row; combine: codes + scales
        # + an 8-byte (position, slot) tag per GEMM2 row (a BF16 row alone would be 2H bytes)
        assert c["wire"] == (H + H // 32 + 4 * K, H + H // 32 + 8), c["wire"]
        assert zero_ok
        assert small == "decode" and large == "large"
    # what rank a sends to rank b is what b receives from a
    assert res[0][5][1] == res[1][6][0] and res[1][5][0] == res[0][6][1]


def test_plan_routes_each_row_once_per_owner():
    from block_scaled_moe_gb300 import ep
    ids = torch.tensor([[0, 5], [1, 2], [7, 6], [-1, 3], [4, 4]], dtype=torch.int32)
    w = torch.tensor([[0.6, 0.4], [0.5, 0.5], [0.9, 0.1], [0.0, 1.0], [0.3, 0.7]])
    plan = ep.make_plan(ids, w, E=8, world=2, rank=0, num_valid_rows=4)
    # experts 0-3 on rank 0, 4-7 on rank 1; row 4 is past the row count
    assert plan.send_counts == [3, 2]
    assert plan.send_rows.tolist() == [0, 1, 3, 0, 2]
    assert plan.ids.tolist() == [[0, -1], [1, 2], [-1, 3], [-1, 1], [3, 2]]
    assert torch.allclose(plan.weights, torch.tensor([[0.6, 0], [0.5, 0.5], [0, 1.0], [0, 0.4], [0.9, 0.1]]))
    with pytest.raises(ValueError):
        ep.make_plan(ids, w, E=8, world=3, rank=0)


def _leave(result_q):
    """End this process at once (no process-group teardown), after the queued result is sent."""
    result_q.close()
    result_q.join_thread()
    os._exit(0)


def _leaving_worker(rank, world, port, result_q):
    import torch.distributed as dist
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
        from block_scaled_moe_gb300 import ep

        w = synth.micro(24, 64, 64, 4, 2, nvr=24, routing="uniform", invalid_frac=0.0, seed=5)
        x, ids, wts, _ = synth.make_all(w)
        lo, hi = (0, 12) if rank == 0 else (12, 24)
        plan = ep.make_plan(torch.from_numpy(ids[lo:hi]), torch.from_numpy(wts[lo:hi]), w.E, world, rank)
        rcv = ep.dispatch(plan, x[lo:hi])                  # step 1, both ranks
        rt = ep.routes(rcv)
        ep.combine(plan, rcv, rt, rt.x, torch.from_numpy(wts[lo:hi]), hi - lo)  # any rows stand in for the layer's
        if rank == 1:
            result_q.put((1, "left", 0.0))                 # leaves between steps
            _leave(result_q)
        t0 = time.monotonic()
        try:
            ep.dispatch(plan, x[lo:hi])                    # step 2: the peer is gone
            result_q.put((0, "no error", time.monotonic() - t0))
        except Exception as exc:  # the collective's error is the detection
            result_q.put((0, type(exc).__name__, time.monotonic() - t0))
        _leave(result_q)
    except Exception as exc:  # pragma: no cover - reported to the parent
        result_q.put((rank, "setup: " + repr(exc), -1.0))


def test_rank_leaving_between_steps_is_detected():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_leaving_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(2):
            r = q.get(timeout=120)
            res[r[0]] = r
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():  # only this test's own child processes
                p.kill()
                p.join(timeout=10)
    assert res[1][1] == "left", res
    assert res[0][1] not in ("no error",) and not res[0][1].startswith("setup"), res
    assert 0.0 <= res[0][2] < 60.0, res  # ended by the peer's closed connection or the 5 s timeout


def test_mxfp8_rows_on_the_wire_are_exact():
    """The wire format of the exchange: the OCP MX quantisation of BF16 rows equals the oracle's, and
    dequantising then quantising again returns the same codes and scales (the receiving layer sees the
    sender's quantised rows)."""
    import oracle
    from block_scaled_moe_gb300 import ep
    oracle.build()
    g = torch.Generator().manual_seed(3)
    x = (torch.randn((37, 512), generator=g) * torch.logspace(-6, 6, 37)[:, None]).to(torch.bfloat16)
    x[5, 64:96] = 0
    x[6, :32] = -0.0
    codes, scales = ep.mxfp8_rows(x)
    oc, os_ = oracle.quant_mxfp8_rows(x)
    assert np.array_equal(codes.numpy(), oc) and np.array_equal(scales.numpy(), os_)
    back = ep.mxfp8_values(codes, scales).to(torch.bfloat16)
    c2, s2 = ep.mxfp8_rows(back)
    assert torch.equal(c2, codes) and torch.equal(s2, scales)
