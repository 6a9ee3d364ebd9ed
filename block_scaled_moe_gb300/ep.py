"""Expert-parallel exchange around the layer: host logic for boxes with several GPUs.

The pages' deployment (ROCm/aiter PR #6881, Motivation: one MegaMoEV2 instance per rank with expert
parallelism over 8 ranks; vLLM PR #61262 review notes: the decode or the large runtime is picked by the
largest token count across the data-parallel ranks) shards the experts over the ranks of a group:

* dispatch: each token row goes once to every rank that owns at least one of its valid top-k experts,
  with its top-k slots rewritten to that rank's local expert ids (-1 for slots owned elsewhere) and the
  matching weights (0 elsewhere);
* each rank runs the layer on what it received, over its own experts only;
* combine: every rank sends its partial output rows back to the tokens' owners, which add them in
  float, in ascending rank order, and round to BF16 once.

The exchanges use `torch.distributed.all_to_all_single` with split sizes agreed by a first exchange of
row counts, so the same code runs on NCCL (GPU buffers) or gloo (CPU tensors).  Experts are split in
contiguous blocks of E / world.  Only the host logic lives here; on one GPU the layer is not sharded.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch


def experts_per_rank(E: int, world: int) -> int:
    if world < 1 or E % world:
        raise ValueError(f"E={E} experts do not split evenly over {world} ranks")
    return E // world


@dataclass
class EPPlan:
    """Where this rank's token rows go.

    send_rows   int64 [S]: local token row of each outgoing row, destination-major (rank ascending),
                token ascending within a destination
    send_counts list[int]: rows per destination rank
    ids         int32 [S, K]: the row's slots as the destination's local expert ids, -1 elsewhere
    weights     float32 [S, K]: the slots' weights, 0 where ids is -1
    """
    world: int
    rank: int
    E: int
    send_rows: torch.Tensor
    send_counts: List[int]
    ids: torch.Tensor
    weights: torch.Tensor


def make_plan(topk_ids: torch.Tensor, topk_weights: torch.Tensor, E: int, world: int, rank: int,
              num_valid_rows: Optional[int] = None) -> EPPlan:
    """Dispatch plan of this rank's tokens (host tensors or device tensors; computed on their device)."""
    per = experts_per_rank(E, world)
    ids = topk_ids.to(torch.int64)
    T, K = ids.shape
    nvr = T if num_valid_rows is None else max(0, min(T, int(num_valid_rows)))
    rows_ok = (torch.arange(T, device=ids.device) < nvr)[:, None]
    valid = rows_ok & (ids >= 0) & (ids < E)
    dest = torch.where(valid, ids // per, torch.full_like(ids, -1))
    send_rows, send_ids, send_w, counts = [], [], [], []
    for r in range(world):
        mine = dest == r                                   # [T, K]
        rows = torch.nonzero(mine.any(dim=1)).flatten()    # ascending token rows
        sel = mine[rows]
        send_rows.append(rows)
        send_ids.append(torch.where(sel, ids[rows] - r * per, torch.full_like(ids[rows], -1)).to(torch.int32))
        send_w.append(torch.where(sel, topk_weights[rows].to(torch.float32),
                                  torch.zeros((), dtype=torch.float32, device=ids.device)))
        counts.append(int(rows.numel()))
    return EPPlan(world, rank, E, torch.cat(send_rows), counts,
                  torch.cat(send_ids).reshape(-1, K), torch.cat(send_w).reshape(-1, K))


def _exchange(t: torch.Tensor, send_counts: List[int], recv_counts: List[int], group=None) -> torch.Tensor:
    import torch.distributed as dist
    rows = t.shape[1:] if t.dim() > 1 else ()
    out = torch.empty((sum(recv_counts),) + tuple(rows), dtype=t.dtype, device=t.device)
    # BF16 rows travel as their bytes (a [rows, 2H] uint8 view keeps the row split)
    send = t.contiguous().view(torch.uint8) if t.dtype == torch.bfloat16 else t.contiguous()
    recv = out.view(torch.uint8) if t.dtype == torch.bfloat16 else out
    dist.all_to_all_single(recv, send, recv_counts, send_counts, group=group)
    return out


@dataclass
class Received:
    """Rows this rank computes: x [R, H], ids [R, K] (local expert ids), weights [R, K]."""
    x: torch.Tensor
    ids: torch.Tensor
    weights: torch.Tensor
    recv_counts: List[int]


def dispatch(plan: EPPlan, x: torch.Tensor, group=None) -> Received:
    """Send every planned row (x: this rank's BF16 rows [T, H]) and its slots to their ranks."""
    import torch.distributed as dist
    sc = torch.tensor(plan.send_counts, dtype=torch.int64, device=x.device)
    rc = torch.empty_like(sc)
    dist.all_to_all_single(rc, sc, group=group)
    recv_counts = [int(v) for v in rc.tolist()]
    xs = x[plan.send_rows]
    return Received(_exchange(xs, plan.send_counts, recv_counts, group),
                    _exchange(plan.ids, plan.send_counts, recv_counts, group),
                    _exchange(plan.weights, plan.send_counts, recv_counts, group),
                    recv_counts)


def combine(plan: EPPlan, received: Received, partial: torch.Tensor, T: int, group=None) -> torch.Tensor:
    """Return the partial rows (BF16 [R, H], in received order) to their owners and add them there:
    float sum in ascending source-rank order, one BF16 rounding.  Rows no rank computed are +0."""
    back = _exchange(partial, received.recv_counts, plan.send_counts, group)  # destination-major = rank order
    H = partial.shape[1]
    acc = torch.zeros((T, H), dtype=torch.float32, device=partial.device)
    hit = torch.zeros(T, dtype=torch.bool, device=partial.device)
    off = 0
    for n in plan.send_counts:                         # ranks ascending
        rows = plan.send_rows[off:off + n]
        acc[rows] += back[off:off + n].to(torch.float32)
        hit[rows] = True
        off += n
    out = acc.to(torch.bfloat16)
    out[~hit] = 0
    return out


def select_runtime(local_T: int, small_max: int, group=None, device=None) -> str:
    """"decode" (the fixed-slot runtime sized for at most `small_max` rows) when the largest token count
    over the group's ranks fits it, else "large"; every rank gets the same answer."""
    import torch.distributed as dist
    t = torch.tensor([int(local_T)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return "decode" if int(t.item()) <= small_max else "large"
