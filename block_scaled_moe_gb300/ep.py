"""Expert-parallel exchange around the layer: host logic for boxes with several GPUs.

The pages' deployment (ROCm/aiter PR #6881, Motivation: one MegaMoEV2 instance per rank with expert
parallelism over 8 ranks; vLLM PR #61262 review notes: the decode or the large runtime is picked by the
largest token count across the data-parallel ranks) shards the experts over the ranks of a group:

* dispatch: each token row goes once to every rank that owns at least one of its valid top-k experts,
  as MXFP8 (E4M3 codes and one E8M0 scale per 1x32 block along H, the layer's own input format), with
  its top-k slots rewritten to that rank's local expert ids (-1 for slots owned elsewhere);
* each rank runs the layer on one row per valid local slot (`routes`), weight 1 and MXFP8 GEMM2 rows,
  so its outputs are the routes' GEMM2 rows exactly;
* combine: the GEMM2 rows travel back as MXFP8 in the main path's 1x32 format (aiter #6881 Technical
  Details, small input: GEMM2 rows sent to the combine as FP8) and the owner adds, per token, its own
  top-k weights times the rows in ascending k, in float, rounding to BF16 once.

Both formats are exact for what they carry: re-quantising a dequantised MXFP8 row by the OCP rule
returns the same codes and scales, so the receiving layer sees the sender's quantised row, and the
owner's sum is the layer's combine over MXFP8 GEMM2 rows.  The exchanges use
`torch.distributed.all_to_all_single` with split sizes agreed by a first exchange of row counts, so the
same code runs on NCCL (GPU buffers) or gloo (CPU tensors).  Experts are split in contiguous blocks of
E / world.  Only the host logic lives here; on one GPU the layer is not sharded.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch


def experts_per_rank(E: int, world: int) -> int:
    if world < 1 or E % world:
        raise ValueError(f"E={E} experts do not split evenly over {world} ranks")
    return E // world


# ------------------------------------------------------------------ MXFP8 rows on the wire

def mxfp8_rows(x: torch.Tensor):
    """MXFP8 of rows [n, H] (any float dtype, H % 32 == 0) by the OCP MX rule: per 1x32 block, E8M0 code
    clamp(floor(log2 amax) - 8 + 127, 0, 254) (0 for an all-zero block), elements E4M3 round to nearest
    even of x / 2^(code - 127), saturating at +-448.  Returns (codes uint8 [n, H], scales uint8 [n, H/32])."""
    n, H = x.shape
    b = x.to(torch.float32).reshape(n, H // 32, 32)
    amax = b.abs().amax(dim=-1)
    ex = torch.frexp(amax)[1].to(torch.int32) - 1           # floor(log2 amax) for amax > 0
    code = torch.clamp(ex - 8 + 127, 0, 254)
    code = torch.where(amax > 0, code, torch.zeros_like(code))
    scaled = b * torch.ldexp(torch.ones_like(amax), (127 - code).to(torch.float32))[..., None]
    q = torch.clamp(scaled, -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.reshape(n, H), code.to(torch.uint8)


def mxfp8_values(codes: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """float32 [n, H] of MXFP8 rows (exact: every value is an E4M3 value times a power of two)."""
    n, H = codes.shape
    v = codes.view(torch.float8_e4m3fn).to(torch.float32).reshape(n, H // 32, 32)
    s = torch.ldexp(torch.ones(scales.shape, dtype=torch.float32, device=scales.device),
                    scales.to(torch.float32) - 127.0)
    return (v * s[..., None]).reshape(n, H)


@dataclass
class EPPlan:
    """Where this rank's token rows go.

    send_rows   int64 [S]: local token row of each outgoing row, destination-major (rank ascending),
                token ascending within a destination
    send_counts list[int]: rows per destination rank
    ids         int32 [S, K]: the row's slots as the destination's local expert ids, -1 elsewhere
    weights     float32 [S, K]: the slots' weights, 0 where ids is -1 (kept by the owner)
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
    dist.all_to_all_single(out, t.contiguous(), recv_counts, send_counts, group=group)
    return out


def _counts(send_counts: List[int], device, group=None) -> List[int]:
    import torch.distributed as dist
    sc = torch.tensor(send_counts, dtype=torch.int64, device=device)
    rc = torch.empty_like(sc)
    dist.all_to_all_single(rc, sc, group=group)
    return [int(v) for v in rc.tolist()]


@dataclass
class Received:
    """Rows this rank computes, in source-rank order: x [R, H] BF16 (the senders' MXFP8 rows, exactly),
    ids [R, K] (local expert ids, -1 elsewhere), recv_counts (rows per source rank) and the bytes per
    row that crossed the wire."""
    x: torch.Tensor
    ids: torch.Tensor
    recv_counts: List[int]
    wire_bytes_per_row: int = 0


def dispatch(plan: EPPlan, x: torch.Tensor, group=None) -> Received:
    """Send every planned row (x: this rank's BF16 rows [T, H]) as MXFP8 with its local slot ids."""
    recv_counts = _counts(plan.send_counts, x.device, group)
    codes, scales = mxfp8_rows(x[plan.send_rows])
    rc = _exchange(codes, plan.send_counts, recv_counts, group)
    rs = _exchange(scales, plan.send_counts, recv_counts, group)
    ri = _exchange(plan.ids, plan.send_counts, recv_counts, group)
    H = x.shape[1]
    K = plan.ids.shape[1]
    return Received(mxfp8_values(rc, rs).to(torch.bfloat16), ri, recv_counts,
                    wire_bytes_per_row=H + H // 32 + 4 * K)


@dataclass
class Routes:
    """One row per valid local slot of the received rows, for the layer: x [R', H], ids [R', K] (the local
    expert in column 0, -1 elsewhere), weights [R', K] (1 in column 0), and where each route came from:
    its received row, its top-k slot k, and the number of routes per source rank."""
    x: torch.Tensor
    ids: torch.Tensor
    weights: torch.Tensor
    row: torch.Tensor
    k: torch.Tensor
    counts: List[int] = field(default_factory=list)


def routes(received: Received) -> Routes:
    """Expand the received rows into their valid local slots (received-row order, k ascending, so the
    routes of a source rank stay contiguous)."""
    ids = received.ids
    R, K = ids.shape
    r_idx, k_idx = torch.nonzero(ids >= 0, as_tuple=True)     # row-major: rows ascending, then k
    n = r_idx.numel()
    rid = torch.full((n, K), -1, dtype=torch.int32, device=ids.device)
    rid[:, 0] = ids[r_idx, k_idx]
    rw = torch.zeros((n, K), dtype=torch.float32, device=ids.device)
    rw[:, 0] = 1.0
    bounds = torch.tensor([0] + list(torch.cumsum(torch.tensor(received.recv_counts), 0)), device=ids.device)
    counts = [int(((r_idx >= bounds[i]) & (r_idx < bounds[i + 1])).sum()) for i in range(len(received.recv_counts))]
    return Routes(received.x[r_idx], rid, rw, r_idx, k_idx.to(torch.int32), counts)


def combine(plan: EPPlan, received: Received, rt: Routes, y_rows: torch.Tensor, topk_weights: torch.Tensor,
            T: int, group=None):
    """Return the routes' GEMM2 rows (y_rows [R', H]: the layer's output for `rt`, which is the routes'
    MXFP8 GEMM2 rows exactly) to their owners as MXFP8, and combine them there: per token, its own top-k
    weights times the rows in ascending k, float sums (each product rounded, then added), one BF16
    rounding.  Returns (out BF16 [T, H], wire bytes per returned row); rows with no route are +0."""
    H = y_rows.shape[1] if y_rows.dim() == 2 else 0
    dev = topk_weights.device
    codes, scales = mxfp8_rows(y_rows) if y_rows.shape[0] else (
        torch.zeros((0, H), dtype=torch.uint8, device=dev), torch.zeros((0, H // 32), dtype=torch.uint8, device=dev))
    # route tag: the row's position in its source's send order, and its slot k
    first = torch.tensor([0] + list(torch.cumsum(torch.tensor(received.recv_counts), 0))[:-1], device=rt.row.device)
    src = torch.bucketize(rt.row, torch.tensor(list(torch.cumsum(torch.tensor(received.recv_counts), 0)),
                                                device=rt.row.device), right=True)
    tag = torch.stack([(rt.row - first[src]).to(torch.int32), rt.k], dim=1) if rt.row.numel() else \
        torch.zeros((0, 2), dtype=torch.int32, device=dev)
    back_counts = _counts(rt.counts, dev, group)               # routes each destination returns to this rank
    bc = _exchange(codes, rt.counts, back_counts, group)
    bs = _exchange(scales, rt.counts, back_counts, group)
    bt = _exchange(tag, rt.counts, back_counts, group)
    K = topk_weights.shape[1]
    y = torch.zeros((T, K, H), dtype=torch.float32, device=dev)
    have = torch.zeros((T, K), dtype=torch.bool, device=dev)
    off, sent_off = 0, 0
    vals = mxfp8_values(bc, bs) if bc.shape[0] else torch.zeros((0, H), dtype=torch.float32, device=dev)
    for r, n in enumerate(back_counts):                         # source ranks ascending
        if n:
            pos, kk = bt[off:off + n, 0].to(torch.int64), bt[off:off + n, 1].to(torch.int64)
            tok = plan.send_rows[sent_off + pos]
            y[tok, kk] = vals[off:off + n]
            have[tok, kk] = True
        off += n
        sent_off += plan.send_counts[r]
    acc = torch.zeros((T, H), dtype=torch.float32, device=dev)
    w = topk_weights.to(torch.float32)
    for k in range(K):                                         # ascending k, like the layer's combine
        contrib = (w[:, k:k + 1] * y[:, k]).to(torch.float32)
        acc = torch.where(have[:, k:k + 1], acc + contrib, acc)
    out = acc.to(torch.bfloat16)
    out[~have.any(dim=1)] = 0
    return out, H + H // 32 + 8


def select_runtime(local_T: int, small_max: int, group=None, device=None) -> str:
    """"decode" (the fixed-slot runtime sized for at most `small_max` rows) when the largest token count
    over the group's ranks fits it, else "large"; every rank gets the same answer."""
    import torch.distributed as dist
    t = torch.tensor([int(local_T)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return "decode" if int(t.item()) <= small_max else "large"
