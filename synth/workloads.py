"""Seeded synthetic workloads for the fused block-scaled MoE layer.

This module only *generates inputs*.  It holds none of the layer's arithmetic
(no activation quantisation, no GEMM, no SwiGLU, no combine); both the CUDA
library and the CPU oracle consume the arrays it returns.

Workload shapes follow the pages:
  * DeepSeek-V4-Pro MoE: H=7168, I=3072, 384 experts, top-6
    (ROCm/aiter PR #6881 "MegaMoEV2: fuse Dispatch, GEMM1, GEMM2 and Combine
    into one kernel", Test Result table header).
  * DeepSeek-V4.1-Flash MoE: H=5120, I=2304, 384 experts, top-6
    (ROCm/aiter PR #6154 "Add full-expert DeepSeek V4.1 Flash MegaMoE tuning
    for gfx950", Summary).
  * Expert weights are MXFP4 (E2M1 codes, one E8M0 scale per 32 along K);
    activations enter as BF16 rows.

Recipe (all seeded):
  * x: float32 N(0,1) from numpy PCG64, rounded to BF16 (round-to-nearest-even).
  * routing: Gumbel-top-K over per-expert logits (equal logits = uniform,
    log Zipf(s) over a seeded expert order = skewed); K distinct experts per row.
    The "hot" workload instead draws every slot independently (25% one seeded
    expert, else Zipf over the others), so a row may repeat an expert.
  * invalid slots: exactly floor(p*T*K) flat slots chosen by a seeded
    permutation get id -1; rows at or past num_valid_rows of the skewed
    prefill workload are routed entirely to -1.
  * routing weights: float32 softmax of N(0,1) logits over the K slots.
  * expert weights: N(0, 0.02) drawn with a seeded torch generator on the device
    that will hold them, quantised to MXFP4 by the OCP MX rule
    (scale = 2^(floor(log2 amax) - 2), E2M1 round-to-nearest-even, saturate at 6),
    two codes per byte with element 2j in the low nibble.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    nvr: int                 # num_valid_rows passed to the layer
    routing: str             # "uniform" | "zipf" | "hot_zipf"
    invalid_frac: float      # fraction of flat slots set to -1
    swiglu_limit: float      # 0 = plain SwiGLU, 10 = clamp-10 SwiGLU
    dispatch: str            # "fixed" | "compact"
    capacity: int            # rows the layer instance is sized for (MTPR)
    zipf_s: float = 1.3
    hot_frac: float = 0.0
    seed: int = 0

    @property
    def weight_bytes_per_expert(self) -> int:
        # W13 [2I,H] + W2 [H,I]: 1/2 byte per code, 1/32 byte per scale
        return 3 * self.H * self.I // 2 + 3 * self.H * self.I // 32


WORKLOADS = {
    # Tiny MoE: parity case that the oracle finishes within seconds.
    "tiny": Workload("tiny", T=64, H=256, I=128, E=8, K=2, nvr=60, routing="uniform",
                     invalid_frac=0.10, swiglu_limit=0.0, dispatch="compact", capacity=64),
    # Decode, fixed-slot, V4-Flash shape, MTPR=128.
    "decode_flash": Workload("decode_flash", T=128, H=5120, I=2304, E=384, K=6, nvr=128,
                             routing="uniform", invalid_frac=0.0, swiglu_limit=10.0,
                             dispatch="fixed", capacity=128),
    # Small-M single-launch case, V4-Pro shape, Zipf(1.3) skew, 5% invalid slots.
    "smallm_pro": Workload("smallm_pro", T=512, H=7168, I=3072, E=384, K=6, nvr=480,
                           routing="zipf", invalid_frac=0.05, swiglu_limit=0.0,
                           dispatch="compact", capacity=512),
    # Large-M persistent case, V4-Pro shape, uniform, 2% invalid slots.
    "largem_pro": Workload("largem_pro", T=8192, H=7168, I=3072, E=384, K=6, nvr=8192,
                           routing="uniform", invalid_frac=0.02, swiglu_limit=0.0,
                           dispatch="compact", capacity=8192),
    # Skewed prefill, V4-Flash shape: Zipf(1.3) plus one expert taking 25% of routes.
    "skewed_flash": Workload("skewed_flash", T=4096, H=5120, I=2304, E=384, K=6, nvr=3500,
                             routing="hot_zipf", invalid_frac=0.0, swiglu_limit=10.0,
                             dispatch="compact", capacity=4096, hot_frac=0.25),
    # Profiling stand-in for the decode workload: same H, I, top-k and clamp,
    # 64 experts (1.2 GB of MXFP4 weights) so a full ncu capture stays small.
    "decode_flash_e64": Workload("decode_flash_e64", T=32, H=5120, I=2304, E=64, K=6, nvr=32,
                                 routing="uniform", invalid_frac=0.0, swiglu_limit=10.0,
                                 dispatch="fixed", capacity=32),
    # Profiling stand-in for the large-input workload: Pro shape, 48 experts (1.7 GB of MXFP4
    # weights) and 1024 rows, so experts hold ~128 routes each as in the 8192-row case.
    "largem_pro_e48": Workload("largem_pro_e48", T=1024, H=7168, I=3072, E=48, K=6, nvr=1024,
                               routing="uniform", invalid_frac=0.02, swiglu_limit=10.0,
                               dispatch="compact", capacity=1024),
}


def get(name: str, **overrides) -> Workload:
    return dataclasses.replace(WORKLOADS[name], **overrides)


def micro(T: int, H: int, I: int, E: int, K: int, *, nvr: Optional[int] = None,
          routing: str = "uniform", invalid_frac: float = 0.1, swiglu_limit: float = 0.0,
          dispatch: str = "compact", capacity: Optional[int] = None, seed: int = 0,
          hot_frac: float = 0.0) -> Workload:
    """An ad-hoc small workload (tests)."""
    return Workload(f"micro_T{T}_H{H}_I{I}_E{E}_K{K}", T=T, H=H, I=I, E=E, K=K,
                    nvr=T if nvr is None else nvr, routing=routing, invalid_frac=invalid_frac,
                    swiglu_limit=swiglu_limit, dispatch=dispatch,
                    capacity=T if capacity is None else capacity, seed=seed,
                    hot_frac=hot_frac)


# ----------------------------------------------------------------------------- streams

_STREAMS = ("x", "route", "mask", "wlogit", "order", "hot", "weights")


def _rngs(seed: int) -> dict:
    children = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    return {k: np.random.Generator(np.random.PCG64(c)) for k, c in zip(_STREAMS, children)}


def _weight_seed(seed: int) -> int:
    child = np.random.SeedSequence(seed).spawn(len(_STREAMS))[_STREAMS.index("weights")]
    return int(child.generate_state(1, dtype=np.uint64)[0] & ((1 << 62) - 1))


# ----------------------------------------------------------------------------- activations

def make_x(w: Workload) -> torch.Tensor:
    """BF16 [T,H] hidden rows, N(0,1) rounded to nearest-even BF16 (CPU tensor)."""
    r = _rngs(w.seed)["x"]
    x32 = r.standard_normal((w.T, w.H), dtype=np.float32)
    return torch.from_numpy(x32).to(torch.bfloat16)


# ----------------------------------------------------------------------------- routing

def _zipf_logits(E: int, s: float, order: np.ndarray) -> np.ndarray:
    ranks = np.empty(E, dtype=np.float64)
    ranks[order] = np.arange(1, E + 1, dtype=np.float64)
    return -s * np.log(ranks)


def make_routing(w: Workload):
    """Returns (topk_ids int32 [T,K], topk_weights float32 [T,K]) as numpy arrays."""
    rs = _rngs(w.seed)
    T, E, K = w.T, w.E, w.K
    if w.routing in ("uniform", "zipf"):
        if K > E:
            raise ValueError("distinct top-k needs K <= E")
        if w.routing == "uniform":
            logits = np.zeros(E)
        else:
            logits = _zipf_logits(E, w.zipf_s, rs["order"].permutation(E))
        g = rs["route"].gumbel(size=(T, E)) + logits[None, :]
        ids = np.argsort(-g, axis=1, kind="stable")[:, :K].astype(np.int32)
    elif w.routing == "hot_zipf":
        hot = int(rs["hot"].integers(E))
        others = np.array([e for e in range(E) if e != hot], dtype=np.int64)
        others = others[rs["order"].permutation(E - 1)]
        p = np.arange(1, E, dtype=np.float64) ** (-w.zipf_s)
        p /= max(p.sum(), 1.0)
        pick_hot = rs["route"].random((T, K)) < w.hot_frac
        if E == 1:
            pick_hot[:] = True
            z = np.zeros((T, K), np.int64)
        else:
            z = others[rs["route"].choice(E - 1, size=(T, K), p=p)]
        ids = np.where(pick_hot, hot, z).astype(np.int32)
    else:
        raise ValueError(w.routing)
    n_mask = int(math.floor(w.invalid_frac * T * K))
    if n_mask:
        flat = rs["mask"].permutation(T * K)[:n_mask]
        ids.reshape(-1)[flat] = -1
    if w.routing == "hot_zipf":
        ids[w.nvr:, :] = -1
    lg = rs["wlogit"].standard_normal((T, K), dtype=np.float32)
    lg = lg - lg.max(axis=1, keepdims=True)
    ex = np.exp(lg, dtype=np.float32)
    wts = (ex / ex.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    return ids, wts


# ----------------------------------------------------------------------------- weights

def _mxfp4_encode(w32: torch.Tensor):
    """OCP MX FP4 encoding of float32 [..., K] (K % 32 == 0) -> (packed u8 [..., K/2], scales u8 [..., K/32])."""
    *lead, Kd = w32.shape
    b = w32.reshape(*lead, Kd // 32, 32)
    amax = b.abs().amax(dim=-1)
    _, ex = torch.frexp(amax)                       # amax = m * 2^ex, m in [0.5, 1)
    code = (ex - 1 - 2 + 127).clamp(0, 254)          # floor(log2 amax) - emax(E2M1) + bias
    code = torch.where(amax == 0, torch.zeros_like(code), code)
    v = torch.ldexp(b.abs(), (127 - code).unsqueeze(-1).to(b.dtype))  # |x| / 2^(code-127)
    # nearest-even onto {0,.5,1,1.5,2,3,4,6} (codes 0..7), saturating at 6
    q = ((v > 0.25).to(torch.uint8) + (v >= 0.75) + (v > 1.25) + (v >= 1.75)
         + (v > 2.5) + (v >= 3.5) + (v > 5.0)).to(torch.uint8)
    nib = q | (torch.signbit(b).to(torch.uint8) << 3)
    nib = nib.reshape(*lead, Kd)
    packed = nib[..., 0::2] | (nib[..., 1::2] << 4)
    return packed.contiguous(), code.to(torch.uint8).contiguous()


def make_weights(w: Workload, device="cpu", std: float = 0.02, w13_gain: float = 1.0):
    """MXFP4 expert weights on `device`:
    w13 u8 [E,2I,H/2], w13_sf u8 [E,2I,H/32], w2 u8 [E,H,I/2], w2_sf u8 [E,H,I/32].
    Rows [0,I) of W13 are the gate projection, rows [I,2I) the up projection.
    Values depend on (seed, device type): CPU and CUDA generators differ."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(_weight_seed(w.seed))
    E, H, I = w.E, w.H, w.I
    w13 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=device)
    w13s = torch.empty((E, 2 * I, H // 32), dtype=torch.uint8, device=device)
    w2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=device)
    w2s = torch.empty((E, H, I // 32), dtype=torch.uint8, device=device)
    for e in range(E):
        a = torch.randn((2 * I, H), generator=gen, device=device, dtype=torch.float32) * (std * w13_gain)
        w13[e], w13s[e] = _mxfp4_encode(a)
        b = torch.randn((H, I), generator=gen, device=device, dtype=torch.float32) * std
        w2[e], w2s[e] = _mxfp4_encode(b)
    return w13, w13s, w2, w2s


def make_all(w: Workload, weight_device="cpu", **kw):
    x = make_x(w)
    ids, wts = make_routing(w)
    return x, ids, wts, make_weights(w, weight_device, **kw)


def active_experts(ids: np.ndarray, E: int, nvr: int) -> np.ndarray:
    v = ids[:nvr].reshape(-1)
    v = v[(v >= 0) & (v < E)]
    return np.unique(v)
