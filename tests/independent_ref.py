"""A second, independent CPU formulation of the layer, used only to pin the oracle.

The oracle (C) loops token by token over its k slots.  This module instead
groups the routes by expert (gather -> dense GEMM -> scatter), vectorises with
numpy/torch, decodes E4M3/E8M0 with torch's casts and encodes E4M3 with torch's
round-to-nearest-even cast.  It shares no code with the oracle or with the CUDA
library.  Format facts come from the OCP Microscaling Formats (MX) v1.0 spec:
E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, E4M3 max normal 448, E8M0 = 2^(c-127).
"""

from __future__ import annotations

import numpy as np
import torch

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def fp4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes u8 [..., K/2] (element 2j low nibble), scales u8 [..., K/32] -> float64 [..., K]."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = codes & 0xF
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    mag = E2M1_MAG[nib & 7]
    val = np.where(nib & 8, -mag, mag)
    sc = np.ldexp(1.0, np.asarray(scales, dtype=np.int64) - 127)
    return val * np.repeat(sc, 32, axis=-1)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e8m0_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e8m0fnu).to(torch.float64).numpy()


def q8(x32: np.ndarray):
    """MXFP8 1x32 quantisation of float32 [..., K] -> (codes u8, scales u8)."""
    x32 = np.asarray(x32, dtype=np.float32)
    *lead, K = x32.shape
    b = x32.reshape(*lead, K // 32, 32)
    amax = np.abs(b).max(axis=-1)
    _, ex = np.frexp(amax.astype(np.float64))
    code = np.clip(ex.astype(np.int64) - 1 - 8 + 127, 0, 254)
    code = np.where(amax == 0, 0, code)
    scaled = b.astype(np.float64) * np.ldexp(1.0, 127 - code)[..., None]
    scaled = np.clip(scaled, -448.0, 448.0).astype(np.float32)
    c = torch.from_numpy(np.ascontiguousarray(scaled)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return c.reshape(*lead, K), code.astype(np.uint8)


def q8_dequant(codes, scales) -> np.ndarray:
    return e4m3_decode(codes) * np.repeat(e8m0_decode(scales), 32, axis=-1)


def bf16_round(a32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def bf16_bits(a32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def swiglu(g: np.ndarray, I: int, limit: float) -> np.ndarray:
    a = g[:, :I].astype(np.float32)
    b = g[:, I:].astype(np.float32)
    if limit > 0:
        L = np.float32(limit)
        a = np.minimum(a, L)
        b = np.clip(b, -L, L)
    one = np.float32(1.0)
    sig = one / (one + np.exp(-a.astype(np.float64)).astype(np.float32))
    return (a * sig * b).astype(np.float32)


def grouped_forward(x_bf16: torch.Tensor, ids: np.ndarray, wts: np.ndarray, weights, nvr=None,
                    swiglu_limit: float = 0.0, y_fp32: bool = False, y_mxfp8: bool = False,
                    swiglu_fn=None) -> np.ndarray:
    """Per-expert grouped formulation.  Returns BF16 bits [T,H].  `swiglu_fn(g, I, limit)` replaces
    the activation (tests use it to plant wrong readings of the clamp)."""
    w13, w13s, w2, w2s = (np.asarray(a.cpu().numpy() if isinstance(a, torch.Tensor) else a) for a in weights)
    E, I2, _ = w13.shape
    I = I2 // 2
    x32 = x_bf16.float().numpy()
    T, H = x32.shape
    K = ids.shape[1]
    nvr = T if nvr is None else max(0, min(T, int(nvr)))
    xq, xs = q8(x32)
    xdq = q8_dequant(xq, xs)
    valid = (np.arange(T)[:, None] < nvr) & (ids >= 0) & (ids < E)
    Y = np.zeros((T, K, H), np.float32)
    for e in range(E):
        t_idx, k_idx = np.nonzero(valid & (ids == e))
        if len(t_idx) == 0:
            continue
        A = xdq[t_idx]
        G = (A @ fp4_dequant(w13[e], w13s[e]).T).astype(np.float32)
        h = (swiglu_fn or swiglu)(G, I, swiglu_limit)
        hq, hs = q8(h)
        Yv = (q8_dequant(hq, hs) @ fp4_dequant(w2[e], w2s[e]).T).astype(np.float32)
        if y_mxfp8:
            yq, ys = q8(Yv)
            Y[t_idx, k_idx] = q8_dequant(yq, ys).astype(np.float32)
        else:
            Y[t_idx, k_idx] = Yv if y_fp32 else bf16_round(Yv)
    acc = np.zeros((T, H), np.float32)
    for k in range(K):
        contrib = (wts[:, k:k + 1].astype(np.float32) * Y[:, k]).astype(np.float32)
        acc = (acc + np.where(valid[:, k:k + 1], contrib, np.float32(0))).astype(np.float32)
    out = bf16_bits(acc)
    out[~valid.any(axis=1)] = 0
    return out


def sort_dispatch(ids: np.ndarray, E: int, nvr=None):
    """Compact dispatch by a stable sort of (expert, flat slot id)."""
    T, K = ids.shape
    nvr = T if nvr is None else max(0, min(T, int(nvr)))
    flat = ids.reshape(-1).astype(np.int64)
    sid = np.arange(T * K)
    ok = ((sid // K) < nvr) & (flat >= 0) & (flat < E)
    keys = np.where(ok, flat, E)
    order = np.lexsort((sid, keys))
    order = order[ok[order]]
    counts = np.bincount(flat[ok], minlength=E).astype(np.int32)
    route_row = np.full(T * K, -1, np.int32)
    route_row[order] = np.arange(len(order), dtype=np.int32)
    return counts, np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), order.astype(np.int32), \
        route_row.reshape(T, K)
