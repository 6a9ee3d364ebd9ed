"""CPU oracle of the fused block-scaled MoE layer -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this package.  The product library never does, and this
package imports nothing from the product library.

The arithmetic lives in `moe_oracle.c` (plain C, fp64 dot products); this file
compiles it with gcc and wraps it with ctypes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over token rows)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
            lib.orc_e2m1_value.restype = ctypes.c_double
            lib.orc_e2m1_value.argtypes = [i32]
            lib.orc_e4m3_value.restype = ctypes.c_double
            lib.orc_e4m3_value.argtypes = [i32]
            lib.orc_e8m0_value.restype = ctypes.c_double
            lib.orc_e8m0_value.argtypes = [i32]
            lib.orc_e4m3_encode.restype = i32
            lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
            lib.orc_float_to_bf16.restype = ctypes.c_uint16
            lib.orc_float_to_bf16.argtypes = [f32]
            lib.orc_quant_mxfp8_block.argtypes = [P, P, P]
            lib.orc_quant_mxfp8_rows.argtypes = [P, i64, i32, P, P]
            lib.orc_dispatch_compact.argtypes = [P, i32, i32, i32, P, P, P, P, P]
            lib.orc_dispatch_fixed.argtypes = [P, i32, i32, i32, P, i32, P, P, P]
            lib.orc_moe_forward.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P, P,
                                            f32, i32, P, i32, P, i32]
            lib.orc_route_intermediates.argtypes = [P, i32, i32, i32, i32, P, P, P, P, f32, P, P, P, P]
            lib.orc_topk_softmax.argtypes = [P, i32, i32, i32, P, i32, P, P]
            lib.orc_max_threads.restype = i32
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _bf16_bits(x):
    """torch bf16 tensor or uint16 array -> contiguous uint16 numpy bits."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.uint16)


def _np(a, dtype):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ formats

def e2m1_value(nib: int) -> float:
    return _load().orc_e2m1_value(int(nib))


def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(int(code))


def e8m0_value(code: int) -> float:
    return _load().orc_e8m0_value(int(code))


def e4m3_encode(v: float) -> int:
    return _load().orc_e4m3_encode(float(v))


def float_to_bf16_bits(f: float) -> int:
    return _load().orc_float_to_bf16(float(f))


def quant_mxfp8_block(x32) -> tuple:
    x = np.ascontiguousarray(x32, dtype=np.float32)
    assert x.shape == (32,)
    codes = np.zeros(32, np.uint8)
    sc = np.zeros(1, np.uint8)
    _load().orc_quant_mxfp8_block(_p(x), _p(codes), _p(sc))
    return codes, int(sc[0])


def quant_mxfp8_rows(x_bf16) -> tuple:
    """BF16 [rows, cols] -> (E4M3 codes u8 [rows, cols], E8M0 scales u8 [rows, cols/32])."""
    xb = _bf16_bits(x_bf16)
    rows, cols = xb.shape
    codes = np.zeros((rows, cols), np.uint8)
    scales = np.zeros((rows, cols // 32), np.uint8)
    rc = _load().orc_quant_mxfp8_rows(_p(xb), rows, cols, _p(codes), _p(scales))
    if rc:
        raise ValueError(f"orc_quant_mxfp8_rows: {rc}")
    return codes, scales


# ------------------------------------------------------------------ dispatch

def dispatch_compact(ids, E: int, num_valid_rows=None) -> dict:
    ids = _np(ids, np.int32)
    T, K = ids.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.full(max(T * K, 1), -1, np.int32)
    route_row = np.zeros(T * K, np.int32) if T * K else np.zeros(1, np.int32)
    nvr = None if num_valid_rows is None else np.array([num_valid_rows], np.int32)
    rc = _load().orc_dispatch_compact(_p(ids) if T else None, T, K, E, _p(nvr), _p(counts), _p(offsets),
                                      _p(perm), _p(route_row))
    if rc:
        raise ValueError(f"orc_dispatch_compact: {rc}")
    R = int(offsets[-1])
    return {"counts": counts, "offsets": offsets, "perm": perm[:R].copy(),
            "route_row": route_row[:T * K].reshape(T, K)}


def dispatch_fixed(ids, E: int, mtpr: int, num_valid_rows=None) -> dict:
    ids = _np(ids, np.int32)
    T, K = ids.shape
    words = (mtpr + 31) // 32
    occ = np.zeros((E, words), np.uint32)
    counts = np.zeros(E, np.int32)
    route_slot = np.zeros(max(T * K, 1), np.int32)
    nvr = None if num_valid_rows is None else np.array([num_valid_rows], np.int32)
    rc = _load().orc_dispatch_fixed(_p(ids) if T else None, T, K, E, _p(nvr), mtpr, _p(occ), _p(counts),
                                    _p(route_slot))
    if rc:
        raise ValueError(f"orc_dispatch_fixed: {rc}")
    return {"occ": occ, "counts": counts, "route_slot": route_slot[:T * K].reshape(T, K)}


# ------------------------------------------------------------------ forward

def w13_rows_concat(w13_rows, layout: str):
    """W13 codes or scales [E, 2I, n] in the concatenated order (gate rows [0,I), up rows [I,2I)).

    layout "interleaved": gate row j is row 2j and up row j is row 2j+1 (the gate-up-interleaved
    experts of the mega_moe reference linked from ROCm/aiter PR #6881; the row-by-row reading is
    ours)."""
    a = _np(w13_rows, np.uint8)
    if layout == "concat":
        return a
    if layout != "interleaved":
        raise ValueError(layout)
    return np.ascontiguousarray(np.concatenate([a[:, 0::2, :], a[:, 1::2, :]], axis=1))


def moe_forward(x_bf16, ids, wts, weights, num_valid_rows=None, swiglu_limit: float = 0.0,
                y_fp32: bool = False, rows=None, nthreads: int = 0, w13_layout: str = "concat",
                y_format: str = None):
    """Returns BF16 bits (uint16) [T or len(rows), H].  y_format: GEMM2 rows handed to the combine as
    "bf16" (default), "fp32" (same as y_fp32=True) or "mxfp8" (1x32 E4M3 + E8M0 along H)."""
    y_mode = {"bf16": 0, "fp32": 1, "mxfp8": 2}[y_format or ("fp32" if y_fp32 else "bf16")]
    w13, w13s, w2, w2s = (_np(a, np.uint8) for a in weights)
    w13, w13s = w13_rows_concat(w13, w13_layout), w13_rows_concat(w13s, w13_layout)
    E, I2, Hh = w13.shape
    H, I = Hh * 2, I2 // 2
    xb = _bf16_bits(x_bf16)
    T = xb.shape[0]
    ids = _np(ids, np.int32)
    ids = ids if ids.ndim == 2 else ids.reshape(T, -1)
    K = ids.shape[1]
    wts = _np(wts, np.float32).reshape(T, K)
    assert xb.shape == (T, H) and w2.shape == (E, H, I // 2)
    assert w13s.shape == (E, 2 * I, H // 32) and w2s.shape == (E, H, I // 32)
    rws = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = T if rws is None else len(rws)
    out = np.zeros((max(n, 1), H), np.uint16)
    nvr = None if num_valid_rows is None else np.array([num_valid_rows], np.int32)
    if T == 0:
        xb = np.zeros((1, H), np.uint16)
        ids = np.zeros((1, K), np.int32)
        wts = np.zeros((1, K), np.float32)
    rc = _load().orc_moe_forward(_p(xb), _p(ids), _p(wts), T, H, I, E, K, _p(nvr), _p(w13), _p(w13s),
                                 _p(w2), _p(w2s), float(swiglu_limit), y_mode, _p(rws), n, _p(out),
                                 int(nthreads))
    if rc:
        raise ValueError(f"orc_moe_forward: {rc}")
    return out[:n]


def route_intermediates(x_row_bf16, e: int, weights, swiglu_limit: float = 0.0) -> dict:
    w13, w13s, w2, w2s = (_np(a, np.uint8) for a in weights)
    E, I2, Hh = w13.shape
    H, I = Hh * 2, I2 // 2
    xb = _bf16_bits(x_row_bf16).reshape(-1)
    g = np.zeros(2 * I, np.float32)
    hq = np.zeros(I, np.uint8)
    hs = np.zeros(I // 32, np.uint8)
    y = np.zeros(H, np.float32)
    rc = _load().orc_route_intermediates(_p(xb), H, I, E, int(e), _p(w13), _p(w13s), _p(w2), _p(w2s),
                                         float(swiglu_limit), _p(g), _p(hq), _p(hs), _p(y))
    if rc:
        raise ValueError(f"orc_route_intermediates: {rc}")
    return {"g": g, "hq": hq, "hs": hs, "y": y}


def topk_softmax(logits, K: int, num_valid_rows=None, renormalize: bool = True) -> dict:
    """Router top-k: logits float32 [T, E] (BF16 logits: pass them widened) -> ids int32 [T, K],
    weights float32 [T, K]."""
    lg = np.ascontiguousarray(_np(logits, np.float32))
    T, E = lg.shape
    ids = np.zeros((max(T, 1), K), np.int32)
    w = np.zeros((max(T, 1), K), np.float32)
    nvr = None if num_valid_rows is None else np.array([num_valid_rows], np.int32)
    if T == 0:
        lg = np.zeros((1, E), np.float32)
    rc = _load().orc_topk_softmax(_p(lg), T, E, K, _p(nvr), int(bool(renormalize)), _p(ids), _p(w))
    if rc:
        raise ValueError(f"orc_topk_softmax: {rc}")
    return {"ids": ids[:T], "weights": w[:T]}


def max_threads() -> int:
    return _load().orc_max_threads()


def bf16_bits_to_float(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)
