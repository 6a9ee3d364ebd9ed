"""Python binding of libblockmoe.so, the fused block-scaled MoE layer for GB300 (sm_103a).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C ABI's names (include/blockmoe.h); the
`BlockScaledMoE` class wraps a handle for torch tensors (torch provides device
memory and streams).  Importing the package does not need a GPU; loading the
library raises if it has not been built, and there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
# BMOE_LIB_VARIANT=bounds loads the bounds-checking build (libblockmoe_bounds.so) instead, =trace the
# tracing build (libblockmoe_trace.so); other values are refused at load time
LIB_VARIANTS = ("", "bounds", "trace")
LIB_VARIANT = os.environ.get("BMOE_LIB_VARIANT", "")
LIB_PATH = os.path.join(PKG, "lib", f"libblockmoe_{LIB_VARIANT}.so" if LIB_VARIANT else "libblockmoe.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "blockmoe.h")

_lock = threading.Lock()
_lib = None


def _header_constants() -> dict:
    out = {}
    with open(HEADER) as f:
        for m in re.finditer(r"#define\s+(MOE_\w+)\s+\(?(-?(?:0x)?[0-9a-fA-F]+)u?\)?", f.read()):
            out[m.group(1)] = int(m.group(2), 0)
    return out


C = _header_constants()
globals().update(C)


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def load(path: Optional[str] = None):
    """Load libblockmoe.so (built in-tree by `__graft_entry__.build()`)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if path is None and LIB_VARIANT not in LIB_VARIANTS:
            raise ImportError(f"BMOE_LIB_VARIANT={LIB_VARIANT!r} is not a build variant; known: {LIB_VARIANTS}")
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{os.path.basename(p)} is not built ({p}); run __graft_entry__.build()"
                              + (f" or _build.build(variant={LIB_VARIANT!r})" if LIB_VARIANT else ""))
        lib = ctypes.CDLL(p)
        vp, i32, f64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
        lib.moe_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32]
        lib.moe_create.restype = i32
        lib.moe_bind_weights.argtypes = [vp, vp, vp, vp, vp]
        lib.moe_bind_weights.restype = i32
        lib.moe_forward.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp]
        lib.moe_forward.restype = i32
        lib.moe_destroy.argtypes = [vp]
        lib.moe_destroy.restype = None
        lib.moe_set_option.argtypes = [vp, i32, f64]
        lib.moe_set_option.restype = i32
        lib.moe_get_option.argtypes = [vp, i32, ctypes.POINTER(f64)]
        lib.moe_get_option.restype = i32
        lib.moe_workspace_bytes.argtypes = [vp]
        lib.moe_workspace_bytes.restype = sz
        lib.moe_set_workspace.argtypes = [vp, vp, sz]
        lib.moe_set_workspace.restype = i32
        lib.moe_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        lib.moe_read_status.restype = i32
        lib.moe_last_error.argtypes = [vp]
        lib.moe_last_error.restype = ctypes.c_char_p
        lib.moe_dispatch_scheme.argtypes = [vp]
        lib.moe_dispatch_scheme.restype = i32
        lib.moe_debug_copy.argtypes = [vp, i32, vp, ctypes.POINTER(sz), vp]
        lib.moe_debug_copy.restype = i32
        lib.moe_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), i32]
        lib.moe_profile_read.restype = i32
        lib.moe_last_path.argtypes = [vp]
        lib.moe_last_path.restype = i32
        lib.moe_bind_layer.argtypes = [vp, i32, vp, vp, vp, vp]
        lib.moe_bind_layer.restype = i32
        lib.moe_select_layer.argtypes = [vp, i32]
        lib.moe_select_layer.restype = i32
        lib.moe_topk_softmax.argtypes = [vp, i32, i32, i32, i32, vp, i32, vp, vp, vp]
        lib.moe_topk_softmax.restype = i32
        lib.moe_forward_routed.argtypes = [vp, vp, vp, i32, i32, vp, vp, i32, vp]
        lib.moe_forward_routed.restype = i32
        lib.moe_dispatch_compact_noalloc.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.moe_dispatch_compact_noalloc.restype = i32
        lib.moe_set_path_table.argtypes = [vp, vp, vp, i32]
        lib.moe_set_path_table.restype = i32
        lib.moe_get_path_table.argtypes = [vp, vp, vp, i32]
        lib.moe_get_path_table.restype = i32
        lib.moe_autotune.argtypes = [vp, vp, i32, i32, vp]
        lib.moe_autotune.restype = i32
        _lib = lib
        return lib


def exported_symbols_from_header() -> list:
    """Names of the functions include/blockmoe.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"^\s*(?:int|void|size_t|const char\*)\s+(moe_\w+)\s*\(", text, flags=re.M)


# ---------------------------------------------------------------- C ABI names

def _check(h, rc: int):
    if rc != 0:
        msg = load().moe_last_error(h)
        raise MoeError(rc, msg.decode() if msg else "")


def moe_create(H: int, I: int, E: int, topk: int, capacity: int):
    lib = load()
    h = ctypes.c_void_p()
    rc = lib.moe_create(ctypes.byref(h), H, I, E, topk, capacity)
    _check(None, rc)
    return h


def moe_bind_weights(h, w13_fp4: int, w13_sf: int, w2_fp4: int, w2_sf: int):
    _check(h, load().moe_bind_weights(h, w13_fp4, w13_sf, w2_fp4, w2_sf))


def moe_bind_layer(h, slot: int, w13_fp4: int, w13_sf: int, w2_fp4: int, w2_sf: int):
    _check(h, load().moe_bind_layer(h, slot, w13_fp4, w13_sf, w2_fp4, w2_sf))


def moe_select_layer(h, slot: int):
    _check(h, load().moe_select_layer(h, slot))


def moe_forward(h, x: int, topk_ids: int, topk_weights: int, num_valid_rows: Optional[int], out: int, T: int,
                stream: int = 0):
    _check(h, load().moe_forward(h, x, topk_ids, topk_weights, num_valid_rows, out, T, stream))


def moe_topk_softmax(logits: int, logits_dtype: int, T: int, E: int, topk: int, num_valid_rows: Optional[int],
                     renormalize: bool, topk_ids: int, topk_weights: int, stream: int = 0):
    _check(None, load().moe_topk_softmax(logits, logits_dtype, T, E, topk, num_valid_rows, int(bool(renormalize)),
                                         topk_ids, topk_weights, stream))


def moe_forward_routed(h, x: int, router_logits: int, logits_dtype: int, renormalize: bool,
                       num_valid_rows: Optional[int], out: int, T: int, stream: int = 0):
    _check(h, load().moe_forward_routed(h, x, router_logits, logits_dtype, int(bool(renormalize)), num_valid_rows,
                                        out, T, stream))


def _logits_dtype(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return MOE_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return MOE_DTYPE_BF16
    raise ValueError(f"router logits must be float32 or bfloat16, not {t.dtype}")


def topk_softmax(router_logits, topk: int, num_valid_rows=None, renormalize: bool = True, stream=None):
    """Router top-k with softmax weights on the GPU: logits [T, E] -> (ids int32 [T, topk], weights float32)."""
    import torch
    if not (isinstance(router_logits, torch.Tensor) and router_logits.is_cuda and router_logits.is_contiguous()
            and router_logits.dim() == 2):
        raise ValueError("router_logits must be a contiguous 2-D CUDA tensor")
    T, E = router_logits.shape
    dev = router_logits.device
    ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
    w = torch.empty((T, topk), dtype=torch.float32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    moe_topk_softmax(router_logits.data_ptr(), _logits_dtype(router_logits), T, E, topk,
                     None if num_valid_rows is None else num_valid_rows.data_ptr(), renormalize, ids.data_ptr(),
                     w.data_ptr(), s.cuda_stream)
    return ids, w


def _i32_array(vals):
    arr = (ctypes.c_int32 * max(1, len(vals)))(*[int(v) for v in vals])
    return arr


def moe_set_path_table(h, t: list, path: list):
    if len(t) != len(path):
        raise ValueError("t and path must have the same length")
    ta, pa = _i32_array(t), _i32_array(path)
    _check(h, load().moe_set_path_table(h, ctypes.cast(ta, ctypes.c_void_p), ctypes.cast(pa, ctypes.c_void_p), len(t)))


def moe_get_path_table(h) -> tuple:
    lib = load()
    n = lib.moe_get_path_table(h, None, None, 0)
    if n < 0:
        _check(h, n)
    ta, pa = _i32_array([0] * n), _i32_array([0] * n)
    lib.moe_get_path_table(h, ctypes.cast(ta, ctypes.c_void_p), ctypes.cast(pa, ctypes.c_void_p), n)
    return list(ta)[:n], list(pa)[:n]


def moe_autotune(h, t_buckets: list, reps: int = 5, stream: int = 0):
    ta = _i32_array(t_buckets)
    _check(h, load().moe_autotune(h, ctypes.cast(ta, ctypes.c_void_p), len(t_buckets), reps, stream))


def moe_destroy(h):
    load().moe_destroy(h)


def moe_set_option(h, key: int, value: float):
    _check(h, load().moe_set_option(h, key, float(value)))


def moe_get_option(h, key: int) -> float:
    v = ctypes.c_double()
    _check(h, load().moe_get_option(h, key, ctypes.byref(v)))
    return v.value


def moe_workspace_bytes(h) -> int:
    return load().moe_workspace_bytes(h)


def moe_set_workspace(h, ptr: int, nbytes: int):
    _check(h, load().moe_set_workspace(h, ptr, nbytes))


def moe_read_status(h, stream: int = 0) -> int:
    v = ctypes.c_uint32()
    _check(h, load().moe_read_status(h, ctypes.byref(v), stream))
    return v.value


def moe_last_error(h=None) -> str:
    m = load().moe_last_error(h)
    return m.decode() if m else ""


def moe_dispatch_scheme(h) -> int:
    return load().moe_dispatch_scheme(h)


def moe_profile_read(h) -> list:
    ms = (ctypes.c_float * 5)()
    _check(h, load().moe_profile_read(h, ms, 5))
    return list(ms)


def moe_dispatch_compact_noalloc(topk_ids: int, T: int, topk: int, E: int, num_valid_rows: Optional[int],
                                 counts: int, offsets: int, perm: int, route_row: int, stream: int = 0):
    """Compact dispatch without any device allocation (raw device pointers)."""
    _check(None, load().moe_dispatch_compact_noalloc(topk_ids, T, topk, E, num_valid_rows, counts, offsets, perm,
                                                     route_row, stream))


def moe_debug_copy(h, which: int, stream: int = 0) -> bytes:
    lib = load()
    n = ctypes.c_size_t(0)
    _check(h, lib.moe_debug_copy(h, which, None, ctypes.byref(n), stream))
    buf = ctypes.create_string_buffer(max(n.value, 1))
    _check(h, lib.moe_debug_copy(h, which, buf, ctypes.byref(n), stream))
    return buf.raw[: n.value]


# ---------------------------------------------------------------- torch wrapper

class BlockScaledMoE:
    """One layer instance: torch tensors in, torch tensors out (CUDA, contiguous)."""

    def __init__(self, H: int, I: int, E: int, topk: int, capacity: int, *, dispatch: Optional[str] = None,
                 swiglu_limit: float = 0.0, route_tile: int = 0, debug: bool = False,
                 fixed_slot_max: Optional[int] = None, workspace=None, path: Optional[str] = None,
                 w13_layout: str = "concat", layer_slots: int = 1, y_format: str = "bf16"):
        self.H, self.I, self.E, self.topk, self.capacity = H, I, E, topk, capacity
        self.h = moe_create(H, I, E, topk, capacity)
        try:
            if fixed_slot_max is not None:
                moe_set_option(self.h, MOE_OPT_FIXED_SLOT_MAX, fixed_slot_max)
            if dispatch is not None:
                moe_set_option(self.h, MOE_OPT_DISPATCH,
                               {"auto": MOE_DISPATCH_AUTO, "fixed": MOE_DISPATCH_FIXED,
                                "compact": MOE_DISPATCH_COMPACT}[dispatch])
            if route_tile:
                moe_set_option(self.h, MOE_OPT_ROUTE_TILE, route_tile)
            if debug:
                moe_set_option(self.h, MOE_OPT_DEBUG_CAPTURE, 1)
            moe_set_option(self.h, MOE_OPT_SWIGLU_LIMIT, swiglu_limit)
            moe_set_option(self.h, MOE_OPT_W13_LAYOUT,
                           {"concat": MOE_W13_CONCAT, "interleaved": MOE_W13_INTERLEAVED}[w13_layout])
            if layer_slots != 1:
                moe_set_option(self.h, MOE_OPT_LAYER_SLOTS, layer_slots)
            moe_set_option(self.h, MOE_OPT_Y_FORMAT, {"bf16": MOE_Y_BF16, "mxfp8": MOE_Y_MXFP8}[y_format])
            if path is not None:
                moe_set_option(self.h, MOE_OPT_PATH, {"auto": MOE_PATH_AUTO, "fused": MOE_PATH_FUSED,
                                                      "multi": MOE_PATH_MULTI}[path])
            if workspace is not None:
                moe_set_workspace(self.h, workspace.data_ptr(), workspace.numel() * workspace.element_size())
        except Exception:
            moe_destroy(self.h)
            self.h = None
            raise
        self._weights = {}

    def close(self):
        if getattr(self, "h", None) is not None:
            moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def scheme(self) -> str:
        return "fixed" if moe_dispatch_scheme(self.h) == MOE_DISPATCH_FIXED else "compact"

    @property
    def workspace_bytes(self) -> int:
        return moe_workspace_bytes(self.h)

    @property
    def last_path(self) -> str:
        return {MOE_PATH_FUSED: "fused", MOE_PATH_MULTI: "multi"}.get(load().moe_last_path(self.h), "none")

    def autotune(self, t_buckets, reps: int = 5, stream=None) -> dict:
        """Measure the paths for each bucket T on synthetic inputs; returns {T: "fused" | "multi"}."""
        import torch
        s = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        moe_autotune(self.h, list(t_buckets), reps, s)
        return self.path_table

    @property
    def path_table(self) -> dict:
        t, p = moe_get_path_table(self.h)
        return {ti: {MOE_PATH_FUSED: "fused", MOE_PATH_MULTI: "multi"}[pi] for ti, pi in zip(t, p)}

    def set_path_table(self, table: dict):
        """Replace the T-bucketed path table ({T: "fused" | "multi"}; empty dict clears it)."""
        items = sorted(table.items())
        code = {"fused": MOE_PATH_FUSED, "multi": MOE_PATH_MULTI}
        moe_set_path_table(self.h, [t for t, _ in items], [code[p] for _, p in items])

    @property
    def launches(self) -> int:
        return int(moe_get_option(self.h, MOE_OPT_LAUNCHES))

    def set_profile(self, on: bool = True):
        moe_set_option(self.h, MOE_OPT_PROFILE, 1 if on else 0)

    def profile_ms(self) -> list:
        """[dispatch, quant, GEMM1, GEMM2, combine] ms of the last profiled forward."""
        return moe_profile_read(self.h)

    def _dev(self, t, name, shape, dtypes):
        import torch
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (strided views are refused, not copied)")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
        if t.dtype not in dtypes:
            raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
        return t.data_ptr()

    def _weight_ptrs(self, w13, w13_sf, w2, w2_sf):
        import torch
        E, H, I = self.E, self.H, self.I
        fp4 = (torch.uint8,) + ((torch.float4_e2m1fn_x2,) if hasattr(torch, "float4_e2m1fn_x2") else ())
        sf = (torch.uint8,) + ((torch.float8_e8m0fnu,) if hasattr(torch, "float8_e8m0fnu") else ())
        return (self._dev(w13, "w13", (E, 2 * I, H // 2), fp4), self._dev(w13_sf, "w13_sf", (E, 2 * I, H // 32), sf),
                self._dev(w2, "w2", (E, H, I // 2), fp4), self._dev(w2_sf, "w2_sf", (E, H, I // 32), sf))

    @property
    def layer(self) -> int:
        return int(moe_get_option(self.h, MOE_OPT_LAYER))

    def set_w13_layout(self, layout: str):
        """Row order assumed by the next bind: "concat" or "interleaved"."""
        moe_set_option(self.h, MOE_OPT_W13_LAYOUT, {"concat": MOE_W13_CONCAT, "interleaved": MOE_W13_INTERLEAVED}[layout])

    def bind_weights(self, w13, w13_sf, w2, w2_sf):
        ptrs = self._weight_ptrs(w13, w13_sf, w2, w2_sf)
        moe_bind_weights(self.h, *ptrs)
        self._weights[self.layer] = (w13, w13_sf, w2, w2_sf)  # keep caller tensors alive while bound

    def bind_layer(self, slot: int, w13, w13_sf, w2, w2_sf):
        ptrs = self._weight_ptrs(w13, w13_sf, w2, w2_sf)
        moe_bind_layer(self.h, slot, *ptrs)
        self._weights[slot] = (w13, w13_sf, w2, w2_sf)

    def select_layer(self, slot: int):
        moe_select_layer(self.h, slot)

    def forward(self, x, topk_ids, topk_weights, num_valid_rows=None, out=None, stream=None):
        import torch
        T = x.shape[0]
        xp = self._dev(x, "x", (T, self.H), (torch.bfloat16,))
        ip = self._dev(topk_ids, "topk_ids", (T, self.topk), (torch.int32,))
        wp = self._dev(topk_weights, "topk_weights", (T, self.topk), (torch.float32,))
        nvr = None
        if num_valid_rows is not None:
            if not (isinstance(num_valid_rows, torch.Tensor) and num_valid_rows.is_cuda
                    and num_valid_rows.dtype == torch.int32 and num_valid_rows.numel() >= 1):
                raise ValueError("num_valid_rows must be a CUDA int32 tensor (its first element is read)")
            nvr = num_valid_rows.data_ptr()
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        op = self._dev(out, "out", (T, self.H), (torch.bfloat16,))
        s = (stream if stream is not None else torch.cuda.current_stream(x.device)).cuda_stream
        moe_forward(self.h, xp, ip, wp, nvr, op, T, s)
        return out

    __call__ = forward

    def forward_routed(self, x, router_logits, num_valid_rows=None, out=None, stream=None, renormalize=True):
        """Router top-k from `router_logits` [T, E] (float32 or bf16), then the layer."""
        import torch
        T = x.shape[0]
        self._dev(x, "x", (T, self.H), (torch.bfloat16,))
        self._dev(router_logits, "router_logits", (T, self.E), (torch.float32, torch.bfloat16))
        if num_valid_rows is not None:
            self._dev(num_valid_rows, "num_valid_rows", (1,), (torch.int32,))
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        else:
            self._dev(out, "out", (T, self.H), (torch.bfloat16,))
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        moe_forward_routed(self.h, x.data_ptr(), router_logits.data_ptr(), _logits_dtype(router_logits), renormalize,
                           None if num_valid_rows is None else num_valid_rows.data_ptr(), out.data_ptr(), T,
                           s.cuda_stream)
        return out

    def read_status(self, stream=None) -> int:
        import torch
        s = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        return moe_read_status(self.h, s)

    def debug_array(self, which: str):
        import numpy as np
        import torch
        ids = {"counts": (MOE_DBG_COUNTS, np.int32), "offsets": (MOE_DBG_OFFSETS, np.int32),
               "perm": (MOE_DBG_PERM, np.int32), "route_row": (MOE_DBG_ROUTE_ROW, np.int32),
               "route_slot": (MOE_DBG_ROUTE_SLOT, np.int32), "occ": (MOE_DBG_OCC, np.uint32),
               "xq": (MOE_DBG_XQ, np.uint8), "xs": (MOE_DBG_XS, np.uint8), "yrow": (MOE_DBG_YROW, np.int32),
               "hq": (MOE_DBG_HQ, np.uint8), "g": (MOE_DBG_G, np.float32), "y": (MOE_DBG_Y, np.uint16),
               "tiles": (MOE_DBG_TILES, np.int32), "topk_ids": (MOE_DBG_TOPK_IDS, np.int32),
               "topk_weights": (MOE_DBG_TOPK_WEIGHTS, np.float32), "bounds": (MOE_DBG_BOUNDS, np.uint32)}
        code, dt = ids[which]
        raw = moe_debug_copy(self.h, code, torch.cuda.current_stream().cuda_stream)
        return np.frombuffer(raw, dtype=dt).copy()
