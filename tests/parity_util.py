"""Helpers shared by the GPU parity tests: run the CUDA layer and the oracle on
the same seeded inputs and compare with the stated tolerances."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Output tolerance (applied to BF16 outputs as float64):
#   relative L2 error <= 1e-2, and elementwise |d| <= 0.08*|ref| + 1e-2*rms(ref).
REL_L2 = 1e-2
ELEM_REL = 0.08
ELEM_RMS = 1e-2


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_float(bits).astype(np.float64)


def torch_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def compare(got_bits: np.ndarray, ref_bits: np.ndarray) -> dict:
    g = bits_to_f64(got_bits)
    r = bits_to_f64(ref_bits)
    d = np.abs(g - r)
    nr = np.linalg.norm(r)
    rel = float(np.linalg.norm(g - r) / nr) if nr > 0 else float(np.linalg.norm(g))
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    bound = ELEM_REL * np.abs(r) + ELEM_RMS * rms
    bad = int(np.count_nonzero(d > bound))
    return {"rel_l2": rel, "bad": bad, "max_abs": float(d.max()) if d.size else 0.0, "rms": rms,
            "nan": int(np.count_nonzero(~np.isfinite(g)))}


def assert_close(got_bits, ref_bits, what=""):
    c = compare(got_bits, ref_bits)
    assert c["nan"] == 0, (what, c)
    assert c["rel_l2"] <= REL_L2, (what, c)
    assert c["bad"] == 0, (what, c)
    return c


class Case:
    """Inputs of one workload on the host (for the oracle) and on the device."""

    def __init__(self, w: synth.Workload, device="cuda", weights_on_device=False, w13_gain=1.0):
        self.w = w
        self.x = synth.make_x(w)
        self.ids, self.wts = synth.make_routing(w)
        wdev = device if weights_on_device else "cpu"
        W = synth.make_weights(w, wdev, w13_gain=w13_gain)
        self.Wd = [t.to(device) for t in W]
        self.Wh = [t.cpu() for t in W]
        self.xd = self.x.to(device)
        self.idsd = torch.from_numpy(self.ids).to(device)
        self.wtsd = torch.from_numpy(self.wts).to(device)
        self.nvrd = torch.tensor([w.nvr], dtype=torch.int32, device=device)

    def layer(self, **kw):
        import block_scaled_moe_gb300 as bm
        w = self.w
        opts = dict(dispatch=w.dispatch, swiglu_limit=w.swiglu_limit)
        opts.update(kw)
        L = bm.BlockScaledMoE(w.H, w.I, w.E, w.K, w.capacity, **opts)
        L.bind_weights(*self.Wd)
        return L

    def run(self, L, nvr=True, out=None, stream=None):
        return L.forward(self.xd, self.idsd, self.wtsd, self.nvrd if nvr else None, out=out, stream=stream)

    def oracle(self, rows=None, nvr=True, nthreads=0):
        return oracle.moe_forward(self.x, self.ids, self.wts, self.Wh, num_valid_rows=self.w.nvr if nvr else None,
                                  swiglu_limit=self.w.swiglu_limit, rows=rows, nthreads=nthreads)


def cover_rows(ids: np.ndarray, E: int, nvr: int, route_tile: int, dispatch: str, extra: int = 0, seed: int = 0):
    """Rows to compare at full size, chosen so that every active expert's first and last route tile
    (the ragged one) holds at least one compared route: a greedy cover over the (expert, tile) pairs,
    plus `extra` rows drawn at random.  A route's tile is its rank among the expert's packed rows
    (compact: flat slot order t*K+k; fixed: one row per distinct token, tokens ascending) over the
    route tile width."""
    T, K = ids.shape
    nvr = max(0, min(T, int(nvr)))
    tile_of = {}        # (t, k) -> (e, j)
    last = {}
    seen = {}
    for t in range(nvr):
        for k in range(K):
            e = int(ids[t, k])
            if e < 0 or e >= E:
                continue
            if dispatch == "fixed":
                key = (e, t)
                if key not in seen:
                    seen[key] = last.get(e, -1) + 1
                    last[e] = seen[key]
                rank = seen[key]
            else:
                rank = last.get(e, -1) + 1
                last[e] = rank
            tile_of[(t, k)] = (e, rank // route_tile)
    need = set()
    for e, r in last.items():
        need.add((e, 0))
        need.add((e, r // route_tile))
    covers = {}
    for (t, k), ej in tile_of.items():
        if ej in need:
            covers.setdefault(t, set()).add(ej)
    chosen = []
    while need:
        t = max(covers, key=lambda r: (len(covers[r] & need), -r))
        got = covers[t] & need
        assert got, "uncoverable tile"
        chosen.append(t)
        need -= got
    rng = np.random.default_rng(seed)
    pool = np.setdiff1d(np.arange(nvr), chosen)
    if extra and pool.size:
        chosen += list(rng.choice(pool, size=min(extra, pool.size), replace=False))
    return np.sort(np.array(chosen, dtype=np.int64))
