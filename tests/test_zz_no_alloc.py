"""The allocation-free compact dispatch, checked against the oracle's dispatch and
against moe_forward's own.

Some callers may not allocate device memory at all (code running during CUDA
graph capture, engines that reserve the whole GPU up front), so the library
offers moe_dispatch_compact_noalloc, which keeps its scratch in an array built
into the library.  This file runs last so that a failure here comes after every
other test has run; it also passes on its own in a fresh process.
"""

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    torch.cuda.set_device(0)


def _forward_dispatch(ids: np.ndarray, E: int, nvr: int):
    """Dispatch arrays as moe_forward computes them (compact scheme, zero weights)."""
    import block_scaled_moe_gb300 as bm
    T, K = ids.shape
    H = I = 128
    L = bm.BlockScaledMoE(H, I, E, K, T, dispatch="compact")
    Wz = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in
          [(E, 2 * I, H // 2), (E, 2 * I, H // 32), (E, H, I // 2), (E, H, I // 32)]]
    L.bind_weights(*Wz)
    L.forward(torch.zeros((T, H), dtype=torch.bfloat16, device="cuda"), torch.from_numpy(ids).cuda(),
              torch.ones((T, K), dtype=torch.float32, device="cuda"),
              torch.tensor([nvr], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    out = {k: L.debug_array(k) for k in ("counts", "offsets", "perm", "route_row")}
    L.close()
    return out


def _noalloc_dispatch(ids: np.ndarray, E: int, nvr):
    import block_scaled_moe_gb300 as bm
    T, K = ids.shape
    dev = torch.device("cuda")
    ids_d = torch.from_numpy(ids).to(dev)
    nvr_d = None if nvr is None else torch.tensor([nvr], dtype=torch.int32, device=dev)
    # sentinel-filled outputs: everything the call must produce gets overwritten
    counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    perm = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
    route_row = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    bm.moe_dispatch_compact_noalloc(ids_d.data_ptr() if T else 0, T, K, E,
                                    None if nvr_d is None else nvr_d.data_ptr(), counts.data_ptr(),
                                    offsets.data_ptr(), perm.data_ptr() if T else 0,
                                    route_row.data_ptr() if T else 0, stream)
    torch.cuda.synchronize()
    return {"counts": counts.cpu().numpy(), "offsets": offsets.cpu().numpy(), "perm": perm.cpu().numpy(),
            "route_row": route_row.cpu().numpy()}


def _same(a, b):
    R = int(b["offsets"][-1])
    assert np.array_equal(a["counts"], b["counts"])
    assert np.array_equal(a["offsets"], b["offsets"])
    assert np.array_equal(a["perm"][:R], b["perm"][:R])
    assert np.array_equal(np.asarray(a["route_row"]).reshape(-1), np.asarray(b["route_row"]).reshape(-1))


def _oracle(ids: np.ndarray, E: int, nvr):
    import oracle
    oracle.build()
    return oracle.dispatch_compact(ids, E, nvr)


def test_noalloc_dispatch_matches_forward_two_calls_in_a_row():
    # call 1: skewed small-M routing (T=512, E=384, 5% invalid slots, 480 valid rows)
    w1 = synth.get("smallm_pro")
    ids1, _ = synth.make_routing(w1)
    a1 = _noalloc_dispatch(ids1, w1.E, w1.nvr)
    # call 2 right after, on other sizes (T=64, E=8): the shared scratch keeps call 1's contents
    w2 = synth.get("tiny")
    ids2, _ = synth.make_routing(w2)
    a2 = _noalloc_dispatch(ids2, w2.E, w2.nvr)
    _same(a1, _oracle(ids1, w1.E, w1.nvr))
    _same(a2, _oracle(ids2, w2.E, w2.nvr))
    _same(a1, _forward_dispatch(ids1, w1.E, w1.nvr))
    _same(a2, _forward_dispatch(ids2, w2.E, w2.nvr))
    # and once more on the first input: identical to its first result
    _same(_noalloc_dispatch(ids1, w1.E, w1.nvr), a1)


def test_noalloc_dispatch_refuses_sizes_beyond_its_scratch():
    import block_scaled_moe_gb300 as bm
    T, K, E = 8192 * 4, 8, 4096          # about 2.1M chunk counters: far above the 1 MiB array
    with pytest.raises(bm.MoeError) as ei:
        bm.moe_dispatch_compact_noalloc(0, T, K, E, None, 1, 1, 1, 1, 0)
    assert ei.value.code == bm.MOE_ECAPACITY
    assert "scratch" in bm.moe_last_error(None)


def test_noalloc_dispatch_empty_null_count_and_many_experts():
    # T = 0: zero counts and offsets, nothing else touched
    a0 = _noalloc_dispatch(np.zeros((0, 6), np.int32), 384, None)
    assert not a0["counts"].any() and not a0["offsets"].any()
    # no row count: every row is valid, as with num_valid_rows = T
    rng = np.random.default_rng(7)
    ids = rng.integers(-1, 40, size=(300, 4)).astype(np.int32)
    _same(_noalloc_dispatch(ids, 40, None), _oracle(ids, 40, None))
    _same(_noalloc_dispatch(ids, 40, None), _noalloc_dispatch(ids, 40, 300))
    # E = 4096, the largest the library accepts (the count kernel then needs 64 KB of shared memory)
    ids = rng.integers(-1, 4096, size=(200, 8)).astype(np.int32)
    _same(_noalloc_dispatch(ids, 4096, 150), _oracle(ids, 4096, 150))
