"""Host-side checks of the C ABI that need no GPU: the library builds, loads,
exports every function include/blockmoe.h declares, and refuses bad shapes
before touching the device."""

import ctypes

import pytest

import block_scaled_moe_gb300 as bm


@pytest.fixture(scope="module")
def lib():
    from block_scaled_moe_gb300 import _build
    _build.build()
    return bm.load()


def test_every_declared_symbol_is_exported(lib):
    names = bm.exported_symbols_from_header()
    expected = {"moe_create", "moe_bind_weights", "moe_forward", "moe_destroy", "moe_set_option",
                "moe_get_option", "moe_workspace_bytes", "moe_set_workspace", "moe_read_status",
                "moe_last_error", "moe_dispatch_scheme", "moe_debug_copy", "moe_profile_read",
                "moe_last_path", "moe_dispatch_compact_noalloc", "moe_bind_layer", "moe_select_layer", "moe_topk_softmax",
                "moe_set_path_table", "moe_get_path_table", "moe_autotune",
                "moe_forward_routed"}
    assert expected <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_header_constants_parse():
    assert bm.MOE_OK == 0 and bm.MOE_ECAPACITY == -4 and bm.MOE_ST_TIMEOUT == 2
    assert bm.MOE_DISPATCH_COMPACT == 2 and bm.MOE_DBG_TILES == 13


@pytest.mark.parametrize("H,I,E,topk,cap,code", [
    (100, 128, 8, 2, 64, -3),      # H not a multiple of 128
    (256, 96, 8, 2, 64, -3),       # I not a multiple of 128
    (256, 128, 0, 2, 64, -3),      # no experts
    (256, 128, 8, 17, 64, -3),     # top-k above 16
    (256, 128, 8, 2, 0, -1),       # zero capacity
])
def test_create_refuses_bad_shapes_before_cuda(lib, H, I, E, topk, cap, code):
    h = ctypes.c_void_p()
    rc = lib.moe_create(ctypes.byref(h), H, I, E, topk, cap)
    assert rc == code
    assert not h.value
    assert lib.moe_last_error(None)


def test_null_handle_calls_are_refused(lib):
    assert lib.moe_forward(None, None, None, None, None, None, 0, None) == bm.MOE_EINVAL
    assert lib.moe_bind_weights(None, None, None, None, None) == bm.MOE_EINVAL
    assert lib.moe_set_option(None, 1, 0.0) == bm.MOE_EINVAL
    assert lib.moe_workspace_bytes(None) == 0
    lib.moe_destroy(None)


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = lib.moe_create(ctypes.byref(h), 256, 128, 8, 2, 64)
    assert rc in (bm.MOE_ECUDA, bm.MOE_EDEVICE)
    assert not h.value


@pytest.mark.parametrize("dtype,T,E,K", [(7, 4, 8, 2), (0, -1, 8, 2), (0, 4, 0, 1), (0, 4, 4097, 1),
                                         (0, 4, 8, 0), (0, 4, 8, 17), (1, 4, 3, 4), (0, 4, 8, 2)])
def test_topk_softmax_refuses_bad_arguments_before_cuda(lib, dtype, T, E, K):
    """Argument checks run on the host before any CUDA call (the last case: NULL buffers)."""
    import block_scaled_moe_gb300 as bm
    rc = lib.moe_topk_softmax(None, dtype, T, E, K, None, 1, None, None, None)
    assert rc == bm.MOE_EINVAL
    assert bm.moe_last_error(None)


def test_topk_softmax_empty_batch_is_a_no_op(lib):
    import block_scaled_moe_gb300 as bm
    assert lib.moe_topk_softmax(None, bm.MOE_DTYPE_BF16, 0, 384, 6, None, 1, None, None, None) == bm.MOE_OK


def test_bounds_checking_build_builds_and_exports_everything():
    """libblockmoe_bounds.so (-DMOE_DEBUG_BOUNDS) compiles and exports the same functions; an
    unknown build variant is refused."""
    from block_scaled_moe_gb300 import _build
    path = _build.build(variant="bounds")
    assert path.endswith("libblockmoe_bounds.so")
    blib = ctypes.CDLL(path)
    for n in bm.exported_symbols_from_header():
        assert hasattr(blib, n), n
    with pytest.raises(ValueError):
        _build.build(variant="asan")
    assert bm.MOE_ST_BOUNDS == 8 and bm.MOE_DBG_BOUNDS == 16 and bm.MOE_OPT_BOUNDS_BUILD == 16


def test_variant_switch_loads_the_bounds_library():
    """BMOE_LIB_VARIANT=bounds makes the binding load libblockmoe_bounds.so (checked in a child
    process, since the parent already holds the normal library)."""
    import os
    import subprocess
    import sys
    from block_scaled_moe_gb300 import _build
    _build.build(variant="bounds")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import block_scaled_moe_gb300 as bm, os; lib = bm.load(); "
            "print(os.path.basename(lib._name))")
    env = dict(os.environ, BMOE_LIB_VARIANT="bounds")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "libblockmoe_bounds.so"


def test_every_option_and_debug_region_is_handled():
    """Each MOE_OPT_* key and MOE_DBG_* region the header defines has a case in the library's option
    and debug-copy switches (the header and the implementation do not drift apart)."""
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = open(os.path.join(root, "block_scaled_moe_gb300", "csrc", "moe_api.cu")).read()
    cases = set(re.findall(r"case\s+(MOE_(?:OPT|DBG)_\w+)\s*:", src))
    keys = [k for k in bm.C if k.startswith("MOE_OPT_") or k.startswith("MOE_DBG_")]
    assert keys
    missing = [k for k in keys if k not in cases]
    assert not missing, missing


def test_unknown_variant_is_refused():
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, BMOE_LIB_VARIANT="../../elsewhere")
    r = subprocess.run([sys.executable, "-c", "import block_scaled_moe_gb300 as bm; bm.load()"], cwd=root, env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "not a build variant" in r.stderr
