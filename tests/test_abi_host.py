"""The C-ABI library loads, exports every symbol include/moe.h declares, and
its host-only calls (create, options, workspace sizing) behave; no GPU."""
import ctypes

import pytest

import persistent_megakernel_sm_gb300 as pkg
from persistent_megakernel_sm_gb300 import build as cuda_build


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return pkg.load_library()


def test_header_declares_the_boundary():
    names = pkg.header_symbols()
    for must in ("moe_layer_create", "moe_layer_reserve", "moe_layer_forward",
                 "moe_layer_destroy", "moe_layer_status", "moe_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in pkg.header_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


@pytest.mark.parametrize("args,ok", [
    ((4096, 14336, 8, 2, 0), True),
    ((7168, 2048, 256, 8, 1), True),
    ((100, 512, 8, 2, 0), False),     # d not a multiple of 128
    ((256, 200, 8, 2, 0), False),     # f not a multiple of 128
    ((256, 512, 8, 9, 0), False),     # k > E
    ((256, 512, 300, 2, 0), False),   # E > 256
    ((256, 512, 64, 17, 0), False),   # k > 16
    ((256, 512, 8, 2, 2), False),     # two shared experts
    ((32768, 512, 8, 2, 0), True),    # the largest d: a 64 KB row fits a gather round
    ((32896, 512, 8, 2, 0), False),   # d > 32768: a row could overrun the gather's stages
])
def test_create_validates(lib, args, ok):
    h = lib.moe_layer_create(*args)
    if ok:
        assert h
        lib.moe_layer_destroy(h)
    else:
        assert not h
        assert lib.moe_last_error()


def test_options_and_workspace_without_device(lib):
    h = lib.moe_layer_create(4096, 14336, 8, 2, 0)
    try:
        assert lib.moe_layer_set_option(h, pkg.OPTIONS["mode"], 1) == 0
        assert lib.moe_layer_set_option(h, pkg.OPTIONS["mode"], 7) == pkg.MOE_E_INVAL
        assert lib.moe_layer_set_option(h, pkg.OPTIONS["split_k"], 3) == pkg.MOE_E_INVAL
        assert lib.moe_layer_set_option(h, pkg.OPTIONS["tokens_per_tile"], 48) == 0
        assert lib.moe_layer_set_option(h, pkg.OPTIONS["tokens_per_tile"], 50) == pkg.MOE_E_INVAL
        assert lib.moe_layer_set_option(h, 999, 1) == pkg.MOE_E_INVAL
        # forward before reserve is a state error, not a crash
        rc = lib.moe_layer_forward(h, 1, 16, 16, 16, 16, 16, 16, None)
        assert rc == pkg.MOE_E_STATE
        small = lib.moe_layer_workspace_bytes(h, 256)
        big = lib.moe_layer_workspace_bytes(h, 4096)
        # the permuted activations alone are T*k*d*2 bytes
        assert small >= 256 * 2 * 4096 * 2 and big > small
        assert lib.moe_layer_get_stat(h, pkg.STATS["tasks"]) == -1
    finally:
        lib.moe_layer_destroy(h)
    lib.moe_layer_destroy(None)


def test_new_options_validate_without_device(lib):
    h = lib.moe_layer_create(2048, 768, 128, 8, 0)
    try:
        opt = pkg.OPTIONS
        assert lib.moe_layer_set_option(h, opt["mode"], pkg.MOE_MODE_STATIC) == 0
        assert lib.moe_layer_set_option(h, opt["bands"], 0) == 0
        assert lib.moe_layer_set_option(h, opt["bands"], 1) == 0
        assert lib.moe_layer_set_option(h, opt["route_splits"], 8) == 0
        assert lib.moe_layer_set_option(h, opt["route_splits"], 9) == pkg.MOE_E_INVAL
        assert lib.moe_layer_set_option(h, opt["l2_prefetch"], -1) == 0
        assert lib.moe_layer_set_option(h, opt["l2_prefetch"], -2) == pkg.MOE_E_INVAL
        assert lib.moe_layer_set_option(h, opt["release"], 2) == pkg.MOE_E_INVAL
        for v in (0, 64, 128):
            assert lib.moe_layer_set_option(h, opt["route_tokens"], v) == 0
        assert lib.moe_layer_set_option(h, opt["route_tokens"], 96) == pkg.MOE_E_INVAL
    finally:
        lib.moe_layer_destroy(h)


def test_worker_width_split_and_fault_options_validate_without_device(lib):
    h = lib.moe_layer_create(2048, 768, 128, 8, 0)
    try:
        opt = pkg.OPTIONS
        for v in (0, 1, 2):
            assert lib.moe_layer_set_option(h, opt["pair"], v) == 0
        for v in (-1, 3, 4):
            assert lib.moe_layer_set_option(h, opt["pair"], v) == pkg.MOE_E_INVAL
        for v in (-1, 0, 1):
            assert lib.moe_layer_set_option(h, opt["front_split"], v) == 0
        assert lib.moe_layer_set_option(h, opt["front_split"], 2) == pkg.MOE_E_INVAL
        for v in (0, 2, 3, 4):
            assert lib.moe_layer_set_option(h, opt["fault_drop_type"], v) == 0
        for v in (1, 5, -1):  # router tiles and combines feed no counter
            assert lib.moe_layer_set_option(h, opt["fault_drop_type"], v) == pkg.MOE_E_INVAL
        assert lib.moe_layer_set_option(h, opt["fault_corrupt_count"], 3) == 0
        assert lib.moe_layer_set_option(h, opt["fault_corrupt_count"], 1 << 21) == pkg.MOE_E_INVAL
        assert lib.moe_layer_set_option(h, opt["fault_repush"], 5) == 0
        assert lib.moe_layer_set_option(h, opt["debug_claims"], 1) == 0
        # statistics of a layer that has not run a forward
        assert lib.moe_layer_get_stat(h, pkg.STATS["pair"]) == -1
    finally:
        lib.moe_layer_destroy(h)


def test_residual_norm_entry_validates_without_device(lib):
    h = lib.moe_layer_create(2048, 768, 128, 8, 0)
    try:
        f = lib.moe_layer_forward_residual_norm
        ptrs = [16] * 5
        # missing residual / gamma / norm_out
        assert f(h, 1, *ptrs, None, 16, 1e-5, 16, 16, None) == pkg.MOE_E_INVAL
        assert f(h, 1, *ptrs, 16, 16, 1e-5, 16, None, None) == pkg.MOE_E_INVAL
        # misaligned residual, negative eps
        assert f(h, 1, *ptrs, 8, 16, 1e-5, 16, 16, None) == pkg.MOE_E_INVAL
        assert f(h, 1, *ptrs, 16, 16, -1.0, 16, 16, None) == pkg.MOE_E_INVAL
        # well-formed but before reserve: a state error, not a crash
        assert f(h, 1, *ptrs, 16, 16, 1e-5, 16, 16, None) == pkg.MOE_E_STATE
    finally:
        lib.moe_layer_destroy(h)


def test_calibrate_validates_without_device(lib):
    assert lib.moe_layer_calibrate(None, 8, 16, 16, 16, 16, 16, 16, 3, None, None) == \
        pkg.MOE_E_INVAL
    h = lib.moe_layer_create(2048, 768, 128, 8, 0)
    try:
        # before reserve: a state error, not a crash
        assert lib.moe_layer_calibrate(h, 8, 16, 16, 16, 16, 16, 16, 3, None, None) == \
            pkg.MOE_E_STATE
        assert lib.moe_layer_get_stat(h, pkg.STATS["tile_tokens"]) == -1
    finally:
        lib.moe_layer_destroy(h)
