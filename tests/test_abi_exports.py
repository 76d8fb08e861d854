"""The C-ABI library builds, loads without a GPU and exports every declared symbol."""
import ctypes
import os
import re

import pytest

import aux_loss_free_gb300 as M
from aux_loss_free_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    return B.build()


def test_header_declares_the_documented_calls():
    names = declared_functions()
    for required in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine",
                     "moe_bias_update", "moe_layer_fwd"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    assert sorted(M.SIGNATURES) == declared_functions()


def test_pure_host_entry_points(lib_path):
    lib = M.load_library(lib_path)
    assert lib.moe_abi_version() == 2
    assert lib.moe_status_string(0) == b"ok"
    assert [lib.moe_gate_up_block(w) for w in (512, 2048, 64, 32, 96)] == [128, 128, 64, 32, 32]


def test_host_validation_rejects_bad_shapes_before_any_launch(lib_path):
    M.load_library(lib_path)
    bad = [
        M.make_shape(0, 1024, 64, 512, 2048, 2),      # T = 0
        M.make_shape(16, 1000, 64, 512, 2048, 2),     # d % 64 != 0
        M.make_shape(16, 1024, 300, 512, 2048, 2),    # E > 256
        M.make_shape(16, 1024, 4, 512, 2048, 5),      # k > E
        M.make_shape(16, 1024, 64, 500, 2048, 2),     # f % 32 != 0
        M.make_shape(16, 1024, 64, 512, 2048, 2, w_format=M.MOE_W_INT4_G32),  # int4 needs k = 1
    ]
    for s in bad:
        assert M.moe_layer_workspace_size(s) == 0
        assert M.moe_permute_workspace_size(s) == 0
    good = M.make_shape(8192, 1024, 64, 512, 2048, 2)
    assert M.moe_layer_workspace_size(good) > 8192 * 2 * 1024 * 2
    lib = M.load_library()
    # Null pointers are rejected on the host (no device touched).
    assert lib.moe_route(ctypes.byref(good), None, None, None, None, None, None, None, None,
                         None, 0, None) == 1
    assert M.moe_route_workspace_size(good) == 3 * 64 * 1024 * 2
    assert M.moe_route_workspace_size(M.make_shape(64, 1024, 64, 512, 2048, 2)) == 0  # small T: CUDA-core router
    assert M.moe_route_workspace_size(M.make_shape(64, 64, 8, 32, 128, 2, x_dtype=M.MOE_X_F32)) == 0
    assert lib.moe_bias_update(0, 16, None, 1e-3, None, None) == 1
    p = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation first
    assert lib.moe_bias_update(64, -2, p, ctypes.c_float(1e-3), p, None) == 1  # only -1 means "sum the loads"
    assert lib.moe_load_balance(0, p, p, None) == 1                       # no experts
    assert lib.moe_load_balance(64, p, ctypes.c_void_p(20), None) == 1    # balance not 8-byte aligned
    assert lib.moe_load_balance(64, None, p, None) == 1


def test_noalloc_permute_validates_like_permute(lib_path):
    """moe_permute_noalloc returns the status moe_permute returns for every bad shape
    (both validate before touching the device)."""
    lib = M.load_library(lib_path)
    p = ctypes.c_void_p(16)
    bad = [
        M.make_shape(0, 1024, 64, 512, 2048, 2),
        M.make_shape(16, 1000, 64, 512, 2048, 2),
        M.make_shape(16, 1024, 300, 512, 2048, 2),
        M.make_shape(16, 1024, 4, 512, 2048, 5),
        M.make_shape(16, 1024, 64, 500, 2048, 2),
        M.make_shape(16, 1024, 64, 512, 2048, 2, renorm=True, x_dtype=7),
        M.make_shape(16, 1024, 64, 512, 2048, 2, w_format=M.MOE_W_INT4_G32),
    ]
    for s in bad:
        want = lib.moe_permute(ctypes.byref(s), p, p, p, p, p, 1 << 20, None)
        assert want != 0
        assert lib.moe_permute_noalloc(ctypes.byref(s), p, p, p, p, None) == want
    good = M.make_shape(64, 1024, 64, 512, 2048, 2)
    assert lib.moe_permute_noalloc(ctypes.byref(good), None, p, p, p, None) == 1  # null idx


def test_expert_parallel_calls_validate_on_the_host(lib_path):
    """moe_gather_rows and moe_ep_regroup reject bad sizes and null pointers before any
    launch (MOE_ERR_INVALID_ARG = 1), so this runs without a GPU."""
    lib = M.load_library(lib_path)
    p = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation first
    assert lib.moe_gather_rows(-1, 256, p, p, p, None) == 1     # negative row count
    assert lib.moe_gather_rows(4, 12, p, p, p, None) == 1       # d not a multiple of 8
    assert lib.moe_gather_rows(4, 16384, p, p, p, None) == 1    # d too wide
    assert lib.moe_gather_rows(4, 256, None, p, p, None) == 1   # null source
    assert lib.moe_gather_rows(4, 256, ctypes.c_void_p(24), p, p, None) == 1  # misaligned source
    assert lib.moe_ep_regroup(0, 8, p, p, p, p, None) == 1      # no ranks
    assert lib.moe_ep_regroup(2, 0, p, p, p, p, None) == 1      # no local experts
    assert lib.moe_ep_regroup(64, 128, p, p, p, p, None) == 1   # count table too large
    assert lib.moe_ep_regroup(2, 8, p, None, p, p, None) == 1   # null output


def test_selftest_call_validates_on_the_host(lib_path):
    lib = M.load_library(lib_path)
    out = ctypes.c_int32(0)
    assert lib.moe_selftest_bounded_wait(0, ctypes.byref(out), None) == 1              # no limit
    assert lib.moe_selftest_bounded_wait(2_000_000_000, ctypes.byref(out), None) == 1  # over 1 s
    assert lib.moe_selftest_bounded_wait(1000, None, None) == 1                        # no output


def test_short_workspace_name_matches_the_layer_query(lib_path):
    M.load_library(lib_path)
    lib = M.load_library()
    for s in (M.make_shape(8192, 1024, 64, 512, 2048, 2), M.make_shape(64, 64, 8, 32, 128, 2),
              M.make_shape(0, 1024, 64, 512, 2048, 2)):
        assert lib.moe_workspace_size(ctypes.byref(s)) == M.moe_layer_workspace_size(s)


def test_attention_calls_validate_on_the_host(lib_path):
    lib = M.load_library(lib_path)
    p = ctypes.c_void_p(16)
    good = M.make_attn_shape(4, 2048, 1024, 8, 2)
    # q, k, v rows [8192][(8 + 2 + 2) * 128] and the attention output [8192][8 * 128], bf16
    assert M.moe_attention_workspace_size(good) == 2 * 8192 * 12 * 128 + 2 * 8192 * 8 * 128
    for bad, code in ((M.make_attn_shape(4, 2048, 1024, 8, 2, head_dim=64), 2),   # head width other than 128
                      (M.make_attn_shape(4, 2048, 1024, 8, 3), 2),                 # 8 heads do not group by 3
                      (M.make_attn_shape(4, 2048, 1000, 8, 2), 2),                 # d % 64 != 0
                      (M.make_attn_shape(0, 2048, 1024, 8, 2), 1),                 # no sequences
                      (M.make_attn_shape(4, 2048, 1024, 8, 2, eps=0.0), 1)):       # eps must be positive
        assert M.moe_attention_workspace_size(bad) == 0
        assert lib.moe_attention_fwd(ctypes.byref(bad), p, p, p, 1, p, p, 1 << 30, None) == code
        assert lib.moe_attention_core(ctypes.byref(bad), p, p, None) == code
    assert lib.moe_attention_fwd(ctypes.byref(good), None, p, p, 1, p, p, 1 << 30, None) == 1
    assert lib.moe_attention_fwd(ctypes.byref(good), p, p, p, 1, p, p, 16, None) == 3  # workspace too small
