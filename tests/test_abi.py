"""The C-ABI library loads and exports every function include/*.h declares (CPU only).

Only host-side entry points are called here (version, workspace sizing, argument checks
that return before any launch); nothing touches a GPU.
"""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_pft_gb300 import build as bld

    path = bld.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ["moe_route", "moe_route_bwd", "moe_pft_build", "moe_dispatch", "moe_dispatch_bwd",
              "moe_expert_ffn", "moe_expert_ffn_bwd", "moe_combine", "moe_combine_bwd",
              "moe_workspace_size", "moe_check_status", "moe_status_reset", "moe_last_error"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_signatures_cover_the_header():
    from mixture_experts_layer_pft_gb300 import binding

    assert set(declared_functions()) <= set(binding.SIGNATURES) | {"moe_abi_version"}


def test_host_only_entry_points(lib):
    from mixture_experts_layer_pft_gb300 import binding as B

    lib.moe_abi_version.restype = ctypes.c_int
    assert lib.moe_abi_version() == 2
    f = lib.moe_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 7
    sizes = [f(op, 4096, 7168, 256, 8, 2048, B.MOE_BF16) for op in range(B.MOE_OP_ALL)]
    assert all(s >= 256 and s % 256 == 0 for s in sizes)
    assert f(B.MOE_OP_ALL, 4096, 7168, 256, 8, 2048, B.MOE_BF16) == max(sizes)
    # the expert backward keeps dh1 and dh3 (Tk x f each) in the workspace
    assert sizes[B.MOE_OP_EXPERT_FFN_BWD] >= 256 + 2 * 4096 * 8 * 2048 * 2


def test_argument_errors_return_before_any_launch(lib):
    from mixture_experts_layer_pft_gb300 import binding as B

    fn = lib.moe_dispatch
    fn.restype = ctypes.c_int
    fn.argtypes = B.SIGNATURES["moe_dispatch"][1]
    ws = ctypes.create_string_buffer(512)
    p = ctypes.c_void_p(16)  # never dereferenced: the checks fail first
    # h not a multiple of 8 -> unsupported
    assert fn(p, p, 4, 2, 12, B.MOE_BF16, p, ws, 512, None) == B.MOE_ERR_UNSUPPORTED
    # bad dtype -> invalid argument
    assert fn(p, p, 4, 2, 16, 7, p, ws, 512, None) == B.MOE_ERR_INVALID_ARG
    # workspace too small
    assert fn(p, p, 4, 2, 16, B.MOE_BF16, p, ws, 16, None) == B.MOE_ERR_WORKSPACE
    lib.moe_last_error.restype = ctypes.c_char_p
    assert b"workspace" in lib.moe_last_error()
    r = lib.moe_route
    r.restype = ctypes.c_int
    r.argtypes = B.SIGNATURES["moe_route"][1]
    # k > E
    assert r(p, p, None, 4, 16, 8, 9, B.MOE_F32, 0, p, p, p, p, ws, 512, None) == B.MOE_ERR_INVALID_ARG


def test_withhold_hook_checks_its_arguments(lib):
    from mixture_experts_layer_pft_gb300 import binding as B

    fn = lib.moe_debug_withhold_stage
    fn.restype = ctypes.c_int
    fn.argtypes = B.SIGNATURES["moe_debug_withhold_stage"][1]
    assert fn(-1, 0) == B.MOE_ERR_INVALID_ARG
    assert fn(1, 1000) == B.MOE_ERR_INVALID_ARG  # below 1 ms
    assert fn(1, 3_000_000_000) == B.MOE_ERR_INVALID_ARG  # above 2 s
    assert fn(0, 0) == B.MOE_OK  # cancel: nothing pending
