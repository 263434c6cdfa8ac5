"""The C-ABI library builds, loads and exports every entry point include/moe.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_six_path_calls():
    names = declared_symbols()
    for n in ["moe_gating_softmax_topk", "moe_indices_to_multihot", "moe_multihot_to_indices",
              "moe_align_by_expert", "moe_grouped_ffn", "moe_layer_forward"]:
        assert n in names


@pytest.fixture(scope="module")
def built_lib():
    from mixture_experts_routing_token_gb300.build import build
    return build()


def test_library_exports_every_declared_symbol(built_lib):
    lib = ctypes.CDLL(built_lib)
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_signatures_cover_header(built_lib):
    import mixture_experts_routing_token_gb300 as moe
    assert set(moe.SIGNATURES) == set(declared_symbols())
    moe.lib()
    assert "sm_103a" in moe.version()


def test_workspace_sizes_without_gpu(built_lib):
    import mixture_experts_routing_token_gb300 as moe
    # pure host arithmetic
    S = 4096 * 2
    n = moe.moe_layer_workspace_size(moe.MOE_BF16, 4096, 4096, 14336, 8, 2)
    assert n >= S * 14336 * 2 + S * 4096 * 2 + S * 4096 * 2   # act, bf16 staging, sorted token rows
    # decode batches (T <= 64) keep float32 staging rows
    assert moe.moe_layer_workspace_size(moe.MOE_BF16, 64, 2048, 1408, 64, 8) >= 512 * 1408 * 2 + 512 * 2048 * 4
    assert moe.moe_align_workspace_size(1, 8, 64) == 0          # single chunk: no scratch
    assert moe.moe_align_workspace_size(32768, 8, 128) >= 64 * 128 * 4
    assert moe.moe_grouped_ffn_workspace_size(moe.MOE_F32, 0, 8, 8, 4, 2) >= 0


def test_host_argument_checks_without_gpu(built_lib):
    """Invalid shapes are rejected on the host before any device work."""
    lib = ctypes.CDLL(built_lib)
    f = lib.moe_gating_softmax_topk
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert f(None, 4, 8, 9, 1, None, None, None) == 1            # k > E
    assert f(None, 4, 8, 0, 1, None, None, None) == 1            # k < 1
    assert f(None, 4, 2000, 2, 1, None, None, None) == 1         # E too large
    assert f(None, -1, 8, 2, 1, None, None, None) == 1           # T < 0
    assert f(None, 0, 8, 2, 1, None, None, None) == 0            # empty is fine, nothing launched
    lib.moe_last_error.restype = ctypes.c_char_p
    assert lib.moe_last_error() == b""
