"""The C ABI library (CPU-side checks, no GPU needed): it loads, exports
every entry point include/fp8bs.h declares, and rejects bad arguments on the
host before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def fp8():
    import fp8_block_scaled_07_gb300 as m
    return m


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ["fp8_act_quant", "fp8_gemm", "fp8_grouped_gemm", "fp8_weight_dequant",
              "fp8_gemm_workspace_size", "fp8_device_status", "fp8_status_string"]:
        assert s in syms


def test_library_exports_every_declared_symbol(fp8):
    lib = ctypes.CDLL(fp8.LIB_PATH)
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_status_strings(fp8):
    for code in range(6):
        assert fp8.lib.fp8_status_string(code)
    assert fp8.lib.fp8_status_string(99) == b"unknown status"


def test_host_validation_rejects_bad_arguments(fp8):
    L, NULL = fp8.lib, None
    # K not a multiple of 128
    assert L.fp8_act_quant(NULL, NULL, NULL, 4, 100, 0, NULL) == 1
    # unknown scale format
    assert L.fp8_act_quant(NULL, NULL, NULL, 4, 128, 7, NULL) == 1
    # null pointers with a real shape
    assert L.fp8_act_quant(NULL, NULL, NULL, 4, 128, 0, NULL) == 1
    # misaligned pointer
    assert L.fp8_act_quant(ctypes.c_void_p(8), ctypes.c_void_p(16), ctypes.c_void_p(16), 4, 128, 0, NULL) == 1
    assert L.fp8_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 4, 4, 100, NULL, 0, NULL) == 1
    assert L.fp8_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 4, 4, 128, NULL, 0, NULL) == 1
    assert L.fp8_grouped_gemm(NULL, NULL, NULL, NULL, NULL, 4, 16, NULL, NULL, 100, 128, NULL) == 1
    assert L.fp8_weight_dequant(NULL, NULL, NULL, 4, 15, NULL) == 1
    assert L.fp8_silu_mul_quant(NULL, NULL, 256, 4, 100, NULL, NULL, NULL, 0, NULL) == 1
    assert L.fp8_moe_route(NULL, 4, 8, 2000, NULL, NULL, NULL, NULL) == 1
    assert L.fp8_moe_combine(NULL, NULL, NULL, 4, 8, 12, NULL, NULL, NULL) == 1
    # fp8_gemm_noalloc checks its arguments before it touches the device
    assert L.fp8_gemm_noalloc(NULL, NULL, NULL, NULL, NULL, NULL, 4, 4, 100, NULL) == 1
    assert L.fp8_gemm_noalloc(NULL, NULL, NULL, NULL, NULL, NULL, 4, 4, 128, NULL) == 1
    assert L.fp8_gemm_noalloc(ctypes.c_void_p(8), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                              ctypes.c_void_p(16), NULL, 4, 4, 128, NULL) == 1
    # fp8_linear: unknown scale format
    assert L.fp8_linear(NULL, NULL, NULL, NULL, NULL, 4, 4, 128, 7, NULL, 0, NULL) == 1


def test_empty_problems_are_no_ops(fp8):
    L, NULL = fp8.lib, None
    assert L.fp8_act_quant(NULL, NULL, NULL, 0, 128, 0, NULL) == 0
    assert L.fp8_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 0, 16, 128, NULL, 0, NULL) == 0
    assert L.fp8_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 16, 0, 128, NULL, 0, NULL) == 0
    assert L.fp8_grouped_gemm(NULL, NULL, NULL, NULL, NULL, 0, 16, NULL, NULL, 128, 128, NULL) == 0
    assert L.fp8_weight_dequant(NULL, NULL, NULL, 0, 16, NULL) == 0
