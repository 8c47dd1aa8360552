"""The C ABI without a GPU: the library builds and loads, exports every symbol
the header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from nvfp4_weight_only_gb300 import ffi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    return ffi.load(build_if_missing=True)


def header_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_binding_exports():
    assert len(HEADERS) == 2
    assert header_functions() == sorted(ffi.EXPORTS + ffi.TESTING_EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in ffi.STATUS_NAMES.items():
        s = lib.nvfp4_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0, name
    assert lib.nvfp4_status_string(99) == b"unknown status"


def test_repacked_sizes(lib):
    # aligned shapes keep the canonical byte count N*K*9/16
    for N, K in ((5120, 17408), (17408, 5120), (4096, 4096), (256, 256), (21504, 5376)):
        assert lib.nvfp4_repacked_bytes(N, K) == N * K * 9 // 16
        assert lib.nvfp4_repacked_gate_up_bytes(N, K) == 2 * N * K * 9 // 16
    # ragged shapes are zero-padded to 256 rows x 256 columns
    assert lib.nvfp4_repacked_bytes(200, 272) == 256 * 512 * 9 // 16
    assert lib.nvfp4_repacked_bytes(300, 16) == 512 * 256 * 9 // 16
    assert lib.nvfp4_repacked_bytes(0, 64) == 0


def test_workspace_queries_are_positive(lib):
    for M in (1, 2, 8, 9, 16):
        assert lib.nvfp4_gemv_workspace_bytes(M, 5120, 17408) > 256
        assert lib.ffn_swiglu_nvfp4_workspace_bytes(M, 5120, 17408) > 256 + M * 17408 * 2
    assert lib.nvfp4_gemv_workspace_bytes(0, 5120, 17408) == 0
    assert lib.nvfp4_gemv_workspace_bytes(64, 5120, 17408) > 0
    assert lib.nvfp4_gemv_workspace_bytes(65, 5120, 17408) == 0
    assert lib.nvfp4_quantize_scratch_bytes(5120, 17408) >= 8


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x10004)
NULL = ctypes.c_void_p(0)
S = ctypes.c_void_p(0)


def test_gemv_validation(lib):
    g = lib.nvfp4_gemv
    assert g(NULL, 1, 64, FAKE, 1.0, 64, FAKE, FAKE, 1 << 20, S) == 1
    assert g(FAKE, 0, 64, FAKE, 1.0, 64, FAKE, FAKE, 1 << 20, S) == 4
    assert g(FAKE, 65, 64, FAKE, 1.0, 64, FAKE, FAKE, 1 << 20, S) == 4
    assert g(FAKE, 1, 40, FAKE, 1.0, 64, FAKE, FAKE, 1 << 20, S) == 2
    assert g(FAKE, 1, 64, FAKE, 1.0, 0, FAKE, FAKE, 1 << 20, S) == 2
    assert g(MISALIGNED, 1, 64, FAKE, 1.0, 64, ctypes.c_void_p(0x20000), FAKE, 1 << 20, S) == 3
    # x and y overlap
    assert g(FAKE, 1, 64, ctypes.c_void_p(0x30000), 1.0, 64, ctypes.c_void_p(0x10020), FAKE,
             1 << 20, S) == 8


def test_ffn_validation(lib):
    f = lib.ffn_swiglu_nvfp4
    A = [ctypes.c_void_p(0x10000 * i) for i in range(1, 6)]
    assert f(NULL, 1, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3], A[4], 1 << 24, S) == 1
    assert f(A[0], 0, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3], A[4], 1 << 24, S) == 4
    assert f(A[0], 1, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 2, A[3], A[4], 1 << 24, S) == 4
    assert f(A[0], 1, 250, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3], A[4], 1 << 24, S) == 2
    assert f(A[0], 1, 256, 500, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3], A[4], 1 << 24, S) == 2
    assert f(A[0], 1, 256, 512, MISALIGNED, 1.0, 1.0, A[2], 1.0, 0, A[3], A[4], 1 << 24, S) == 3
    assert f(A[0], 1, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, A[0], A[4], 1 << 24, S) == 8


def test_quantize_and_repack_validation(lib):
    s2 = ctypes.c_float()
    q = lib.nvfp4_quantize
    assert q(NULL, 0, 16, 64, FAKE, FAKE, ctypes.byref(s2), FAKE, 256, S) == 1
    assert q(FAKE, 3, 16, 64, FAKE, FAKE, ctypes.byref(s2), FAKE, 256, S) == 4
    assert q(FAKE, 0, 16, 24, FAKE, FAKE, ctypes.byref(s2), FAKE, 256, S) == 2
    assert q(FAKE, 0, 0, 64, FAKE, FAKE, ctypes.byref(s2), FAKE, 256, S) == 2
    assert q(FAKE, 0, 16, 64, FAKE, FAKE, ctypes.byref(s2), FAKE, 4, S) == 5
    assert lib.nvfp4_repack(NULL, FAKE, 16, 64, FAKE, S) == 1
    assert lib.nvfp4_repack(FAKE, FAKE, 16, 40, FAKE, S) == 2
    assert lib.nvfp4_repack(FAKE, FAKE, 16, 64, MISALIGNED, S) == 3
    assert lib.nvfp4_repack_gate_up(FAKE, FAKE, FAKE, NULL, 16, 64, FAKE, S) == 1
    assert lib.nvfp4_unpack(FAKE, 16, 8, FAKE, FAKE, S) == 2
    assert lib.nvfp4_workspace_init(NULL, 16, S) == 1
    assert lib.nvfp4_workspace_status(NULL, S) == 1


def test_binding_raises_without_cuda_tensors():
    import torch
    with pytest.raises(ValueError):
        ffi.nvfp4_gemv(torch.zeros(1, 64, dtype=torch.bfloat16), torch.zeros(10, dtype=torch.uint8),
                       1.0, 64)


def test_shared_memory_plans_are_aligned(lib):
    """Every shared-memory plan the GEMV kernel can be launched with keeps the
    alignment its accesses assume (bulk-copy stages and vector loads on 16
    bytes, mbarriers on 8, the misc area on 128) and fits the per-block limit,
    for every M, odd stage counts included, across SM counts and shapes."""
    shapes = [(5120, 17408), (17408, 5120), (4096, 12288), (12288, 4096), (5376, 21504),
              (21504, 5376), (65536, 21504), (65536, 4096), (4096, 4096), (200, 272), (16, 16),
              (1, 2048), (300, 21504), (384, 1024)]
    for streams in (1, 2):
        for M in range(1, 17):
            for N, K in shapes:
                for sms in (152, 148, 132, 160, 7, 1):
                    assert lib.nvfp4_testing_plan_aligned(streams, M, N, K, sms) == 1, \
                        (streams, M, N, K, sms)
    assert lib.nvfp4_testing_plan_aligned(3, 1, 256, 256, 152) == -1
    assert lib.nvfp4_testing_plan_aligned(1, 17, 256, 256, 152) == -1


def test_testing_stall_switch_validates_its_limit(lib):
    assert lib.nvfp4_testing_inject_stall(1, 10) == 4          # below 1 us: NVFP4_ERR_RANGE
    assert lib.nvfp4_testing_inject_stall(1, 2 * 10 ** 9) == 4  # above 1 s
    assert lib.nvfp4_testing_inject_stall(0, 0) == 0           # off: always accepted


def test_noalloc_validation_touches_nothing(lib):
    """Argument errors of the fixed-workspace FFN are found on the host before
    any device set-up (these calls run without a GPU)."""
    f = lib.ffn_swiglu_nvfp4_noalloc
    A = [ctypes.c_void_p(0x10000 * i) for i in range(1, 5)]
    assert f(NULL, 1, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3], S) == 1
    assert f(A[0], 17, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3], S) == 4
    assert f(A[0], 1, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 7, A[3], S) == 4
    assert f(A[0], 1, 250, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3], S) == 2
    assert f(A[0], 1, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, MISALIGNED, S) == 3
    assert f(A[0], 1, 256, 512, A[1], 1.0, 1.0, A[2], 1.0, 0, A[0], S) == 8
    B = [ctypes.c_void_p(0x10000000 * i) for i in range(1, 5)]  # disjoint at this size
    assert f(B[0], 16, 8192, 32768, B[1], 1.0, 1.0, B[2], 1.0, 0, B[3], S) == 5


def test_w8a16_repacked_sizes(lib):
    """FP8 blobs: the codes (N*K bytes for shapes that are multiples of 256)
    plus one fp32 scale per 16-row tile and 64-K chunk (1/256 more)."""
    for N, K in ((5120, 17408), (17408, 5120), (4096, 4096), (256, 256)):
        assert lib.w8a16_repacked_bytes(N, K) == N * K + N * K // 256
        assert lib.w8a16_repacked_gate_up_bytes(N, K) == 2 * (N * K + N * K // 256)
    assert lib.w8a16_repacked_bytes(200, 272) == 256 * 512 * (1 + 1 / 256)
    assert lib.w8a16_repacked_bytes(0, 64) == 0


def test_w8a16_plans_are_aligned(lib):
    shapes = [(5120, 17408), (17408, 5120), (4096, 12288), (12288, 4096), (65536, 21504),
              (4096, 4096), (200, 272), (16, 16), (1, 2048), (300, 21504)]
    for streams in (1, 2):
        for M in range(1, 17):
            for N, K in shapes:
                for sms in (152, 148, 7, 1):
                    assert lib.nvfp4_testing_plan_aligned_w8a16(streams, M, N, K, sms) == 1, \
                        (streams, M, N, K, sms)


def test_w8a16_validation_before_any_launch(lib):
    """Argument errors of the FP8 calls come back without a GPU."""
    p = ctypes.c_void_p(0x10000000)
    q = ctypes.c_void_p(0x20000000)
    ws = ctypes.c_void_p(0x30000000)
    f = lib.ffn_swiglu_w8a16
    assert f(None, 1, 256, 512, p, q, 0, ws, ws, 1 << 20, None) == 1           # null x
    assert f(p, 0, 256, 512, p, q, 0, q, ws, 1 << 20, None) == 4              # M = 0
    assert f(p, 65, 256, 512, p, q, 0, q, ws, 1 << 20, None) == 4             # M = 65
    assert f(p, 1, 250, 512, p, q, 0, q, ws, 1 << 20, None) == 2              # H % 16
    assert f(p, 1, 256, 512, p, q, 7, q, ws, 1 << 20, None) == 4              # act
    assert f(ctypes.c_void_p(0x10000004), 1, 256, 512, p, q, 0, q, ws, 1 << 20, None) == 3
    g = lib.w8a16_gemv
    assert g(p, 1, 250, q, 64, ws, ws, 1 << 20, None) == 2                    # K % 16
    assert g(p, 1, 256, q, 64, p, ws, 1 << 20, None) == 8                     # x and y overlap
    r = lib.w8a16_repack
    assert r(p, ctypes.c_void_p(0x20000002), 256, 256, q, None) == 3         # grid alignment
    assert r(p, q, 256, 8, q, None) == 2
