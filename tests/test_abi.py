"""The C ABI without a GPU: the library loads, exports every declared entry point, and
refuses bad arguments on the host before any CUDA call (no compute is launched here)."""
import os
import re

import pytest

import q8_block_quantized_act_gb300 as q8
from q8_block_quantized_act_gb300 import build as q8build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q8act.h")


@pytest.fixture(scope="module")
def L():
    q8build.build()
    return q8.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q8act_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(L, name), f"{name} declared in q8act.h but not exported"
    assert set(names) == set(q8.EXPORTED)


def test_version_and_strerror(L):
    assert q8.q8act_version() >= 100
    for rc in (0, -1, -2, -3, -4, -5, -6, -7, 1002):
        assert isinstance(q8.strerror(rc), str) and q8.strerror(rc)


def test_gemv_workspace_query(L):
    # int8 quants then f32 scales, each rounded up to 256 bytes; 0 for invalid m or k
    assert q8.q8act_gemv_workspace_bytes(1, 4096) == 4096 + 512
    assert q8.q8act_gemv_workspace_bytes(3, 256) == 768 + 256
    assert q8.q8act_gemv_workspace_bytes(0, 4096) == 0
    assert q8.q8act_gemv_workspace_bytes(q8.Q8ACT_GEMV_MAX_M + 1, 4096) == 0
    assert q8.q8act_gemv_workspace_bytes(1, 100) == 0


def test_workspace_query(L):
    assert q8.q8act_gemm_workspace_bytes(512, 4096) >= 512 * 4096 * 2 + 4096 // 32 * 512 * 4
    assert q8.q8act_gemm_workspace_bytes(0, 4096) == 0
    assert q8.q8act_gemm_workspace_bytes(16, 4000) == 0
    assert q8.q8act_gemm_workspace_bytes(16, -256) == 0
    assert q8.q8act_mmq_ldm(1) == 4 and q8.q8act_mmq_ldm(4) == 4 and q8.q8act_mmq_ldm(5) == 8
    assert q8.q8act_mmq_ldm(0) == 0
    assert q8.q8act_repack_ldn(1) == 4 and q8.q8act_repack_ldn(4096) == 4096
    assert q8.q8act_repack_ldn(4097) == 4100 and q8.q8act_repack_ldn(0) == 0


A = 1 << 20          # a fake, 16-byte aligned address: never dereferenced by these calls
MIS = A + 4          # misaligned
S0 = 0               # legacy stream handle


@pytest.mark.parametrize("call,want", [
    (lambda: q8.q8act_quantize_q8_1(None, A, A, 1, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_quantize_q8_1(A, A, A, 1, 100, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_quantize_q8_1(A, A, A, 0, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_quantize_q8_1(MIS, A, A, 1, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_quantize_q8_1_mmq(A, None, A, 1, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_quantize_q8_0(A, A, 4, 288, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0(A, A, A, None, 1, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemv_q8_0(A, A, A, A, q8.Q8ACT_GEMV_MAX_M + 1, 8, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0(A, A, A, A, 0, 8, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0(A, A, A, A, 1, 0, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0(A, A, A, A, 1, 8, 1280 + 32, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0(A, A, A, A, 1, 8, 2 * q8.Q8ACT_MAX_K, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0(MIS, A, A, A, 1, 8, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_gemm_q8_0(A, A, A, 16, 8, 256, None, 1 << 30, S0), q8.Q8ACT_ERR_WORKSPACE),
    (lambda: q8.q8act_gemm_q8_0(A, A, A, 16, 8, 256, A, 16, S0), q8.Q8ACT_ERR_WORKSPACE),
    (lambda: q8.q8act_gemm_q8_0(A, A, A, 16, 8, 255, A, 1 << 30, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemm_q8_0(A, MIS, A, 16, 8, 256, A, 1 << 30, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_gemm_q8_0_preq(A, A, A, None, 16, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemm_q8_0_preq(A, A, A, A, 16, 0, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_dequant_q8_0_f16(A, None, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_dequant_q8_0_f16(A, MIS, 8, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_debug_gemv_block_dots(A, A, None, 1, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_debug_gemm_block_dots(A, A, None, 1, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_repack_q8_0(A, A, None, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_repack_q8_0(A, A, A, 8, 300, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_repack_q8_0(A, MIS, A, 8, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_gemm_q8_0_repacked(A, None, A, A, 16, 8, 256, A, 1 << 30, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemm_q8_0_repacked(A, A, A, A, 16, 8, 256, A, 16, S0), q8.Q8ACT_ERR_WORKSPACE),
    (lambda: q8.q8act_gemm_q8_0_repacked(A, A, A, A, 16, 8, 255, A, 1 << 30, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemm_q8_0_repacked(A, MIS, A, A, 16, 8, 256, A, 1 << 30, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_debug_gemm_repacked_block_dots(A, A, A, None, 1, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemv_q8_0_group([], [], [], A, A, 1, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0_group([A] * 9, [A] * 9, [8] * 9, A, A, 1, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0_group([A, None], [A, A], [8, 8], A, A, 1, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemv_q8_0_group([A, A], [A, A], [8, 0], A, A, 1, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0_group([A, MIS], [A, A], [8, 8], A, A, 1, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_gemv_q8_0_group([A], [A], [8], A, A, q8.Q8ACT_GEMV_MAX_M + 1, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_quantize_q4_0(None, A, 4, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_quantize_q4_0(A, A, 4, 288, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_quantize_q4_0(A, MIS, 4, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_dequant_q4_0_f16(A, None, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_dequant_q4_0_f16(A, A, 0, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_dequant_q4_0_f16(MIS, A, 8, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_gemv_q4_0(A, A, A, None, 1, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemv_q4_0(A, A, A, A, q8.Q8ACT_GEMV_MAX_M + 1, 8, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q4_0(A, A, A, A, 1, 8, 1280 + 32, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q4_0(A, A, MIS, A, 1, 8, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_debug_gemv_q4_0_block_dots(A, A, None, 1, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemv_q8_0_f32(A, None, A, 1, 8, 256, A, 1 << 20, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemv_q8_0_f32(A, A, A, 0, 8, 256, A, 1 << 20, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0_f32(A, A, A, q8.Q8ACT_GEMV_MAX_M + 1, 8, 256, A, 1 << 20, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0_f32(A, A, A, 1, 8, 300, A, 1 << 20, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q8_0_f32(A, A, A, 1, 8, 256, None, 1 << 20, S0), q8.Q8ACT_ERR_WORKSPACE),
    (lambda: q8.q8act_gemv_q8_0_f32(A, A, A, 1, 8, 256, A, 16, S0), q8.Q8ACT_ERR_WORKSPACE),
    (lambda: q8.q8act_gemv_q8_0_f32(A, MIS, A, 1, 8, 256, A, 1 << 20, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_gemm_q8_0_noalloc(None, A, A, 16, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemm_q8_0_noalloc(A, None, A, 16, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemm_q8_0_noalloc(A, A, None, 16, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemm_q8_0_noalloc(A, A, A, 0, 8, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemm_q8_0_noalloc(A, A, A, 16, 0, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemm_q8_0_noalloc(A, A, A, 16, 8, 300, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemm_q8_0_noalloc(A, A, A, 2892, 8, 4096, S0), q8.Q8ACT_ERR_WORKSPACE),
    (lambda: q8.q8act_debug_wait_timeout(0, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_dequant_q6_k_f16(A, None, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_dequant_q4_k_f16(A, A, 8, 100, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_dequant_q5_k_f16(MIS, A, 8, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_gemv_q6_k(A, A, A, None, 1, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_gemv_q4_k(A, A, A, A, 9, 8, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q5_k(A, A, A, A, 1, 0, 256, S0), q8.Q8ACT_ERR_DIMS),
    (lambda: q8.q8act_gemv_q5_k(A, MIS, A, A, 1, 8, 256, S0), q8.Q8ACT_ERR_ALIGN),
    (lambda: q8.q8act_debug_gemv_q6_k_block_dots(A, A, None, 1, 8, 256, S0), q8.Q8ACT_ERR_NULL),
    (lambda: q8.q8act_debug_wait_timeout(10 ** 10, S0), q8.Q8ACT_ERR_DIMS),
])
def test_host_side_refusals(L, call, want):
    assert call() == want
