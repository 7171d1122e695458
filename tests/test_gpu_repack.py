"""Load-time repack (exact binary16 quant plane + transposed f32 scale plane) and the GEMM on
repacked weights, vs the oracle: bit-exact planes, exact block dots, outputs within 1e-5 * S,
and bitwise equality with the GEMM on raw Q8_0 (same dots, same fold order)."""
import numpy as np
import pytest
import torch

import oracle
import q8_block_quantized_act_gb300 as q8
from gpu_util import (assert_within_tolerance, cuda, device_ok, ensure_built, host, problem,
                      sample_rows)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,k", [(8, 256), (130, 1280), (33, 8192), (4096, 4096), (5, 65536)])
def test_repack_bit_exact(n, k):
    ensure_built()
    _, _, wb, _, _ = problem(1, n, k)
    wq16, wdt = q8.repack_q8_0(cuda(wb), n, k)
    device_ok()
    ref16, refdt = oracle.repack_q8_0(wb, k, q8.q8act_repack_ldn(n))
    assert np.array_equal(host(wq16).view(np.uint16), ref16)
    assert np.array_equal(host(wdt).view(np.uint32), refdt.view(np.uint32))


@pytest.mark.parametrize("m,n,k", [(128, 128, 256), (130, 200, 512), (17, 300, 1280)])
def test_gemm_repacked_block_dots_exact(m, n, k):
    ensure_built()
    _, x, wb, xq, _ = problem(m, n, k, "token_scales")
    wq16, wdt = q8.repack_q8_0(cuda(wb), n, k)
    xqh, _ = q8.quantize_q8_1_mmq(cuda(x))
    D = torch.full((m, n, k // 32), -7, dtype=torch.int32, device="cuda")
    q8.check(q8.q8act_debug_gemm_repacked_block_dots(wq16, wdt, xqh, D, m, n, k))
    device_ok()
    assert np.array_equal(host(D), oracle.block_dots(wb, xq, k))


@pytest.mark.parametrize("m,n,k,kind", [
    (128, 128, 256, "normal"),
    (130, 200, 512, "token_scales"),     # ragged in m and n
    (1, 77, 4096, "normal"),
    (300, 520, 2048, "outliers"),
])
def test_gemm_repacked_matches_oracle_and_raw(m, n, k, kind):
    """Within 1e-5 * S of the oracle; and, with the last-wave split off (the two paths tile
    differently, so a split cuts k at different places), bitwise the raw-Q8_0 GEMM."""
    ensure_built()
    _, x, wb, xq, xd = problem(m, n, k, kind)
    w_d, x_d = cuda(wb), cuda(x)
    wq16, wdt = q8.repack_q8_0(w_d, n, k)
    y = host(q8.gemm_q8_0_repacked(wq16, wdt, x_d))
    small = torch.empty(q8.q8act_gemm_workspace_bytes(m, k) - q8.Q8ACT_GEMM_SPLIT_BYTES,
                        dtype=torch.uint8, device="cuda")
    y_whole = host(q8.gemm_q8_0_repacked(wq16, wdt, x_d, ws=small))
    y_raw = host(q8.gemm_q8_0(w_d, x_d, n, ws=small))
    device_ok()
    _, y64, S = oracle.matmul(wb, xq, xd, k)
    assert_within_tolerance(y, y64, S)
    assert np.array_equal(y_whole.view(np.uint32), y_raw.view(np.uint32))


@pytest.mark.parametrize("m,n", [(512, 4096), (512, 5152), (512, 20480), (2048, 20480), (512, 64448),
                                 (2048, 64448)])
def test_gemm_repacked_serving_shapes_sampled(m, n):
    ensure_built()
    k = 4096
    _, x, wb, xq, xd = problem(m, n, k, "token_scales" if n > 5152 else "normal")
    wq16, wdt = q8.repack_q8_0(cuda(wb), n, k)
    y = host(q8.gemm_q8_0_repacked(wq16, wdt, cuda(x)))
    device_ok()
    rows = sample_rows(n, 256)
    _, y64, S = oracle.matmul(wb, xq, xd, k, rows=rows)
    assert_within_tolerance(y[:, rows], y64, S)
