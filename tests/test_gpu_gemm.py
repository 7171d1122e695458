"""GPU GEMM (prefill MMQ on tcgen05) vs the oracle: exact block dots from the tensor-core
path, outputs within 1e-5 * S, fused and pre-quantized entry points, ragged tiles."""
import numpy as np
import pytest
import torch

import oracle
import q8_block_quantized_act_gb300 as q8
from gpu_util import (assert_within_tolerance, cuda, device_ok, ensure_built, host, problem,
                      sample_rows)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,n,k", [(128, 128, 256), (130, 200, 512), (1, 64, 256),
                                   (17, 300, 1280), (256, 384, 4096)])
def test_gemm_block_dots_exact(m, n, k):
    ensure_built()
    _, x, wb, xq, _ = problem(m, n, k, "token_scales")
    xqh, xdt = q8.quantize_q8_1_mmq(cuda(x))
    D = torch.full((m, n, k // 32), -7, dtype=torch.int32, device="cuda")
    q8.check(q8.q8act_debug_gemm_block_dots(cuda(wb), xqh, D, m, n, k))
    device_ok()
    assert np.array_equal(host(D), oracle.block_dots(wb, xq, k))


@pytest.mark.parametrize("m,n,k,kind", [
    (128, 128, 256, "normal"),
    (130, 200, 512, "token_scales"),     # ragged in m and n
    (1, 77, 4096, "normal"),             # m below the prefill threshold
    (16, 4096, 1280, "normal"),
    (300, 520, 2048, "outliers"),
])
def test_gemm_matches_oracle(m, n, k, kind):
    ensure_built()
    _, x, wb, xq, xd = problem(m, n, k, kind)
    y = host(q8.gemm_q8_0(cuda(wb), cuda(x), n))
    device_ok()
    _, y64, S = oracle.matmul(wb, xq, xd, k)
    assert_within_tolerance(y, y64, S)


def _min_workspace(m, k):
    """A workspace without the split region (every tile is then done by one CTA over the whole
    of k)."""
    return torch.empty(q8.q8act_gemm_workspace_bytes(m, k) - q8.Q8ACT_GEMM_SPLIT_BYTES,
                       dtype=torch.uint8, device="cuda")


def test_gemm_preq_equals_fused():
    """Without the split region the fused call is the quantizer followed by the pre-quantized
    GEMM, bit for bit."""
    ensure_built()
    m, n, k = 200, 260, 1024
    _, x, wb, xq, xd = problem(m, n, k, "token_scales")
    w_d, x_d = cuda(wb), cuda(x)
    y_fused = host(q8.gemm_q8_0(w_d, x_d, n, ws=_min_workspace(m, k)))
    xqh, xdt = q8.quantize_q8_1_mmq(x_d)
    y_pre = host(q8.gemm_q8_0_preq(w_d, xqh, xdt, n))
    device_ok()
    assert np.array_equal(y_fused.view(np.uint32), y_pre.view(np.uint32))


def _balanced(m, n, k):
    """The fused GEMM's schedule choice (mirrors the library's plan): True when its cost model
    prefers equal contiguous runs of (tile, k group) units per CTA over one CTA per tile."""
    slots = min(torch.cuda.get_device_properties(0).multi_processor_count, 160)
    tiles = -(-n // 128) * -(-m // 128)
    G = k // 256
    U = tiles * G
    if tiles % slots == 0:
        return False
    C = min(slots, U)
    waves = -(-tiles // slots)
    per = U // C
    balanced_cost = -(-U // C) + 2 + (-(-G // per) + 1)
    return balanced_cost < waves * G + waves - 1


@pytest.mark.parametrize("m,n,k", [
    (512, 5152, 4096),    # 164 tiles on 152 SMs
    (256, 20480, 1024),   # 320 tiles, 4 groups each
    (64, 9000, 4096),     # ragged in m and n; tiles cut into up to 3 pieces
    (512, 2048, 4096),    # 64 tiles, every one cut
])
def test_gemm_balanced_schedule(m, n, k):
    """The balanced schedule: within 1e-5 * S of the oracle, deterministic, and within the same
    bound of the one-CTA-per-tile schedule (only the order of the fold's f32 additions
    differs); on the repacked weights too."""
    ensure_built()
    assert _balanced(m, n, k), "shape does not take the balanced schedule"
    _, x, wb, xq, xd = problem(m, n, k, "token_scales")
    w_d, x_d = cuda(wb), cuda(x)
    y_bal = host(q8.gemm_q8_0(w_d, x_d, n))
    y_again = host(q8.gemm_q8_0(w_d, x_d, n))
    y_plain = host(q8.gemm_q8_0(w_d, x_d, n, ws=_min_workspace(m, k)))
    wq16, wdt = q8.repack_q8_0(w_d, n, k)
    y_rp = host(q8.gemm_q8_0_repacked(wq16, wdt, x_d))
    device_ok()
    rows = sample_rows(n, 256)
    _, y64, S = oracle.matmul(wb, xq, xd, k, rows=rows)
    assert_within_tolerance(y_bal[:, rows], y64, S)
    assert_within_tolerance(y_plain[:, rows], y64, S)
    assert_within_tolerance(y_rp[:, rows], y64, S)
    assert np.array_equal(y_bal.view(np.uint32), y_again.view(np.uint32)), "not deterministic"
    # the raw and the repacked kernels share the schedule and the fold: bitwise equal
    assert np.array_equal(y_bal.view(np.uint32), y_rp.view(np.uint32))


def edge_and_sampled_rows(n, count, tail=40):
    """A seeded sample of weight rows plus the last `tail` rows (the ragged last tile)."""
    rows = np.union1d(sample_rows(n, count), np.arange(max(0, n - tail), n))
    return rows.astype(np.int64)


@pytest.mark.parametrize("repacked", [False, True])
def test_gemm_block_dots_full_shape_sampled(repacked):
    """m = 512, 4096 -> 5152 (164 tiles, the last one ragged): the production block dots of the
    raw and the repacked GEMM at full size, exact on a seeded row sample and the last rows."""
    ensure_built()
    m, n, k = 512, 5152, 4096
    _, x, wb, xq, _ = problem(m, n, k, "token_scales")
    xqh, _ = q8.quantize_q8_1_mmq(cuda(x))
    D = torch.full((m, n, k // 32), -7, dtype=torch.int32, device="cuda")
    if repacked:
        wq16, wdt = q8.repack_q8_0(cuda(wb), n, k)
        q8.check(q8.q8act_debug_gemm_repacked_block_dots(wq16, wdt, xqh, D, m, n, k))
    else:
        q8.check(q8.q8act_debug_gemm_block_dots(cuda(wb), xqh, D, m, n, k))
    device_ok()
    rows = edge_and_sampled_rows(n, 256)
    got = host(D[:, torch.from_numpy(rows).cuda(), :])
    assert np.array_equal(got, oracle.block_dots(wb, xq, k, rows=rows))


@pytest.mark.parametrize("m,n", [(512, 4096), (512, 5152), (512, 20480), (2048, 20480), (512, 64448),
                                 (2048, 64448)])
def test_gemm_serving_shapes_sampled(m, n):
    """The prefill shapes at full size: every token, a seeded sample of weight rows."""
    ensure_built()
    k = 4096
    _, x, wb, xq, xd = problem(m, n, k, "token_scales" if n > 5152 else "normal")
    y = host(q8.gemm_q8_0(cuda(wb), cuda(x), n))
    device_ok()
    rows = sample_rows(n, 256)
    _, y64, S = oracle.matmul(wb, xq, xd, k, rows=rows)
    assert_within_tolerance(y[:, rows], y64, S)
    again = host(q8.gemm_q8_0(cuda(wb), cuda(x), n))
    assert np.array_equal(again.view(np.uint32), y.view(np.uint32)), "not deterministic"
