"""GPU GEMV (decode / verify, m = 1..15) vs the oracle: exact block dots, outputs within
1e-5 * S, bitwise batch invariance (decode == verify) and determinism."""
import numpy as np
import pytest
import torch

import oracle
import q8_block_quantized_act_gb300 as q8
from q8_block_quantized_act_gb300 import inputs
from gpu_util import (assert_within_tolerance, cuda, device_ok, ensure_built, host, problem,
                      sample_rows)

pytestmark = pytest.mark.gpu


def run_gemv(wb, xq, xd, n):
    return host(q8.gemv_q8_0(cuda(wb), cuda(xq), cuda(xd), n))


@pytest.mark.parametrize("m,n,k,kind", [
    (1, 512, 256, "normal"),          # tiny decode shape
    (1, 4096, 4096, "outliers"),      # o_proj
    (1, 5152, 4096, "outliers"),      # fused qkv (ragged chunk tail)
    (3, 1000, 1280, "normal"),        # short rows, ragged n, odd m
    (8, 777, 4096, "normal"),
    (2, 1, 256, "normal"),            # a single row
    (5, 33, 8192, "token_scales"),
    (9, 640, 4096, "outliers"),       # verify tier, K = 8 drafted tokens
    (12, 300, 2048, "token_scales"),
    (15, 1000, 4096, "normal"),       # largest m below the prefill threshold
    (15, 40, 10752, "normal"),        # largest k at m = 15 (shrunken chunks)
    (8, 24, 18688, "outliers"),       # largest k at m = 8
])
def test_gemv_matches_oracle(m, n, k, kind):
    ensure_built()
    _, _, wb, xq, xd = problem(m, n, k, kind)
    y = run_gemv(wb, xq, xd, n)
    device_ok()
    _, y64, S = oracle.matmul(wb, xq, xd, k)
    assert y.shape == (m, n)
    assert_within_tolerance(y, y64, S)


@pytest.mark.parametrize("m,n,k", [(1, 512, 256), (2, 77, 1280), (4, 300, 1280), (8, 130, 4096), (15, 70, 4096)])
def test_gemv_block_dots_exact(m, n, k):
    ensure_built()
    _, _, wb, xq, _ = problem(m, n, k)
    D = torch.zeros((m, n, k // 32), dtype=torch.int32, device="cuda")
    q8.check(q8.q8act_debug_gemv_block_dots(cuda(wb), cuda(xq), D, m, n, k))
    device_ok()
    assert np.array_equal(host(D), oracle.block_dots(wb, xq, k))


@pytest.mark.parametrize("m", [1, 8, 15])
def test_gemv_block_dots_full_shape_sampled(m):
    """4096 -> 64448 (the LM-head half; its last row chunk is ragged): the production block
    dots of the GEMV at full size -- dp4a at m = 1, int8 mma.sync at m = 8, binary16 mma.sync
    at m = 15 -- exact on a seeded row sample plus the last 40 rows."""
    ensure_built()
    n, k = 64448, 4096
    _, _, wb, xq, _ = problem(m, n, k, "outliers")
    D = torch.full((m, n, k // 32), -7, dtype=torch.int32, device="cuda")
    q8.check(q8.q8act_debug_gemv_block_dots(cuda(wb), cuda(xq), D, m, n, k))
    device_ok()
    rows = np.union1d(sample_rows(n, 256), np.arange(n - 40, n)).astype(np.int64)
    got = host(D[:, torch.from_numpy(rows).cuda(), :])
    assert np.array_equal(got, oracle.block_dots(wb, xq, k, rows=rows))


@pytest.mark.parametrize("n,k", [(4096, 4096), (4096, 1280), (20480, 4096), (64448, 4096)])
def test_gemv_serving_shapes_batch_invariant(n, k):
    """decode == verify: token t's output is bitwise the same for every m of the GEMV."""
    ensure_built()
    mmax = q8.Q8ACT_GEMV_MAX_M
    _, _, wb, xq, xd = problem(mmax, n, k)
    w_d = cuda(wb)
    ys = {}
    for m in (mmax, 12, 9, 8, 4, 2, 1):
        ys[m] = host(q8.gemv_q8_0(w_d, cuda(xq[:m]), cuda(xd[:m]), n))
    device_ok()
    for m in (12, 9, 8, 4, 2, 1):
        assert np.array_equal(ys[m].view(np.uint32), ys[mmax][:m].view(np.uint32)), f"m={m}"
    again = host(q8.gemv_q8_0(w_d, cuda(xq), cuda(xd), n))
    assert np.array_equal(again.view(np.uint32), ys[mmax].view(np.uint32)), "not deterministic"
    rows = sample_rows(n, 1024)
    _, y64, S = oracle.matmul(wb, xq, xd, k, rows=rows)
    assert_within_tolerance(ys[mmax][:, rows], y64, S)


@pytest.mark.parametrize("m,kmax", [(1, 65536), (8, 18688), (15, 10752)])
def test_gemv_k_limit(m, kmax):
    """The documented largest k per m is accepted and the next multiple of 256 is refused
    before any launch (the activation cache no longer fits beside two weight stages)."""
    ensure_built()
    _, _, wb, xq, xd = problem(m, 8, kmax)
    y = run_gemv(wb, xq, xd, 8)
    device_ok()
    _, y64, S = oracle.matmul(wb, xq, xd, kmax)
    assert_within_tolerance(y, y64, S)
    k = kmax + 256
    w = torch.zeros(8 * k // 32 * 34, dtype=torch.uint8, device="cuda")
    aq = torch.zeros((m, k), dtype=torch.int8, device="cuda")
    ad = torch.zeros((m, k // 32), dtype=torch.float32, device="cuda")
    out = torch.zeros((m, 8), dtype=torch.float32, device="cuda")
    rc = q8.q8act_gemv_q8_0(w, aq, ad, out, m, 8, k)
    assert rc == q8.Q8ACT_ERR_DIMS


@pytest.mark.parametrize("m,k,ns", [(1, 4096, (4096, 5152, 777)), (2, 1280, (4096, 33)),
                                    (4, 4096, (64, 4096, 20480, 1)), (9, 2048, (300, 200, 100)),
                                    # the largest group; 5 groups per row (64-row chunks), ragged sizes
                                    (12, 1280, (130, 64, 1, 777, 65, 200, 1000, 63))])
def test_gemv_group_equals_single_calls(m, k, ns):
    """One grouped launch gives each matrix bitwise the result of its own GEMV."""
    ensure_built()
    ws = [problem(m, n, k, wseed=10 + i)[2] for i, n in enumerate(ns)]
    _, _, _, xq, xd = problem(m, 8, k, "outliers")
    xq_d, xd_d = cuda(xq), cuda(xd)
    w_d = [cuda(wb) for wb in ws]
    ys = [host(t) for t in q8.gemv_q8_0_group(w_d, xq_d, xd_d, list(ns))]
    singles = [host(q8.gemv_q8_0(wd, xq_d, xd_d, n)) for wd, n in zip(w_d, ns)]
    device_ok()
    for i, (a, b) in enumerate(zip(ys, singles)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"matrix {i}"
    _, y64, S = oracle.matmul(ws[-1], xq, xd, k)
    assert_within_tolerance(ys[-1], y64, S)


@pytest.mark.parametrize("m,n,k", [(1, 64448, 4096), (2, 5152, 4096), (3, 4096, 1280), (8, 20480, 4096),
                                   (15, 777, 2048)])
def test_gemv_f32_equals_two_calls(m, n, k):
    """The fused decode call (q8_1 quantization, then the GEMV as its programmatic dependent)
    gives bitwise the y of the two separate calls, also when two fused calls run back to back
    on different activations; and it is within 1e-5 * S of the oracle."""
    ensure_built()
    w, x, wb, xq, xd = problem(m, n, k, "outliers")
    x2 = inputs.activations_f32(m, k, kind="token_scales", seed=7)
    w_d = cuda(wb)
    ws = q8.gemv_workspace(m, k, w_d.device)
    y1 = q8.gemv_q8_0_f32(w_d, cuda(x), n, ws=ws)
    y2 = q8.gemv_q8_0_f32(w_d, cuda(x2), n, ws=ws)       # reuses the workspace right away
    y1h, y2h = host(y1), host(y2)
    xq1, xd1 = q8.quantize_q8_1(cuda(x))
    ref1 = host(q8.gemv_q8_0(w_d, xq1, xd1, n))
    xq2, xd2 = q8.quantize_q8_1(cuda(x2))
    ref2 = host(q8.gemv_q8_0(w_d, xq2, xd2, n))
    device_ok()
    assert np.array_equal(y1h.view(np.uint32), ref1.view(np.uint32))
    assert np.array_equal(y2h.view(np.uint32), ref2.view(np.uint32))
    rows = sample_rows(n, 256)
    _, y64, S = oracle.matmul(wb, xq, xd, k, rows=rows)
    assert_within_tolerance(y1h[:, rows], y64, S)
