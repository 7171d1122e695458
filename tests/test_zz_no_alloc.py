"""q8act_gemm_q8_0_noalloc: the fused GEMM for callers that cannot allocate device memory.

Such callers (an allocator's own hooks, a serving loop that forbids allocation after
start-up, a runtime that only passes buffers it owns) cannot hand q8act_gemm_q8_0 a
workspace; this entry point uses the library's fixed device scratch instead.  The test calls
it through the C ABI twice in a row with different activations and compares each result with
the workspace entry point's on the same inputs, within the tolerance the parity tests use
(|y - y_ref| <= 1e-5 * S, S = sum_b |d_w d_a D| from the oracle).  It lives in a file that
pytest collects last and passes both alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
import q8_block_quantized_act_gb300 as q8
from gpu_util import RTOL, assert_within_tolerance, cuda, ensure_built, host, problem, sample_rows


@pytest.mark.gpu
def test_noalloc_gemm_matches_workspace_gemm_twice():
    ensure_built()
    m, n, k = 300, 520, 2048
    _, x1, wb, _, _ = problem(m, n, k, "token_scales", xseed=1)
    x2 = problem(m, n, k, "outliers", xseed=7)[1]
    w_d = cuda(wb)
    ws = q8.gemm_workspace(m, k, w_d.device)
    for x in (x1, x2):
        x_d = cuda(x)
        y_ref = torch.empty((m, n), dtype=torch.float32, device="cuda")
        y_na = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        q8.check(q8.q8act_gemm_q8_0(w_d, x_d, y_ref, m, n, k, ws, ws.numel()))
        q8.check(q8.q8act_gemm_q8_0_noalloc(w_d, x_d, y_na, m, n, k))
        torch.cuda.synchronize()
        q8.device_status()
        xq, xd = oracle.quantize_q8_1(x)
        _, y64, S = oracle.matmul(wb, xq, xd, k)
        a, b = host(y_na), host(y_ref)
        err = np.abs(a.astype(np.float64) - b.astype(np.float64))
        assert np.all(err <= RTOL * S), float((err / np.maximum(S, 1e-300)).max())
        assert_within_tolerance(a, y64, S)


@pytest.mark.gpu
@pytest.mark.parametrize("m", [1024, 2891])
def test_noalloc_gemm_prefill_sizes(m):
    """Prefill sizes where the split region no longer fits beside the quantized activation
    (every tile then done by one CTA), up to the largest m the scratch holds at k = 4096: the
    result matches the workspace entry point's within the parity tolerance, twice in a row."""
    ensure_built()
    n, k = 640, 4096
    _, x1, wb, _, _ = problem(m, n, k, "token_scales", xseed=1)
    x2 = problem(m, n, k, "outliers", xseed=5)[1]
    w_d = cuda(wb)
    ws = q8.gemm_workspace(m, k, w_d.device)
    rows = sample_rows(n, 96)
    for x in (x1, x2):
        x_d = cuda(x)
        y_ref = torch.empty((m, n), dtype=torch.float32, device="cuda")
        y_na = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        q8.check(q8.q8act_gemm_q8_0(w_d, x_d, y_ref, m, n, k, ws, ws.numel()))
        q8.check(q8.q8act_gemm_q8_0_noalloc(w_d, x_d, y_na, m, n, k))
        torch.cuda.synchronize()
        q8.device_status()
        xq, xd = oracle.quantize_q8_1(x)
        _, y64, S = oracle.matmul(wb, xq, xd, k, rows=rows)
        a, b = host(y_na)[:, rows], host(y_ref)[:, rows]
        err = np.abs(a.astype(np.float64) - b.astype(np.float64))
        assert np.all(err <= RTOL * S), float((err / np.maximum(S, 1e-300)).max())
        assert_within_tolerance(a, y64, S)


@pytest.mark.gpu
def test_noalloc_gemm_refuses_beyond_its_scratch():
    ensure_built()
    k = 4096
    # the quantized activation must fit in the scratch (the split region is optional)
    m_ok = max(mm for mm in range(2800, 3000)
               if q8.q8act_gemm_workspace_bytes(mm, k) - q8.Q8ACT_GEMM_SPLIT_BYTES <= q8.Q8ACT_NOALLOC_WS_BYTES)
    assert m_ok == 2891
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    rc = q8.q8act_gemm_q8_0_noalloc(dummy, dummy, dummy, m_ok + 1, 64, k)
    assert rc == q8.Q8ACT_ERR_WORKSPACE
