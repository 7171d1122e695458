"""GPU Q4_0 path vs the oracle: the writer's bytes, the fp16 dequant and the GEMV's block
dots bit for bit, the GEMV's outputs within 1e-5 * S of the oracle, and decode == verify
(token t's output bitwise the same for every m)."""
import numpy as np
import pytest
import torch

import oracle
import q8_block_quantized_act_gb300 as q8
from q8_block_quantized_act_gb300 import inputs
from gpu_util import assert_within_tolerance, cuda, device_ok, ensure_built, host, sample_rows

pytestmark = pytest.mark.gpu


def q4_problem(m, n, k, kind="normal"):
    """Seeded f32 weights/activations, the oracle's Q4_0 weights and q8_1 activation."""
    w = inputs.weights_f32(n, k, seed=0)
    x = inputs.activations_f32(m, k, kind=kind, seed=1)
    wb = oracle.quantize_q4_0(w)
    xq, xd = oracle.quantize_q8_1(x)
    return w, x, wb, xq, xd


@pytest.mark.parametrize("n,k", [(1, 256), (37, 768), (512, 4096)])
def test_q4_0_writer_bytes(n, k):
    ensure_built()
    w = inputs.weights_f32(n, k, seed=3)
    w[0, :32] = 0.0                                            # a zero block
    w[-1, 32:64] = (np.arange(32, dtype=np.float32) - 15.5)   # a ramp over the full range
    w[-1, 64:96] = np.float32(np.nan)                          # out of contract: quantizes to 0
    got = host(q8.quantize_q4_0(cuda(w)))
    device_ok()
    assert np.array_equal(got, oracle.quantize_q4_0(w))


@pytest.mark.parametrize("n,k", [(1, 256), (13, 768), (300, 4096), (4096, 4096), (7, 65536)])
def test_q4_0_dequant_bit_exact(n, k):
    ensure_built()
    _, _, wb, _, _ = q4_problem(1, n, k)
    got = host(q8.dequant_q4_0_f16(cuda(wb), n, k)).view(np.uint16)
    device_ok()
    assert np.array_equal(got, oracle.dequant_q4_0_f16(wb, k))


@pytest.mark.parametrize("m,n,k", [(1, 64, 256), (3, 200, 1280), (5, 40, 1280), (8, 129, 4096), (15, 40, 2048)])
def test_q4_0_gemv_block_dots_exact(m, n, k):
    ensure_built()
    _, _, wb, xq, _ = q4_problem(m, n, k, "outliers")
    D = torch.full((m, n, k // 32), -7, dtype=torch.int32, device="cuda")
    q8.check(q8.q8act_debug_gemv_q4_0_block_dots(cuda(wb), cuda(xq), D, m, n, k))
    device_ok()
    assert np.array_equal(host(D), oracle.block_dots_q4_0(wb, xq, k))


@pytest.mark.parametrize("m,n,k,kind", [
    (1, 512, 256, "normal"),
    (2, 5152, 4096, "outliers"),
    (8, 1000, 1280, "token_scales"),     # k = 5 groups: the shared-memory reduction path
    (15, 77, 4096, "normal"),
    (5, 333, 1280, "outliers"),          # the tensor-core kernel's first m; 5 groups, ragged n
    (11, 50, 6144, "token_scales"),      # two token groups, 24 groups per row
])
def test_q4_0_gemv_matches_oracle(m, n, k, kind):
    ensure_built()
    _, _, wb, xq, xd = q4_problem(m, n, k, kind)
    y = host(q8.gemv_q4_0(cuda(wb), cuda(xq), cuda(xd), n))
    device_ok()
    _, y64, S = oracle.matmul_q4_0(wb, xq, xd, k)
    assert_within_tolerance(y, y64, S)


@pytest.mark.parametrize("n,k", [(4096, 4096), (64448, 4096)])
def test_q4_0_gemv_serving_shapes_batch_invariant(n, k):
    """decode == verify for Q4_0, determinism, and a seeded sample of rows at full size."""
    ensure_built()
    mmax = q8.Q8ACT_GEMV_MAX_M
    _, _, wb, xq, xd = q4_problem(mmax, n, k)
    w_d = cuda(wb)
    ys = {m: host(q8.gemv_q4_0(w_d, cuda(xq[:m]), cuda(xd[:m]), n)) for m in (mmax, 8, 4, 2, 1)}
    device_ok()
    for m in (8, 4, 2, 1):
        assert np.array_equal(ys[m].view(np.uint32), ys[mmax][:m].view(np.uint32)), f"m={m}"
    again = host(q8.gemv_q4_0(w_d, cuda(xq), cuda(xd), n))
    assert np.array_equal(again.view(np.uint32), ys[mmax].view(np.uint32)), "not deterministic"
    rows = sample_rows(n, 1024)
    _, y64, S = oracle.matmul_q4_0(wb, xq, xd, k, rows=rows)
    assert_within_tolerance(ys[mmax][:, rows], y64, S)
