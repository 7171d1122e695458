"""GPU K-quant superblocks (GGUF Q6_K 210 B, Q4_K 144 B, Q5_K 176 B) vs the oracle: the fp16
mirror bit for bit (including the hand-built golden superblocks), the GEMV's exact per-block
integers, its outputs within 1e-5 * S, and bitwise decode == verify across m."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import q8_block_quantized_act_gb300 as q8
from q8_block_quantized_act_gb300 import inputs
from gpu_util import assert_within_tolerance, cuda, device_ok, ensure_built, host, sample_rows

pytestmark = pytest.mark.gpu

FORMATS = ("q6_k", "q4_k", "q5_k")
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kquant_superblocks.json")


def kq_problem(fmt, m, n, k, kind="normal", seed=0):
    wb = inputs.kquant_superblocks(fmt, n, k, seed=seed)
    x = inputs.activations_f32(m, k, kind=kind)
    xq, xd = oracle.quantize_q8_1(x)
    return wb, xq, xd


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("n,k", [(8, 256), (130, 1280), (33, 4096), (1000, 4096), (17, 2304)])
def test_kq_dequant_bit_exact(fmt, n, k):
    """Ragged shapes included: Q6_K rows of 1280 and 2304 weights are not 16-byte multiples."""
    ensure_built()
    wb = inputs.kquant_superblocks(fmt, n, k, seed=3)
    w16 = host(q8.dequant_kq_f16(fmt, cuda(wb), n, k))
    device_ok()
    assert np.array_equal(w16.view(np.uint16), oracle.dequant_kq_f16(fmt, wb, k))


@pytest.mark.parametrize("fmt", FORMATS)
def test_kq_dequant_bit_exact_any_finite_scales(fmt):
    """Scale fields (d, dmin) drawn from every finite binary16 pattern: both signs, zeros,
    subnormals, exponent gaps of any width between d and dmin (the mirror takes one exact FMA
    for close exponents and a rounding to odd otherwise), products beyond the binary16 range."""
    ensure_built()
    n, k = 600, 4096
    nbytes, offsets = inputs.KQUANT_LAYOUT[fmt]
    wb = inputs.kquant_superblocks(fmt, n, k, seed=9)
    sb = wb.reshape(-1, nbytes)
    rng = np.random.default_rng(1234)
    for off in offsets:
        bits = rng.integers(0, 65536, size=sb.shape[0]).astype(np.uint32)
        bits = (bits & 0x83FF) | (rng.integers(0, 31, size=sb.shape[0]).astype(np.uint32) << 10)
        sb[:, off] = (bits & 0xFF).astype(np.uint8)
        sb[:, off + 1] = (bits >> 8).astype(np.uint8)
    wb = sb.reshape(n, -1)
    w16 = host(q8.dequant_kq_f16(fmt, cuda(wb), n, k))
    device_ok()
    assert np.array_equal(w16.view(np.uint16), oracle.dequant_kq_f16(fmt, wb, k))


def test_kq_dequant_golden_superblocks():
    """The hand-built superblocks: the GPU mirror carries the hand-worked binary16 values."""
    ensure_built()
    for sb in json.load(open(GOLDEN))["superblocks"]:
        wb = np.frombuffer(bytes.fromhex(sb["bytes"]), dtype=np.uint8).reshape(1, -1).copy()
        h = host(q8.dequant_kq_f16(sb["format"], cuda(wb), 1, 256)).view(np.uint16)[0]
        device_ok()
        for w in sb["worked"]:
            if "f16" in w:
                assert int(h[w["e"]]) == int(w["f16"], 16), (sb["format"], w["e"])
        assert np.array_equal(h, oracle.dequant_kq_f16(sb["format"], wb, 256)[0])


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("m,n,k", [(1, 64, 256), (2, 77, 1280), (5, 300, 4096), (8, 130, 2048)])
def test_kq_gemv_block_integers_exact(fmt, m, n, k):
    ensure_built()
    wb, xq, _ = kq_problem(fmt, m, n, k, "outliers")
    D = torch.full((m, n, k // 32), -7, dtype=torch.int32, device="cuda")
    fn = {"q6_k": q8.q8act_debug_gemv_q6_k_block_dots, "q4_k": q8.q8act_debug_gemv_q4_k_block_dots,
          "q5_k": q8.q8act_debug_gemv_q5_k_block_dots}[fmt]
    q8.check(fn(cuda(wb), cuda(xq), D, m, n, k))
    device_ok()
    assert np.array_equal(host(D), oracle.block_dots_kq(fmt, wb, xq, k))


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("m", [1, 8])
def test_kq_gemv_block_integers_full_shape_sampled(fmt, m):
    """4096 -> 20493 (a serving width with a ragged last 16-row tile): the production block
    integers of the dp4a kernel (m = 1) and of the tensor-core kernel (m = 8), exact on a
    seeded row sample plus the last 40 rows."""
    ensure_built()
    n, k = 20493, 4096
    wb, xq, _ = kq_problem(fmt, m, n, k, "outliers")
    D = torch.full((m, n, k // 32), -7, dtype=torch.int32, device="cuda")
    fn = {"q6_k": q8.q8act_debug_gemv_q6_k_block_dots, "q4_k": q8.q8act_debug_gemv_q4_k_block_dots,
          "q5_k": q8.q8act_debug_gemv_q5_k_block_dots}[fmt]
    q8.check(fn(cuda(wb), cuda(xq), D, m, n, k))
    device_ok()
    rows = np.union1d(sample_rows(n, 256), np.arange(n - 40, n)).astype(np.int64)
    got = host(D[:, torch.from_numpy(rows).cuda(), :])
    assert np.array_equal(got, oracle.block_dots_kq(fmt, wb, xq, k, rows=rows))


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("m,n,k,kind", [(1, 512, 256, "normal"), (1, 4096, 4096, "outliers"),
                                         (3, 1000, 1280, "normal"), (4, 777, 4096, "token_scales"),
                                         (8, 300, 4096, "outliers"), (2, 1, 256, "normal")])
def test_kq_gemv_matches_oracle(fmt, m, n, k, kind):
    ensure_built()
    wb, xq, xd = kq_problem(fmt, m, n, k, kind)
    y = host(q8.gemv_kq(fmt, cuda(wb), cuda(xq), cuda(xd), n))
    device_ok()
    _, y64, S = oracle.matmul_kq(fmt, wb, xq, xd, k)
    assert_within_tolerance(y, y64, S)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("n,k", [(64448, 4096), (4096, 1280)])
def test_kq_gemv_serving_shapes_batch_invariant(fmt, n, k):
    """decode == verify: token t's output is bitwise the same for m = 1..8; sampled rows (with
    the ragged end) against the oracle."""
    ensure_built()
    wb, xq, xd = kq_problem(fmt, 8, n, k)
    w_d = cuda(wb)
    ys = {m: host(q8.gemv_kq(fmt, w_d, cuda(xq[:m]), cuda(xd[:m]), n)) for m in (8, 5, 4, 2, 1)}
    device_ok()
    for m in (5, 4, 2, 1):
        assert np.array_equal(ys[m].view(np.uint32), ys[8][:m].view(np.uint32)), m
    rows = np.union1d(sample_rows(n, 256), np.arange(n - 20, n)).astype(np.int64)
    _, y64, S = oracle.matmul_kq(fmt, wb, xq, xd, k, rows=rows)
    assert_within_tolerance(ys[8][:, rows], y64, S)


def test_kq_refusals():
    ensure_built()
    w = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    a = torch.zeros(4096, dtype=torch.int8, device="cuda")
    s = torch.zeros(4096, dtype=torch.float32, device="cuda")
    assert q8.q8act_gemv_q6_k(w, a, s, s, q8.Q8ACT_GEMV_KQ_MAX_M + 1, 8, 256) == q8.Q8ACT_ERR_DIMS
    assert q8.q8act_gemv_q4_k(w, a, s, s, 1, 8, 300) == q8.Q8ACT_ERR_DIMS
    assert q8.q8act_dequant_q5_k_f16(w, None, 8, 256) == q8.Q8ACT_ERR_NULL
