"""GPU quantizers and dequant vs the oracle: bit-exact quants, scales, bytes and fp16."""
import numpy as np
import pytest
import torch

import oracle
import q8_block_quantized_act_gb300 as q8
from gpu_util import cuda, device_ok, ensure_built, host
from oracle_pins import _block
import json, os

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def edge_rows(k):
    """Rows exercising ties, zero blocks, sign-dominant blocks, and extreme magnitudes."""
    g = json.load(open(os.path.join(GOLDEN, "q8_1_worked_cases.json")))
    golden = np.concatenate([_block(c["x"]) for c in g["cases"]])
    rows = []
    rng = np.random.Generator(np.random.PCG64(21))
    for scale in (1.0, 1e-30, 1e30, 2.0 ** -140, 3.0e-39):
        r = rng.standard_normal(k).astype(np.float32) * np.float32(scale)
        r[: golden.size] = golden[:k] * np.float32(scale if scale < 1e29 else 1.0)
        r[64:96] = 0.0
        rows.append(r)
    r = np.zeros(k, np.float32)
    r[5] = -7.0
    rows.append(r)
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("m,k,kind", [(1, 256, "normal"), (3, 4096, "outliers"),
                                      (37, 1280, "normal"), (512, 4096, "token_scales"),
                                      (2048, 4096, "token_scales")])
def test_quantize_q8_1_bit_exact(m, k, kind):
    ensure_built()
    from q8_block_quantized_act_gb300 import inputs
    x = inputs.activations_f32(m, k, kind=kind)
    xq_ref, xd_ref = oracle.quantize_q8_1(x)
    xq, xd = q8.quantize_q8_1(cuda(x))
    device_ok()
    assert np.array_equal(host(xq), xq_ref)
    assert np.array_equal(host(xd).view(np.uint32), xd_ref.view(np.uint32))


def test_quantize_q8_1_edge_cases():
    ensure_built()
    x = edge_rows(256)
    xq_ref, xd_ref = oracle.quantize_q8_1(x)
    xq, xd = q8.quantize_q8_1(cuda(x))
    device_ok()
    assert np.array_equal(host(xq), xq_ref)
    assert np.array_equal(host(xd).view(np.uint32), xd_ref.view(np.uint32))
    assert np.all(np.isfinite(host(xd)))


def test_quantize_nonfinite_inputs():
    """NaN and infinite entries are out of contract: no fault, and the same quants and scales
    as the oracle (NaN entries quantize to 0; a block with an infinity gets d = inf, q = 0)."""
    ensure_built()
    x = edge_rows(256)
    x[0, 3] = np.nan
    x[0, 40] = np.nan
    x[1, 100] = np.inf
    x[2, 200] = -np.inf
    x[3, 128:160] = np.nan               # a whole block of NaNs (d = 0)
    x[3, 7] = np.nan                     # and one NaN in an otherwise finite block
    xq_ref, xd_ref = oracle.quantize_q8_1(x)
    xq, xd = q8.quantize_q8_1(cuda(x))
    xqh, xdt = q8.quantize_q8_1_mmq(cuda(x))
    device_ok()
    assert np.array_equal(host(xq), xq_ref)
    assert np.array_equal(host(xd).view(np.uint32), xd_ref.view(np.uint32))
    assert np.array_equal(host(xqh).view(np.float16).astype(np.float32), xq_ref.astype(np.float32))
    assert np.array_equal(host(xdt)[:, :x.shape[0]].T.copy().view(np.uint32), xd_ref.view(np.uint32))


@pytest.mark.parametrize("m,k", [(1, 256), (5, 512), (130, 4096), (512, 4096)])
def test_quantize_q8_1_mmq_layout(m, k):
    ensure_built()
    from q8_block_quantized_act_gb300 import inputs
    x = inputs.activations_f32(m, k, kind="token_scales")
    xq_ref, xd_ref = oracle.quantize_q8_1(x)
    xqh, xdt = q8.quantize_q8_1_mmq(cuda(x))
    device_ok()
    vals = host(xqh).view(np.float16).astype(np.float32)
    assert np.array_equal(vals, xq_ref.astype(np.float32))
    ldm = q8.q8act_mmq_ldm(m)
    assert xdt.shape == (k // 32, ldm)
    assert np.array_equal(host(xdt)[:, :m].T.copy().view(np.uint32), xd_ref.view(np.uint32))


@pytest.mark.parametrize("n,k", [(1, 256), (512, 256), (77, 1280), (4096, 4096)])
def test_quantize_q8_0_bit_exact(n, k):
    ensure_built()
    from q8_block_quantized_act_gb300 import inputs
    w = inputs.weights_f32(n, k)
    ref = oracle.quantize_q8_0(w)
    got = q8.quantize_q8_0(cuda(w))
    device_ok()
    assert np.array_equal(host(got), ref)


def test_quantize_q8_0_edge_cases():
    ensure_built()
    w = edge_rows(256) * np.float32(1e-3)
    ref = oracle.quantize_q8_0(w.astype(np.float32))
    got = q8.quantize_q8_0(cuda(w.astype(np.float32)))
    device_ok()
    assert np.array_equal(host(got), ref)


@pytest.mark.parametrize("n,k", [(1, 256), (13, 512), (4096, 4096), (5152, 4096)])
def test_dequant_f16_bit_exact(n, k):
    ensure_built()
    from q8_block_quantized_act_gb300 import inputs
    w = inputs.weights_f32(n, k)
    wb = oracle.quantize_q8_0(w)
    ref = oracle.dequant_f16(wb, k)
    got = q8.dequant_q8_0_f16(cuda(wb), n, k)
    device_ok()
    assert np.array_equal(host(got).view(np.uint16), ref)


def test_dequant_f16_extreme_scales():
    """Scales near the binary16 limits: products that overflow to inf or round to subnormals."""
    ensure_built()
    rng = np.random.Generator(np.random.PCG64(5))
    n, k = 64, 256
    wb = oracle.quantize_q8_0(rng.standard_normal((n, k)).astype(np.float32))
    blocks = wb.reshape(n, k // 32, 34)
    scales = rng.integers(0, 0x7c00, size=(n, k // 32), dtype=np.uint16)   # any finite binary16
    blocks[:, :, 0:2] = scales.view(np.uint8).reshape(n, k // 32, 2)
    ref = oracle.dequant_f16(wb, k)
    got = q8.dequant_q8_0_f16(cuda(wb), n, k)
    device_ok()
    assert np.array_equal(host(got).view(np.uint16), ref)
