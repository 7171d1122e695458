"""GB300 (sm_103a) Q8_0 weight x q8_1 activation block-quantized matmul.

The compute lives in libq8act.so (hand-written CUDA kernels behind the C ABI of
include/q8act.h).  This package is its Python face:

  * the raw ABI under the C names (``q8act_quantize_q8_1``, ``q8act_gemv_q8_0``, ...), which
    take torch tensors or integer device addresses and return the C return code;
  * torch conveniences (``quantize_q8_1``, ``gemv_q8_0``, ``gemm_q8_0``, ...) that allocate
    outputs with torch on the input's device, call the ABI on torch's current stream and
    raise ``Q8ActError`` on a non-zero return code.

There is no CPU or PyTorch fallback: without the built library every call raises.
"""
from __future__ import annotations

from ._lib import (  # noqa: F401  (re-exported ABI)
    EXPORTED, LIB_PATH, Q8ACT_ERR_ALIGN, Q8ACT_ERR_CUDA_BASE, Q8ACT_ERR_DEVICE, Q8ACT_ERR_DIMS,
    Q8ACT_ERR_NULL, Q8ACT_ERR_TIMEOUT, Q8ACT_ERR_WORKSPACE, Q8ACT_GEMV_MAX_M, Q8ACT_MAX_K,
    Q8ACT_NOALLOC_WS_BYTES, Q8ACT_GEMM_SPLIT_BYTES, Q8ACT_OK, Q8ActError, check, lib, q8act_debug_gemm_block_dots, q8act_debug_gemv_block_dots,
    q8act_dequant_q8_0_f16, q8act_device_status, q8act_gemm_q8_0, q8act_gemm_q8_0_preq,
    q8act_gemm_q8_0_noalloc, q8act_gemm_workspace_bytes, q8act_gemv_q8_0, q8act_mmq_ldm, q8act_quantize_q8_0,
    q8act_quantize_q8_1, q8act_quantize_q8_1_mmq, q8act_strerror, q8act_version, strerror,
    q8act_repack_q8_0, q8act_repack_ldn, q8act_gemm_q8_0_repacked, q8act_debug_gemm_repacked_block_dots,
    q8act_gemv_q8_0_group, Q8ACT_GEMV_MAX_GROUP, q8act_quantize_q4_0, q8act_dequant_q4_0_f16,
    q8act_gemv_q4_0, q8act_debug_gemv_q4_0_block_dots, q8act_gemv_workspace_bytes, q8act_gemv_q8_0_f32,
    q8act_debug_wait_timeout, Q8ACT_ERR_DRAIN_TIMEOUT, Q8ACT_GEMV_KQ_MAX_M,
    q8act_dequant_q6_k_f16, q8act_dequant_q4_k_f16, q8act_dequant_q5_k_f16,
    q8act_gemv_q6_k, q8act_gemv_q4_k, q8act_gemv_q5_k,
    q8act_debug_gemv_q6_k_block_dots, q8act_debug_gemv_q4_k_block_dots, q8act_debug_gemv_q5_k_block_dots)

QK = 32
Q8_0_BYTES = 34
Q4_0_BYTES = 18


def row_bytes(k: int) -> int:
    """Bytes of one Q8_0 row of k values (k/32 blocks of 34 bytes)."""
    return k // QK * Q8_0_BYTES


def quantize_q8_0(w):
    """f32 [n, k] CUDA tensor -> Q8_0 bytes, uint8 [n, k/32*34]."""
    import torch
    n, k = w.shape
    out = torch.empty((n, row_bytes(k)), dtype=torch.uint8, device=w.device)
    check(q8act_quantize_q8_0(w, out, n, k), "q8act_quantize_q8_0")
    return out


def quantize_q8_1(x):
    """f32 [m, k] -> (xq int8 [m, k], xd f32 [m, k/32])."""
    import torch
    m, k = x.shape
    xq = torch.empty((m, k), dtype=torch.int8, device=x.device)
    xd = torch.empty((m, k // QK), dtype=torch.float32, device=x.device)
    check(q8act_quantize_q8_1(x, xq, xd, m, k), "q8act_quantize_q8_1")
    return xq, xd


def quantize_q8_1_mmq(x):
    """f32 [m, k] -> (xqh uint16 [m, k] binary16 quants, xdt f32 [k/32, ldm] scales)."""
    import torch
    m, k = x.shape
    xqh = torch.empty((m, k), dtype=torch.uint16, device=x.device)
    xdt = torch.empty((k // QK, q8act_mmq_ldm(m)), dtype=torch.float32, device=x.device)
    check(q8act_quantize_q8_1_mmq(x, xqh, xdt, m, k), "q8act_quantize_q8_1_mmq")
    return xqh, xdt


def gemv_q8_0(w, xq, xd, n: int, out=None):
    """Decode GEMV: Q8_0 bytes w (n rows), q8_1 activation (xq, xd) of m <= Q8ACT_GEMV_MAX_M (15) tokens."""
    import torch
    m, k = xq.shape
    y = out if out is not None else torch.empty((m, n), dtype=torch.float32, device=xq.device)
    check(q8act_gemv_q8_0(w, xq, xd, y, m, n, k), "q8act_gemv_q8_0")
    return y


def gemv_q8_0_group(ws, xq, xd, ns, outs=None):
    """Grouped decode GEMV: weight matrices ws (Q8_0 bytes of ns[i] rows each) sharing the
    q8_1 activation (xq, xd) of m tokens, one launch; returns the list of outputs."""
    import torch
    m, k = xq.shape
    ys = outs if outs is not None else [torch.empty((m, n), dtype=torch.float32, device=xq.device) for n in ns]
    check(q8act_gemv_q8_0_group(ws, ys, ns, xq, xd, m, k), "q8act_gemv_q8_0_group")
    return ys


def gemm_workspace(m: int, k: int, device):
    import torch
    nbytes = q8act_gemm_workspace_bytes(m, k)
    if nbytes == 0:
        raise Q8ActError(Q8ACT_ERR_DIMS, "q8act_gemm_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def gemm_q8_0(w, x, n: int, ws=None, out=None):
    """Prefill GEMM with the q8_1 quantization of x fused into the call."""
    import torch
    m, k = x.shape
    if ws is None:
        ws = gemm_workspace(m, k, x.device)
    y = out if out is not None else torch.empty((m, n), dtype=torch.float32, device=x.device)
    check(q8act_gemm_q8_0(w, x, y, m, n, k, ws, ws.numel()), "q8act_gemm_q8_0")
    return y


def gemm_q8_0_preq(w, xqh, xdt, n: int, out=None):
    """Prefill GEMM on an activation already in the MMQ layout (quantize_q8_1_mmq)."""
    import torch
    m, k = xqh.shape
    y = out if out is not None else torch.empty((m, n), dtype=torch.float32, device=xqh.device)
    check(q8act_gemm_q8_0_preq(w, xqh, xdt, y, m, n, k), "q8act_gemm_q8_0_preq")
    return y


def repack_q8_0(w, n: int, k: int):
    """Load-time repack of Q8_0 bytes for the tensor-core GEMM: (wq16 float16 [n, k] holding
    the exact quants, wdt float32 [k/32, q8act_repack_ldn(n)] holding the block scales)."""
    import torch
    wq16 = torch.empty((n, k), dtype=torch.float16, device=w.device)
    wdt = torch.zeros((k // QK, q8act_repack_ldn(n)), dtype=torch.float32, device=w.device)
    check(q8act_repack_q8_0(w, wq16, wdt, n, k), "q8act_repack_q8_0")
    return wq16, wdt


def gemm_q8_0_repacked(wq16, wdt, x, ws=None, out=None):
    """Prefill GEMM (q8_1 quantization fused) on repacked weights (repack_q8_0)."""
    import torch
    m, k = x.shape
    n = wq16.shape[0]
    if ws is None:
        ws = gemm_workspace(m, k, x.device)
    y = out if out is not None else torch.empty((m, n), dtype=torch.float32, device=x.device)
    check(q8act_gemm_q8_0_repacked(wq16, wdt, x, y, m, n, k, ws, ws.numel()), "q8act_gemm_q8_0_repacked")
    return y


def dequant_q8_0_f16(w, n: int, k: int, out=None):
    """Q8_0 bytes -> row-major float16 [n, k]."""
    import torch
    w16 = out if out is not None else torch.empty((n, k), dtype=torch.float16, device=w.device)
    check(q8act_dequant_q8_0_f16(w, w16, n, k), "q8act_dequant_q8_0_f16")
    return w16


def device_status(stream=None) -> None:
    """Synchronize and raise if a kernel recorded a pipeline timeout since the last check."""
    check(q8act_device_status(stream), "q8act_device_status")


def row_bytes_q4_0(k: int) -> int:
    """Bytes of one Q4_0 row of k values (k/32 blocks of 18 bytes)."""
    return k // QK * Q4_0_BYTES


def quantize_q4_0(w):
    """f32 [n, k] CUDA tensor -> Q4_0 bytes, uint8 [n, k/32*18] (data preparation)."""
    import torch
    n, k = w.shape
    out = torch.empty((n, row_bytes_q4_0(k)), dtype=torch.uint8, device=w.device)
    check(q8act_quantize_q4_0(w, out, n, k), "q8act_quantize_q4_0")
    return out


def dequant_q4_0_f16(w, n: int, k: int, out=None):
    """Q4_0 bytes -> row-major float16 [n, k]."""
    import torch
    w16 = out if out is not None else torch.empty((n, k), dtype=torch.float16, device=w.device)
    check(q8act_dequant_q4_0_f16(w, w16, n, k), "q8act_dequant_q4_0_f16")
    return w16


def gemv_q4_0(w, xq, xd, n: int, out=None):
    """Q4_0 weights x pre-quantized q8_1 activation: y f32 [m, n] (1 <= m <= 15)."""
    import torch
    m, k = xq.shape
    y = out if out is not None else torch.empty((m, n), dtype=torch.float32, device=xq.device)
    check(q8act_gemv_q4_0(w, xq, xd, y, m, n, k), "q8act_gemv_q4_0")
    return y


def gemv_workspace(m: int, k: int, device):
    """A workspace for the fused GEMV (q8act_gemv_q8_0_f32)."""
    import torch
    nbytes = q8act_gemv_workspace_bytes(m, k)
    if nbytes == 0:
        raise Q8ActError(Q8ACT_ERR_DIMS, "q8act_gemv_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def gemv_q8_0_f32(w, x, n: int, ws=None, out=None):
    """Decode GEMV with the q8_1 quantization fused: f32 x [m, k] -> y f32 [m, n]."""
    import torch
    m, k = x.shape
    if ws is None:
        ws = gemv_workspace(m, k, x.device)
    y = out if out is not None else torch.empty((m, n), dtype=torch.float32, device=x.device)
    check(q8act_gemv_q8_0_f32(w, x, y, m, n, k, ws, ws.numel()), "q8act_gemv_q8_0_f32")
    return y


KQ_BYTES = {"q6_k": 210, "q4_k": 144, "q5_k": 176}   # bytes per 256-weight superblock


def dequant_kq_f16(fmt: str, w, n: int, k: int, out=None):
    """K-quant superblocks (fmt "q6_k", "q4_k" or "q5_k") -> row-major float16 [n, k]."""
    import torch
    w16 = out if out is not None else torch.empty((n, k), dtype=torch.float16, device=w.device)
    fn = {"q6_k": q8act_dequant_q6_k_f16, "q4_k": q8act_dequant_q4_k_f16, "q5_k": q8act_dequant_q5_k_f16}[fmt]
    check(fn(w, w16, n, k), f"q8act_dequant_{fmt}_f16")
    return w16


def gemv_kq(fmt: str, w, xq, xd, n: int, out=None):
    """Decode GEMV over K-quant weights (n rows) with the q8_1 activation of m <= 8 tokens."""
    import torch
    m, k = xq.shape
    y = out if out is not None else torch.empty((m, n), dtype=torch.float32, device=xq.device)
    fn = {"q6_k": q8act_gemv_q6_k, "q4_k": q8act_gemv_q4_k, "q5_k": q8act_gemv_q5_k}[fmt]
    check(fn(w, xq, xd, y, m, n, k), f"q8act_gemv_{fmt}")
    return y
