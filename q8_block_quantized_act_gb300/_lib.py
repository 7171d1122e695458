"""ctypes binding of libq8act.so: the C ABI of include/q8act.h under the same names.

Argument marshalling only.  Every q8act_* function here accepts, for each pointer argument,
a torch tensor (its data_ptr() is passed), a plain integer address, or None (NULL); and for
`stream`, a torch.cuda.Stream, an integer cudaStream_t, or None (torch's current stream on
the current device).  They return the C return code unchanged; `check(rc)` turns a non-zero
code into a Q8ActError.

The library must have been built (q8_block_quantized_act_gb300.build); loading fails loudly
otherwise -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libq8act.so")

Q8ACT_OK = 0
Q8ACT_ERR_NULL = -1
Q8ACT_ERR_DIMS = -2
Q8ACT_ERR_ALIGN = -3
Q8ACT_ERR_WORKSPACE = -4
Q8ACT_ERR_DEVICE = -5
Q8ACT_ERR_TIMEOUT = -6
Q8ACT_ERR_DRAIN_TIMEOUT = -7
Q8ACT_ERR_CUDA_BASE = 1000
Q8ACT_MAX_K = 65536
Q8ACT_GEMV_MAX_M = 15
Q8ACT_GEMV_MAX_GROUP = 8

EXPORTED = (
    "q8act_version", "q8act_strerror", "q8act_quantize_q8_1", "q8act_quantize_q8_1_mmq",
    "q8act_mmq_ldm", "q8act_quantize_q8_0", "q8act_gemv_q8_0", "q8act_gemm_workspace_bytes",
    "q8act_gemm_q8_0", "q8act_gemm_q8_0_preq", "q8act_dequant_q8_0_f16",
    "q8act_debug_gemv_block_dots", "q8act_debug_gemm_block_dots", "q8act_device_status",
    "q8act_gemm_q8_0_noalloc", "q8act_repack_q8_0", "q8act_repack_ldn",
    "q8act_gemm_q8_0_repacked", "q8act_debug_gemm_repacked_block_dots", "q8act_gemv_q8_0_group",
    "q8act_quantize_q4_0", "q8act_dequant_q4_0_f16", "q8act_gemv_q4_0", "q8act_debug_gemv_q4_0_block_dots",
    "q8act_gemv_workspace_bytes", "q8act_gemv_q8_0_f32", "q8act_debug_wait_timeout",
    "q8act_dequant_q6_k_f16", "q8act_dequant_q4_k_f16", "q8act_dequant_q5_k_f16",
    "q8act_gemv_q6_k", "q8act_gemv_q4_k", "q8act_gemv_q5_k",
    "q8act_debug_gemv_q6_k_block_dots", "q8act_debug_gemv_q4_k_block_dots", "q8act_debug_gemv_q5_k_block_dots",
)
Q8ACT_GEMV_KQ_MAX_M = 8
Q8ACT_NOALLOC_WS_BYTES = 24 << 20
Q8ACT_GEMM_SPLIT_BYTES = 320 * 65536 + 160 * 64


class Q8ActError(RuntimeError):
    def __init__(self, rc: int, what: str = ""):
        self.rc = rc
        super().__init__(f"{what}: q8act error {rc} ({strerror(rc)})" if what else
                         f"q8act error {rc} ({strerror(rc)})")


_LOCK = threading.Lock()
_LIB = None


def lib() -> ctypes.CDLL:
    """Load libq8act.so (once).  Raises if it has not been built."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libq8act.so not found at {LIB_PATH}; build it with "
                    "`python -m q8_block_quantized_act_gb300.build` (no CPU fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            sig = {
                "q8act_version": ([], I32),
                "q8act_strerror": ([I32], ctypes.c_char_p),
                "q8act_quantize_q8_1": ([P, P, P, I64, I64, P], I32),
                "q8act_quantize_q8_1_mmq": ([P, P, P, I64, I64, P], I32),
                "q8act_mmq_ldm": ([I64], I64),
                "q8act_quantize_q8_0": ([P, P, I64, I64, P], I32),
                "q8act_gemv_q8_0": ([P, P, P, P, I64, I64, I64, P], I32),
                "q8act_gemm_workspace_bytes": ([I64, I64], SZ),
                "q8act_gemm_q8_0": ([P, P, P, I64, I64, I64, P, SZ, P], I32),
                "q8act_gemm_q8_0_preq": ([P, P, P, P, I64, I64, I64, P], I32),
                "q8act_dequant_q8_0_f16": ([P, P, I64, I64, P], I32),
                "q8act_debug_gemv_block_dots": ([P, P, P, I64, I64, I64, P], I32),
                "q8act_debug_gemm_block_dots": ([P, P, P, I64, I64, I64, P], I32),
                "q8act_device_status": ([P], I32),
                "q8act_gemm_q8_0_noalloc": ([P, P, P, I64, I64, I64, P], I32),
                "q8act_repack_q8_0": ([P, P, P, I64, I64, P], I32),
                "q8act_repack_ldn": ([I64], I64),
                "q8act_gemm_q8_0_repacked": ([P, P, P, P, I64, I64, I64, P, SZ, P], I32),
                "q8act_debug_gemm_repacked_block_dots": ([P, P, P, P, I64, I64, I64, P], I32),
                "q8act_gemv_q8_0_group": ([P, P, P, I32, P, P, I64, I64, P], I32),
                "q8act_quantize_q4_0": ([P, P, I64, I64, P], I32),
                "q8act_dequant_q4_0_f16": ([P, P, I64, I64, P], I32),
                "q8act_gemv_q4_0": ([P, P, P, P, I64, I64, I64, P], I32),
                "q8act_debug_gemv_q4_0_block_dots": ([P, P, P, I64, I64, I64, P], I32),
                "q8act_gemv_workspace_bytes": ([I64, I64], SZ),
                "q8act_gemv_q8_0_f32": ([P, P, P, I64, I64, I64, P, SZ, P], I32),
                "q8act_debug_wait_timeout": ([I64, P], I32),
            }
            for f in ("q6_k", "q4_k", "q5_k"):
                sig[f"q8act_dequant_{f}_f16"] = ([P, P, I64, I64, P], I32)
                sig[f"q8act_gemv_{f}"] = ([P, P, P, P, I64, I64, I64, P], I32)
                sig[f"q8act_debug_gemv_{f}_block_dots"] = ([P, P, P, I64, I64, I64, P], I32)
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _LIB = L
    return _LIB


def _p(v):
    """Pointer argument: tensor -> data_ptr, int -> itself, None -> NULL."""
    if v is None:
        return None
    if isinstance(v, int):
        return v
    return v.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def strerror(rc: int) -> str:
    return lib().q8act_strerror(int(rc)).decode()


def check(rc: int, what: str = "") -> None:
    if rc != Q8ACT_OK:
        raise Q8ActError(rc, what)


def q8act_version() -> int:
    return lib().q8act_version()


def q8act_strerror(rc: int) -> str:
    return strerror(rc)


def q8act_quantize_q8_1(x, xq, xd, m, k, stream=None) -> int:
    return lib().q8act_quantize_q8_1(_p(x), _p(xq), _p(xd), m, k, _s(stream))


def q8act_quantize_q8_1_mmq(x, xqh, xdt, m, k, stream=None) -> int:
    return lib().q8act_quantize_q8_1_mmq(_p(x), _p(xqh), _p(xdt), m, k, _s(stream))


def q8act_mmq_ldm(m) -> int:
    return lib().q8act_mmq_ldm(m)


def q8act_quantize_q8_0(w, wq, n, k, stream=None) -> int:
    return lib().q8act_quantize_q8_0(_p(w), _p(wq), n, k, _s(stream))


def q8act_gemv_q8_0(w, xq, xd, y, m, n, k, stream=None) -> int:
    return lib().q8act_gemv_q8_0(_p(w), _p(xq), _p(xd), _p(y), m, n, k, _s(stream))


def q8act_gemm_workspace_bytes(m, k) -> int:
    return lib().q8act_gemm_workspace_bytes(m, k)


def q8act_gemm_q8_0(w, x, y, m, n, k, ws, ws_bytes, stream=None) -> int:
    return lib().q8act_gemm_q8_0(_p(w), _p(x), _p(y), m, n, k, _p(ws), ws_bytes, _s(stream))


def q8act_gemm_q8_0_preq(w, xqh, xdt, y, m, n, k, stream=None) -> int:
    return lib().q8act_gemm_q8_0_preq(_p(w), _p(xqh), _p(xdt), _p(y), m, n, k, _s(stream))


def q8act_dequant_q8_0_f16(w, w16, n, k, stream=None) -> int:
    return lib().q8act_dequant_q8_0_f16(_p(w), _p(w16), n, k, _s(stream))


def q8act_debug_gemv_block_dots(w, xq, D, m, n, k, stream=None) -> int:
    return lib().q8act_debug_gemv_block_dots(_p(w), _p(xq), _p(D), m, n, k, _s(stream))


def q8act_debug_gemm_block_dots(w, xqh, D, m, n, k, stream=None) -> int:
    return lib().q8act_debug_gemm_block_dots(_p(w), _p(xqh), _p(D), m, n, k, _s(stream))


def q8act_device_status(stream=None) -> int:
    return lib().q8act_device_status(_s(stream))


def q8act_gemm_q8_0_noalloc(w, x, y, m, n, k, stream=None) -> int:
    """The fused GEMM using the library's fixed device scratch instead of a caller workspace
    (for callers that cannot allocate device memory)."""
    return lib().q8act_gemm_q8_0_noalloc(_p(w), _p(x), _p(y), m, n, k, _s(stream))


def q8act_repack_q8_0(w, wq16, wdt, n, k, stream=None) -> int:
    return lib().q8act_repack_q8_0(_p(w), _p(wq16), _p(wdt), n, k, _s(stream))


def q8act_repack_ldn(n) -> int:
    return lib().q8act_repack_ldn(n)


def q8act_gemm_q8_0_repacked(wq16, wdt, x, y, m, n, k, ws, ws_bytes, stream=None) -> int:
    return lib().q8act_gemm_q8_0_repacked(_p(wq16), _p(wdt), _p(x), _p(y), m, n, k, _p(ws), ws_bytes,
                                          _s(stream))


def q8act_debug_gemm_repacked_block_dots(wq16, wdt, xqh, D, m, n, k, stream=None) -> int:
    return lib().q8act_debug_gemm_repacked_block_dots(_p(wq16), _p(wdt), _p(xqh), _p(D), m, n, k,
                                                      _s(stream))


def q8act_gemv_q8_0_group(w, y, n, xq, xd, m, k, stream=None) -> int:
    """w, y: sequences of tensors (or device addresses), n: sequence of row counts; the
    pointer and size arrays are marshalled into host memory for the call."""
    count = len(w)
    Parr = ctypes.c_void_p * max(count, 1)
    Narr = ctypes.c_int64 * max(count, 1)
    wa = Parr(*[_p(v) for v in w])
    ya = Parr(*[_p(v) for v in y])
    na = Narr(*[int(v) for v in n])
    return lib().q8act_gemv_q8_0_group(wa, ya, na, count, _p(xq), _p(xd), m, k, _s(stream))


def q8act_quantize_q4_0(w, wq, n, k, stream=None) -> int:
    return lib().q8act_quantize_q4_0(_p(w), _p(wq), n, k, _s(stream))


def q8act_dequant_q4_0_f16(w, w16, n, k, stream=None) -> int:
    return lib().q8act_dequant_q4_0_f16(_p(w), _p(w16), n, k, _s(stream))


def q8act_gemv_q4_0(w, xq, xd, y, m, n, k, stream=None) -> int:
    return lib().q8act_gemv_q4_0(_p(w), _p(xq), _p(xd), _p(y), m, n, k, _s(stream))


def q8act_debug_gemv_q4_0_block_dots(w, xq, D, m, n, k, stream=None) -> int:
    return lib().q8act_debug_gemv_q4_0_block_dots(_p(w), _p(xq), _p(D), m, n, k, _s(stream))


def q8act_gemv_workspace_bytes(m, k) -> int:
    return lib().q8act_gemv_workspace_bytes(m, k)


def q8act_gemv_q8_0_f32(w, x, y, m, n, k, ws, ws_bytes, stream=None) -> int:
    return lib().q8act_gemv_q8_0_f32(_p(w), _p(x), _p(y), m, n, k, _p(ws), ws_bytes, _s(stream))


def q8act_debug_wait_timeout(limit_ns, stream=None) -> int:
    """Test hook: a kernel whose bounded wait on a barrier nobody arrives on runs out after
    limit_ns nanoseconds and records a pipeline timeout in the device status word."""
    return lib().q8act_debug_wait_timeout(int(limit_ns), _s(stream))


def q8act_dequant_q6_k_f16(w, w16, n, k, stream=None) -> int:
    return lib().q8act_dequant_q6_k_f16(_p(w), _p(w16), n, k, _s(stream))


def q8act_dequant_q4_k_f16(w, w16, n, k, stream=None) -> int:
    return lib().q8act_dequant_q4_k_f16(_p(w), _p(w16), n, k, _s(stream))


def q8act_dequant_q5_k_f16(w, w16, n, k, stream=None) -> int:
    return lib().q8act_dequant_q5_k_f16(_p(w), _p(w16), n, k, _s(stream))


def q8act_gemv_q6_k(w, xq, xd, y, m, n, k, stream=None) -> int:
    return lib().q8act_gemv_q6_k(_p(w), _p(xq), _p(xd), _p(y), m, n, k, _s(stream))


def q8act_gemv_q4_k(w, xq, xd, y, m, n, k, stream=None) -> int:
    return lib().q8act_gemv_q4_k(_p(w), _p(xq), _p(xd), _p(y), m, n, k, _s(stream))


def q8act_gemv_q5_k(w, xq, xd, y, m, n, k, stream=None) -> int:
    return lib().q8act_gemv_q5_k(_p(w), _p(xq), _p(xd), _p(y), m, n, k, _s(stream))


def q8act_debug_gemv_q6_k_block_dots(w, xq, D, m, n, k, stream=None) -> int:
    return lib().q8act_debug_gemv_q6_k_block_dots(_p(w), _p(xq), _p(D), m, n, k, _s(stream))


def q8act_debug_gemv_q4_k_block_dots(w, xq, D, m, n, k, stream=None) -> int:
    return lib().q8act_debug_gemv_q4_k_block_dots(_p(w), _p(xq), _p(D), m, n, k, _s(stream))


def q8act_debug_gemv_q5_k_block_dots(w, xq, D, m, n, k, stream=None) -> int:
    return lib().q8act_debug_gemv_q5_k_block_dots(_p(w), _p(xq), _p(D), m, n, k, _s(stream))
