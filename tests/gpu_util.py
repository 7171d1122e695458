"""Helpers of the GPU parity tests: seeded inputs, oracle references, the tolerance rule."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import q8_block_quantized_act_gb300 as q8
from q8_block_quantized_act_gb300 import build as q8build
from q8_block_quantized_act_gb300 import inputs

QK = 32
RTOL = 1e-5   # |y - y64| <= RTOL * S,  S = sum_b |d_w d_a D|  (f32 fold-order difference only)

_built = False


def ensure_built():
    global _built
    if not _built:
        q8build.build()
        assert torch.cuda.is_available(), "GPU tests need a CUDA device"
        _built = True


def cuda(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def problem(m, n, k, kind="normal", wseed=0, xseed=1):
    """Seeded f32 weights/activations and their oracle quantizations (numpy)."""
    w = inputs.weights_f32(n, k, seed=wseed)
    x = inputs.activations_f32(m, k, kind=kind, seed=xseed)
    wb = oracle.quantize_q8_0(w)
    xq, xd = oracle.quantize_q8_1(x)
    return w, x, wb, xq, xd


# One line per checked output set: (label, max |dy|/S, max plain |dy|/|y64| over the outputs
# with |y64| >= 1e-3 S, how many such outputs, how many outputs).  conftest.py prints them
# after the run, so the plain relative error appears next to the error-scale bound.
ERROR_REPORT: list = []


def current_test_label() -> str:
    import os
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


def plain_relative_error(y_gpu: np.ndarray, y64: np.ndarray, S: np.ndarray):
    """Max |y_gpu - y64| / |y64| over the outputs with |y64| >= 1e-3 * S (outputs nearer zero
    than that are sums that cancel, where a plain relative error says nothing), and how many
    outputs that covers."""
    err = np.abs(y_gpu.astype(np.float64) - y64)
    sel = np.abs(y64) >= 1e-3 * S
    if not sel.any():
        return 0.0, 0
    return float((err[sel] / np.abs(y64[sel])).max()), int(sel.sum())


def assert_within_tolerance(y_gpu: np.ndarray, y64: np.ndarray, S: np.ndarray, rtol=RTOL):
    err = np.abs(y_gpu.astype(np.float64) - y64)
    bound = rtol * S
    bad = np.argwhere(err > bound)
    worst = float((err / np.where(S > 0, S, 1)).max()) if err.size else 0.0
    plain, counted = plain_relative_error(y_gpu, y64, S)
    ERROR_REPORT.append((current_test_label(), worst, plain, counted, int(err.size)))
    assert bad.size == 0, (
        f"{len(bad)} outputs outside {rtol}*S; first {tuple(bad[0])}: gpu={y_gpu[tuple(bad[0])]!r} "
        f"oracle={y64[tuple(bad[0])]!r} S={S[tuple(bad[0])]!r}")
    return worst


def sample_rows(n, count, seed=11):
    rng = np.random.Generator(np.random.PCG64(seed))
    if n <= count:
        return np.arange(n, dtype=np.int64)
    rows = rng.choice(n, size=count, replace=False)
    rows[:2] = [0, n - 1]                    # always include both edges (ragged last tile)
    return np.sort(rows).astype(np.int64)


def device_ok():
    torch.cuda.synchronize()
    q8.device_status()
