"""Seeded synthetic inputs for the Q8_0 x q8_1 matmul: shapes and random values only.

This module holds none of the method's arithmetic (no quantization, no dot products, no
folding): it draws f32 weights and activations with numpy's PCG64 generator, whose streams
are the same on every platform, so the product path and the oracle can be fed identical
inputs on x86 and Arm hosts alike.

Distributions (the pages give no dataset; these stand in for a decoder's weights and
hidden states at the pages' serving shapes):
  weights       N(0, 0.02), seed 0
  activations   N(0, 1), seed 1, optionally
                  "outliers":     each entry independently (p = 0.01, seed 2) scaled by 20
                  "token_scales": each token row scaled by s_t, ln s_t ~ U(ln 0.1, ln 10)
                                  (seed 2)
"""
from __future__ import annotations

import numpy as np

WEIGHT_SEED = 0
ACT_SEED = 1
AUX_SEED = 2
WEIGHT_STD = 0.02


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def weights_f32(n: int, k: int, seed: int = WEIGHT_SEED, std: float = WEIGHT_STD) -> np.ndarray:
    """f32 [n, k] weights drawn from N(0, std^2)."""
    w = _rng(seed).standard_normal((n, k), dtype=np.float32)
    w *= np.float32(std)
    return w


def activations_f32(m: int, k: int, kind: str = "normal", seed: int = ACT_SEED,
                    aux_seed: int = AUX_SEED) -> np.ndarray:
    """f32 [m, k] activations: N(0, 1), with the optional outlier or per-token-scale mix."""
    x = _rng(seed).standard_normal((m, k), dtype=np.float32)
    if kind == "normal":
        pass
    elif kind == "outliers":
        mask = _rng(aux_seed).random((m, k), dtype=np.float32) < np.float32(0.01)
        x[mask] *= np.float32(20.0)
    elif kind == "token_scales":
        lo, hi = np.log(0.1), np.log(10.0)
        s = np.exp(_rng(aux_seed).uniform(lo, hi, size=(m, 1))).astype(np.float32)
        x *= s
    else:
        raise ValueError(f"unknown activation kind {kind!r}")
    return x


KQUANT_LAYOUT = {
    # bytes per 256-weight superblock, and the byte offsets of its binary16 scale fields
    "q6_k": (210, (208,)),
    "q4_k": (144, (0, 2)),
    "q5_k": (176, (0, 2)),
}


def kquant_superblocks(fmt: str, n: int, k: int, seed: int = WEIGHT_SEED) -> np.ndarray:
    """uint8 [n, k/256 * bytes] of K-quant superblocks: every code and sub-block scale byte
    drawn uniformly from all its bit patterns, and each binary16 scale field (d, and dmin for
    Q4_K / Q5_K) a positive binary16 with a uniformly drawn fraction and an exponent field in
    5..8 (2^-10 .. 2^-7 times 1..2).  Random bits cover every code, every sub-block scale
    and min and every sign of the Q6_K scales; the weight magnitudes (up to ~16 for Q6_K) are
    not those of a trained model, which neither the exact integers nor the relative error
    bound depend on."""
    nbytes, scale_offsets = KQUANT_LAYOUT[fmt]
    rng = _rng(seed)
    nsb = n * (k // 256)
    sb = rng.integers(0, 256, size=(nsb, nbytes), dtype=np.uint16).astype(np.uint8)
    for off in scale_offsets:
        frac = rng.integers(0, 1024, size=nsb, dtype=np.uint16)
        expo = rng.integers(5, 9, size=nsb, dtype=np.uint16)
        bits = (expo << 10) | frac
        sb[:, off] = (bits & 0xFF).astype(np.uint8)
        sb[:, off + 1] = (bits >> 8).astype(np.uint8)
    return sb.reshape(n, (k // 256) * nbytes)


# The serving shapes the pages time (decode_kernel_census.rs main, accprobe_bench.rs): each
# case is (name, m, n, k, activation kind).
GEMV_CASES = [
    ("tiny_256x512", 1, 512, 256, "normal"),
    ("o_proj_4096x4096", 1, 4096, 4096, "outliers"),
    ("qkv_4096x5152", 1, 5152, 4096, "outliers"),
] + [
    (f"{name}_m{m}", m, n, k, "normal")
    for (name, n, k) in (("head_half_4096x64448", 64448, 4096),
                         ("shexp_down_1280x4096", 4096, 1280),
                         ("expert_gate_up_4096x20480", 20480, 4096))
    for m in (1, 2, 4, 8)
]

GEMM_CASES = [
    ("prefill_m512_4096x4096", 512, 4096, 4096, "normal"),
    ("prefill_m512_4096x5152", 512, 5152, 4096, "normal"),
    ("prefill_m512_4096x20480", 512, 20480, 4096, "token_scales"),
    ("prefill_m2048_4096x20480", 2048, 20480, 4096, "token_scales"),
    ("prefill_m512_4096x64448", 512, 64448, 4096, "token_scales"),
    ("prefill_m2048_4096x64448", 2048, 64448, 4096, "token_scales"),
]
