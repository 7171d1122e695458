"""Pins of the CPU oracle to facts outside itself.

Each ``pin_*`` function takes a namespace with the oracle's public functions (the real
oracle, or a copy with a planted mistake) and raises AssertionError when the oracle
disagrees with what the pages or the mathematics fix:

  * hand-derived worked cases under tests/golden/ (each cites its page);
  * independent libraries: numpy's binary16 conversion, numpy int64 / float64 matmuls;
  * closed forms and invariants of the quantizer (range, amax -> +-127, odd symmetry,
    power-of-two scaling, zero blocks, re-quantization idempotence);
  * brute force on tiny inputs: the block fold equals the plain float64 dot product of
    the dequantized operands (sum_b d_w d_a D_b = sum_i (d_w q_w,i)(d_a q_a,i)).

Nothing here calls the CUDA library.
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
QK = 32


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def parse_q8_0(wb: np.ndarray, n: int, k: int):
    """Decode Q8_0 bytes with numpy alone: (d_w float64 [n, k/32], q int64 [n, k/32, 32])."""
    nb = k // QK
    blocks = np.ascontiguousarray(wb).reshape(n, nb, 34)
    d = np.ascontiguousarray(blocks[:, :, 0:2]).view("<f2").reshape(n, nb).astype(np.float64)
    q = np.ascontiguousarray(blocks[:, :, 2:]).view(np.int8).astype(np.int64)
    return d, q


def _block(entries: dict) -> np.ndarray:
    v = np.zeros(QK, dtype=np.float32)
    for i, val in entries.items():
        v[int(i)] = np.float32(val)
    return v


def _rand_blocks(rng, rows, k, lo=-40, hi=40):
    """Blocks whose magnitudes span binades 2^lo..2^hi (all f32 scales stay normal)."""
    x = rng.standard_normal((rows, k)).astype(np.float32)
    scale = np.exp2(rng.integers(lo, hi, size=(rows, k // QK))).astype(np.float32)
    x *= np.repeat(scale, QK, axis=1)
    # a few exact ties and a few zero blocks
    x[0, :QK] = np.arange(QK, dtype=np.float32) - 15.5
    if rows > 1:
        x[1, QK:2 * QK] = 0.0 if k >= 2 * QK else x[1, QK:2 * QK]
    return x


# ---------------------------------------------------------------------------------------
# O0: binary16 conversions
# ---------------------------------------------------------------------------------------
def pin_f16_decode_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = o.f16_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # and every finite value survives the round trip
    back = o.f32_to_f16(got[~nan])
    assert np.array_equal(back, bits[~nan])


def pin_f16_encode_vs_numpy(o, n_random=1 << 20, seed=7):
    rng = np.random.Generator(np.random.PCG64(seed))
    raw = rng.integers(0, 1 << 32, size=n_random, dtype=np.uint64).astype(np.uint32)
    x = raw.view(np.float32)
    # every midpoint between adjacent finite binary16 values, and its f32 neighbours
    h = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mid = ((h[:-1] + h[1:]) / 2).astype(np.float32)
    near = np.concatenate([mid, np.nextafter(mid, np.float32(np.inf)),
                           np.nextafter(mid, np.float32(0))])
    x = np.concatenate([x, near, -near]).astype(np.float32)
    x = x[~np.isnan(x)]
    got = o.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[0]]!r}"


def pin_f16_golden(o):
    g = _golden("f16_conversions.json")
    xs = np.array([float(c["f32"]) for c in g["cases"]], dtype=np.float32)
    want = np.array([int(c["f16"], 16) for c in g["cases"]], dtype=np.uint16)
    got = o.f32_to_f16(xs)
    for c, gv, wv in zip(g["cases"], got, want):
        assert gv == wv, f"{c['f32']}: got {gv:#06x}, want {wv:#06x} ({c['why']})"


# ---------------------------------------------------------------------------------------
# O1 / O2: quantizers
# ---------------------------------------------------------------------------------------
def pin_q8_1_golden(o):
    g = _golden("q8_1_worked_cases.json")
    x = np.stack([_block(c["x"]) for c in g["cases"]]).reshape(1, -1)
    xq, xd = o.quantize_q8_1(x)
    for j, c in enumerate(g["cases"]):
        want_q = np.zeros(QK, dtype=np.int8)
        for i, v in c["q"].items():
            want_q[int(i)] = v
        assert xd[0, j] == np.float32(c["d"]), f"{c['name']}: d={xd[0, j]!r} ({c['why']})"
        assert np.array_equal(xq[0, j * QK:(j + 1) * QK], want_q), f"{c['name']}: {c['why']}"


def pin_q8_0_layout_golden(o):
    g = _golden("q8_0_block_layout.json")
    k = g["k"]
    w = np.zeros((1, k), dtype=np.float32)
    for i, v in g["row"].items():
        w[0, int(i)] = v
    got = o.quantize_q8_0(w)
    assert got.shape == (1, k // QK * 34)
    assert got.tobytes().hex() == g["bytes_hex"], g["why"]


def _check_quant_block_invariants(x, xq, d):
    """x [rows, k] f32, xq [rows, k] int, d [rows, k/32] f32 (the f32 scale used)."""
    rows, k = x.shape
    nb = k // QK
    xb = x.reshape(rows, nb, QK)
    qb = xq.reshape(rows, nb, QK).astype(np.int64)
    amax = np.abs(xb).max(axis=2)
    assert np.all(np.abs(qb) <= 127)
    nz = amax > 0
    assert np.all(np.abs(qb).max(axis=2)[nz] == 127), "a nonzero block must reach +-127"
    # the entry holding the block amax maps to +-127 with its own sign
    idx = np.abs(xb).argmax(axis=2)
    top_q = np.take_along_axis(qb, idx[..., None], axis=2)[..., 0]
    top_x = np.take_along_axis(xb, idx[..., None], axis=2)[..., 0]
    assert np.all(top_q[nz] == np.where(top_x[nz] > 0, 127, -127))
    assert np.all(qb[~nz] == 0) and np.all(d[~nz] == 0)
    assert np.all(np.isfinite(d))
    # d = amax / 127 up to one rounding (both are f32)
    rel = np.abs(d[nz].astype(np.float64) * 127 - amax[nz]) / amax[nz]
    assert np.all(rel <= 2.0 ** -23)
    # each quant is within half a step of x/d, measured in float64
    ratio = xb.astype(np.float64) / np.where(d > 0, d, 1)[..., None]
    err = np.abs(ratio - qb)[nz]
    assert np.all(err <= 0.5 + 1e-5), f"max |x/d - q| = {err.max()}"


def pin_quant_invariants(o, seed=3):
    rng = np.random.Generator(np.random.PCG64(seed))
    for k in (32, 256, 1280):
        x = _rand_blocks(rng, 17, k)
        xq, xd = o.quantize_q8_1(x)
        _check_quant_block_invariants(x, xq, xd)
        # odd symmetry (fails for floor(x + 0.5) style rounding)
        nq, nd = o.quantize_q8_1(-x)
        assert np.array_equal(nq, -xq) and np.array_equal(nd, xd)
        # power-of-two scaling is exact in binary floating point
        for s in (-9, 1, 13):
            sq, sd = o.quantize_q8_1(x * np.float32(2.0 ** s))
            assert np.array_equal(sq, xq)
            assert np.array_equal(sd, xd * np.float32(2.0 ** s))
        # Q8_0 weights: same quants (computed with the f32 d), scale stored as binary16
        wb = o.quantize_q8_0(x)
        dh, wq = parse_q8_0(wb, x.shape[0], k)
        assert np.array_equal(wq.reshape(x.shape[0], k), xq.astype(np.int64))
        want_h = xd.astype(np.float16).view(np.uint16)
        got_h = np.ascontiguousarray(wb.reshape(x.shape[0], k // QK, 34)[:, :, 0:2]).view("<u2")
        assert np.array_equal(got_h.reshape(want_h.shape), want_h)


def pin_requant_idempotent(o, seed=4):
    rng = np.random.Generator(np.random.PCG64(seed))
    k = 512
    x = _rand_blocks(rng, 9, k)
    xq, xd = o.quantize_q8_1(x)
    back = (np.repeat(xd, QK, axis=1) * xq.astype(np.float32)).astype(np.float32)
    q2, d2 = o.quantize_q8_1(back)
    assert np.array_equal(q2, xq)
    ulp = np.spacing(xd)
    assert np.all(np.abs(d2 - xd) <= ulp)
    # Q8_0: with the binary16 scale the dequantized block re-quantizes to the same bytes
    # (scales kept inside the binary16 range so that no scale rounds to 0 or infinity)
    x = _rand_blocks(rng, 9, k, lo=-6, hi=6)
    wb = o.quantize_q8_0(x)
    dh, wq = parse_q8_0(wb, x.shape[0], k)
    deq = (np.repeat(dh.astype(np.float32), QK, axis=1) * wq.reshape(x.shape[0], k).astype(np.float32))
    assert np.array_equal(o.quantize_q8_0(deq.astype(np.float32)), wb)


# ---------------------------------------------------------------------------------------
# O3 / O4: block dots and the fold, by brute force
# ---------------------------------------------------------------------------------------
def _tiny_problem(rng, m, n, k, o):
    w = rng.standard_normal((n, k)).astype(np.float32) * np.float32(0.02)
    x = rng.standard_normal((m, k)).astype(np.float32)
    x *= np.exp2(rng.integers(-6, 6, size=(m, 1))).astype(np.float32)
    wb = o.quantize_q8_0(w)
    xq, xd = o.quantize_q8_1(x)
    return wb, xq, xd


def pin_block_dots_bruteforce(o, seed=5):
    rng = np.random.Generator(np.random.PCG64(seed))
    for (m, n, k) in ((1, 3, 32), (3, 5, 64), (4, 8, 256), (2, 7, 96)):
        wb, xq, xd = _tiny_problem(rng, m, n, k, o)
        _, wq = parse_q8_0(wb, n, k)
        aq = xq.reshape(m, k // QK, QK).astype(np.int64)
        ref = np.einsum("rbi,tbi->trb", wq, aq)
        got = o.block_dots(wb, xq, k)
        assert got.shape == (m, n, k // QK)
        assert np.array_equal(got.astype(np.int64), ref)
        rows = np.array([n - 1, 0, n // 2], dtype=np.int64)
        assert np.array_equal(o.block_dots(wb, xq, k, rows=rows).astype(np.int64), ref[:, rows])


def pin_fold_bruteforce(o, seed=6):
    rng = np.random.Generator(np.random.PCG64(seed))
    for (m, n, k) in ((1, 3, 32), (3, 5, 64), (4, 8, 256), (2, 6, 4096)):
        wb, xq, xd = _tiny_problem(rng, m, n, k, o)
        dw, wq = parse_q8_0(wb, n, k)
        Wd = (dw[:, :, None] * wq).reshape(n, k)                     # exact in float64
        Xd = (xd.astype(np.float64)[:, :, None]
              * xq.reshape(m, k // QK, QK).astype(np.float64)).reshape(m, k)
        ref = Xd @ Wd.T                                              # [m, n]
        absref = np.abs((Xd[:, None, :] * Wd[None, :, :]).reshape(m, n, k // QK, QK)
                        .sum(axis=3)).sum(axis=2)
        y32, y64, S = o.matmul(wb, xq, xd, k)
        assert np.allclose(S, absref, rtol=1e-12, atol=0)
        assert np.all(np.abs(y64 - ref) <= 1e-12 * S + 1e-300)
        # the f32 fold stays inside the error bound the tolerance is built on
        nb = k // QK
        bound = (nb + 2) * 2.0 ** -24 * S
        assert np.all(np.abs(y32.astype(np.float64) - ref) <= bound + 1e-300)
        rows = np.array([n - 1, 0], dtype=np.int64)
        sy32, sy64, sS = o.matmul(wb, xq, xd, k, rows=rows)
        assert np.array_equal(sy32, y32[:, rows]) and np.array_equal(sy64, y64[:, rows])


# ---------------------------------------------------------------------------------------
# O5: fp16 dequant
# ---------------------------------------------------------------------------------------
def pin_dequant_vs_numpy(o, seed=8):
    rng = np.random.Generator(np.random.PCG64(seed))
    n, k = 13, 512
    w = _rand_blocks(rng, n, k, lo=-16, hi=6)
    wb = o.quantize_q8_0(w)
    dw, wq = parse_q8_0(wb, n, k)
    prod = (dw.astype(np.float32)[:, :, None] * wq.astype(np.float32)).reshape(n, k)
    with np.errstate(over="ignore"):
        ref = prod.astype(np.float16).view(np.uint16)
    got = o.dequant_f16(wb, k)
    assert np.array_equal(got, ref)


def pin_repack(o, seed=9):
    """The repacked planes hold exactly the Q8_0 quants and scales: numpy's own binary16
    decode of wq16 gives back the int8 quants, wdt is numpy's binary16 -> f32 of the stored
    scale bits (transposed), and re-rounding wdt * wq16 to fp16 reproduces the dequant."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n, k, ldn = 11, 768, 16
    w = _rand_blocks(rng, n, k, lo=-16, hi=6)
    wb = o.quantize_q8_0(w)
    dw, wq = parse_q8_0(wb, n, k)
    wq16, wdt = o.repack_q8_0(wb, k, ldn)
    assert np.array_equal(wq16.view(np.float16).astype(np.float64),
                          wq.reshape(n, k).astype(np.float64))
    assert np.array_equal(wdt[:, :n], dw.astype(np.float32).T)
    assert not wdt[:, n:].any()
    prod = wdt[:, :n].T.repeat(32, axis=1) * wq16.view(np.float16).astype(np.float32)
    with np.errstate(over="ignore"):
        assert np.array_equal(prod.astype(np.float16).view(np.uint16), o.dequant_f16(wb, k))


def pin_nonfinite_inputs(o):
    """Out-of-contract entries do not poison a block: a NaN entry is skipped by amax and
    quantizes to 0; an infinite entry makes d infinite, so every finite entry quantizes to 0
    and the infinite one (inf / inf) too."""
    v = np.zeros((1, QK), np.float32)
    v[0, :4] = [np.nan, 127.0, -63.5, 1.0]
    q, d = o.quantize_q8_1(v)
    assert d[0, 0] == np.float32(1.0)
    assert q[0, :4].tolist() == [0, 127, -64, 1]
    v[0, 0] = np.inf
    q, d = o.quantize_q8_1(v)
    assert np.isinf(d[0, 0]) and not q.any()


# ---------------------------------------------------------------------------------------
# O7: Q4_0 (the GGUF 18-byte block named by f16_ffi.rs memra_q4_0_dequant_f16)
# ---------------------------------------------------------------------------------------
def parse_q4_0(wb: np.ndarray, n: int, k: int):
    """Decode Q4_0 bytes with numpy alone: (d float64 [n, k/32], signed values int64
    [n, k/32, 32]) -- element i < 16 from the low nibble of quant byte i, element i + 16
    from its high nibble, minus 8."""
    nb = k // QK
    blocks = np.ascontiguousarray(wb).reshape(n, nb, 18)
    d = np.ascontiguousarray(blocks[:, :, 0:2]).view("<f2").reshape(n, nb).astype(np.float64)
    qs = blocks[:, :, 2:].astype(np.int64)
    q = np.concatenate([qs & 0x0F, qs >> 4], axis=2) - 8
    return d, q


def pin_q4_0_layout_golden(o):
    g = _golden("q4_0_block_layout.json")
    for blk in g["blocks"]:
        raw = np.frombuffer(bytes.fromhex(blk["bytes"].replace(" ", "")), dtype=np.uint8)
        assert raw.size == 18
        h = o.dequant_q4_0_f16(raw.reshape(1, 18), QK)[0]
        d = float(raw[:2].view("<f2")[0])
        for i, v in blk["values"].items():
            # a one-hot activation picks element i's signed value out of the block dot
            onehot = np.zeros((1, QK), np.int8)
            onehot[0, int(i)] = 1
            D = int(o.block_dots_q4_0(raw.reshape(1, 18), onehot, QK)[0, 0, 0])
            assert d * D == v, (i, d * D, v)
        for i, bits in blk["f16"].items():
            assert int(h[int(i)]) == int(bits, 16), (i, hex(h[int(i)]), bits)
        xq = np.zeros((1, QK), np.int8)
        for i, x in blk["xq"].items():
            xq[0, int(i)] = x
        assert o.block_dots_q4_0(raw.reshape(1, 18), xq, QK)[0, 0, 0] == blk["dot"]


def pin_q4_0_dequant_vs_numpy(o, seed=10):
    rng = np.random.Generator(np.random.PCG64(seed))
    n, k = 9, 768
    w = _rand_blocks(rng, n, k, lo=-12, hi=8)
    wb = o.quantize_q4_0(w)
    d, q = parse_q4_0(wb, n, k)
    prod = (d.astype(np.float32)[:, :, None] * q.astype(np.float32)).reshape(n, k)
    with np.errstate(over="ignore"):
        ref = prod.astype(np.float16).view(np.uint16)
    assert np.array_equal(o.dequant_q4_0_f16(wb, k), ref)


def pin_q4_0_writer_invariants(o, seed=11):
    """The Q4_0 writer (data preparation): nibbles stay in 1..15 (values -7..7), a block's
    largest magnitude maps to +-7, a zero block stores d = 0 and nibbles 8, negating the
    input negates the values, and every value is within half a step of the input."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n, k = 7, 512
    w = _rand_blocks(rng, n, k, lo=-10, hi=10)
    wb = o.quantize_q4_0(w)
    d, q = parse_q4_0(wb, n, k)
    assert q.min() >= -7 and q.max() <= 7
    wblk = w.reshape(n, k // QK, QK).astype(np.float64)
    amax = np.abs(wblk).max(axis=2)
    nz = amax > 0
    assert (np.abs(q).max(axis=2)[nz] == 7).all()
    assert (d[~nz] == 0).all() and (q[~nz] == 0).all()
    d32 = (amax / 7.0).astype(np.float32).astype(np.float64)   # the f32 divisor
    err = np.abs(wblk - d32[:, :, None] * q)
    assert (err <= 0.5 * d32[:, :, None] * (1 + 1e-6) + 1e-30).all()
    wb_neg = o.quantize_q4_0(-w)
    d2, q2 = parse_q4_0(wb_neg, n, k)
    assert np.array_equal(d2, d) and np.array_equal(q2, -q)


def pin_q4_0_dots_and_fold_bruteforce(o, seed=12):
    """Block dots equal numpy int64 dots of the decoded values; the fold (y64) equals the
    plain float64 dot of the dequantized operands; y32 is within the f32 summation bound."""
    rng = np.random.Generator(np.random.PCG64(seed))
    for m, n, k in [(1, 5, 32), (3, 8, 256), (2, 4, 1024)]:
        w = _rand_blocks(rng, n, k, lo=-6, hi=6)
        x = rng.standard_normal((m, k)).astype(np.float32)
        wb = o.quantize_q4_0(w)
        xq, xd = o.quantize_q8_1(x)
        d, q = parse_q4_0(wb, n, k)
        nb = k // QK
        D = o.block_dots_q4_0(wb, xq, k)
        ref = np.einsum("rbi,tbi->trb", q, xq.astype(np.int64).reshape(m, nb, QK))
        assert np.array_equal(D.astype(np.int64), ref)
        y32, y64, S = o.matmul_q4_0(wb, xq, xd, k)
        wv = (d[:, :, None] * q).reshape(n, k)
        xv = (xd.astype(np.float64)[:, :, None] * xq.astype(np.float64).reshape(m, nb, QK)).reshape(m, k)
        plain = xv @ wv.T
        assert np.all(np.abs(y64 - plain) <= 1e-12 * np.maximum(S, 1e-300))
        assert np.all(np.abs(y32.astype(np.float64) - y64) <= (nb + 2) * 2.0 ** -23 * S + 1e-30)
        rows = np.array([n - 1, 0], dtype=np.int64)
        sy32, sy64, _ = o.matmul_q4_0(wb, xq, xd, k, rows=rows)
        assert np.array_equal(sy32, y32[:, rows]) and np.array_equal(sy64, y64[:, rows])


# ---------------------------------------------------------------------------------------
# K-quant superblocks (Q6_K, Q4_K, Q5_K): tests/golden/kquant_superblocks.json holds one
# superblock of each format built from chosen codes and scales (the encoding direction of
# the GGUF layouts), with hand-worked values; the oracle must read those choices back.
# ---------------------------------------------------------------------------------------
def _kq_golden():
    return _golden("kquant_superblocks.json")["superblocks"]


def _kq_expected(sb):
    """The exact values of the golden superblock's 256 weights, from its chosen codes and
    scales (float64: every one is exact)."""
    e = np.arange(256)
    codes = np.array(sb["codes"], dtype=np.float64)
    if sb["format"] == "q6_k":
        return sb["d"] * np.array(sb["scales"], dtype=np.float64)[e // 16] * (codes - 32)
    sc = np.array(sb["sub_scales"], dtype=np.float64)[e // 32]
    mn = np.array(sb["sub_mins"], dtype=np.float64)[e // 32]
    return sb["d"] * sc * codes - sb["dmin"] * mn


def _kq_bytes(sb):
    return np.frombuffer(bytes.fromhex(sb["bytes"]), dtype=np.uint8).reshape(1, -1).copy()


def pin_kq_golden_dequant(o):
    """The fp16 mirror of each golden superblock: numpy's binary16 rounding of the chosen
    exact values, and the hand-worked encodings (including round-to-even ties)."""
    for sb in _kq_golden():
        h = o.dequant_kq_f16(sb["format"], _kq_bytes(sb), 256)[0]
        want = _kq_expected(sb).astype(np.float16).view(np.uint16)
        assert np.array_equal(h, want), sb["format"]
        for w in sb["worked"]:
            assert abs(_kq_expected(sb)[w["e"]] - w["value"]) == 0.0, (sb["format"], w["e"])
            if "f16" in w:
                assert int(h[w["e"]]) == int(w["f16"], 16), (sb["format"], w["e"])


def pin_kq_golden_onehot(o):
    """Each weight read alone through the block integers and the fold: with the one-hot
    activation of element e (quant 1, scale 1) the block integer is the weight's scaled code
    (Q6_K: scale * (code - 32); Q4_K / Q5_K: the code) and y64 is the weight's exact value."""
    for sb in _kq_golden():
        fmt = sb["format"]
        wb = _kq_bytes(sb)
        xq = np.eye(256, dtype=np.int8)
        xd = np.ones((256, 8), dtype=np.float32)
        D = o.block_dots_kq(fmt, wb, xq, 256)[:, 0, :]
        codes = np.array(sb["codes"], dtype=np.int64)
        e = np.arange(256)
        if fmt == "q6_k":
            want = np.array(sb["scales"], dtype=np.int64)[e // 16] * (codes - 32)
        else:
            want = codes
        got = D[e, e // 32]
        assert np.array_equal(got.astype(np.int64), want), fmt
        mask = np.ones_like(D, dtype=bool)
        mask[e, e // 32] = False
        assert not D[mask].any(), fmt
        _, y64, S = o.matmul_kq(fmt, wb, xq, xd, 256)
        assert np.array_equal(y64[:, 0], _kq_expected(sb)), fmt
        assert np.all(S[:, 0] >= np.abs(y64[:, 0]))


def pin_kq_fold_bruteforce(o, seed=13):
    """y64 over rows of golden superblocks (repeated, and with one superblock's scale bytes
    changed) equals the plain float64 dot of the exact weights with the dequantized
    activation; y32 is within the f32 summation bound; a row subset gives the same rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    for sb in _kq_golden():
        fmt = sb["format"]
        one = _kq_bytes(sb)[0]
        vals = _kq_expected(sb)
        k = 512
        row = np.concatenate([one, one])
        w = np.stack([row, row[::1]]).copy()
        m = 3
        x = rng.standard_normal((m, k)).astype(np.float32) * np.float32(3.0)
        xq, xd = o.quantize_q8_1(x)
        _, y64, S = o.matmul_kq(fmt, w, xq, xd, k)
        wv = np.concatenate([vals, vals])
        xv = (xd.astype(np.float64)[:, :, None] * xq.astype(np.float64).reshape(m, k // QK, QK)).reshape(m, k)
        plain = xv @ wv
        assert np.all(np.abs(y64[:, 0] - plain) <= 1e-12 * np.maximum(S[:, 0], 1e-300)), fmt
        y32, _, _ = o.matmul_kq(fmt, w, xq, xd, k)
        assert np.all(np.abs(y32.astype(np.float64) - y64) <= (k // QK + 4) * 2.0 ** -23 * S + 1e-30), fmt
        sy32, sy64, _ = o.matmul_kq(fmt, w, xq, xd, k, rows=np.array([1], dtype=np.int64))
        assert np.array_equal(sy64[:, 0], y64[:, 1]) and np.array_equal(sy32[:, 0], y32[:, 1])


def pin_f64_to_f16_vs_numpy(o, seed=14):
    """binary64 -> binary16 against numpy's own conversion: random values over the whole
    binary16 range (and past it), every midpoint between neighbouring binary16 values of a
    few binades and its neighbours one double ulp away, zeros, infinities."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-28, 18, size=20000))
    h = np.arange(0, 0x7c00, 97, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    x = np.concatenate([x, mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf), -mid,
                        [0.0, -0.0, np.inf, -np.inf, 65504.0, 65519.99, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26]])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(o.f64_to_f16(x), want)


ALL_PINS = [
    pin_f16_decode_exhaustive,
    pin_f16_encode_vs_numpy,
    pin_f16_golden,
    pin_q8_1_golden,
    pin_q8_0_layout_golden,
    pin_quant_invariants,
    pin_requant_idempotent,
    pin_block_dots_bruteforce,
    pin_fold_bruteforce,
    pin_dequant_vs_numpy,
    pin_repack,
    pin_nonfinite_inputs,
    pin_q4_0_layout_golden,
    pin_q4_0_dequant_vs_numpy,
    pin_q4_0_writer_invariants,
    pin_q4_0_dots_and_fold_bruteforce,
    pin_kq_golden_dequant,
    pin_kq_golden_onehot,
    pin_kq_fold_bruteforce,
    pin_f64_to_f16_vs_numpy,
]
