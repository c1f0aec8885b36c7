"""Pins for the oracle: checks against what the pages and mathematics fix.

Each check takes an ``oracle.Oracle`` instance and raises AssertionError on a
mismatch, so the same checks run against the real build and against builds
with a planted mistake (``test_oracle_mutants.py``).  None of them retypes the
oracle's formulas: they use stored hand-worked values, brute-force searches,
library routines (numpy matmul and float16 rounding), closed-form bounds and
invariants.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

from w4a8_quantized_serving_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (t.strip() for t in line.split("=", 1))
            vals = [int(t, 0) for t in v.split()]
            out[k] = vals if len(vals) > 1 else vals[0]
    return out


def f16(values) -> np.ndarray:
    return np.asarray(values, dtype=np.float64).astype(np.float16)


def half_val(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def nearest_int_half_even(x: Fraction) -> int:
    """Brute-force nearest integer to x, ties to the even one."""
    lo = x.numerator // x.denominator
    best = None
    for c in range(lo - 1, lo + 3):
        d = abs(x - c)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


# --------------------------------------------------------------------------
# binary16 conversions against numpy's IEEE float16
# --------------------------------------------------------------------------

def check_half_to_double(o) -> None:
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    for b in range(0, 65536, 7):  # every 7th pattern covers all exponents
        v = o.half_to_double(b)
        r = ref[b]
        if np.isnan(r):
            assert np.isnan(v), b
        else:
            assert v == r, (hex(b), v, r)


def check_double_to_half(o) -> None:
    rng = np.random.default_rng(1234)
    xs = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 6, 3000),
        # exact ties between neighbouring fp16 values
        (np.arange(2048, 4096, 3, dtype=np.float64) + 0.5) * 2.0 ** -11,
        (np.arange(1, 1024, 5, dtype=np.float64) + 0.5) * 2.0 ** -24,  # subnormal ties
        np.array([65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -25, 2.0 ** -26, 6.1e-5, 0.0, -0.0]),
    ])
    with np.errstate(over="ignore"):
        wants = xs.astype(np.float16).view(np.uint16)
    for x, want in zip(xs, wants):
        got = o.double_to_half(float(x))
        want = int(want)
        assert got == want, (x, hex(got), hex(want))


# --------------------------------------------------------------------------
# the hand-worked example and the printed dequant literal
# --------------------------------------------------------------------------

def _appendix_inputs(gold: dict, K: int = 8, g: int = 4, embed: bool = False):
    Q8 = np.array(gold["Q8"], np.int64)
    Xq = np.array(gold["Xq"], np.int64)
    if not embed:
        W = f16(Q8 * 2.0 ** -7).reshape(1, K)
        X = f16(Xq * 2.0 ** -6).reshape(1, K)
        return W, X
    # g = 128 embedding: group j of the example sits at k = 128 j + 0..3, zeros elsewhere
    Wl = np.zeros(K, np.float64)
    Xl = np.zeros(K, np.float64)
    for j in range(2):
        Wl[128 * j:128 * j + 4] = Q8[4 * j:4 * j + 4] * 2.0 ** -7
        Xl[128 * j:128 * j + 4] = Xq[4 * j:4 * j + 4] * 2.0 ** -6
    return f16(Wl).reshape(1, K), f16(Xl).reshape(1, K)


def check_appendix_a(o) -> None:
    gold = load_golden("appendix_a_g4.txt")
    g = gold["g"]
    W, X = _appendix_inputs(gold)
    r = o.weight_quant(synth.bits(W), g)
    assert int(r["s1"][0]) == gold["s1_bits"]
    assert r["Q8"][0].tolist() == gold["Q8"]
    assert r["s2"][0].tolist() == gold["s2"]
    assert r["z"][0].tolist() == gold["z"]
    assert r["q4"][0].tolist() == gold["q4"]
    w8 = o.dequant_weights(r["q4"], r["s2"], r["z"], g)
    assert w8[0].tolist() == gold["w8"]
    Xq, sx = o.act_quant(synth.bits(X))
    assert Xq[0].tolist() == gold["Xq"]
    assert int(sx[0]) == gold["sx_bits"]
    acc, Y = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g)
    assert int(acc[0, 0]) == gold["acc"] != gold["acc_half_away"]
    assert int(Y[0, 0]) == gold["Y_bits"]


def check_appendix_a_g128(o) -> None:
    """The same example embedded at g = 128 (K = 256), rows replicated to N = 128."""
    gold = load_golden("appendix_a_g4.txt")
    W1, X = _appendix_inputs(gold, K=256, embed=True)
    W = np.repeat(W1, 128, axis=0)
    r = o.weight_quant(synth.bits(W), 128)
    assert (r["s2"] == np.array(gold["s2"], np.uint8)).all()
    assert (r["z"] == np.array(gold["z"], np.uint8)).all()
    Xq, sx = o.act_quant(synth.bits(X))
    acc, Y = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], 128)
    assert (acc == gold["acc"]).all()
    assert (Y == gold["Y_bits"]).all()


def check_fig3_literal(o) -> None:
    """QFactory notes, Fig. 3: (6 - 2) x (-0.4) = -1.6; the integer form of the same rule."""
    assert o.dequant_real(6, 2, -0.4) == -1.6
    assert o.dequant_code(6, 2, 4) == 16
    assert o.dequant_code(2, 6, 4) == -16


# --------------------------------------------------------------------------
# brute force on tiny inputs
# --------------------------------------------------------------------------

def _tiny_rows(seed: int, n: int, k: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((n, k)) * 0.05
    W[:, rng.integers(0, k)] *= 8.0
    W[0, :] = np.abs(W[0, :])  # an all-positive row
    W[1, :] = -np.abs(W[1, :])  # an all-negative row
    return f16(W)


def check_level1_bruteforce(o) -> None:
    W = _tiny_rows(7, 24, 16)
    r = o.weight_quant(synth.bits(W), 8)
    s1 = half_val(r["s1"])
    for n in range(W.shape[0]):
        amax = float(np.max(np.abs(W[n].astype(np.float64))))
        # s1 is the fp16 nearest to amax/119 up to one fp16 half-ulp plus an fp32 rounding
        assert abs(s1[n] - amax / 119) <= s1[n] * (2.0 ** -11 + 2.0 ** -23) + 1e-30
        sf = Fraction(float(s1[n]))
        for k in range(W.shape[1]):
            w = Fraction(float(W[n, k]))
            # nearest code in [-119, 119] to w/s1, ties to even
            want = max(-119, min(119, nearest_int_half_even(w / sf)))
            assert int(r["Q8"][n, k]) == want, (n, k)


def check_level2_bruteforce(o) -> None:
    W = _tiny_rows(11, 32, 16)
    g = 4
    r = o.weight_quant(synth.bits(W), g)
    for n in range(W.shape[0]):
        for j in range(W.shape[1] // g):
            grp = [int(v) for v in r["Q8"][n, j * g:(j + 1) * g]]
            lo, hi = min(0, min(grp)), max(0, max(grp))
            # smallest integer scale >= 1 whose 16-level grid spans [lo, hi]
            s2 = next(s for s in range(1, 64) if 15 * s >= hi - lo)
            # zero point: the grid index of 0, nearest integer to -lo/s2, ties to even
            zero = nearest_int_half_even(Fraction(-lo, s2))
            assert int(r["s2"][n, j]) == s2, (n, j)
            assert int(r["z"][n, j]) == zero, (n, j)
            for t, q8 in enumerate(grp):
                c = nearest_int_half_even(Fraction(q8, s2))
                assert int(r["q4"][n, j * g + t]) == max(0, min(15, c + zero)), (n, j, t)


# --------------------------------------------------------------------------
# invariants and closed-form bounds
# --------------------------------------------------------------------------

def _adversarial_weights() -> np.ndarray:
    rng = np.random.default_rng(5)
    K = 256
    rows = [
        np.full(K, 0.5), np.full(K, -0.25), np.zeros(K),
        np.where(np.arange(K) % 2 == 0, 1.0, -1.0),
        np.linspace(-3, 3, K), rng.standard_normal(K) * 1e-3,
        np.where(np.arange(K) % 128 == 5, 40.0, rng.standard_normal(K) * 0.01),
        (rng.integers(-119, 120, K) * 2.0 ** -7),
    ]
    return f16(np.stack(rows + [rng.standard_normal(K) * 0.02 for _ in range(56)]))


def check_invariants(o) -> None:
    W = np.concatenate([_adversarial_weights(), synth.weights(64, 256, 99)])
    g = 128
    r = o.weight_quant(synth.bits(W), g)
    Q8 = r["Q8"].astype(np.int64)
    s2 = r["s2"].astype(np.int64)
    z = r["z"].astype(np.int64)
    q4 = r["q4"].astype(np.int64)
    w8 = o.dequant_weights(r["q4"], r["s2"], r["z"], g).astype(np.int64)
    s2e = np.repeat(s2, g, axis=1)
    assert Q8.min() >= -119 and Q8.max() <= 119
    assert s2.min() >= 1 and s2.max() <= 16
    assert z.min() >= 0 and z.max() <= 15
    assert q4.min() >= 0 and q4.max() <= 15
    assert (2 * np.abs(w8 - Q8) <= s2e).all()  # group error at most s2/2
    assert w8.min() >= -127 and w8.max() <= 127  # the protective range works
    # w8 is the dequant of the stored codes with the stored parameters
    assert (w8 == (q4 - np.repeat(z, g, axis=1)) * s2e).all()


def check_error_bounds(o) -> None:
    W = synth.weights(64, 512, 3)
    X = synth.activations(16, 512, 3)
    g = 128
    r = o.weight_quant(synth.bits(W), g)
    w8 = o.dequant_weights(r["q4"], r["s2"], r["z"], g).astype(np.float64)
    s1 = half_val(r["s1"])[:, None]
    s2e = np.repeat(r["s2"].astype(np.float64), g, axis=1)
    Wd = W.astype(np.float64)
    assert (np.abs(s1 * w8 - Wd) <= s1 * (0.5 + s2e / 2) * (1 + 1e-12)).all()
    Xq, sx = o.act_quant(synth.bits(X))
    sxv = half_val(sx)[:, None]
    assert (np.abs(sxv * Xq - X.astype(np.float64)) <= sxv / 2 * (1 + 1e-12)).all()
    assert np.abs(Xq).max() <= 127


def check_lossless_grid(o) -> None:
    """When a group already lies on its 16-level grid, level 2 loses nothing.

    Group 0 holds multiples of 7 spanning exactly [-49, 56] (15 steps of 7), so
    s2 = 7, z = 7 and every value is a grid point; group 2 spans [-7, 8]
    (s2 = 1).  Group 1 holds the row maximum 119 * 2^-7, which pins s1 = 2^-7
    so that the level-1 codes are the integers written here.
    """
    k = np.arange(128)
    g0 = ((k % 16) - 7) * 7  # -49 .. 56
    g1 = np.zeros(128, np.int64)
    g1[17] = 119
    g2 = (k % 16) - 7  # -7 .. 8
    q8 = np.concatenate([g0, g1, g2]).astype(np.int64)
    W = f16(q8 * 2.0 ** -7).reshape(1, -1)
    r = o.weight_quant(synth.bits(W), 128)
    assert int(r["s1"][0]) == 0x2000
    assert (r["Q8"][0] == q8).all()
    assert r["s2"][0].tolist() == [7, 8, 1] and r["z"][0].tolist() == [7, 0, 7]
    w8 = o.dequant_weights(r["q4"], r["s2"], r["z"], 128)[0]
    assert (w8[:128] == q8[:128]).all() and (w8[256:] == q8[256:]).all()


def check_zero_and_underflow(o) -> None:
    W = np.zeros((3, 256), np.float16)
    W[1, 3] = np.float16(2.0 ** -24)  # amax/119 underflows fp16 -> treated as a zero row
    W[2, :] = np.float16(1.0)
    r = o.weight_quant(synth.bits(W), 128)
    for n in (0, 1):
        assert int(r["s1"][n]) == 0
        assert (r["Q8"][n] == 0).all() and (r["q4"][n] == 0).all()
        assert (r["s2"][n] == 1).all() and (r["z"][n] == 0).all()
    X = np.zeros((2, 256), np.float16)
    X[1, :] = np.float16(-3.0)
    Xq, sx = o.act_quant(synth.bits(X))
    assert int(sx[0]) == 0 and (Xq[0] == 0).all()
    assert (Xq[1] == -127).all()


# --------------------------------------------------------------------------
# the GEMM against a library matmul
# --------------------------------------------------------------------------

def check_gemm_library(o) -> None:
    M, N, K, g = 9, 40, 384, 128
    W = synth.weights(N, K, 21)
    X = synth.activations(M, K, 21)
    r = o.weight_quant(synth.bits(W), g)
    Xq, sx = o.act_quant(synth.bits(X))
    acc, Y = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g)
    w8 = o.dequant_weights(r["q4"], r["s2"], r["z"], g).astype(np.int64)
    assert (acc == Xq.astype(np.int64) @ w8.T).all()
    # float dequant-then-matmul in float64 agrees with the scaled integer sum
    Xf = half_val(sx)[:, None] * Xq
    Wf = half_val(r["s1"])[:, None] * w8
    Yf = Xf @ Wf.T
    scaled = acc * half_val(sx)[:, None] * half_val(r["s1"])[None, :]
    assert np.allclose(Yf, scaled, rtol=1e-12, atol=1e-300)
    # the fp16 result is the library's round-to-nearest of the exact product
    assert (Y == scaled.astype(np.float16).view(np.uint16)).all()
    # sampled entries agree with the full product
    mi = np.array([0, 3, 8, 8], np.int32)
    ni = np.array([0, 39, 1, 17], np.int32)
    a2, y2 = o.gemm_entries(mi, ni, Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g)
    assert (a2 == acc[mi, ni]).all() and (y2 == Y[mi, ni]).all()
    # an operand swap would be caught: W rows are output channels
    assert acc.shape == (M, N)


def check_gemm_threads(o) -> None:
    """The multi-threaded product (output channels cut into ranges, one
    dequantized weight row at a time) equals the single-threaded oracle and
    numpy's int64 matmul of the dequantized weights, element for element, for
    thread counts that divide N, do not divide it, and exceed it."""
    M, N, K, g = 5, 44, 640, 64
    W = synth.weights(N, K, 23)
    X = synth.activations(M, K, 23)
    r = o.weight_quant(synth.bits(W), g)
    Xq, sx = o.act_quant(synth.bits(X))
    acc1, Y1 = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g)
    w8 = o.dequant_weights(r["q4"], r["s2"], r["z"], g).astype(np.int64)
    ref = Xq.astype(np.int64) @ w8.T
    for threads in (2, 3, 4, 7, 44, 100):
        acc, Y = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g, threads=threads)
        assert np.array_equal(acc, ref) and np.array_equal(acc, acc1), threads
        assert np.array_equal(Y, Y1), threads
    # worst-case magnitudes through the threaded path: 127 * 120 * K
    Kw = 2048
    r = o.weight_quant(synth.bits(np.full((3, Kw), np.float16(1.0))), 128)
    Xq, sx = o.act_quant(synth.bits(np.full((2, Kw), np.float16(1.0))))
    acc, _ = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], 128, threads=2)
    assert (acc == 127 * 120 * Kw).all()


def check_zero_folded_appendix(o) -> None:
    """The zero-point-folded product on the hand-worked example: the per-group
    row sums and the total, as worked by hand in the golden file."""
    gold = load_golden("appendix_a_g4.txt")
    zf = load_golden("appendix_a_zero_folded_g4.txt")
    g = gold["g"]
    W, X = _appendix_inputs(gold)
    r = o.weight_quant(synth.bits(W), g)
    Xq, sx = o.act_quant(synth.bits(X))
    acc, Y, RS = o.gemm_zero_folded(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g)
    assert RS[0].tolist() == zf["RS"]
    assert (r["z"][0].astype(int) * r["s2"][0]).tolist() == zf["zs"]
    assert int(acc[0, 0]) == zf["acc"] == sum(zf["scaled"]) - sum(zf["correction"])
    assert int(Y[0, 0]) == gold["Y_bits"]
    # embedded at g = 128: the same numbers
    W1, X1 = _appendix_inputs(gold, K=256, embed=True)
    r = o.weight_quant(synth.bits(np.repeat(W1, 128, axis=0)), 128)
    Xq, sx = o.act_quant(synth.bits(X1))
    acc, Y, RS = o.gemm_zero_folded(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], 128)
    assert RS[0].tolist() == zf["RS"] and (acc == zf["acc"]).all() and (Y == gold["Y_bits"]).all()


def check_zero_folded_equals_direct(o) -> None:
    """Distributivity: the folded form equals the direct product of the
    dequantized weights for every group size, including codes and zeros at
    their extremes; row sums equal numpy's per-group sums."""
    rng = np.random.default_rng(31)
    for g in (32, 64, 128, 256):
        M, N, K = 3, 20, 512
        W = synth.weights(N, K, 40 + g)
        X = synth.activations(M, K, 40 + g)
        W[:8] = np.tile(_adversarial_weights()[:8], (1, K // 256))  # constant, zero, alternating, tiny rows
        r = o.weight_quant(synth.bits(W), g)
        Xq, sx = o.act_quant(synth.bits(X))
        acc0, Y0 = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g)
        acc, Y, RS = o.gemm_zero_folded(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g)
        assert np.array_equal(acc, acc0) and np.array_equal(Y, Y0), g
        assert np.array_equal(RS, Xq.astype(np.int64).reshape(M, K // g, g).sum(axis=2)), g
    # raw codes and zero points at their extremes (not produced by the quantizer)
    M, N, K, g = 2, 5, 256, 128
    q4 = rng.integers(0, 16, (N, K)).astype(np.uint8)
    s2 = rng.integers(1, 17, (N, K // g)).astype(np.uint8)
    z = rng.integers(0, 16, (N, K // g)).astype(np.uint8)
    Xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    sx = np.full(M, 0x2000, np.uint16)
    s1 = np.full(N, 0x1000, np.uint16)
    acc0, _ = o.gemm(Xq, sx, q4, s2, z, s1, g)
    acc, _, _ = o.gemm_zero_folded(Xq, sx, q4, s2, z, s1, g)
    assert np.array_equal(acc, acc0)


# ----------------------------------------------------------------- W4Ax --
# COMET explainer, FMPQ and the W4Ax kernel: 128-channel activation blocks,
# the n8 leading (outlier) blocks at 8 bits, the rest at 4 bits, one scale per
# (token, block); the product scales each block's integer partial sum.

def _w4ax_golden_inputs(gold: dict, zf: dict):
    """X [1][256] and W [128][256] of the hand-worked W4Ax example."""
    appx = load_golden("appendix_a_g4.txt")
    K = 256
    Wl = np.zeros(K)
    for j in range(2):
        Wl[128 * j:128 * j + 4] = np.array(appx["Q8"][4 * j:4 * j + 4]) * 2.0 ** -7
    Xl = np.zeros(K)
    Xl[0:4] = np.array(gold["codes0"]) * 2.0 ** -6
    Xl[128:132] = np.array(gold["codes1"]) * 2.0 ** -3
    return f16(Xl).reshape(1, K), np.repeat(f16(Wl).reshape(1, K), 128, axis=0), appx


def check_w4ax_golden(o) -> None:
    gold = load_golden("w4ax_two_blocks.txt")
    X, W, appx = _w4ax_golden_inputs(gold, None)
    codes, sxb = o.act_quant_w4ax(synth.bits(X), gold["n8"])
    assert codes[0, 0:4].tolist() == gold["codes0"] and codes[0, 128:132].tolist() == gold["codes1"]
    assert not codes[0, 4:128].any() and not codes[0, 132:].any()
    assert sxb[0].tolist() == gold["scale_bits"]
    r = o.weight_quant(synth.bits(W), 128)
    acc, Y, blocks = o.gemm_w4ax(codes, sxb, r["q4"], r["s2"], r["z"], r["s1"], 128, want_blocks=True)
    assert (blocks[0] == np.array(gold["acc_blocks"])).all()
    assert (acc == gold["acc_sum"]).all() and (Y == gold["Y_bits"]).all()


def check_w4ax_8bit_blocks(o) -> None:
    """An 8-bit block is the per-token quantizer applied to that block alone."""
    M, K = 5, 512
    X = synth.activations(M, K, 61)
    codes, sxb = o.act_quant_w4ax(synth.bits(X), K // 128)
    for b in range(K // 128):
        cq, cs = o.act_quant(synth.bits(X[:, 128 * b:128 * b + 128]))
        assert np.array_equal(codes[:, 128 * b:128 * b + 128], cq) and np.array_equal(sxb[:, b], cs)


def check_w4ax_4bit_bruteforce(o) -> None:
    """4-bit blocks: s = fp16(amax / 7) and each code the integer in [-7, 7]
    nearest x / s (ties to even), from exact rationals; |s c - x| <= s / 2
    wherever x / s lies within the range."""
    rng = np.random.default_rng(62)
    M, K, n8 = 4, 384, 1
    X = f16(rng.standard_normal((M, K)) * np.array([1.0, 30.0, 0.01, 1.0])[:, None])
    X[3, 128:256] = f16(((np.arange(128) % 15) - 7 + 0.5) * 2.0 ** -4)  # exact ties, amax = 7.5 * 2^-4
    codes, sxb = o.act_quant_w4ax(synth.bits(X), n8)
    for m in range(M):
        for b in range(n8, K // 128):
            blk = X[m, 128 * b:128 * b + 128].astype(np.float64)
            amax = float(np.abs(blk).max())
            s_bits = int(f16(np.float32(amax) / np.float32(7.0)).view(np.uint16)) if amax > 0 else 0
            assert int(sxb[m, b]) == s_bits, (m, b)
            s = float(np.uint16(s_bits).view(np.float16))
            for k in range(128):
                want = 0 if s == 0 else max(-7, min(7, nearest_int_half_even(Fraction(blk[k]) / Fraction(s))))
                assert int(codes[m, 128 * b + k]) == want, (m, b, k)
                if s and abs(blk[k] / s) <= 7.5:
                    assert abs(s * want - blk[k]) <= s / 2 + 1e-12


def check_w4ax_gemm_reduces_to_w4a8(o) -> None:
    """With every block 8-bit and every block of a row sharing its max-abs,
    the block scales all equal the per-token scale: the W4Ax product is the
    W4A8 product, bit for bit."""
    M, N, K = 3, 24, 512
    X = f16(np.clip(synth.activations(M, K, 63).astype(np.float64), -1.0, 1.0))
    X[:, ::128] = f16(np.array([5.0, -2.0, 9.0]))[:, None]  # the row max sits in every block
    W = synth.weights(N, K, 63)
    r = o.weight_quant(synth.bits(W), 128)
    codes, sxb = o.act_quant_w4ax(synth.bits(X), K // 128)
    Xq, sx = o.act_quant(synth.bits(X))
    assert (sxb == sx[:, None]).all() and np.array_equal(codes, Xq)
    acc_ref, Y_ref = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], 128)
    acc, Y = o.gemm_w4ax(codes, sxb, r["q4"], r["s2"], r["z"], r["s1"], 128)
    assert np.array_equal(acc, acc_ref) and np.array_equal(Y, Y_ref)


def check_w4ax_gemm_float_reference(o) -> None:
    """Y against float64 dequant-then-matmul (s_b c) (s1 w8) rounded to fp16:
    equal, or one fp16 unit apart where the two summation orders straddle a
    rounding boundary; the per-block sums against numpy's int64 matmul."""
    M, N, K = 6, 40, 640
    X = synth.activations(M, K, 64)
    W = synth.weights(N, K, 64)
    r = o.weight_quant(synth.bits(W), 64)
    codes, sxb = o.act_quant_w4ax(synth.bits(X), 2)
    acc, Y, blocks = o.gemm_w4ax(codes, sxb, r["q4"], r["s2"], r["z"], r["s1"], 64, want_blocks=True)
    w8 = o.dequant_weights(r["q4"], r["s2"], r["z"], 64).astype(np.int64)
    c = codes.astype(np.int64)
    for b in range(K // 128):
        sl = slice(128 * b, 128 * b + 128)
        assert np.array_equal(blocks[:, :, b], c[:, sl] @ w8[:, sl].T)
    assert np.array_equal(acc, c @ w8.T)
    xd = c * np.repeat(half_val(sxb), 128, axis=1)
    yd = (xd @ (w8 * half_val(r["s1"])[:, None]).T).astype(np.float16)
    ulp = np.abs(Y.view(np.float16).astype(np.int32) - yd.view(np.int16).astype(np.int32))
    got, ref = Y.view(np.int16).astype(np.int32), yd.view(np.int16).astype(np.int32)
    assert (np.abs(got - ref) <= 1).all() and (got == ref).mean() > 0.99


def check_acc_range(o) -> None:
    """|acc| <= 127 * 127 * K stays below 2^31 for K <= 131072 (worst case)."""
    K = 1024
    W = np.full((1, K), np.float16(1.0))
    X = np.full((1, K), np.float16(1.0))
    r = o.weight_quant(synth.bits(W), 128)
    Xq, sx = o.act_quant(synth.bits(X))
    acc, _ = o.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], 128)
    # Q8 = 119 everywhere: group range [0, 119] -> s2 = 8, z = 0, q4 = 15, w8 = 120
    assert int(acc[0, 0]) == 127 * 120 * K


# ------------------------------------------------------------------- norm --
# The norm fused with the activation quantizer ([QS] "Precision Data Flow and
# Activation Quantization Fusion").  Pins: exact rational sums, closed forms
# (constant rows, unit rows), an error bound against the exact normalization
# computed with rationals, and the composition with the pinned quantizer.

def _ulp16(v: float) -> float:
    """Spacing of binary16 values at magnitude v (2^-24 in the subnormal range)."""
    v = abs(v)
    if v < 2.0 ** -14:
        return 2.0 ** -24
    e = int(np.floor(np.log2(v)))
    return 2.0 ** (e - 10)


def _bits16(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def check_norm_exact_stats(o) -> None:
    """S1 = sum x and S2 = sum x^2 are exact (rationals), even across the full
    fp16 range in one row."""
    rng = np.random.default_rng(11)
    K = 512
    X = rng.standard_normal((3, K)).astype(np.float16)
    X[0, :6] = [65504.0, -65504.0, 2.0 ** -24, -(2.0 ** -24), 2.0 ** -14, 3.0 * 2.0 ** -24]
    X[1, :] = np.float16(2.0 ** -24) * rng.integers(1, 1024, K).astype(np.float16)  # subnormals only
    X[2, ::7] = np.float16(60000.0)
    r = o.norm_quant_act(_bits16(X), _bits16(np.ones(K)), kind="rms", eps=1e-3)
    for m in range(3):
        xs = [Fraction(float(v)) for v in X[m].astype(np.float64)]
        s1, s2 = sum(xs), sum(v * v for v in xs)
        assert int(r["S1"][m]) == s1 * 2 ** 24, m
        assert r["S2"][m] == s2 * 2 ** 48, m


def check_norm_layer_constant_row(o) -> None:
    """LayerNorm of a constant row: x - mu = 0, so y = beta exactly, whatever gamma."""
    K = 384
    rng = np.random.default_rng(12)
    X = np.full((2, K), 0.75, np.float16)
    X[1] = np.float16(-3.5)
    gamma = rng.uniform(0.5, 2.0, K).astype(np.float16)
    beta = rng.uniform(-1.0, 1.0, K).astype(np.float16)
    r = o.norm_quant_act(_bits16(X), _bits16(gamma), _bits16(beta), kind="layer", eps=1e-5)
    assert np.array_equal(r["Y"], np.tile(_bits16(beta), (2, 1)))
    assert float(r["mu"][0]) == 0.75 and float(r["mu"][1]) == -3.5


def check_norm_rms_unit_row(o) -> None:
    """RMSNorm of a row of +-1 with gamma = 1 and eps = 2^-30: the mean square is
    1 and 1/sqrt(1 + 2^-30) rounds to 1 in fp32, so y = x."""
    K = 256
    rng = np.random.default_rng(13)
    X = np.where(rng.random((2, K)) < 0.5, -1.0, 1.0).astype(np.float16)
    r = o.norm_quant_act(_bits16(X), _bits16(np.ones(K)), kind="rms", eps=2.0 ** -30)
    assert np.all(r["r"] == np.float32(1.0))
    assert np.array_equal(r["Y"], _bits16(X))


def check_norm_error_bound(o) -> None:
    """y is within half an fp16 ulp plus a few fp32 roundings of the exact
    normalization, computed with rationals (sqrt to 40 digits).  A large eps
    keeps it visible in y."""
    from decimal import Decimal, getcontext

    getcontext().prec = 40
    rng = np.random.default_rng(14)
    K = 96
    X = (rng.standard_normal((4, K)) * np.array([[0.3], [1.0], [0.05], [2.0]])).astype(np.float16)
    X[3] += np.float16(1.5)  # a row with a mean far from zero
    gamma = rng.uniform(0.5, 2.0, K).astype(np.float16)
    beta = rng.uniform(-0.5, 0.5, K).astype(np.float16)
    for kind, eps in (("rms", 0.25), ("layer", 0.125)):
        r = o.norm_quant_act(_bits16(X), _bits16(gamma), _bits16(beta) if kind == "layer" else None,
                             kind=kind, eps=eps)
        y = r["Y"].view(np.float16).astype(np.float64)
        for m in range(X.shape[0]):
            xs = [Fraction(float(v)) for v in X[m].astype(np.float64)]
            mu = sum(xs) / K if kind == "layer" else Fraction(0)
            spread = sum((v - mu) ** 2 for v in xs) / K
            rstar = 1 / (Decimal(spread.numerator) / Decimal(spread.denominator) + Decimal(eps)).sqrt()
            for k in range(K):
                c = (Decimal((xs[k] - mu).numerator) / Decimal((xs[k] - mu).denominator)) * rstar * \
                    Decimal(float(gamma[k]))
                b = Decimal(float(beta[k])) if kind == "layer" else Decimal(0)
                ystar = float(c + b)
                bound = 0.5 * _ulp16(max(abs(ystar), abs(y[m, k]))) + 2.0 ** -24 * (
                    8 * abs(float(c)) + 2 * abs(float(mu)) * float(rstar) * float(gamma[k]) + 2 * abs(float(b))) + 2.0 ** -40
                assert abs(y[m, k] - ystar) <= bound, (kind, m, k, y[m, k], ystar)


def _round_f32(q: Fraction) -> np.float32:
    """The float32 nearest to the rational q, ties to even (no double rounding
    through float64)."""
    c = np.float32(float(q))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = min(cands, key=lambda v: (abs(Fraction(float(v)) - q), int(np.float32(v).view(np.uint32)) & 1))
    return np.float32(best)


def _norm_chain(X, gamma, beta, kind, eps, dtype):
    """The fused norm's arithmetic written out step by step: exact integer row
    statistics, each rounded once to `dtype`, then every operation in `dtype`
    (numpy float32 / float64 operations are IEEE, rounded to nearest), y
    rounded to fp16."""
    f = dtype
    K = X.shape[1]
    Y = np.empty(X.shape, np.float16)
    for m in range(X.shape[0]):
        a = [int(Fraction(float(v)) * 2 ** 24) for v in X[m].astype(np.float64)]
        S1, S2 = sum(a), sum(v * v for v in a)
        rnd = _round_f32 if f is np.float32 else (lambda q: np.float64(float(q)))
        if kind == "rms":
            spread = f(rnd(Fraction(S2)) * f(2.0 ** -48)) / f(K)
            mu = f(0.0)
        else:
            v = K * S2 - S1 * S1
            spread = f(rnd(Fraction(v)) * f(2.0 ** -48)) / (f(K) * f(K))
            mu = f(rnd(Fraction(S1)) * f(2.0 ** -24)) / f(K)
        r = f(1.0) / np.sqrt(f(spread + f(eps)))
        for k in range(K):
            x = f(X[m, k])
            t = f(x - mu) if kind == "layer" else x
            w = f(f(t * r) * f(gamma[k]))
            if kind == "layer":
                w = f(w + f(beta[k]))
            Y[m, k] = np.float16(w)
    return Y


def check_norm_fp32_chain(o) -> None:
    """The norm's reading (every step after the exact row sums in fp32) against
    that chain written out with numpy float32 on exact rationals, bit for bit;
    and, on the same rows, a float64 chain gives other fp16 values, so the pin
    tells the two readings apart."""
    rng = np.random.default_rng(16)
    K = 4096
    X = (rng.standard_normal((6, K)) * np.array([[1.0], [0.07], [3.0], [0.5], [20.0], [0.01]])).astype(np.float16)
    X[2] += np.float16(0.75)
    gamma = rng.uniform(0.5, 1.5, K).astype(np.float16)
    beta = rng.uniform(-0.3, 0.3, K).astype(np.float16)
    eps = 1e-5
    for kind in ("rms", "layer"):
        r = o.norm_quant_act(_bits16(X), _bits16(gamma), _bits16(beta) if kind == "layer" else None,
                             kind=kind, eps=eps)
        y32 = _norm_chain(X, gamma, beta, kind, np.float32(eps), np.float32)
        assert np.array_equal(r["Y"], y32.view(np.uint16)), kind
        y64 = _norm_chain(X, gamma, beta, kind, eps, np.float64)
        assert (y64.view(np.uint16) != r["Y"]).any(), f"{kind}: the rows do not separate the two chains"
        Xq, sx = o.act_quant(y32.view(np.uint16))
        assert np.array_equal(Xq, r["Xq"]) and np.array_equal(sx, r["sx"])


def check_norm_quant_composition(o) -> None:
    """The fused quantization equals the per-token quantizer applied to the
    normalized fp16 rows."""
    rng = np.random.default_rng(15)
    X = (rng.standard_normal((3, 640)) * 3).astype(np.float16)
    gamma = rng.uniform(0.5, 2.0, 640).astype(np.float16)
    beta = rng.uniform(-1, 1, 640).astype(np.float16)
    for kind in ("rms", "layer"):
        r = o.norm_quant_act(_bits16(X), _bits16(gamma), _bits16(beta), kind=kind, eps=1e-6)
        Xq, sx = o.act_quant(r["Y"])
        assert np.array_equal(Xq, r["Xq"]) and np.array_equal(sx, r["sx"])


ALL_CHECKS = [
    check_half_to_double, check_double_to_half, check_appendix_a, check_appendix_a_g128,
    check_fig3_literal, check_level1_bruteforce, check_level2_bruteforce, check_invariants,
    check_error_bounds, check_lossless_grid, check_zero_and_underflow, check_gemm_library,
    check_gemm_threads, check_w4ax_golden, check_w4ax_8bit_blocks, check_w4ax_4bit_bruteforce,
    check_w4ax_gemm_reduces_to_w4a8, check_w4ax_gemm_float_reference, check_zero_folded_appendix, check_zero_folded_equals_direct, check_acc_range, check_norm_exact_stats, check_norm_layer_constant_row, check_norm_rms_unit_row,
    check_norm_error_bound, check_norm_fp32_chain, check_norm_quant_composition,
]
