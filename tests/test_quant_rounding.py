"""The quantizers' divide-free rounding (quant_bits in csrc/ptx.cuh) equals
clamp(rint(fl32(x / s)), -q, q) with an IEEE fp32 divide -- the rule the
oracle follows -- for fp16 x and s (CPU emulation of the same float32
operations, with an exactly emulated fused multiply-add; exhaustive over x).

Two forms are checked.  The clamped one, for any scale, and the unclamped
one the kernels take when s = fp16_rn(fl32(amax / q)) is a normal fp16
number: then |x / s| <= q (1 + 2^-11) for every |x| <= amax, which never
rounds past q, so the clamp can be left out."""
import numpy as np

MAGIC = np.float32(12582912.0)  # 1.5 * 2^23: adding it rounds to an integer, ties to even
MAGIC_BITS = 0x4B400000


def _fma32(a: np.ndarray, b, c: np.ndarray) -> np.ndarray:
    """fp32 fused multiply-add, rounded once to nearest even.  a * b is
    exact in float64; TwoSum gives the float64 sum and its exact error; the
    float64 sum rounds to the right fp32 value unless it sits exactly on an
    fp32 midpoint, where the error's sign decides."""
    a64, b64, c64 = (np.asarray(v, np.float32).astype(np.float64) for v in (a, b, c))
    p = a64 * b64  # exact (24 + 24 bits)
    s = p + c64
    bb = s - p
    err = (p - (s - bb)) + (c64 - bb)  # s + err = p + c exactly
    r = s.astype(np.float32)
    r64 = r.astype(np.float64)
    toward = np.where(s > r64, np.float32(np.inf), np.float32(-np.inf))
    n = np.nextafter(r, toward.astype(np.float32))
    mid = (s != r64) & ((r64 + n.astype(np.float64)) * 0.5 == s)
    # exactly on a midpoint: round away from it on the side the error points to
    go_n = mid & (err != 0) & ((err > 0) == (n.astype(np.float64) > r64))
    return np.where(go_n, n, r).astype(np.float32)


def _quant(x: np.ndarray, s: np.float32, q: float, clamp: bool) -> np.ndarray:
    """The GPU's steps in float32: y1 = x * rcp_rn(s); e = fma(-y1, s, x), the
    exact remainder; y = fma(e, rcp_rn(s), y1), which is exact wherever x / s
    is a half-integer; optionally clamp y to [-q, q]; the code is the bit
    pattern of y + 1.5 * 2^23 less 0x4B400000 (round to nearest, ties even)."""
    x = x.astype(np.float32)
    rc = np.float32(1.0) / s if s != 0 else np.float32(0.0)  # rcp_rn: the correctly rounded reciprocal
    y1 = (x * rc).astype(np.float32)
    e = _fma32(-y1, s, x)
    y = _fma32(e, rc, y1)
    if clamp:
        y = np.minimum(np.maximum(y, np.float32(-q)), np.float32(q))
    t = (y + MAGIC).astype(np.float32)
    return (t.view(np.int32).astype(np.int64) - MAGIC_BITS).astype(np.float32)


def _reference(x: np.ndarray, s: np.float32, q: float) -> np.ndarray:
    d = (x.astype(np.float32) / s).astype(np.float32)  # IEEE binary32 divide
    return np.clip(np.rint(d), -q, q).astype(np.float32)  # ties to even, then the code range


def _fp16(bits) -> np.float32:
    return np.float32(np.array([bits], np.uint16).view(np.float16)[0])


_ALLX = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
_ALLX = _ALLX[np.isfinite(_ALLX)].astype(np.float32)


def test_fma32_emulation_is_exact():
    """The emulated fma against exact rational arithmetic on random and
    midpoint-heavy operands."""
    from fractions import Fraction
    rng = np.random.default_rng(1)
    a = rng.standard_normal(4000).astype(np.float32)
    b = rng.standard_normal(4000).astype(np.float32)
    c = (-(a.astype(np.float64) * b.astype(np.float64))).astype(np.float32)  # cancellation
    c[::2] = rng.standard_normal(2000).astype(np.float32) * np.float32(2.0 ** -30)
    # a * b exactly on an fp32 midpoint ((1 + k 2^-23) 1.5 with k odd), c far below it
    k = 2 * rng.integers(0, 1 << 20, 1000) + 1
    a[:1000] = (1.0 + k * 2.0 ** -23).astype(np.float32)
    b[:1000] = np.float32(1.5)
    c[:1000] = np.float32(2.0 ** -60) * rng.choice([-1, 0, 1], 1000).astype(np.float32)
    got = _fma32(a, b, c)
    for i in range(a.size):
        exact = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        lo = np.float32(float(exact))  # float() rounds the rational once to float64
        # pick the nearest fp32 (ties even) to the exact rational
        cands = [np.nextafter(lo, np.float32(-np.inf)), lo, np.nextafter(lo, np.float32(np.inf))]
        best = min(cands, key=lambda v: (abs(Fraction(float(v)) - exact), int(np.array(v).view(np.int32)) & 1))
        assert got[i] == best, (a[i], b[i], c[i], got[i], best)


def test_unclamped_codes_match_ieee_divide():
    """s = fp16_rn(fl32(amax / q)) normal: every |x| <= amax gets the IEEE
    divide's code without the clamp, for q = 127 (activations), 119 (level-1
    weights) and 7 (4-bit activation blocks)."""
    rng = np.random.default_rng(0)
    amaxes = set(int(b) for b in rng.integers(0x0400, 0x7BFF, 900))
    for e in range(1, 31):  # powers of two and their neighbours (exact ties live there)
        for m in (0, 1, 2, 0x3FF, 0x200):
            amaxes.add((e << 10) | m)
    checked = 0
    for i, b in enumerate(sorted(amaxes)):
        amax = _fp16(b)
        for q in ((127.0, 119.0, 7.0)[i % 3], (127.0, 119.0, 7.0)[(i + 1) % 3]):
            s = np.float32(np.float16(np.float32(amax) / np.float32(q)))
            if not (s >= np.float32(2.0 ** -14)) or not np.isfinite(s):
                continue
            x = _ALLX[np.abs(_ALLX) <= amax]
            got = _quant(x, s, q, clamp=False)
            want = _reference(x, s, q)
            bad = got != want
            assert not bad.any(), (float(amax), q, x[bad][:5], got[bad][:5], want[bad][:5])
            checked += x.size
    assert checked > 5_000_000


def test_clamped_codes_match_ieee_divide():
    """The clamped form for any positive fp16 scale (subnormal ones too, where
    x / s can pass q) and |x| well past q s."""
    rng = np.random.default_rng(2)
    scales = set(int(b) for b in rng.integers(1, 0x7BFF, 600))
    for m in range(1, 1024, 37):  # subnormal scales
        scales.add(m)
    checked = 0
    for i, b in enumerate(sorted(scales)):
        s = _fp16(b)
        q = (127.0, 119.0, 7.0)[i % 3]
        x = _ALLX[np.abs(_ALLX) <= np.float32(2 * q + 4) * s]
        if x.size == 0:
            continue
        got = _quant(x, s, q, clamp=True)
        want = _reference(x, s, q)
        bad = got != want
        assert not bad.any(), (float(s), q, x[bad][:5], got[bad][:5], want[bad][:5])
        checked += x.size
    assert checked > 300_000


def test_zero_scale_gives_zero_codes():
    """s = 0 (an all-zero row) with rcp = 0: every code is 0, clamped or not."""
    x = _ALLX[np.abs(_ALLX) < 1]
    assert (_quant(x, np.float32(0.0), 127.0, clamp=True) == 0).all()
    assert (_quant(x, np.float32(0.0), 127.0, clamp=False) == 0).all()


def test_rounding_ties_go_to_even():
    """Exact ties x / s = n + 1/2 go to the even code, on both sides of zero,
    including scales that are not powers of two (x = (n + 1/2) s exact in
    fp16)."""
    found = 0
    for sb in (0x2400, 0x3C00, 0x4800, 0x3E00, 0x3A80, 0x2D40):
        s = _fp16(sb)
        n = np.arange(-127, 127, dtype=np.float64)
        x64 = (n + 0.5) * np.float64(s)
        x = x64.astype(np.float16).astype(np.float32)
        x = x[x.astype(np.float64) == x64]  # the tie is representable in fp16
        found += x.size
        got = _quant(x, s, 127.0, clamp=True)
        assert np.array_equal(got, _reference(x, s, 127.0))
        assert (got % 2 == 0).all()
    assert found > 400
