"""The quantizers' divide-free rounding (rint_div_fp16 in csrc/ptx.cuh) equals
rint(fl32(x / s)) with an IEEE fp32 divide -- the rule the oracle follows --
for every fp16 x and a broad set of fp16 scales s (CPU emulation of the same
float32 operations; exhaustive over x)."""
import numpy as np


def _rint_div_fp16(x: np.ndarray, s: np.float32) -> np.ndarray:
    x = x.astype(np.float32)
    r = np.float32(1.0) / s  # rcp_rn: the correctly rounded reciprocal
    y = (x * r).astype(np.float32)
    f = np.floor(y).astype(np.float32)
    # fma(f + 0.5, s, -x) == 0, evaluated exactly ((f + 1/2) * s fits in 53 bits)
    tie = ((f.astype(np.float64) + 0.5) * np.float64(s) - x.astype(np.float64)) == 0.0
    even = np.where(f.astype(np.int64) % 2 == 0, f, f + 1)
    return np.where(tie, even, np.rint(y)).astype(np.float32)


def _reference(x: np.ndarray, s: np.float32) -> np.ndarray:
    q = (x.astype(np.float32) / s).astype(np.float32)  # IEEE binary32 divide
    return np.rint(q).astype(np.float32)  # ties to even


def test_divide_free_rounding_matches_ieee_divide():
    allx = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    allx = allx[np.isfinite(allx)].astype(np.float32)
    rng = np.random.default_rng(0)
    scales = set()
    for b in rng.integers(1, 0x7BFF, 3000):  # random positive finite fp16 scales
        scales.add(int(b))
    for e in range(1, 31):  # powers of two and their neighbours (exact ties live there)
        for m in (0, 1, 2, 0x3FF, 0x200):
            scales.add((e << 10) | m)
    for m in range(1, 1024, 37):  # subnormal scales
        scales.add(m)
    checked = 0
    for b in sorted(scales):
        s = np.float32(np.array([b], np.uint16).view(np.float16)[0])
        if not np.isfinite(s) or s <= 0:
            continue
        x = allx[np.abs(allx) <= np.float32(130.0) * s]
        if x.size == 0:
            continue
        got = _rint_div_fp16(x, s)
        want = _reference(x, s)
        bad = got != want
        assert not bad.any(), (float(s), x[bad][:5], got[bad][:5], want[bad][:5])
        checked += x.size
    assert checked > 1_000_000
