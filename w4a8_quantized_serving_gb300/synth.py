"""Seeded synthetic inputs for the W4A8 linear layer (no method arithmetic here).

Both the oracle tests and the CUDA path draw their inputs from this module; it
holds only random-number generation, nothing of the quantization method.

Recipe (the workload shapes are those of the decode/prefill projections the
QServe write-up and the lecture notes discuss; the value distributions follow
the usual LLM picture of Gaussian weights and activations with a few outlier
input channels):

* generator: splitmix64 (Steele, Lea, Flood 2014), counter-based, so any
  chunk can be produced independently: output i of a stream with start state
  S is mix(S + (i + 1) * 0x9E3779B97F4A7C15), with mix the splitmix64
  finaliser.  A stream's start state is mix(seed * 0x9E3779B97F4A7C15 + tag).
* uniforms: u = (x >> 11) * 2^-53, in [0, 1).
* normals: Box-Muller on consecutive pairs (u1, u2):
  r = sqrt(-2 ln(1 - u1)); n0 = r cos(2 pi u2); n1 = r sin(2 pi u2),
  in float64, row-major over the tensor.
* W [N][K] = N(0, 0.02^2); 2 distinct input channels (columns k) scaled x10.
* X [M][K] = N(0, 1); 4 distinct input channels scaled x20.
* outlier channels: uniforms from a separate stream, k = floor(u * K),
  duplicates skipped, in draw order.
* every value is rounded once from float64 to fp16 (nearest-even).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TAG_W = 0x57
TAG_X = 0x58
TAG_OUTLIER = 0x100


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_start(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(int(seed) * int(GAMMA) + int(tag)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(s)[0]


def u64(start: np.uint64, offset: int, n: int) -> np.ndarray:
    """Outputs offset .. offset+n-1 of the splitmix64 stream with start state `start`."""
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(start + i * GAMMA)


def uniforms(start: np.uint64, offset: int, n: int) -> np.ndarray:
    return (u64(start, offset, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(start: np.uint64, offset: int, n: int) -> np.ndarray:
    """Normals offset .. offset+n-1 (offset must be even)."""
    assert offset % 2 == 0
    npairs = (n + 1) // 2
    u = uniforms(start, offset, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    out = np.empty(2 * npairs, np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:n]


def outlier_channels(seed: int, tag: int, K: int, count: int) -> np.ndarray:
    start = stream_start(seed, tag + TAG_OUTLIER)
    picked: list[int] = []
    off = 0
    while len(picked) < min(count, K):
        u = uniforms(start, off, 64)
        off += 64
        for v in u:
            k = int(v * K)
            if k not in picked:
                picked.append(k)
                if len(picked) == min(count, K):
                    break
    return np.array(picked, dtype=np.int64)


def _gaussian_fp16(seed: int, tag: int, rows: int, K: int, sigma: float, n_out: int, out_scale: float,
                   chunk_rows: int | None = None) -> np.ndarray:
    start = stream_start(seed, tag)
    cols = outlier_channels(seed, tag, K, n_out)
    colscale = np.ones(K, np.float64)
    colscale[cols] = out_scale
    out = np.empty((rows, K), np.float16)
    if chunk_rows is None:
        chunk_rows = max(1, (1 << 20) // max(K, 1))
    # keep chunk offsets even so Box-Muller pairs never straddle a chunk edge
    if (chunk_rows * K) % 2:
        chunk_rows += 1

    def fill(r0: int) -> None:
        r1 = min(rows, r0 + chunk_rows)
        v = normals(start, r0 * K, (r1 - r0) * K).reshape(r1 - r0, K)
        out[r0:r1] = (v * sigma * colscale).astype(np.float16)

    starts = list(range(0, rows, chunk_rows))
    if len(starts) > 1:
        # chunks are independent (counter-based stream); numpy releases the GIL
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, starts))
    else:
        for r0 in starts:
            fill(r0)
    return out


def weights(N: int, K: int, seed: int) -> np.ndarray:
    """fp16 W [N][K]: N(0, 0.02^2) with 2 outlier input channels x10."""
    return _gaussian_fp16(seed, TAG_W, N, K, 0.02, 2, 10.0)


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """fp16 X [M][K]: N(0, 1) with 4 outlier input channels x20."""
    return _gaussian_fp16(seed, TAG_X, M, K, 1.0, 4, 20.0)


def bits(a: np.ndarray) -> np.ndarray:
    """fp16 array -> its uint16 bit patterns (a view)."""
    return np.ascontiguousarray(a, dtype=np.float16).view(np.uint16)


# The five workloads: (M, N, K, seed).  g = 128 for all of them.
WORKLOADS = {
    0: dict(name="tiny", M=8, N=256, K=512, seed=0),
    1: dict(name="decode_qkv_7b", M=16, N=12288, K=4096, seed=1),
    2: dict(name="decode_gate_up_7b", M=128, N=22016, K=4096, seed=2),
    3: dict(name="decode_down_8b_b256", M=256, N=4096, K=14336, seed=3),
    4: dict(name="prefill_up_70b", M=4096, N=28672, K=8192, seed=4),
}
