"""Plain CPU oracle for the QoQ W4A8 g128 linear layer (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA product path never imports it.

The arithmetic lives in ``qoq_oracle.c`` (plain C, one function per step of
the method, each citing the page passage it follows).  This module compiles it
with gcc on first use and wraps it with numpy-level functions; it adds no
arithmetic of its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "qoq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_LOCK = threading.Lock()

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]


def compile_source(src: str, out: str) -> str:
    """gcc one C file into a shared library (portable C11, no target flags)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm", "-lpthread"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile qoq_oracle.c into oracle/_build/liboracle.so."""
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SRC):
        compile_source(SRC, LIB_PATH)
    return LIB_PATH


class OracleError(RuntimeError):
    pass


def host_cores() -> int:
    """Host threads this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc == 1:
        raise OracleError(f"{what}: bad arguments")
    return rc


class Oracle:
    """numpy-level wrapper around one build of qoq_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        lib.qoq_oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.qoq_oracle_half_to_double.restype = ctypes.c_double
        lib.qoq_oracle_double_to_half.argtypes = [ctypes.c_double]
        lib.qoq_oracle_double_to_half.restype = ctypes.c_uint16
        lib.qoq_oracle_dequant_code.argtypes = [ctypes.c_int64] * 3
        lib.qoq_oracle_dequant_code.restype = ctypes.c_int64
        lib.qoq_oracle_dequant_real.argtypes = [ctypes.c_double] * 3
        lib.qoq_oracle_dequant_real.restype = ctypes.c_double
        lib.qoq_oracle_weight_quant.argtypes = [i32, i32, i32, P, P, P, P, P, P]
        lib.qoq_oracle_weight_quant.restype = i32
        lib.qoq_oracle_dequant_weights.argtypes = [i32, i32, i32, P, P, P, P]
        lib.qoq_oracle_dequant_weights.restype = i32
        lib.qoq_oracle_act_quant.argtypes = [i32, i32, P, P, P]
        lib.qoq_oracle_act_quant.restype = i32
        lib.qoq_oracle_gemm.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P]
        lib.qoq_oracle_gemm.restype = i32
        lib.qoq_oracle_gemm_threads.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, i32]
        lib.qoq_oracle_gemm_threads.restype = i32
        lib.qoq_oracle_gemm_zero_folded.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
        lib.qoq_oracle_gemm_zero_folded.restype = i32
        lib.qoq_oracle_act_quant_w4ax.argtypes = [i32, i32, i32, P, P, P]
        lib.qoq_oracle_act_quant_w4ax.restype = i32
        lib.qoq_oracle_gemm_w4ax.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
        lib.qoq_oracle_gemm_w4ax.restype = i32
        lib.qoq_oracle_gemm_entries.argtypes = [i32, P, P, i32, i32, P, P, P, P, P, P, P, P]
        lib.qoq_oracle_gemm_entries.restype = i32
        lib.qoq_oracle_norm_quant_act.argtypes = [i32, i32, i32, ctypes.c_float, P, P, P, P, P, P, P, P]
        lib.qoq_oracle_norm_quant_act.restype = i32
        self.lib = lib
        self.path = path

    # ------------------------------------------------------------ scalars --
    def half_to_double(self, b: int) -> float:
        return self.lib.qoq_oracle_half_to_double(int(b) & 0xFFFF)

    def double_to_half(self, x: float) -> int:
        return int(self.lib.qoq_oracle_double_to_half(float(x)))

    def dequant_code(self, q: int, zero: int, scale: int) -> int:
        return int(self.lib.qoq_oracle_dequant_code(q, zero, scale))

    def dequant_real(self, q: float, zero: float, scale: float) -> float:
        return float(self.lib.qoq_oracle_dequant_real(q, zero, scale))

    # ------------------------------------------------------------- arrays --
    def weight_quant(self, W_bits: np.ndarray, g: int = 128) -> dict:
        """Progressive group quantization of fp16 weights W [N][K] (uint16 bits).

        Returns s1 [N] (fp16 bits), Q8 [N][K] int8, q4 [N][K] uint8 (one code
        per byte), s2 [N][K/g] uint8 and z [N][K/g] uint8.
        """
        W = _c(W_bits, np.uint16)
        N, K = W.shape
        G = K // g if g > 0 else 0
        s1 = np.empty(N, np.uint16)
        Q8 = np.empty((N, K), np.int8)
        q4 = np.empty((N, K), np.uint8)
        s2 = np.empty((N, max(G, 1)), np.uint8)
        z = np.empty((N, max(G, 1)), np.uint8)
        _check(self.lib.qoq_oracle_weight_quant(N, K, g, _p(W), _p(s1), _p(Q8), _p(q4), _p(s2),
                                                _p(z)), "weight_quant")
        return {"s1": s1, "Q8": Q8, "q4": q4, "s2": np.ascontiguousarray(s2[:, :G]),
                "z": np.ascontiguousarray(z[:, :G])}

    def dequant_weights(self, q4, s2, z, g: int = 128) -> np.ndarray:
        q4 = _c(q4, np.uint8)
        N, K = q4.shape
        w8 = np.empty((N, K), np.int16)
        _check(self.lib.qoq_oracle_dequant_weights(N, K, g, _p(q4), _p(_c(s2, np.uint8)),
                                                   _p(_c(z, np.uint8)), _p(w8)), "dequant_weights")
        return w8

    def act_quant(self, X_bits: np.ndarray):
        """Per-token symmetric int8 quantization of fp16 X [M][K] -> (Xq, sx bits)."""
        X = _c(X_bits, np.uint16)
        M, K = X.shape
        Xq = np.empty((M, K), np.int8)
        sx = np.empty(M, np.uint16)
        _check(self.lib.qoq_oracle_act_quant(M, K, _p(X), _p(Xq), _p(sx)), "act_quant")
        return Xq, sx

    def gemm(self, Xq, sx, q4, s2, z, s1, g: int = 128, want_acc: bool = True, threads: int = 1):
        """acc [M][N] int64 (or None) and Y [M][N] fp16 bits.  threads > 1 runs
        qoq_oracle_gemm_threads on that many host threads (0: all cores)."""
        Xq = _c(Xq, np.int8)
        q4 = _c(q4, np.uint8)
        M, K = Xq.shape
        N = q4.shape[0]
        acc = np.empty((M, N), np.int64) if want_acc else None
        Y = np.empty((M, N), np.uint16)
        if threads == 0:
            threads = host_cores()
        args = (M, N, K, g, _p(Xq), _p(_c(sx, np.uint16)), _p(q4), _p(_c(s2, np.uint8)), _p(_c(z, np.uint8)),
                _p(_c(s1, np.uint16)), _p(acc), _p(Y))
        if threads == 1:
            rc = _check(self.lib.qoq_oracle_gemm(*args), "gemm")
        else:
            rc = _check(self.lib.qoq_oracle_gemm_threads(*args, int(threads)), "gemm_threads")
        if rc == 2:
            raise OracleError("gemm: |acc| reached 2^31")
        return acc, Y

    def gemm_zero_folded(self, Xq, sx, q4, s2, z, s1, g: int = 128):
        """The product in its zero-point-folded form: returns (acc [M][N] int64,
        Y [M][N] fp16 bits, RS [M][K/g] int64 per-group row sums of Xq)."""
        Xq = _c(Xq, np.int8)
        q4 = _c(q4, np.uint8)
        M, K = Xq.shape
        N = q4.shape[0]
        acc = np.empty((M, N), np.int64)
        Y = np.empty((M, N), np.uint16)
        RS = np.empty((M, K // g), np.int64)
        rc = _check(self.lib.qoq_oracle_gemm_zero_folded(M, N, K, g, _p(Xq), _p(_c(sx, np.uint16)), _p(q4),
                                                         _p(_c(s2, np.uint8)), _p(_c(z, np.uint8)),
                                                         _p(_c(s1, np.uint16)), _p(RS), _p(acc), _p(Y)),
                    "gemm_zero_folded")
        if rc == 2:
            raise OracleError("gemm_zero_folded: |acc| reached 2^31")
        return acc, Y, RS

    def act_quant_w4ax(self, X_bits: np.ndarray, n8: int):
        """W4Ax activations of fp16 X [M][K]: the n8 leading 128-channel blocks
        8-bit, the rest 4-bit, one symmetric scale per (token, block).
        Returns (codes [M][K] int8, sxb [M][K/128] fp16 bits)."""
        X = _c(X_bits, np.uint16)
        M, K = X.shape
        codes = np.empty((M, K), np.int8)
        sxb = np.empty((M, K // 128), np.uint16)
        _check(self.lib.qoq_oracle_act_quant_w4ax(M, K, int(n8), _p(X), _p(codes), _p(sxb)), "act_quant_w4ax")
        return codes, sxb

    def gemm_w4ax(self, codes, sxb, q4, s2, z, s1, g: int = 128, want_blocks: bool = False):
        """W4Ax product: (acc_sum [M][N] int64, Y [M][N] fp16 bits, and
        acc_blocks [M][N][K/128] int64 when want_blocks)."""
        codes = _c(codes, np.int8)
        q4 = _c(q4, np.uint8)
        M, K = codes.shape
        N = q4.shape[0]
        acc = np.empty((M, N), np.int64)
        Y = np.empty((M, N), np.uint16)
        blocks = np.empty((M, N, K // 128), np.int64) if want_blocks else None
        _check(self.lib.qoq_oracle_gemm_w4ax(M, N, K, g, _p(codes), _p(_c(sxb, np.uint16)), _p(q4),
                                             _p(_c(s2, np.uint8)), _p(_c(z, np.uint8)), _p(_c(s1, np.uint16)),
                                             _p(blocks), _p(acc), _p(Y)), "gemm_w4ax")
        return (acc, Y, blocks) if want_blocks else (acc, Y)

    def gemm_entries(self, m_idx, n_idx, Xq, sx, q4, s2, z, s1, g: int = 128):
        """acc and Y for the listed (m, n) entries only."""
        m_idx = _c(m_idx, np.int32)
        n_idx = _c(n_idx, np.int32)
        Xq = _c(Xq, np.int8)
        q4 = _c(q4, np.uint8)
        K = Xq.shape[1]
        cnt = int(m_idx.shape[0])
        acc = np.empty(cnt, np.int64)
        Y = np.empty(cnt, np.uint16)
        _check(self.lib.qoq_oracle_gemm_entries(cnt, _p(m_idx), _p(n_idx), K, g, _p(Xq),
                                                _p(_c(sx, np.uint16)), _p(q4), _p(_c(s2, np.uint8)),
                                                _p(_c(z, np.uint8)), _p(_c(s1, np.uint16)), _p(acc),
                                                _p(Y)), "gemm_entries")
        return acc, Y


    def norm_quant_act(self, X_bits, gamma_bits, beta_bits=None, kind: str = "rms", eps: float = 1e-6):
        """The norm (RMSNorm, or LayerNorm with beta) fused with the per-token
        int8 quantizer, on fp16 X [M][K] (uint16 bits).  Returns a dict with
        Y (the fp16 normalized rows, bits), Xq, sx (bits), r and mu per row
        (float32) and the exact row sums S1 (units 2^-24) and S2 (units 2^-48,
        as a Python int per row)."""
        X = _c(X_bits, np.uint16)
        M, K = X.shape
        k = {"rms": 0, "layer": 1}[kind]
        g = _c(gamma_bits, np.uint16)
        b = None if beta_bits is None else _c(beta_bits, np.uint16)
        Y = np.empty((M, K), np.uint16)
        Xq = np.empty((M, K), np.int8)
        sx = np.empty(M, np.uint16)
        rmu = np.empty((M, 2), np.float32)
        st = np.empty((M, 4), np.int64)
        _check(self.lib.qoq_oracle_norm_quant_act(M, K, k, float(eps), _p(X), _p(g), None if b is None else _p(b),
                                                  _p(Y), _p(Xq), _p(sx), _p(rmu), _p(st)), "norm_quant_act")
        S2 = [int(np.uint64(st[i, 1])) + (int(np.uint64(st[i, 2])) << 64) for i in range(M)]
        return {"Y": Y, "Xq": Xq, "sx": sx, "r": rmu[:, 0].copy(), "mu": rmu[:, 1].copy(),
                "S1": st[:, 0].copy(), "S2": S2}


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    global _DEFAULT
    with _LOCK:
        if _DEFAULT is None:
            _DEFAULT = Oracle(build())
    return _DEFAULT


def __getattr__(name):
    # module-level shortcuts: oracle.weight_quant(...) etc. use the default build
    if name in ("half_to_double", "double_to_half", "dequant_code", "dequant_real", "weight_quant",
                "dequant_weights", "act_quant", "gemm", "gemm_entries", "norm_quant_act",
                "gemm_zero_folded", "act_quant_w4ax", "gemm_w4ax"):
        return getattr(default(), name)
    raise AttributeError(name)
