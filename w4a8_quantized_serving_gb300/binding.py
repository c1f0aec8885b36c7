"""ctypes binding of libqoq.so (include/qoq.h): argument marshalling only.

Each function takes torch CUDA tensors (fp16 values as torch.float16, whose
bits are the ABI's uint16), allocates outputs with torch when the caller
passes none, and calls the C entry point of the same name on the current
torch stream (or the given one).  A non-zero status raises QoQError.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .csrc import build as _build

QOQ_ERRORS = {
    0: "QOQ_OK", 1: "QOQ_ERR_NULL", 2: "QOQ_ERR_SHAPE", 3: "QOQ_ERR_UNSUPPORTED",
    4: "QOQ_ERR_MISALIGNED", 5: "QOQ_ERR_WORKSPACE", 6: "QOQ_ERR_CUDA",
    7: "QOQ_ERR_DEVICE_TIMEOUT", 8: "QOQ_ERR_ARCH",
}

EXPORTED = (
    "qoq_status_str", "qoq_version", "qoq_packed_weight_bytes", "qoq_gemm_workspace_bytes",
    "qoq_pack_weights", "qoq_quant_act", "qoq_norm_quant_act", "qoq_w4a8_gemm", "qoq_unpack_weights_debug",
    "qoq_last_device_status", "qoq_no_alloc_last_status", "qoq_set_debug", "qoq_w4a8_gemm_no_alloc", "qoq_w4a8_gemm_zero_folded",
    "qoq_w4ax_act_bytes", "qoq_quant_act_w4ax", "qoq_w4ax_workspace_bytes", "qoq_w4ax_gemm",
)

_LOCK = threading.Lock()
_LIB = None


class QoQError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {QOQ_ERRORS.get(code, code)}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def build(force: bool = False) -> str:
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = library_path()
            if not os.path.exists(path):
                raise QoQError(6, f"libqoq.so not found at {path} (run __graft_entry__.build())")
            L = ctypes.CDLL(path)
            i32, u64, sz, P = ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
            L.qoq_status_str.argtypes = [i32]
            L.qoq_status_str.restype = ctypes.c_char_p
            L.qoq_version.argtypes = []
            L.qoq_version.restype = i32
            L.qoq_packed_weight_bytes.argtypes = [i32, i32, i32]
            L.qoq_packed_weight_bytes.restype = sz
            L.qoq_gemm_workspace_bytes.argtypes = [i32, i32, i32, i32]
            L.qoq_gemm_workspace_bytes.restype = sz
            L.qoq_pack_weights.argtypes = [i32, i32, i32, P, P, P, P]
            L.qoq_pack_weights.restype = i32
            L.qoq_quant_act.argtypes = [i32, i32, P, P, P, P]
            L.qoq_quant_act.restype = i32
            L.qoq_norm_quant_act.argtypes = [i32, i32, i32, ctypes.c_float, P, P, P, P, P, P]
            L.qoq_norm_quant_act.restype = i32
            L.qoq_w4a8_gemm.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
            L.qoq_w4a8_gemm.restype = i32
            L.qoq_w4ax_act_bytes.argtypes = [i32, i32, i32]
            L.qoq_w4ax_act_bytes.restype = sz
            L.qoq_w4ax_workspace_bytes.argtypes = [i32, i32, i32, i32]
            L.qoq_w4ax_workspace_bytes.restype = sz
            L.qoq_quant_act_w4ax.argtypes = [i32, i32, i32, P, P, P, P]
            L.qoq_quant_act_w4ax.restype = i32
            L.qoq_w4ax_gemm.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
            L.qoq_w4ax_gemm.restype = i32
            L.qoq_w4a8_gemm_zero_folded.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
            L.qoq_w4a8_gemm_zero_folded.restype = i32
            L.qoq_w4a8_gemm_no_alloc.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P]
            L.qoq_w4a8_gemm_no_alloc.restype = i32
            L.qoq_no_alloc_last_status.argtypes = [P]
            L.qoq_no_alloc_last_status.restype = i32
            L.qoq_unpack_weights_debug.argtypes = [i32, i32, i32, P, P, P, P, P]
            L.qoq_unpack_weights_debug.restype = i32
            L.qoq_last_device_status.argtypes = [P, P]
            L.qoq_last_device_status.restype = i32
            L.qoq_set_debug.argtypes = [u64, i32]
            L.qoq_set_debug.restype = i32
            _LIB = L
    return _LIB


def _check(code: int, what: str) -> None:
    if code != 0:
        raise QoQError(code, what)


def _torch():
    import torch

    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t, dtype, name: str, shape=None, host_ok: bool = False):
    """Device address of tensor t, checked; with host_ok, a pinned (page-locked)
    host tensor is accepted too and the kernels access it in place."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_cuda and not (host_ok and t.device.type == "cpu" and t.is_pinned()):
        raise TypeError(f"{name} must be a CUDA tensor" + (" or a pinned host tensor" if host_ok else ""))
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


# ---------------------------------------------------------------- host-only --

def qoq_status_str(code: int) -> str:
    return lib().qoq_status_str(int(code)).decode()


def qoq_version() -> int:
    return int(lib().qoq_version())


def qoq_packed_weight_bytes(N: int, K: int, g: int = 128) -> int:
    return int(lib().qoq_packed_weight_bytes(N, K, g))


def qoq_gemm_workspace_bytes(M: int, N: int, K: int, g: int = 128) -> int:
    return int(lib().qoq_gemm_workspace_bytes(M, N, K, g))


def qoq_set_debug(wait_timeout_ns: int = 0, fault: int = 0) -> None:
    _check(lib().qoq_set_debug(int(wait_timeout_ns), int(fault)), "qoq_set_debug")


# ------------------------------------------------------------------- device --

def qoq_pack_weights(W, g: int = 128, packed=None, s1=None, stream=None):
    """W fp16 [N][K] -> (packed uint8 blob, s1 fp16 [N])."""
    torch = _torch()
    N, K = W.shape
    nbytes = qoq_packed_weight_bytes(N, K, g)
    if packed is None:
        packed = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=W.device)
    if s1 is None:
        s1 = torch.empty(N, dtype=torch.float16, device=W.device)
    _check(lib().qoq_pack_weights(N, K, g, _dev(W, torch.float16, "W"), _dev(packed, torch.uint8, "packed"),
                                  _dev(s1, torch.float16, "s1", (N,)), _stream(stream)), "qoq_pack_weights")
    return packed, s1


def _out_device(t):
    """Where outputs go by default: t's device, or the current CUDA device for
    a pinned host tensor."""
    torch = _torch()
    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def qoq_quant_act(X, Xq=None, sx=None, stream=None):
    """X fp16 [M][K] (CUDA, or pinned host: read in place) -> (Xq int8 [M][K], sx fp16 [M])."""
    torch = _torch()
    M, K = X.shape
    xp = _dev(X, torch.float16, "X", host_ok=True)
    if Xq is None:
        Xq = torch.empty((M, K), dtype=torch.int8, device=_out_device(X))
    if sx is None:
        sx = torch.empty(M, dtype=torch.float16, device=_out_device(X))
    _check(lib().qoq_quant_act(M, K, xp, _dev(Xq, torch.int8, "Xq", (M, K)),
                               _dev(sx, torch.float16, "sx", (M,)), _stream(stream)), "qoq_quant_act")
    return Xq, sx


NORM_KINDS = {"rms": 0, "layer": 1}


def qoq_norm_quant_act(X, gamma, beta=None, kind: str = "rms", eps: float = 1e-6, Xq=None, sx=None, stream=None):
    """RMSNorm (or LayerNorm with beta) fused with the per-token int8 quantizer:
    X fp16 [M][K] (CUDA, or pinned host: read in place), gamma (and beta) fp16
    [K] -> (Xq int8 [M][K], sx fp16 [M])."""
    torch = _torch()
    M, K = X.shape
    if kind not in NORM_KINDS:
        raise ValueError(f"kind must be one of {sorted(NORM_KINDS)}")
    xp = _dev(X, torch.float16, "X", host_ok=True)
    if Xq is None:
        Xq = torch.empty((M, K), dtype=torch.int8, device=_out_device(X))
    if sx is None:
        sx = torch.empty(M, dtype=torch.float16, device=_out_device(X))
    bptr = None if beta is None else _dev(beta, torch.float16, "beta", (K,))
    _check(lib().qoq_norm_quant_act(M, K, NORM_KINDS[kind], float(eps), xp,
                                    _dev(gamma, torch.float16, "gamma", (K,)), bptr,
                                    _dev(Xq, torch.int8, "Xq", (M, K)), _dev(sx, torch.float16, "sx", (M,)),
                                    _stream(stream)), "qoq_norm_quant_act")
    return Xq, sx


def qoq_w4a8_gemm(Xq, sx, packed, s1, N: int | None = None, g: int = 128, Y=None, acc_debug=None,
                  workspace=None, stream=None):
    """Y fp16 [M][N] = W4A8 GEMM of (Xq, sx) with the packed weights (and s1).
    Y may be a pinned host tensor: the kernel writes it in place."""
    return _gemm("qoq_w4a8_gemm", Xq, sx, packed, s1, N, g, Y, acc_debug, workspace, stream)


def qoq_w4a8_gemm_zero_folded(Xq, sx, packed, s1, N: int | None = None, g: int = 128, Y=None, acc_debug=None,
                              workspace=None, stream=None):
    """The same GEMM with the zero points folded into the epilogue (q4 * s2 in
    the main loop, minus z * s2 times the per-group row sums of Xq); g must be
    a multiple of 128."""
    return _gemm("qoq_w4a8_gemm_zero_folded", Xq, sx, packed, s1, N, g, Y, acc_debug, workspace, stream)


def _gemm(name, Xq, sx, packed, s1, N, g, Y, acc_debug, workspace, stream):
    torch = _torch()
    M, K = Xq.shape
    if N is None:
        N = s1.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=Xq.device)
    ws_need = qoq_gemm_workspace_bytes(M, N, K, g)
    if workspace is None:  # zero-filled once; every completed call leaves it zeroed
        workspace = torch.zeros(max(ws_need, 16), dtype=torch.uint8, device=Xq.device)
    acc_ptr = None if acc_debug is None else _dev(acc_debug, torch.int32, "acc_debug", (M, N))
    code = getattr(lib(), name)(M, N, K, g, _dev(Xq, torch.int8, "Xq"), _dev(sx, torch.float16, "sx", (M,)),
                                _dev(packed, torch.uint8, "packed"), _dev(s1, torch.float16, "s1", (N,)),
                                _dev(Y, torch.float16, "Y", (M, N), host_ok=True), acc_ptr,
                                _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(code, name)
    return Y


def qoq_w4a8_gemm_no_alloc(Xq, sx, packed, s1, N: int | None = None, g: int = 128, Y=None,
                           acc_debug=None, stream=None):
    """qoq_w4a8_gemm with the library's own fixed device scratch instead of a
    caller workspace (for callers that cannot allocate device memory; calls
    that overlap on the GPU race on that scratch).  Pass Y (and acc_debug) to
    keep the call itself free of allocation."""
    torch = _torch()
    M, K = Xq.shape
    if N is None:
        N = s1.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=Xq.device)
    acc_ptr = None if acc_debug is None else _dev(acc_debug, torch.int32, "acc_debug", (M, N))
    code = lib().qoq_w4a8_gemm_no_alloc(M, N, K, g, _dev(Xq, torch.int8, "Xq"),
                                        _dev(sx, torch.float16, "sx", (M,)),
                                        _dev(packed, torch.uint8, "packed"),
                                        _dev(s1, torch.float16, "s1", (N,)),
                                        _dev(Y, torch.float16, "Y", (M, N), host_ok=True), acc_ptr, _stream(stream))
    _check(code, "qoq_w4a8_gemm_no_alloc")
    return Y


def qoq_w4ax_act_bytes(M: int, K: int, n8: int) -> int:
    return int(lib().qoq_w4ax_act_bytes(M, K, n8))


def qoq_w4ax_workspace_bytes(M: int, N: int, K: int, g: int = 128) -> int:
    return int(lib().qoq_w4ax_workspace_bytes(M, N, K, g))


def qoq_quant_act_w4ax(X, n8: int, Xa=None, sxb=None, stream=None):
    """W4Ax activations of fp16 X [M][K]: the n8 leading 128-channel blocks
    8-bit, the rest 4-bit (two codes per byte), one fp16 scale per (token,
    block).  Returns (Xa uint8 [M][row bytes], sxb fp16 [M][K/128])."""
    torch = _torch()
    M, K = X.shape
    dev = _out_device(X)
    row = qoq_w4ax_act_bytes(1, K, n8)
    if Xa is None:
        Xa = torch.empty((M, row), dtype=torch.uint8, device=dev)
    if sxb is None:
        sxb = torch.empty((M, K // 128), dtype=torch.float16, device=dev)
    _check(lib().qoq_quant_act_w4ax(M, K, n8, _dev(X, torch.float16, "X", (M, K), host_ok=True),
                                    _dev(Xa, torch.uint8, "Xa"), _dev(sxb, torch.float16, "sxb", (M, K // 128)),
                                    _stream(stream)), "qoq_quant_act_w4ax")
    return Xa, sxb


def qoq_w4ax_gemm(Xa, sxb, n8: int, packed, s1, K: int, N: int | None = None, g: int = 128, Y=None,
                  acc_debug=None, workspace=None, stream=None):
    """Y fp16 [M][N] = the W4Ax GEMM of (Xa, sxb) with the packed 4-bit weights."""
    torch = _torch()
    M = sxb.shape[0]
    if N is None:
        N = s1.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=sxb.device)
    if workspace is None:
        workspace = torch.zeros(max(qoq_w4ax_workspace_bytes(M, N, K, g), 16), dtype=torch.uint8,
                                device=sxb.device)
    acc_ptr = None if acc_debug is None else _dev(acc_debug, torch.int32, "acc_debug", (M, N))
    code = lib().qoq_w4ax_gemm(M, N, K, g, n8, _dev(Xa, torch.uint8, "Xa"),
                               _dev(sxb, torch.float16, "sxb", (M, K // 128)), _dev(packed, torch.uint8, "packed"),
                               _dev(s1, torch.float16, "s1", (N,)), _dev(Y, torch.float16, "Y", (M, N), host_ok=True),
                               acc_ptr, _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(code, "qoq_w4ax_gemm")
    return Y


def qoq_unpack_weights_debug(packed, N: int, K: int, g: int = 128, stream=None):
    """packed -> (q4 uint8 [N][K], s2 uint8 [N][K/g], z uint8 [N][K/g])."""
    torch = _torch()
    dev = packed.device
    q4 = torch.empty((N, K), dtype=torch.uint8, device=dev)
    s2 = torch.empty((N, K // g), dtype=torch.uint8, device=dev)
    z = torch.empty((N, K // g), dtype=torch.uint8, device=dev)
    _check(lib().qoq_unpack_weights_debug(N, K, g, _dev(packed, torch.uint8, "packed"), q4.data_ptr(),
                                          s2.data_ptr(), z.data_ptr(), _stream(stream)),
           "qoq_unpack_weights_debug")
    return q4, s2, z


def workspace_for(M: int, N: int, K: int, g: int = 128, device="cuda"):
    """A zero-filled workspace for qoq_w4a8_gemm at (M, N, K)."""
    torch = _torch()
    return torch.zeros(max(qoq_gemm_workspace_bytes(M, N, K, g), 16), dtype=torch.uint8, device=device)


def qoq_last_device_status(workspace, stream=None) -> int:
    """Synchronize and return (then clear) the last GEMM's device status code."""
    torch = _torch()
    return int(lib().qoq_last_device_status(_dev(workspace, torch.uint8, "workspace"), _stream(stream)))


def qoq_no_alloc_last_status(stream=None) -> int:
    """Synchronize and return (then reset) the sticky device status of the
    qoq_w4a8_gemm_no_alloc calls since the previous read."""
    return int(lib().qoq_no_alloc_last_status(_stream(stream)))


class QoQLinear:
    """A W4A8 linear layer: weights packed once, Y = X W^T per call.

    Holds the packed weights, s1, and one workspace per token count M.  X may
    be a CUDA tensor or a pinned host tensor; `out` (optional) receives Y and
    may be either as well.
    """

    def __init__(self, W, g: int = 128):
        self.N, self.K = W.shape
        self.g = g
        self.packed, self.s1 = qoq_pack_weights(W, g)
        self._ws = {}

    def workspace(self, M: int):
        torch = _torch()
        if M not in self._ws:
            need = qoq_gemm_workspace_bytes(M, self.N, self.K, self.g)
            self._ws[M] = torch.zeros(need, dtype=torch.uint8, device=self.packed.device)
        return self._ws[M]

    def __call__(self, X, out=None, stream=None):
        Xq, sx = qoq_quant_act(X, stream=stream)
        return qoq_w4a8_gemm(Xq, sx, self.packed, self.s1, self.N, self.g, Y=out,
                             workspace=self.workspace(X.shape[0]), stream=stream)
