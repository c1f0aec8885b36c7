"""The C-ABI library: loads, exports what include/qoq.h declares, validates
arguments on the host before any device access (CPU only, no compute)."""
import ctypes
import os
import re

import pytest

import w4a8_quantized_serving_gb300 as q
from w4a8_quantized_serving_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qoq.h")
FAKE = 0x7F0000001000  # 16-byte aligned, never dereferenced: every call below fails validation first
MIS = FAKE + 8


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qoq_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("qoq_pack_weights", "qoq_quant_act", "qoq_w4a8_gemm", "qoq_packed_weight_bytes",
                 "qoq_gemm_workspace_bytes", "qoq_last_device_status", "qoq_unpack_weights_debug"):
        assert must in names


def test_library_exports_every_declared_symbol():
    L = q.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(binding.EXPORTED) <= set(declared_functions())


def test_library_is_built_for_sm103a_only():
    """Every translation unit is compiled for one target, sm_103a, and the
    library is linked for it alone (the build's own flags, not a binary tool)."""
    from w4a8_quantized_serving_gb300.csrc import build as cbuild

    assert cbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert cbuild.NVCC_FLAGS[:2] == cbuild.ARCH
    assert not any("sm_" in f or "compute_" in f for f in cbuild.NVCC_FLAGS[2:])


def test_status_strings_and_version():
    assert q.qoq_version() >= 100
    for code, name in binding.QOQ_ERRORS.items():
        assert q.qoq_status_str(code) == name
    assert q.qoq_status_str(99) == "QOQ_ERR_UNKNOWN"


def test_packed_weight_bytes_closed_form():
    # 4 bits per code plus one uint8 scale and one uint8 zero per 128-channel group:
    # 4 + 16/128 bits per weight (lecture 15: 4 + 16/128 = 4.125 effective bits)
    for N, K in [(128, 128), (256, 512), (12288, 4096), (28672, 8192)]:
        nb = q.qoq_packed_weight_bytes(N, K, 128)
        assert nb == N * K // 2 + 2 * N * (K // 128)
        assert nb * 8 / (N * K) == pytest.approx(4.125)
    assert q.qoq_packed_weight_bytes(100, 128, 128) == 0
    assert q.qoq_packed_weight_bytes(128, 128, 96) == 0  # not 32, 64 or a multiple of 128
    assert q.qoq_packed_weight_bytes(128, 384, 256) == 0  # g must divide K


def test_packed_weight_bytes_other_group_sizes():
    # one uint8 scale and one uint8 zero per group for g < 128; for g >= 128
    # every 128-channel k-tile repeats its group's scale pair
    N, K = 256, 1024
    for g, bits in [(32, 4 + 16 / 32), (64, 4 + 16 / 64), (128, 4.125), (256, 4.125), (1024, 4.125)]:
        nb = q.qoq_packed_weight_bytes(N, K, g)
        assert nb * 8 / (N * K) == pytest.approx(bits), g


def test_workspace_bytes_host_pure_and_monotone():
    for (M, N, K) in [(8, 256, 512), (16, 12288, 4096), (128, 22016, 4096), (256, 4096, 14336),
                      (4096, 28672, 8192)]:
        ws = q.qoq_gemm_workspace_bytes(M, N, K, 128)
        assert ws > 0 and ws % 256 == 0
        # holds at least the fp16 copy of the activations
        assert ws >= 2 * M * K
    assert q.qoq_gemm_workspace_bytes(0, 128, 128, 128) == 0
    assert q.qoq_gemm_workspace_bytes(1, 128, 131072 + 128, 128) == 0


L = None


def _lib():
    return q.lib()


def test_quant_act_validation():
    L = _lib()
    assert L.qoq_quant_act(16, 4096, None, FAKE, FAKE, None) == 1
    assert L.qoq_quant_act(0, 4096, FAKE, FAKE, FAKE, None) == 2
    assert L.qoq_quant_act(16, 100, FAKE, FAKE, FAKE, None) == 2
    assert L.qoq_quant_act(16, 4096, MIS, FAKE, FAKE, None) == 4


def test_norm_quant_act_validation():
    L = _lib()
    f = ctypes.c_float
    assert L.qoq_norm_quant_act(16, 4096, 0, f(1e-6), None, FAKE, None, FAKE, FAKE, None) == 1
    assert L.qoq_norm_quant_act(16, 4096, 1, f(1e-6), FAKE, FAKE, None, FAKE, FAKE, None) == 1  # LayerNorm needs beta
    assert L.qoq_norm_quant_act(16, 4096, 2, f(1e-6), FAKE, FAKE, FAKE, FAKE, FAKE, None) == 3
    assert L.qoq_norm_quant_act(16, 4096, 0, f(0.0), FAKE, FAKE, None, FAKE, FAKE, None) == 3
    assert L.qoq_norm_quant_act(16, 4096, 0, f(float("nan")), FAKE, FAKE, None, FAKE, FAKE, None) == 3
    assert L.qoq_norm_quant_act(16, 4096, 0, f(float("inf")), FAKE, FAKE, None, FAKE, FAKE, None) == 3
    assert L.qoq_norm_quant_act(16, 100, 0, f(1e-6), FAKE, FAKE, None, FAKE, FAKE, None) == 2
    assert L.qoq_norm_quant_act(16, 4096, 0, f(1e-6), FAKE, MIS, None, FAKE, FAKE, None) == 4
    assert L.qoq_norm_quant_act(16, 4096, 1, f(1e-6), FAKE, FAKE, MIS, FAKE, FAKE, None) == 4


def test_pack_validation():
    L = _lib()
    assert L.qoq_pack_weights(128, 256, 128, FAKE, None, FAKE, None) == 1
    assert L.qoq_pack_weights(128, 256, 96, FAKE, FAKE, FAKE, None) == 3
    assert L.qoq_pack_weights(100, 256, 128, FAKE, FAKE, FAKE, None) == 2
    assert L.qoq_pack_weights(128, 256, 128, FAKE, MIS, FAKE, None) == 4


@pytest.mark.parametrize("entry", ["qoq_w4a8_gemm", "qoq_w4a8_gemm_zero_folded"])
def test_gemm_validation(entry):
    L = _lib()
    ws = q.qoq_gemm_workspace_bytes(16, 256, 512)

    def call(M=16, N=256, K=512, g=128, Xq=FAKE, sx=FAKE, pk=FAKE, s1=FAKE, Y=FAKE, acc=None, w=FAKE,
             wb=ws):
        return getattr(L, entry)(M, N, K, g, Xq, sx, pk, s1, Y, acc, w, wb, None)

    if entry.endswith("zero_folded"):
        # the folded variant reads one scale set per 128-channel k-tile: g >= 128 only
        assert call(g=64) == 3 and call(g=32) == 3
    assert call(Xq=None) == 1
    assert call(Y=None) == 1
    assert call(g=48) == 3
    assert call(N=200) == 2
    assert call(K=131072 + 128) == 2
    assert call(M=0) == 2
    assert call(pk=MIS) == 4
    assert call(acc=MIS) == 4
    assert call(wb=ws - 1) == 5
    assert call(w=None) == 5
    assert call(w=MIS) == 4


def test_unpack_and_status_validation():
    L = _lib()
    assert L.qoq_unpack_weights_debug(128, 256, 128, None, FAKE, FAKE, FAKE, None) == 1
    assert L.qoq_unpack_weights_debug(128, 256, 96, FAKE, FAKE, FAKE, FAKE, None) == 3
    assert L.qoq_last_device_status(None, None) == 1
    assert L.qoq_set_debug(0, 5) == 3
    assert L.qoq_set_debug(0, 0) == 0


def test_binding_refuses_pageable_host_tensors():
    """Pinned host memory is accepted for X and Y (the kernels access it in
    place); pageable host memory is refused before any device work."""
    import torch

    X = torch.zeros((4, 128), dtype=torch.float16)  # pageable
    with pytest.raises(TypeError, match="pinned host"):
        q.qoq_quant_act(X)
    with pytest.raises(TypeError, match="pinned host"):
        q.qoq_norm_quant_act(X, X[0])
    with pytest.raises(TypeError, match="CUDA tensor$"):
        binding._dev(X, torch.float16, "Xq")  # device-only arguments take no host tensor


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_LIB", None)
    monkeypatch.setattr(binding._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(binding.QoQError):
        binding.lib()


def test_w4ax_sizes_and_validation():
    """W4Ax activation bytes follow the documented row layout; argument errors
    return before any device access (fake pointers)."""
    L = _lib()
    for M, K, n8 in [(1, 128, 0), (1, 128, 1), (16, 4096, 1), (4096, 8192, 5)]:
        G = K // 128
        assert q.qoq_w4ax_act_bytes(M, K, n8) == M * (128 * n8 + 64 * (G - n8))
    assert q.qoq_w4ax_act_bytes(16, 4096, 33) == 0 and q.qoq_w4ax_act_bytes(16, 4096, -1) == 0
    assert q.qoq_w4ax_workspace_bytes(16, 12288, 4096) > 0 and q.qoq_w4ax_workspace_bytes(16, 100, 4096) == 0
    assert L.qoq_quant_act_w4ax(16, 512, 5, FAKE, FAKE, FAKE, None) == 3
    assert L.qoq_quant_act_w4ax(16, 512, 1, None, FAKE, FAKE, None) == 1
    assert L.qoq_quant_act_w4ax(16, 500, 1, FAKE, FAKE, FAKE, None) == 2
    assert L.qoq_quant_act_w4ax(16, 512, 1, FAKE, MIS, FAKE, None) == 4
    ws = q.qoq_w4ax_workspace_bytes(16, 256, 512)

    def call(M=16, N=256, K=512, g=128, n8=1, Xa=FAKE, sx=FAKE, pk=FAKE, s1=FAKE, Y=FAKE, acc=None, w=FAKE, wb=ws):
        return L.qoq_w4ax_gemm(M, N, K, g, n8, Xa, sx, pk, s1, Y, acc, w, wb, None)

    assert call(Xa=None) == 1 and call(Y=None) == 1
    assert call(n8=5) == 3 and call(n8=-1) == 3 and call(g=96) == 3
    assert call(N=200) == 2 and call(M=0) == 2
    assert call(pk=MIS) == 4 and call(acc=MIS) == 4
    assert call(wb=ws - 1) == 5 and call(w=None) == 5

