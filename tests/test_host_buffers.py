"""Host buffers at the ends of the path (GPU): X read in place from pinned host
memory by the quantizers, Y written in place into pinned host memory by the
GEMM.  The results must equal the oracle's, and the device-buffer path's bit
for bit, since only where the bytes live changes."""
import numpy as np
import pytest

from tests import gpu_cases as gc
from tests.conftest import gpu_available
from w4a8_quantized_serving_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


def q():
    import w4a8_quantized_serving_gb300 as mod

    return mod


def pinned_f16(a: np.ndarray):
    t = gc.torch()
    h = t.empty(a.shape, dtype=t.float16, pin_memory=True)
    h.copy_(t.from_numpy(np.ascontiguousarray(a, dtype=np.float16)))
    return h


@pytest.mark.parametrize("M,N,K", [(16, 1280, 1152), (5, 384, 4096), (64, 512, 640), (200, 640, 1024)])
def test_host_x_and_host_y_match_oracle(M, N, K):
    mod, t = q(), gc.torch()
    W = synth.weights(N, K, 31 + M)
    X = synth.activations(M, K, 32 + M)
    o = gc.oracle_layer(W, X)
    packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(W))
    Xh = pinned_f16(X)
    Xq, sx = mod.qoq_quant_act(Xh)  # X read from host memory
    assert Xq.is_cuda and sx.is_cuda
    Yh = t.empty((M, N), dtype=t.float16, pin_memory=True)
    ws = t.zeros(mod.qoq_gemm_workspace_bytes(M, N, K, 128), dtype=t.uint8, device="cuda")
    acc = t.empty((M, N), dtype=t.int32, device="cuda")
    mod.qoq_w4a8_gemm(Xq, sx, packed, s1, N, Y=Yh, acc_debug=acc, workspace=ws)  # Y written to host memory
    assert mod.qoq_last_device_status(ws) == 0
    t.cuda.synchronize()
    assert np.array_equal(Xq.cpu().numpy(), o["Xq"])
    assert np.array_equal(gc.f16_bits(sx), o["sx"])
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), o["acc"])
    ok, rel, ab = gc.y_close(Yh.numpy().view(np.uint16), o["Y"])
    assert ok, (rel, ab)
    # and bit for bit what the device-buffer path writes
    Yd = mod.qoq_w4a8_gemm(Xq, sx, packed, s1, N, workspace=ws)
    t.cuda.synchronize()
    assert np.array_equal(Yh.numpy().view(np.uint16), gc.f16_bits(Yd))


def test_host_x_norm_quant_matches_device_x():
    mod, t = q(), gc.torch()
    M, K = 16, 4096
    X = synth.activations(M, K, 41)
    gamma = gc.to_dev_f16(1.0 + 0.25 * np.random.default_rng(42).standard_normal(K))
    beta = gc.to_dev_f16(0.1 * np.random.default_rng(43).standard_normal(K))
    for kind, b in (("rms", None), ("layer", beta)):
        Xq_h, sx_h = mod.qoq_norm_quant_act(pinned_f16(X), gamma, b, kind=kind)
        Xq_d, sx_d = mod.qoq_norm_quant_act(gc.to_dev_f16(X), gamma, b, kind=kind)
        t.cuda.synchronize()
        assert np.array_equal(Xq_h.cpu().numpy(), Xq_d.cpu().numpy()), kind
        assert np.array_equal(gc.f16_bits(sx_h), gc.f16_bits(sx_d)), kind


def test_linear_layer_with_host_buffers():
    """QoQLinear with X and Y in pinned host memory gives the device path's Y."""
    mod, t = q(), gc.torch()
    M, N, K = 16, 1280, 1024
    W = gc.to_dev_f16(synth.weights(N, K, 51))
    X = synth.activations(M, K, 52)
    layer = mod.QoQLinear(W)
    Yd = layer(gc.to_dev_f16(X))
    Yh = t.empty((M, N), dtype=t.float16, pin_memory=True)
    assert layer(pinned_f16(X), out=Yh) is Yh
    t.cuda.synchronize()
    assert np.array_equal(Yh.numpy().view(np.uint16), gc.f16_bits(Yd))
