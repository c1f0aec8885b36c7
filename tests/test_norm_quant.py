"""The norm fused with the per-token quantizer (GPU): qoq_norm_quant_act
against the oracle, bit-exact in Xq and s_x, for RMSNorm and LayerNorm.

QServe talk write-up, "Precision Data Flow and Activation Quantization
Fusion": a linear layer's activation quantization is fused into the preceding
layer, such as LayerNorm, whose output is quantized to 8 bits directly.  The
row statistics are exact integers on both sides, so the codes do not depend on
the GPU's reduction order."""
import numpy as np
import pytest

from tests import gpu_cases as gc
from tests.conftest import gpu_available
from w4a8_quantized_serving_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


def q():
    import w4a8_quantized_serving_gb300 as mod

    return mod


def _edge_rows(X):
    """Rows that stress the statistics and the rounding: zeros, a constant, the
    fp16 extremes with subnormals, a single spike, and exact-halves."""
    M, K = X.shape
    if M > 0:
        X[0] = 0.0
    if M > 1:
        X[1] = np.float16(0.75)
    if M > 2:
        X[2] = np.float16(2.0 ** -24) * np.arange(K) % 1024
        X[2, :4] = [65504.0, -65504.0, 2.0 ** -24, -(2.0 ** -14)]
    if M > 3:
        X[3] = 0.0
        X[3, K // 2] = np.float16(-7.0)
    if M > 4:
        X[4] = (np.arange(K) % 255 - 127 + 0.5).astype(np.float16)
    return X


@pytest.mark.parametrize("kind", ["rms", "layer"])
@pytest.mark.parametrize("M,K", [(1, 128), (7, 512), (16, 4096), (33, 1152), (5, 16384), (3, 65536), (2, 131072),
                                 (1100, 1152), (1024, 4096)])
def test_norm_quant_bit_exact(kind, M, K):
    """Shapes from one row to the M >= 1024 prefill range, K up to 131072."""
    rng = np.random.default_rng(M * 1000 + K)
    X = (synth.activations(M, K, 40 + M) * 0.5).astype(np.float16)
    X = _edge_rows(X)
    gamma = rng.uniform(0.25, 2.0, K).astype(np.float16)
    beta = rng.uniform(-1.0, 1.0, K).astype(np.float16) if kind == "layer" else None
    eps = 1e-5
    Xq, sx = q().qoq_norm_quant_act(gc.to_dev_f16(X), gc.to_dev_f16(gamma),
                                    None if beta is None else gc.to_dev_f16(beta), kind=kind, eps=eps)
    o = gc.oracle.norm_quant_act(synth.bits(X), synth.bits(gamma), None if beta is None else synth.bits(beta),
                                 kind=kind, eps=eps)
    xq = Xq.cpu().numpy()
    bad = np.argwhere(xq != o["Xq"])
    assert len(bad) == 0, f"Xq differs at {bad[:5].tolist()}"
    assert np.array_equal(gc.f16_bits(sx), o["sx"])


@pytest.mark.parametrize("kind", ["rms", "layer"])
def test_norm_quant_feeds_the_gemm(kind):
    """norm -> int8 -> W4A8 GEMM on the decode shape: the fused codes give the
    oracle's int32 accumulators."""
    M, N, K = 16, 1280, 4096
    rng = np.random.default_rng(5)
    X = synth.activations(M, K, 61)
    gamma = rng.uniform(0.5, 1.5, K).astype(np.float16)
    beta = rng.uniform(-0.5, 0.5, K).astype(np.float16) if kind == "layer" else None
    W = synth.weights(N, K, 62)
    packed, s1 = q().qoq_pack_weights(gc.to_dev_f16(W))
    Xq, sx = q().qoq_norm_quant_act(gc.to_dev_f16(X), gc.to_dev_f16(gamma),
                                    None if beta is None else gc.to_dev_f16(beta), kind=kind, eps=1e-6)
    import torch

    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    Y = q().qoq_w4a8_gemm(Xq, sx, packed, s1, N, acc_debug=acc)
    o = gc.oracle.norm_quant_act(synth.bits(X), synth.bits(gamma), None if beta is None else synth.bits(beta),
                                 kind=kind, eps=1e-6)
    w = gc.oracle.weight_quant(synth.bits(W), 128)
    oacc, oY = gc.oracle.gemm(o["Xq"], o["sx"], w["q4"], w["s2"], w["z"], w["s1"], 128)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), oacc)
    ok, rel, ab = gc.y_close(gc.f16_bits(Y), oY)
    assert ok, (rel, ab)
