"""Level-2 group sizes other than 128 (GPU): g = 32 and 64, where a packed
128-channel k-tile carries 4 or 2 scale sets, and g = 256 .. K, where a group
spans several k-tiles (g = K: one group per output channel).  Each case runs
the C ABI through the binding and checks it against the oracle at the same g:
codes, scales and the packed layout bit-exact, int32 accumulators bit-exact,
fp16 Y within the parity tolerance.

QServe talk write-up, "Progressive Group Quantization for W4A8 GEMM", and
lecture 15 notes, section 15.6: the group size trades scale bytes per weight
(4 + 16/g bits here) against the level-2 reconstruction error."""
import numpy as np
import pytest

from tests import gpu_cases as gc
from tests.conftest import gpu_available
from w4a8_quantized_serving_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


def q():
    import w4a8_quantized_serving_gb300 as mod

    return mod


@pytest.mark.parametrize("g", [32, 64, 256, 512, 1024])
def test_pack_bit_exact_and_layout_other_g(g):
    N, K = 256, 1024
    W = synth.weights(N, K, 300 + g)
    W[0, : K // 2] = 0.0  # groups that are all zero in one half of a row
    packed, s1 = q().qoq_pack_weights(gc.to_dev_f16(W), g=g)
    o = gc.oracle.weight_quant(synth.bits(W), g)
    gc.check_weights(q(), dict(packed=packed, s1=s1), o, N, K, group=g)
    want = gc.pack_reference_layout(o["q4"], o["s2"], o["z"], g)
    assert packed.numel() == q().qoq_packed_weight_bytes(N, K, g) == want.size
    assert np.array_equal(packed.cpu().numpy(), want)


@pytest.mark.parametrize("g", [32, 64, 256, "K"])
@pytest.mark.parametrize("M,N,K", [(16, 384, 1024), (40, 640, 1152), (200, 384, 1024), (200, 512, 1152), (1, 128, 768)])
def test_gemm_other_g(g, M, N, K):
    """Decode token tiles (M <= 64) and 128-token tiles (M > 64), with split-K
    tiles, at each group size; N = 512 runs the 128-token tiles on CTA pairs,
    N = 384 on single CTAs."""
    gg = K if g == "K" else g
    if K % gg:
        pytest.skip("g must divide K")
    W = synth.weights(N, K, 7 + M)
    X = synth.activations(M, K, 8 + M)
    gl = gc.gpu_layer(W, X, g=gg)
    o = gc.oracle_layer(W, X, g=gg)
    gc.check_weights(q(), gl, o, N, K, group=gg)
    gc.check_acts(gl, o)
    acc = gl["acc"].cpu().numpy()
    assert np.array_equal(acc.astype(np.int64), o["acc"]), f"acc mismatch at {np.argwhere(acc != o['acc'])[:5].tolist()}"
    ok, rel, ab = gc.y_close(gc.f16_bits(gl["Y"]), o["Y"])
    assert ok, (rel, ab)


@pytest.mark.parametrize("g", [32, 64])
def test_gemm_small_groups_worst_case(g):
    """Largest |acc| per fold chunk with distinct scales in every scale set of a
    k-tile: weights that put codes at the range ends with s2 = 16 in some groups
    and small ranges in others, and saturated activations."""
    N, K, M = 128, 2048, 16
    rng = np.random.default_rng(g)
    W = np.where(rng.random((N, K)) < 0.5, -1.0, 1.0) * 0.125
    # a range per group: full (codes 0 and 14 with s2 = 16, w8 = +-112) or
    # 1/16 of it (s2 = 1, w8 = +-7)
    W = (W.reshape(N, K // g, g) * rng.choice([0.0625, 1.0], size=(N, K // g, 1))).reshape(N, K)
    X = np.where(rng.random((M, K)) < 0.5, -1.0, 1.0) * 4.0
    gl = gc.gpu_layer(W.astype(np.float16), X.astype(np.float16), g=g)
    o = gc.oracle_layer(W.astype(np.float16), X.astype(np.float16), g=g)
    assert np.array_equal(gl["acc"].cpu().numpy().astype(np.int64), o["acc"])
