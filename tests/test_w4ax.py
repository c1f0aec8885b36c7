"""The W4Ax path (COMET-style 4-bit activation blocks with 8-bit outlier
blocks) against the oracle (GPU).

qoq_quant_act_w4ax: codes and block scales bit-exact, and the activation
bytes equal a host re-pack of the oracle's codes in the documented layout.
qoq_w4ax_gemm: sum_b acc_b bit-exact (acc_debug) and Y within the parity
tolerance, at small shapes and at the large-batch workloads with the outlier
channels permuted into the leading 8-bit block.
"""
import numpy as np
import pytest

from tests import gpu_cases as gc
from tests.conftest import gpu_available
from w4a8_quantized_serving_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


def q():
    import w4a8_quantized_serving_gb300 as mod

    return mod


def pack_w4ax_reference(codes: np.ndarray, n8: int) -> np.ndarray:
    """Activation rows in the layout of include/qoq.h, rebuilt on the host from
    codes [M][K] (test-side, independent of the kernels)."""
    M, K = codes.shape
    rows = []
    for b in range(K // 128):
        blk = codes[:, 128 * b:128 * b + 128].astype(np.int16)
        if b < n8:
            rows.append(blk.astype(np.int8).view(np.uint8))
        else:
            nib = (blk & 0xF).astype(np.uint8)
            rows.append(nib[:, 0::2] | (nib[:, 1::2] << 4))
    return np.concatenate(rows, axis=1)


def outlier_first_permutation(seed: int, K: int) -> np.ndarray:
    """Channel order with the activation generator's outlier channels first,
    so that they fall into the leading block (the rest in their order)."""
    out = synth.outlier_channels(seed, synth.TAG_X, K, 4)
    rest = np.setdiff1d(np.arange(K), out)
    return np.concatenate([out, rest])


def _check_quant(X, n8):
    mod = q()
    M, K = X.shape
    Xa, sxb = mod.qoq_quant_act_w4ax(gc.to_dev_f16(X), n8)
    codes, osx = gc.oracle.act_quant_w4ax(synth.bits(X), n8)
    assert np.array_equal(gc.f16_bits(sxb), osx), "block scales"
    assert np.array_equal(Xa.cpu().numpy(), pack_w4ax_reference(codes, n8)), "activation bytes"
    return Xa, sxb, codes, osx


@pytest.mark.parametrize("M,K,n8", [(1, 128, 0), (3, 384, 1), (16, 4096, 1), (129, 1024, 3), (7, 512, 4)])
def test_quant_act_w4ax_bit_exact(M, K, n8):
    X = synth.activations(M, K, 600 + M)
    if M >= 3:
        X[0] = 0  # zero blocks: scale 0, codes 0
        X[1, :256] = ((np.arange(256) % 15) - 7 + 0.5) * 2.0 ** -4  # exact ties in 4-bit blocks
        X[2, 5] = np.float16(60000.0)  # a block dominated by one value
    _check_quant(X, n8)


def _run_gemm(M, N, K, n8, g=128, seed=0, perm=None, sample_cols=None):
    mod = q()
    t = gc.torch()
    W = synth.weights(N, K, seed)
    X = synth.activations(M, K, seed)
    if perm is not None:  # the channel permutation applied to both operands upstream
        W = np.ascontiguousarray(W[:, perm])
        X = np.ascontiguousarray(X[:, perm])
    Xa, sxb, codes, osx = _check_quant(X, n8)
    packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(W), g=g)
    acc = t.empty((M, N), dtype=t.int32, device="cuda")
    ws = t.zeros(mod.qoq_w4ax_workspace_bytes(M, N, K, g), dtype=t.uint8, device="cuda")
    Y = mod.qoq_w4ax_gemm(Xa, sxb, n8, packed, s1, K, N, g=g, acc_debug=acc, workspace=ws)
    assert mod.qoq_last_device_status(ws) == 0
    o = gc.oracle.weight_quant(synth.bits(W), g)
    # sum_b acc_b is the plain integer product of the codes (pinned in the oracle)
    acc_ref, _ = gc.oracle.gemm(codes, np.zeros(M, np.uint16), o["q4"], o["s2"], o["z"], o["s1"], g, threads=0)
    got = acc.cpu().numpy().astype(np.int64)
    bad = got != acc_ref
    assert not bad.any(), f"{int(bad.sum())} accumulators differ, first at {np.argwhere(bad)[:5].tolist()}"
    Yg = gc.f16_bits(Y)
    if sample_cols is None:
        _, y_ref = gc.oracle.gemm_w4ax(codes, osx, o["q4"], o["s2"], o["z"], o["s1"], g)
        ok, rel, ab = gc.y_close(Yg, y_ref)
    else:  # the oracle's W4Ax product on a sample of output channels
        cols = np.sort(np.random.default_rng(seed).choice(N, sample_cols, replace=False))
        G = K // g
        _, y_ref = gc.oracle.gemm_w4ax(codes, osx, o["q4"][cols], o["s2"][cols], o["z"][cols], o["s1"][cols], g)
        ok, rel, ab = gc.y_close(np.ascontiguousarray(Yg[:, cols]), y_ref)
    assert ok, (rel, ab)


@pytest.mark.parametrize("M,N,K,n8,g", [
    (1, 128, 256, 1, 128), (16, 384, 1152, 1, 128), (100, 256, 1024, 2, 64), (128, 1024, 2048, 0, 128),
    (200, 384, 1152, 9, 128), (33, 2048, 4096, 3, 256),
])
def test_w4ax_gemm_matches_oracle(M, N, K, n8, g):
    _run_gemm(M, N, K, n8, g=g, seed=610 + M)


def test_w4ax_gemm_golden_example():
    """The hand-worked two-block example of the oracle's pins, through the GPU."""
    from tests.oracle_pins import load_golden, _w4ax_golden_inputs

    mod = q()
    t = gc.torch()
    gold = load_golden("w4ax_two_blocks.txt")
    X, W, _ = _w4ax_golden_inputs(gold, None)
    Xa, sxb, codes, osx = _check_quant(X, gold["n8"])
    packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(W))
    acc = t.empty((1, 128), dtype=t.int32, device="cuda")
    Y = mod.qoq_w4ax_gemm(Xa, sxb, gold["n8"], packed, s1, 256, acc_debug=acc)
    assert (acc.cpu().numpy() == gold["acc_sum"]).all()
    assert (gc.f16_bits(Y) == gold["Y_bits"]).all()


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_w4ax_workloads(cfg):
    """The large-batch workloads, outlier channels permuted into block 0
    (n8 = 1): every accumulator compared, Y on 128 sampled output channels."""
    c = synth.WORKLOADS[cfg]
    perm = outlier_first_permutation(c["seed"], c["K"])
    _run_gemm(c["M"], c["N"], c["K"], 1, seed=c["seed"], perm=perm, sample_cols=128)
