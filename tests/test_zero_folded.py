"""qoq_w4a8_gemm_zero_folded against the oracle (GPU).

The variant feeds q4 * s2 to the tensor cores and subtracts the zero points'
share, sum_j z s2 RS[m, j], in the epilogue (QFactory notes, section 4.3,
Table 2: the matmul with the all-ones J matrix).  Its int32 accumulators must
equal the oracle's bit for bit (the oracle's folded and direct forms are
pinned equal), and Y must be within the parity tolerance.
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


def _run(M, N, K, seed, g=128, W=None, X=None, oracle_form="folded"):
    mod = q()
    t = gc.torch()
    if W is None:
        W = synth.weights(N, K, seed)
    if X is None:
        X = synth.activations(M, K, seed)
    packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(W), g=g)
    Xq, sx = mod.qoq_quant_act(gc.to_dev_f16(X))
    acc = t.empty((M, N), dtype=t.int32, device="cuda")
    ws = t.zeros(mod.qoq_gemm_workspace_bytes(M, N, K, g), dtype=t.uint8, device="cuda")
    Y = mod.qoq_w4a8_gemm_zero_folded(Xq, sx, packed, s1, N, g=g, acc_debug=acc, workspace=ws)
    assert mod.qoq_last_device_status(ws) == 0
    o = gc.oracle.weight_quant(synth.bits(W), g)
    oXq, osx = gc.oracle.act_quant(synth.bits(X))
    assert np.array_equal(Xq.cpu().numpy(), oXq)
    if oracle_form == "folded":
        acc_ref, y_ref, _ = gc.oracle.gemm_zero_folded(oXq, osx, o["q4"], o["s2"], o["z"], o["s1"], g)
    else:  # the direct form on all host threads (pinned equal to the folded one)
        acc_ref, y_ref = gc.oracle.gemm(oXq, osx, o["q4"], o["s2"], o["z"], o["s1"], g, threads=0)
    got = acc.cpu().numpy().astype(np.int64)
    bad = got != acc_ref
    assert not bad.any(), f"{int(bad.sum())} accumulators differ, first at {np.argwhere(bad)[:5].tolist()}"
    ok, rel, ab = gc.y_close(gc.f16_bits(Y), y_ref)
    assert ok, (rel, ab)


@pytest.mark.parametrize("M", [1, 5, 16, 17, 33, 64, 65, 128, 200])
def test_zero_folded_token_counts(M):
    # 9 k-tiles: crosses the 8-group fold boundary; split-K on every tile
    _run(M, 384, 1152, 500 + M)


@pytest.mark.parametrize("M,N,K,g", [(16, 2048, 4096, 256), (130, 1024, 2048, 2048), (8, 128, 16384, 128)])
def test_zero_folded_shapes_and_group_sizes(M, N, K, g):
    _run(M, N, K, 510 + M, g=g)


def test_zero_folded_extreme_zero_points():
    """Rows whose groups have zero points at both ends of [0, 15] (all-negative
    and all-positive groups) and saturating activations."""
    M, N, K = 16, 256, 1024
    W = synth.weights(N, K, 520)
    W[0::4] = -np.abs(W[0::4])  # all-negative groups: z = 15
    W[1::4] = np.abs(W[1::4])   # all-positive groups: z = 0
    X = synth.activations(M, K, 520)
    X[0] = np.float16(3.0)
    X[1, ::2] = np.float16(-3.0)
    _run(M, N, K, 0, W=W, X=X)


@pytest.mark.parametrize("cfg", [1, 4])
def test_zero_folded_workload_full(cfg):
    """The two workloads of the A/B (decode M=16 and prefill M=4096), every
    output compared."""
    c = synth.WORKLOADS[cfg]
    _run(c["M"], c["N"], c["K"], c["seed"], oracle_form="direct")


@pytest.mark.parametrize("M", [16, 256])
def test_zero_folded_largest_operands(M):
    """The folded operand q4 * s2 reaches 224 here (s2 = 16, z = 7, q4 = 14 on
    127 of every group's 128 channels) against activations of 127: eight
    groups of such products would pass 2^24 in an fp32 accumulator, so the
    variant must fold more often than the direct form.  Whole tiles only, so
    the fold chunks start at group 0 (decode M=16, 128-token tiles M=256)."""
    import torch

    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 160)
    N = 128 * (sms if M <= 64 else sms // 2)
    K = 2048
    s1 = 2.0 ** -10
    W = np.full((N, K), 119 * s1)
    W[:, ::128] = -119 * s1  # one channel per group at the low end: s2 = 16, z = 7
    X = np.full((M, K), 1.0)
    o = gc.oracle.weight_quant(synth.bits(np.float16(W)), 128)
    assert (o["s2"] == 16).all() and (o["z"] == 7).all() and int(o["q4"].max()) == 14
    _run(M, N, K, 0, W=np.float16(W), X=np.float16(X), oracle_form="direct")
