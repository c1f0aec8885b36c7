"""qoq_w4a8_gemm_no_alloc: the W4A8 GEMM for callers that cannot allocate
device memory.

Examples of such callers:
- a plugin that a host program hands only its input and output buffers,
  without access to the host's allocator;
- a serving process that reserved nearly all device memory for its caches at
  start-up;
- a step that must not synchronise the device, as cudaMalloc and cudaFree may.

The entry point keeps its scratch in a fixed 16 MiB device array inside the
library and must give the same results as qoq_w4a8_gemm with a caller
workspace.

This file is named so that pytest collects it last: a run that stops at its
first failure has then already run every other test.  Its GPU test also
passes on its own in a fresh process, where its first call does the per-device
set-up.
"""
import numpy as np
import pytest

from tests import gpu_cases as gc
from tests.conftest import gpu_available
from w4a8_quantized_serving_gb300 import synth

FAKE = 0x7F0000001000  # 16-byte aligned, never dereferenced: every CPU call below fails validation
MIS = FAKE + 8
MAX_SCRATCH = 16 << 20


def q():
    import w4a8_quantized_serving_gb300 as mod

    return mod


def test_no_alloc_limit_matches_the_header():
    """The documented limit: every shape with M <= 64 fits, whatever N and K,
    as qoq_gemm_workspace_bytes counts; large prefill shapes do not."""
    ws = q().qoq_gemm_workspace_bytes
    for K in (128, 4096, 131072):
        for M in (1, 16, 17, 32, 33, 64):
            for N in (128, 12288, 524288):
                assert 0 < ws(M, N, K) <= MAX_SCRATCH
    assert ws(4096, 28672, 8192) > MAX_SCRATCH  # 70B prefill does not fit


def test_no_alloc_rejects_before_touching_the_device():
    """Argument errors, and shapes that need more scratch than the array
    holds, return their code on the host (the pointers here are fake)."""
    L = q().lib()

    def call(M=16, N=256, K=512, g=128, Xq=FAKE, sx=FAKE, pk=FAKE, s1=FAKE, Y=FAKE, acc=None):
        return L.qoq_w4a8_gemm_no_alloc(M, N, K, g, Xq, sx, pk, s1, Y, acc, None)

    assert call(Xq=None) == 1
    assert call(Y=None) == 1
    assert call(g=96) == 3
    assert call(K=384, g=256) == 3  # g must divide K
    assert call(N=200) == 2
    assert call(M=0) == 2
    assert call(K=131072 + 128) == 2
    assert call(pk=MIS) == 4
    assert call(acc=MIS) == 4
    assert call(M=4096, N=28672, K=8192) == 5  # needs ~100 MB of scratch
    assert call(M=1024, N=4096, K=14336) == 5
    assert call(M=2048, N=4096, K=4096) == 5
    assert q().qoq_status_str(5) == "QOQ_ERR_WORKSPACE"


@pytest.mark.gpu
@pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")
@pytest.mark.parametrize("M,N,K", [(16, 12288, 4096), (40, 1664, 1152), (128, 1024, 1024)])
def test_no_alloc_matches_workspace_entry_point(M, N, K):
    """Two no-alloc calls in a row, on different activations, each equal to
    qoq_w4a8_gemm with a zero-filled caller workspace.  The int32 accumulators
    must be bit-exact; Y must be within the tolerance of the parity tests."""
    import torch

    mod = q()
    mod.qoq_set_debug(0, 0)
    assert 0 < mod.qoq_gemm_workspace_bytes(M, N, K) <= MAX_SCRATCH
    W = gc.to_dev_f16(synth.weights(N, K, 71))
    packed, s1 = mod.qoq_pack_weights(W)

    inputs, refs = [], []
    for call in range(2):
        Xq, sx = mod.qoq_quant_act(gc.to_dev_f16(synth.activations(M, K, 72 + call)))
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        ws = torch.zeros(mod.qoq_gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        Y = mod.qoq_w4a8_gemm(Xq, sx, packed, s1, N, acc_debug=acc, workspace=ws)
        inputs.append((Xq, sx))
        refs.append((Y, acc))
    torch.cuda.synchronize()

    outs = [(torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda"),
             torch.full((M, N), -1, dtype=torch.int32, device="cuda")) for _ in range(2)]
    for (Xq, sx), (Y, acc) in zip(inputs, outs):  # the two calls, back to back on one stream
        mod.qoq_w4a8_gemm_no_alloc(Xq, sx, packed, s1, N, Y=Y, acc_debug=acc)
    torch.cuda.synchronize()

    for call, ((Y, acc), (Yr, accr)) in enumerate(zip(outs, refs)):
        assert np.array_equal(acc.cpu().numpy(), accr.cpu().numpy()), f"call {call}: acc differs"
        ok, rel, ab = gc.y_close(gc.f16_bits(Y), gc.f16_bits(Yr))
        assert ok, f"call {call}: Y differs (max rel {rel}, max abs {ab})"


@pytest.mark.gpu
@pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")
def test_no_alloc_timeout_is_reported_after_later_calls():
    """A no-alloc call that runs out of a device-side wait limit (test hook:
    the producer skips one stage, 5 ms limit) is reported by
    qoq_no_alloc_last_status even after a later call has cleared the array:
    the status is sticky until read, the read resets it, and the later call
    is bit-exact against the workspace entry point."""
    import torch

    mod = q()
    M, N, K = 16, 128 * 152, 8192
    W = gc.to_dev_f16(synth.weights(N, K, 75))
    packed, s1 = mod.qoq_pack_weights(W)
    Xq, sx = mod.qoq_quant_act(gc.to_dev_f16(synth.activations(M, K, 76)))
    assert mod.qoq_no_alloc_last_status() == 0  # nothing pending from earlier tests
    try:
        mod.qoq_set_debug(5_000_000, 1)
        mod.qoq_w4a8_gemm_no_alloc(Xq, sx, packed, s1, N)
    finally:
        mod.qoq_set_debug(0, 0)
    acc = torch.full((M, N), -1, dtype=torch.int32, device="cuda")
    mod.qoq_w4a8_gemm_no_alloc(Xq, sx, packed, s1, N, acc_debug=acc)  # clears the array, keeps the status
    assert mod.qoq_no_alloc_last_status() == 7  # QOQ_ERR_DEVICE_TIMEOUT
    assert mod.qoq_no_alloc_last_status() == 0  # the read reset it
    ref = torch.empty((M, N), dtype=torch.int32, device="cuda")
    ws = torch.zeros(mod.qoq_gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    mod.qoq_w4a8_gemm(Xq, sx, packed, s1, N, acc_debug=ref, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(acc, ref)
    assert mod.qoq_last_device_status(ws) == 0
