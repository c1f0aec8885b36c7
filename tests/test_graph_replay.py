"""qoq_w4a8_gemm inside a captured CUDA graph, replayed with new inputs (GPU).

A serving loop captures its decode step once and replays it every step with
new activations in the same buffers.  Each replay runs the captured launches
with identical parameters, so nothing that tells one call's split-K partial
sums from another's may come from the launch parameters: the decode kernel
tags them with an epoch it keeps in the workspace header.  These tests replay
graphs many times, change the inputs between replays, and compare every
replay's int32 accumulators with the oracle's, bit for bit.
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


def _input_sets(o, M: int, K: int, n_sets: int, seed0: int):
    """n_sets activation sets as (Xq, s_x) device tensors plus the oracle's
    int32 accumulators for each, on the device for a fast comparison."""
    t = gc.torch()
    sets = []
    for i in range(n_sets):
        Xq, sx = gc.oracle.act_quant(synth.bits(synth.activations(M, K, seed0 + i)))
        acc, Y = gc.oracle.gemm(Xq, sx, o["q4"], o["s2"], o["z"], o["s1"], threads=0)
        sets.append(dict(Xq=t.from_numpy(Xq).cuda(), sx=t.from_numpy(sx.view(np.float16)).cuda(),
                         acc=t.from_numpy(acc.astype(np.int32)).cuda(), Y=Y))
    return sets


def test_graph_replays_with_new_inputs_are_exact():
    """Four GEMM calls at the 7B fused-QKV decode shape (M=16, N=12288,
    K=4096: every tile split along K) captured in one graph, two calls per
    workspace; 60 replays, each with new activations in the captured buffers
    (five input sets in rotation, so that consecutive replays of a call always
    differ); every replay's accumulators bit-exact against the oracle."""
    mod = q()
    t = gc.torch()
    M, N, K = 16, 12288, 4096
    W = synth.weights(N, K, 91)
    packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(W))
    o = gc.oracle.weight_quant(synth.bits(W), 128)
    n_sets, n_calls, n_replays = 5, 4, 60
    sets = _input_sets(o, M, K, n_sets, 900)

    xq = [t.empty((M, K), dtype=t.int8, device="cuda") for _ in range(n_calls)]
    sx = [t.empty(M, dtype=t.float16, device="cuda") for _ in range(n_calls)]
    acc = [t.empty((M, N), dtype=t.int32, device="cuda") for _ in range(n_calls)]
    Y = [t.empty((M, N), dtype=t.float16, device="cuda") for _ in range(n_calls)]
    ws_bytes = mod.qoq_gemm_workspace_bytes(M, N, K)
    ws = [t.zeros(ws_bytes, dtype=t.uint8, device="cuda") for _ in range(2)]

    def load(r: int):
        for j in range(n_calls):
            s = sets[(r + j) % n_sets]
            xq[j].copy_(s["Xq"])
            sx[j].copy_(s["sx"])
            acc[j].fill_(-1)

    def calls():
        for j in range(n_calls):
            mod.qoq_w4a8_gemm(xq[j], sx[j], packed, s1, N, Y=Y[j], acc_debug=acc[j], workspace=ws[j // 2])

    load(0)
    calls()  # direct calls first: per-device set-up happens outside the capture
    t.cuda.synchronize()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph):
        calls()
    t.cuda.synchronize()

    bad = []
    for r in range(n_replays):
        load(r)
        graph.replay()
        for j in range(n_calls):
            if not t.equal(acc[j], sets[(r + j) % n_sets]["acc"]):
                bad.append((r, j))
    t.cuda.synchronize()
    for w in ws:
        assert mod.qoq_last_device_status(w) == 0
    assert not bad, f"(replay, call) pairs with wrong accumulators: {bad[:10]} ({len(bad)} in all)"
    # the last replay's fp16 outputs, against the oracle's
    for j in range(n_calls):
        ok, rel, ab = gc.y_close(gc.f16_bits(Y[j]), sets[(n_replays - 1 + j) % n_sets]["Y"])
        assert ok, (j, rel, ab)


def test_graph_replays_pair_kernel_with_new_inputs_are_exact():
    """128-token tiles on CTA pairs (M=200, N=4096, K=4096: two token tiles,
    sixteen pair tiles, every one split along K over the pairs): three calls
    in one graph over two workspaces, 20 replays with new activations in the
    captured buffers; every replay's accumulators bit-exact against the
    oracle."""
    mod = q()
    t = gc.torch()
    M, N, K = 200, 4096, 4096
    W = synth.weights(N, K, 95)
    packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(W))
    o = gc.oracle.weight_quant(synth.bits(W), 128)
    n_sets, n_calls, n_replays = 4, 3, 20
    sets = _input_sets(o, M, K, n_sets, 970)
    xq = [t.empty((M, K), dtype=t.int8, device="cuda") for _ in range(n_calls)]
    sx = [t.empty(M, dtype=t.float16, device="cuda") for _ in range(n_calls)]
    acc = [t.empty((M, N), dtype=t.int32, device="cuda") for _ in range(n_calls)]
    ws_bytes = mod.qoq_gemm_workspace_bytes(M, N, K)
    ws = [t.zeros(ws_bytes, dtype=t.uint8, device="cuda") for _ in range(2)]

    def load(r: int):
        for j in range(n_calls):
            s = sets[(r + j) % n_sets]
            xq[j].copy_(s["Xq"])
            sx[j].copy_(s["sx"])
            acc[j].fill_(-1)

    def calls():
        for j in range(n_calls):
            mod.qoq_w4a8_gemm(xq[j], sx[j], packed, s1, N, acc_debug=acc[j], workspace=ws[j % 2])

    load(0)
    calls()
    t.cuda.synchronize()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph):
        calls()
    t.cuda.synchronize()
    bad = []
    for r in range(n_replays):
        load(r)
        graph.replay()
        for j in range(n_calls):
            if not t.equal(acc[j], sets[(r + j) % n_sets]["acc"]):
                bad.append((r, j))
    t.cuda.synchronize()
    for w in ws:
        assert mod.qoq_last_device_status(w) == 0
    assert not bad, f"(replay, call) pairs with wrong accumulators: {bad[:10]} ({len(bad)} in all)"


def test_workspace_shared_across_token_counts():
    """One workspace, sized for the largest call, serves a sequence of calls
    whose token counts switch between the decode kernel (M <= 64) and the
    128-token-tile kernel, directly and replayed from a graph: each call's
    accumulators bit-exact against the oracle."""
    mod = q()
    t = gc.torch()
    N, K = 2048, 2048
    W = synth.weights(N, K, 93)
    packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(W))
    o = gc.oracle.weight_quant(synth.bits(W), 128)
    Ms = [16, 200, 16, 64, 130, 33, 16]
    ws = t.zeros(max(mod.qoq_gemm_workspace_bytes(M, N, K) for M in Ms), dtype=t.uint8, device="cuda")
    cases = []
    for i, M in enumerate(Ms):
        s = _input_sets(o, M, K, 1, 950 + i)[0]
        s["out"] = t.empty((M, N), dtype=t.int32, device="cuda")
        cases.append(s)

    def calls():
        for s in cases:
            mod.qoq_w4a8_gemm(s["Xq"], s["sx"], packed, s1, N, acc_debug=s["out"], workspace=ws)

    calls()
    t.cuda.synchronize()
    for M, s in zip(Ms, cases):
        assert t.equal(s["out"], s["acc"]), f"direct call, M={M}"
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph):
        calls()
    for r in range(10):
        for s in cases:
            s["out"].fill_(-1)
        graph.replay()
        t.cuda.synchronize()
        for M, s in zip(Ms, cases):
            assert t.equal(s["out"], s["acc"]), f"replay {r}, M={M}"
    assert mod.qoq_last_device_status(ws) == 0
