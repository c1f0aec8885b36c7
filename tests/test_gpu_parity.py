"""CUDA path vs the oracle, element by element, on seeded inputs (GPU).

Integer outputs (Xq, s_x, q4, s2, z, s1, the int32 accumulators) must be
bit-exact; fp16 Y within |dY| <= 2e-3 |Y_ref| or |dY| <= 1e-2.
"""
import numpy as np
import pytest

from tests import gpu_cases as gc
from tests.conftest import gpu_available
from tests.oracle_pins import f16, load_golden
from w4a8_quantized_serving_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


def q():
    import w4a8_quantized_serving_gb300 as mod

    return mod


def _edge_rows(K: int, seed: int) -> np.ndarray:
    """Rows that stress the quantizers: zeros, constants, saturation, a row
    whose values sit exactly on rounding ties (amax = 127 * 2^-6 makes the
    activation scale 2^-6 and X / s_x = n + 1/2), subnormals, large values."""
    rng = np.random.default_rng(seed)
    ties = ((np.arange(K) % 254) - 127 + 0.5) * 2.0 ** -6
    ties[0] = 127 * 2.0 ** -6
    rows = [ties,
        np.zeros(K), np.full(K, 0.5), np.full(K, -3.0), np.linspace(-2, 2, K),
        np.where(np.arange(K) % 2 == 0, 1.0, -1.0), rng.standard_normal(K) * 1e-6,
        np.where(np.arange(K) == 7, 60000.0, 0.0),
    ]
    return f16(np.stack(rows))


# ------------------------------------------------------------------ act quant --

@pytest.mark.parametrize("M,K", [(1, 128), (7, 256), (8, 512), (16, 4096), (129, 384), (33, 8192), (300, 8192),
                                 (80, 65536)])
def test_act_quant_bit_exact(M, K):
    X = synth.activations(M, K, 100 + M)
    if M >= 8:
        X[:8] = _edge_rows(K, M)
    Xd = gc.to_dev_f16(X)
    Xq, sx = q().qoq_quant_act(Xd)
    oXq, osx = gc.oracle.act_quant(synth.bits(X))
    assert np.array_equal(Xq.cpu().numpy(), oXq)
    assert np.array_equal(gc.f16_bits(sx), osx)


# ---------------------------------------------------------------------- pack --

@pytest.mark.parametrize("N,K", [(128, 128), (256, 512), (384, 1152), (128, 8192)])
def test_pack_bit_exact_and_layout(N, K):
    W = synth.weights(N, K, 200 + N)
    W[:8] = _edge_rows(K, N) * 0.01
    # exact level-1 ties: amax = 119 * 2^-7 makes s1 = 2^-7 and W / s1 = n + 1/2
    wt = ((np.arange(K) % 238) - 119 + 0.5) * 2.0 ** -7
    wt[0] = 119 * 2.0 ** -7
    W[8] = f16(wt)
    Wd = gc.to_dev_f16(W)
    packed, s1 = q().qoq_pack_weights(Wd)
    o = gc.oracle.weight_quant(synth.bits(W), 128)
    gc.check_weights(q(), dict(packed=packed, s1=s1), o, N, K)
    # the blob itself follows the documented layout
    want = gc.pack_reference_layout(o["q4"], o["s2"], o["z"])
    assert np.array_equal(packed.cpu().numpy()[:want.size], want)


# ---------------------------------------------------------------------- GEMM --

def _run_full(M, N, K, seed, W=None, X=None):
    if W is None:
        W = synth.weights(N, K, seed)
    if X is None:
        X = synth.activations(M, K, seed)
    g = gc.gpu_layer(W, X)
    o = gc.oracle_layer(W, X)
    gc.check_weights(q(), g, o, N, K)
    gc.check_acts(g, o)
    acc = g["acc"].cpu().numpy()
    assert np.array_equal(acc.astype(np.int64), o["acc"]), \
        f"acc mismatch at {np.argwhere(acc != o['acc'])[:5].tolist()}"
    ok, rel, ab = gc.y_close(gc.f16_bits(g["Y"]), o["Y"])
    assert ok, (rel, ab)
    return g, o


def test_gemm_appendix_example_g128():
    gold = load_golden("appendix_a_g4.txt")
    K = 256
    Wl = np.zeros(K)
    Xl = np.zeros(K)
    for j in range(2):
        Wl[128 * j:128 * j + 4] = np.array(gold["Q8"][4 * j:4 * j + 4]) * 2.0 ** -7
        Xl[128 * j:128 * j + 4] = np.array(gold["Xq"][4 * j:4 * j + 4]) * 2.0 ** -6
    W = np.repeat(f16(Wl).reshape(1, K), 128, axis=0)
    X = f16(Xl).reshape(1, K)
    g, o = _run_full(1, 128, K, 0, W=W, X=X)
    assert (g["acc"].cpu().numpy() == gold["acc"]).all()
    assert (gc.f16_bits(g["Y"]) == gold["Y_bits"]).all()


def test_gemm_config0_tiny():
    c = synth.WORKLOADS[0]
    _run_full(c["M"], c["N"], c["K"], c["seed"])


@pytest.mark.parametrize("M", [1, 7, 15, 16, 17, 32, 33, 64, 65, 128, 129, 200])
def test_gemm_token_counts(M):
    # 9 groups: crosses the 8-group fp32 -> int32 fold boundary
    _run_full(M, 384, 1152, 300 + M)


@pytest.mark.parametrize("M", [65, 128, 129, 200, 256, 300])
def test_gemm_pair_token_counts(M):
    """N a multiple of 256: 128-token tiles run on CTA pairs (two weight tiles
    per pair tile, M=256 MMAs, each CTA staging half of every token tile); 9
    groups cross the fold boundary, and two pair tiles per token tile are
    split along K over the pairs."""
    _run_full(M, 512, 1152, 500 + M)


@pytest.mark.parametrize("M,N,K", [(16, 128, 4096), (64, 1024, 2048), (128, 2048, 1024), (5, 128, 16384)])
def test_gemm_split_k_shapes(M, N, K):
    _run_full(M, N, K, 400 + M)


@pytest.mark.parametrize("K", [1024, 8192])
def test_gemm_worst_case_magnitudes(K):
    """All codes at their extremes: every chunk's fp32 partial sums reach the
    largest values the format allows (127 * 120 * 1024 < 2^24)."""
    M, N = 16, 256
    W = np.full((N, K), np.float16(1.0))
    W[1::2] = np.float16(-1.0)  # Q8 = -119: group [-119, 0] -> w8 = -120
    X = np.full((M, K), np.float16(2.0))
    X[1::2] = np.float16(-2.0)
    g, o = _run_full(M, N, K, 0, W=W, X=X)
    assert int(np.abs(o["acc"]).max()) == 127 * 120 * K


def test_gemm_max_k():
    """K = 131072, the largest K the int32 accumulator admits."""
    M, N, K = 2, 128, 131072
    W = np.full((N, K), np.float16(0.5))
    X = np.full((M, K), np.float16(0.25))  # Xq = 127; Y stays within the fp16 range
    g, o = _run_full(M, N, K, 0, W=W, X=X)
    assert int(o["acc"].max()) == 127 * 120 * K


def test_gemm_zero_inputs():
    M, N, K = 4, 128, 256
    W = synth.weights(N, K, 9)
    X = np.zeros((M, K), np.float16)
    g, o = _run_full(M, N, K, 0, W=W, X=X)
    assert (g["acc"].cpu().numpy() == 0).all()


def test_gemm_deterministic_and_workspace_reuse():
    M, N, K = 24, 512, 3072
    W = synth.weights(N, K, 51)
    X = synth.activations(M, K, 51)
    g1 = gc.gpu_layer(W, X)
    g2 = gc.gpu_layer(W, X, ws=g1["ws"])
    assert np.array_equal(g1["acc"].cpu().numpy(), g2["acc"].cpu().numpy())
    assert np.array_equal(gc.f16_bits(g1["Y"]), gc.f16_bits(g2["Y"]))


# ------------------------------------------------------- full-size workloads --

@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_gemm_workload_full(cfg):
    """Full-size workloads in the benchmark's launch configuration, compared
    element by element: the quantization outputs and every int32 accumulator
    bit-exact, every fp16 Y within the tolerance.  The oracle's product runs
    on all host threads (its threaded form is pinned to the single-threaded
    one)."""
    c = synth.WORKLOADS[cfg]
    M, N, K = c["M"], c["N"], c["K"]
    W = synth.weights(N, K, c["seed"])
    X = synth.activations(M, K, c["seed"])
    g = gc.gpu_layer(W, X)
    o = gc.oracle_layer(W, X, full_gemm=False)
    gc.check_weights(q(), g, o, N, K)
    gc.check_acts(g, o)
    del W, X
    acc_ref, y_ref = gc.oracle.gemm(o["Xq"], o["sx"], o["q4"], o["s2"], o["z"], o["s1"], threads=0)
    acc = g["acc"].cpu().numpy()
    bad = acc.astype(np.int64) != acc_ref
    assert not bad.any(), f"{int(bad.sum())} accumulators differ, first at {np.argwhere(bad)[:5].tolist()}"
    ok, rel, ab = gc.y_close(gc.f16_bits(g["Y"]), y_ref)
    assert ok, (rel, ab)


# ------------------------------------------- fp32 accumulation, adversarial --

def _accumulation_case(M: int, N: int, K: int, small_group):
    """Weights and activations whose fp32 partial sums first climb into
    [2^23, 2^24) with maximal products and then take +-1 products.

    Group j of every weight row is "big" (Q8 = 119 on all 128 channels: s2 = 8,
    z = 0, w8 = 120) unless small_group(j), where it is "small" (Q8 in {0, 1}
    or {-1, 0}: s2 = 1, w8 = +-1).  The activations are given as codes: 127
    on big channels (the sign alternates per token) and a fixed +-1 pattern on
    small ones, so that a dropped +-1 changes the exact sum.  In the fp32
    accumulator of one fold chunk (8 groups per accumulator), seven big groups
    reach 7 * 128 * 127 * 120 = 13,655,040 units, where the fp32 spacing is 1,
    and the small group's products then land one unit at a time."""
    G = K // 128
    s1 = 2.0 ** -10
    W = np.empty((N, K), np.float64)
    row_sign = np.where(np.arange(N) % 2 == 0, 1.0, -1.0)[:, None]
    for j in range(G):
        cols = slice(128 * j, 128 * j + 128)
        if small_group(j):
            pat = (np.arange(128) % 3 != 1).astype(np.float64)  # codes 0 / 1
            W[:, cols] = row_sign * pat[None, :] * s1
        else:
            W[:, cols] = 119 * s1
    Xq = np.empty((M, K), np.int8)
    tok_sign = np.where(np.arange(M) % 2 == 0, 1, -1)[:, None]
    for j in range(G):
        cols = slice(128 * j, 128 * j + 128)
        if small_group(j):
            Xq[:, cols] = np.where(np.arange(128) % 4 == 1, -1, 1)[None, :]
        else:
            Xq[:, cols] = 127 * tok_sign
    sx = np.full(M, 0x0400, np.uint16)  # 2^-14: Y stays well inside the fp16 range
    return f16(W), Xq, sx


@pytest.mark.parametrize("kernel", ["decode", "bulk"])
def test_gemm_fp32_accumulation_large_then_unit_products(kernel):
    """The exact-integer product runs on fp32 tensor-core accumulators, exact
    while partial sums stay below 2^24.  Drive each accumulator's partial sums
    to 13.7M units (past 2^23, where only integers are representable) with
    maximal products, then add +-1 products: any truncation in the tensor
    core's accumulation shows as a wrong int32 result.  Whole tiles only (N is
    chosen so that every CTA takes one tile and no split-K applies), so the
    fold chunks start at group 0: the decode kernel's four slots take groups
    j, j + 4, ... of each 32-group chunk, the bulk kernel folds every 8
    consecutive groups."""
    import torch

    mod = q()
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 160)
    if kernel == "decode":
        M, K = 16, 8192
        N = 128 * sms
        small = lambda j: j % 32 >= 28  # each slot: 7 big groups, then 1 small, per chunk
    else:
        M, K = 256, 4096
        N = 128 * (sms // 2)
        small = lambda j: j % 8 == 7    # 7 big groups, then 1 small, per chunk
    W, Xq, sx = _accumulation_case(M, N, K, small)
    o = gc.oracle.weight_quant(synth.bits(W), 128)
    w8 = gc.oracle.dequant_weights(o["q4"], o["s2"], o["z"], 128)
    assert set(np.unique(w8).tolist()) == {-1, 0, 1, 120}, "case construction"
    acc_ref, y_ref = gc.oracle.gemm(Xq, sx, o["q4"], o["s2"], o["z"], o["s1"], threads=0)
    packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(W))
    t = gc.torch()
    Xq_d = t.from_numpy(Xq).cuda()
    sx_d = t.from_numpy(sx.view(np.float16)).cuda()
    acc = t.empty((M, N), dtype=t.int32, device="cuda")
    ws = t.zeros(mod.qoq_gemm_workspace_bytes(M, N, K), dtype=t.uint8, device="cuda")
    Y = mod.qoq_w4a8_gemm(Xq_d, sx_d, packed, s1, N, acc_debug=acc, workspace=ws)
    assert mod.qoq_last_device_status(ws) == 0
    assert np.array_equal(gc.f16_bits(s1), o["s1"])
    got = acc.cpu().numpy().astype(np.int64)
    bad = got != acc_ref
    assert not bad.any(), f"{int(bad.sum())} accumulators differ, e.g. {got[bad][:3]} vs {acc_ref[bad][:3]}"
    ok, rel, ab = gc.y_close(gc.f16_bits(Y), y_ref)
    assert ok, (rel, ab)


# ------------------------------------------------------- failure detection --

@pytest.mark.parametrize("M,N,K", [(16, 12288, 4096), (256, 4096, 14336)])
def test_gemm_exact_across_alternating_inputs(M, N, K):
    """Repeated calls that alternate between two input sets (different weights
    and activations), with a call that times out on purpose now and then:
    every int32 accumulator must equal that input set's first result, bit for
    bit.  Any pipeline wait that passes before its data is ready reads what
    the previous call left in shared or tensor memory, which here always
    belongs to the other input set."""
    mod = q()
    t = gc.torch()
    sets = []
    for seed in (81, 82):
        packed, s1 = mod.qoq_pack_weights(gc.to_dev_f16(synth.weights(N, K, seed)))
        Xq, sx = mod.qoq_quant_act(gc.to_dev_f16(synth.activations(M, K, seed)))
        sets.append((Xq, sx, packed, s1))
    ws = t.zeros(mod.qoq_gemm_workspace_bytes(M, N, K), dtype=t.uint8, device="cuda")
    refs = []
    for Xq, sx, packed, s1 in sets:
        acc = t.empty((M, N), dtype=t.int32, device="cuda")
        mod.qoq_w4a8_gemm(Xq, sx, packed, s1, N, acc_debug=acc, workspace=ws)
        refs.append(acc)
    # a small call that times out on purpose (test hook), with its own workspace
    Mt, Nt, Kt = 16, 128 * 152, 4096  # 32 groups per CTA: the hook (group 17) fires
    pt, s1t = mod.qoq_pack_weights(gc.to_dev_f16(synth.weights(Nt, Kt, 83)))
    Xqt, sxt = mod.qoq_quant_act(gc.to_dev_f16(synth.activations(Mt, Kt, 83)))
    wst = t.zeros(mod.qoq_gemm_workspace_bytes(Mt, Nt, Kt), dtype=t.uint8, device="cuda")
    acc = t.empty((M, N), dtype=t.int32, device="cuda")
    bad = []
    for i in range(120):
        if i % 20 == 19:
            try:
                mod.qoq_set_debug(2_000_000, 1)
                mod.qoq_w4a8_gemm(Xqt, sxt, pt, s1t, Nt, workspace=wst)
                mod.qoq_last_device_status(wst)
            finally:
                mod.qoq_set_debug(0, 0)
            wst.zero_()
        j = i % 2
        acc.fill_(-1)
        mod.qoq_w4a8_gemm(*sets[j], N, acc_debug=acc, workspace=ws)
        if not t.equal(acc, refs[j]):
            bad.append(i)
    assert mod.qoq_last_device_status(ws) == 0
    assert not bad, f"calls {bad} differ from their input set's first result"


@pytest.mark.parametrize("M,N,K", [(16, 128 * 152, 8192), (200, 4096, 8192)])
def test_device_wait_timeout_is_reported_and_context_survives(M, N, K):
    """A producer that skips one pipeline stage (test hook) makes the waits
    downstream run out after a short limit; the kernel returns, the status
    reads QOQ_ERR_DEVICE_TIMEOUT, and the next call is correct.  M=16: the
    decode kernel; M=200, N=4096: the CTA-pair kernel, where the other CTA of
    the pair and the leading CTA's MMA issuer run out as well."""
    mod = q()
    t = gc.torch()
    W = synth.weights(N, K, 61)
    X = synth.activations(M, K, 61)
    Wd, Xd = gc.to_dev_f16(W), gc.to_dev_f16(X)
    packed, s1 = mod.qoq_pack_weights(Wd)
    Xq, sx = mod.qoq_quant_act(Xd)
    ws = t.zeros(mod.qoq_gemm_workspace_bytes(M, N, K), dtype=t.uint8, device="cuda")
    try:
        mod.qoq_set_debug(5_000_000, 1)  # 5 ms wait limit, skip one stage
        mod.qoq_w4a8_gemm(Xq, sx, packed, s1, N, workspace=ws)
        assert mod.qoq_last_device_status(ws) == 7
    finally:
        mod.qoq_set_debug(0, 0)
    ws.zero_()  # an aborted call leaves split-K state behind: clear before reuse
    acc = t.empty((M, N), dtype=t.int32, device="cuda")
    mod.qoq_w4a8_gemm(Xq, sx, packed, s1, N, acc_debug=acc, workspace=ws)
    assert mod.qoq_last_device_status(ws) == 0
    # the oracle quantizes rows independently: only the sampled rows are needed
    rows = np.arange(0, N, N // 8)
    o = gc.oracle.weight_quant(synth.bits(W[rows]), 128)
    oXq, osx = gc.oracle.act_quant(synth.bits(X))
    mi = np.arange(0, M).repeat(len(rows))
    ni = np.tile(np.arange(len(rows)), M)
    acc_ref, _ = gc.oracle.gemm_entries(mi, ni, oXq, osx, o["q4"], o["s2"], o["z"], o["s1"])
    assert np.array_equal(acc.cpu().numpy()[mi, rows[ni]].astype(np.int64), acc_ref)
