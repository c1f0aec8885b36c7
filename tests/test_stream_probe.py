"""The benchmark's probes (libqoq_probe.so): the streaming-read probe
(csrc/probe_stream.cu) and the tcgen05.mma issue-rate probe (csrc/probe_mma.cu).

It sets the GEMM call's HBM figure beside what a launch that only reads the
same bytes takes, so it must really read every byte once: the GPU cases check
its word sum against numpy's, for sizes that leave ragged tails of the
unrolled loop, in both launch forms and every grid shape.  The CPU cases check
that it is built, exported, and rejects bad arguments on the host."""
import ctypes
import os

import numpy as np
import pytest

from tests.conftest import gpu_available

FAKE = 0x7F0000001000  # 16-byte aligned, never dereferenced: the calls below fail validation first
CUDA_ERROR_INVALID_VALUE = 1


def probe():
    from w4a8_quantized_serving_gb300.csrc import build as cbuild

    if not os.path.exists(cbuild.PROBE_LIB):
        pytest.skip("libqoq_probe.so not built")
    L = ctypes.CDLL(cbuild.PROBE_LIB)
    L.qoq_probe_stream_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p]
    L.qoq_probe_stream_read.restype = ctypes.c_int
    L.qoq_probe_stream_ring.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    L.qoq_probe_stream_ring.restype = ctypes.c_int
    L.qoq_probe_mma_issue.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    L.qoq_probe_mma_issue.restype = ctypes.c_int
    return L


def test_probe_is_built_beside_the_library_and_not_into_it():
    from w4a8_quantized_serving_gb300.csrc import build as cbuild

    for src in ("probe_stream.cu", "probe_mma.cu"):
        assert src in cbuild.PROBE_SOURCES and src not in cbuild.SOURCES
    L = probe()
    for name in ("qoq_probe_stream_read", "qoq_probe_stream_ring", "qoq_probe_mma_issue"):
        assert hasattr(L, name)


def test_probe_rejects_bad_arguments_on_the_host():
    L = probe()
    sink = FAKE + 0x1000
    assert L.qoq_probe_stream_read(FAKE, 0, sink, 2, 1, None) == 0  # nothing to read: no launch
    assert L.qoq_probe_stream_read(None, 64, sink, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert L.qoq_probe_stream_read(FAKE, 64, None, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert L.qoq_probe_stream_read(FAKE + 8, 64, sink, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert L.qoq_probe_stream_read(FAKE, 72, sink, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert L.qoq_probe_stream_read(FAKE, 64, sink + 4, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    for bad in (0, 5, -1):
        assert L.qoq_probe_stream_read(FAKE, 64, sink, bad, 1, None) == CUDA_ERROR_INVALID_VALUE
    err = FAKE + 0x2000
    ring = L.qoq_probe_stream_ring
    assert ring(FAKE, 0, sink, err, 8192, 2, 1, None) == 0
    assert ring(None, 64, sink, err, 8192, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert ring(FAKE, 64, sink, None, 8192, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert ring(FAKE + 8, 64, sink, err, 8192, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert ring(FAKE, 72, sink, err, 8192, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert ring(FAKE, 64, sink + 4, err, 8192, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    assert ring(FAKE, 64, sink, err + 2, 8192, 2, 1, None) == CUDA_ERROR_INVALID_VALUE
    for chunk, prod in ((4096, 1), (12288, 1), (8192, 0), (8192, 3)):
        assert ring(FAKE, 64, sink, err, chunk, prod, 1, None) == CUDA_ERROR_INVALID_VALUE
    mma = L.qoq_probe_mma_issue
    for pair, n, iters, out in ((2, 128, 64, FAKE), (0, 48, 64, FAKE), (1, 64, 64, FAKE), (0, 128, 1, FAKE),
                                (0, 128, (1 << 20) + 1, FAKE), (0, 128, 64, None), (1, 256, 64, FAKE + 4)):
        assert mma(pair, n, iters, out, None) == CUDA_ERROR_INVALID_VALUE


@pytest.mark.gpu
@pytest.mark.skipif(not gpu_available(), reason="needs a GPU")
@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 5 * (1 << 20) + 48, 26435616, 64 << 20])
@pytest.mark.parametrize("dependent", [0, 1])
@pytest.mark.parametrize("ctas_per_sm", [1, 2, 4])
def test_probe_reads_every_byte_once(nbytes, dependent, ctas_per_sm):
    import torch

    L = probe()
    rng = np.random.default_rng(nbytes + 7 * dependent + ctas_per_sm)
    host = rng.integers(0, 256, nbytes, dtype=np.uint8)
    buf = torch.from_numpy(host).cuda()
    sink = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # twice: the sum accumulates
        assert L.qoq_probe_stream_read(buf.data_ptr(), nbytes, sink.data_ptr(), ctas_per_sm, dependent, st) == 0
    torch.cuda.synchronize()
    want = (2 * int(host.view(np.uint32).astype(np.uint64).sum(dtype=np.uint64))) % (1 << 64)
    got = int(sink.cpu().numpy().view(np.uint64)[0])
    assert got == want


@pytest.mark.gpu
@pytest.mark.skipif(not gpu_available(), reason="needs a GPU")
@pytest.mark.parametrize("nbytes", [16, 8192, 16384 + 16, 24 * 8192 * 152 + 48, 26435616, (64 << 20) + 16])
@pytest.mark.parametrize("prefetch", [0, 1])
@pytest.mark.parametrize("chunk,producers", [(8192, 2), (8192, 1), (16384, 2), (16384, 1)])
def test_ring_probe_reads_every_byte_once(nbytes, prefetch, chunk, producers):
    """The ring form: one chunk, a ragged last chunk, exactly one lap per SM
    plus a tail, the decode GEMM's bytes, several laps per SM."""
    import torch

    L = probe()
    rng = np.random.default_rng(nbytes + 3 * prefetch + chunk + 5 * producers)
    host = rng.integers(0, 256, nbytes, dtype=np.uint8)
    buf = torch.from_numpy(host).cuda()
    sink = torch.zeros(1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        assert L.qoq_probe_stream_ring(buf.data_ptr(), nbytes, sink.data_ptr(), err.data_ptr(), chunk, producers,
                                       prefetch, st) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = (2 * int(host.view(np.uint32).astype(np.uint64).sum(dtype=np.uint64))) % (1 << 64)
    assert int(sink.cpu().numpy().view(np.uint64)[0]) == want


@pytest.mark.gpu
@pytest.mark.skipif(not gpu_available(), reason="needs a GPU")
def test_probe_chain_in_a_graph_times_like_the_bench():
    """The benchmark's own harness: a graph of dependent launches over a buffer
    pool larger than 3x L2, replayed; the result is a positive time below the
    one a launch would take at 1% of the copy bandwidth."""
    import importlib.util
    import types

    import torch

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)

    for form in ("read", "ring"):
        r = bench.stream_floor(torch, torch.device("cuda", 0), 26435616, steps=8, repeats=2, form=form)
        assert r["bytes"] == 26435616 and len(r["regions_ms_per_launch"]) == 2 and r["form"] == form
        assert 0 < r["ms_per_launch"] < 26435616 / (0.01 * 6.6e12) * 1e3
    peaks, _ = bench.load_peaks()
    fl = bench.hbm_floor_of(torch, torch.device("cuda", 0), 76304, 0.01,
                            types.SimpleNamespace(steps=8, repeats=2), peaks)
    assert fl["read"]["dependent"] and fl["ring"]["gemm_ms_over_floor"] > 0


@pytest.mark.gpu
@pytest.mark.skipif(not gpu_available(), reason="needs a GPU")
@pytest.mark.parametrize("pair,n", [(False, 16), (False, 64), (False, 128), (False, 256), (True, 128), (True, 256)])
def test_mma_issue_probe_completes_with_plausible_rates(pair, n):
    """Every launch completes (its bounded wait did not give up), the issue
    stamps rise, and the rates lie between a few and a few thousand cycles."""
    import importlib.util

    import torch

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    r = bench.mma_issue_probe(torch, torch.device("cuda", 0), pair, n, iters=512, reps=2)
    assert r["completed"] and r["iters"] == 512
    assert 4 < r["issue_cycles_per_mma"] < 5000
    assert r["issue_cycles_per_mma"] <= r["complete_cycles_per_mma"] + 1
    assert all(g > 0 for g in r["first_issue_gaps"])
