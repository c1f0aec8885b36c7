"""bench.py's host logic (CPU): the algorithmic byte count behind the roofline,
the DRAM-traffic record's source check, and the reference arm's JSON line,
which runs the oracle on the host cores and needs no GPU."""
import importlib.util
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes_decode_workload(bench):
    # M=16, N=12288, K=4096, g=128: nibbles N K / 2, one s2 and one z byte per
    # (row, group), fp16 s1, int8 Xq, fp16 s_x, fp16 Y
    M, N, K = 16, 12288, 4096
    b = bench.algorithmic_bytes(M, N, K, 128)
    assert b["gemm"] == 25165824 + 786432 + 24576 + 65536 + 32 + 393216 == 26435616
    # the quantizer reads fp16 X, writes int8 Xq and fp16 s_x
    assert b["act"] == 2 * M * K + M * K + 2 * M
    assert b["step"] == b["gemm"] + b["act"]
    # smaller groups carry more scale bytes, larger ones fewer (minimal bytes)
    assert bench.algorithmic_bytes(M, N, K, 32)["gemm"] - b["gemm"] == 2 * N * (K // 32 - K // 128)
    assert bench.algorithmic_bytes(M, N, K, 256)["gemm"] < b["gemm"]


def test_traffic_record_follows_the_gemm_sources(bench, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["decode_qkv_7b"]
    assert rec["algorithmic_bytes_per_launch"] == bench.algorithmic_bytes(16, 12288, 4096)["gemm"]
    traffic, src = bench.recorded_traffic("decode_qkv_7b")
    if rec["source_sha256"] == bench.gemm_source_hash():
        assert traffic == rec["dram_bytes_per_launch"]
    else:
        assert traffic is None
    # any change to the GEMM sources voids the record
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 64)
    assert bench.recorded_traffic("decode_qkv_7b")[0] is None


def test_reference_arm_json_line(bench):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "decode_qkv_7b"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    # the reference arm times the same workload as the GPU arm, on all host cores
    assert "full workload" in cb["sample"]
    import oracle

    assert cb["cores"] == oracle.host_cores()
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_sample_is_bounded(bench):
    """The full workload where the product is small; otherwise a multiple of
    128 output channels that keeps the oracle's work near the bound."""
    from w4a8_quantized_serving_gb300 import synth

    W = synth.WORKLOADS
    assert bench.oracle_sample_channels(W[1], 2e10) == W[1]["N"]
    n4 = bench.oracle_sample_channels(W[4], 2e10)
    assert n4 % 128 == 0 and 128 <= n4 < W[4]["N"]
    assert W[4]["M"] * n4 * W[4]["K"] <= 2e10
    assert bench.oracle_sample_channels(W[4], 1.0) == 128


def test_roofline_picks_the_binding_roof(bench):
    """Below the ridge the GEMM is reported against HBM (algorithmic bytes per
    launch / time), above it against the tensor peak (2MNK / time)."""
    peaks = {"hbm_gbs": 6666.9, "bf16_tflops": 1967.3, "bf16_tflops_sustained": 1756.1}
    r = bench.roofline_of(16, 12288, 4096, 128, 0.01, 20, peaks, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(26435616 / 1e-5 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6666.9)
    r = bench.roofline_of(4096, 28672, 8192, 128, 1.4, 20, peaks, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1967.3
    assert r["achieved"] == pytest.approx(2.0 * 4096 * 28672 * 8192 / 1.4e-3 / 1e12)
    # a long timed region runs under the power cap: the sustained peak
    assert bench.roofline_of(4096, 28672, 8192, 128, 1.4, 1000, peaks, "measured")["peak"] == 1756.1


def _max_over_ranks_worker(rank, world, port, q):
    import torch.distributed as dist

    spec = importlib.util.spec_from_file_location("bench_in_rank", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 5.0 - rank, 2.5]  # each rank's timings
        q.put((rank, mod.max_over_ranks(dist, mine, "cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    """The job's time is the slowest rank's, element by element, on every
    rank (world size 2, gloo on CPU)."""
    import socket

    import torch.multiprocessing as mp

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_max_over_ranks_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [2.0, 5.0, 2.5]


def test_job_throughput_counts_every_rank(bench):
    ops = 2.0 * 16 * 12288 * 4096
    assert bench.job_tops(1, ops, 0.01) == pytest.approx(ops / 1e-5 / 1e12)
    assert bench.job_tops(4, ops, 0.01) == pytest.approx(4 * bench.job_tops(1, ops, 0.01))
    assert bench.max_over_ranks(None, [1, 2.5], "cpu") == [1.0, 2.5]


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT,
                         env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    assert not [l for l in out.stdout.splitlines() if l.startswith("{")]
