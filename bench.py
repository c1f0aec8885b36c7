"""Benchmark of the W4A8 g128 linear layer on GB300.

One step = one pass of the hot path over one batch: per-token int8
quantization of the activations (qoq_quant_act) and the W4A8 GEMM
(qoq_w4a8_gemm), with the weights packed offline (qoq_pack_weights, timed
separately).  Default workload: the 7B fused-QKV decode projection,
M=16, N=12288, K=4096, g=128 (seed 1).

Timing: W untimed warm-up steps, then timed regions of exactly K steps each
(a CUDA graph of K steps, replayed), every region between CUDA events on the
launching stream with a barrier and a device synchronize on both sides; the
line reports the median region.  The inputs of consecutive steps rotate
through a pool of independent buffer sets larger than 3x L2, so every step
streams its weights from HBM.

Output: one JSON line (rank 0).  Keys beyond the metric: roofline of the
dominant kernel (the GEMM call), the oracle's CPU baseline (all host cores and
one), the end-to-end number through the public API with host buffers, clocks
sampled during the timed regions, the count of kernel launches inside a
region, and a per_config block with the same measurements for every workload
of the metric (M = 8 .. 4096).

--impl reference times the oracle (the plain CPU implementation the tests
check against) on all host cores instead: it is the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from w4a8_quantized_serving_gb300 import synth  # noqa: E402

METRIC = "W4A8 g128 GEMM effective TOPS & HBM GB/s (% of roofline), M=1..4096"
UNIT = "TOPS"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def algorithmic_bytes(M: int, N: int, K: int, g: int = 128, n8: int | None = None) -> dict:
    """Bytes the GEMM call must move at least once: q4 nibbles, per-group s2 and
    z, s1, Xq, s_x, and the fp16 output; plus the activation quantizer's.
    With n8 (the W4Ax path): the activations are the n8 8-bit blocks (128 bytes
    per token) and the 4-bit ones (64 bytes), with one fp16 scale per (token,
    block)."""
    weights = N * K // 2 + 2 * N * (K // g) + 2 * N
    if n8 is None:
        acts = M * K + 2 * M
    else:
        G = K // 128
        acts = M * (128 * n8 + 64 * (G - n8)) + 2 * M * G
    gemm = weights + acts + 2 * M * N
    act = 2 * M * K + acts
    return {"gemm": gemm, "act": act, "step": gemm + act}


def outlier_first_permutation(seed: int, K: int) -> np.ndarray:
    """Channel order with the activation generator's outlier channels first
    (the W4Ax path's channel permutation: they fall into the leading 8-bit
    block), the other channels in their order."""
    out = synth.outlier_channels(seed, synth.TAG_X, K, 4)
    return np.concatenate([out, np.setdiff1d(np.arange(K), out)])


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


GEMM_SOURCES = ["gemm.cu", "gemm_decode.cu", "gemm_common.cuh", "ptx.cuh", "internal.h"]


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "w4a8_quantized_serving_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(workload: str) -> tuple[float | None, str]:
    """DRAM bytes per GEMM launch from the committed ncu record, if the GEMM
    sources are unchanged since it was taken (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None, "no ncu record"
    if not rec:
        return None, "no ncu record for this workload"
    if rec.get("source_sha256") != gemm_source_hash():
        return None, "GEMM sources changed since the ncu capture"
    return float(rec["dram_bytes_per_launch"]), rec.get("capture", "")


def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(dist, vals: list, device) -> list:
    """Element-wise maximum of per-rank timings, returned on every rank (the
    slowest rank sets the job's time); the values themselves without a group."""
    if dist is None:
        return [float(v) for v in vals]
    import torch

    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tops(world: int, ops: float, ms: float) -> float:
    """Whole-job throughput: every rank does `ops` per step in `ms` (the max
    over ranks), so the job does world * ops per step."""
    return world * ops / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power), "reasons": sorted(reasons)}


# ------------------------------------------------------------- CPU oracle --

def oracle_sample_channels(c: dict, macs_per_step: float) -> int:
    """Output channels of a bounded oracle sample: all N when the workload's
    product is at most `macs_per_step` multiply-adds, else a multiple of 128
    that keeps it near that size."""
    M, N, K = c["M"], c["N"], c["K"]
    if M * N * K <= macs_per_step:
        return N
    return max(128, int(macs_per_step / (M * K)) // 128 * 128)


def oracle_step_timing(c: dict, budget_s: float, threads: int, n_sample: int | None = None) -> dict:
    """Time the oracle on a (bounded) sample of the workload: all M tokens
    quantized, the GEMM over the first n_sample output channels (weights
    quantized beforehand, outside the timing, as on the GPU).  threads: host
    threads of the oracle's product (0: all cores; its per-token quantizer is
    single-threaded)."""
    import oracle

    M, N, K = c["M"], c["N"], c["K"]
    g = c.get("g", 128)
    n_sample = min(N, N if n_sample is None else n_sample)
    W = synth.weights(n_sample, K, c["seed"])  # the first n_sample output channels
    X = synth.activations(M, K, c["seed"])
    wq = oracle.weight_quant(synth.bits(W), g)
    cores = oracle.host_cores() if threads == 0 else threads
    times = []
    t_end = time.perf_counter() + budget_s
    while True:
        t0 = time.perf_counter()
        Xq, sx = oracle.act_quant(synth.bits(X))
        oracle.gemm(Xq, sx, wq["q4"], wq["s2"], wq["z"], wq["s1"], g, want_acc=False, threads=threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() >= t_end or len(times) >= 50:
            break
    t = statistics.median(times)
    ops = 2.0 * M * n_sample * K
    what = "the full workload" if n_sample == N else f"GEMM over {n_sample} of {N} output channels"
    return {"value": ops / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"act-quant of all {M} tokens + {what}, K={K}; median of {len(times)} runs of "
                      f"{t:.4f} s (C oracle, {cores} host thread{'s' if cores > 1 else ''})",
            "seconds_per_sample": t}


def cpu_baselines(c: dict, budget_s: float) -> dict:
    """The oracle on all host cores (the reported baseline) and, on a smaller
    bounded sample, on one core."""
    allc = oracle_step_timing(c, budget_s * 0.5, threads=0, n_sample=oracle_sample_channels(c, 2e10))
    one = oracle_step_timing(c, budget_s * 0.5, threads=1, n_sample=oracle_sample_channels(c, 8e8))
    allc["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}
    return allc


def run_reference(args, c: dict) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    M, N, K = c["M"], c["N"], c["K"]
    g = c.get("g", 128)
    import oracle

    n_sample = oracle_sample_channels(c, 2e10)  # the full workload for M <= 1024-class shapes
    W = synth.weights(n_sample, K, c["seed"])
    X = synth.activations(M, K, c["seed"])
    wq = oracle.weight_quant(synth.bits(W), g)

    def step():
        Xq, sx = oracle.act_quant(synth.bits(X))
        oracle.gemm(Xq, sx, wq["q4"], wq["s2"], wq["z"], wq["s1"], g, want_acc=False, threads=0)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = 2.0 * M * n_sample * K / dt / 1e12
    cores = oracle.host_cores()
    what = "the full workload" if n_sample == N else f"GEMM over {n_sample} of {N} output channels"
    sample = f"per step: act-quant of {M} tokens + {what}, K={K}, on {cores} host threads"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int64", "data": "synthetic",
        "config": config_dict(c),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(c: dict, extra: dict | None = None) -> dict:
    d = {"workload": c["name"], "M": c["M"], "N": c["N"], "K": c["K"], "g": c.get("g", 128), "seed": c["seed"]}
    if extra:
        d.update(extra)
    return d


# ------------------------------------------------------------------ GPU arm --

def roofline_of(M: int, N: int, K: int, g: int, gemm_ms: float, steps: int, peaks: dict, peak_src: str,
                n8: int | None = None) -> dict:
    """The GEMM call against the roofline that binds it: HBM below the ridge
    (algorithmic bytes / time), the tensor pipe above it (2MNK / time)."""
    ops = 2.0 * M * N * K
    nbytes = algorithmic_bytes(M, N, K, g, n8)["gemm"]
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if ops / nbytes < ridge:
        achieved = nbytes / (gemm_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
    else:
        achieved = ops / (gemm_ms * 1e-3) / 1e12
        sustained = steps * gemm_ms > 1000
        pk = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s", "frac": achieved / pk,
                "peak_source": f"{peak_src} bf16 dense {'sustained' if sustained else 'burst'} "
                               "(fp16 operands run at the bf16 rate)"}
    roof["algorithmic_bytes_per_launch"] = nbytes
    roof["ms_per_launch"] = gemm_ms
    roof["gb_per_s_algorithmic"] = nbytes / (gemm_ms * 1e-3) / 1e9
    roof["tops_effective"] = ops / (gemm_ms * 1e-3) / 1e12
    return roof


_PROBE = None


def probe_lib():
    """libqoq_probe.so (the streaming-read probe, csrc/probe_stream.cu), built
    beside libqoq.so; measurement support, not part of the W4A8 path."""
    global _PROBE
    if _PROBE is None:
        import ctypes

        from w4a8_quantized_serving_gb300.csrc import build as _b

        if not os.path.exists(_b.PROBE_LIB):
            raise SystemExit(f"{_b.PROBE_LIB} not found (run __graft_entry__.build())")
        L = ctypes.CDLL(_b.PROBE_LIB)
        P, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        L.qoq_probe_stream_read.argtypes = [P, sz, P, i32, i32, P]
        L.qoq_probe_stream_read.restype = i32
        L.qoq_probe_stream_ring.argtypes = [P, sz, P, P, i32, i32, i32, P]
        L.qoq_probe_stream_ring.restype = i32
        L.qoq_probe_mma_issue.argtypes = [i32, i32, i32, P, P]
        L.qoq_probe_mma_issue.restype = i32
        _PROBE = L
    return _PROBE


def stream_floor(torch, dev, nbytes: int, steps: int, repeats: int, form: str = "read", dependent: bool = True,
                 ctas_per_sm: int = 2, chunk: int = 8192, producers: int = 2) -> dict:
    """Time per launch of a chain of `steps` streaming reads of `nbytes` each
    (rounded up to 16), timed like the GEMM call: a CUDA graph of the chain,
    `repeats` replays between events, the median; consecutive launches read
    distinct buffers of a pool of at least 8 and larger than 3x L2, each
    launch a programmatic dependent of the one before.
    form "read": 16-byte loads from ctas_per_sm CTAs per SM, waiting for the
    preceding launch before the first read if `dependent`.
    form "ring": the decode GEMM's way (one CTA per SM, `producers` threads
    bulk-copying `chunk`-byte pieces into a 192 KB shared-memory ring,
    consumer warps); `dependent` then means the first lap is copied before the
    wait and consumed after it, as the GEMM does with its weights (else
    nothing is read before the wait).
    The HBM time one launch of that size needs on this GPU."""
    L = probe_lib()
    nbytes = (int(nbytes) + 15) // 16 * 16
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nbuf = max(8, int(np.ceil(3 * l2 / nbytes)))
    bufs = [torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev) for _ in range(nbuf)]
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def chain(n: int):
        st = torch.cuda.current_stream().cuda_stream
        for i in range(n):
            if form == "ring":
                e = L.qoq_probe_stream_ring(bufs[i % nbuf].data_ptr(), nbytes, sink.data_ptr(), err.data_ptr(),
                                            chunk, producers, 1 if dependent else 0, st)
            else:
                e = L.qoq_probe_stream_read(bufs[i % nbuf].data_ptr(), nbytes, sink.data_ptr(), ctas_per_sm,
                                            1 if dependent else 0, st)
            if e != 0:
                raise RuntimeError(f"stream probe ({form}): cudaError {e}")

    chain(3)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain(steps)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    out = []
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / steps)
    if int(err.item()) != 0:
        raise RuntimeError(f"stream probe ({form}): a wait inside the kernel gave up")
    del graph, bufs
    ms = statistics.median(out)
    r = {"form": form, "bytes": nbytes, "ms_per_launch": ms, "gb_per_s": nbytes / (ms * 1e-3) / 1e9,
         "regions_ms_per_launch": [round(v, 6) for v in out], "dependent": dependent}
    if form == "read":
        r["ctas_per_sm"] = ctas_per_sm
    else:
        r["chunk_bytes"], r["producers"] = chunk, producers
    return r


def hbm_floor_of(torch, dev, nbytes: int, gemm_ms: float, args, peaks: dict) -> dict:
    """Two streaming-read chains at the GEMM call's algorithmic bytes, beside
    the GEMM call's own time per launch: plain loads that wait for the
    preceding launch first ("read"), and the GEMM's own copy structure with its
    first lap copied before that wait ("ring")."""
    out = {}
    for form in ("read", "ring"):
        fl = stream_floor(torch, dev, nbytes, args.steps, args.repeats, form=form, dependent=True)
        fl["frac_of_peak"] = fl["gb_per_s"] / peaks["hbm_gbs"]
        fl["gemm_ms_over_floor"] = gemm_ms / fl["ms_per_launch"]
        out[form] = fl
    out["kernel"] = ("libqoq_probe.so: one read of the GEMM call's algorithmic bytes per launch, each launch a "
                     "programmatic dependent of the one before, timed like the GEMM call; 'read': 16-byte loads "
                     "after the wait for the preceding launch; 'ring': the decode GEMM's copy structure (one CTA "
                     "per SM, two producer threads, 8 KB bulk copies into a 192 KB ring), first lap copied before "
                     "that wait")
    return out


def run_stream_sweep(args) -> None:
    """--stream-sweep: the streaming-read chains over launch sizes from 1 MiB
    to 1 GiB (and the algorithmic bytes of the two HBM-bound workloads): plain
    loads, dependent and independent, also over 1, 2 and 4 CTAs per SM at the
    decode size; the GEMM-like ring (two producers, 8 KB copies) with and
    without its first lap copied before the wait, and at the decode size and
    1 GiB with one producer or 16 KB copies.  One JSON line."""
    import torch

    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    decode = synth.WORKLOADS[1]
    dec_bytes = algorithmic_bytes(decode["M"], decode["N"], decode["K"])["gemm"]
    tiny = synth.WORKLOADS[0]
    sizes = sorted({1 << 20, 1 << 22, 1 << 24, dec_bytes, 1 << 26, 1 << 28, 1 << 30,
                    algorithmic_bytes(tiny["M"], tiny["N"], tiny["K"])["gemm"]})
    if args.stream_bytes:
        sizes = [int(b) for b in args.stream_bytes.split(",")]
    sampler = ClockSampler(local)
    sampler.start()
    rows = []
    for nb in sizes:
        for dep in (True, False):
            r = stream_floor(torch, dev, nb, args.steps, args.repeats, dependent=dep)
            r["frac_of_peak"] = r["gb_per_s"] / peaks["hbm_gbs"]
            rows.append(r)
    for cps in (1, 4) if not args.stream_bytes else ():
        r = stream_floor(torch, dev, dec_bytes, args.steps, args.repeats, dependent=True, ctas_per_sm=cps)
        r["frac_of_peak"] = r["gb_per_s"] / peaks["hbm_gbs"]
        rows.append(r)
    for nb in sizes:
        for pre in (True, False):
            r = stream_floor(torch, dev, nb, args.steps, args.repeats, form="ring", dependent=pre)
            r["frac_of_peak"] = r["gb_per_s"] / peaks["hbm_gbs"]
            rows.append(r)
    for nb in (dec_bytes, 1 << 30) if not args.stream_bytes else ():  # the copy size and the number of issuing threads
        for chunk, prod in ((8192, 1), (16384, 1), (16384, 2)):
            r = stream_floor(torch, dev, nb, args.steps, args.repeats, form="ring", dependent=True, chunk=chunk,
                             producers=prod)
            r["frac_of_peak"] = r["gb_per_s"] / peaks["hbm_gbs"]
            rows.append(r)
    clocks = sampler.stop()
    print(json.dumps({"stream_sweep": rows, "peak_hbm_gbs": peaks["hbm_gbs"], "peak_source": peak_src,
                      "steps": args.steps, "repeats": args.repeats, "clocks": clocks}), flush=True)


def mma_issue_probe(torch, dev, pair: bool, n: int, iters: int = 2048, reps: int = 3) -> dict:
    """One thread issuing `iters` tcgen05.mma of the GEMM's shape back to back
    (csrc/probe_mma.cu): cycles per issue over the whole run, cycles per MMA
    until all completed, and the spacing of the first 64 issues (median of the
    first 8 and of issues 48-63).  The last of `reps` launches is reported."""
    L = probe_lib()
    out = torch.zeros(68, dtype=torch.int64, device=dev)
    h = None
    for _ in range(reps):
        e = L.qoq_probe_mma_issue(1 if pair else 0, n, iters, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        if e != 0:
            raise RuntimeError(f"qoq_probe_mma_issue: cudaError {e}")
        torch.cuda.synchronize()
        h = out.cpu().numpy().astype(np.int64)
    stamps = h[4:4 + 64]
    gaps = np.diff(np.concatenate([[0], stamps]))
    return {"cta_group": 2 if pair else 1, "M": 256 if pair else 128, "N": n, "iters": int(h[3]),
            "completed": bool(h[2]), "issue_cycles_per_mma": float(h[0]) / iters,
            "complete_cycles_per_mma": float(h[1]) / iters,
            "first_issue_gaps": [int(x) for x in gaps[:16]],
            "gap_median_first8": float(np.median(gaps[1:9])), "gap_median_48_63": float(np.median(gaps[48:64]))}


def run_mma_probe(args) -> None:
    """--mma-probe: the issue probe for N=16 .. 256 on one CTA and N=128, 256 on
    a CTA pair; one JSON line."""
    import torch

    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sampler = ClockSampler(local)
    sampler.start()
    rows = [mma_issue_probe(torch, dev, False, n) for n in (16, 32, 64, 128, 256)]
    rows += [mma_issue_probe(torch, dev, True, n) for n in (128, 256)]
    clocks = sampler.stop()
    print(json.dumps({"mma_issue_probe": rows, "clocks": clocks}), flush=True)


def bench_workload(q, torch, c: dict, args, dev, stream, dist, rank: int) -> dict:
    """Every GPU measurement of one workload: the step, the GEMM call alone and
    the step's quantizer alone (each a CUDA graph of K steps, timed over
    args.repeats regions of exactly K steps; the median region is reported),
    and the two end-to-end routes through the public API with host buffers."""
    M, N, K = c["M"], c["N"], c["K"]
    G = c.get("g", 128)
    K_steps, repeats = args.steps, args.repeats

    # weights: generated once, packed on the GPU (timed separately), cloned into a pool
    w4ax = args.path == "w4ax"
    n8 = args.n8
    Wn = synth.weights(N, K, c["seed"])
    Xn = synth.activations(M, K, c["seed"] + rank)
    if w4ax:  # the channel permutation, applied upstream to both operands
        perm = outlier_first_permutation(c["seed"] + rank, K)
        Wn, Xn = np.ascontiguousarray(Wn[:, perm]), np.ascontiguousarray(Xn[:, perm])
    W = torch.from_numpy(Wn).to(dev)
    X = torch.from_numpy(Xn).to(dev)
    del Wn, Xn
    packed, s1 = q.qoq_pack_weights(W, g=G)
    torch.cuda.synchronize()
    pk_ev0, pk_ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pk_ev0.record()
    for _ in range(3):
        q.qoq_pack_weights(W, g=G, packed=packed, s1=s1)
    pk_ev1.record()
    torch.cuda.synchronize()
    pack_ms = pk_ev0.elapsed_time(pk_ev1) / 3
    del W

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ws_bytes = q.qoq_w4ax_workspace_bytes(M, N, K, G) if w4ax else q.qoq_gemm_workspace_bytes(M, N, K, G)
    act_row = q.qoq_w4ax_act_bytes(1, K, n8) if w4ax else K
    set_bytes = packed.numel() + 2 * N + 2 * M * K + M * act_row + 2 * M * (K // 128) + 2 * M * N + ws_bytes
    nsets = max(2, int(np.ceil(3 * l2 / set_bytes)))
    sets = []
    for _ in range(nsets):
        st_ = dict(packed=packed.clone(), s1=s1.clone(), X=X.clone(),
                   Y=torch.empty((M, N), dtype=torch.float16, device=dev),
                   ws=torch.zeros(ws_bytes, dtype=torch.uint8, device=dev))
        if w4ax:
            st_["Xa"] = torch.empty((M, act_row), dtype=torch.uint8, device=dev)
            st_["sxb"] = torch.empty((M, K // 128), dtype=torch.float16, device=dev)
        else:
            st_["Xq"] = torch.empty((M, K), dtype=torch.int8, device=dev)
            st_["sx"] = torch.empty(M, dtype=torch.float16, device=dev)
        sets.append(st_)
    del packed, s1

    # the step's activation quantizer: the per-token quantizer alone, or fused
    # with the preceding RMSNorm (gamma drawn once, eps 1e-6)
    norm_step = args.step == "norm"
    gamma = torch.from_numpy(np.random.default_rng(c["seed"]).uniform(0.5, 1.5, K).astype(np.float16)).to(dev)

    def quantize(s, X_src=None):
        src = s["X"] if X_src is None else X_src
        if w4ax:
            q.qoq_quant_act_w4ax(src, n8, Xa=s["Xa"], sxb=s["sxb"])
        elif norm_step:
            q.qoq_norm_quant_act(src, gamma, kind="rms", eps=1e-6, Xq=s["Xq"], sx=s["sx"])
        else:
            q.qoq_quant_act(src, Xq=s["Xq"], sx=s["sx"])

    gemm_call = q.qoq_w4a8_gemm_zero_folded if args.variant == "zero_folded" else q.qoq_w4a8_gemm

    def gemm(s, Y=None):
        if w4ax:
            q.qoq_w4ax_gemm(s["Xa"], s["sxb"], n8, s["packed"], s["s1"], K, N, g=G, Y=s["Y"] if Y is None else Y,
                            workspace=s["ws"])
        else:
            gemm_call(s["Xq"], s["sx"], s["packed"], s["s1"], N, g=G, Y=s["Y"] if Y is None else Y,
                      workspace=s["ws"])

    def steps_full(n: int):
        for i in range(n):
            s = sets[i % nsets]
            quantize(s)
            gemm(s)

    def steps_gemm(n: int):
        for i in range(n):
            gemm(sets[i % nsets])

    def steps_act(n: int):
        for i in range(n):
            quantize(sets[i % nsets])

    steps_full(max(3, args.warmup))
    torch.cuda.synchronize()
    st = q.qoq_last_device_status(sets[0]["ws"])
    if st != 0:
        raise SystemExit(f"device status after warm-up: {q.qoq_status_str(st)}")

    use_graph = not args.no_graph

    def timed(run_steps, name: str) -> tuple[list[float], bool]:
        """ms per step of each of `repeats` timed regions of exactly K steps."""
        graph = None
        run_steps(3)
        torch.cuda.synchronize()
        if use_graph:
            try:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    run_steps(K_steps)
                for _ in range(2):  # untimed warm replays
                    graph.replay()
                torch.cuda.synchronize()
            except Exception as exc:  # capture unsupported: time direct calls instead
                print(f"{name}: graph capture failed ({exc}); timing direct calls", file=sys.stderr)
                graph = None
                torch.cuda.synchronize()
        out = []
        for _ in range(repeats):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if dist:
                dist.barrier()
            torch.cuda.synchronize()
            e0.record(stream)
            if graph is not None:
                graph.replay()
            else:
                run_steps(K_steps)
            e1.record(stream)
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            out.append(e0.elapsed_time(e1) / K_steps)
        return out, graph is not None

    step_regions, step_graph = timed(steps_full, "step")
    gemm_regions, _ = timed(steps_gemm, "gemm")
    act_regions, _ = timed(steps_act, "quantizer")
    for s in sets:
        st = q.qoq_last_device_status(s["ws"])
        if st != 0:
            raise SystemExit(f"device status: {q.qoq_status_str(st)}")

    # ---- end to end through the public API with host buffers.  Route 1: each
    # step copies its X from pinned host memory and its Y back to pinned host
    # memory on copy streams, so that step i+1's upload and step i-1's
    # download overlap step i's kernels (events keep each set's reuse in order).
    Xh = torch.empty((M, K), dtype=torch.float16, pin_memory=True)
    Xh.copy_(X.cpu())
    Yh = [torch.empty((M, N), dtype=torch.float16, pin_memory=True) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = [{k: torch.cuda.Event() for k in ("x_ready", "x_free", "y_ready", "y_free")} for _ in range(nsets)]
    used = [False] * nsets

    def e2e_step(i: int):
        j = i % nsets
        s, e = sets[j], ev[j]
        comp = torch.cuda.current_stream()
        with torch.cuda.stream(h2d):
            if used[j]:
                h2d.wait_event(e["x_free"])
            s["X"].copy_(Xh, non_blocking=True)
            e["x_ready"].record(h2d)
        comp.wait_event(e["x_ready"])
        if used[j]:
            comp.wait_event(e["y_free"])
        quantize(s)
        e["x_free"].record(comp)
        gemm(s)
        e["y_ready"].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(e["y_ready"])
            Yh[i % 2].copy_(s["Y"], non_blocking=True)
            e["y_free"].record(d2h)
        used[j] = True

    def e2e_steps(n: int):
        comp = torch.cuda.current_stream()
        h2d.wait_stream(comp)  # fork the copy streams from the compute stream
        d2h.wait_stream(comp)
        for j in range(nsets):
            used[j] = False
        for i in range(n):
            e2e_step(i)
        comp.wait_stream(h2d)  # and join them back
        comp.wait_stream(d2h)

    # Route 2: the same calls with the host buffers themselves.  The quantizer
    # reads X in place from pinned host memory and the GEMM writes Y in place
    # into pinned host memory (unified addressing over the host link), so no
    # copy engine or cross-stream event sits between the kernels.
    Xh2 = [torch.empty((M, K), dtype=torch.float16, pin_memory=True) for _ in range(2)]
    for h in Xh2:
        h.copy_(Xh)

    def direct_steps(n: int):
        for i in range(n):
            s = sets[i % nsets]
            quantize(s, Xh2[i % 2])
            gemm(s, Y=Yh[i % 2])

    copy_regions, copy_graph = timed(e2e_steps, "e2e (copy engines)")
    direct_regions, direct_graph = timed(direct_steps, "e2e (host buffers in place)")
    for s in sets:
        st = q.qoq_last_device_status(s["ws"])
        if st != 0:
            raise SystemExit(f"device status: {q.qoq_status_str(st)}")

    med = statistics.median
    ms_per_step, gemm_ms, act_ms, copy_ms, direct_ms = max_over_ranks(
        dist, [med(step_regions), med(gemm_regions), med(act_regions), med(copy_regions), med(direct_regions)],
        dev)
    quant_name = "qoq_quant_act_w4ax" if w4ax else ("qoq_norm_quant_act" if norm_step else "qoq_quant_act")
    if direct_ms <= copy_ms:
        e2e_ms, e2e_how = direct_ms, (
            f"public API per step with host buffers: {quant_name} reads X in place from pinned host memory and "
            "qoq_w4a8_gemm writes Y in place into pinned host memory, every step (unified addressing over the "
            "host link, no staging copy); " + ("the K steps captured once in a CUDA graph and replayed"
                                               if direct_graph else "direct calls"))
    else:
        e2e_ms, e2e_how = copy_ms, (
            "public API per step; X uploaded from and Y read back to pinned host memory every step, on copy "
            "streams that overlap the neighbouring steps' kernels; " +
            ("the K steps captured once in a CUDA graph and replayed" if copy_graph else "direct calls"))
    out = dict(
        ms_per_step=ms_per_step, gemm_ms=gemm_ms, act_ms=act_ms, e2e_ms=e2e_ms, e2e_how=e2e_how,
        copy_ms=copy_ms, direct_ms=direct_ms, pack_ms=pack_ms, use_graph=step_graph,
        regions={"step": step_regions, "gemm": gemm_regions, "quantizer": act_regions},
        l2_policy=f"rotating pool of {nsets} buffer sets, {nsets * set_bytes / 1e6:.0f} MB "
                  f"(>= 3x L2 {l2 / 1e6:.0f} MB)",
        norm_step=norm_step, quant_name=quant_name, n8=n8 if w4ax else None)
    del sets
    torch.cuda.empty_cache()
    return out


def config_summary(c: dict, r: dict, args, world: int, peaks: dict, peak_src: str) -> dict:
    """The per-workload entry of the per_config block."""
    M, N, K = c["M"], c["N"], c["K"]
    G = c.get("g", 128)
    ops = 2.0 * M * N * K
    roof = roofline_of(M, N, K, G, r["gemm_ms"], args.steps, peaks, peak_src, r["n8"])
    roof_out = {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "peak_source")}
    if G == 128 and r["n8"] is None and args.variant == "direct":
        roof_out["traffic"], roof_out["traffic_source"] = recorded_traffic(c["name"])
        roof_out["algorithmic_bytes_per_launch"] = roof["algorithmic_bytes_per_launch"]
    return {
        "workload": c["name"], "M": M, "N": N, "K": K, "g": G,
        "value": job_tops(world, ops, r["ms_per_step"]), "unit": UNIT, "ms_per_step": r["ms_per_step"],
        "ms_per_launch": r["gemm_ms"], "roofline": roof_out,
        "gemm_tops": roof["tops_effective"], "gemm_gb_per_s": roof["gb_per_s_algorithmic"],
        "quantizer_ms": r["act_ms"],
        "e2e": {"value": job_tops(world, ops, r["e2e_ms"]), "unit": UNIT, "ms_per_step": r["e2e_ms"],
                "h2d_bytes_per_step": 2 * M * K, "d2h_bytes_per_step": 2 * M * N,
                "routes_ms_per_step": {"host_buffers_in_place": r["direct_ms"], "copy_engines": r["copy_ms"]}},
        "regions_ms_per_step": {k: [round(v, 6) for v in vs] for k, vs in r["regions"].items()},
    }


def run_ours(args, c: dict) -> None:
    import torch

    import w4a8_quantized_serving_gb300 as q

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    M, N, K = c["M"], c["N"], c["K"]
    G = c.get("g", 128)
    peaks, peak_src = load_peaks()

    sampler = ClockSampler(local)
    sampler.start()
    r = bench_workload(q, torch, c, args, dev, stream, dist, rank)
    clocks = sampler.stop()

    ops = 2.0 * M * N * K
    nbytes = algorithmic_bytes(M, N, K, G, r["n8"])
    value = job_tops(world, ops, r["ms_per_step"])
    roof = roofline_of(M, N, K, G, r["gemm_ms"], args.steps, peaks, peak_src, r["n8"])
    roof["traffic"] = args.traffic
    if roof["traffic"] is None:
        if r["n8"] is not None or args.variant != "direct":
            roof["traffic_source"] = "no ncu record for this path"
        elif G == 128:
            roof["traffic"], roof["traffic_source"] = recorded_traffic(c["name"])
        else:
            roof["traffic_source"] = f"no ncu record at g = {G}"
    roof["kernel"] = ("qoq_w4a8_gemm call (the GEMM kernel; + B-operand convert for M > 64), timed alone over "
                      "regions of K launches")
    # the step's activation quantizer alone: 2 bytes read and 1 written per
    # element, 2 per token for s_x, plus gamma (2K) when the norm is fused
    act_bytes = nbytes["act"] + (2 * K if r["norm_step"] else 0)
    act_gbs = act_bytes / (r["act_ms"] * 1e-3) / 1e9
    act_roof = {"kernel": r["quant_name"] + (" (RMSNorm)" if r["norm_step"] else ""),
                "bound": "hbm", "achieved": act_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": act_gbs / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": act_bytes,
                "ms_per_launch": r["act_ms"],
                "timing": "alone, same pool, " + ("CUDA graph" if r["use_graph"] else "direct")}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded splitmix64 Gaussians with outlier channels)",
        "config": config_dict(c, {
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2_policy": r["l2_policy"],
            "step": f"{r['quant_name']}{' (RMSNorm)' if r['norm_step'] else ''} + qoq_w4a8_gemm",
            "timing": (f"{args.repeats} timed regions of exactly K steps each "
                       f"({'a CUDA graph of K steps, replayed' if r['use_graph'] else 'direct launches'}); "
                       "median region reported"),
            "mma": "tcgen05 kind::f16, exact integer operands, fp32 TMEM folded to int32",
            "variant": ("qoq_w4ax_gemm (W4Ax: the outlier channels permuted into the first "
                        f"{r['n8']} 8-bit 128-channel block(s), 4-bit blocks elsewhere)" if r["n8"] is not None else
                        "qoq_w4a8_gemm_zero_folded (q4*s2 in the main loop, zero points' share subtracted in "
                        "the epilogue)" if args.variant == "zero_folded" else "qoq_w4a8_gemm")}),
        "regions_ms_per_step": {k: [round(v, 6) for v in vs] for k, vs in r["regions"].items()},
        "hbm_gb_per_s_step": world * nbytes["step"] / (r["ms_per_step"] * 1e-3) / 1e9,
        "roofline": roof,
        "act_roofline": act_roof,
        "e2e": {"value": job_tops(world, ops, r["e2e_ms"]), "unit": UNIT,
                "h2d_bytes_per_step": 2 * M * K, "d2h_bytes_per_step": 2 * M * N,
                "ms_per_step": r["e2e_ms"], "how": r["e2e_how"],
                "routes_ms_per_step": {"host_buffers_in_place": r["direct_ms"], "copy_engines": r["copy_ms"]}},
        "clocks": clocks,
        # inside one timed region of K steps: act-quant + GEMM per step, and
        # for M > 64 also the B-operand convert
        "gpu_launches": ((3 if r["n8"] is not None else (2 if M <= 64 else 3)) +
                         (1 if args.variant == "zero_folded" else 0)) * args.steps,
        "pack_ms": r["pack_ms"],
    }

    # a launch that only reads the GEMM call's algorithmic bytes, timed the
    # same way: the HBM time one launch of this size needs here
    if roof["bound"] == "hbm" and not args.no_floor:
        line["hbm_floor"] = hbm_floor_of(torch, dev, nbytes["gemm"], r["gemm_ms"], args, peaks)

    # the other workloads of the metric, measured the same way
    if not args.no_per_config:
        per = {}
        for idx, wc in synth.WORKLOADS.items():
            cc = dict(wc)
            if G != 128:
                cc["g"] = G
            if idx == args.config:
                entry = config_summary(cc, r, args, world, peaks, peak_src)
                entry["clocks"] = clocks
                if "hbm_floor" in line:
                    entry["hbm_floor"] = line["hbm_floor"]
            else:
                smp = ClockSampler(local)
                smp.start()
                rr = bench_workload(q, torch, cc, args, dev, stream, dist, rank)
                cl = smp.stop()
                entry = config_summary(cc, rr, args, world, peaks, peak_src)
                entry["clocks"] = cl
                if entry["roofline"]["bound"] == "hbm" and not args.no_floor:
                    entry["hbm_floor"] = hbm_floor_of(
                        torch, dev, algorithmic_bytes(cc["M"], cc["N"], cc["K"], cc.get("g", 128))["gemm"],
                        entry["ms_per_launch"], args, peaks)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                entry["cpu_baseline"] = oracle_step_timing(cc, args.cpu_budget_per_config, threads=0,
                                                           n_sample=oracle_sample_channels(cc, 2e10))
            per[cc["name"]] = entry
        line["per_config"] = per

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baselines(c, args.cpu_budget)
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed regions of exactly K steps each; the median is reported (default 5)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, help="workload index 0..4 (default 1)")
    ap.add_argument("--g", type=int, default=128,
                    help="level-2 group size: 32, 64 or a multiple of 128 dividing K (default 128, the pages' g128)")
    ap.add_argument("--step", choices=["quant", "norm"], default="quant",
                    help="activation quantizer of the step: qoq_quant_act (default) or qoq_norm_quant_act (RMSNorm fused)")
    ap.add_argument("--variant", choices=["direct", "zero_folded"], default="direct",
                    help="GEMM entry point: qoq_w4a8_gemm (default) or qoq_w4a8_gemm_zero_folded")
    ap.add_argument("--path", choices=["w4a8", "w4ax"], default="w4a8",
                    help="w4a8 (default): QoQ W4A8; w4ax: 4-bit activation blocks with 8-bit outlier blocks")
    ap.add_argument("--n8", type=int, default=1, help="W4Ax: leading 8-bit blocks (outlier channels permuted there)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle CPU timing (headline)")
    ap.add_argument("--cpu-budget-per-config", type=float, default=3.0,
                    help="seconds of oracle CPU timing per workload in per_config")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="measure the headline workload only")
    ap.add_argument("--no-graph", action="store_true", help="time direct launches instead of a CUDA graph")
    ap.add_argument("--no-floor", action="store_true",
                    help="skip the streaming-read chain timed beside HBM-bound workloads")
    ap.add_argument("--stream-sweep", action="store_true",
                    help="only time the streaming-read chain over launch sizes (one JSON line)")
    ap.add_argument("--mma-probe", action="store_true",
                    help="only run the tcgen05.mma issue-rate probe (one JSON line)")
    ap.add_argument("--stream-bytes", default="",
                    help="with --stream-sweep: only these launch sizes (comma-separated bytes)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per GEMM launch from an ncu capture of the current library, if known")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.repeats = max(1, args.repeats)
    c = dict(synth.WORKLOADS[args.config])
    if args.g != 128:
        c["g"] = args.g
    if args.mma_probe:
        run_mma_probe(args)
    elif args.stream_sweep:
        run_stream_sweep(args)
    elif args.impl == "reference":
        run_reference(args, c)
    else:
        run_ours(args, c)


if __name__ == "__main__":
    main()
