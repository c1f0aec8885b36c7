"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding (which calls the C ABI) and the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np

import oracle
from w4a8_quantized_serving_gb300 import synth

# fp16 Y tolerance: |Y - Y_ref| <= 2e-3 |Y_ref|  or  |Y - Y_ref| <= 1e-2
Y_RTOL = 2e-3
Y_ATOL = 1e-2


def torch():
    import torch as t

    return t


def to_dev_f16(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).cuda()


def f16_bits(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def gpu_layer(W: np.ndarray, X: np.ndarray, want_acc: bool = True, ws=None, g: int = 128):
    """Run pack -> quant_act -> gemm on the GPU at group size g. Returns the tensors."""
    import w4a8_quantized_serving_gb300 as q

    t = torch()
    Wd, Xd = to_dev_f16(W), to_dev_f16(X)
    N, K = W.shape
    M = X.shape[0]
    packed, s1 = q.qoq_pack_weights(Wd, g=g)
    Xq, sx = q.qoq_quant_act(Xd)
    acc = t.empty((M, N), dtype=t.int32, device="cuda") if want_acc else None
    if ws is None:
        ws = t.zeros(q.qoq_gemm_workspace_bytes(M, N, K, g), dtype=t.uint8, device="cuda")
    Y = q.qoq_w4a8_gemm(Xq, sx, packed, s1, N, g=g, acc_debug=acc, workspace=ws)
    status = q.qoq_last_device_status(ws)
    assert status == 0, f"device status {status}"
    t.cuda.synchronize()
    return dict(packed=packed, s1=s1, Xq=Xq, sx=sx, Y=Y, acc=acc, ws=ws)


def oracle_layer(W: np.ndarray, X: np.ndarray, full_gemm: bool = True, g: int = 128):
    r = oracle.weight_quant(synth.bits(W), g)
    Xq, sx = oracle.act_quant(synth.bits(X))
    r["Xq"], r["sx"] = Xq, sx
    if full_gemm:
        acc, Y = oracle.gemm(Xq, sx, r["q4"], r["s2"], r["z"], r["s1"], g)
        r["acc"], r["Y"] = acc, Y
    return r


def y_close(Y_bits: np.ndarray, Yref_bits: np.ndarray):
    """Element-wise fp16 tolerance; returns (ok, max_rel, max_abs)."""
    Y = Y_bits.view(np.float16).astype(np.float64)
    R = Yref_bits.view(np.float16).astype(np.float64)
    same = Y_bits == Yref_bits  # identical values, including infinities
    with np.errstate(invalid="ignore"):
        d = np.where(same, 0.0, np.abs(Y - R))
    ok = same | (d <= Y_RTOL * np.abs(R)) | (d <= Y_ATOL)
    rel = d / np.maximum(np.abs(R), 1e-30)
    return bool(ok.all()), float(rel[np.abs(R) > Y_ATOL].max(initial=0.0)), float(d.max(initial=0.0))


def check_weights(q_mod, g, o, N, K, group: int = 128):
    q4, s2, z = q_mod.qoq_unpack_weights_debug(g["packed"], N, K, group)
    assert np.array_equal(q4.cpu().numpy(), o["q4"]), "q4 mismatch"
    assert np.array_equal(s2.cpu().numpy(), o["s2"]), "s2 mismatch"
    assert np.array_equal(z.cpu().numpy(), o["z"]), "z mismatch"
    assert np.array_equal(f16_bits(g["s1"]), o["s1"]), "s1 mismatch"


def check_acts(g, o):
    assert np.array_equal(g["Xq"].cpu().numpy(), o["Xq"]), "Xq mismatch"
    assert np.array_equal(f16_bits(g["sx"]), o["sx"]), "sx mismatch"


def pack_reference_layout(q4: np.ndarray, s2: np.ndarray, z: np.ndarray, g: int = 128) -> np.ndarray:
    """The packed blob rebuilt on the host from logical codes, following the
    layout written in include/qoq.h (test-side, independent of the kernels):
    per 128-channel k-tile, S = max(1, 128 / g) sets of s2[128] + z[128], then
    the four code chunks."""
    N, K = q4.shape
    G = K // 128
    S = max(1, 128 // g)
    nib = 256 * S
    out = np.zeros((N // 128, G, nib + 8192), np.uint8)
    for nt in range(N // 128):
        rows = slice(nt * 128, nt * 128 + 128)
        for j in range(G):
            tile = out[nt, j]
            for u in range(S):
                grp = (j * 128 + u * g) // g  # the group of the set's first channel
                tile[256 * u:256 * u + 128] = s2[rows, grp]
                tile[256 * u + 128:256 * u + 256] = z[rows, grp]
            codes = q4[rows, j * 128:(j + 1) * 128].astype(np.uint32)  # [128 rows][128 k]
            for c in range(4):
                for w in range(4):
                    word = np.zeros(128, np.uint32)
                    for i in range(4):
                        word |= codes[:, 32 * c + 8 * w + 2 * i] << (4 * i)
                        word |= codes[:, 32 * c + 8 * w + 2 * i + 1] << (16 + 4 * i)
                    off = nib + c * 2048
                    blk = tile[off:off + 2048].reshape(128, 16)
                    blk[:, 4 * w:4 * w + 4] = word.view(np.uint8).reshape(128, 4)
    return out.reshape(-1)
