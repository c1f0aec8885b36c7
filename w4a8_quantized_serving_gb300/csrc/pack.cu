// pack.cu -- offline weight preparation: progressive group quantization and
// the compute-aware packed layout, plus its inverse for testing.
//
// QServe talk write-up, "Progressive Group Quantization for W4A8 GEMM", and
// lecture 15 notes, section 15.6 (two-level scales):
//   level 1 (per output channel n, protective range):
//     s1[n]  = fp16_rn(fp32(max_k |W[n,k]|) / 119)        (IEEE fp32 divide)
//     Q8     = clamp(rint(W / s1), -119, 119)               (fp32 divide, ties even)
//   level 2 (per group of g channels, asymmetric uint4, exact integers):
//     lo = min(0, min Q8), hi = max(0, max Q8)
//     s2 = max(1, ceil((hi - lo) / 15)),  z = rne(-lo / s2)
//     q4 = clamp(rne(Q8 / s2) + z, 0, 15)
// QServe "compute-aware weight reordering": the codes are stored in the order
// and grouping the GEMM's dequant threads consume them (layout in qoq.h).
//
// One warp per output row; lane l owns channels 4l .. 4l+3 of each 128-channel
// k-tile.  For g <= 128 a group is g / 4 consecutive lanes of a k-tile; for
// g > 128 a group spans g / 128 k-tiles, whose codes are computed twice (once
// for the group's range, once to store them).
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace qoq {
namespace {

constexpr int kRowsPerBlock = 8;

// a / b rounded to nearest with ties to even, for b > 0 (exact integers):
// round-half-up as floor((2a + b) / 2b), then step back on an exact tie that
// landed on an odd quotient.
__device__ __forceinline__ int div_round_even(int a, int b) {
  const int num = 2 * a + b, den = 2 * b;
  int q = num >= 0 ? num / den : -((den - 1 - num) / den);
  if (q * den == num && (q & 1)) q -= 1;
  return q;
}

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Bit position of channel kk (0..7) inside its 32-bit word: even channels in
// the low half-word, odd channels in the high half-word, 4 bits apart.
__device__ __forceinline__ int nibble_shift(int kk) { return (kk & 1) * 16 + (kk >> 1) * 4; }

// Level-1 codes of channels 4 lane .. 4 lane + 3 of k-tile t of one row.
__device__ __forceinline__ void level1_codes(const uint16_t* wr, int t, int lane, float s1f, float r1f, int (&q8)[4]) {
  uint2 raw = __ldg(reinterpret_cast<const uint2*>(wr + t * kGroup + 4 * lane));
  const __half* h = reinterpret_cast<const __half*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    q8[i] = quant_code(__half2float(h[i]), s1f, r1f, 119.0f);  // 0 where s1 = 0
  }
}

// Level 2 for the lane's 4 channels with the group's (s2, z): the codes go
// into k-tile `tile` (layout of include/qoq.h); lane `writer` of the group
// writes s2 and z into scale set u.
__device__ __forceinline__ void store_codes(uint8_t* tile, int nib, int r, int lane, const int (&q8)[4], int s2, int z,
                                            int u, bool writer) {
  // channels 4*lane .. 4*lane+3 sit in word (lane / 2), positions 4*(lane & 1) + i
  uint32_t part = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q4 = min(15, max(0, div_round_even(q8[i], s2) + z));
    part |= (uint32_t)q4 << nibble_shift(4 * (lane & 1) + i);
  }
  const uint32_t word = part | __shfl_xor_sync(0xffffffffu, part, 1);
  if ((lane & 1) == 0) {
    const int wd = lane >> 1;  // word 0..15 of the row's 64 bytes
    const int chunk = wd >> 2, wi = wd & 3;
    *reinterpret_cast<uint32_t*>(tile + nib + chunk * kWChunkBytes + r * 16 + wi * 4) = word;
  }
  if (writer) {
    tile[u * 256 + r] = (uint8_t)s2;
    tile[u * 256 + 128 + r] = (uint8_t)z;
  }
}

__global__ void __launch_bounds__(kRowsPerBlock * 32) pack_kernel(const uint16_t* __restrict__ W,
                                                                  uint8_t* __restrict__ packed,
                                                                  uint16_t* __restrict__ s1out,
                                                                  int N, int K, int g) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kRowsPerBlock + warp;
  if (n >= N) return;
  const uint16_t* wr = W + (size_t)n * K;
  const int KT = K / kGroup;  // k-tiles per row
  const int gpt = g >= kGroup ? 1 : kGroup / g;
  const int tile_bytes = w_tile_bytes(gpt), nib = w_nib_offset(gpt);

  // level 1: row max-abs -> s1
  float amax = 0.0f;
  for (int k = lane * 8; k < K; k += 256) {
    uint4 raw = __ldg(reinterpret_cast<const uint4*>(wr + k));
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __half22float2(__habs2(h[i]));
      amax = fmaxf(amax, fmaxf(f.x, f.y));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  __half s1 = __float2half_rn(0.0f);
  if (amax > 0.0f) s1 = __float2half_rn(__fdiv_rn(amax, 119.0f));
  const float s1f = __half2float(s1);
  const float r1f = s1f != 0.0f ? __frcp_rn(s1f) : 0.0f;
  if (lane == 0) s1out[n] = __half_as_ushort(s1);

  const int nt = n / kTileN, r = n % kTileN;
  uint8_t* const row_tiles = packed + (size_t)nt * KT * tile_bytes;
  int q8[4];
  if (g <= kGroup) {
    // level 2, g <= 128: groups of g / 4 lanes inside each k-tile
    const int width = g / 4, u = lane / width;
    for (int t = 0; t < KT; ++t) {
      level1_codes(wr, t, lane, s1f, r1f, q8);
      int lo = min(0, min(min(q8[0], q8[1]), min(q8[2], q8[3])));
      int hi = max(0, max(max(q8[0], q8[1]), max(q8[2], q8[3])));
      for (int off = width / 2; off > 0; off >>= 1) {  // stays inside the lane's group
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
      }
      const int s2 = max(1, (hi - lo + 14) / 15);
      const int z = div_round_even(-lo, s2);
      store_codes(row_tiles + (size_t)t * tile_bytes, nib, r, lane, q8, s2, z, u, lane % width == 0);
    }
  } else {
    // level 2, g > 128: the group's range over its g / 128 k-tiles first
    const int R = g / kGroup;
    for (int t0 = 0; t0 < KT; t0 += R) {
      int lo = 0, hi = 0;
      for (int t = t0; t < t0 + R; ++t) {
        level1_codes(wr, t, lane, s1f, r1f, q8);
        lo = min(lo, min(min(q8[0], q8[1]), min(q8[2], q8[3])));
        hi = max(hi, max(max(q8[0], q8[1]), max(q8[2], q8[3])));
      }
      lo = warp_min(lo);
      hi = warp_max(hi);
      const int s2 = max(1, (hi - lo + 14) / 15);
      const int z = div_round_even(-lo, s2);
      for (int t = t0; t < t0 + R; ++t) {  // the same level-1 codes again (same arithmetic)
        level1_codes(wr, t, lane, s1f, r1f, q8);
        store_codes(row_tiles + (size_t)t * tile_bytes, nib, r, lane, q8, s2, z, 0, lane == 0);
      }
    }
  }
}

// Inverse of the layout: one thread per (row, k-tile).  Writes the k-tile's
// 128 codes and the (s2, z) of every group that starts in it.
__global__ void unpack_kernel(const uint8_t* __restrict__ packed, uint8_t* __restrict__ q4,
                              uint8_t* __restrict__ s2, uint8_t* __restrict__ z, int N, int K, int g) {
  const int KT = K / kGroup, NG = K / g;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)N * KT) return;
  const int n = (int)(idx / KT), t = (int)(idx % KT);
  const int gpt = g >= kGroup ? 1 : kGroup / g;
  const int nt = n / kTileN, r = n % kTileN;
  const uint8_t* tile = packed + ((size_t)nt * KT + t) * w_tile_bytes(gpt);
  if (g <= kGroup) {
    for (int u = 0; u < gpt; ++u) {
      const size_t j = (size_t)n * NG + (size_t)t * gpt + u;
      s2[j] = tile[u * 256 + r];
      z[j] = tile[u * 256 + 128 + r];
    }
  } else if (t % (g / kGroup) == 0) {
    const size_t j = (size_t)n * NG + (size_t)(t / (g / kGroup));
    s2[j] = tile[r];
    z[j] = tile[128 + r];
  }
  uint8_t* out = q4 + (size_t)n * K + (size_t)t * kGroup;
  for (int c = 0; c < 4; ++c) {
    const uint32_t* words = reinterpret_cast<const uint32_t*>(tile + w_nib_offset(gpt) + c * kWChunkBytes + r * 16);
    for (int w = 0; w < 4; ++w) {
      const uint32_t v = words[w];
      for (int kk = 0; kk < 8; ++kk) out[c * 32 + w * 8 + kk] = (v >> nibble_shift(kk)) & 0xF;
    }
  }
}

}  // namespace

cudaError_t launch_pack(int N, int K, int g, const uint16_t* W, uint8_t* packed, uint16_t* s1,
                        cudaStream_t s) {
  dim3 grid((N + kRowsPerBlock - 1) / kRowsPerBlock);
  pack_kernel<<<grid, kRowsPerBlock * 32, 0, s>>>(W, packed, s1, N, K, g);
  return cudaGetLastError();
}

cudaError_t launch_unpack(int N, int K, int g, const uint8_t* packed, uint8_t* q4, uint8_t* s2, uint8_t* z,
                          cudaStream_t s) {
  const long long total = (long long)N * (K / kGroup);
  const int threads = 256;
  dim3 grid((unsigned)((total + threads - 1) / threads));
  unpack_kernel<<<grid, threads, 0, s>>>(packed, q4, s2, z, N, K, g);
  return cudaGetLastError();
}

}  // namespace qoq
