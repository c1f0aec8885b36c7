// pack.cu -- offline weight preparation: progressive group quantization and
// the compute-aware packed layout, plus its inverse for testing.
//
// QServe talk write-up, "Progressive Group Quantization for W4A8 GEMM", and
// lecture 15 notes, section 15.6 (two-level scales):
//   level 1 (per output channel n, protective range):
//     s1[n]  = fp16_rn(fp32(max_k |W[n,k]|) / 119)        (IEEE fp32 divide)
//     Q8     = clamp(rint(W / s1), -119, 119)               (fp32 divide, ties even)
//   level 2 (per 128-channel group, asymmetric uint4, exact integers):
//     lo = min(0, min Q8), hi = max(0, max Q8)
//     s2 = max(1, ceil((hi - lo) / 15)),  z = rne(-lo / s2)
//     q4 = clamp(rne(Q8 / s2) + z, 0, 15)
// QServe "compute-aware weight reordering": the codes are stored in the order
// and grouping the GEMM's dequant threads consume them (layout in qoq.h).
//
// One warp per output row; lane l owns channels 4l .. 4l+3 of each group.
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

__global__ void __launch_bounds__(kRowsPerBlock * 32) pack_kernel(const uint16_t* __restrict__ W,
                                                                  uint8_t* __restrict__ packed,
                                                                  uint16_t* __restrict__ s1out,
                                                                  int N, int K) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kRowsPerBlock + warp;
  if (n >= N) return;
  const uint16_t* wr = W + (size_t)n * K;
  const int G = K / kGroup;

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
  for (int j = 0; j < G; ++j) {
    uint8_t* tile = packed + ((size_t)nt * G + j) * kWTileBytes;
    uint2 raw = __ldg(reinterpret_cast<const uint2*>(wr + j * kGroup + 4 * lane));
    const __half* h = reinterpret_cast<const __half*>(&raw);
    int q8[4];
    int lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int q = 0;
      if (s1f != 0.0f) q = (int)fminf(119.0f, fmaxf(-119.0f, rint_div_fp16(__half2float(h[i]), s1f, r1f)));
      q8[i] = q;
      lo = min(lo, q);
      hi = max(hi, q);
    }
    lo = warp_min(lo);
    hi = warp_max(hi);
    const int s2 = max(1, (hi - lo + 14) / 15);
    const int z = div_round_even(-lo, s2);

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
      *reinterpret_cast<uint32_t*>(tile + kWNibOffset + chunk * kWChunkBytes + r * 16 + wi * 4) = word;
    }
    if (lane == 0) {
      tile[r] = (uint8_t)s2;
      tile[128 + r] = (uint8_t)z;
    }
  }
}

// Inverse of the layout: one thread per (row, group).
__global__ void unpack_kernel(const uint8_t* __restrict__ packed, uint8_t* __restrict__ q4,
                              uint8_t* __restrict__ s2, uint8_t* __restrict__ z, int N, int K) {
  const int G = K / kGroup;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)N * G) return;
  const int n = (int)(idx / G), j = (int)(idx % G);
  const int nt = n / kTileN, r = n % kTileN;
  const uint8_t* tile = packed + ((size_t)nt * G + j) * kWTileBytes;
  s2[(size_t)n * G + j] = tile[r];
  z[(size_t)n * G + j] = tile[128 + r];
  uint8_t* out = q4 + (size_t)n * K + (size_t)j * kGroup;
  for (int c = 0; c < 4; ++c) {
    const uint32_t* words = reinterpret_cast<const uint32_t*>(tile + kWNibOffset + c * kWChunkBytes + r * 16);
    for (int w = 0; w < 4; ++w) {
      const uint32_t v = words[w];
      for (int kk = 0; kk < 8; ++kk) out[c * 32 + w * 8 + kk] = (v >> nibble_shift(kk)) & 0xF;
    }
  }
}

}  // namespace

cudaError_t launch_pack(int N, int K, const uint16_t* W, uint8_t* packed, uint16_t* s1,
                        cudaStream_t s) {
  dim3 grid((N + kRowsPerBlock - 1) / kRowsPerBlock);
  pack_kernel<<<grid, kRowsPerBlock * 32, 0, s>>>(W, packed, s1, N, K);
  return cudaGetLastError();
}

cudaError_t launch_unpack(int N, int K, const uint8_t* packed, uint8_t* q4, uint8_t* s2, uint8_t* z,
                          cudaStream_t s) {
  const long long total = (long long)N * (K / kGroup);
  const int threads = 256;
  dim3 grid((unsigned)((total + threads - 1) / threads));
  unpack_kernel<<<grid, threads, 0, s>>>(packed, q4, s2, z, N, K);
  return cudaGetLastError();
}

}  // namespace qoq
