// act_quant.cu -- per-token symmetric int8 activation quantization.
//
// QServe talk write-up, "Precision Data Flow and Activation Quantization
// Fusion": every linear layer takes 8-bit activations (the write-up fuses the
// quantizer into the preceding LayerNorm; here it is a standalone kernel).
//   s_x[m]  = fp16_rn(fp32(max_k |X[m,k]|) / 127)        (IEEE fp32 divide)
//   Xq[m,k] = clamp(rint(X[m,k] / s_x[m]), -127, 127)      (fp32 divide, ties even;
//             computed without a divide by quant_bits, which gives the same codes)
// An all-zero row gets s_x = 0 and Xq = 0.
//
// Each token row is owned by T threads (T a power of two, 32..1024), each
// holding up to MAXV (4, 8 or 16, fixed at compile time) vectors of 8 fp16
// values in registers, so X is read from HBM once; the row max-abs is reduced
// with warp shuffles (and shared memory when T > 32).  CTAs have 128 threads
// when T <= 128 (several rows each) so that they fit beside the decode GEMM's
// persistent CTAs.  Both kernels chain by programmatic dependent launch: this
// kernel lets the dependent GEMM launch at once, and the GEMM streams its
// weights while this kernel runs; it is itself launched as a dependent, so it
// can sit resident beside a preceding GEMM and starts reading X the moment
// that kernel completes.  HBM bound: 2 bytes read and 1 byte written per
// element.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace qoq {
namespace {

// Running max-abs of fp16 values, kept in fp16 (exact) two lanes at a time.
__device__ __forceinline__ __half2 absmax8(uint4 v, __half2 m) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) m = __hmax2(m, __habs2(h[i]));
  return m;
}
__device__ __forceinline__ float hmax_float(__half2 m) {
  const float2 f = __half22float2(m);
  return fmaxf(f.x, f.y);
}

// int8 codes of 8 fp16 values (one 16-byte vector), packed little-endian.
template <bool CLAMP>
__device__ __forceinline__ uint2 quant8(uint4 v, float sf, float rf) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    b[2 * i] = quant_bits<CLAMP>(f.x, sf, rf, 127.0f);
    b[2 * i + 1] = quant_bits<CLAMP>(f.y, sf, rf, 127.0f);
  }
  // low byte of each biased pattern is the code byte
  const uint32_t lo = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
  const uint32_t hi = __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410);
  return make_uint2(lo, hi);
}

// Max-abs of a token row held by T threads (thread t has `amax` of its
// elements), combined over the row's warps through shared memory when T > 32.
__device__ __forceinline__ float row_absmax(float amax, int T, float* warp_max) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (T > 32) {  // combine the T/32 warps of this row
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    const int w0 = (threadIdx.x / T) * (T / 32);
    amax = 0.0f;
    for (int w = 0; w < T / 32; ++w) amax = fmaxf(amax, warp_max[w0 + w]);
  }
  return amax;
}

// Symmetric int8 quantization of a token row whose values this thread holds
// as fp16 vectors v[i] (vector t + i T of the row), given the row's max-abs:
// s_x = fp16_rn(amax / 127) (IEEE fp32 divide), Xq = clamp(rint(x / s_x), +-127).
template <int MAXV>
__device__ __forceinline__ void quant_row(const uint4 (&v)[MAXV], float amax, int row, int t, int T, int nvec,
                                          int K, int8_t* __restrict__ Xq, uint16_t* __restrict__ sx) {
  __half s = __float2half_rn(0.0f);
  if (amax > 0.0f) s = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float sf = __half2float(s);
  const float rf = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
  if (t == 0) sx[row] = __half_as_ushort(s);
  uint2* qr = reinterpret_cast<uint2*>(Xq + (size_t)row * K);
  if (sf >= kFp16MinNormal) {  // |x / s| <= 127 (1 + 2^-11): no clamp
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int idx = t + i * T;
      if (idx < nvec) qr[idx] = quant8<false>(v[i], sf, rf);
    }
  } else {  // subnormal or zero scale (zero gives zero codes)
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int idx = t + i * T;
      if (idx < nvec) qr[idx] = quant8<true>(v[i], sf, rf);
    }
  }
}

template <int MAXV>
__global__ void __launch_bounds__(1024) act_quant_kernel(const uint16_t* __restrict__ X,
                                                         int8_t* __restrict__ Xq,
                                                         uint16_t* __restrict__ sx, int M, int K,
                                                         int T) {
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the preceding kernel; Xq and s_x may still be read by it
  __shared__ float warp_max[32];
  const int rows_per_cta = blockDim.x / T;
  const int row = blockIdx.x * rows_per_cta + threadIdx.x / T;
  const int t = threadIdx.x % T;
  const int nvec = K / 8;
  const bool live = row < M;
  const uint4* xr = reinterpret_cast<const uint4*>(X + (size_t)(live ? row : 0) * K);
  uint4 v[MAXV];
  __half2 m2 = __float2half2_rn(0.0f);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = t + i * T;
    if (live && idx < nvec) {
      v[i] = __ldcg(xr + idx);  // L2: X may have been written by the preceding kernel
      m2 = absmax8(v[i], m2);
    }
  }
  const float amax = row_absmax(hmax_float(m2), T, warp_max);
  if (!live) return;
  quant_row<MAXV>(v, amax, row, t, T, nvec, K, Xq, sx);
}

// ------------------------------------------------------------------ norm --
// QServe talk write-up, "Precision Data Flow and Activation Quantization
// Fusion": the quantizer is fused into the preceding layer, such as
// LayerNorm, so its output goes to 8 bits without an fp16 round trip
// through HBM.  The row statistics are exact integers (x = a 2^-24 with a an
// integer for every fp16 x): S1 = sum a, S2 = sum a^2 (128 bits), so they do
// not depend on the reduction order.  Then, in fp32 with every operation
// rounded to nearest (fl32(S): the exact integer rounded once):
//   RMSNorm:   r = 1 / sqrt(fl32(S2) 2^-48 / K + eps),
//              y = fp16_rn(fl32(fl32(x r) gamma));
//   LayerNorm: mu = fl32(S1) 2^-24 / K,
//              r = 1 / sqrt(fl32(K S2 - S1^2) 2^-48 / K^2 + eps),
//              y = fp16_rn(fl32(fl32(fl32(fl32(x - mu) r) gamma) + beta));
// and y is quantized per token as by act_quant_kernel.  Every thread of a row
// computes r and mu from the same sums, so no broadcast is needed.

typedef unsigned __int128 u128;

// x = +-m 2^(s - 24) for a finite fp16 x: mantissa m < 2^11 and shift s <= 29,
// so a = x 2^24 = +-m 2^s and a^2 = m^2 2^(2s) < 2^80.
__device__ __forceinline__ uint32_t half_mantissa(uint32_t h, uint32_t& s, bool& neg) {
  const uint32_t e = (h >> 10) & 31, f = h & 1023;
  neg = (h >> 15) & 1;
  s = e == 0 ? 0 : e - 1;
  return e == 0 ? f : (f | 1024);
}

// Round-to-nearest-even conversion of a 128-bit unsigned integer (< 2^127) to fp32.
__device__ __forceinline__ float u128_to_float_rn(u128 v) {
  const uint64_t hi = (uint64_t)(v >> 64), lo = (uint64_t)v;
  if (hi == 0) return __ull2float_rn(lo);
  const int sh = 64 - __clzll((long long)hi);  // v >> sh has its top bit at 63
  uint64_t top = (uint64_t)(v >> sh);
  if ((v & (((u128)1 << sh) - 1)) != 0) top |= 1;  // sticky: bit 0 lies below the 24-bit rounding point
  return __fmul_rn(__ull2float_rn(top), __int_as_float((127 + sh) << 23));  // exact scaling by 2^sh
}

__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int off) {
  const uint64_t lo = __shfl_xor_sync(0xffffffffu, (unsigned long long)v, off);
  const uint64_t hi = __shfl_xor_sync(0xffffffffu, (unsigned long long)(v >> 64), off);
  return ((u128)hi << 64) | lo;
}

// At most 32 registers per thread for rows of up to 32768 channels (MAXV 4),
// like act_quant_kernel: a 128-thread CTA then fits, on every SM
// sub-partition, beside a decode GEMM CTA, so it becomes resident while that
// GEMM runs and starts the moment it completes.
template <int MAXV, bool LN>
__global__ void __launch_bounds__(1024, MAXV == 4 ? 2 : 1) norm_quant_kernel(const uint16_t* __restrict__ X,
                                                          const uint16_t* __restrict__ gamma,
                                                          const uint16_t* __restrict__ beta,
                                                          int8_t* __restrict__ Xq, uint16_t* __restrict__ sx,
                                                          int M, int K, int T, float eps) {
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the preceding kernel; Xq and s_x may still be read by it
  __shared__ float warp_max[32];
  __shared__ unsigned long long warp_s2[32][2];
  __shared__ long long warp_s1[32];
  const int rows_per_cta = blockDim.x / T;
  const int row = blockIdx.x * rows_per_cta + threadIdx.x / T;
  const int t = threadIdx.x % T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = K / 8;
  const bool live = row < M;
  const uint4* xr = reinterpret_cast<const uint4*>(X + (size_t)(live ? row : 0) * K);
  uint4 v[MAXV];
  // this thread's part of S2 as lo + hi 2^32: a^2 = m^2 2^(2s) goes to lo when
  // 2s < 32 (< 2^52) and to hi as m^2 2^(2s-32) otherwise (< 2^48); at most
  // 128 terms each, so neither 64-bit sum can wrap
  uint64_t s2lo = 0, s2hi = 0;
  long long s1 = 0;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = t + i * T;
    if (live && idx < nvec) {
      v[i] = __ldcg(xr + idx);  // L2: X may have been written by the preceding kernel
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        bool neg;
        uint32_t sh;
        const uint32_t mnt = half_mantissa((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, sh, neg);
        const uint64_t sq = (uint64_t)(mnt * mnt);
        if (sh >= 16)
          s2hi += sq << (2 * sh - 32);
        else
          s2lo += sq << (2 * sh);
        if (LN) {
          const long long a = (long long)((uint64_t)mnt << sh);
          s1 += neg ? -a : a;
        }
      }
    }
  }
  u128 s2 = ((u128)s2hi << 32) + s2lo;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    s2 += shfl_xor_u128(s2, off);
    if (LN) s1 += __shfl_xor_sync(0xffffffffu, s1, off);
  }
  if (T > 32) {  // the row's warps, summed in the same order by every thread
    if (lane == 0) {
      warp_s2[warp][0] = (unsigned long long)s2;
      warp_s2[warp][1] = (unsigned long long)(s2 >> 64);
      warp_s1[warp] = s1;
    }
    __syncthreads();
    const int w0 = (threadIdx.x / T) * (T / 32);
    s2 = 0;
    s1 = 0;
    for (int w = 0; w < T / 32; ++w) {
      s2 += ((u128)warp_s2[w0 + w][1] << 64) | warp_s2[w0 + w][0];
      s1 += warp_s1[w0 + w];
    }
  }

  float spread, mu = 0.0f;  // mean square (RMSNorm) or variance (LayerNorm)
  if (LN) {
    const u128 a1 = (u128)(unsigned long long)(s1 < 0 ? -s1 : s1);
    const u128 var_num = (u128)(unsigned)K * s2 - a1 * a1;  // K S2 - S1^2 >= 0, exact
    spread = __fdiv_rn(__fmul_rn(u128_to_float_rn(var_num), 0x1p-48f), (float)K * (float)K);
    mu = __fdiv_rn(__fmul_rn(__ll2float_rn(s1), 0x1p-24f), (float)K);
  } else {
    spread = __fdiv_rn(__fmul_rn(u128_to_float_rn(s2), 0x1p-48f), (float)K);
  }
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(spread, eps)));

  // y in place of x (fp16), and its max-abs
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = t + i * T;
    if (live && idx < nvec) {
      const uint4 gv = __ldcg(reinterpret_cast<const uint4*>(gamma) + idx);
      uint4 bv = make_uint4(0, 0, 0, 0);
      if (LN) bv = __ldcg(reinterpret_cast<const uint4*>(beta) + idx);
      __half* h = reinterpret_cast<__half*>(&v[i]);
      const __half* gh = reinterpret_cast<const __half*>(&gv);
      const __half* bh = reinterpret_cast<const __half*>(&bv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float y = __half2float(h[j]);
        if (LN) y = __fsub_rn(y, mu);
        y = __fmul_rn(__fmul_rn(y, r), __half2float(gh[j]));
        if (LN) y = __fadd_rn(y, __half2float(bh[j]));
        h[j] = __float2half_rn(y);
        amax = fmaxf(amax, fabsf(__half2float(h[j])));
      }
    }
  }
  amax = row_absmax(amax, T, warp_max);
  if (!live) return;
  quant_row<MAXV>(v, amax, row, t, T, nvec, K, Xq, sx);
}

}  // namespace

namespace {

// Threads per token row: a power of two, ~4 vectors of 8 values each (latency),
// at most 16 (T = 1024 for K up to 131072).
struct RowLayout {
  int T, threads, grid, vpt;
};

// vmax: vectors per thread to aim for.  4 keeps a CTA at 32 registers per
// thread, so that it fits beside a decode GEMM CTA (M <= 64); above that the
// quantizer never shares an SM with the GEMM, and 8 per thread (fewer threads
// per row, more loads in flight each) is faster: M=4096, K=8192 23.5 -> 19.2
// us; M=256, K=14336 5.7 -> 4.5 us.
RowLayout row_layout(int M, int K, int vmax = 4) {
  const int nvec = K / 8;
  RowLayout L;
  L.T = 32;
  while (L.T * vmax < nvec && L.T < 1024) L.T *= 2;
  L.threads = L.T < 128 ? 128 : L.T;
  const int rows_per_cta = L.threads / L.T;
  L.grid = (M + rows_per_cta - 1) / rows_per_cta;
  L.vpt = (nvec + L.T - 1) / L.T;  // <= 4 unless T = 1024; <= 16 for K <= 131072
  return L;
}

cudaLaunchConfig_t row_config(const RowLayout& L, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(L.threads);
  cfg.stream = s;
  attr[0] = pdl_attr();
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <bool LN>
cudaError_t launch_norm_kind(const RowLayout& L, cudaLaunchConfig_t& cfg, int M, int K, float eps, const uint16_t* X,
                             const uint16_t* gamma, const uint16_t* beta, int8_t* Xq, uint16_t* sx) {
  if (L.vpt <= 4) return cudaLaunchKernelEx(&cfg, norm_quant_kernel<4, LN>, X, gamma, beta, Xq, sx, M, K, L.T, eps);
  if (L.vpt <= 8) return cudaLaunchKernelEx(&cfg, norm_quant_kernel<8, LN>, X, gamma, beta, Xq, sx, M, K, L.T, eps);
  if (L.vpt <= 16) return cudaLaunchKernelEx(&cfg, norm_quant_kernel<16, LN>, X, gamma, beta, Xq, sx, M, K, L.T, eps);
  return cudaErrorInvalidValue;
}

// ----------------------------------------------------------------- W4Ax --
// COMET explainer, FMPQ: activations in 128-channel blocks, the outlier
// channels clustered (by a channel permutation) into the n8 leading blocks,
// which stay at 8 bits, every other block at 4 bits; one symmetric scale per
// (token, block):
//   s = fp16_rn(fp32(max |x|) / q) (IEEE fp32 divide), code = clamp(rint(x / s), +-q),
// q = 127 for 8-bit blocks, 7 for 4-bit blocks.  Storage per token row, blocks
// in order: an 8-bit block is 128 int8 codes, a 4-bit block 64 bytes with the
// code of channel 2i in the low nibble of byte i and that of 2i + 1 in the
// high nibble (two's complement).  One warp per (row, pair of blocks): each
// half-warp owns a block, 8 channels per lane, and reduces its max-abs with
// shuffles inside the half.
__global__ void __launch_bounds__(256) act_quant_w4ax_kernel(const uint16_t* __restrict__ X, uint8_t* __restrict__ Xa,
                                                             uint16_t* __restrict__ sxb, int M, int K, int n8) {
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the preceding kernel; Xa and the scales may still be read by it
  const int G = K / 128;
  const int pairs = (G + 1) / 2;
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (long long)M * pairs) return;  // whole warps
  const int lane = threadIdx.x & 31, l = lane & 15;
  const int m = (int)(wid / pairs);
  const int b = 2 * (int)(wid % pairs) + (lane >> 4);
  const bool live = b < G;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (live) v = __ldcg(reinterpret_cast<const uint4*>(X + (size_t)m * K + (size_t)b * 128) + l);
  float amax = hmax_float(absmax8(v, __float2half2_rn(0.0f)));
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (!live) return;
  const bool eight = b < n8;
  const float q = eight ? 127.0f : 7.0f;
  __half sh = __float2half_rn(0.0f);
  if (amax > 0.0f) sh = __float2half_rn(__fdiv_rn(amax, q));
  const float sf = __half2float(sh);
  const float rf = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
  if (l == 0) sxb[(size_t)m * G + b] = __half_as_ushort(sh);
  const __half* h = reinterpret_cast<const __half*>(&v);
  uint32_t c[8];  // biased patterns: the low byte (nibble) is the code's 8-bit (4-bit) two's complement
  if (sf >= kFp16MinNormal) {  // |x / s| <= q (1 + 2^-11): no clamp
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = quant_bits<false>(__half2float(h[i]), sf, rf, q);
  } else {  // subnormal or zero scale (zero gives zero codes)
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = quant_bits<true>(__half2float(h[i]), sf, rf, q);
  }
  const size_t row_bytes = (size_t)128 * n8 + (size_t)64 * (G - n8);
  uint8_t* row = Xa + (size_t)m * row_bytes;
  if (eight) {
    uint2 out;
    out.x = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
    out.y = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
    *reinterpret_cast<uint2*>(row + (size_t)128 * b + 8 * l) = out;
  } else {
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) out |= (c[i] & 0xfu) << (4 * i);
    *reinterpret_cast<uint32_t*>(row + (size_t)128 * n8 + (size_t)64 * (b - n8) + 4 * l) = out;
  }
}

}  // namespace

cudaError_t launch_act_quant(int M, int K, const uint16_t* X, int8_t* Xq, uint16_t* sx,
                             cudaStream_t s) {
  const RowLayout L = row_layout(M, K, M > 64 ? 8 : 4);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = row_config(L, s, attr);
  if (L.vpt <= 4) return cudaLaunchKernelEx(&cfg, act_quant_kernel<4>, X, Xq, sx, M, K, L.T);
  if (L.vpt <= 8) return cudaLaunchKernelEx(&cfg, act_quant_kernel<8>, X, Xq, sx, M, K, L.T);
  if (L.vpt <= 16) return cudaLaunchKernelEx(&cfg, act_quant_kernel<16>, X, Xq, sx, M, K, L.T);
  return cudaErrorInvalidValue;
}

cudaError_t launch_norm_quant(int M, int K, int kind, float eps, const uint16_t* X, const uint16_t* gamma,
                              const uint16_t* beta, int8_t* Xq, uint16_t* sx, cudaStream_t s) {
  const RowLayout L = row_layout(M, K);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = row_config(L, s, attr);
  return kind == 1 ? launch_norm_kind<true>(L, cfg, M, K, eps, X, gamma, beta, Xq, sx)
                   : launch_norm_kind<false>(L, cfg, M, K, eps, X, gamma, beta, Xq, sx);
}

cudaError_t launch_act_quant_w4ax(int M, int K, int n8, const uint16_t* X, uint8_t* Xa, uint16_t* sxb,
                                  cudaStream_t s) {
  const long long warps = (long long)M * ((K / 128 + 1) / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, act_quant_w4ax_kernel, X, Xa, sxb, M, K, n8);
}

}  // namespace qoq
