// act_quant.cu -- per-token symmetric int8 activation quantization.
//
// QServe talk write-up, "Precision Data Flow and Activation Quantization
// Fusion": every linear layer takes 8-bit activations (the write-up fuses the
// quantizer into the preceding LayerNorm; here it is a standalone kernel).
//   s_x[m]  = fp16_rn(fp32(max_k |X[m,k]|) / 127)        (IEEE fp32 divide)
//   Xq[m,k] = clamp(rint(X[m,k] / s_x[m]), -127, 127)      (fp32 divide, ties even)
// An all-zero row gets s_x = 0 and Xq = 0.
//
// One warp per token row: 16-byte vector loads, a 5-step shuffle max, then a
// second sweep (served from L1/L2) that writes 8 codes per 8-byte store.
// The work is HBM bound: 2 bytes read and 1 byte written per element.
#include <cuda_fp16.h>

#include "internal.h"

namespace qoq {
namespace {

constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ float absmax8(uint4 v, float m) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(__habs2(h[i]));
    m = fmaxf(m, fmaxf(f.x, f.y));
  }
  return m;
}

__device__ __forceinline__ int quant1(float x, float sf) {
  int q = __float2int_rn(__fdiv_rn(x, sf));
  return min(127, max(-127, q));
}

__global__ void __launch_bounds__(kRowsPerBlock * 32) act_quant_kernel(const uint16_t* __restrict__ X,
                                                                       int8_t* __restrict__ Xq,
                                                                       uint16_t* __restrict__ sx,
                                                                       int M, int K) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  if (row >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(X + (size_t)row * K);
  const int nvec = K / 8;

  float amax = 0.0f;
  for (int v = lane; v < nvec; v += 32) amax = absmax8(__ldg(xr + v), amax);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

  __half s = __float2half_rn(0.0f);
  if (amax > 0.0f) s = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float sf = __half2float(s);
  if (lane == 0) sx[row] = __half_as_ushort(s);

  uint2* qr = reinterpret_cast<uint2*>(Xq + (size_t)row * K);
  for (int v = lane; v < nvec; v += 32) {
    uint4 raw = __ldg(xr + v);
    const __half* h = reinterpret_cast<const __half*>(&raw);
    uint32_t lo = 0, hi = 0;
    if (sf != 0.0f) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        lo |= (uint32_t)(quant1(__half2float(h[i]), sf) & 0xff) << (8 * i);
        hi |= (uint32_t)(quant1(__half2float(h[4 + i]), sf) & 0xff) << (8 * i);
      }
    }
    qr[v] = make_uint2(lo, hi);
  }
}

}  // namespace

cudaError_t launch_act_quant(int M, int K, const uint16_t* X, int8_t* Xq, uint16_t* sx,
                             cudaStream_t s) {
  dim3 grid((M + kRowsPerBlock - 1) / kRowsPerBlock);
  act_quant_kernel<<<grid, kRowsPerBlock * 32, 0, s>>>(X, Xq, sx, M, K);
  return cudaGetLastError();
}

}  // namespace qoq
