// act_quant.cu -- per-token symmetric int8 activation quantization.
//
// QServe talk write-up, "Precision Data Flow and Activation Quantization
// Fusion": every linear layer takes 8-bit activations (the write-up fuses the
// quantizer into the preceding LayerNorm; here it is a standalone kernel).
//   s_x[m]  = fp16_rn(fp32(max_k |X[m,k]|) / 127)        (IEEE fp32 divide)
//   Xq[m,k] = clamp(rint(X[m,k] / s_x[m]), -127, 127)      (fp32 divide, ties even)
// An all-zero row gets s_x = 0 and Xq = 0.
//
// One CTA per token row: each thread loads up to 16 vectors of 8 fp16 values
// (16 bytes) into registers, the CTA reduces the max-abs (warp shuffles, then
// shared memory), and the same registers are quantized and stored, so X is
// read from HBM once.  The work is HBM bound: 2 bytes read and 1 byte written
// per element.
#include <cuda_fp16.h>

#include "internal.h"

namespace qoq {
namespace {

constexpr int kMaxVecPerThread = 16;  // K <= 131072 with 1024 threads

__device__ __forceinline__ float absmax8(uint4 v, float m) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(__habs2(h[i]));
    m = fmaxf(m, fmaxf(f.x, f.y));
  }
  return m;
}

__device__ __forceinline__ uint32_t quant4(const __half* h, float sf) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = min(127, max(-127, __float2int_rn(__fdiv_rn(__half2float(h[i]), sf))));
    r |= (uint32_t)(q & 0xff) << (8 * i);
  }
  return r;
}

__global__ void __launch_bounds__(1024) act_quant_kernel(const uint16_t* __restrict__ X,
                                                         int8_t* __restrict__ Xq,
                                                         uint16_t* __restrict__ sx, int K) {
  __shared__ float warp_max[32];
  const int row = blockIdx.x;
  const int nvec = K / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(X + (size_t)row * K);
  uint4 v[kMaxVecPerThread];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nvec) {
      v[i] = __ldg(xr + idx);
      amax = absmax8(v[i], amax);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    float m = lane < nw ? warp_max[lane] : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) warp_max[0] = m;
  }
  __syncthreads();
  amax = warp_max[0];

  __half s = __float2half_rn(0.0f);
  if (amax > 0.0f) s = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float sf = __half2float(s);
  if (threadIdx.x == 0) sx[row] = __half_as_ushort(s);

  uint2* qr = reinterpret_cast<uint2*>(Xq + (size_t)row * K);
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nvec) {
      uint2 out = make_uint2(0, 0);
      if (sf != 0.0f) {
        const __half* h = reinterpret_cast<const __half*>(&v[i]);
        out = make_uint2(quant4(h, sf), quant4(h + 4, sf));
      }
      qr[idx] = out;
    }
  }
}

}  // namespace

cudaError_t launch_act_quant(int M, int K, const uint16_t* X, int8_t* Xq, uint16_t* sx,
                             cudaStream_t s) {
  const int nvec = K / 8;
  // one vector per thread up to 1024 threads (latency), up to 16 beyond (K <= 131072)
  int threads = (nvec + 31) / 32 * 32;
  if (threads > 1024) threads = 1024;
  act_quant_kernel<<<M, threads, 0, s>>>(X, Xq, sx, K);
  return cudaGetLastError();
}

}  // namespace qoq
