// act_quant.cu -- per-token symmetric int8 activation quantization.
//
// QServe talk write-up, "Precision Data Flow and Activation Quantization
// Fusion": every linear layer takes 8-bit activations (the write-up fuses the
// quantizer into the preceding LayerNorm; here it is a standalone kernel).
//   s_x[m]  = fp16_rn(fp32(max_k |X[m,k]|) / 127)        (IEEE fp32 divide)
//   Xq[m,k] = clamp(rint(X[m,k] / s_x[m]), -127, 127)      (fp32 divide, ties even;
//             computed without a divide by rint_div_fp16, which gives the same codes)
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

__device__ __forceinline__ float absmax8(uint4 v, float m) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(__habs2(h[i]));
    m = fmaxf(m, fmaxf(f.x, f.y));
  }
  return m;
}

__device__ __forceinline__ uint32_t quant4(const __half* h, float sf, float rf) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float q = fminf(127.0f, fmaxf(-127.0f, rint_div_fp16(__half2float(h[i]), sf, rf)));
    r |= (uint32_t)((int)q & 0xff) << (8 * i);
  }
  return r;
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = K / 8;
  const bool live = row < M;
  const uint4* xr = reinterpret_cast<const uint4*>(X + (size_t)(live ? row : 0) * K);
  uint4 v[MAXV];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = t + i * T;
    if (live && idx < nvec) {
      v[i] = __ldcg(xr + idx);  // L2: X may have been written by the preceding kernel
      amax = absmax8(v[i], amax);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (T > 32) {  // combine the T/32 warps of this row
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    const int w0 = (threadIdx.x / T) * (T / 32);
    amax = 0.0f;
    for (int w = 0; w < T / 32; ++w) amax = fmaxf(amax, warp_max[w0 + w]);
  }
  if (!live) return;

  __half s = __float2half_rn(0.0f);
  if (amax > 0.0f) s = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float sf = __half2float(s);
  const float rf = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
  if (t == 0) sx[row] = __half_as_ushort(s);

  uint2* qr = reinterpret_cast<uint2*>(Xq + (size_t)row * K);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = t + i * T;
    if (idx < nvec) {
      uint2 out = make_uint2(0, 0);
      if (sf != 0.0f) {
        const __half* h = reinterpret_cast<const __half*>(&v[i]);
        out = make_uint2(quant4(h, sf, rf), quant4(h + 4, sf, rf));
      }
      qr[idx] = out;
    }
  }
}

}  // namespace

cudaError_t launch_act_quant(int M, int K, const uint16_t* X, int8_t* Xq, uint16_t* sx,
                             cudaStream_t s) {
  const int nvec = K / 8;
  // threads per row: a power of two, ~4 vectors each (latency), at most 16
  int T = 32;
  while (T * 4 < nvec && T < 1024) T *= 2;
  const int threads = T < 128 ? 128 : T;
  const int rows_per_cta = threads / T;
  const int grid = (M + rows_per_cta - 1) / rows_per_cta;
  const int vpt = (nvec + T - 1) / T;  // <= 4 unless T = 1024; <= 16 for K <= 131072
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (vpt <= 4) return cudaLaunchKernelEx(&cfg, act_quant_kernel<4>, X, Xq, sx, M, K, T);
  if (vpt <= 8) return cudaLaunchKernelEx(&cfg, act_quant_kernel<8>, X, Xq, sx, M, K, T);
  if (vpt <= 16) return cudaLaunchKernelEx(&cfg, act_quant_kernel<16>, X, Xq, sx, M, K, T);
  return cudaErrorInvalidValue;
}

}  // namespace qoq
