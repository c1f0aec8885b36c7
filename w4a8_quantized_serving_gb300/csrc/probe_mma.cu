// probe_mma.cu -- how fast one thread issues tcgen05.mma, for the design of
// the GEMM kernels' MMA issue (built into libqoq_probe.so with the streaming
// probe; measurement support, not part of the W4A8 path).
//
// One thread issues `iters` MMAs of the GEMM's shape back to back (kind::f16,
// K=16, M=128 per CTA -- 256 for a CTA pair, cta_group::2 -- and N tokens; A
// from tensor memory, B a zero tile in shared memory, one accumulator), reads
// the SM clock before each of issues 2 .. 65, then commits and waits for them
// all to complete.  When the issue spacing stays at the thread's own
// rate while the tensor pipe needs less time per MMA, one issuing thread
// cannot keep the pipe busy; when the spacing grows to the pipe's time per
// MMA after a few issues, the thread runs ahead and later issues wait for
// room.  out[0]: cycles to issue all, out[1]: cycles until the commit's
// barrier completed, out[2]: 1 if it did (the wait is bounded), out[3]:
// iters, out[4 + i]: cycles from the start to just before issue i + 1
// (i < 64).
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_common.cuh"

namespace {

using namespace qoq;

constexpr int kBTile = 32768;  // the zero B operand: 128-byte swizzled, K-major, up to 256 rows
constexpr int kProbeSmem = kBTile + 64 + 1024;

template <bool PAIR, int N>
__global__ void __launch_bounds__(128, 1) mma_issue_kernel(unsigned long long* out, int iters) {
  __shared__ unsigned long long stamps[64];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;
  const uint32_t bar = sb + kBTile, slot = sb + kBTile + 8;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < kBTile / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();  // the zero tile -> the MMAs' operand reads
  if (warp == 0) {
    if constexpr (PAIR)
      tmem_alloc_pair(slot, kTmemCols);
    else
      tmem_alloc(slot, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kBTile + 8);
  {  // a zero A operand at columns 256 .. 271 of this warp's lanes
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0;
    tmem_st16(tmem + ((uint32_t)(warp * 32) << 16) + 256, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();
  tc_fence_after();
  if (rank == 0 && warp == 0) {
    __syncwarp();
    if (threadIdx.x == 0) {
      constexpr uint32_t kIdesc = mma_idesc(N, PAIR ? 2 * kTileN : kTileN);
      const uint32_t dl = desc_sw128_lo(sb);
      const long long t0 = clock64();
      for (int i = 0; i < iters; ++i) {
        if (i > 0 && i <= 64) stamps[i - 1] = (unsigned long long)(clock64() - t0);
        if constexpr (PAIR)
          tc_mma_ts_pair(tmem, tmem + 256, dl, kDescSw128Hi, kIdesc, 1u);
        else
          tc_mma_ts(tmem, tmem + 256, dl, kDescSw128Hi, kIdesc, 1u);
      }
      const long long t1 = clock64();
      if constexpr (PAIR)
        tc_commit_pair_mc(bar, 1);  // this (the leading) CTA's barrier
      else
        tc_commit(bar);
      unsigned ok = 0;
      for (int i = 0; i < (1 << 24) && !ok; ++i) ok = mbar_try_wait(bar, 0) ? 1u : 0u;
      const long long t2 = clock64();
      out[0] = (unsigned long long)(t1 - t0);
      out[1] = (unsigned long long)(t2 - t0);
      out[2] = ok;
      out[3] = (unsigned long long)iters;
      const int ns = iters - 1 < 64 ? iters - 1 : 64;
      for (int i = 0; i < 64; ++i) out[4 + i] = i < ns ? stamps[i] : 0ull;
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // the pair's MMAs read both CTAs' memory
  if (warp == 0) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool PAIR, int N>
cudaError_t launch_probe(unsigned long long* out, int iters, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(PAIR ? 2 : 1);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kProbeSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mma_issue_kernel<PAIR, N>, out, iters);
}

}  // namespace

// out: 68 unsigned 64-bit words in device memory (8-byte aligned), written as
// described at the head of this file.  pair: 0 (one CTA, cta_group::1) or 1
// (a cluster of two, cta_group::2); n: the MMA's N, 16, 32, 64, 128 or 256
// for one CTA (the decode kernel's token tiles are 16, 32 or 64), 128 or 256
// for a pair; iters: 2 .. 1 << 20.  Returns a cudaError_t:
// cudaErrorInvalidValue for other arguments (before any launch);
// cudaErrorNoDevice off an sm_103 device; otherwise the launch's status.
extern "C" int qoq_probe_mma_issue(int pair, int n, int iters, unsigned long long* out, void* stream) {
  const bool n_ok = n == 128 || n == 256 || (!pair && (n == 16 || n == 32 || n == 64));
  if (!out || ((uintptr_t)out & 7u) || (pair != 0 && pair != 1) || !n_ok || iters < 2 || iters > (1 << 20))
    return cudaErrorInvalidValue;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return cudaErrorNoDevice;
  if (major != 10 || minor != 3) return cudaErrorNoDevice;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (pair)
    e = n == 128 ? launch_probe<true, 128>(out, iters, s) : launch_probe<true, 256>(out, iters, s);
  else if (n == 16)
    e = launch_probe<false, 16>(out, iters, s);
  else if (n == 32)
    e = launch_probe<false, 32>(out, iters, s);
  else if (n == 64)
    e = launch_probe<false, 64>(out, iters, s);
  else
    e = n == 128 ? launch_probe<false, 128>(out, iters, s) : launch_probe<false, 256>(out, iters, s);
  return (int)e;
}
