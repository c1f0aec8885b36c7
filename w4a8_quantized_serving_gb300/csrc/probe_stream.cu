// probe_stream.cu -- a streaming-read kernel that measures what one launch of
// a given size can reach on this GPU's HBM, for the GEMM's roofline figures.
//
// Measurement support only, built into its own library (libqoq_probe.so) and
// used by the benchmark and its tests; the W4A8 path neither links nor calls
// it.  The kernel reads `bytes` of device memory once and does nothing else
// with them but sum their 32-bit words (mod 2^64) into *sink, so the reads
// cannot be dropped and a test can check that every byte was read.  Each
// launch is a programmatic dependent of the preceding kernel, as the GEMM
// calls are: it lets the next launch become resident at once and, when
// `dependent` is set, waits for the preceding kernel before its first read,
// as a layer whose input comes from the previous layer must.  Timed the way
// the GEMM call is timed, the time per launch of a chain of such launches is
// the HBM time one launch of that many bytes needs here: launch, DRAM latency,
// ramp-up and drain included, which a bandwidth figure measured on gigabytes
// leaves out.
//
// A second form, qoq_probe_stream_ring, moves the bytes the way the decode
// GEMM moves its weights: one CTA per SM, one or two producer threads that
// bulk-copy 8 KB (or 16 KB) chunks of the CTA's contiguous share into a
// 192 KB shared-memory ring (so no second CTA fits beside it), consumer warps
// that wait on each stage, read it and release it.  With `prefetch` set, the
// producers issue the ring's first lap before they wait for the preceding
// kernel and the consumers wait for that kernel before their first read, as
// the GEMM's weight copies and MMAs do: the GEMM's memory traffic with no
// arithmetic.  Each producer thread issues about one copy per 0.2 us, so the
// copy size and the producer count bound the rate an SM streams at.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "ptx.cuh"

namespace {

using namespace qoq;

constexpr int kThreads = 256;
constexpr int kUnroll = 8;  // 16-byte loads in flight per thread: 128 B, 64 KB per SM at 2 CTAs

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned long long word_sum(const uint4& v) {
  return (unsigned long long)v.x + v.y + v.z + v.w;
}

template <bool DEPENDENT>
__global__ void __launch_bounds__(kThreads) stream_read_kernel(const uint4* __restrict__ src, size_t n16,
                                                               unsigned long long* sink) {
  if (DEPENDENT) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t stride = (size_t)gridDim.x * kThreads;
  size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
  unsigned long long acc = 0;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) v[j] = ld_stream(src + i + j * stride);
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) acc += word_sum(v[j]);
  }
  for (; i < n16; i += stride) acc += word_sum(ld_stream(src + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc != 0) atomicAdd(sink, acc);
}

// ------------------------------------------------------------ ring form --

constexpr int kRingBytes = 24 * 8192;  // 192 KB of stages: one CTA per SM
constexpr int kMaxProducers = 2;       // warps 0 .. 1 (warp 1 idles with one producer)
constexpr int kConsumers = 4;          // warps 2 .. 5
constexpr int kRingThreads = 32 * (kMaxProducers + kConsumers);
constexpr int kRingSmem = kRingBytes + 2 * 24 * 8 + 1024;  // + barriers, + slack for 1024-byte alignment
constexpr long long kWaitCycles = 4000000000LL;           // ~2 s at 2 GHz: a wait gives up

// Bounded phase wait: false once ~kWaitCycles have passed without the phase.
__device__ __noinline__ bool ring_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 0 && clock64() - t0 > kWaitCycles) return false;
  }
}

// CHUNK-byte copies into STAGES = kRingBytes / CHUNK stages.  Chunk i of the
// CTA's share goes to stage i % STAGES; producer warp i % nprod issues it and
// consumer warp i % kConsumers reads it (STAGES is a multiple of both, so each
// stage has one producer and one consumer).
template <int CHUNK, bool PREFETCH>
__global__ void __launch_bounds__(kRingThreads, 1) stream_ring_kernel(const uint8_t* __restrict__ src, size_t bytes,
                                                                     int nprod, unsigned long long* sink,
                                                                     unsigned* err) {
  constexpr int STAGES = kRingBytes / CHUNK;
  static_assert(STAGES % kConsumers == 0 && STAGES % kMaxProducers == 0 && STAGES <= 32, "stage ownership");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t rbase = smem_addr(ring);
  const uint32_t full = rbase + kRingBytes, empty = full + 8 * STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t nchunks = (bytes + CHUNK - 1) / CHUNK;
  const size_t c0 = nchunks * blockIdx.x / gridDim.x, c1 = nchunks * (blockIdx.x + 1) / gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + 8 * s, 1);   // the producer's arrive.expect_tx (+ the copy's bytes)
      mbar_init(empty + 8 * s, 1);  // the stage's consumer warp
    }
    fence_mbar_init();
  }
  __syncthreads();
  grid_dep_launch_dependents();
  unsigned long long acc = 0;
  if (warp < kMaxProducers) {
    if (lane == 0 && warp < nprod) {
      const uint64_t pol = policy_evict_first();
      uint32_t issued = 0, par = 0;  // per stage: a copy in its latest lap; that lap's parity
      bool waited = !PREFETCH;
      if (!PREFETCH) grid_dep_wait();
      for (size_t c = c0 + warp; c < c1; c += nprod) {
        const uint32_t i = (uint32_t)(c - c0), s = i % STAGES, lap = i / STAGES;
        if (!waited && lap > 0) {  // the first lap is issued before the preceding kernel ends
          grid_dep_wait();
          waited = true;
        }
        if (lap > 0 && !ring_wait(empty + 8 * s, (lap - 1) & 1)) {
          atomicExch(err, 1u);
          break;
        }
        const size_t left = bytes - c * CHUNK;
        const uint32_t n = left < (size_t)CHUNK ? (uint32_t)left : (uint32_t)CHUNK;
        mbar_arrive_expect_tx(full + 8 * s, n);
        bulk_g2s(rbase + s * CHUNK, src + c * CHUNK, n, full + 8 * s, pol);
        issued |= 1u << s;
        par = (par & ~(1u << s)) | ((lap & 1) << s);
      }
      // every copy still in flight lands before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) ring_wait(full + 8 * s, (par >> s) & 1u);
    }
  } else {
    grid_dep_wait();
    for (size_t c = c0 + (warp - kMaxProducers); c < c1; c += kConsumers) {
      const uint32_t i = (uint32_t)(c - c0), s = i % STAGES, lap = i / STAGES;
      if (!__all_sync(0xffffffffu, ring_wait(full + 8 * s, lap & 1))) {
        if (lane == 0) atomicExch(err, 1u);
        break;
      }
      const size_t left = bytes - c * CHUNK;
      const uint32_t n = left < (size_t)CHUNK ? (uint32_t)left : (uint32_t)CHUNK;
      for (uint32_t off = 16u * lane; off < n; off += 512u)
        acc += word_sum(*reinterpret_cast<const uint4*>(ring + s * CHUNK + off));
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + 8 * s);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
  if (lane == 0 && acc != 0) atomicAdd(sink, acc);
}

template <int CHUNK, bool PREFETCH>
cudaError_t launch_ring(const cudaLaunchConfig_t& cfg, const uint8_t* src, size_t bytes, int nprod,
                        unsigned long long* sink, unsigned* err) {
  static int attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(stream_ring_kernel<CHUNK, PREFETCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRingSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = 1;
  }
  return cudaLaunchKernelEx(&cfg, stream_ring_kernel<CHUNK, PREFETCH>, src, bytes, nprod, sink, err);
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

// Reads `bytes` at `src` (device memory, 16-byte aligned, `bytes` a multiple
// of 16) once on `stream` (a cudaStream_t; null: the legacy default stream)
// and adds the sum of its 32-bit words, mod 2^64, to *sink (device memory,
// 8-byte aligned; the caller zeroes it).  Grid: ctas_per_sm (1..4) CTAs of 256
// threads per SM.  dependent != 0: the launch waits for the preceding kernel
// before its first read.  bytes == 0 launches nothing.  Returns a
// cudaError_t: cudaErrorInvalidValue for a null pointer, a misaligned
// address or size, or ctas_per_sm outside 1..4; otherwise the launch's status.
extern "C" int qoq_probe_stream_read(const void* src, size_t bytes, unsigned long long* sink, int ctas_per_sm,
                                     int dependent, void* stream) {
  if (bytes == 0) return cudaSuccess;
  if (!src || !sink || ((uintptr_t)src & 15u) || (bytes & 15u) || ((uintptr_t)sink & 7u) || ctas_per_sm < 1 ||
      ctas_per_sm > 4)
    return cudaErrorInvalidValue;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms * ctas_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint4* s = static_cast<const uint4*>(src);
  const size_t n16 = bytes / 16;
  const cudaError_t e = dependent ? cudaLaunchKernelEx(&cfg, stream_read_kernel<true>, s, n16, sink)
                                  : cudaLaunchKernelEx(&cfg, stream_read_kernel<false>, s, n16, sink);
  return (int)e;
}

// The ring form (see the head of this file): one CTA per SM of 192 threads and
// ~194 KB of shared memory.  Arguments as qoq_probe_stream_read's, and:
// chunk_bytes (8192 or 16384) per copy; producers (1 or 2) copy-issuing
// threads per CTA; err (device memory, 4-byte aligned, zeroed by the caller)
// becomes non-zero if a wait inside the kernel gave up (~2 s), in which case
// the sum is partial.  prefetch != 0: the first lap of copies is issued before
// the wait for the preceding kernel; otherwise nothing is read before it.
extern "C" int qoq_probe_stream_ring(const void* src, size_t bytes, unsigned long long* sink, unsigned* err,
                                     int chunk_bytes, int producers, int prefetch, void* stream) {
  if (bytes == 0) return cudaSuccess;
  if (!src || !sink || !err || ((uintptr_t)src & 15u) || (bytes & 15u) || ((uintptr_t)sink & 7u) ||
      ((uintptr_t)err & 3u) || (chunk_bytes != 8192 && chunk_bytes != 16384) || producers < 1 ||
      producers > kMaxProducers)
    return cudaErrorInvalidValue;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = kRingSmem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint8_t* s = static_cast<const uint8_t*>(src);
  cudaError_t e;
  if (chunk_bytes == 8192)
    e = prefetch ? launch_ring<8192, true>(cfg, s, bytes, producers, sink, err)
                 : launch_ring<8192, false>(cfg, s, bytes, producers, sink, err);
  else
    e = prefetch ? launch_ring<16384, true>(cfg, s, bytes, producers, sink, err)
                 : launch_ring<16384, false>(cfg, s, bytes, producers, sink, err);
  return (int)e;
}
