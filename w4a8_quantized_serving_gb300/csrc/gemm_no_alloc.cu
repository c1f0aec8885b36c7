// gemm_no_alloc.cu -- qoq_w4a8_gemm for callers that cannot allocate device
// memory (declared in include/qoq.h as qoq_w4a8_gemm_no_alloc).
//
// qoq_w4a8_gemm needs a caller-supplied workspace (status header, split-K
// counters and partial sums, and for M > 64 the fp16 B-operand copy of Xq).
// Some callers have no way to provide one:
//  - a plugin handed only its input and output buffers by a host program that
//    does not expose its allocator;
//  - a serving process that reserved nearly all device memory for its caches
//    at start-up, so that a later cudaMalloc fails;
//  - a step that must not synchronise the device, which cudaMalloc and
//    cudaFree may do.
// For them this entry point runs the same GEMM with its workspace in a
// file-scope device array of fixed size, QOQ_NO_ALLOC_SCRATCH_BYTES.
//
// In host code `g_no_alloc_scratch` names a host-side stand-in, not device
// memory; its device address is taken once per device with
// cudaGetSymbolAddress (with that device current) and passed to the kernels.
// Device code here names the array directly.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/qoq.h"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[QOQ_NO_ALLOC_SCRATCH_BYTES];
// Sticky device status of the calls since the last qoq_no_alloc_last_status:
// each call's clear kernel folds in the status its predecessor left in the
// header before clearing it.
static __device__ int g_no_alloc_sticky;

constexpr int kMaxDevices = 64;

struct ScratchSetup {
  std::once_flag once;
  void* ptr = nullptr;
  qoq_status status = QOQ_ERR_CUDA;
};
ScratchSetup g_setup[kMaxDevices];

// Once per device, with that device current: check the architecture (the
// array lives in an sm_103a-only module), then take the array's device address.
qoq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return QOQ_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return QOQ_ERR_CUDA;
  ScratchSetup& s = g_setup[dev];
  std::call_once(s.once, [&] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      s.status = QOQ_ERR_CUDA;
      return;
    }
    if (major != 10 || minor != 3) {
      s.status = QOQ_ERR_ARCH;
      return;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      s.status = QOQ_ERR_CUDA;
      return;
    }
    s.ptr = p;
    s.status = QOQ_OK;
  });
  *out = s.ptr;
  return s.status;
}

// Zeroes the part of the workspace that the GEMM requires to start at zero:
// the header's status and abort words (after folding a non-zero status of the
// previous call into g_no_alloc_sticky), and the 16-byte words [lo16, hi16)
// (split-K counters and partial sums of 128-token tiles).  The decode
// kernel's hand-off epoch and CTA exit counter (header words 2 and 3) are
// kept: every launch leaves the counter at zero and advances the epoch, so
// partial sums that a call which ran out of its wait limit left behind carry
// an older tag than any later call's.
__global__ void __launch_bounds__(256) no_alloc_clear_kernel(size_t lo16, size_t hi16) {
  uint4* p = reinterpret_cast<uint4*>(g_no_alloc_scratch);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid == 0) {
    const int prev = *reinterpret_cast<volatile int*>(g_no_alloc_scratch);  // stream-ordered after that call
    if (prev != 0) g_no_alloc_sticky = prev;
    *reinterpret_cast<uint2*>(g_no_alloc_scratch) = make_uint2(0u, 0u);  // status and abort words
  }
  for (size_t i = lo16 + tid; i < hi16; i += stride) p[i] = make_uint4(0u, 0u, 0u, 0u);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" qoq_status qoq_w4a8_gemm_no_alloc(int M, int N, int K, int g, const int8_t* Xq,
                                             const uint16_t* sx_f16, const uint8_t* packed,
                                             const uint16_t* s1_f16, uint16_t* Y_f16,
                                             int32_t* acc_debug, qoq_stream_t stream) {
  // Argument checks in the order qoq_w4a8_gemm takes them, all before any
  // device access.
  if (!Xq || !sx_f16 || !packed || !s1_f16 || !Y_f16) return QOQ_ERR_NULL;
  const size_t need = qoq_gemm_workspace_bytes(M, N, K, qoq::kGroup);  // 0: bad shape (any g)
  if (need == 0) return QOQ_ERR_SHAPE;
  if (!qoq::group_size_ok(K, g)) return QOQ_ERR_UNSUPPORTED;
  if (!aligned16(Xq) || !aligned16(sx_f16) || !aligned16(packed) || !aligned16(s1_f16) ||
      !aligned16(Y_f16) || (acc_debug && !aligned16(acc_debug)))
    return QOQ_ERR_MISALIGNED;
  if (need > QOQ_NO_ALLOC_SCRATCH_BYTES) return QOQ_ERR_WORKSPACE;

  void* scratch = nullptr;
  const qoq_status st = scratch_address(&scratch);
  if (st != QOQ_OK) return st;

  // The array keeps whatever the previous call left (normally zeros, but not
  // after a call that ran out of its wait limit), so clear the zero-start part
  // on the stream before every GEMM.
  const qoq::WsLayout L = qoq::gemm_ws_layout(M, N, K);
  const size_t lo16 = L.cnt_off / 16, hi16 = L.zero_bytes / 16;
  size_t blocks = (hi16 - lo16 + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 1024) blocks = 1024;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  // The launch's own return code: an error left pending by unrelated work is
  // neither reported as this call's nor cleared here.
  if (cudaLaunchKernelEx(&cfg, no_alloc_clear_kernel, lo16, hi16) != cudaSuccess) {
    cudaGetLastError();  // clear the launch's own (non-sticky) error, as qoq_w4a8_gemm does
    return QOQ_ERR_CUDA;
  }

  return qoq_w4a8_gemm(M, N, K, g, Xq, sx_f16, packed, s1_f16, Y_f16, acc_debug, scratch,
                       QOQ_NO_ALLOC_SCRATCH_BYTES, stream);
}

extern "C" qoq_status qoq_no_alloc_last_status(qoq_stream_t stream) {
  void* scratch = nullptr;
  const qoq_status st = scratch_address(&scratch);
  if (st != QOQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  int sticky = 0, last = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&sticky, g_no_alloc_sticky, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpy(&last, scratch, sizeof(int), cudaMemcpyDeviceToHost);  // the latest call's
  const int zero = 0;
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_no_alloc_sticky, &zero, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpy(scratch, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QOQ_ERR_CUDA;
  }
  const int code = sticky != 0 ? sticky : last;
  return code == 0 ? QOQ_OK : (code == QOQ_ERR_DEVICE_TIMEOUT ? QOQ_ERR_DEVICE_TIMEOUT : QOQ_ERR_CUDA);
}
