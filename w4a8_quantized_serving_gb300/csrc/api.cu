// api.cu -- the extern "C" boundary of libqoq.so (declared in include/qoq.h).
// Host-side argument validation, per-device attribute cache, dispatch to the
// kernel launchers, and the device status read-back.  No allocation, no
// printing, no exceptions across the boundary.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/qoq.h"
#include "internal.h"

namespace {

using qoq::kGroup;

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s

std::atomic<unsigned long long> g_timeout_ns{0};
std::atomic<int> g_fault{0};
std::atomic<unsigned long long*> g_trace{nullptr};
std::atomic<unsigned> g_call_id{0};

struct DevInfo {
  std::once_flag once;
  int sms = 0;
  int major = 0, minor = 0;
  cudaError_t err = cudaSuccess;
};
DevInfo g_dev[kMaxDevices];

// Current device's SM count and compute capability (cached, thread-safe).
qoq_status device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return QOQ_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return QOQ_ERR_CUDA;
  DevInfo& d = g_dev[dev];
  std::call_once(d.once, [&] {
    d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
  });
  if (d.err != cudaSuccess) return QOQ_ERR_CUDA;
  if (d.major != 10 || d.minor != 3) return QOQ_ERR_ARCH;
  if (sms) *sms = d.sms;
  return QOQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool shape_ok_mk(int M, int K) {
  return M >= 1 && M <= (1 << 24) && K >= kGroup && K <= 131072 && K % kGroup == 0;
}

bool shape_ok_nk(int N, int K) {
  return N >= qoq::kTileN && N <= (1 << 24) && N % qoq::kTileN == 0 && K >= kGroup && K <= 131072 &&
         K % kGroup == 0;
}

qoq_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return QOQ_OK;
  cudaGetLastError();  // clear a non-sticky error so later calls are not blamed
  return QOQ_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* qoq_status_str(int s) {
  switch (s) {
    case QOQ_OK: return "QOQ_OK";
    case QOQ_ERR_NULL: return "QOQ_ERR_NULL";
    case QOQ_ERR_SHAPE: return "QOQ_ERR_SHAPE";
    case QOQ_ERR_UNSUPPORTED: return "QOQ_ERR_UNSUPPORTED";
    case QOQ_ERR_MISALIGNED: return "QOQ_ERR_MISALIGNED";
    case QOQ_ERR_WORKSPACE: return "QOQ_ERR_WORKSPACE";
    case QOQ_ERR_CUDA: return "QOQ_ERR_CUDA";
    case QOQ_ERR_DEVICE_TIMEOUT: return "QOQ_ERR_DEVICE_TIMEOUT";
    case QOQ_ERR_ARCH: return "QOQ_ERR_ARCH";
    default: return "QOQ_ERR_UNKNOWN";
  }
}

int qoq_version(void) { return 100; }

size_t qoq_packed_weight_bytes(int N, int K, int g) {
  if (!shape_ok_nk(N, K) || !qoq::group_size_ok(K, g)) return 0;
  return (size_t)(N / qoq::kTileN) * (size_t)(K / kGroup) * (size_t)qoq::w_tile_bytes(qoq::gpt_for_group(g));
}

size_t qoq_gemm_workspace_bytes(int M, int N, int K, int g) {
  if (!shape_ok_mk(M, K) || !shape_ok_nk(N, K) || !qoq::group_size_ok(K, g)) return 0;
  return qoq::gemm_ws_layout(M, N, K).total;
}

qoq_status qoq_pack_weights(int N, int K, int g, const uint16_t* W_f16, uint8_t* packed,
                            uint16_t* s1_f16, qoq_stream_t stream) {
  if (!W_f16 || !packed || !s1_f16) return QOQ_ERR_NULL;
  if (!shape_ok_nk(N, K)) return QOQ_ERR_SHAPE;
  if (!qoq::group_size_ok(K, g)) return QOQ_ERR_UNSUPPORTED;
  if (!aligned16(W_f16) || !aligned16(packed) || !aligned16(s1_f16)) return QOQ_ERR_MISALIGNED;
  qoq_status st = device_info(nullptr);
  if (st != QOQ_OK) return st;
  return from_cuda(qoq::launch_pack(N, K, g, W_f16, packed, s1_f16, reinterpret_cast<cudaStream_t>(stream)));
}

qoq_status qoq_quant_act(int M, int K, const uint16_t* X_f16, int8_t* Xq, uint16_t* sx_f16,
                         qoq_stream_t stream) {
  if (!X_f16 || !Xq || !sx_f16) return QOQ_ERR_NULL;
  if (!shape_ok_mk(M, K)) return QOQ_ERR_SHAPE;
  if (!aligned16(X_f16) || !aligned16(Xq) || !aligned16(sx_f16)) return QOQ_ERR_MISALIGNED;
  qoq_status st = device_info(nullptr);
  if (st != QOQ_OK) return st;
  return from_cuda(qoq::launch_act_quant(M, K, X_f16, Xq, sx_f16, reinterpret_cast<cudaStream_t>(stream)));
}

qoq_status qoq_norm_quant_act(int M, int K, int kind, float eps, const uint16_t* X_f16,
                              const uint16_t* gamma_f16, const uint16_t* beta_f16, int8_t* Xq,
                              uint16_t* sx_f16, qoq_stream_t stream) {
  if (!X_f16 || !gamma_f16 || !Xq || !sx_f16 || (kind == QOQ_NORM_LAYER && !beta_f16)) return QOQ_ERR_NULL;
  if (kind != QOQ_NORM_RMS && kind != QOQ_NORM_LAYER) return QOQ_ERR_UNSUPPORTED;
  if (!(eps > 0.0f) || !(eps <= 3.4e38f)) return QOQ_ERR_UNSUPPORTED;  // positive and finite
  if (!shape_ok_mk(M, K)) return QOQ_ERR_SHAPE;
  if (!aligned16(X_f16) || !aligned16(gamma_f16) || (kind == QOQ_NORM_LAYER && !aligned16(beta_f16)) ||
      !aligned16(Xq) || !aligned16(sx_f16))
    return QOQ_ERR_MISALIGNED;
  qoq_status st = device_info(nullptr);
  if (st != QOQ_OK) return st;
  return from_cuda(qoq::launch_norm_quant(M, K, kind, eps, X_f16, gamma_f16, beta_f16, Xq, sx_f16,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The two GEMM entry points share their checks and launch path.
qoq_status gemm_entry(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx_f16,
                      const uint8_t* packed, const uint16_t* s1_f16, uint16_t* Y_f16, int32_t* acc_debug,
                      void* workspace, size_t ws_bytes, qoq_stream_t stream, bool zero_folded) {
  if (!Xq || !sx_f16 || !packed || !s1_f16 || !Y_f16) return QOQ_ERR_NULL;
  if (!shape_ok_mk(M, K) || !shape_ok_nk(N, K)) return QOQ_ERR_SHAPE;
  if (!qoq::group_size_ok(K, g) || (zero_folded && g < kGroup)) return QOQ_ERR_UNSUPPORTED;
  if (!aligned16(Xq) || !aligned16(sx_f16) || !aligned16(packed) || !aligned16(s1_f16) ||
      !aligned16(Y_f16) || (acc_debug && !aligned16(acc_debug)))
    return QOQ_ERR_MISALIGNED;
  if (!workspace || ws_bytes < qoq_gemm_workspace_bytes(M, N, K, g)) return QOQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QOQ_ERR_MISALIGNED;
  int sms = 0;
  qoq_status st = device_info(&sms);
  if (st != QOQ_OK) return st;
  unsigned long long tmo = g_timeout_ns.load();
  if (tmo == 0) tmo = kDefaultTimeoutNs;
  unsigned call_id = g_call_id.fetch_add(1) + 1;
  if (call_id == 0) call_id = g_call_id.fetch_add(1) + 1;  // skip 0 on wrap-around
  return from_cuda(qoq::launch_gemm(M, N, K, g, Xq, sx_f16, packed, s1_f16, Y_f16, acc_debug, workspace,
                                    sms, tmo, g_fault.load(), call_id, g_trace.load(), zero_folded,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

qoq_status qoq_w4a8_gemm(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx_f16,
                         const uint8_t* packed, const uint16_t* s1_f16, uint16_t* Y_f16,
                         int32_t* acc_debug, void* workspace, size_t ws_bytes,
                         qoq_stream_t stream) {
  return gemm_entry(M, N, K, g, Xq, sx_f16, packed, s1_f16, Y_f16, acc_debug, workspace, ws_bytes, stream, false);
}

qoq_status qoq_w4a8_gemm_zero_folded(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx_f16,
                                     const uint8_t* packed, const uint16_t* s1_f16, uint16_t* Y_f16,
                                     int32_t* acc_debug, void* workspace, size_t ws_bytes,
                                     qoq_stream_t stream) {
  return gemm_entry(M, N, K, g, Xq, sx_f16, packed, s1_f16, Y_f16, acc_debug, workspace, ws_bytes, stream, true);
}

size_t qoq_w4ax_act_bytes(int M, int K, int n8) {
  if (!shape_ok_mk(M, K) || n8 < 0 || n8 > K / kGroup) return 0;
  return (size_t)M * ((size_t)128 * n8 + (size_t)64 * (K / kGroup - n8));
}

size_t qoq_w4ax_workspace_bytes(int M, int N, int K, int g) {
  if (!shape_ok_mk(M, K) || !shape_ok_nk(N, K) || !qoq::group_size_ok(K, g)) return 0;
  return qoq::w4ax_ws_layout(M, N, K).total;
}

qoq_status qoq_quant_act_w4ax(int M, int K, int n8, const uint16_t* X_f16, uint8_t* Xa, uint16_t* sxb_f16,
                              qoq_stream_t stream) {
  if (!X_f16 || !Xa || !sxb_f16) return QOQ_ERR_NULL;
  if (!shape_ok_mk(M, K)) return QOQ_ERR_SHAPE;
  if (n8 < 0 || n8 > K / kGroup) return QOQ_ERR_UNSUPPORTED;
  if (!aligned16(X_f16) || !aligned16(Xa) || !aligned16(sxb_f16)) return QOQ_ERR_MISALIGNED;
  qoq_status st = device_info(nullptr);
  if (st != QOQ_OK) return st;
  return from_cuda(qoq::launch_act_quant_w4ax(M, K, n8, X_f16, Xa, sxb_f16, reinterpret_cast<cudaStream_t>(stream)));
}

qoq_status qoq_w4ax_gemm(int M, int N, int K, int g, int n8, const uint8_t* Xa, const uint16_t* sxb_f16,
                         const uint8_t* packed, const uint16_t* s1_f16, uint16_t* Y_f16, int32_t* acc_debug,
                         void* workspace, size_t ws_bytes, qoq_stream_t stream) {
  if (!Xa || !sxb_f16 || !packed || !s1_f16 || !Y_f16) return QOQ_ERR_NULL;
  if (!shape_ok_mk(M, K) || !shape_ok_nk(N, K)) return QOQ_ERR_SHAPE;
  if (!qoq::group_size_ok(K, g) || n8 < 0 || n8 > K / kGroup) return QOQ_ERR_UNSUPPORTED;
  if (!aligned16(Xa) || !aligned16(sxb_f16) || !aligned16(packed) || !aligned16(s1_f16) || !aligned16(Y_f16) ||
      (acc_debug && !aligned16(acc_debug)))
    return QOQ_ERR_MISALIGNED;
  if (!workspace || ws_bytes < qoq_w4ax_workspace_bytes(M, N, K, g)) return QOQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QOQ_ERR_MISALIGNED;
  int sms = 0;
  qoq_status st = device_info(&sms);
  if (st != QOQ_OK) return st;
  unsigned long long tmo = g_timeout_ns.load();
  if (tmo == 0) tmo = kDefaultTimeoutNs;
  unsigned call_id = g_call_id.fetch_add(2) + 1;  // two ids: the W4Ax launch and the integer-sum launch
  if (call_id == 0 || call_id + 1 == 0) call_id = g_call_id.fetch_add(2) + 1;
  return from_cuda(qoq::launch_w4ax(M, N, K, g, n8, Xa, sxb_f16, packed, s1_f16, Y_f16, acc_debug, workspace, sms,
                                    tmo, call_id, reinterpret_cast<cudaStream_t>(stream)));
}

qoq_status qoq_unpack_weights_debug(int N, int K, int g, const uint8_t* packed, uint8_t* q4,
                                    uint8_t* s2, uint8_t* z, qoq_stream_t stream) {
  if (!packed || !q4 || !s2 || !z) return QOQ_ERR_NULL;
  if (!shape_ok_nk(N, K)) return QOQ_ERR_SHAPE;
  if (!qoq::group_size_ok(K, g)) return QOQ_ERR_UNSUPPORTED;
  if (!aligned16(packed)) return QOQ_ERR_MISALIGNED;
  qoq_status st = device_info(nullptr);
  if (st != QOQ_OK) return st;
  return from_cuda(qoq::launch_unpack(N, K, g, packed, q4, s2, z, reinterpret_cast<cudaStream_t>(stream)));
}

qoq_status qoq_last_device_status(void* workspace, qoq_stream_t stream) {
  if (!workspace) return QOQ_ERR_NULL;
  if (!aligned16(workspace)) return QOQ_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int host[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(host, workspace, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return from_cuda(e);
  e = cudaMemsetAsync(workspace, 0, sizeof(int), s);  // the sticky status word
  if (e != cudaSuccess) return from_cuda(e);
  return host[0] == 0 ? QOQ_OK : (host[0] == QOQ_ERR_DEVICE_TIMEOUT ? QOQ_ERR_DEVICE_TIMEOUT : QOQ_ERR_CUDA);
}

qoq_status qoq_set_debug(uint64_t wait_timeout_ns, int fault) {
  if (fault < 0 || fault > 1) return QOQ_ERR_UNSUPPORTED;
  g_timeout_ns.store(wait_timeout_ns);
  g_fault.store(fault);
  return QOQ_OK;
}

#ifdef QOQ_TRACE
// Trace builds only: device buffer of (grid size x kTraceSlots) uint64 that
// the next GEMM launches fill with pipeline event clocks (NULL disables).
void qoq_debug_set_trace(void* device_buffer) {
  g_trace.store(static_cast<unsigned long long*>(device_buffer));
}
#endif

}  // extern "C"
