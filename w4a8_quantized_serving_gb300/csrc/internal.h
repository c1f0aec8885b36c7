// internal.h -- layout constants, the GEMM schedule and the kernel launchers
// shared by the translation units of libqoq.so (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace qoq {

// ---------------------------------------------------------------- layouts --
constexpr int kGroup = 128;        // g: input channels per level-2 group
constexpr int kTileN = 128;        // output channels per packed tile / MMA M
constexpr int kWTileBytes = 8448;  // s2[128] + z[128] + 4 chunks x 128 rows x 16 B
constexpr int kWNibOffset = 256;   // offset of the nibble chunks inside a tile
constexpr int kWChunkBytes = 2048; // one 32-channel chunk for all 128 rows
constexpr int kFoldGroups = 8;     // fp32 TMEM partials are folded to int32 every 8 groups
                                   // (1024 channels: 127*127*1024 < 2^24, exact in fp32)
constexpr int kMaxSkTiles = 512;   // upper bound of split-K tiles per call (workspace sizing)
constexpr int kMaxGrid = 256;      // upper bound of persistent CTAs per call

constexpr int kWsHeaderBytes = 256;  // [0] status, [1] abort flag

// Token-tile width (MMA N) used for a given M.
inline int gemm_bn_for_m(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace partition for (M, N, K); device independent.
struct WsLayout {
  size_t cnt_off, acc_off, xh_off, total;
};

inline WsLayout gemm_ws_layout(int M, int N, int K) {
  const int BN = gemm_bn_for_m(M);
  const long long MT = (M + BN - 1) / BN;
  const long long T = MT * (N / kTileN);
  const long long skmax = T < kMaxSkTiles ? T : kMaxSkTiles;
  WsLayout L;
  L.cnt_off = kWsHeaderBytes;
  L.acc_off = align_up(L.cnt_off + (size_t)skmax * 4, 256);
  L.xh_off = align_up(L.acc_off + (size_t)skmax * BN * kTileN * 4, 1024);
  L.total = align_up(L.xh_off + (size_t)MT * K * BN * 2, 256);
  return L;
}

// --------------------------------------------------------------- schedule --
// Tiles: tile t -> weight tile nt = t / MT, token tile mt = t % MT.
// Tiles [0, T_dp) are processed whole, round-robin over the P CTAs; the
// remaining T_sk tiles are split along K: their T_sk * G group-iterations are
// cut into P equal contiguous ranges (stream-K), and partial int32 sums meet
// in the workspace, where the last contributor of a tile writes the output.
struct GemmParams {
  const uint8_t* packed;
  const uint16_t* xh;  // tiled fp16 copy of Xq (B operand layout)
  const uint16_t* sx;
  const uint16_t* s1;
  uint16_t* Y;
  int32_t* acc_debug;
  int32_t* sk_acc;  // [T_sk][BN][128]
  int32_t* sk_cnt;  // [T_sk]
  int* status;      // workspace header
  int M, N, K, G, MT, NT, T, T_dp, T_sk, P;
  long long I_sk;
  unsigned long long timeout_ns;
  int fault;
};

struct ConvertParams {
  const int8_t* Xq;
  uint16_t* xh;
  int32_t* zero_words;  // workspace region cleared each call (header + split-K state)
  long long zero_count; // number of int32 words to clear
  int M, K, BN, MT;
};

// ---------------------------------------------------------------- launchers --
cudaError_t launch_act_quant(int M, int K, const uint16_t* X, int8_t* Xq, uint16_t* sx,
                             cudaStream_t s);
cudaError_t launch_pack(int N, int K, const uint16_t* W, uint8_t* packed, uint16_t* s1,
                        cudaStream_t s);
cudaError_t launch_unpack(int N, int K, const uint8_t* packed, uint8_t* q4, uint8_t* s2, uint8_t* z,
                          cudaStream_t s);
cudaError_t launch_gemm(int M, int N, int K, const int8_t* Xq, const uint16_t* sx,
                        const uint8_t* packed, const uint16_t* s1, uint16_t* Y, int32_t* acc_debug,
                        void* ws, int num_sms, unsigned long long timeout_ns, int fault,
                        cudaStream_t s);

}  // namespace qoq
