// internal.h -- layout constants, the GEMM schedule and the kernel launchers
// shared by the translation units of libqoq.so (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace qoq {

// ---------------------------------------------------------------- layouts --
constexpr int kGroup = 128;        // input channels per k-tile (the GEMM's unit of K)
constexpr int kTileN = 128;        // output channels per packed tile / MMA M
constexpr int kWChunkBytes = 2048; // one 32-channel chunk for all 128 rows

// Level-2 group size g: 32, 64, or a multiple of 128 dividing K.  A packed
// k-tile (128 rows x 128 channels) holds GPT = max(1, 128 / g) scale sets of
// s2[128] + z[128] (for g > 128, a group's s2 and z are repeated in each of
// its k-tiles), then the four 32-channel code chunks.
inline bool group_size_ok(int K, int g) {
  return g == 32 || g == 64 || (g >= kGroup && g % kGroup == 0 && K % g == 0);
}
inline int gpt_for_group(int g) { return g >= kGroup ? 1 : kGroup / g; }
__host__ __device__ constexpr int w_nib_offset(int gpt) { return 256 * gpt; }
__host__ __device__ constexpr int w_tile_bytes(int gpt) { return w_nib_offset(gpt) + 4 * kWChunkBytes; }
constexpr int kWTileBytes = w_tile_bytes(1);  // g >= 128: 8448 bytes
constexpr int kFoldGroups = 8;     // fp32 TMEM partials are folded to int32 every 8 groups
                                   // (1024 channels: 127*127*1024 < 2^24, exact in fp32)
constexpr int kFoldGroupsZf = 4;   // the zero-point-folded variant's operand q4 * s2 reaches 240:
                                   // every 4 groups (512 channels: 240*127*512 < 2^24)
constexpr int kMaxSkTiles = 512;   // upper bound of split-K tiles per call (workspace sizing)
constexpr int kMaxGrid = 160;      // upper bound of persistent CTAs per call (GB300: 152 SMs)

// Workspace header, 32-bit words: [0] sticky status, [1] id of a call that
// aborted, [2] hand-off epoch of the decode kernel (advanced by the last CTA
// of every decode launch), [3] that kernel's CTA exit counter.
constexpr int kWsHeaderBytes = 256;
constexpr int kWsEpochWord = 2;
constexpr int kWsExitWord = 3;

// Token-tile width (MMA N) used for a given M.
inline int gemm_bn_for_m(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace partition for (M, N, K); device independent.
//   token tiles of <= 64 (one tile): header, then one split-K slot per CTA
//     ([BN][128] entries of {int32 partial sum, uint32 epoch tag});
//   128-token tiles: header, split-K tile counters, int32 partial tiles, and
//     the fp16 B-operand copy of Xq.
// Both end with the per-k-tile row sums of Xq that the zero-point-folded
// variant subtracts in its epilogue: int32 [K/128][rs_ld], rs_ld = M rounded
// up to a multiple of 4 (rewritten by every call of that variant).
// Zero-start state: the header's status words and [cnt_off, zero_bytes)
// (empty for decode-sized calls, whose split-K entries carry epoch tags).
struct WsLayout {
  size_t cnt_off, acc_off, slot_off, xh_off, rs_off, zero_bytes, total;
  int rs_ld;
};

// Every region a decode-sized call (M <= 64) can touch lies below
// kDecodeArea: the header, its split-K slots (at most kMaxGrid x 64 x 128
// entries of 8 bytes) and its row sums (at most 1024 k-tiles x 64 tokens of 4
// bytes).  The 128-token-tile layout starts its zero-start state above it, so
// calls of both kinds can share a workspace without clearing anything.
constexpr size_t kDecodeArea = kWsHeaderBytes + (size_t)kMaxGrid * 64 * kTileN * 8 + (size_t)1024 * 64 * 4;

inline WsLayout gemm_ws_layout(int M, int N, int K) {
  const int BN = gemm_bn_for_m(M);
  const long long MT = (M + BN - 1) / BN;
  const long long T = MT * (N / kTileN);
  const long long skmax = T < kMaxSkTiles ? T : kMaxSkTiles;
  WsLayout L;
  L.rs_ld = (M + 3) / 4 * 4;
  const size_t rs_bytes = (size_t)(K / kGroup) * L.rs_ld * 4;
  if (BN <= 64) {
    L.acc_off = 0;  // unused
    L.slot_off = kWsHeaderBytes;
    L.xh_off = align_up(L.slot_off + (size_t)kMaxGrid * BN * kTileN * 8, 1024);  // no B copy: end of slots
    L.rs_off = L.xh_off;
    L.cnt_off = L.zero_bytes = kWsHeaderBytes;
    L.total = align_up(L.rs_off + rs_bytes, 256);
    return L;
  }
  L.slot_off = 0;  // unused
  L.cnt_off = align_up(kDecodeArea, 1024);
  L.acc_off = align_up(L.cnt_off + (size_t)skmax * 4, 256);
  L.xh_off = align_up(L.acc_off + (size_t)skmax * BN * kTileN * 4, 1024);
  L.rs_off = align_up(L.xh_off + (size_t)MT * K * BN * 2, 256);
  L.zero_bytes = L.xh_off;
  L.total = align_up(L.rs_off + rs_bytes, 256);
  return L;
}

// --------------------------------------------------------------- schedule --
// Tiles: tile t -> weight tile nt = t / MT, token tile mt = t % MT.
// Split-K state lives in the workspace.  128-token tiles: int32 sums and
// counts that every completed call leaves zeroed (the last contributor clears
// them).  Decode tiles: each CTA's slot holds its partial sums tagged with the
// launch's epoch, read from the workspace header on the device, so a launch
// replayed from a CUDA graph gets a fresh tag too and stale entries never
// need clearing.
// Tiles [0, T_dp) are processed whole, round-robin over the P CTAs; the
// remaining T_sk tiles are split along K: their T_sk * G group-iterations are
// cut into P equal contiguous ranges (stream-K), and partial int32 sums meet
// in the workspace, where the last contributor of a tile writes the output.
struct GemmParams {
  const uint8_t* packed;
  const uint16_t* xh;  // tiled fp16 copy of Xq (B operand layout), 128-token tiles
  const int8_t* xq;    // Xq itself, read directly for token tiles of <= 64 rows
  const uint16_t* sx;
  const uint16_t* s1;
  uint16_t* Y;
  int32_t* acc_debug;
  int32_t* sk_acc;  // [T_sk][BN][128]  (128-token tiles)
  int32_t* sk_cnt;  // [T_sk]           (128-token tiles)
  unsigned long long* sk_slot;  // [P][BN][128] {int32 partial, uint32 epoch tag} (decode tiles)
  int* status;      // workspace header
  int M, N, K, G, MT, NT, T, T_dp, T_sk, P;  // G: k-tiles (K / 128)
  int gpt;                                    // scale sets per k-tile (the kernel's template argument)
  uint32_t I_sk;  // T_sk * G <= 511 * 1024, so 32-bit schedule arithmetic suffices
  unsigned long long timeout_ns;
  int fault;
  unsigned call_id;           // non-zero: the abort word names the aborting call (not a hand-off tag)
  unsigned long long* trace;  // per-CTA event clock, only with -DQOQ_TRACE (else unused)
  const int32_t* rs;          // zero-point-folded variant: row sums of Xq per k-tile, [G][rs_ld]
  int rs_ld;
  const uint16_t* sxT;        // W4Ax: activation block scales by block, [G][sxT_ld] fp16 (0 past M)
  int sxT_ld;
};

// Event tracing for pipeline studies: compiled in only with -DQOQ_TRACE.
// Per CTA kTraceSlots 64-bit slots of %globaltimer (ns, common to all warps):
// [0], [1] start, [2] end, [3] dependency wait passed (decode dequant);
// producer issue of group i at 16+i; MMA issue at 128+i; dequant slice load,
// stage full, start, end (quadrant 0 of the group's slot) at 192+i, 320+i,
// 256+i, 384+i; epilogue chunk ready/folded at 512+c / 576+c; unit done at
// 640+u; per-warp final barrier arrive/depart at 700+2w / 701+2w; MMA warp
// group start/end at 800+i / 900+i; decode A tile stored / slot barrier
// passed at 832+i / 896+i; split-K hand-off steps at 960+4u+{0,1,2}.
constexpr int kTraceSlots = 1024;
#ifdef QOQ_TRACE
#define QOQ_TRACE_AT(p, slot, value)                                                     \
  do {                                                                                    \
    if ((p).trace && (slot) < kTraceSlots) {                                              \
      (void)(value);                                                                      \
      unsigned long long qoq_t_;                                                          \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(qoq_t_));                         \
      (p).trace[(size_t)blockIdx.x * kTraceSlots + (slot)] = qoq_t_;                      \
    }                                                                                     \
  } while (0)
#else
#define QOQ_TRACE_AT(p, slot, value) \
  do {                               \
  } while (0)
#endif

// split: the CTA-pair layout, each [128][128] token x channel block stored as
// two [64][128] halves (tokens 0..63, then 64..127), each [2][64][64] (the
// 64-channel halves), so that each CTA of a pair copies its half in one piece.
struct ConvertParams {
  const int8_t* Xq;
  uint16_t* xh;
  int M, K, BN, MT;
  int split;
};

// W4Ax activations (mixed 8-bit / 4-bit 128-channel blocks, n8 leading 8-bit
// blocks) -> the fp16 B-operand copy and the transposed block scales.
struct ConvertAxParams {
  const uint8_t* Xa;
  const uint16_t* sxb;  // [M][G]
  uint16_t* xh;
  uint16_t* sxT;        // [G][sxT_ld]
  int M, K, n8, MT, sxT_ld;
};

// Workspace of qoq_w4ax_gemm: the 128-token-tile layout for any M, then the
// transposed block scales, fp16 [K/128][MT * 128].
inline WsLayout w4ax_ws_layout(int M, int N, int K) {
  const int MT = (M + 127) / 128;
  const long long T = (long long)MT * (N / kTileN);
  const long long skmax = T < kMaxSkTiles ? T : kMaxSkTiles;
  WsLayout L;
  L.slot_off = 0;  // unused
  L.cnt_off = kWsHeaderBytes;
  L.acc_off = align_up(L.cnt_off + (size_t)skmax * 4, 256);
  L.xh_off = align_up(L.acc_off + (size_t)skmax * 128 * kTileN * 4, 1024);
  L.rs_off = align_up(L.xh_off + (size_t)MT * K * 128 * 2, 256);  // here: the block scales
  L.rs_ld = MT * 128;
  L.zero_bytes = L.xh_off;
  L.total = align_up(L.rs_off + (size_t)(K / kGroup) * L.rs_ld * 2, 256);
  return L;
}

// Row sums of Xq per 128-channel k-tile, for the zero-point-folded variant.
struct RowSumParams {
  const int8_t* Xq;
  int32_t* rs;  // [K/128][rs_ld]
  int M, K, rs_ld;
};

// Launch attribute for programmatic dependent launch: the kernel may start
// before the preceding kernel on the stream has finished, once that kernel
// has triggered (griddepcontrol.launch_dependents) or exited; it must execute
// griddepcontrol.wait before touching anything the preceding kernels write
// or read.
inline cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// ---------------------------------------------------------------- launchers --
cudaError_t launch_act_quant(int M, int K, const uint16_t* X, int8_t* Xq, uint16_t* sx,
                             cudaStream_t s);
cudaError_t launch_norm_quant(int M, int K, int kind, float eps, const uint16_t* X, const uint16_t* gamma,
                              const uint16_t* beta, int8_t* Xq, uint16_t* sx, cudaStream_t s);
cudaError_t launch_pack(int N, int K, int g, const uint16_t* W, uint8_t* packed, uint16_t* s1,
                        cudaStream_t s);
cudaError_t launch_act_quant_w4ax(int M, int K, int n8, const uint16_t* X, uint8_t* Xa, uint16_t* sxb,
                                  cudaStream_t s);
cudaError_t launch_unpack(int N, int K, int g, const uint8_t* packed, uint8_t* q4, uint8_t* s2, uint8_t* z,
                          cudaStream_t s);
cudaError_t launch_gemm_decode(const GemmParams& p, int BN, bool zero_folded, cudaStream_t s);
// The W4Ax GEMM (mixed 4/8-bit activation blocks, per-block scales): always
// the 128-token-tile kernel; with acc_debug a second launch of the plain
// kernel on the same operand copy writes sum_b acc_b.
cudaError_t launch_w4ax(int M, int N, int K, int g, int n8, const uint8_t* Xa, const uint16_t* sxb,
                        const uint8_t* packed, const uint16_t* s1, uint16_t* Y, int32_t* acc_debug, void* ws,
                        int num_sms, unsigned long long timeout_ns, unsigned call_id, cudaStream_t s);
// zero_folded: the variant that feeds q4 * s2 to the tensor cores and
// subtracts the zero points' share, sum_j z s2 RS[m, j], in the epilogue
// (g >= 128 only); it first launches the row-sum pre-pass.
cudaError_t launch_gemm(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx,
                        const uint8_t* packed, const uint16_t* s1, uint16_t* Y, int32_t* acc_debug,
                        void* ws, int num_sms, unsigned long long timeout_ns, int fault,
                        unsigned call_id, unsigned long long* trace, bool zero_folded, cudaStream_t s);

}  // namespace qoq
