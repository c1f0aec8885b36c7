// gemm.cu -- the W4A8 g128 GEMM on sm_103a tensor cores.
//
// Computes, for Xq [M][K] int8 (per-token scale s_x) and the packed weights
// (level-2 codes q4, integer scale s2, zero z per 128-channel group; level-1
// fp16 scale s1 per output channel):
//   acc[m,n] = sum_k Xq[m,k] * ((q4[n,k] - z[n,k/128]) * s2[n,k/128])   (exact)
//   Y[m,n]   = fp16_rn(float(acc) * (float(s_x[m]) * float(s1[n])))
// QServe talk write-up, "Quantized Matrix Multiplication (GEMM) Kernel on
// GPUs" and "Challenges and Design Details": the 4-bit weights are
// dequantized to 8-bit integers before the tensor cores (never partial-sum
// dequant), the main loop is tensor-core work only, and the per-channel
// scales go to the epilogue.  Lecture 15 notes, section 15.5: the dequant
// instruction count per weight is what decides whether the weight stream can
// reach the HBM floor.
//
// sm_103a has no integer tcgen05 MMA, so the exact int8 x int8 product runs on
// tcgen05.mma kind::f16: both operands are small integers times a power of
// two, exact in fp16; each product and each partial sum below 2^24 units is
// exact in the fp32 accumulator, and the epilogue folds the fp32 TMEM partials
// into int32 every 8 groups (1024 channels, 127*127*1024 < 2^24).
//
// Data path per CTA (one persistent CTA per SM, warp-specialised):
//   warp 0      producer: per 128-channel group, one bulk copy of the packed
//               weight tile (8448 B) and the activation tile into an S-stage
//               ring: for token tiles of <= 64 rows the int8 Xq tile by 2D TMA
//               (converted to fp16 in shared memory by the dequant warps), for
//               128-row tiles a pre-swizzled fp16 tile made by convert_kernel.
//   warps 2..   dequant: NSLOT slots of 4 warps (one per TMEM lane quadrant);
//               slot j takes every NSLOT-th group, so NSLOT groups are in
//               flight.  Thread r owns weight row r of the tile and expands its
//               64 code bytes to 128 fp16 values with one mask and one packed
//               FMA per pair (see dequant_pair), storing them straight into
//               tensor memory (tcgen05.st): the MMA's A operand.  Dequantized
//               weights never touch shared memory.
//   warp 1      MMA issuer: 8 x tcgen05.mma (M=128, N=BN, K=16) per group, A
//               from TMEM, B from shared memory, D in one of two TMEM
//               accumulators (double-buffered per fold chunk).  The warp stays
//               converged and one elected lane issues: a diverged single
//               thread issues tcgen05 ops about 2.5x slower, and each mbarrier
//               wait costs ~100 cycles even when the phase is complete, so the
//               loop waits once per group.
//   last NEPI   epilogue: sum the R chains, fold fp32 to int32, then write Y
//               (whole-K tiles) or add int32 partials into the workspace
//               (split-K tiles; the last contributor writes Y and clears them).
// Every mbarrier wait is bounded; on expiry the CTA records
// QOQ_ERR_DEVICE_TIMEOUT in the workspace header, drains its copies and MMAs,
// frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace qoq {
namespace {

constexpr int kTmemCols = 512;
constexpr int kACol0 = 256;  // A buffers: TMEM columns 256 + 64 a
constexpr int kNABuf = 4;
constexpr int kStatusTimeout = 7;  // QOQ_ERR_DEVICE_TIMEOUT
// The A operand carries w8 * 2^-13 (see dequant_pair); the epilogue undoes it.
constexpr float kAccScale = 8192.0f;
constexpr int kSmemBudget = 228 * 1024;

template <int BN>
struct Cfg {
  static constexpr bool IN_KERNEL_B = BN <= 64;  // int8 tile by TMA, fp16 made in shared memory
  static constexpr int R = 1;                                   // accumulator chains per set
  static constexpr int ACC_COLS = R * BN;                       // TMEM columns per accumulator set
  static constexpr int NACC = 2;                                // accumulator sets (double buffer)
  static constexpr int NSLOT = BN <= 32 ? 3 : 2;               // groups dequantized concurrently
  static constexpr int NDQ = 4 * NSLOT;                        // dequant warps
  static constexpr int NEPI = BN == 128 ? 16 : (BN == 64 ? 8 : 4);  // epilogue warps
  static constexpr int EPI_TOK = BN / (NEPI / 4);              // tokens per epilogue thread
  static constexpr int WARPS = 2 + NDQ + NEPI;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int EPI_WARP0 = 2 + NDQ;
  static constexpr int B_BYTES = BN * kGroup * 2;               // fp16 B tile per group
  static constexpr int X8_BYTES = IN_KERNEL_B ? BN * kGroup : 0; // int8 staging per group
  static constexpr int STAGE_BYTES = B_BYTES + X8_BYTES + kWTileBytes;
  static constexpr int STAGES_FIT = (kSmemBudget - 2048) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 16 ? 16 : STAGES_FIT;
  static constexpr int B_OFF = 0;
  static constexpr int X8_OFF = STAGES * B_BYTES;
  static constexpr int W_OFF = X8_OFF + STAGES * X8_BYTES;
  static constexpr int BAR_OFF = W_OFF + STAGES * kWTileBytes;
  static constexpr int NBARS = 2 * STAGES + 2 * kNABuf + 2 * NACC + 1;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int FLAG_OFF = TMEM_SLOT_OFF + 8;
  static constexpr int SMEM_BYTES = FLAG_OFF + 8 + 1024;  // + slack for 1024-B alignment
  // tcgen05 instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B
  // fp16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0),
  // N >> 3 in bits 17-22, M >> 4 in bits 24-28.
  static constexpr uint32_t IDESC =
      (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kTileN >> 4) << 24);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert(8 % R == 0, "chains divide the 8 K-steps of a group");
  static_assert(NACC * ACC_COLS <= kACol0, "accumulators overlap A buffers");
  static_assert(kNABuf >= NSLOT + 1, "A buffers");
  static_assert(B_BYTES % 1024 == 0 && X8_BYTES % 1024 == 0, "1024-B aligned tiles");
  static_assert(EPI_TOK % 16 == 0, "epilogue loads 16 columns at a time");
  static_assert(STAGES >= 3, "pipeline depth");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Exact dequant of a pair of 4-bit codes (QServe "subtraction after
// multiplication": the zero point enters after the scale, as one packed FMA).
// `h` holds the two codes q in the same 4-bit field of each fp16 half, at bit
// p (p = 0 or 4) and nothing else, i.e. the fp16 subnormals q * 2^(p-24).
// With sc = s2 * 2^(11-p) and c = -(z * s2) * 2^-13 (both exact in fp16),
//   fma(h, sc, c) = (q - z) * s2 * 2^-13
// computed exactly then rounded once; the result is representable (|.| <= 240
// units of 2^-13, and every non-zero value is a normal fp16), so it is exact.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t h, uint32_t sc, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(h), "r"(sc), "r"(c));
  return d;
}

// Four int8 lanes of `x` -> two fp16x2 (exact): the biased byte u = b ^ 0x80
// becomes the fp16 1024 + u through its mantissa, and 1024 + 128 is removed.
__device__ __forceinline__ void int8x4_to_half2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = x ^ 0x80808080u;
  const uint32_t bias = 0x64806480u;  // fp16 (1152, 1152)
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

// Shared-memory matrix descriptor: 128-byte swizzle, K-major, 8-row groups
// 1024 B apart (SBO), version 1 (bit 46), layout code 2 (bits 61-63).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

struct Unit {
  int tile, g0, g1;
};

// The CTA's sequence of (tile, group range) units: whole tiles first, then
// its stream-K range.  Every role walks the same sequence.
struct UnitIter {
  int dp_next;
  long long it, it_end;
  __device__ __forceinline__ void init(const GemmParams& p) {
    dp_next = blockIdx.x;
    it = (long long)blockIdx.x * p.I_sk / p.P;
    it_end = (long long)(blockIdx.x + 1) * p.I_sk / p.P;
  }
  __device__ __forceinline__ bool next(const GemmParams& p, Unit& u) {
    if (dp_next < p.T_dp) {
      u.tile = dp_next;
      u.g0 = 0;
      u.g1 = p.G;
      dp_next += p.P;
      return true;
    }
    if (it < it_end) {
      const long long sk = it / p.G;
      const int g0 = (int)(it - sk * p.G);
      const long long rem = it_end - it;
      const long long g1 = rem < (long long)(p.G - g0) ? g0 + rem : (long long)p.G;
      u.tile = p.T_dp + (int)sk;
      u.g0 = g0;
      u.g1 = (int)g1;
      it += g1 - g0;
      return true;
    }
    return false;
  }
};

// Bounded wait on an mbarrier phase.  Returns false if the wait ran out (the
// timeout is recorded) or, when honor_abort, if another thread of this call
// already recorded one.  The loop polls only the barrier for the first ~100k
// cycles; the global timer and the abort word in global memory are read after
// that, so a normal hand-off never waits behind a global load.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const GemmParams& p,
                                       bool honor_abort) {
  volatile unsigned* abort_word = reinterpret_cast<volatile unsigned*>(p.status + 1);
  const long long c0 = clock64();
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 0 && clock64() - c0 > 100000) {
      const uint64_t now = global_timer_ns();
      if (t0 == 0) t0 = now;
      if (honor_abort && *abort_word == p.call_id) return false;
      if (now - t0 > p.timeout_ns) {
        atomicExch(p.status, kStatusTimeout);
        atomicExch(reinterpret_cast<unsigned*>(p.status + 1), p.call_id);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const GemmParams& p,
                                         bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, p, honor_abort);
}

template <int NTHREADS>
__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory");
}

// Y[m, n] for the COLS tokens m = m0 .. m0+COLS-1 held by this thread.
template <int COLS>
__device__ __forceinline__ void write_tile_out(const GemmParams& p, const int32_t (&run)[COLS], int m0,
                                               int n) {
  const float s1f = __half2float(__ushort_as_half(p.s1[n]));
#pragma unroll
  for (int i = 0; i < COLS; ++i) {
    const int m = m0 + i;
    if (m < p.M) {
      const float sxf = __half2float(__ushort_as_half(p.sx[m]));
      const float y = (float)run[i] * (sxf * s1f);
      p.Y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(y));
      if (p.acc_debug) p.acc_debug[(size_t)m * p.N + n] = run[i];
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(Cfg<BN>::THREADS, 1)
    gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap xmap) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + C::BAR_OFF;
  const uint32_t bar_full = bars, bar_empty = bars + 8 * C::STAGES;
  const uint32_t bar_afull = bars + 8 * (2 * C::STAGES), bar_aempty = bar_afull + 8 * kNABuf;
  const uint32_t bar_accfull = bar_aempty + 8 * kNABuf, bar_accempty = bar_accfull + 8 * C::NACC;
  const uint32_t bar_drain = bar_accempty + 8 * C::NACC;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1 + 4);  // MMA commit + the 4 warps of one dequant slot
    }
    for (int a = 0; a < kNABuf; ++a) {
      mbar_init(bar_afull + 8 * a, 4);
      mbar_init(bar_aempty + 8 * a, 1);
    }
    for (int b = 0; b < C::NACC; ++b) {
      mbar_init(bar_accfull + 8 * b, 1);
      mbar_init(bar_accempty + 8 * b, C::NEPI);
    }
    mbar_init(bar_drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(sbase + C::TMEM_SLOT_OFF, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::TMEM_SLOT_OFF);
  if (threadIdx.x == 0) {
    QOQ_TRACE_AT(p, 0, 0);
    QOQ_TRACE_AT(p, 1, 0);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      const uint64_t pol_w = p.MT == 1 ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_x = policy_evict_last();
      if (C::IN_KERNEL_B) prefetch_tensormap(&xmap);
      UnitIter iter;
      iter.init(p);
      Unit u;
      bool have = iter.next(p, u);
      int g = have ? u.g0 : 0;
      uint32_t issued_mask = 0, issued_par = 0;  // per stage: last issue and its parity
      constexpr uint32_t kStageTx = kWTileBytes + (C::IN_KERNEL_B ? C::X8_BYTES : C::B_BYTES);
      auto issue_w = [&](int s, int tile, int gg) {
        const uint8_t* src = p.packed + ((size_t)(tile / p.MT) * p.G + gg) * kWTileBytes;
        bulk_g2s(sbase + C::W_OFF + s * kWTileBytes, src, kWTileBytes, bar_full + 8 * s, pol_w);
      };
      auto issue_x = [&](int s, int tile, int gg) {
        const int mt = tile % p.MT;
        if (C::IN_KERNEL_B) {
          tma_load_2d(sbase + C::X8_OFF + s * C::X8_BYTES, &xmap, gg * kGroup, mt * BN, bar_full + 8 * s,
                      pol_x);
        } else {
          const uint16_t* src = p.xh + ((size_t)mt * p.G + gg) * (C::B_BYTES / 2);
          bulk_g2s(sbase + C::B_OFF + s * C::B_BYTES, src, C::B_BYTES, bar_full + 8 * s, pol_x);
        }
      };
      // Weights do not depend on the preceding kernels (activation quant,
      // B-operand convert): stream the first ring's worth before waiting on them.
      int npre = 0;
      int pre_tile[C::STAGES], pre_g[C::STAGES];
      while (have && npre < C::STAGES) {
        const int s = npre;
        mbar_arrive_expect_tx(bar_full + 8 * s, kStageTx);
        issue_w(s, u.tile, g);
        QOQ_TRACE_AT(p, 16 + npre, 0);
        pre_tile[npre] = u.tile;
        pre_g[npre] = g;
        issued_mask |= 1u << s;
        ++npre;
        if (++g >= u.g1) {
          have = iter.next(p, u);
          if (have) g = u.g0;
        }
      }
      grid_dep_wait();
      for (int i = 0; i < npre; ++i) issue_x(i, pre_tile[i], pre_g[i]);
      uint32_t gi = npre;
      while (have) {
        const int s = gi % C::STAGES;
        const uint32_t ph = (gi / C::STAGES) & 1;
        if (!wait_bar(bar_empty + 8 * s, ph ^ 1, p)) break;
        if (!(p.fault == 1 && gi == (uint32_t)C::STAGES + 1)) {  // test hook: skip one stage
          mbar_arrive_expect_tx(bar_full + 8 * s, kStageTx);
          issue_w(s, u.tile, g);
          issue_x(s, u.tile, g);
          QOQ_TRACE_AT(p, 16 + (int)gi, 0);
          issued_mask |= 1u << s;
          issued_par = (issued_par & ~(1u << s)) | (ph << s);
        } else {
          issued_mask &= ~(1u << s);
        }
        ++gi;
        if (++g >= u.g1) {
          have = iter.next(p, u);
          if (have) g = u.g0;
        }
      }
      // Let every copy still in flight land before the CTA may exit.
      for (int s = 0; s < C::STAGES; ++s)
        if (issued_mask & (1u << s)) wait_bar(bar_full + 8 * s, (issued_par >> s) & 1, p, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer --
    // The whole warp walks the loop; lane 0 waits and broadcasts the outcome,
    // one elected lane issues the MMAs and commits.
    grid_dep_wait();
    UnitIter iter;
    iter.init(p);
    Unit u;
    uint32_t gi = 0, chunk = 0;
    bool ok = true;
    while (ok && iter.next(p, u)) {
      for (int c0 = u.g0; c0 < u.g1; c0 += kFoldGroups) {
        const int c1 = min(u.g1, c0 + kFoldGroups);
        const int b = chunk % C::NACC;
        int w_ok = 1;
        if (lane == 0) w_ok = wait_bar(bar_accempty + 8 * b, ((chunk / C::NACC) & 1) ^ 1, p);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_base = tmem + b * C::ACC_COLS;
        for (int g = c0; g < c1; ++g, ++gi) {
          const int s = gi % C::STAGES;
          const int a = gi % kNABuf;
          // the dequant slot of this group waited for the stage's copies before
          // arriving, so A-full also means the B tile is in shared memory
          if (lane == 0) w_ok = wait_bar(bar_afull + 8 * a, (gi / kNABuf) & 1, p);
          if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) QOQ_TRACE_AT(p, 128 + (int)gi, 0);
          const uint32_t b_base = sbase + C::B_OFF + s * C::B_BYTES;
          if (lane == 0) QOQ_TRACE_AT(p, 800 + (int)gi, 0);
          if (elect_one()) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t b_addr = b_base + (j >> 2) * (BN * 128) + (j & 3) * 32;
              const int r = j % C::R;
              tc_mma_ts(d_base + r * BN, tmem + kACol0 + a * 64 + 8 * j, desc_sw128(b_addr), C::IDESC,
                        (g > c0 || j >= C::R) ? 1u : 0u);
            }
            tc_commit(bar_empty + 8 * s);
            tc_commit(bar_aempty + 8 * a);
          }
          __syncwarp();
          if (lane == 0) QOQ_TRACE_AT(p, 900 + (int)gi, 0);
        }
        if (!ok) break;
        if (elect_one()) tc_commit(bar_accfull + 8 * b);
        __syncwarp();
        ++chunk;
      }
    }
    // all MMAs issued by this warp complete before TMEM is released
    if (elect_one()) tc_commit(bar_drain);
    __syncwarp();
    if (lane == 0) wait_bar(bar_drain, 0, p, false);
    __syncwarp();
  } else if (warp < C::EPI_WARP0) {
    // ------------------------------------------------------------- dequant --
    grid_dep_wait();
    const int quad = warp & 3;
    const int slot = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const int stid = ((warp - 2) & 3) * 32 + lane;  // 0..127 within the slot
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    UnitIter iter;
    iter.init(p);
    Unit u;
    uint32_t gi = 0;
    bool ok = true;
    while (ok && iter.next(p, u)) {
      for (int g = u.g0; g < u.g1; ++g, ++gi) {
        if ((int)(gi % C::NSLOT) != slot) continue;
        const int s = gi % C::STAGES;
        const int a = gi % kNABuf;
        if (!wait_bar(bar_full + 8 * s, (gi / C::STAGES) & 1, p) ||
            !wait_bar(bar_aempty + 8 * a, ((gi / kNABuf) & 1) ^ 1, p)) {
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read this A buffer are complete
        if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 256 + (int)gi, 0);
        if (C::IN_KERNEL_B) {
          // int8 [BN][128] tile -> fp16 B operand: two [BN][64] 128B-swizzled halves
          const uint8_t* x8 = smem + C::X8_OFF + s * C::X8_BYTES;
          uint8_t* bt = smem + C::B_OFF + s * C::B_BYTES;
#pragma unroll
          for (int i = 0; i < BN / 16; ++i) {
            const int q = stid + i * 128;  // 16-byte int8 chunk: row q / 8, channels 16 (q % 8) ..
            const int r = q >> 3, kc = q & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(x8 + q * 16);
            uint32_t h[8];
            int8x4_to_half2x2(v.x, h[0], h[1]);
            int8x4_to_half2x2(v.y, h[2], h[3]);
            int8x4_to_half2x2(v.z, h[4], h[5]);
            int8x4_to_half2x2(v.w, h[6], h[7]);
            const int c = 2 * (kc & 3);  // first 16-byte fp16 chunk inside the 64-channel half
            uint8_t* line = bt + (kc >> 2) * (BN * 128) + r * 128;
            *reinterpret_cast<uint4*>(line + ((c ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(line + (((c + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
          }
          fence_proxy_async_smem();  // generic-proxy writes -> the MMA's async-proxy reads
        }
        const uint8_t* wt = smem + C::W_OFF + s * kWTileBytes;
        const uint32_t s2 = wt[row], z = wt[128 + row];
        // sc0 = s2 * 2^11 (codes at bit 0), sc4 = s2 * 2^7 (codes at bit 4),
        // c = -(z * s2) * 2^-13; all exact in fp16 (s2 <= 16, z * s2 <= 240)
        const uint32_t sc0 = (uint32_t)__half_as_ushort(__float2half_rn((float)(s2 << 11))) * 0x00010001u;
        const uint32_t sc4 = (uint32_t)__half_as_ushort(__float2half_rn((float)(s2 << 7))) * 0x00010001u;
        const uint32_t cz =
            (uint32_t)__half_as_ushort(__float2half_rn(-(float)(z * s2) * (1.0f / 8192.0f))) * 0x00010001u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(wt + kWNibOffset + c * kWChunkBytes + row * 16);
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
          uint32_t out[16];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t x = wv[w], y = wv[w] >> 8;
            out[4 * w + 0] = dequant_pair(x & 0x000F000Fu, sc0, cz);  // channels 8w + 0, 1
            out[4 * w + 1] = dequant_pair(x & 0x00F000F0u, sc4, cz);  // channels 8w + 2, 3
            out[4 * w + 2] = dequant_pair(y & 0x000F000Fu, sc0, cz);  // channels 8w + 4, 5
            out[4 * w + 3] = dequant_pair(y & 0x00F000F0u, sc4, cz);  // channels 8w + 6, 7
          }
          tmem_st16(tmem + lane_base + kACol0 + a * 64 + c * 16, out);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_afull + 8 * a);
          mbar_arrive(bar_empty + 8 * s);
          if (quad == 0) QOQ_TRACE_AT(p, 384 + (int)gi, 0);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    grid_dep_wait();
    const int e = warp - C::EPI_WARP0;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int tok0 = (e >> 2) * C::EPI_TOK;  // this thread's tokens within the tile
    const int etid = threadIdx.x - C::EPI_WARP0 * 32;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::FLAG_OFF);
    UnitIter iter;
    iter.init(p);
    Unit u;
    uint32_t chunk = 0;
    int unit_no = 0;
    bool ok = true;  // once false, keep the control flow (named barriers) but do no work
    while (iter.next(p, u)) {
      const int nt = u.tile / p.MT, mt = u.tile % p.MT;
      const int n = nt * kTileN + row;
      int32_t run[C::EPI_TOK];
#pragma unroll
      for (int i = 0; i < C::EPI_TOK; ++i) run[i] = 0;
      for (int c0 = u.g0; c0 < u.g1; c0 += kFoldGroups, ++chunk) {
        const int b = chunk % C::NACC;
        if (ok) ok = wait_bar(bar_accfull + 8 * b, (chunk / C::NACC) & 1, p);
        if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 512 + (int)chunk, 0);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int r = 0; r < C::R; ++r) {
#pragma unroll
            for (int piece = 0; piece < C::EPI_TOK / 16; ++piece) {
              uint32_t v[16];
              tmem_ld16_wait(tmem + lane_base + b * C::ACC_COLS + r * BN + tok0 + piece * 16, v);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                run[piece * 16 + i] += __float2int_rn(__uint_as_float(v[i]) * kAccScale);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_accempty + 8 * b);
          if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 576 + (int)chunk, 0);
        }
      }
      if (u.g0 == 0 && u.g1 == p.G) {
        if (ok) write_tile_out<C::EPI_TOK>(p, run, mt * BN + tok0, n);
      } else {
        const int sk = u.tile - p.T_dp;
        int32_t* part = p.sk_acc + (size_t)sk * BN * kTileN + (size_t)tok0 * kTileN;
        if (ok) {
#pragma unroll
          for (int i = 0; i < C::EPI_TOK; ++i) red_add_relaxed(part + i * kTileN + row, run[i]);
        }
        // The barrier orders every epilogue thread's partial sums before one
        // thread's acq_rel count update (release is cumulative over the
        // barrier); the last contributor's acquire makes the other CTAs' sums
        // visible, and the second barrier passes that on to its warps.
        epi_bar_sync<C::NEPI * 32>();
        if (etid == 0) {
          int last = 0;
          if (ok) {
            const int add = u.g1 - u.g0;
            last = (atom_add_acq_rel(p.sk_cnt + sk, add) + add == p.G) ? 1 : 0;
            if (last) p.sk_cnt[sk] = 0;  // every contributor has counted: reset for the next call
          }
          *last_flag = last;
        }
        epi_bar_sync<C::NEPI * 32>();
        if (ok && *last_flag) {
#pragma unroll
          for (int i = 0; i < C::EPI_TOK; ++i) {
            run[i] = ld_relaxed(part + i * kTileN + row);
            part[i * kTileN + row] = 0;  // leave the workspace zeroed
          }
          write_tile_out<C::EPI_TOK>(p, run, mt * BN + tok0, n);
        }
      }
      if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 640 + unit_no, 0);
      ++unit_no;
    }
  }

  tc_fence_before();
  if (lane == 0) QOQ_TRACE_AT(p, 700 + 2 * warp, 0);
  __syncthreads();
  if (lane == 0) QOQ_TRACE_AT(p, 701 + 2 * warp, 0);
  if (threadIdx.x == 0) QOQ_TRACE_AT(p, 2, 0);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// fp16 copy of Xq in the B-operand layout for 128-token tiles: [MT][G][2][128][64]
// fp16, each [128][64] block 128B-swizzled (16-byte chunk c of row r stored at
// chunk c ^ (r & 7)), rows m >= M zero.
__global__ void __launch_bounds__(256) convert_kernel(const ConvertParams c) {
  grid_dep_launch_dependents();  // the GEMM may launch and start streaming weights
  grid_dep_wait();               // Xq comes from the preceding kernel
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int kc_per_row = c.K / 16;
  const int G = c.K / kGroup;
  const long long total = (long long)c.MT * c.BN * kc_per_row;
  for (long long idx = tid; idx < total; idx += stride) {
    const int m = (int)(idx / kc_per_row);
    const int k0 = (int)(idx % kc_per_row) * 16;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (m < c.M) raw = __ldg(reinterpret_cast<const uint4*>(c.Xq + (size_t)m * c.K + k0));
    const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      h[i] = (uint32_t)__half_as_ushort(__int2half_rn(b[2 * i])) |
             ((uint32_t)__half_as_ushort(__int2half_rn(b[2 * i + 1])) << 16);
    const int g = k0 / kGroup, kk = k0 % kGroup, half = kk / 64, chunk0 = (kk % 64) / 8;
    const int mt = m / c.BN, r = m % c.BN;
    uint16_t* blk = c.xh + ((size_t)(mt * G + g) * 2 + half) * c.BN * 64 + (size_t)r * 64;
    *reinterpret_cast<uint4*>(blk + ((chunk0 ^ (r & 7)) * 8)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(blk + (((chunk0 + 1) ^ (r & 7)) * 8)) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// Opt the kernel into its dynamic shared memory once per device (not a
// stream operation; done before any graph capture can reach it).
template <int BN>
cudaError_t set_smem_attr_once() {
  static std::mutex mu;
  static uint64_t done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && (done_mask >> dev) & 1) return cudaSuccess;
  e = cudaFuncSetAttribute(gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<BN>::SMEM_BYTES);
  if (e == cudaSuccess && dev < 64) done_mask |= 1ull << dev;
  return e;
}

cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

template <int BN>
cudaError_t launch_gemm_bn(const GemmParams& p, const CUtensorMap& xmap, cudaStream_t s) {
  using C = Cfg<BN>;
  cudaError_t e = set_smem_attr_once<BN>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.P);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BN>, p, xmap);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

// 2D map over int8 Xq [M][K]: boxes of 128 channels x BN tokens, rows past M
// read as zero.
cudaError_t make_xq_map(CUtensorMap* map, const int8_t* Xq, int M, int K, int BN) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {(cuuint32_t)kGroup, (cuuint32_t)BN};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(Xq), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm(int M, int N, int K, const int8_t* Xq, const uint16_t* sx,
                        const uint8_t* packed, const uint16_t* s1, uint16_t* Y, int32_t* acc_debug,
                        void* ws, int num_sms, unsigned long long timeout_ns, int fault,
                        unsigned call_id, unsigned long long* trace, cudaStream_t s) {
  const int BN = gemm_bn_for_m(M);
  const WsLayout L = gemm_ws_layout(M, N, K);
  GemmParams p = {};
  p.M = M;
  p.N = N;
  p.K = K;
  p.G = K / kGroup;
  p.MT = (M + BN - 1) / BN;
  p.NT = N / kTileN;
  p.T = p.MT * p.NT;
  const int P0 = std::max(1, std::min(num_sms, kMaxGrid));
  if (p.T >= P0) {
    const int rem = p.T % P0;
    p.T_sk = rem == 0 ? 0 : std::min(p.T, rem + P0);
    p.T_dp = p.T - p.T_sk;
    p.P = P0;
  } else {
    p.T_dp = 0;
    p.T_sk = p.T;
    const long long want = ((long long)p.T * p.G + 3) / 4;  // at least ~4 groups per CTA
    p.P = (int)std::max<long long>(1, std::min<long long>(P0, want));
  }
  p.I_sk = (long long)p.T_sk * p.G;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.status = reinterpret_cast<int*>(w);
  p.sk_cnt = reinterpret_cast<int32_t*>(w + L.cnt_off);
  p.sk_acc = reinterpret_cast<int32_t*>(w + L.acc_off);
  p.xh = reinterpret_cast<const uint16_t*>(w + L.xh_off);
  p.packed = packed;
  p.sx = sx;
  p.s1 = s1;
  p.Y = Y;
  p.acc_debug = acc_debug;
  p.timeout_ns = timeout_ns;
  p.fault = fault;
  p.call_id = call_id;
  p.trace = trace;

  CUtensorMap xmap;
  std::memset(&xmap, 0, sizeof(xmap));
  if (BN <= 64) {
    cudaError_t e = make_xq_map(&xmap, Xq, M, K, BN);
    if (e != cudaSuccess) return e;
  } else {
    ConvertParams c = {};
    c.Xq = Xq;
    c.xh = reinterpret_cast<uint16_t*>(w + L.xh_off);
    c.M = M;
    c.K = K;
    c.BN = BN;
    c.MT = p.MT;
    const long long work = (long long)p.MT * BN * (K / 16);
    const int cblocks = (int)std::max<long long>(1, std::min<long long>((work + 255) / 256, (long long)P0 * 4));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cblocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, convert_kernel, c);
    if (e != cudaSuccess) return e;
  }

  switch (BN) {
    case 16: return launch_gemm_bn<16>(p, xmap, s);
    case 32: return launch_gemm_bn<32>(p, xmap, s);
    case 64: return launch_gemm_bn<64>(p, xmap, s);
    default: return launch_gemm_bn<128>(p, xmap, s);
  }
}

}  // namespace qoq
