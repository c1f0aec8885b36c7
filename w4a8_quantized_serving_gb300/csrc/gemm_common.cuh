// gemm_common.cuh -- pieces shared by the two W4A8 GEMM kernels (the
// register-fed decode kernel for token tiles of <= 64 rows and the
// bulk-copy-fed kernel for 128-token tiles): exact dequant arithmetic, the
// work schedule, bounded waits, and the MMA-issue and epilogue roles.
//
// Exactness (QServe talk write-up, "Quantized Matrix Multiplication (GEMM)
// Kernel on GPUs": the product runs on tensor cores in 8-bit integers):
// sm_103a has no integer tcgen05 MMA, so the int8 x int8 product runs on
// tcgen05.mma kind::f16 with operands that are small integers times a power of
// two (exact in fp16).  Each product and each partial sum below 2^24 units is
// exact in the fp32 accumulator; the epilogue folds the TMEM partials into
// int32 every 8 groups (1024 channels, 127 * 127 * 1024 < 2^24).
#pragma once

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace qoq {

constexpr int kTmemCols = 512;
constexpr int kStatusTimeout = 7;  // QOQ_ERR_DEVICE_TIMEOUT
// The A operand carries w8 * 2^-13 (see dequant_pair); the epilogue undoes it.
constexpr float kAccScale = 8192.0f;
constexpr int kSmemBudget = 227 * 1024;  // per-CTA dynamic shared memory limit

// tcgen05 instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B
// fp16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28; M = 128 (one weight tile), or 256 for the
// CTA-pair MMA (one weight tile in each CTA).
__host__ __device__ constexpr uint32_t mma_idesc(int n, int m = kTileN) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

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

// Per-row constants of dequant_pair for a group with scale s2 and zero z:
// sc0 = s2 * 2^11 (codes at bit 0), sc4 = s2 * 2^7 (codes at bit 4),
// c = -(z * s2) * 2^-13, each duplicated into both fp16 halves.
struct DequantConsts {
  uint32_t sc0, sc4, cz;
};

__device__ __forceinline__ DequantConsts dequant_consts(uint32_t s2, uint32_t z) {
  DequantConsts k;
  k.sc0 = (uint32_t)__half_as_ushort(__float2half_rn((float)(s2 << 11))) * 0x00010001u;
  k.sc4 = (uint32_t)__half_as_ushort(__float2half_rn((float)(s2 << 7))) * 0x00010001u;
  k.cz = (uint32_t)__half_as_ushort(__float2half_rn(-(float)(z * s2) * (1.0f / 8192.0f))) * 0x00010001u;
  return k;
}

// 16 packed code bytes (32 channels, layout of include/qoq.h) -> 16 fp16x2
// words in channel order, ready for tcgen05.st (column c holds channels 2c, 2c+1).
__device__ __forceinline__ void dequant_chunk(const uint4& v, const DequantConsts& k, uint32_t (&out)[16]) {
  const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t x = wv[w], y = wv[w] >> 8;
    out[4 * w + 0] = dequant_pair(x & 0x000F000Fu, k.sc0, k.cz);  // channels 8w + 0, 1
    out[4 * w + 1] = dequant_pair(x & 0x00F000F0u, k.sc4, k.cz);  // channels 8w + 2, 3
    out[4 * w + 2] = dequant_pair(y & 0x000F000Fu, k.sc0, k.cz);  // channels 8w + 4, 5
    out[4 * w + 3] = dequant_pair(y & 0x00F000F0u, k.sc4, k.cz);  // channels 8w + 6, 7
  }
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

// 16 int8 activations (one 16-byte chunk: row r, channels 16 kc .. 16 kc + 15
// of a 128-channel group) -> fp16 into the B operand tile: two [BN][64]
// halves, K-major, 128-byte swizzled (16-byte chunk c of row r at c ^ (r & 7)).
__device__ __forceinline__ void store_b_chunk(uint8_t* btile, int bn, int r, int kc, const uint4& v) {
  uint32_t h[8];
  int8x4_to_half2x2(v.x, h[0], h[1]);
  int8x4_to_half2x2(v.y, h[2], h[3]);
  int8x4_to_half2x2(v.z, h[4], h[5]);
  int8x4_to_half2x2(v.w, h[6], h[7]);
  const int c = 2 * (kc & 3);  // first 16-byte fp16 chunk inside the 64-channel half
  uint8_t* line = btile + (kc >> 2) * (bn * 128) + r * 128;
  *reinterpret_cast<uint4*>(line + ((c ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(line + (((c + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
}

// Shared-memory matrix descriptor: 128-byte swizzle, K-major, 8-row groups
// 1024 B apart (SBO), version 1 (bit 46), layout code 2 (bits 61-63).
// Given as its two 32-bit halves: shared addresses stay below 2^18, so moving
// the start address by a multiple of 16 bytes is an add of (bytes >> 4) to
// the low half.
__device__ __forceinline__ uint32_t desc_sw128_lo(uint32_t saddr) { return ((saddr & 0x3FFFFu) >> 4) | (1u << 16); }
constexpr uint32_t kDescSw128Hi = (1024u >> 4) | (1u << 14) | (2u << 29);

// ------------------------------------------------------------------ schedule --

struct Unit {
  int tile, g0, g1;
};

// The CTA's sequence of (tile, group range) units: whole tiles first, then
// its stream-K range.  Every role walks the same sequence.  All quantities fit
// 32 bits (blockIdx.x * I_sk < 256 * 2^19), which keeps the divisions short.
struct UnitIter {
  int dp_next;
  uint32_t it, it_end;
  // idx: this worker's index among the p.P workers (a CTA, or a CTA pair)
  __device__ __forceinline__ void init(const GemmParams& p, uint32_t idx = blockIdx.x) {
    dp_next = (int)idx;
    it = idx * p.I_sk / (uint32_t)p.P;
    it_end = (idx + 1) * p.I_sk / (uint32_t)p.P;
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
      const uint32_t G = (uint32_t)p.G;
      const uint32_t sk = it / G;
      const uint32_t g0 = it - sk * G;
      const uint32_t rem = it_end - it;
      const uint32_t g1 = rem < G - g0 ? g0 + rem : G;
      u.tile = p.T_dp + (int)sk;
      u.g0 = (int)g0;
      u.g1 = (int)g1;
      it += g1 - g0;
      return true;
    }
    return false;
  }
};

// Tile t -> (weight tile nt, token tile mt) for 128-token tiles.  Tiles go in
// bands of kTileBand token tiles: inside a band the token tile changes
// fastest, so the CTAs running at one time share ~P / kTileBand weight tiles
// and kTileBand token tiles, and their operands stay in L2 (all token tiles of
// a large prefill at once would not).  A band narrower than kTileBand (the
// last one, or MT < kTileBand) keeps the same order.
constexpr int kTileBand = 16;
struct TileXY {
  int nt, mt;
};
__device__ __forceinline__ TileXY tile_xy(const GemmParams& p, int t) {
  const int band_tiles = kTileBand * p.NT;
  const int band = t / band_tiles, r = t - band * band_tiles;
  const int width = min(kTileBand, p.MT - band * kTileBand);
  TileXY c;
  c.nt = r / width;
  c.mt = band * kTileBand + (r - c.nt * width);
  return c;
}

// ------------------------------------------------------------------- waits --

// Bounded wait on an mbarrier phase.  Returns false if the wait ran out (the
// timeout is recorded) or, when honor_abort, if another thread of this call
// already recorded one.  The loop polls only the barrier for the first ~100k
// cycles; the global timer and the abort word in global memory are read after
// that, so a normal hand-off never waits behind a global load.
template <bool CL = false>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const GemmParams& p, bool honor_abort) {
  volatile unsigned* abort_word = reinterpret_cast<volatile unsigned*>(p.status + 1);
  const long long c0 = clock64();
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (CL ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
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

// CL: acquire at cluster scope, for barriers that the other CTA of a CTA pair
// (or the pair's tensor-core operations) arrive on.
template <bool CL = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const GemmParams& p,
                                         bool honor_abort = true) {
  if (CL ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  return wait_slow<CL>(bar, parity, p, honor_abort);
}

// Per-stage sequence words in shared memory: the producer publishes, with
// release semantics, the group it armed a stage for; a consumer that is not
// the stage's previous consumer first waits (acquire) for its own group's
// number, which proves that the stage's previous phase completed, and only
// then waits on the stage's phase parity.
__device__ __forceinline__ void st_release_shared(uint32_t addr, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_shared(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
// Bounded like wait_slow.
__device__ __noinline__ inline bool wait_seq_slow(uint32_t addr, uint32_t want, const GemmParams& p) {
  volatile unsigned* abort_word = reinterpret_cast<volatile unsigned*>(p.status + 1);
  const long long c0 = clock64();
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire_shared(addr) == want) return true;
    if ((i & 255) == 0 && clock64() - c0 > 100000) {
      const uint64_t now = global_timer_ns();
      if (t0 == 0) t0 = now;
      if (*abort_word == p.call_id) return false;
      if (now - t0 > p.timeout_ns) {
        atomicExch(p.status, kStatusTimeout);
        atomicExch(reinterpret_cast<unsigned*>(p.status + 1), p.call_id);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_seq(uint32_t addr, uint32_t want, const GemmParams& p) {
  if (ld_acquire_shared(addr) == want) return true;
  return wait_seq_slow(addr, want, p);
}

// For spin loops on global memory: false once the call's wait limit has run
// out (recorded as a timeout) or another thread of the call recorded one.
// t0: 0 before the first check.
__device__ __noinline__ inline bool spin_ok(const GemmParams& p, uint64_t& t0) {
  const uint64_t now = global_timer_ns();
  if (t0 == 0) t0 = now;
  if (*reinterpret_cast<volatile unsigned*>(p.status + 1) == p.call_id) return false;
  if (now - t0 > p.timeout_ns) {
    atomicExch(p.status, kStatusTimeout);
    atomicExch(reinterpret_cast<unsigned*>(p.status + 1), p.call_id);
    return false;
  }
  return true;
}

// Lane 0 waits, the warp learns the outcome (keeps the warp converged).
template <bool CL = false>
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, const GemmParams& p) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = wait_bar<CL>(bar, parity, p);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Every lane waits, then the warp votes.  Lanes that spin on their own leave
// the loop at different times, and nothing else guarantees that the warp is
// converged again when it reaches a warp-collective instruction (tcgen05.ld /
// st .sync.aligned, elect.sync); so a wait followed by one, with no
// __syncwarp in between, takes this form or warp_wait_bar's.  The vote
// returns the warp converged, with one outcome for all lanes.
template <bool CL = false>
__device__ __forceinline__ bool conv_wait_bar(uint32_t bar, uint32_t parity, const GemmParams& p) {
  const bool ok = wait_bar<CL>(bar, parity, p);
  return __all_sync(0xffffffffu, ok);
}

template <int NTHREADS>
__device__ __forceinline__ void named_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory");
}

// Called once per CTA (one thread), after a CTA-wide barrier that follows
// every read of the hand-off epoch in the CTA: counts the CTA out, and the
// last CTA of the launch resets the counter and advances the epoch.  The
// counter's acq_rel update orders each CTA's epoch reads before the last
// CTA's advance; the next launch reads the epoch only after
// griddepcontrol.wait, i.e. after this launch has completed.  A launch that
// ran out of a wait limit still reaches this point in every CTA.
__device__ __forceinline__ void advance_epoch_at_exit(const GemmParams& p) {
  int32_t* const hdr = p.status;
  if (atom_add_acq_rel(hdr + kWsExitWord, 1) == p.P - 1) {
    hdr[kWsExitWord] = 0;
    hdr[kWsEpochWord] = (int32_t)((uint32_t)hdr[kWsEpochWord] + 1u);
  }
}

// -------------------------------------------------- zero-point folding --
// The zero-point-folded variant (QFactory notes, section 4.3: a matmul whose
// weight operand carries an offset splits into the offset-free product and a
// product with the all-ones matrix, i.e. row sums): the tensor cores see
// q4 * s2, and this subtracts the zero points' share of k-tiles g0 .. g1-1 of
// weight tile nt for tokens m0 .. m0 + COLS - 1 of weight row `row`:
//   run[i] -= (z * s2)[row, g] * RS[g][m0 + i]   for every k-tile g,
// with s2 and z read from the packed tile (one scale set per k-tile, g >= 128)
// and RS the row sums the pre-pass wrote.  Tokens past M (whose RS chunks may
// lie past the array) are skipped; their outputs are never written.
template <int COLS, int TILE>
__device__ __forceinline__ void zero_point_share(const GemmParams& p, int nt, int g0, int g1, int m0, int row,
                                                 int32_t (&run)[COLS]) {
  static_assert(COLS % 4 == 0, "row sums are read four tokens at a time");
  const uint8_t* t = p.packed + ((size_t)nt * p.G + g0) * TILE;
  for (int g = g0; g < g1; ++g, t += TILE) {
    const int zs = (int)__ldg(t + row) * (int)__ldg(t + 128 + row);  // s2 * z
    const int4* r = reinterpret_cast<const int4*>(p.rs + (size_t)g * p.rs_ld + m0);
#pragma unroll
    for (int q = 0; q < COLS / 4; ++q) {
      if (m0 + 4 * q < p.rs_ld) {
        const int4 v = __ldcg(r + q);
        run[4 * q + 0] -= zs * v.x;
        run[4 * q + 1] -= zs * v.y;
        run[4 * q + 2] -= zs * v.z;
        run[4 * q + 3] -= zs * v.w;
      }
    }
  }
}

// ------------------------------------------------------------------ output --
// ------------------------------------------------------------------ output --

// Y[m, n] for the COLS tokens m = m0 .. m0+COLS-1 held by this thread.
template <int COLS>
__device__ __forceinline__ void write_tile_out(const GemmParams& p, const int32_t (&run)[COLS], int m0,
                                               int n) {
  const float s1f = p.Y ? __half2float(__ushort_as_half(p.s1[n])) : 0.0f;
#pragma unroll
  for (int i = 0; i < COLS; ++i) {
    const int m = m0 + i;
    if (m < p.M) {
      if (p.Y) {  // (the W4Ax kernels' integer-sum launch writes acc_debug alone)
        const float sxf = __half2float(__ushort_as_half(p.sx[m]));
        const float y = (float)run[i] * (sxf * s1f);
        p.Y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(y));
      }
      if (p.acc_debug) p.acc_debug[(size_t)m * p.N + n] = run[i];
    }
  }
}

// The epilogue scales of a row: s1[n] and s_x of tokens m0 .. m0 + COLS - 1
// (0 past M), loaded into registers ahead of time, two fp16 per register.
template <int COLS>
struct RowScales {
  uint16_t s1;
  uint32_t sx2[COLS / 2];
};

// m0 is a multiple of COLS and s_x is 16-byte aligned, so a pair of s_x
// values is one aligned 4-byte load; a pair that straddles M loads its first.
template <int COLS>
__device__ __forceinline__ RowScales<COLS> load_row_scales(const GemmParams& p, int m0, int n) {
  static_assert(COLS % 2 == 0, "s_x pairs");
  RowScales<COLS> r;
  r.s1 = p.s1[n];
#pragma unroll
  for (int i = 0; i < COLS / 2; ++i) {
    const int m = m0 + 2 * i;
    r.sx2[i] = m + 1 < p.M ? *reinterpret_cast<const uint32_t*>(p.sx + m) : m < p.M ? (uint32_t)p.sx[m] : 0u;
  }
  return r;
}

// write_tile_out with the scales already loaded.
template <int COLS>
__device__ __forceinline__ void write_tile_out(const GemmParams& p, const int32_t (&run)[COLS], int m0, int n,
                                               const RowScales<COLS>& sc) {
  const float s1f = __half2float(__ushort_as_half(sc.s1));
#pragma unroll
  for (int i = 0; i < COLS; ++i) {
    const int m = m0 + i;
    if (m < p.M) {
      const uint16_t sx = (uint16_t)(sc.sx2[i / 2] >> (16 * (i & 1)));
      const float y = (float)run[i] * (__half2float(__ushort_as_half(sx)) * s1f);
      p.Y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(y));
      if (p.acc_debug) p.acc_debug[(size_t)m * p.N + n] = run[i];
    }
  }
}

// ------------------------------------------------------------- MMA issuer --
// One converged warp; lane 0 waits, one elected lane issues 8 MMAs per group
// (M=128, N=BN, K=16; A = dequantized weights in TMEM, B = fp16 activations
// in shared memory) and commits.  A diverged single thread issues tcgen05 ops
// about 2.5x slower, and an mbarrier wait costs ~100 cycles even on a completed
// phase, so the loop waits once per group.  `b_tile(gi, a)` gives the shared
// address of group gi's B tile; the group's A-full barrier covers it too.
// After each MMA group: commits to `bar_aempty[a]` and to `extra_commit(gi)`
// (0 = none).
// PAIR: the warp of the pair's leading CTA issues the pair's MMAs (M=256:
// each CTA's weight tile from its own TMEM; N=BN tokens, the first BN/2 from
// this CTA's B half, the rest from the other CTA's, at the same offset), its
// waits are cluster-scope (the other CTA arrives on the A-full and
// accumulator-empty barriers too), and every commit but the drain arrives on
// the same barrier in both CTAs.
template <int BN, int NACC, int NABUF, int ACOL0, int FOLD, bool PAIR = false, typename BTile,
          typename ExtraCommit>
__device__ __forceinline__ void mma_role(const GemmParams& p, uint32_t tmem, uint32_t bar_afull,
                                         uint32_t bar_aempty, uint32_t bar_accfull, uint32_t bar_accempty,
                                         uint32_t bar_drain, BTile b_tile, ExtraCommit extra_commit) {
  constexpr uint32_t kIdesc = mma_idesc(BN, PAIR ? 2 * kTileN : kTileN);
  constexpr uint32_t kBRows = PAIR ? BN / 2 : BN;  // rows of this CTA's B tile
  auto commit = [](uint32_t bar) {
    if constexpr (PAIR)
      tc_commit_pair_mc(bar, 3);
    else
      tc_commit(bar);
  };
  UnitIter iter;
  iter.init(p, PAIR ? blockIdx.x >> 1 : blockIdx.x);
  Unit u;
  uint32_t gi = 0, chunk = 0;
  bool ok = true;
  while (ok && iter.next(p, u)) {
    for (int c0 = u.g0; c0 < u.g1; c0 += FOLD) {
      const int c1 = min(u.g1, c0 + FOLD);
      const int b = chunk % NACC;
      if (!warp_wait_bar<PAIR>(bar_accempty + 8 * b, ((chunk / NACC) & 1) ^ 1, p)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + b * BN;
      for (int g = c0; g < c1; ++g, ++gi) {
        const int a = gi % NABUF;
        if (!warp_wait_bar<PAIR>(bar_afull + 8 * a, (gi / NABUF) & 1, p)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if ((threadIdx.x & 31) == 0) QOQ_TRACE_AT(p, 128 + (int)gi, 0);
        const uint32_t b_lo = desc_sw128_lo(b_tile(gi, a));
        const uint32_t a_col = tmem + ACOL0 + a * 64;
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {  // K step j: 64-channel half j / 4, 32-byte chunk j % 4
            const uint32_t bl = b_lo + (j >> 2) * (kBRows * 8) + (j & 3) * 2;
            const uint32_t acc = (g > c0 || j > 0) ? 1u : 0u;
            if constexpr (PAIR)
              tc_mma_ts_pair(d_tmem, a_col + 8 * j, bl, kDescSw128Hi, kIdesc, acc);
            else
              tc_mma_ts(d_tmem, a_col + 8 * j, bl, kDescSw128Hi, kIdesc, acc);
          }
          commit(bar_aempty + 8 * a);
          const uint32_t xc = extra_commit(gi);
          if (xc) commit(xc);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) commit(bar_accfull + 8 * b);
      __syncwarp();
      ++chunk;
    }
  }
  // all MMAs issued by this warp complete before TMEM is released
  if (elect_one()) {
    if constexpr (PAIR)
      tc_commit_pair_mc(bar_drain, 1);  // this (the leading) CTA only
    else
      tc_commit(bar_drain);
  }
  __syncwarp();
  if ((threadIdx.x & 31) == 0) wait_bar<PAIR>(bar_drain, 0, p, false);
  __syncwarp();
}

// ---------------------------------------------------------------- epilogue --
// End of a unit for the NEPI epilogue warps: a whole-K tile is written; a
// split tile's int32 partial sums are added into the workspace, and the last
// contributor writes Y and leaves the workspace zeroed.  `run` holds tokens
// tok0 .. tok0 + TOK - 1 of weight row `row` (output channel n; first token m0).
// `sk` indexes the split tile's partial sums and count (for a CTA pair, each
// CTA's half of a pair tile has its own).
template <int BN, int NEPI, int TOK>
__device__ __forceinline__ void finish_unit(const GemmParams& p, const Unit& u, int sk, int32_t (&run)[TOK], int m0,
                                            int n, int tok0, int row, int etid, bool ok, volatile int* last_flag,
                                            bool tracer, int unit_no) {
  (void)tracer;
  (void)unit_no;
  if (u.g0 == 0 && u.g1 == p.G) {
    if (ok) write_tile_out<TOK>(p, run, m0, n);
    return;
  }
  int32_t* part = p.sk_acc + (size_t)sk * BN * kTileN + (size_t)tok0 * kTileN;
  if (ok) {
#pragma unroll
    for (int i = 0; i < TOK; ++i) red_add_relaxed(part + i * kTileN + row, run[i]);
  }
  // The barrier orders every epilogue thread's partial sums before one
  // thread's acq_rel count update (release is cumulative over the barrier);
  // the last contributor's acquire makes the other CTAs' sums visible, and the
  // second barrier passes that on to its warps.
  if (tracer) QOQ_TRACE_AT(p, 960 + 4 * (unit_no & 7) + 0, 0);
  named_bar_sync<NEPI * 32>();
  if (etid == 0) {
    int last = 0;
    if (ok) {
      const int add = u.g1 - u.g0;
      last = (atom_add_acq_rel(p.sk_cnt + sk, add) + add == p.G) ? 1 : 0;
      if (last) p.sk_cnt[sk] = 0;  // every contributor has counted: reset for the next call
    }
    *last_flag = last;
  }
  named_bar_sync<NEPI * 32>();
  if (tracer) QOQ_TRACE_AT(p, 960 + 4 * (unit_no & 7) + 2, 0);
  if (ok && *last_flag) {
#pragma unroll
    for (int i = 0; i < TOK; ++i) run[i] = __ldcg(part + i * kTileN + row);
#pragma unroll
    for (int i = 0; i < TOK; ++i) __stcg(part + i * kTileN + row, 0);  // leave it zeroed
    write_tile_out<TOK>(p, run, m0, n);
  }
}

// NEPI warps (a multiple of 4: warp w reads TMEM lanes 32 (w % 4) ..); warp e
// owns tokens (e / 4) * TOK .. + TOK of the tile for weight row 32 (w % 4) +
// lane.  Per fold chunk: read the fp32 accumulator, convert to int32 (exact),
// add.  At a unit's end: write Y (whole-K tile), or add the int32 partials
// into the workspace and let the last contributor write Y and clear them.
// PAIR: this CTA holds weight tile 2 nt + rank of pair tile nt, and releases
// an accumulator on the leading CTA's barrier (where the pair's MMAs are
// issued).
template <int BN, int NEPI, int NACC, bool ZF = false, int TILE = kWTileBytes,
          int FOLD = ZF ? kFoldGroupsZf : kFoldGroups, bool PAIR = false>
__device__ __forceinline__ void epilogue_role(const GemmParams& p, uint32_t tmem, int epi_warp0,
                                              uint32_t bar_accfull, uint32_t bar_accempty,
                                              volatile int* last_flag) {
  static_assert(!(PAIR && ZF), "the pair kernel has no zero-point-folded form");
  constexpr int TOK = BN / (NEPI / 4);
  static_assert(TOK % 16 == 0, "epilogue loads 16 columns at a time");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = warp - epi_warp0;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;
  const int tok0 = (e >> 2) * TOK;
  const int etid = threadIdx.x - epi_warp0 * 32;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const uint32_t rank = PAIR ? blockIdx.x & 1 : 0;
  UnitIter iter;
  iter.init(p, PAIR ? blockIdx.x >> 1 : blockIdx.x);
  Unit u;
  uint32_t chunk = 0;
  int unit_no = 0;
  bool ok = true;  // once false, keep the control flow (named barriers) but do no work
  while (iter.next(p, u)) {
    const TileXY xy = tile_xy(p, u.tile);
    const int nt = xy.nt, mt = xy.mt;
    const int n = (PAIR ? 2 * nt + (int)rank : nt) * kTileN + row;
    int32_t run[TOK];
#pragma unroll
    for (int i = 0; i < TOK; ++i) run[i] = 0;
    for (int c0 = u.g0; c0 < u.g1; c0 += FOLD, ++chunk) {
      const int b = chunk % NACC;
      // zero points' share of the chunk, while its MMAs still run
      if constexpr (ZF) zero_point_share<TOK, TILE>(p, nt, c0, min(u.g1, c0 + FOLD), mt * BN + tok0, row, run);
      if (ok) ok = conv_wait_bar<PAIR>(bar_accfull + 8 * b, (chunk / NACC) & 1, p);
      if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 512 + (int)chunk, 0);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int piece = 0; piece < TOK / 16; ++piece) {
          uint32_t v[16];
          tmem_ld16_wait(tmem + lane_base + b * BN + tok0 + piece * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) run[piece * 16 + i] += __float2int_rn(__uint_as_float(v[i]) * kAccScale);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && rank != 0)
            mbar_arrive_remote(bar_accempty + 8 * b, 0);
          else
            mbar_arrive(bar_accempty + 8 * b);
        }
        if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 576 + (int)chunk, 0);
      }
    }
    const int sk = PAIR ? 2 * (u.tile - p.T_dp) + (int)rank : u.tile - p.T_dp;
    finish_unit<BN, NEPI, TOK>(p, u, sk, run, mt * BN + tok0, n, tok0, row, etid, ok, last_flag,
                                e == 0 && lane == 0, unit_no);
    if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 640 + unit_no, 0);
    ++unit_no;
  }
}

// ------------------------------------------------------------- W4Ax epilogue --
// COMET explainer, the W4Ax kernel: each activation block's integer partial
// sums are scaled by that block's scale on the general-purpose cores.  The
// MMA warp commits one accumulator per 128-channel group (fold chunk of one
// group); per group this thread adds, for its weight row and its TOK tokens,
//   run[i] += D[i] * s[m_i, g]        (D = acc_g * 2^-13, exact in fp32),
// and at a unit's end writes Y = fp16_rn(run * 2^13 * s1[n]), or adds its
// float partial sums into the workspace for a split tile, where the last
// contributor writes Y (the order of those additions is not fixed, so a split
// tile's Y may differ between calls in the last fp32 bit before rounding).
template <int COLS>
__device__ __forceinline__ void write_tile_out_ax(const GemmParams& p, const float (&run)[COLS], int m0, int n) {
  const float sc = kAccScale * __half2float(__ushort_as_half(p.s1[n]));  // exact: s1 times 2^13
#pragma unroll
  for (int i = 0; i < COLS; ++i) {
    const int m = m0 + i;
    if (m < p.M) p.Y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(run[i] * sc));
  }
}

// The block scales of group number q arrive in shared-memory slot q % SCR
// (sc_smem + 256 slot: 128 fp16, one per token of the tile), announced on
// barrier sc_bars + 8 slot; every epilogue warp arrives on sc_bars + 8 (SCR +
// slot) when it is done with them.
template <int BN, int NEPI, int NACC, int SCR>
__device__ __forceinline__ void epilogue_role_ax(const GemmParams& p, uint32_t tmem, int epi_warp0,
                                                 uint32_t bar_accfull, uint32_t bar_accempty,
                                                 volatile int* last_flag, uint32_t sc_smem, uint32_t sc_bars) {
  constexpr int TOK = BN / (NEPI / 4);
  static_assert(TOK % 16 == 0, "epilogue loads 16 columns at a time");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = warp - epi_warp0;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;
  const int tok0 = (e >> 2) * TOK;
  const int etid = threadIdx.x - epi_warp0 * 32;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  UnitIter iter;
  iter.init(p);
  Unit u;
  uint32_t chunk = 0;
  bool ok = true;  // once false, keep the control flow (named barriers) but do no work
  while (iter.next(p, u)) {
    const TileXY xy = tile_xy(p, u.tile);
    const int nt = xy.nt, mt = xy.mt;
    const int n = nt * kTileN + row;
    float run[TOK];
#pragma unroll
    for (int i = 0; i < TOK; ++i) run[i] = 0.0f;
    for (int g = u.g0; g < u.g1; ++g, ++chunk) {
      const int b = chunk % NACC;
      const int slot = (int)(chunk % SCR);
      if (ok) ok = conv_wait_bar(sc_bars + 8 * slot, (chunk / SCR) & 1, p);
      if (ok) ok = conv_wait_bar(bar_accfull + 8 * b, (chunk / NACC) & 1, p);
      if (ok) tc_fence_after();
#pragma unroll
      for (int piece = 0; piece < TOK / 16; ++piece) {
        if (ok) {
          // this group's scales of these 16 tokens, from the ring
          const uint32_t sa = sc_smem + 256 * slot + 2 * (tok0 + piece * 16);
          uint4 s0, s1v;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(s0.x), "=r"(s0.y), "=r"(s0.z), "=r"(s0.w) : "r"(sa));
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(s1v.x), "=r"(s1v.y), "=r"(s1v.z), "=r"(s1v.w) : "r"(sa + 16));
          uint32_t v[16];
          tmem_ld16_wait(tmem + lane_base + b * BN + tok0 + piece * 16, v);
          const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1v.x, s1v.y, s1v.z, s1v.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(&sw[i]));
            run[piece * 16 + 2 * i] = fmaf(__uint_as_float(v[2 * i]), sc.x, run[piece * 16 + 2 * i]);
            run[piece * 16 + 2 * i + 1] = fmaf(__uint_as_float(v[2 * i + 1]), sc.y, run[piece * 16 + 2 * i + 1]);
          }
        }
      }
      if (ok) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_accempty + 8 * b);
          mbar_arrive(sc_bars + 8 * (SCR + slot));
        }
      }
    }
    const int m0 = mt * BN + tok0;
    if (u.g0 == 0 && u.g1 == p.G) {
      if (ok) write_tile_out_ax<TOK>(p, run, m0, n);
      continue;
    }
    // split tile: float partial sums meet in the workspace (see finish_unit)
    const int sk = u.tile - p.T_dp;
    float* part = reinterpret_cast<float*>(p.sk_acc) + (size_t)sk * BN * kTileN + (size_t)tok0 * kTileN;
    if (ok) {
#pragma unroll
      for (int i = 0; i < TOK; ++i) red_add_relaxed_f32(part + i * kTileN + row, run[i]);
    }
    named_bar_sync<NEPI * 32>();
    if (etid == 0) {
      int last = 0;
      if (ok) {
        const int add = u.g1 - u.g0;
        last = (atom_add_acq_rel(p.sk_cnt + sk, add) + add == p.G) ? 1 : 0;
        if (last) p.sk_cnt[sk] = 0;  // every contributor has counted: reset for the next call
      }
      *last_flag = last;
    }
    named_bar_sync<NEPI * 32>();
    if (ok && *last_flag) {
#pragma unroll
      for (int i = 0; i < TOK; ++i) run[i] = __ldcg(part + i * kTileN + row);
#pragma unroll
      for (int i = 0; i < TOK; ++i) __stcg(part + i * kTileN + row, 0.0f);  // leave it zeroed
      write_tile_out_ax<TOK>(p, run, m0, n);
    }
  }
}

// Opt a kernel into its dynamic shared memory once per device (not a stream
// operation; done before any graph capture can reach it).
template <typename Kernel>
cudaError_t set_smem_attr_once(Kernel kernel, int bytes, uint64_t& done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && (done_mask >> dev) & 1) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) done_mask |= 1ull << dev;
  return e;
}


}  // namespace qoq
