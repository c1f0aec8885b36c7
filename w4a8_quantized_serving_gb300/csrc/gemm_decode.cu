// gemm_decode.cu -- the W4A8 g128 GEMM for decode-sized token counts
// (M <= 64, one token tile of BN = 16, 32 or 64 rows).
//
// Lecture 15 notes, section 15.5: at decode sizes the weight stream is the
// floor, and the dequant instructions per weight decide whether the kernel
// reaches it.  Roles:
//   warps 0, 1    producers (lane 0 of each): per 128-channel group one bulk
//                 copy of the packed weight tile (8448 B) into shared memory.
//                 Group gi of the CTA's work belongs to dequant slot
//                 gi % NSLOT, which owns a sub-ring of SPS stages; each
//                 producer serves half of the slots.  Warp 1 also allocates
//                 tensor memory (and frees it at the end).
//   warps 2..     NSLOT dequant slots of 4 warps, one per TMEM lane quadrant.
//                 Per group a slot's 128 threads read the group's int8
//                 activation slice from L2 (issued before their stage wait) and
//                 write it as the fp16 B tile into the slot's shared buffer;
//                 thread r expands weight row r's 64 code bytes with one mask
//                 and one FMA per pair (exact) into the slot's TMEM A buffer.
//                 After a named barrier of the slot, one elected thread issues
//                 the group's 8 tcgen05.mma (M=128 weight rows, N=BN tokens,
//                 K=16) into the slot's own accumulator.  Each slot issues its
//                 own MMAs: no MMA warp serialises the groups, and no hand-off
//                 of A buffers between warps is needed.
//   last NEPI     epilogue: per fold chunk (up to 8 groups per slot) it sums
//                 the slots' accumulators into int32, and at a unit's end
//                 writes Y, or hands a split tile's part to the tile's owner
//                 (see slot_store / slot_gather).
//
// Barrier protocol.  mbarrier waits test only the parity of a phase, so each
// wait must start after the phase before the one it wants has completed, and
// before the phase after it can complete.  Here every barrier's waiters take
// part in each of its phases: a weight stage has one producer and one
// consumer slot, both in order; a slot's MMA-done barrier is waited on only
// by that slot; every slot waits for and arrives on every fold chunk's
// accumulator barriers, also in chunks where it has no group.
#include <mutex>

#include "gemm_common.cuh"

namespace qoq {
namespace {

// BN: token tile width; GPT: level-2 scale sets per packed k-tile (g = 128 / GPT,
// or a multiple of 128 with GPT = 1).
template <int BN, int GPT>
struct DecCfg {
  static constexpr int TILE = w_tile_bytes(GPT);  // packed k-tile bytes
  static constexpr int NIB = w_nib_offset(GPT);   // offset of its code chunks
  static constexpr int NSLOT = BN == 64 ? 2 : 4;
  static constexpr int NDQ = 4 * NSLOT;
  static constexpr int NEPI = BN == 64 ? 8 : 4;
  static constexpr int DQ_WARP0 = 2;
  static constexpr int EPI_WARP0 = 2 + NDQ;
  static constexpr int THREADS = (2 + NDQ + NEPI) * 32;
  static constexpr int NACC = 2;
  // Fold chunk: up to CH(fold) consecutive groups of a unit, so at most
  // `fold` groups of each slot go into one fp32 accumulator (exact below 2^24).
  __host__ __device__ static constexpr int chunk(int fold) { return fold * NSLOT; }
  // TMEM columns: accumulator b of slot j at (j * NACC + b) * BN; slot j's A
  // buffer (128 rows x 128 fp16 = 64 columns) at ACOL0 + 64 j.
  static constexpr int ACOL0 = (NSLOT * NACC * BN + 63) / 64 * 64;
  static constexpr int B_BYTES = BN * kGroup * 2;  // slot j's B tile at j * B_BYTES
  static constexpr int W_OFF = NSLOT * B_BYTES;
  static constexpr int STAGES_FIT = (kSmemBudget - 2048 - W_OFF) / TILE;
  static constexpr int STAGES = (STAGES_FIT > 24 ? 24 : STAGES_FIT) / NSLOT * NSLOT;
  static constexpr int SPS = STAGES / NSLOT;  // stages per slot
  static constexpr int BAR_OFF = W_OFF + STAGES * TILE;
  static constexpr int NBARS = 2 * STAGES + NSLOT + 2 * NACC;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SMEM_BYTES = TMEM_SLOT_OFF + 8 + 1024;  // + slack for 1024-B alignment
  static_assert(BN == 16 || BN == 32 || BN == 64, "decode tiles");
  static_assert(ACOL0 + 64 * NSLOT <= kTmemCols, "TMEM columns");
  static_assert(SPS >= 2 && STAGES <= 32, "pipeline depth per slot, stage masks");
  static_assert(B_BYTES % 1024 == 0, "1024-B aligned B tiles");
  static_assert(SMEM_BYTES <= kSmemBudget, "shared memory");
};

// Copy-issuing threads: lane 0 of warps 0 .. kProducers - 1 (warp 1 also
// allocates tensor memory).
constexpr int kProducers = 2;

// Named barrier ID of dequant slot j (0: __syncthreads, 1: the epilogue).
constexpr int kSlotBar0 = 2;

// Slot j's first group in a chunk whose first group has CTA index gc0.
template <int NSLOT>
__device__ __forceinline__ int slot_first(int slot, uint32_t gc0) {
  return (int)(((uint32_t)slot - gc0) & (NSLOT - 1));
}

// Named barrier among the 4 warps (128 threads) of one slot, whole warps.
__device__ __forceinline__ void slot_bar_sync(int slot) {
  asm volatile("bar.sync %0, 128;" ::"r"(kSlotBar0 + slot) : "memory");
}

// The CTA whose stream-K range holds group iteration it (CTA b's range is
// [floor(b I / P), floor((b + 1) I / P)) of the I = T_sk G iterations).
__device__ __forceinline__ int sk_cta_of(const GemmParams& p, uint32_t it) {
  return (int)(((it + 1) * (uint32_t)p.P - 1) / p.I_sk);
}

// Split-K hand-off of the decode kernel.  A split tile is finished by its
// owner, the CTA holding the tile's first group: that part is the last unit
// of its range, so it comes last in time.  Every other contributor holds a
// later part of the tile as the first unit of its range, and stores it into
// its own slot as {int32 partial sum, tag} pairs, which are single-copy
// atomic: the owner reads the slots of the CTAs after it and retries only
// while an entry does not carry this launch's tag yet.  The tag is 2 e + 1 for
// the epoch e in the workspace header, which the last CTA of every launch
// advances (advance_epoch_at_exit), so a launch replayed from a CUDA graph
// never accepts a partial sum that an earlier replay left behind, and nothing
// needs clearing.  Tags are odd, so a zero-filled entry never matches one;
// the state of 128-token-tile calls sharing the workspace lies above the
// decode area (kDecodeArea) and never overlaps the slots.
template <int BN, int TOK>
__device__ __forceinline__ void slot_store(const GemmParams& p, uint32_t tag, int tok0, int row,
                                           const int32_t (&run)[TOK]) {
  unsigned long long* sl = p.sk_slot + (size_t)blockIdx.x * BN * kTileN;
  const unsigned long long hi = (unsigned long long)tag << 32;
#pragma unroll
  for (int i = 0; i < TOK; ++i) st_relaxed_b64(sl + (tok0 + i) * kTileN + row, hi | (uint32_t)run[i]);
}

// Pieces of 16 tokens: all 16 loads in flight at once, without holding more
// registers than that beside the running sums.
template <int BN, int TOK>
__device__ __forceinline__ bool slot_gather(const GemmParams& p, uint32_t tag, int c, int tok0, int row,
                                            int32_t (&run)[TOK]) {
  unsigned long long* sl = p.sk_slot + (size_t)c * BN * kTileN;
  uint64_t t0 = 0;
#pragma unroll
  for (int piece = 0; piece < TOK; piece += 16) {
    int32_t part[16];
    for (uint32_t tries = 1;; ++tries) {
      bool all = true;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const unsigned long long v = ld_relaxed_b64(sl + (tok0 + piece + i) * kTileN + row);
        part[i] = (int32_t)(uint32_t)v;
        all &= (uint32_t)(v >> 32) == tag;
      }
      if (all) break;
      if ((tries & 15) == 0 && !spin_ok(p, t0)) return false;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) run[piece + i] += part[i];
  }
  return true;
}

template <int BN, int GPT, bool ZF>
__global__ void __launch_bounds__(DecCfg<BN, GPT>::THREADS, 1) gemm_decode_kernel(const __grid_constant__ GemmParams p) {
  using C = DecCfg<BN, GPT>;
  constexpr int CH = C::chunk(ZF ? kFoldGroupsZf : kFoldGroups);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + C::BAR_OFF;
  const uint32_t bar_full = bars, bar_empty = bars + 8 * C::STAGES;
  const uint32_t bar_mmadone = bar_empty + 8 * C::STAGES;  // per slot: its MMAs of a group completed
  const uint32_t bar_accfull = bar_mmadone + 8 * C::NSLOT, bar_accempty = bar_accfull + 8 * C::NACC;

  // The next kernel on the stream may launch now: it waits for this one to
  // complete before it touches anything this call reads or writes, and its
  // CTAs take SMs as this call's CTAs leave them.
  grid_dep_launch_dependents();
  if (threadIdx.x == 0) {
    QOQ_TRACE_AT(p, 0, 0);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 4);  // the 4 warps of the slot that owns the stage
    }
    for (int j = 0; j < C::NSLOT; ++j) mbar_init(bar_mmadone + 8 * j, 1);
    for (int b = 0; b < C::NACC; ++b) {
      mbar_init(bar_accfull + 8 * b, C::NSLOT);  // one arrival per slot and chunk
      mbar_init(bar_accempty + 8 * b, C::NEPI);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(sbase + C::TMEM_SLOT_OFF, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::TMEM_SLOT_OFF);
  if (threadIdx.x == 0) QOQ_TRACE_AT(p, 1, 0);

  if (warp < kProducers) {
    // ------------------------------------------------------------ producer --
    // Weights only: they do not depend on the preceding kernel, so the ring
    // fills while it runs.  Before its first wait for a stage to be released
    // (timed, like every wait) the producer waits for that kernel too, so the
    // wait measures this call alone.  Producer warp w copies the groups of the
    // slots j with j % kProducers == w (two issuing threads: a copy takes
    // ~0.2-0.3 us to issue while the SM is busy with dequant work).
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();  // each weight tile is read once
      const uint8_t* const packed = p.packed;     // one token tile: weight tile index = tile
      const size_t tile_stride = (size_t)p.G * C::TILE;
      const uint32_t w_base = sbase + C::W_OFF;
      uint32_t issued_mask = 0, issued_par = 0;  // per stage: a copy in its latest lap; its parity
      UnitIter iter;
      iter.init(p);
      Unit u;
      uint32_t gi = 0;
      bool ok = true;
      while (ok && iter.next(p, u)) {
        const uint8_t* src = packed + (size_t)u.tile * tile_stride + (size_t)u.g0 * C::TILE;
        for (int g = u.g0; g < u.g1; ++g, ++gi, src += C::TILE) {
          const int slot = (int)(gi % C::NSLOT);
          if (slot % kProducers != warp) continue;
          const uint32_t k = gi / C::NSLOT;  // the slot's k-th group
          const int s = slot * C::SPS + (int)(k % C::SPS);
          const uint32_t ph = (k / C::SPS) & 1;
          if (k == (uint32_t)C::SPS) grid_dep_wait();
          if (k >= (uint32_t)C::SPS && !wait_bar(bar_empty + 8 * s, ph ^ 1, p)) {
            ok = false;
            break;
          }
          if (!(p.fault == 1 && gi == 17)) {  // test hook: one copy is never issued
            mbar_arrive_expect_tx(bar_full + 8 * s, C::TILE);
            bulk_g2s(w_base + s * C::TILE, src, C::TILE, bar_full + 8 * s, pol);
            issued_mask |= 1u << s;
            issued_par = (issued_par & ~(1u << s)) | (ph << s);
          } else {
            issued_mask &= ~(1u << s);
          }
          QOQ_TRACE_AT(p, 16 + (int)gi, 0);
        }
      }
      // Let every copy still in flight land before the CTA may exit.
      for (int s = 0; s < C::STAGES; ++s)
        if (issued_mask & (1u << s)) wait_bar(bar_full + 8 * s, (issued_par >> s) & 1, p, false);
    }
    __syncwarp();
  } else if (warp < C::EPI_WARP0) {
    // ------------------------------------------------------ dequant + MMA --
    grid_dep_wait();  // Xq comes from the preceding kernel
    if (warp == C::DQ_WARP0 && lane == 0) QOQ_TRACE_AT(p, 3, 0);
    const int slot = (warp - C::DQ_WARP0) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int stid = ((warp - C::DQ_WARP0) & 3) * 32 + lane;  // 0..127 within the slot
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const bool issuer = quad == (slot & 3);  // the slots' MMA issuers sit on different sub-partitions
    constexpr uint32_t kIdesc = mma_idesc(BN);
    const uint32_t a_col = tmem + C::ACOL0 + 64 * slot;
    const uint32_t b_lo = desc_sw128_lo(sbase + (uint32_t)(slot * C::B_BYTES));
    uint8_t* const btile = smem + slot * C::B_BYTES;
    UnitIter iter;
    iter.init(p);
    Unit u;
    uint32_t gi_u = 0, ch = 0, nown = 0;  // CTA index of the unit's first group; chunk; own groups
    uint32_t nissued = 0;                 // groups whose MMAs this slot issued
    // After a wait runs out, a warp keeps the slot's control flow (so that the
    // slot's other warps never wait at its named barrier for it) but skips its
    // waits and work, and the kernel winds down.
    bool ok = true;
    while (iter.next(p, u)) {
      for (int c0 = u.g0; c0 < u.g1; c0 += CH, ++ch) {
        const int len = min(CH, u.g1 - c0);
        const uint32_t gc0 = gi_u + (uint32_t)(c0 - u.g0);
        const int b = ch % C::NACC;
        const uint32_t d_tmem = tmem + (uint32_t)((slot * C::NACC + b) * BN);
        // Every slot waits for every chunk's accumulator, with or without a
        // group in it (see the protocol note above).
        if (ok) ok = wait_bar(bar_accempty + 8 * b, ((ch / C::NACC) & 1) ^ 1, p);
        const int f = slot_first<C::NSLOT>(slot, gc0);
        if (f >= len) {  // no group of this slot in the chunk
          __syncwarp();
          if (ok && issuer && lane == 0) mbar_arrive(bar_accfull + 8 * b);
          continue;
        }
        for (int off = f; off < len; off += C::NSLOT, ++nown) {
          const int g = c0 + off;
          const uint32_t gi = gc0 + (uint32_t)off;  // the group's index in the CTA's work (traces)
          (void)gi;
          const int s = slot * C::SPS + (int)(nown % C::SPS);
          // int8 activation slice: 16-byte chunk q of the [BN][128] tile is
          // row q / 8, channels 16 (q % 8) .. +15; rows past M read as zero
          uint4 xv[BN / 16];
#pragma unroll
          for (int i = 0; i < BN / 16; ++i) {
            const int q = stid + i * 128;
            const int m = q >> 3;  // one token tile: rows 0 .. BN-1
            xv[i] = m < p.M ? __ldcg(reinterpret_cast<const uint4*>(p.xq + (size_t)m * p.K + g * kGroup + (q & 7) * 16))
                            : make_uint4(0, 0, 0, 0);
          }
          if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 192 + (int)gi, 0);
          if (ok) ok = wait_bar(bar_full + 8 * s, (nown / C::SPS) & 1, p);
          if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 320 + (int)gi, 0);
          // The slot's previous MMAs have read its A buffer and B tile.
          if (ok) ok = wait_bar(bar_mmadone + 8 * slot, (nown & 1) ^ 1, p);
          if (ok) {
            tc_fence_after();
            if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 256 + (int)gi, 0);
            const uint8_t* wt = smem + C::W_OFF + s * C::TILE;
            uint4 wv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) wv[c] = *reinterpret_cast<const uint4*>(wt + C::NIB + c * kWChunkBytes + row * 16);
            uint32_t s2v[GPT], zv[GPT];  // scale set u covers chunks u * 4 / GPT ..
#pragma unroll
            for (int u = 0; u < GPT; ++u) {
              s2v[u] = wt[u * 256 + row];
              zv[u] = wt[u * 256 + 128 + row];
            }
            DequantConsts kc = dequant_consts(s2v[0], ZF ? 0u : zv[0]);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);  // the weight tile is in registers
#pragma unroll
            for (int i = 0; i < BN / 16; ++i) {
              const int q = stid + i * 128;
              store_b_chunk(btile, BN, q >> 3, q & 7, xv[i]);
            }
            fence_proxy_async_smem();  // generic-proxy writes -> the MMA's async-proxy reads
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (GPT > 1 && c > 0 && c % (4 / GPT) == 0)
                kc = dequant_consts(s2v[c / (4 / GPT)], ZF ? 0u : zv[c / (4 / GPT)]);
              uint32_t out[16];
              dequant_chunk(wv[c], kc, out);
              tmem_st16(tmem + lane_base + C::ACOL0 + 64 * slot + c * 16, out);
            }
            tmem_wait_st();
            tc_fence_before();
          }
          if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 832 + (int)gi, 0);
          slot_bar_sync(slot);  // the slot's 4 quadrants and its B tile are written
          if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 896 + (int)gi, 0);
          if (ok && issuer) {
            __syncwarp();  // elect.sync wants the whole warp, converged
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
              for (int j = 0; j < 8; ++j)  // K step j: 64-channel half j / 4, 32-byte chunk j % 4
                tc_mma_ts(d_tmem, a_col + 8 * j, b_lo + (j >> 2) * (BN * 8) + (j & 3) * 2, kDescSw128Hi, kIdesc,
                          (off > f || j > 0) ? 1u : 0u);
              tc_commit(bar_mmadone + 8 * slot);
              if (off + C::NSLOT >= len) tc_commit(bar_accfull + 8 * b);  // the slot's last group of the chunk
            }
            __syncwarp();
            ++nissued;
          }
          if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 384 + (int)gi, 0);
        }
      }
      gi_u += (uint32_t)(u.g1 - u.g0);
    }
    // the slot's MMAs complete before its tensor memory is released
    if (issuer && nissued > 0 && lane == 0) wait_bar(bar_mmadone + 8 * slot, (nissued - 1) & 1, p, false);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue --
    grid_dep_wait();  // also orders the epoch read after the previous launch's advance
    constexpr int TOK = BN / (C::NEPI / 4);
    static_assert(TOK % 16 == 0, "epilogue loads 16 columns at a time");
    const int e = warp - C::EPI_WARP0;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int tok0 = (e >> 2) * TOK;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tag = 2u * (uint32_t)ld_relaxed(p.status + kWsEpochWord) + 1u;  // hand-off tag
    UnitIter iter;
    iter.init(p);
    Unit u;
    uint32_t gi_u = 0, ch = 0;
    int unit_no = 0;
    bool ok = true;  // once false, do no more work
    while (iter.next(p, u)) {
      int32_t run[TOK];
#pragma unroll
      for (int i = 0; i < TOK; ++i) run[i] = 0;
      for (int c0 = u.g0; c0 < u.g1; c0 += CH, ++ch) {
        const int len = min(CH, u.g1 - c0);
        const uint32_t gc0 = gi_u + (uint32_t)(c0 - u.g0);
        const int b = ch % C::NACC;
        // zero points' share of the chunk's groups, while their MMAs still run
        if constexpr (ZF) zero_point_share<TOK, C::TILE>(p, u.tile, c0, c0 + len, tok0, row, run);
        if (ok) ok = conv_wait_bar(bar_accfull + 8 * b, (ch / C::NACC) & 1, p);
        if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 512 + (int)ch, 0);
        if (ok) {
          tc_fence_after();
          // Slots without a group in the chunk left their accumulator unwritten:
          // their loads go to a written one and count zero.
          auto acc_col = [&](int j, int piece) {
            return tmem + lane_base + (uint32_t)((j * C::NACC + b) * BN) + tok0 + piece * 16;
          };
#pragma unroll
          for (int piece = 0; piece < TOK / 16; ++piece) {
#pragma unroll
            for (int j = 0; j < C::NSLOT; j += 2) {
              const bool u0 = slot_first<C::NSLOT>(j, gc0) < len, u1 = slot_first<C::NSLOT>(j + 1, gc0) < len;
              uint32_t v[16], w[16];
              tmem_ld16x2_wait(acc_col(u0 ? j : j + 1, piece), acc_col(u1 ? j + 1 : j, piece), v, w);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int a0 = u0 ? __float2int_rn(__uint_as_float(v[i]) * kAccScale) : 0;
                const int a1 = u1 ? __float2int_rn(__uint_as_float(w[i]) * kAccScale) : 0;
                run[piece * 16 + i] += a0 + a1;
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_accempty + 8 * b);
          if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 576 + (int)ch, 0);
        }
      }
      const int n = u.tile * kTileN + row;  // one token tile: weight tile index = tile
      if (u.g0 == 0 && u.g1 == p.G) {  // whole tile
        if (ok) write_tile_out<TOK>(p, run, tok0, n);
      } else if (u.g0 > 0) {  // a later part of a split tile: its owner adds it
        if (ok) slot_store<BN, TOK>(p, tag, tok0, row, run);
      } else {  // the split tile's owner: add the parts of the CTAs after it, then write
        if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 960 + 4 * (unit_no & 7) + 0, 0);
        // Last contributor first: its part is the first unit of its range and
        // was stored early, while a CTA whose whole range lies inside the tile
        // stores its part only as it finishes.  In this order the early part's
        // round trip overlaps the wait for the late one.
        const int b1 = sk_cta_of(p, (uint32_t)(u.tile - p.T_dp) * (uint32_t)p.G + (uint32_t)p.G - 1);
        if constexpr (TOK <= 16) {
          // the scale loads go out before the gather, so their L2 round trip
          // overlaps the gather's instead of following it (wider rows would
          // spill the prefetched scales)
          const RowScales<TOK> sc = load_row_scales<TOK>(p, tok0, n);
          for (int c = b1; ok && c > (int)blockIdx.x; --c) ok = slot_gather<BN, TOK>(p, tag, c, tok0, row, run);
          if (ok) write_tile_out<TOK>(p, run, tok0, n, sc);
        } else {
          for (int c = b1; ok && c > (int)blockIdx.x; --c) ok = slot_gather<BN, TOK>(p, tag, c, tok0, row, run);
          if (ok) write_tile_out<TOK>(p, run, tok0, n);
        }
        if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 960 + 4 * (unit_no & 7) + 2, 0);
      }
      if (e == 0 && lane == 0) QOQ_TRACE_AT(p, 640 + unit_no, 0);
      ++unit_no;
      gi_u += (uint32_t)(u.g1 - u.g0);
    }
  }

  tc_fence_before();
  if (lane == 0) QOQ_TRACE_AT(p, 700 + 2 * warp, 0);
  __syncthreads();
  if (lane == 0) QOQ_TRACE_AT(p, 701 + 2 * warp, 0);
  if (threadIdx.x == 0) {
    QOQ_TRACE_AT(p, 2, 0);
    advance_epoch_at_exit(p);  // every thread of the CTA is past its epoch read
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BN, int GPT, bool ZF>
cudaError_t launch_bn(const GemmParams& p, cudaStream_t s) {
  using C = DecCfg<BN, GPT>;
  static std::mutex mu;
  static uint64_t done_mask = 0;
  cudaError_t e;
  {
    std::lock_guard<std::mutex> lock(mu);
    e = set_smem_attr_once(gemm_decode_kernel<BN, GPT, ZF>, C::SMEM_BYTES, done_mask);
  }
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.P);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_decode_kernel<BN, GPT, ZF>, p);
}

template <int GPT, bool ZF>
cudaError_t launch_gemm_decode_g(const GemmParams& p, int BN, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_bn<16, GPT, ZF>(p, s);
    case 32: return launch_bn<32, GPT, ZF>(p, s);
    case 64: return launch_bn<64, GPT, ZF>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm_decode(const GemmParams& p, int BN, bool zero_folded, cudaStream_t s) {
  if (zero_folded) return p.gpt == 1 ? launch_gemm_decode_g<1, true>(p, BN, s) : cudaErrorInvalidValue;
  switch (p.gpt) {
    case 1: return launch_gemm_decode_g<1, false>(p, BN, s);
    case 2: return launch_gemm_decode_g<2, false>(p, BN, s);
    case 4: return launch_gemm_decode_g<4, false>(p, BN, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qoq
