// gemm_decode.cu -- the W4A8 g128 GEMM for decode-sized token counts
// (M <= 64, one token tile of BN = 16, 32 or 64 rows).
//
// Lecture 15 notes, section 15.5: at decode sizes the weight stream is the
// floor, and the dequant instructions per weight decide whether the kernel
// reaches it.  Roles:
//   warp 0        producer: per 128-channel group one bulk copy of the packed
//                 weight tile (8448 B) into a 16-stage shared-memory ring.
//   warp 1        MMA issuer (gemm_common.cuh mma_role): per group 8 x
//                 tcgen05.mma M=128 (weight rows), N=BN (tokens), K=16.
//   warps 2..     dequant: NSLOT slots of 4 warps (one per TMEM lane quadrant);
//                 slot j takes every NSLOT-th group of the CTA's work.  The
//                 slot's 128 threads read the group's int8 activation slice
//                 from L2 (issued before their stage wait, so the latency
//                 overlaps it) and write it as the fp16 B tile into shared
//                 memory; thread r expands weight row r's 64 code bytes from the
//                 ring with one mask and one FMA per pair (exact) into the TMEM
//                 A buffer (tcgen05.st).  Dequantized weights never touch
//                 shared memory.
//   last NEPI     epilogue (gemm_common.cuh epilogue_role).
// The A buffer index also names the B tile, so one A-empty commit frees both.
#include <mutex>

#include "gemm_common.cuh"

namespace qoq {
namespace {

template <int BN>
struct DecCfg {
  static constexpr int NSLOT = BN == 64 ? 2 : 4;  // dequant slots (one group each at a time)
  static constexpr int NDQ = 4 * NSLOT;
  static constexpr int NEPI = BN == 64 ? 8 : 4;
  static constexpr int DQ_WARP0 = 2;
  static constexpr int EPI_WARP0 = 2 + NDQ;
  static constexpr int THREADS = (2 + NDQ + NEPI) * 32;
  static constexpr int NACC = 2;
  static constexpr int ACOL0 = (NACC * BN + 63) / 64 * 64;
  // MMA hand-off in batches of 2 groups (16 MMAs per wait and commit): each
  // batch buffer is 2 x 64 TMEM columns of A plus 2 fp16 B tiles.
  static constexpr int NBATCH = (kTmemCols - ACOL0) / 128;
  static constexpr int B_BYTES = BN * kGroup * 2;
  static constexpr int B_TILES = 2 * NBATCH;
  static constexpr int STAGES_FIT = (kSmemBudget - 2048 - B_TILES * B_BYTES) / kWTileBytes;
  static constexpr int STAGES = STAGES_FIT > 16 ? 16 : STAGES_FIT;
  // Each slot has a sub-ring of SPS stages: one producer and one consumer per
  // stage, both in order, so a phase-parity wait can never be a lap ahead.
  static constexpr int SPS = STAGES / NSLOT;
  static constexpr int W_OFF = B_TILES * B_BYTES;
  static constexpr int BAR_OFF = W_OFF + STAGES * kWTileBytes;
  static constexpr int NBARS = 2 * STAGES + 2 * NBATCH + 2 * NACC + 1;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int FLAG_OFF = TMEM_SLOT_OFF + 8;
  static constexpr int SMEM_BYTES = FLAG_OFF + 8 + 1024;  // + slack for 1024-B alignment
  static_assert(BN == 16 || BN == 32 || BN == 64, "decode tiles");
  static_assert(NBATCH >= 2 && ACOL0 + 128 * NBATCH <= kTmemCols, "TMEM columns");
  static_assert(NSLOT % 2 == 0, "slot pairs fill a batch");
  static_assert(SPS >= 2, "pipeline depth per slot");
  static_assert(B_BYTES % 1024 == 0, "1024-B aligned B tiles");
  static_assert(SMEM_BYTES <= kSmemBudget, "shared memory");
};

// Position of a group in the batch sequence: batches of 2 consecutive groups
// start at each unit's first group (units and fold chunks have even group
// offsets, so no batch crosses either), and the last batch of an odd-sized
// unit holds one group.
struct BatchPos {
  uint32_t bi;  // global batch index in the CTA's work
  int pos;      // 0 or 1 within the batch
  int nb;       // groups in the batch (1 or 2)
};

// Per-slot counters of the producer (registers, no indexed local array).
template <int NSLOT>
struct SlotCounters {
  uint32_t c[4] = {0, 0, 0, 0};
  __device__ __forceinline__ uint32_t take(int slot) {
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < NSLOT; ++i)
      if (i == slot) v = c[i]++;
    return v;
  }
  __device__ __forceinline__ uint32_t count(int slot) const {
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < NSLOT; ++i)
      if (i == slot) v = c[i];
    return v;
  }
};

// Walks the groups of one dequant slot.  Within a unit, group g has batch
// position t = t0 + (g - g0), where t0 = 2 x (batches before the unit); its
// batch is t / 2, its place in the batch t % 2, and it belongs to slot
// t % NSLOT.  So a slot steps NSLOT positions at a time and only recomputes
// at unit boundaries (stepping through the other slots' groups one by one
// cost ~0.1 us per step on a sub-partition busy with dequant work).
// A unit of odd length ends with a one-group batch; its empty second place
// t0 + len is walked too, as a dummy entry: the slot that owns it waits for
// the batch's A buffer and arrives on it without writing.  So every slot takes
// part in every batch of its class (every NSLOT / 2-th batch), and its waits
// on an A buffer's phase parity always follow its own wait for the lap before
// (a slot that skipped a batch could otherwise pass a wait a lap early).
template <int NSLOT>
struct SlotWalk {
  UnitIter it;
  Unit u;
  bool have;
  int g, g_end, slot;  // g_end: end of the unit's positions, rounded up to a full batch
  uint32_t gi0, t0;    // index of the unit's first group; its batch position
  __device__ __forceinline__ void enter_unit() {
    g_end = u.g0 + 2 * ((u.g1 - u.g0 + 1) / 2);
    g = u.g0 + (int)(((uint32_t)slot - t0) & (NSLOT - 1));
  }
  __device__ __forceinline__ void init(const GemmParams& p, int slot_) {
    slot = slot_;
    it.init(p);
    gi0 = t0 = 0;
    have = it.next(p, u);
    if (have) enter_unit();
  }
  // dummy: the empty second place of a one-group batch (gi, tile, gg unused).
  __device__ __forceinline__ bool next(const GemmParams& p, int& tile, int& gg, uint32_t& gi, BatchPos& bp,
                                       bool& dummy) {
    while (have && g >= g_end) {
      const uint32_t len = (uint32_t)(u.g1 - u.g0);
      gi0 += len;
      t0 += 2 * ((len + 1) / 2);
      have = it.next(p, u);
      if (have) enter_unit();
    }
    if (!have) return false;
    const int off = g - u.g0;
    dummy = g >= u.g1;
    bp.pos = off & 1;
    bp.bi = (t0 + (uint32_t)off) >> 1;
    bp.nb = min(2, u.g1 - (g - bp.pos));
    tile = u.tile;
    gg = g;
    gi = gi0 + (uint32_t)off;
    g += NSLOT;
    return true;
  }
};

template <int BN>
__global__ void __launch_bounds__(DecCfg<BN>::THREADS, 1) gemm_decode_kernel(const __grid_constant__ GemmParams p) {
  using C = DecCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + C::BAR_OFF;
  const uint32_t bar_full = bars, bar_empty = bars + 8 * C::STAGES;
  const uint32_t bar_afull = bars + 8 * (2 * C::STAGES), bar_aempty = bar_afull + 8 * C::NBATCH;
  const uint32_t bar_accfull = bar_aempty + 8 * C::NBATCH, bar_accempty = bar_accfull + 8 * C::NACC;
  const uint32_t bar_drain = bar_accempty + 8 * C::NACC;

  if (threadIdx.x == 0) {
    QOQ_TRACE_AT(p, 0, 0);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 4);  // the 4 warps of the dequant slot that read the stage
    }
    for (int a = 0; a < C::NBATCH; ++a) {
      mbar_init(bar_afull + 8 * a, 8);  // 4 warps x 2 places (the empty place of a one-group batch too)
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
  if (threadIdx.x == 0) QOQ_TRACE_AT(p, 1, 0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    // Weights only: they do not depend on the preceding kernel, so the ring
    // fills while it runs.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();  // each weight tile is read once
      const uint8_t* const packed = p.packed;     // one token tile: weight tile index = tile
      const size_t tile_stride = (size_t)p.G * kWTileBytes;
      const uint32_t w_base = sbase + C::W_OFF;
      SlotCounters<C::NSLOT> taken;  // groups handed to each slot so far
      UnitIter iter;
      iter.init(p);
      Unit u;
      uint32_t gi = 0, t0 = 0;  // group index; batch position of the unit's first group
      bool ok = true;
      while (ok && iter.next(p, u)) {
        const uint8_t* src = packed + (size_t)u.tile * tile_stride + (size_t)u.g0 * kWTileBytes;
        for (int g = u.g0; g < u.g1; ++g, ++gi, src += kWTileBytes) {
          const int slot = (int)((t0 + (uint32_t)(g - u.g0)) % C::NSLOT);
          const uint32_t k = taken.take(slot);  // the slot's k-th group
          const int s = slot * C::SPS + (int)(k % C::SPS);
          if (k >= (uint32_t)C::SPS && !wait_bar(bar_empty + 8 * s, ((k / C::SPS) & 1) ^ 1, p)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_full + 8 * s, kWTileBytes);
          bulk_g2s(w_base + s * kWTileBytes, src, kWTileBytes, bar_full + 8 * s, pol);
          QOQ_TRACE_AT(p, 16 + (int)gi, 0);
        }
        t0 += 2 * (uint32_t)((u.g1 - u.g0 + 1) / 2);
      }
      // Let every copy still in flight land before the CTA may exit: the last
      // min(k, SPS) copies of each slot, one per stage of its sub-ring.
      for (int slot = 0; slot < C::NSLOT; ++slot) {
        const uint32_t n = taken.count(slot);
        for (uint32_t k = n > (uint32_t)C::SPS ? n - C::SPS : 0; k < n; ++k)
          wait_bar(bar_full + 8 * (slot * C::SPS + (int)(k % C::SPS)), (k / C::SPS) & 1, p, false);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer --
    // One converged warp, one wait and one commit per batch of 2 groups
    // (16 MMAs): the hand-off costs ~200 cycles, the 16 MMAs ~300.
    grid_dep_wait();
    constexpr uint32_t kIdesc = mma_idesc(BN);
    UnitIter iter;
    iter.init(p);
    Unit u;
    uint32_t bi = 0, chunk = 0;
    bool ok = true;
    while (ok && iter.next(p, u)) {
      for (int c0 = u.g0; c0 < u.g1; c0 += kFoldGroups) {
        const int c1 = min(u.g1, c0 + kFoldGroups);
        const int b = chunk % C::NACC;
        if (!warp_wait_bar(bar_accempty + 8 * b, ((chunk / C::NACC) & 1) ^ 1, p)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * BN;
        for (int g = c0; g < c1; g += 2, ++bi) {
          const int nb = min(2, c1 - g);
          const int a = bi % C::NBATCH;
          if (!warp_wait_bar(bar_afull + 8 * a, (bi / C::NBATCH) & 1, p)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) QOQ_TRACE_AT(p, 128 + (int)bi, 0);
          if (elect_one()) {
            for (int q = 0; q < nb; ++q) {
              const uint32_t b_lo = desc_sw128_lo(sbase + (uint32_t)((2 * a + q) * C::B_BYTES));
              const uint32_t a_col = tmem + C::ACOL0 + a * 128 + q * 64;
#pragma unroll
              for (int j = 0; j < 8; ++j)  // K step j: 64-channel half j / 4, 32-byte chunk j % 4
                tc_mma_ts(d_tmem, a_col + 8 * j, b_lo + (j >> 2) * (BN * 8) + (j & 3) * 2, kDescSw128Hi, kIdesc,
                           (g > c0 || q > 0 || j > 0) ? 1u : 0u);
            }
            tc_commit(bar_aempty + 8 * a);
          }
          __syncwarp();
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
    grid_dep_wait();  // Xq comes from the preceding kernel
    const int slot = (warp - C::DQ_WARP0) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int stid = ((warp - C::DQ_WARP0) & 3) * 32 + lane;  // 0..127 within the slot
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    SlotWalk<C::NSLOT> walk;
    walk.init(p, slot);
    int tile, g;
    uint32_t gi, nown = 0;  // groups of this slot so far: its position in its sub-ring
    BatchPos bp;
    bool dummy;
    while (walk.next(p, tile, g, gi, bp, dummy)) {
      const int a = bp.bi % C::NBATCH;
      if (dummy) {  // the empty place of a one-group batch: take part without data
        if (!wait_bar(bar_aempty + 8 * a, ((bp.bi / C::NBATCH) & 1) ^ 1, p)) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_afull + 8 * a);
        continue;
      }
      const int s = slot * C::SPS + (int)(nown % C::SPS);
      const uint32_t sph = (nown / C::SPS) & 1;
      ++nown;
      // int8 activation slice: 16-byte chunk q of the [BN][128] tile is row
      // q / 8, channels 16 (q % 8) .. +15; rows past M read as zero
      uint4 xv[BN / 16];
#pragma unroll
      for (int i = 0; i < BN / 16; ++i) {
        const int q = stid + i * 128;
        const int m = q >> 3;  // one token tile: rows 0 .. BN-1
        xv[i] = m < p.M ? __ldcg(reinterpret_cast<const uint4*>(p.xq + (size_t)m * p.K + g * kGroup + (q & 7) * 16))
                        : make_uint4(0, 0, 0, 0);
      }
      if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 192 + (int)gi, 0);
      if (!wait_bar(bar_full + 8 * s, sph, p)) break;
      if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 320 + (int)gi, 0);
      if (!wait_bar(bar_aempty + 8 * a, ((bp.bi / C::NBATCH) & 1) ^ 1, p)) break;
      tc_fence_after();  // the MMAs that read this batch buffer are complete
      if (quad == 0 && lane == 0) QOQ_TRACE_AT(p, 256 + (int)gi, 0);
      const uint8_t* wt = smem + C::W_OFF + s * kWTileBytes;
      const uint4 wv0 = *reinterpret_cast<const uint4*>(wt + kWNibOffset + 0 * kWChunkBytes + row * 16);
      const uint4 wv1 = *reinterpret_cast<const uint4*>(wt + kWNibOffset + 1 * kWChunkBytes + row * 16);
      const uint4 wv2 = *reinterpret_cast<const uint4*>(wt + kWNibOffset + 2 * kWChunkBytes + row * 16);
      const uint4 wv3 = *reinterpret_cast<const uint4*>(wt + kWNibOffset + 3 * kWChunkBytes + row * 16);
      const DequantConsts k = dequant_consts(wt[row], wt[128 + row]);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);  // the weight tile is in registers
      uint8_t* btile = smem + (2 * a + bp.pos) * C::B_BYTES;
#pragma unroll
      for (int i = 0; i < BN / 16; ++i) {
        const int q = stid + i * 128;
        store_b_chunk(btile, BN, q >> 3, q & 7, xv[i]);
      }
      fence_proxy_async_smem();  // generic-proxy writes -> the MMA's async-proxy reads
      const uint4 wv[4] = {wv0, wv1, wv2, wv3};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t out[16];
        dequant_chunk(wv[c], k, out);
        tmem_st16(tmem + lane_base + C::ACOL0 + a * 128 + bp.pos * 64 + c * 16, out);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (!(p.fault == 1 && gi == 17)) mbar_arrive(bar_afull + 8 * a);  // test hook: one group never arrives
        if (quad == 0) QOQ_TRACE_AT(p, 384 + (int)gi, 0);
        if (quad == 3) QOQ_TRACE_AT(p, 448 + (int)gi, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    grid_dep_wait();
    epilogue_role<BN, C::NEPI, C::NACC>(p, tmem, C::EPI_WARP0, bar_accfull, bar_accempty,
                                        reinterpret_cast<volatile int*>(smem + C::FLAG_OFF));
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

template <int BN>
cudaError_t launch_bn(const GemmParams& p, cudaStream_t s) {
  using C = DecCfg<BN>;
  static std::mutex mu;
  static uint64_t done_mask = 0;
  cudaError_t e;
  {
    std::lock_guard<std::mutex> lock(mu);
    e = set_smem_attr_once(gemm_decode_kernel<BN>, C::SMEM_BYTES, done_mask);
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
  return cudaLaunchKernelEx(&cfg, gemm_decode_kernel<BN>, p);
}

}  // namespace

cudaError_t launch_gemm_decode(const GemmParams& p, int BN, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_bn<16>(p, s);
    case 32: return launch_bn<32>(p, s);
    case 64: return launch_bn<64>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qoq
