// gemm.cu -- the W4A8 g128 GEMM: schedule, dispatch, and the kernel for
// 128-token tiles (M > 64).
//
// Computes, for Xq [M][K] int8 (per-token scale s_x) and the packed weights
// (level-2 codes q4, integer scale s2, zero z per group of g channels;
// level-1 fp16 scale s1 per output channel):
//   acc[m,n] = sum_k Xq[m,k] * ((q4[n,k] - z[n,k/g]) * s2[n,k/g])   (exact)
//   Y[m,n]   = fp16_rn(float(acc) * (float(s_x[m]) * float(s1[n])))
// QServe talk write-up, "Quantized Matrix Multiplication (GEMM) Kernel on
// GPUs" and "Challenges and Design Details": the 4-bit weights are
// dequantized to 8-bit integers before the tensor cores (never partial-sum
// dequant), the main loop is tensor-core work only, and the per-channel
// scales go to the epilogue.
//
// Two kernels share the roles of gemm_common.cuh:
//   * gemm_decode.cu, M <= 64: weights stream HBM -> registers -> TMEM.
//   * here, M > 64 (128-token tiles, compute bound): per 128-channel group a
//     producer warp issues one bulk copy of the packed weight tile (8448 B)
//     and one of the pre-swizzled fp16 activation tile (made once per call by
//     convert_kernel) into an S-stage shared-memory ring; NSLOT dequant slots
//     of 4 warps expand the weight tile from shared memory into the TMEM A
//     buffer; one MMA warp issues 8 x tcgen05.mma (M=128, N=128, K=16) per
//     group into one of two TMEM accumulators; 16 epilogue warps fold and
//     write.
// Every mbarrier wait is bounded; on expiry the CTA records
// QOQ_ERR_DEVICE_TIMEOUT in the workspace header, drains its copies and MMAs,
// frees its tensor memory and returns.
#include <algorithm>
#include <mutex>

#include "gemm_common.cuh"

namespace qoq {
namespace {

constexpr int kPrefetchStages = 4;  // weight stages issued before waiting on the preceding kernel

// GPT: level-2 scale sets per packed k-tile (g = 128 / GPT, or a multiple of
// 128 with GPT = 1).  PAIR: the CTA-pair form (each CTA stages its own weight
// tile and half of the token tile).
template <int GPT, bool PAIR = false>
struct BulkCfg {
  static constexpr int TILE = w_tile_bytes(GPT);  // packed k-tile bytes
  static constexpr int NIB = w_nib_offset(GPT);   // offset of its code chunks
  static constexpr int BN = 128;
  static constexpr int BROWS = PAIR ? BN / 2 : BN;  // token rows of B staged by this CTA
  static constexpr int NSLOT = 2;   // groups dequantized concurrently
  static constexpr int NDQ = 4 * NSLOT;
  static constexpr int NEPI = 16;   // 4 per TMEM lane quadrant, 32 tokens each
  static constexpr int EPI_WARP0 = 2 + NDQ;
  // Copy-issuing warps: warp 0, and with two the last warp of the CTA.  A
  // bulk copy takes a few hundred ns to issue while the SM is busy, so one
  // issuing thread paces the pair kernel's ring (one stage per ~320 ns at
  // M=128 before any wait); producer w serves the groups gi with gi % NPROD
  // == w from its own sub-ring of SPS stages.
  static constexpr int NPROD = PAIR ? 2 : 1;
  static constexpr int PROD2_WARP = EPI_WARP0 + NEPI;
  static constexpr int THREADS = (2 + NDQ + NEPI + (NPROD - 1)) * 32;
  static constexpr int NACC = 2;
  static constexpr int ACOL0 = NACC * BN;
  static constexpr int NABUF = (kTmemCols - ACOL0) / 64;
  static constexpr int B_BYTES = BROWS * kGroup * 2;
  static constexpr int STAGE_BYTES = B_BYTES + TILE;
  static constexpr int STAGES = (kSmemBudget - 4096) / STAGE_BYTES / NPROD * NPROD;  // 4 KB: barriers, scale ring, alignment
  static constexpr int SPS = STAGES / NPROD;  // stages per producer
  static constexpr int W_OFF = STAGES * B_BYTES;
  static constexpr int BAR_OFF = W_OFF + STAGES * TILE;
  static constexpr int NBARS = 2 * STAGES + 2 * NABUF + 2 * NACC + 1;
  static constexpr int SEQ_OFF = BAR_OFF + NBARS * 8;  // one 32-bit sequence word per stage
  static constexpr int TMEM_SLOT_OFF = SEQ_OFF + ((STAGES * 4 + 7) / 8) * 8;
  static constexpr int FLAG_OFF = TMEM_SLOT_OFF + 8;
  // W4Ax: ring of SCR slots of one group's block scales for the tile's 128
  // tokens (fp16, 256 B), filled by the producer's bulk copies, released by
  // the epilogue; its full / empty barriers follow.
  static constexpr int SCR = 8;
  static constexpr int SC_OFF = (FLAG_OFF + 8 + 255) / 256 * 256;
  static constexpr int SC_BAR_OFF = SC_OFF + SCR * 256;
  static constexpr int SMEM_BYTES = SC_BAR_OFF + 2 * SCR * 8 + 1024;  // + slack for 1024-B alignment
  static_assert(NABUF >= NSLOT + 1, "A buffers");
  static_assert(STAGES >= 3 && SPS >= 2, "pipeline depth");
  static_assert(NPROD == 1 || SCR % NPROD == 0, "each producer owns the scale slots of its groups");
  static_assert(SMEM_BYTES <= kSmemBudget, "shared memory");
};

// Stage of group gi (the CTA's gi-th group): sub-ring gi % NPROD, lap k / SPS
// of its k = gi / NPROD-th use.
struct StageRef {
  int s;
  uint32_t lap;
};
template <class C>
__device__ __forceinline__ StageRef stage_of(uint32_t gi) {
  const uint32_t k = gi / C::NPROD;
  return StageRef{(int)((gi % C::NPROD) * C::SPS + k % C::SPS), k / C::SPS};
}

// ZF: the zero-point-folded variant (see zero_point_share).  AX: the W4Ax
// product (one accumulator per group, scaled per activation block; see
// epilogue_role_ax).
// PAIR: launched in clusters of two CTAs (cluster rank = blockIdx.x % 2).  A
// unit's tile is a pair tile (256 weight rows x 128 tokens): CTA r stages
// weight tile 2 nt + r and tokens 64 r .. 64 r + 63 of every k-tile, dequantizes
// its weight tile into its own TMEM, and holds that tile's accumulators; the
// leading CTA (r = 0) issues the pair's M=256 MMAs, which read both CTAs'
// operands, once both CTAs' dequant slots have arrived on its A-full barrier.
// Each CTA's epilogue folds and writes its own 128 rows.  Half of every token
// tile per SM halves the activation bytes each SM stages per group (24.3 KB
// instead of 40.4 KB), so the same shared memory holds nine stages, not five.
template <int GPT, bool ZF, bool AX = false, bool PAIR = false>
__global__ void __launch_bounds__(BulkCfg<GPT, PAIR>::THREADS, 1)
    gemm_bulk_kernel(const __grid_constant__ GemmParams p) {
  static_assert(!(PAIR && (ZF || AX)), "the pair form covers the direct W4A8 product");
  using C = BulkCfg<GPT, PAIR>;
  constexpr int BN = C::BN;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;
  const uint32_t widx = PAIR ? blockIdx.x >> 1 : blockIdx.x;  // worker index of the schedule
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + C::BAR_OFF;
  const uint32_t bar_full = bars, bar_empty = bars + 8 * C::STAGES;
  const uint32_t bar_afull = bars + 8 * (2 * C::STAGES), bar_aempty = bar_afull + 8 * C::NABUF;
  const uint32_t bar_accfull = bar_aempty + 8 * C::NABUF, bar_accempty = bar_accfull + 8 * C::NACC;
  const uint32_t bar_drain = bar_accempty + 8 * C::NACC;
  // Stage s last armed for group seq[s] - 1 (0: never).  The two dequant slots
  // alternate groups over an odd number of stages, so a stage's consumer
  // changes from lap to lap; the sequence word keeps each consumer's parity
  // wait on the right lap.
  const uint32_t seq = sbase + C::SEQ_OFF;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      *reinterpret_cast<volatile uint32_t*>(smem + C::SEQ_OFF + 4 * s) = 0;
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1 + 4);  // MMA commit + the 4 warps of one dequant slot
    }
    for (int a = 0; a < C::NABUF; ++a) {
      mbar_init(bar_afull + 8 * a, PAIR ? 8 : 4);  // one dequant slot's warps (of both CTAs)
      mbar_init(bar_aempty + 8 * a, 1);
    }
    for (int b = 0; b < C::NACC; ++b) {
      mbar_init(bar_accfull + 8 * b, 1);
      mbar_init(bar_accempty + 8 * b, PAIR ? 2 * C::NEPI : C::NEPI);
    }
    mbar_init(bar_drain, 1);
    if (AX)
      for (int j = 0; j < C::SCR; ++j) {
        mbar_init(sbase + C::SC_BAR_OFF + 8 * j, 1);                   // scales landed
        mbar_init(sbase + C::SC_BAR_OFF + 8 * (C::SCR + j), C::NEPI);  // epilogue done with them
      }
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_alloc_pair(sbase + C::TMEM_SLOT_OFF, kTmemCols);
    else
      tmem_alloc(sbase + C::TMEM_SLOT_OFF, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // both CTAs' barriers exist before either arrives remotely
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::TMEM_SLOT_OFF);

  if (warp == 0 || (C::NPROD > 1 && warp == C::PROD2_WARP)) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      const uint32_t w = warp == 0 ? 0u : 1u;  // this producer's groups: gi % NPROD == w
      const uint64_t pol = policy_evict_last();  // weights and activations are both re-read
      UnitIter iter;
      iter.init(p, widx);
      Unit u;
      bool have = iter.next(p, u);
      int g = have ? u.g0 : 0;
      uint32_t gi = 0;
      uint32_t issued_mask = 0, issued_par = 0;  // per stage: last issue and its parity
      constexpr uint32_t kStageTx = C::TILE + C::B_BYTES;
      // the current unit's tile coordinates (computed once per unit)
      TileXY xy = have ? tile_xy(p, u.tile) : TileXY{0, 0};
      auto advance = [&]() {  // to this producer's next group
        do {
          ++gi;
          if (++g >= u.g1) {
            have = iter.next(p, u);
            if (have) {
              g = u.g0;
              xy = tile_xy(p, u.tile);
            }
          }
        } while (have && gi % C::NPROD != w);
      };
      if (have && gi % C::NPROD != w) advance();
      auto issue_w = [&](int s, int nt, int gg) {
        const int wt = PAIR ? 2 * nt + (int)rank : nt;  // this CTA's weight tile
        const uint8_t* src = p.packed + ((size_t)wt * p.G + gg) * C::TILE;
        bulk_g2s(sbase + C::W_OFF + s * C::TILE, src, C::TILE, bar_full + 8 * s, pol);
      };
      auto issue_x = [&](int s, int mt, int gg) {
        // PAIR: this CTA's token half of the block, [2][64][64] fp16 in one piece
        const uint16_t* src = p.xh + ((size_t)mt * p.G + gg) * (BN * kGroup) + (size_t)rank * (C::BROWS * kGroup);
        bulk_g2s(sbase + s * C::B_BYTES, src, C::B_BYTES, bar_full + 8 * s, pol);
      };
      // W4Ax: group number q's block scales into ring slot q % SCR (with two
      // producers, each owns the slots of its groups' parity)
      uint32_t sc_mask = 0, sc_par = 0;  // per slot: a copy in its latest lap; its parity
      auto issue_sc = [&](uint32_t qn, int mt, int gg) -> bool {
        if (!AX) return true;
        const int j = (int)(qn % C::SCR);
        const uint32_t ph = (qn / C::SCR) & 1;
        if (qn >= (uint32_t)C::SCR && !wait_bar(sbase + C::SC_BAR_OFF + 8 * (C::SCR + j), ph ^ 1, p)) return false;
        const uint32_t full = sbase + C::SC_BAR_OFF + 8 * j;
        mbar_arrive_expect_tx(full, 256);
        bulk_g2s(sbase + C::SC_OFF + 256 * j, p.sxT + (size_t)gg * p.sxT_ld + (size_t)mt * BN, 256, full, pol);
        sc_mask |= 1u << j;
        sc_par = (sc_par & ~(1u << j)) | (ph << j);
        return true;
      };
      // Weights do not depend on the preceding kernels: issue a few stages
      // before waiting on them.
      constexpr int kPre = kPrefetchStages / C::NPROD < C::SPS ? kPrefetchStages / C::NPROD : C::SPS;
      int npre = 0;
      int pre_mt[kPre], pre_g[kPre], pre_s[kPre];
      uint32_t pre_gi[kPre];
      while (have && npre < kPre) {  // first lap of the sub-ring: no stage to wait for
        const StageRef st = stage_of<C>(gi);
        mbar_arrive_expect_tx(bar_full + 8 * st.s, kStageTx);
        issue_w(st.s, xy.nt, g);
        st_release_shared(seq + 4 * st.s, gi + 1);
        pre_mt[npre] = xy.mt;
        pre_g[npre] = g;
        pre_s[npre] = st.s;
        pre_gi[npre] = gi;
        issued_mask |= 1u << st.s;
        ++npre;
        advance();
      }
      grid_dep_wait();
      bool sc_ok = true;
      for (int i = 0; i < npre; ++i) {
        issue_x(pre_s[i], pre_mt[i], pre_g[i]);
        if (sc_ok) sc_ok = issue_sc(pre_gi[i], pre_mt[i], pre_g[i]);
      }
      while (have && sc_ok) {
        const StageRef st = stage_of<C>(gi);
        const uint32_t ph = st.lap & 1;
        if (st.lap > 0 && !wait_bar<PAIR>(bar_empty + 8 * st.s, ph ^ 1, p)) break;  // released by the pair's MMA too
        if (!issue_sc(gi, xy.mt, g)) break;
        if (!(p.fault == 1 && gi == (uint32_t)C::STAGES + 1)) {  // test hook: skip one stage
          mbar_arrive_expect_tx(bar_full + 8 * st.s, kStageTx);
          issue_w(st.s, xy.nt, g);
          issue_x(st.s, xy.mt, g);
          st_release_shared(seq + 4 * st.s, gi + 1);
          issued_mask |= 1u << st.s;
          issued_par = (issued_par & ~(1u << st.s)) | (ph << st.s);
        } else {
          issued_mask &= ~(1u << st.s);
        }
        advance();
      }
      // Let every copy still in flight land before the CTA may exit.
      for (int s = 0; s < C::STAGES; ++s)
        if (issued_mask & (1u << s)) wait_bar(bar_full + 8 * s, (issued_par >> s) & 1, p, false);
      for (int j = 0; j < C::SCR; ++j)
        if (sc_mask & (1u << j)) wait_bar(sbase + C::SC_BAR_OFF + 8 * j, (sc_par >> j) & 1, p, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer --
    grid_dep_wait();
    if (rank == 0)  // of a pair, the leading CTA issues
      mma_role<BN, C::NACC, C::NABUF, C::ACOL0, AX ? 1 : (ZF ? kFoldGroupsZf : kFoldGroups), PAIR>(
          p, tmem, bar_afull, bar_aempty, bar_accfull, bar_accempty, bar_drain,
          [&](uint32_t gi, int) { return sbase + (uint32_t)(stage_of<C>(gi).s * C::B_BYTES); },
          [&](uint32_t gi) { return bar_empty + 8 * stage_of<C>(gi).s; });
  } else if (warp < C::EPI_WARP0) {
    // ------------------------------------------------------------- dequant --
    grid_dep_wait();
    const int quad = warp & 3;
    const int slot = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    UnitIter iter;
    iter.init(p, widx);
    Unit u;
    uint32_t gi = 0;
    bool ok = true;
    while (ok && iter.next(p, u)) {
      for (int g = u.g0; g < u.g1; ++g, ++gi) {
        if ((int)(gi % C::NSLOT) != slot) continue;
        const StageRef st = stage_of<C>(gi);
        const int s = st.s;
        const int a = gi % C::NABUF;
        // every lane waits, then the warp votes: it reaches the tensor memory
        // stores below converged (see conv_wait_bar)
        const bool got = wait_seq(seq + 4 * s, gi + 1, p) && wait_bar(bar_full + 8 * s, st.lap & 1, p) &&
                         wait_bar<PAIR>(bar_aempty + 8 * a, ((gi / C::NABUF) & 1) ^ 1, p);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read this A buffer are complete
        const uint8_t* wt = smem + C::W_OFF + s * C::TILE;
        DequantConsts k = dequant_consts(wt[row], ZF ? 0u : wt[128 + row]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (GPT > 1 && c > 0 && c % (4 / GPT) == 0) {  // scale set u covers chunks u * 4 / GPT ..
            const int u = c / (4 / GPT);
            k = dequant_consts(wt[u * 256 + row], ZF ? 0u : wt[u * 256 + 128 + row]);
          }
          uint32_t out[16];
          dequant_chunk(*reinterpret_cast<const uint4*>(wt + C::NIB + c * kWChunkBytes + row * 16), k, out);
          tmem_st16(tmem + lane_base + C::ACOL0 + a * 64 + c * 16, out);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && rank != 0)
            mbar_arrive_remote(bar_afull + 8 * a, 0);  // the pair's MMAs are issued by the leading CTA
          else
            mbar_arrive(bar_afull + 8 * a);
          mbar_arrive(bar_empty + 8 * s);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    grid_dep_wait();
    if constexpr (AX)
      epilogue_role_ax<BN, C::NEPI, C::NACC, C::SCR>(p, tmem, C::EPI_WARP0, bar_accfull, bar_accempty,
                                                    reinterpret_cast<volatile int*>(smem + C::FLAG_OFF),
                                                    sbase + C::SC_OFF, sbase + C::SC_BAR_OFF);
    else
      epilogue_role<BN, C::NEPI, C::NACC, ZF, C::TILE, ZF ? kFoldGroupsZf : kFoldGroups, PAIR>(
          p, tmem, C::EPI_WARP0, bar_accfull, bar_accempty, reinterpret_cast<volatile int*>(smem + C::FLAG_OFF));
  }

  tc_fence_before();
  __syncthreads();
  // A pair's MMAs read both CTAs' shared and tensor memory: neither CTA frees
  // or leaves before the leading CTA's issuer has drained them.
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

// fp16 copy of Xq in the B-operand layout for 128-token tiles: [MT][G][2][128][64]
// fp16, each [128][64] block 128B-swizzled (16-byte chunk c of row r stored at
// chunk c ^ (r & 7)), rows m >= M zero; with c.split, [MT][G][2][2][64][64]
// (token half, then channel half) for the CTA-pair kernel.
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
    if (m < c.M) raw = __ldcg(reinterpret_cast<const uint4*>(c.Xq + (size_t)m * c.K + k0));  // L2: from the preceding kernel
    const int g = k0 / kGroup, kc = (k0 % kGroup) / 16;
    const int mt = m / c.BN, r = m % c.BN;
    uint8_t* blk = reinterpret_cast<uint8_t*>(c.xh + (size_t)(mt * G + g) * c.BN * kGroup);
    if (c.split)  // half r / 64 of the block, rows in the same 128B-swizzle phase (r % 64 = r mod 8 too)
      store_b_chunk(blk + (r / 64) * (64 * kGroup * 2), 64, r % 64, kc, raw);
    else
      store_b_chunk(blk, c.BN, r, kc, raw);
  }
}

// Sixteen 4-bit two's-complement codes (8 bytes, channel 2i in the low nibble
// of byte i) -> sixteen int8 lanes in channel order: flip each code's sign bit
// (offset binary t = code + 8 in [0, 15]), split even and odd channels into
// bytes, interleave them, and sign-extend with ((t | 0x80) - 8) ^ 0x80 = t - 8
// per byte, which borrows across no byte boundary.
__device__ __forceinline__ uint4 expand_nibbles16(uint2 h) {
  uint32_t out[4];
  const uint32_t w2[2] = {h.x, h.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t t = w2[i] ^ 0x88888888u;  // offset binary: code + 8
    const uint32_t ev = t & 0x0F0F0F0Fu, od = (t >> 4) & 0x0F0F0F0Fu;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(a) : "r"(ev), "r"(od));  // channels 0..3 of the word
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(b) : "r"(ev), "r"(od));  // channels 4..7
    out[2 * i] = ((a | 0x80808080u) - 0x08080808u) ^ 0x80808080u;
    out[2 * i + 1] = ((b | 0x80808080u) - 0x08080808u) ^ 0x80808080u;
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// W4Ax: the fp16 B-operand copy ([MT][G][2][128][64], as convert_kernel
// writes it) from the mixed activation rows (n8 leading 8-bit blocks of 128
// bytes, then 4-bit blocks of 64 bytes), and the block scales transposed to
// [G][MT * 128] (0 for tokens past M) for the epilogue's per-group loads.
__global__ void __launch_bounds__(256) convert_w4ax_kernel(const ConvertAxParams c) {
  grid_dep_launch_dependents();  // the GEMM may launch and start streaming weights
  grid_dep_wait();               // the activations come from the preceding kernel
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int G = c.K / kGroup;
  const size_t row_bytes = (size_t)128 * c.n8 + (size_t)64 * (G - c.n8);
  const long long total = (long long)c.MT * 128 * (c.K / 16);
  for (long long idx = tid; idx < total; idx += stride) {
    const int m = (int)(idx / (c.K / 16));
    const int k0 = (int)(idx % (c.K / 16)) * 16;
    const int b = k0 / kGroup, kc = (k0 % kGroup) / 16;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (m < c.M) {
      const uint8_t* rowp = c.Xa + (size_t)m * row_bytes;
      if (b < c.n8)
        raw = __ldcg(reinterpret_cast<const uint4*>(rowp + (size_t)128 * b + 16 * kc));
      else
        raw = expand_nibbles16(__ldcg(reinterpret_cast<const uint2*>(rowp + (size_t)128 * c.n8 +
                                                                   (size_t)64 * (b - c.n8) + 8 * kc)));
    }
    const int mt = m / 128, r = m % 128;
    store_b_chunk(reinterpret_cast<uint8_t*>(c.xh + (size_t)(mt * G + b) * 128 * kGroup), 128, r, kc, raw);
  }
  const long long nsc = (long long)G * c.sxT_ld;
  for (long long idx = tid; idx < nsc; idx += stride) {
    const int b = (int)(idx / c.sxT_ld), m = (int)(idx % c.sxT_ld);
    c.sxT[idx] = m < c.M ? c.sxb[(size_t)m * G + b] : (uint16_t)0;
  }
}

// Row sums of Xq per 128-channel k-tile, RS[j][m] (0 for M <= m < rs_ld),
// for the zero-point-folded variant.  One thread per (j, m): 128 bytes read,
// summed four signed bytes at a time.
__global__ void __launch_bounds__(256) rowsum_kernel(const RowSumParams r) {
  grid_dep_launch_dependents();  // the GEMM may launch and start streaming weights
  grid_dep_wait();               // Xq comes from the preceding kernel
  const long long total = (long long)(r.K / kGroup) * r.rs_ld;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int j = (int)(idx / r.rs_ld), m = (int)(idx % r.rs_ld);
    int sum = 0;
    if (m < r.M) {
      const uint4* x = reinterpret_cast<const uint4*>(r.Xq + (size_t)m * r.K + (size_t)j * kGroup);
#pragma unroll
      for (int q = 0; q < kGroup / 16; ++q) {
        const uint4 v = __ldcg(x + q);
        sum = __dp4a((int)v.x, 0x01010101, sum);
        sum = __dp4a((int)v.y, 0x01010101, sum);
        sum = __dp4a((int)v.z, 0x01010101, sum);
        sum = __dp4a((int)v.w, 0x01010101, sum);
      }
    }
    r.rs[idx] = sum;
  }
}

template <int GPT, bool ZF, bool AX = false>
cudaError_t launch_bulk_g(const GemmParams& p, cudaStream_t s) {
  using C = BulkCfg<GPT>;
  static std::mutex mu;
  static uint64_t done_mask = 0;
  cudaError_t e;
  {
    std::lock_guard<std::mutex> lock(mu);
    e = set_smem_attr_once(gemm_bulk_kernel<GPT, ZF, AX>, C::SMEM_BYTES, done_mask);
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
  return cudaLaunchKernelEx(&cfg, gemm_bulk_kernel<GPT, ZF, AX>, p);
}

cudaError_t launch_bulk_ax(const GemmParams& p, cudaStream_t s) {
  switch (p.gpt) {
    case 1: return launch_bulk_g<1, false, true>(p, s);
    case 2: return launch_bulk_g<2, false, true>(p, s);
    case 4: return launch_bulk_g<4, false, true>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bulk(const GemmParams& p, bool zero_folded, cudaStream_t s) {
  if (zero_folded) return p.gpt == 1 ? launch_bulk_g<1, true>(p, s) : cudaErrorInvalidValue;
  switch (p.gpt) {
    case 1: return launch_bulk_g<1, false>(p, s);
    case 2: return launch_bulk_g<2, false>(p, s);
    case 4: return launch_bulk_g<4, false>(p, s);
    default: return cudaErrorInvalidValue;
  }
}


// The CTA-pair kernel: clusters of two CTAs, p.P pairs.
template <int GPT>
cudaError_t launch_pair_g(const GemmParams& p, cudaStream_t s) {
  using C = BulkCfg<GPT, true>;
  static std::mutex mu;
  static uint64_t done_mask = 0;
  cudaError_t e;
  {
    std::lock_guard<std::mutex> lock(mu);
    e = set_smem_attr_once(gemm_bulk_kernel<GPT, false, false, true>, C::SMEM_BYTES, done_mask);
  }
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.P);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0] = pdl_attr();
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_bulk_kernel<GPT, false, false, true>, p);
}

cudaError_t launch_pair(const GemmParams& p, cudaStream_t s) {
  switch (p.gpt) {
    case 1: return launch_pair_g<1>(p, s);
    case 2: return launch_pair_g<2>(p, s);
    case 4: return launch_pair_g<4>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

// CTA pairs of the pair kernel that fit on the current device at once (one
// CTA per SM; a GPC with an odd number of free SMs leaves one out), cached per
// device.  0 if the query fails.
int pair_capacity() {
  static std::mutex mu;
  static int cached[64];
  static bool have[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && have[dev]) return cached[dev];
  using C = BulkCfg<1, true>;
  uint64_t done_mask = 0;
  if (set_smem_attr_once(gemm_bulk_kernel<1, false, false, true>, C::SMEM_BYTES, done_mask) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (kMaxGrid / 2));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_bulk_kernel<1, false, false, true>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (dev < 64) {
    cached[dev] = n;
    have[dev] = true;
  }
  return n;
}

// Whole tiles round-robin over the P0 persistent workers (CTAs, or CTA pairs);
// when the last wave would be partial, it and one full wave are split along K
// instead (stream-K), so every worker gets the same number of groups.
void make_schedule(GemmParams& p, int P0) {
  P0 = std::max(1, P0);
  if (p.T >= P0) {
    const int rem = p.T % P0;
    p.T_sk = rem == 0 ? 0 : std::min(p.T, rem + P0);
    p.T_dp = p.T - p.T_sk;
    p.P = P0;
  } else {
    p.T_dp = 0;
    p.T_sk = p.T;
    const long long want = ((long long)p.T * p.G + 3) / 4;  // at least ~4 groups per worker
    p.P = (int)std::max<long long>(1, std::min<long long>(P0, want));
  }
  p.I_sk = (uint32_t)p.T_sk * (uint32_t)p.G;  // T_sk <= 2 P0 - 1 <= 511, G <= 1024
}
}  // namespace

cudaError_t launch_gemm(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx,
                        const uint8_t* packed, const uint16_t* s1, uint16_t* Y, int32_t* acc_debug,
                        void* ws, int num_sms, unsigned long long timeout_ns, int fault,
                        unsigned call_id, unsigned long long* trace, bool zero_folded, cudaStream_t s) {
  const int BN = gemm_bn_for_m(M);
  const WsLayout L = gemm_ws_layout(M, N, K);
  GemmParams p = {};
  p.M = M;
  p.N = N;
  p.K = K;
  p.G = K / kGroup;
  p.gpt = gpt_for_group(g);
  p.MT = (M + BN - 1) / BN;
  // The direct product of 128-token tiles runs on CTA pairs (M=256 MMAs, each
  // SM staging half of every token tile) when N is a multiple of 256; then a
  // tile is a pair tile of 256 weight rows.
  const int pairs = std::min(num_sms, kMaxGrid) / 2;
  const int cap = (BN == 128 && !zero_folded && N % (2 * kTileN) == 0 && pairs > 0) ? pair_capacity() : 0;
  const bool pair = cap > 0;
  p.NT = N / (pair ? 2 * kTileN : kTileN);
  p.T = p.MT * p.NT;
  make_schedule(p, pair ? std::min(pairs, cap) : std::min(num_sms, kMaxGrid));
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.status = reinterpret_cast<int*>(w);
  p.sk_cnt = reinterpret_cast<int32_t*>(w + L.cnt_off);
  p.sk_acc = reinterpret_cast<int32_t*>(w + L.acc_off);
  p.sk_slot = reinterpret_cast<unsigned long long*>(w + L.slot_off);
  p.xh = reinterpret_cast<const uint16_t*>(w + L.xh_off);
  p.xq = Xq;
  p.packed = packed;
  p.sx = sx;
  p.s1 = s1;
  p.Y = Y;
  p.acc_debug = acc_debug;
  p.timeout_ns = timeout_ns;
  p.fault = fault;
  p.call_id = call_id;
  p.trace = trace;
  p.rs = reinterpret_cast<const int32_t*>(w + L.rs_off);
  p.rs_ld = L.rs_ld;
  const int P0 = std::max(1, std::min(num_sms, kMaxGrid));

  if (zero_folded) {
    if (p.gpt != 1) return cudaErrorInvalidValue;
    RowSumParams r = {};
    r.Xq = Xq;
    r.rs = reinterpret_cast<int32_t*>(w + L.rs_off);
    r.M = M;
    r.K = K;
    r.rs_ld = L.rs_ld;
    const long long work = (long long)p.G * L.rs_ld;
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3((unsigned)std::max<long long>(1, std::min<long long>((work + 255) / 256, (long long)P0 * 4)));
    rcfg.blockDim = dim3(256);
    rcfg.stream = s;
    cudaLaunchAttribute rattr[1] = {pdl_attr()};
    rcfg.attrs = rattr;
    rcfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&rcfg, rowsum_kernel, r);
    if (e != cudaSuccess) return e;
  }

  if (BN <= 64) {
    if (p.MT != 1) return cudaErrorInvalidValue;  // the decode kernel holds all M tokens in one tile
    return launch_gemm_decode(p, BN, zero_folded, s);
  }

  ConvertParams c = {};
  c.Xq = Xq;
  c.xh = reinterpret_cast<uint16_t*>(w + L.xh_off);
  c.M = M;
  c.K = K;
  c.BN = BN;
  c.MT = p.MT;
  c.split = pair ? 1 : 0;
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
  return pair ? launch_pair(p, s) : launch_bulk(p, zero_folded, s);
}

cudaError_t launch_w4ax(int M, int N, int K, int g, int n8, const uint8_t* Xa, const uint16_t* sxb,
                        const uint8_t* packed, const uint16_t* s1, uint16_t* Y, int32_t* acc_debug, void* ws,
                        int num_sms, unsigned long long timeout_ns, unsigned call_id, cudaStream_t s) {
  constexpr int BN = 128;
  const WsLayout L = w4ax_ws_layout(M, N, K);
  GemmParams p = {};
  p.M = M;
  p.N = N;
  p.K = K;
  p.G = K / kGroup;
  p.gpt = gpt_for_group(g);
  p.MT = (M + BN - 1) / BN;
  p.NT = N / kTileN;
  p.T = p.MT * p.NT;
  const int P0 = std::max(1, std::min(num_sms, kMaxGrid));
  make_schedule(p, P0);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.status = reinterpret_cast<int*>(w);
  p.sk_cnt = reinterpret_cast<int32_t*>(w + L.cnt_off);
  p.sk_acc = reinterpret_cast<int32_t*>(w + L.acc_off);
  p.xh = reinterpret_cast<const uint16_t*>(w + L.xh_off);
  p.sxT = reinterpret_cast<const uint16_t*>(w + L.rs_off);
  p.sxT_ld = L.rs_ld;
  p.packed = packed;
  p.s1 = s1;
  p.Y = Y;
  p.timeout_ns = timeout_ns;
  p.call_id = call_id;

  ConvertAxParams c = {};
  c.Xa = Xa;
  c.sxb = sxb;
  c.xh = reinterpret_cast<uint16_t*>(w + L.xh_off);
  c.sxT = reinterpret_cast<uint16_t*>(w + L.rs_off);
  c.M = M;
  c.K = K;
  c.n8 = n8;
  c.MT = p.MT;
  c.sxT_ld = L.rs_ld;
  const long long work = (long long)p.MT * BN * (K / 16);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max<long long>(1, std::min<long long>((work + 255) / 256, (long long)P0 * 4)));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, convert_w4ax_kernel, c);
  if (e != cudaSuccess) return e;
  e = launch_bulk_ax(p, s);
  if (e != cudaSuccess || !acc_debug) return e;
  // sum_b acc_b for checking: the plain kernel on the same operand copy,
  // integer folds every 8 groups, acc_debug written, no Y
  GemmParams d = p;
  d.Y = nullptr;
  d.acc_debug = acc_debug;
  d.call_id = call_id + 1 ? call_id + 1 : 1;
  return launch_bulk(d, false, s);
}

}  // namespace qoq
