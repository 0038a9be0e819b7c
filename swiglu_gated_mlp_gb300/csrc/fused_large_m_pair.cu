// Large-M fused SwiGLU kernel on CTA pairs: Y = SiLU(A W1) * (A W2) for
// 256-token tiles computed by two SMs with tcgen05.mma.cta_group::2.
//
// Same method as fused_large_m.cu (one packed weight stream, gate and up
// columns side by side in one fp32 TMEM accumulator, SiLU * mul epilogue
// overlapped with the next tile's MMAs; "Tile-Level Activation Overlap for
// Efficient LLM Inference", gist.science, section "Methodology"), with the
// operand traffic of each SM cut by a third:
//
//  * a cluster of two CTAs owns a 256 x 128 output tile; CTA rank r loads A
//    rows [128 r, 128 r + 128) of the tile and packed-weight rows
//    [128 r, 128 r + 128) of the (column block, K slice) tile, i.e. rank 0
//    the 128 gate columns and rank 1 the 128 matching up columns;
//  * rank 0 issues one MMA of M=256, N=256, K=16 per step over both CTAs'
//    shared memory; each CTA's TMEM receives its 128 rows x (128 gate | 128 up)
//    columns, so each CTA's epilogue is the single-CTA one;
//  * per 64-deep K step each CTA pulls 32 KB (16 KB A + 16 KB W) instead of
//    48 KB, and the ring holds 6 stages;
//  * both CTAs' loads complete on rank 0's "full" barrier; rank 0's MMA
//    completions arrive on both CTAs' "empty" and "accumulator full"
//    barriers (multicast commit); both epilogues arrive on rank 0's
//    "accumulator empty" barrier; every wait is bounded (ptx.cuh).
//
// Tile rounds are kept loosely in step across the pairs: pair p takes tiles
// p, p + pairs, p + 2 pairs, ... (round 0, 1, 2, ...), and the tiles of one
// round share A rows and weight columns through L2 only while the pairs are
// near each other. Left alone, pairs drift apart by whole rounds over a long
// run (the 72B prefill read its operands 7-11 times over from DRAM), so the
// even CTA's producer, before the loads of its round r tile, waits until every
// pair has issued all loads of its round r - 2 tile (a per-round counter in
// global memory, tagged with a launch number the CTAs draw on the device, so
// graph replays count apart: every launch takes one block of kPaceBlock
// numbers from a global ticket, pair 0 all but pairs - 1 of them, so blocks
// stay aligned whatever the grid sizes of earlier launches). Every such wait
// is bounded and, if it runs out, only turns pacing off for the rest of the
// launch; results never depend on it. Paced are bf16 gate/up launches with
// K >= 8192 (long tiles; the 72B prefill): DRAM reads 11.0-13.4 -> 7.9-8.8 GB
// per launch at the same time (lag 1: much slower; lag 4: more reads).
// Shorter tiles lose time when paced, since the slowest pair of each round
// then sets everyone's pace. Consecutive rounds share their A rows (a row
// group's tiles run down the columns), so on the paced shapes odd rounds
// walk K backwards and start on the A slices the previous round loaded last,
// while L2 still holds them: the 72B prefill read 8.0 -> 6.3 GB and ran 2 %
// faster. Unpaced launches keep one direction: their pairs drift apart by
// whole rounds, so the tiles in flight would mix both directions (before the
// pacing, alternating directions raised the reads of both 72B forms).
//
// With kDown the same pipeline computes the MLP's down-projection
// Out = Y x W3 + R: a tile is 256 consecutive output columns (rank r loads
// packed rows [128 r, 128 r + 128) of W3's tile), and the epilogue stores
// accumulator + residual for all 256 columns.
//
// With kMx (block-scaled E4M3: one power-of-two scale per 32 K values) each
// CTA also loads, per stage, the scale block of its 128 A rows and both of the
// packed tile's weight-scale blocks (gate, up: the MMA's 256 B columns). A
// warp of the even CTA of its own copies them, as soon as a stage has landed,
// into that stage's slot of both CTAs' tensor memory (tcgen05.cp.cta_group::2,
// each CTA from its own shared memory) and signals their completion on a
// per-stage barrier; the MMA issuer waits for it and issues kind::mxf8f6f4
// MMAs, so the copies never sit in the MMA issuer's own stream of tensor
// instructions (copies issued there, just before the MMAs that read them,
// left the tensor pipe idle for a while at every stage; issuing them one stage
// early there was slower still). The scale slots take the second half of
// tensor memory, so the accumulator is single-buffered: the next tile's MMAs
// wait for the epilogue to have read the previous one. To keep that wait short the
// block-scaled form runs 8 epilogue warps (two per tensor-memory lane
// quarter, 64 output columns each) that load their whole share of the
// accumulator into registers, release it at once, and only then apply
// SiLU(g) * u and store, each through one store-staging buffer of its own
// (the wait on its previous store overlaps the next tile's MMAs).
#include "kernels.h"
#include "ptx.cuh"

namespace swg {
namespace {

template <bool kMx>
struct PairCfg {
  static constexpr int kBN = 128;                        // output columns per tile
  static constexpr int kABytes = 128 * kBlockK * 2;      // 16 KB: this CTA's 128 A rows
  static constexpr int kBBytes = 128 * kBlockK * 2;      // 16 KB: this CTA's 128 weight rows
  static constexpr int kStageBytes = kABytes + kBBytes;  // 32 KB per CTA, 64 KB per pair
  static constexpr int kStages = 6;
  static constexpr int kEpiWarps = kMx ? 8 : 4;          // 2 per lane quarter when block-scaled
  // TMA producer and MMA issuer warps, the epilogue warps, and (block-scaled)
  // a warp that copies each stage's scales into tensor memory
  static constexpr int kThreadsT = 64 + 32 * kEpiWarps + (kMx ? 32 : 0);
  static constexpr int kAccCols = 2 * kBN;               // 256 fp32 columns: gate | up
  static constexpr int kTmemCols = 2 * kAccCols;         // double buffered (bf16, per-tensor FP8)
  static constexpr int kStgBytes = 32 * 32 * 2;          // 32 rows x 64 B store staging
  static constexpr int kNumStg = 8;                      // 2 per warp, or 1 per warp with 8 warps
  static constexpr int kBarBytes = 256;
  // block-scaled FP8: 1.5 KB of scales per stage (A block, gate and up weight blocks)
  static constexpr size_t kSmem = 1024 + size_t(kStages) * kStageBytes +
                                  size_t(kNumStg) * kStgBytes +
                                  (kMx ? size_t(kStages) * kSfStageBytes : 0) + kBarBytes;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(8 * (3 * kStages + 6) + 8 <= kBarBytes, "barrier slots");
  static constexpr int kSfCol = kAccCols;  // scale slots after the single accumulator
  static_assert(!kMx || kSfCol + kStages * kSfTmemCols <= kTmemCols, "tensor memory budget");
};

__device__ __forceinline__ void pair_tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                                 int& mb, int& nb) {
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int gm = min(tiles_m - first_m, group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

// Round pacing state (see the head of this file): the even CTA of every pair
// draws from g_pace_ticket, launch number = ticket / kPaceBlock + 1 (32 bits);
// g_pace_round[r] holds (launch number << 32) | pairs that issued all loads of
// their round r tile; g_pace_run_out counts waits that ran out (testing).
constexpr int kPaceLag = 2;
constexpr int kPaceRounds = 1024;               // rounds beyond this are not paced
constexpr uint64_t kPaceWaitNs = 200000;        // one wait's limit: then pacing stops
constexpr int kPaceMinSlices = 128;             // paced only with K >= 128 slices of 64
constexpr unsigned long long kPaceBlock = 1024;  // tickets per launch (>= pairs)
__device__ unsigned long long g_pace_ticket;
__device__ unsigned long long g_pace_round[kPaceRounds];
__device__ unsigned long long g_pace_run_out;

// Waits (bounded) until `need` pairs of launch `epoch` counted themselves in
// round r; false if the wait ran out or a later launch owns the counter.
__device__ __forceinline__ bool pace_wait(int r, unsigned long long epoch, unsigned need) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    const unsigned long long v = *reinterpret_cast<volatile unsigned long long*>(&g_pace_round[r]);
    if ((v >> 32) == epoch && static_cast<unsigned>(v & 0xffffffffull) >= need) return true;
    if ((v >> 32) > epoch) return false;
    if (globaltimer_ns() - t0 > kPaceWaitNs) {
      atomicAdd(&g_pace_run_out, 1ull);
      return false;
    }
  }
}

// Counts this pair in for round r of launch `epoch` (a counter left by
// another launch restarts at 1).
__device__ __forceinline__ void pace_count(int r, unsigned long long epoch) {
  unsigned long long* c = &g_pace_round[r];
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(c), assumed;
  do {
    assumed = old;
    const unsigned long long next = (assumed >> 32) == epoch ? assumed + 1ull : (epoch << 32) | 1ull;
    old = atomicCAS(c, assumed, next);
  } while (old != assumed);
}

template <bool kFp8, bool kDown, bool kMx>
__global__ void __launch_bounds__(PairCfg<kMx>::kThreadsT, 1)
    fused_large_m_pair_kernel(const __grid_constant__ LargeMParams p) {
  using C = PairCfg<kMx>;
  static_assert(!kMx || (kFp8 && !kDown), "block scales go with E4M3 gate/up inputs");
  constexpr int kAccBufs = kMx ? 1 : 2;  // accumulator buffers in tensor memory
  // K values per stage: 64 bf16 or 128 E4M3, a 128-byte row either way
  constexpr int kBK = kFp8 ? kBlockK8 : kBlockK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem);
  const uint32_t sB = sA + C::kStages * C::kABytes;
  const uint32_t sStg = sB + C::kStages * C::kBBytes;
  const uint32_t sSf = sStg + C::kNumStg * C::kStgBytes;  // scales (kMx): kStages x 1.5 KB
  uint8_t* bar_ptr = smem + size_t(C::kStages) * C::kStageBytes + C::kNumStg * C::kStgBytes +
                     (kMx ? size_t(C::kStages) * kSfStageBytes : 0);
  const uint32_t bar0 = smem_addr(bar_ptr);
  // barrier slots: full[S] | empty[S] | tmem_full[2] | tmem_empty[2] | drain |
  // scales_ready[S] | scale-copy drain
  const uint32_t full0 = bar0, empty0 = bar0 + 8u * C::kStages;
  const uint32_t tfull0 = bar0 + 16u * C::kStages, tempty0 = tfull0 + 16u;
  const uint32_t drain_bar = tempty0 + 16u;
  const uint32_t sready0 = drain_bar + 8u, sdrain_bar = sready0 + 8u * C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (3 * C::kStages + 6));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int pairs = static_cast<int>(cluster_count_x());
  const int num_tiles = p.tiles_m * p.tiles_n;
  const int num_kb = (p.K + kBK - 1) / kBK;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  // rank 0's full and tmem_empty barriers, as seen from either CTA of the pair
  const uint32_t full0_lead = mapa_shared(full0, 0);
  const uint32_t tempty0_lead = mapa_shared(tempty0, 0);

  if (threadIdx.x == 0) {
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_w);
    prefetch_tmap(&p.tmap_y);
    if constexpr (kMx) {
      prefetch_tmap(&p.tmap_sw);
      prefetch_tmap(&p.tmap_sa);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8u * s, 1);   // rank 0's producer arrives (with both CTAs' bytes)
      mbar_init(empty0 + 8u * s, 1);  // rank 0's MMA commit, multicast to both CTAs
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8u * b, 1);   // multicast MMA commit
      mbar_init(tempty0 + 8u * b, 2 * C::kEpiWarps);  // epilogue warps x 2 CTAs (used on rank 0)
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < C::kStages; ++s) mbar_init(sready0 + 8u * s, 1);  // scale-copy commit
    mbar_init(sdrain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t filled = 0, fill_ph = 0;
      bool skip_once = p.inject_stall != 0;
      bool ok = true;
      // round pacing on the even CTA (the odd one follows through the empty
      // barriers); the launch number is drawn after the grid-dependency wait,
      // when the previous launch in the stream has finished. The launch's
      // draws add up to kPaceBlock, so the next launch starts a fresh block.
      const bool can_pace = pairs <= static_cast<int>(kPaceBlock);
      unsigned long long epoch = 0;
      if (leader && can_pace) {
        const unsigned long long take = pair == 0 ? kPaceBlock - static_cast<unsigned long long>(pairs - 1) : 1ull;
        epoch = ((atomicAdd(&g_pace_ticket, take) / kPaceBlock) + 1ull) & 0xffffffffull;
      }
      // only long bf16 gate/up tiles (K >= 8192, the 72B shape): with shorter
      // tiles the slowest pair of each round sets everyone's pace (7B prefill
      // +30 %, FP8 72B +13 %, block-scaled 7B +73 % when paced)
      const bool long_tiles = !kFp8 && !kDown && num_kb >= kPaceMinSlices;  // same in both CTAs
      const bool paced = leader && can_pace && long_tiles;
      bool pacing = paced;  // off for the rest of the launch once a wait runs out
      int round = 0;
      for (int t = pair; ok && t < num_tiles; t += pairs, ++round) {
        if (pacing && round >= kPaceLag && round - kPaceLag < kPaceRounds) {
          const int r = round - kPaceLag;
          pacing = pace_wait(r, epoch, static_cast<unsigned>(min(pairs, num_tiles - r * pairs)));
        }
        int mb, nb;
        pair_tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
        const int m0 = mb * 2 * kTileM + static_cast<int>(rank) * kTileM;
        const int wtile = nb * num_kb;                        // (column block nb, K slice 0)
        const int wrow = static_cast<int>(rank) * kPackBlockN;  // gate rows (0) / up rows (1)
        // paced shapes: odd rounds walk K backwards and start on the A slices
        // the previous round (same row tiles) read last, while L2 holds them
        const bool backwards = long_tiles && (round & 1) != 0;
        for (int i = 0; i < num_kb; ++i) {
          const int kb = backwards ? num_kb - 1 - i : i;
          if (!mbar_wait(empty0 + 8u * s, ph ^ 1u, wc, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          if (skip_once) {
            skip_once = false;  // testing hook: both CTAs leave this stage unfilled
          } else {
            if (leader)
              mbar_arrive_expect_tx(full0 + 8u * s, 2 * (C::kStageBytes + (kMx ? kSfStageBytes : 0)));
            const uint32_t fb = full0_lead + 8u * s;
            tma_load_2d_pair(sA + s * C::kABytes, &p.tmap_a, fb, kb * kBK, m0);
            tma_load_3d_pair(sB + s * C::kBBytes, &p.tmap_w, fb, 0, wrow, wtile + kb);
            if constexpr (kMx) {
              // this CTA's A rows: block (m0 / 128, kb), 2 rows of 256 bytes; both
              // weight-scale blocks of the tile (gate, up), 4 rows
              const uint32_t sf = sSf + s * kSfStageBytes;
              tma_load_2d_pair(sf, &p.tmap_sa, fb, 0, 2 * ((m0 / kTileM) * num_kb + kb));
              tma_load_2d_pair(sf + kSfBlockBytes, &p.tmap_sw, fb, 0, 4 * (wtile + kb));
            }
            filled |= 1u << s;
            fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
          }
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (paced && ok && round < kPaceRounds) pace_count(round, epoch);
      }
      pdl_launch_dependents();
      // Rank 0's full barriers count both CTAs' bytes: once they complete, every
      // copy issued by the pair for those stages has landed.
      if (leader)
        for (int i = 0; i < C::kStages; ++i)
          if (filled & (1u << i)) mbar_wait_drain(full0 + 8u * i, (fill_ph >> i) & 1u, wc);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (rank 0)
    if (leader && lane == 0) {
      constexpr uint32_t kIdesc = kFp8 ? idesc_e4m3_f32(2 * kTileM, 2 * C::kBN)
                                       : idesc_bf16_f32(2 * kTileM, 2 * C::kBN);
      constexpr uint32_t kIdescMx = idesc_mx_e4m3(2 * kTileM, 2 * C::kBN, 0);
      int s = 0;
      uint32_t ph = 0;
      int buf = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int t = pair; ok && t < num_tiles; t += pairs) {
        if (!mbar_wait(tempty0 + 8u * buf, acc_ph ^ 1u, wc, kSiteMmaTmemEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * C::kAccCols;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full0 + 8u * s, ph, wc, kSiteMmaFull)) {
            ok = false;
            break;
          }
          // block-scaled: the scale-copy warp has put this stage's scales in
          // its tensor-memory slot
          if (kMx && !mbar_wait(sready0 + 8u * s, ph, wc, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(sA + s * C::kABytes);
          const uint64_t bdesc = smem_desc_sw128(sB + s * C::kBBytes);
          // scale slot of this stage: A rows [0, 4), B columns 0..127 [4, 8), 128..255 [8, 12)
          const uint32_t tsf = tmem_base + C::kSfCol + uint32_t(s) * kSfTmemCols;
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // four 32-byte K steps per 128-byte row
            if constexpr (kMx)  // K step k consumes scale group k of the slice (IDs at bits 4, 29)
              mma_mx_pair(d, adesc + 2u * k, bdesc + 2u * k,
                          kIdescMx | (uint32_t(k) << 4) | (uint32_t(k) << 29), tsf, tsf + 4,
                          (kb | k) != 0 ? 1u : 0u);
            else if constexpr (kFp8)
              mma_e4m3_pair(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, (kb | k) != 0 ? 1u : 0u);
            else
              mma_bf16_pair(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit_pair_multicast(empty0 + 8u * s, 0x3);  // frees the stage in both CTAs
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_multicast(tfull0 + 8u * buf, 0x3);  // both halves of the accumulator ready
        if (++buf == kAccBufs) {
          buf = 0;
          acc_ph ^= 1u;
        }
      }
      mma_commit_pair_multicast(drain_bar, 0x1);
      mbar_wait_drain(drain_bar, 0, wc);
    }
    __syncwarp();
  } else if (kMx && warp == 2 + C::kEpiWarps) {
    // ------------------------------------------------ scale copies (rank 0)
    // Each stage's scales go from shared to tensor memory (both CTAs, each
    // from its own shared memory) as soon as the stage has landed, in a
    // stream of tcgen05 operations of their own, and the MMA issuer waits
    // for their completion. A slot is refilled only after its stage was
    // refilled, i.e. after the MMAs that read its previous contents completed.
    if (leader && lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = pair; ok && t < num_tiles; t += pairs) {
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full0 + 8u * s, ph, wc, kSiteScaleCopy)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tsf = tmem_base + C::kSfCol + uint32_t(s) * kSfTmemCols;
          const uint32_t sf = sSf + s * kSfStageBytes;
          tmem_cp_sf_pair(tsf, smem_desc_sf(sf));
          tmem_cp_sf_pair(tsf + 4, smem_desc_sf(sf + kSfBlockBytes));
          tmem_cp_sf_pair(tsf + 8, smem_desc_sf(sf + 2 * kSfBlockBytes));
          mma_commit_pair_multicast(sready0 + 8u * s, 0x1);
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      mma_commit_pair_multicast(sdrain_bar, 0x1);
      mbar_wait_drain(sdrain_bar, 0, wc);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int ew = warp - 2;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const float sg = kFp8 ? p.scale_gate : 1.0f, su = kFp8 ? p.scale_up : 1.0f;
    int buf = 0;
    uint32_t acc_ph = 0;
    int sbuf = 0;
    for (int t = pair; t < num_tiles; t += pairs) {
      int mb, nb;
      pair_tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
      const int row0 = mb * 2 * kTileM + static_cast<int>(rank) * kTileM + q * 32;
      const int col0 = nb * (kDown ? 2 * C::kBN : C::kBN);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(tfull0 + 8u * buf, acc_ph, wc, kSiteEpiTmemFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + buf * C::kAccCols;
      if constexpr (kMx) {
        // this warp's 64 output columns [64 h, 64 h + 64): gate and up, all loaded
        // before the accumulator is released to the next tile's MMAs
        const int h = ew >> 2;
        uint32_t g0[32], g1[32], u0[32], u1[32];
        tmem_ld_x32(tacc + 64 * h, g0);
        tmem_ld_x32(tacc + 64 * h + 32, g1);
        tmem_ld_x32(tacc + C::kBN + 64 * h, u0);
        tmem_ld_x32(tacc + C::kBN + 64 * h + 32, u1);
        tmem_wait_ld();
        reg_fence(g0);
        reg_fence(g1);
        reg_fence(u0);
        reg_fence(u1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0_lead + 8u * buf);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t* g = c ? g1 : g0;
          const uint32_t* u = c ? u1 : u0;
          if (lane == 0) bulk_wait_read<0>();  // this warp's one staging buffer is free again
          __syncwarp();
          const uint32_t stg = sStg + ew * C::kStgBytes;
          const uint32_t row_addr = stg + lane * 64;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i0 = 8 * j + 2 * e;
              w[e] = pack_bf16x2(silu_mul(__uint_as_float(g[i0]), __uint_as_float(u[i0])),
                                 silu_mul(__uint_as_float(g[i0 + 1]), __uint_as_float(u[i0 + 1])));
            }
            st_shared_v4(row_addr + ((j ^ ((lane >> 1) & 3)) << 4), w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int ncol = col0 + 64 * h + 32 * c;
            if (ncol < p.N && row0 < p.M) tma_store_2d(&p.tmap_y, stg, ncol, row0);
            bulk_commit();
          }
        }
      } else if constexpr (kDown) {
        // 256 output columns: accumulator + residual, 32 columns per store
        const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(p.residual);
        const int row = row0 + lane;
#pragma unroll 1
        for (int c = 0; c < C::kAccCols / 32; ++c) {
          uint32_t a[32];
          tmem_ld_x32(tacc + c * 32, a);
          tmem_wait_ld();
          reg_fence(a);
          if (c == C::kAccCols / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0_lead + 8u * buf);
          }
          const int ncol = col0 + c * 32;
          float add[32];
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {  // 8 columns (16 bytes) at a time; N % 8 == 0
            const int col = ncol + gq * 8;
            uint4 rv = make_uint4(0u, 0u, 0u, 0u);
            if (res && row < p.M && col < p.N)
              rv = *reinterpret_cast<const uint4*>(res + static_cast<size_t>(row) * p.N + col);
            const uint32_t w4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w4[e]);
              add[gq * 8 + 2 * e] = __low2float(h);
              add[gq * 8 + 2 * e + 1] = __high2float(h);
            }
          }
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          const uint32_t stg = sStg + (ew * 2 + sbuf) * C::kStgBytes;
          const uint32_t row_addr = stg + lane * 64;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i0 = 8 * j + 2 * e;
              w[e] = pack_bf16x2(__uint_as_float(a[i0]) + add[i0],
                                 __uint_as_float(a[i0 + 1]) + add[i0 + 1]);
            }
            st_shared_v4(row_addr + ((j ^ ((lane >> 1) & 3)) << 4), w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (ncol < p.N && row0 < p.M) tma_store_2d(&p.tmap_y, stg, ncol, row0);
            bulk_commit();
          }
          sbuf ^= 1;
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < C::kBN / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_x32(tacc + c * 32, g);
          tmem_ld_x32(tacc + C::kBN + c * 32, u);
          tmem_wait_ld();
          reg_fence(g);
          reg_fence(u);
          if (c == C::kBN / 32 - 1) {  // this CTA's half of the accumulator is read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0_lead + 8u * buf);
          }
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          const uint32_t stg = sStg + (ew * 2 + sbuf) * C::kStgBytes;
          const uint32_t row_addr = stg + lane * 64;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i0 = 8 * j + 2 * e;
              w[e] = pack_bf16x2(
                  silu_mul(sg * __uint_as_float(g[i0]), su * __uint_as_float(u[i0])),
                  silu_mul(sg * __uint_as_float(g[i0 + 1]), su * __uint_as_float(u[i0 + 1])));
            }
            st_shared_v4(row_addr + ((j ^ ((lane >> 1) & 3)) << 4), w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int ncol = col0 + c * 32;
            if (ncol < p.N && row0 < p.M) tma_store_2d(&p.tmap_y, stg, ncol, row0);
            bulk_commit();
          }
          sbuf ^= 1;
        }
      }
      if (++buf == kAccBufs) {
        buf = 0;
        acc_ph ^= 1u;
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  // Neither CTA leaves while the pair's MMAs may still read its shared memory
  // or the peer may still arrive on its barriers.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr,
                               bool with_pdl, bool mx = false) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(mx ? PairCfg<true>::kThreadsT : PairCfg<false>::kThreadsT);
  cfg.dynamicSmemBytes = mx ? PairCfg<true>::kSmem : PairCfg<false>::kSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = with_pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

}  // namespace

cudaError_t configure_large_m_pair(int* max_pairs) {
  cudaError_t e = cudaFuncSetAttribute(fused_large_m_pair_kernel<false, false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(PairCfg<false>::kSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_large_m_pair_kernel<true, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(PairCfg<false>::kSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_large_m_pair_kernel<false, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(PairCfg<false>::kSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_large_m_pair_kernel<true, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(PairCfg<true>::kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(2, nullptr, attr, false);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, fused_large_m_pair_kernel<false, false, false>, &cfg);
  if (e != cudaSuccess) return e;
  *max_pairs = clusters;
  return cudaSuccess;
}

size_t large_m_pair_smem_bytes() { return PairCfg<false>::kSmem; }
int large_m_pair_stages(bool mx) { return mx ? PairCfg<true>::kStages : PairCfg<false>::kStages; }

cudaError_t large_m_pair_pace_run_out(unsigned long long* count) {
  return cudaMemcpyFromSymbol(count, g_pace_run_out, sizeof(*count));
}

cudaError_t launch_large_m_pair(const LargeMParams& p, cudaStream_t stream) {
  if (p.grid < 2 || (p.grid % 2) != 0 || p.bn != PairCfg<false>::kBN) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(p.grid, stream, attr, pdl_enabled(), p.mx != 0);
  if (p.fp8 && p.down) return cudaErrorInvalidValue;  // no FP8 down-projection
  if (p.mx && !p.fp8) return cudaErrorInvalidValue;   // block scales go with E4M3 values
  const cudaError_t e =
      p.down  ? cudaLaunchKernelEx(&cfg, fused_large_m_pair_kernel<false, true, false>, p)
      : p.mx  ? cudaLaunchKernelEx(&cfg, fused_large_m_pair_kernel<true, false, true>, p)
      : p.fp8 ? cudaLaunchKernelEx(&cfg, fused_large_m_pair_kernel<true, false, false>, p)
              : cudaLaunchKernelEx(&cfg, fused_large_m_pair_kernel<false, false, false>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace swg
