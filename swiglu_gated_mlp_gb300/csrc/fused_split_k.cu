// Small-problem fused SwiGLU kernel: Y = SiLU(A W1) * (A W2) with K split over
// the two CTAs of a cluster, one output tile per cluster.
//
// Same method as the other kernels (one packed weight stream, gate and up
// columns side by side in one fp32 TMEM accumulator, SiLU * mul in the
// epilogue; "Tile-Level Activation Overlap for Efficient LLM Inference",
// gist.science, section "Methodology"), shaped for problems that are a single
// wave of small tiles, such as the Qwen-2.5-0.5B MLP at 128 tokens (18.9 MB
// of operands): there every 128 x 32 tile of the single-CTA kernel needs all
// of A plus its weight slice (344 KB), more than one SM's shared memory, so
// its loads come in two DRAM round trips. Here:
//
//  * a cluster of two CTAs owns one 128-token x 64-column output tile; CTA r
//    streams K slices [r * S / 2, (r + 1) * S / 2) of A and of the tile's 64
//    gate + 64 up packed weight rows (32 KB per 64-deep slice) through a
//    7-stage ring, so a K half of up to 448 values is loaded in one round trip;
//  * one MMA of M = 128, N = 128 per 16-deep K step accumulates that CTA's
//    partial Gate | Up in tensor memory (128 columns);
//  * the epilogue sums the two halves through distributed shared memory:
//    CTA r finishes tokens [64 r, 64 r + 64). After a cluster barrier (both
//    rings idle), the two epilogue warps holding the peer's token rows store
//    their fp32 partials into the peer's ring; after a second barrier the two
//    owning warps add them to their own, apply SiLU(g) * u in fp32 and store
//    bf16 rows of Y directly (64 columns = 128 bytes per token row);
//  * every pipeline wait is bounded (ptx.cuh); every thread of both CTAs
//    reaches both cluster barriers whatever the waits returned, so a CTA
//    whose wait ran out never leaves its peer waiting.
//
// Measured on GB300 it is slower than the single-CTA kernel on the 0.5B shape
// (8.0 against 7.35 us before that kernel's two-slice exchanges): the round
// trip it saves is not what that shape waits on. It is a selectable variant
// (SWIGLU_VARIANT_SPLIT_K), not an automatic choice.
#include "kernels.h"
#include "ptx.cuh"

namespace swg {
namespace {

struct SplitCfg {
  static constexpr int kBN = 64;                         // output columns per tile
  static constexpr int kABytes = kTileM * kBlockK * 2;   // 16 KB: 128 token rows
  static constexpr int kBBytes = 2 * kBN * kBlockK * 2;  // 16 KB: 64 gate + 64 up rows
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 7;
  static constexpr int kAccCols = 2 * kBN;               // gate | up, fp32
  static constexpr int kTmemCols = 128;
  static constexpr int kBarBytes = 256;
  static constexpr size_t kSmem = 1024 + size_t(kStages) * kStageBytes + kBarBytes;
  static_assert(kSmem <= 232448, "shared memory budget");
  // exchange buffer (in stage 0 once both rings are idle): 2 warps x 32
  // float4 columns x 32 lanes x 16 bytes
  static_assert(2 * 32 * 32 * 16 <= kStages * kStageBytes, "exchange buffer");
};

// 16-byte store into the shared memory of any CTA of the cluster.
__device__ __forceinline__ void st_shared_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    fused_split_k_kernel(const __grid_constant__ LargeMParams p) {
  using C = SplitCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem);
  const uint32_t sB = sA + C::kStages * C::kABytes;
  uint8_t* bar_ptr = smem + size_t(C::kStages) * C::kStageBytes;
  const uint32_t bar0 = smem_addr(bar_ptr);
  // barrier slots: full[S] | empty[S] | tmem_full | drain
  const uint32_t full0 = bar0, empty0 = bar0 + 8u * C::kStages;
  const uint32_t tfull_bar = bar0 + 16u * C::kStages, drain_bar = tfull_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * C::kStages + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int tile = static_cast<int>(cluster_id_x());
  const int mb = tile % p.tiles_m, nb = tile / p.tiles_m;
  const int num_kb = (p.K + kBlockK - 1) / kBlockK;
  const int kb_begin = static_cast<int>(rank) * num_kb / 2;
  const int kb_end = (static_cast<int>(rank) + 1) * num_kb / 2;
  const bool has_k = kb_end > kb_begin;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_w);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  pdl_wait();

  // epilogue registers: this lane's token row, gate columns [0, 64) then up [0, 64)
  float acc[C::kAccCols];
  int epi_ok = 0;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer -----
    if (lane == 0) {
      const int m0 = mb * kTileM;
      const int col0 = nb * C::kBN;
      const int wtile = (col0 / kPackBlockN) * num_kb;
      const int wrow = col0 % kPackBlockN;
      int s = 0;
      uint32_t ph = 0;
      uint32_t filled = 0, fill_ph = 0;
      bool skip_once = p.inject_stall != 0;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        if (!mbar_wait(empty0 + 8u * s, ph ^ 1u, wc, kSiteProducerEmpty)) break;
        if (skip_once) {
          skip_once = false;  // testing hook: leave this stage unfilled
        } else {
          const uint32_t fb = full0 + 8u * s;
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          tma_load_2d(sA + s * C::kABytes, &p.tmap_a, fb, kb * kBlockK, m0);
          tma_load_3d(sB + s * C::kBBytes, &p.tmap_w, fb, 0, wrow, wtile + kb);
          tma_load_3d(sB + s * C::kBBytes + C::kBN * kBlockK * 2, &p.tmap_w, fb, 0,
                      wrow + kPackBlockN, wtile + kb);
          filled |= 1u << s;
          fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
        }
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      pdl_launch_dependents();
      // copies in flight must land before the ring becomes the exchange buffer
      for (int i = 0; i < C::kStages; ++i)
        if (filled & (1u << i)) mbar_wait_drain(full0 + 8u * i, (fill_ph >> i) & 1u, wc);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer -------
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, C::kAccCols);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        if (!mbar_wait(full0 + 8u * s, ph, wc, kSiteMmaFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = smem_desc_sw128(sA + s * C::kABytes);
        const uint64_t bdesc = smem_desc_sw128(sB + s * C::kBBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem_base, adesc + 2u * k, bdesc + 2u * k, kIdesc,
                   (kb != kb_begin || k != 0) ? 1u : 0u);
        mma_commit(empty0 + 8u * s);
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok) mma_commit(tfull_bar);  // also arrives when no MMA was issued (no K slice)
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, wc);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue: own partial
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    if (lane == 0) epi_ok = mbar_wait(tfull_bar, 0, wc, kSiteEpiTmemFull) ? 1 : 0;
    epi_ok = __shfl_sync(0xffffffffu, epi_ok, 0);
    if (epi_ok && has_k) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C::kAccCols / 32; ++c) {
        uint32_t r[32];
        tmem_ld_x32(tmem_base + lane_off + c * 32, r);
        tmem_wait_ld();
        reg_fence(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[c * 32 + j] = __uint_as_float(r[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < C::kAccCols; ++j) acc[j] = 0.0f;  // no K slice: a zero partial
    }
  }

  // Both CTAs' MMAs and copies are done: both rings are free to exchange through.
  tc_fence_before();
  cluster_sync();

  // CTA r finishes tokens [64 r, 64 r + 64), held by its lane quarters 2r and 2r + 1.
  const int q = warp & 3;
  const bool epi = warp >= 2;
  const bool owner = epi && (q >> 1) == static_cast<int>(rank);
  const uint32_t xbase = smem_addr(smem) + static_cast<uint32_t>((q & 1) * 32 * 32 * 16);
  if (epi && !owner && epi_ok) {
    // the peer's token rows: store this CTA's partials into the peer's exchange buffer
    const uint32_t peer = mapa_shared(xbase, rank ^ 1u);
#pragma unroll
    for (int j = 0; j < C::kAccCols / 4; ++j)
      st_shared_cluster_v4(peer + static_cast<uint32_t>((j * 32 + lane) * 16),
                           make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
  }
  cluster_sync();  // the peer's partials are in this CTA's exchange buffer

  if (owner && epi_ok) {
    const float4* xb = reinterpret_cast<const float4*>(smem + (q & 1) * 32 * 32 * 16);
#pragma unroll
    for (int j = 0; j < C::kAccCols / 4; ++j) {
      const float4 v = xb[j * 32 + lane];
      acc[4 * j] += v.x;
      acc[4 * j + 1] += v.y;
      acc[4 * j + 2] += v.z;
      acc[4 * j + 3] += v.w;
    }
    const int row = mb * kTileM + q * 32 + lane;
    const int col0 = nb * C::kBN;
    if (row < p.M) {
      __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y) + static_cast<size_t>(row) * p.N;
#pragma unroll
      for (int c8 = 0; c8 < C::kBN / 8; ++c8) {  // 8 columns (16 bytes) at a time; N % 8 == 0
        const int col = col0 + c8 * 8;
        if (col < p.N) {
          uint4 o;
          o.x = pack_bf16x2(silu_mul(acc[c8 * 8 + 0], acc[C::kBN + c8 * 8 + 0]),
                            silu_mul(acc[c8 * 8 + 1], acc[C::kBN + c8 * 8 + 1]));
          o.y = pack_bf16x2(silu_mul(acc[c8 * 8 + 2], acc[C::kBN + c8 * 8 + 2]),
                            silu_mul(acc[c8 * 8 + 3], acc[C::kBN + c8 * 8 + 3]));
          o.z = pack_bf16x2(silu_mul(acc[c8 * 8 + 4], acc[C::kBN + c8 * 8 + 4]),
                            silu_mul(acc[c8 * 8 + 5], acc[C::kBN + c8 * 8 + 5]));
          o.w = pack_bf16x2(silu_mul(acc[c8 * 8 + 6], acc[C::kBN + c8 * 8 + 6]),
                            silu_mul(acc[c8 * 8 + 7], acc[C::kBN + c8 * 8 + 7]));
          *reinterpret_cast<uint4*>(y + col) = o;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace

cudaError_t configure_split_k(int* max_clusters) {
  cudaError_t e = cudaFuncSetAttribute(fused_split_k_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SplitCfg::kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SplitCfg::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_clusters, fused_split_k_kernel, &cfg);
}

int split_k_bn() { return SplitCfg::kBN; }
int split_k_stages() { return SplitCfg::kStages; }

cudaError_t launch_split_k(const LargeMParams& p, cudaStream_t stream) {
  if (p.bn != SplitCfg::kBN || p.grid != 2 * p.tiles_m * p.tiles_n || p.fp8 || p.down || p.mx)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SplitCfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_split_k_kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace swg
