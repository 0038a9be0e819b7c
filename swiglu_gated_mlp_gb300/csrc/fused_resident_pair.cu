// Fused SwiGLU for problems whose whole K range fits in shared memory at once
// (K <= 896): Y = SiLU(A W1) * (A W2) on CTA pairs with every K slice loaded
// up front, so that the weights come in one DRAM round trip instead of
// streaming through a ring that is refilled as it is consumed ("Tile-Level
// Activation Overlap for Efficient LLM Inference", gist.science, section
// "Methodology": the gate and up contractions share one A tile and the SiLU *
// mul epilogue consumes them on chip).
//
// On small problems such as a 0.5B model's MLP (M = 128, K = 896, N = 4864) the
// other kernels spend most of a launch waiting: the weight stream is 17 MB,
// but a ring that holds half of each CTA's K range needs two round trips, each
// a DRAM latency plus the pipeline hand-offs of its stages. Here a cluster of
// two CTAs owns a 128-token x 64-column output tile and runs
// tcgen05.mma.cta_group::2 with M = 128: each CTA holds 64 token rows of A
// and, per K slice, 32 gate rows plus the 32 matching up rows of the packed
// weight, i.e. 16 KB per 64-deep slice and 224 KB for 14 slices. With M = 128
// over two CTAs, each CTA's tensor memory holds its 64 token rows twice over:
// lanes 0-63 receive the columns of the even CTA's weight rows and lanes
// 64-127 those of the odd CTA's (measured on GB300). With gate then up rows in
// each CTA's slice, every lane therefore holds the gate and the up value of
// the same 32 output columns side by side (tensor-memory columns 0-31 and
// 32-63), and the epilogue is the single-CTA one: one warp per lane quarter,
// SiLU(g) * u in fp32, bf16, a TMA store of 32 x 32 outputs.
//
// One tile per CTA pair (the grid holds every tile at once): the even CTA's
// "full" barriers count both CTAs' bytes (cta_group::2 loads), its MMA commit
// arrives on both CTAs' "accumulator full" barrier, and every wait is bounded.
//
// Measured on GB300 it is slower than the single-CTA kernel on the 0.5B shape
// (8.4 against 6.9 us): timing copies of that kernel showed the shape waiting
// on per-slice pipeline hand-offs and small MMAs rather than on the second
// round trip, and the M = 128 pair MMAs here follow the loads. It is a
// selectable variant (SWIGLU_VARIANT_RESIDENT_PAIR), not an automatic choice.
#include "kernels.h"
#include "ptx.cuh"

namespace swg {
namespace {

constexpr int kRowsA = 64;                          // token rows of A per CTA
constexpr int kColsTile = 64;                       // output columns per CTA pair
constexpr int kAtomA = kRowsA * kBlockK * 2;        // 8 KB per 64-deep K slice
constexpr int kAtomB = kColsTile * kBlockK * 2;     // 32 gate + 32 up rows: 8 KB
constexpr int kAtom = kAtomA + kAtomB;
constexpr int kMaxSlices = 14;                      // 224 KB: K <= 896
constexpr int kBarBytes = 256;
constexpr size_t kSmem = 1024 + size_t(kMaxSlices) * kAtom + kBarBytes;
static_assert(kSmem <= 232448, "shared memory budget");
constexpr int kTmemCols = 64;                       // N = 128 over two CTAs: 64 columns each
static_assert(8 * (kMaxSlices + 2) + 8 <= kBarBytes, "barrier slots");

__global__ void __launch_bounds__(kThreads, 1)
    fused_resident_pair_kernel(const __grid_constant__ LargeMParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_addr(smem);  // slice kb: A at s0 + kb * kAtom, weights 8 KB after
  uint8_t* bar_ptr = smem + size_t(kMaxSlices) * kAtom;
  const uint32_t bar0 = smem_addr(bar_ptr);
  // barrier slots: full[kMaxSlices] | tmem_full | drain
  const uint32_t full0 = bar0, tfull_bar = bar0 + 8u * kMaxSlices, drain_bar = tfull_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (kMaxSlices + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int tile = static_cast<int>(cluster_id_x());
  const int mb = tile % p.tiles_m, nb = tile / p.tiles_m;
  const int num_kb = (p.K + kBlockK - 1) / kBlockK;  // <= kMaxSlices (checked at launch)
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const uint32_t full0_lead = mapa_shared(full0, 0);

  if (threadIdx.x == 0) {
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_w);
    prefetch_tmap(&p.tmap_y);
    for (int s = 0; s < kMaxSlices; ++s) mbar_init(full0 + 8u * s, 1);  // even CTA's producer
    mbar_init(tfull_bar, 1);  // multicast MMA commit
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const int m0 = mb * kTileM + static_cast<int>(rank) * kRowsA;
      const int c0 = nb * kColsTile;
      const int wtile = (c0 / kPackBlockN) * num_kb;  // packed tile (column block, K slice 0)
      // this CTA's 32 gate rows in the packed tile, and the up rows 128 further
      const int grow = c0 % kPackBlockN + static_cast<int>(rank) * (kColsTile / 2);
      uint32_t filled = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (kb == 0 && p.inject_stall) continue;  // testing hook: both CTAs leave slice 0 unfilled
        const uint32_t fb = full0_lead + 8u * kb;
        const uint32_t sa = s0 + kb * kAtom, sb = sa + kAtomA;
        if (leader) mbar_arrive_expect_tx(full0 + 8u * kb, 2 * kAtom);
        tma_load_2d_pair(sa, &p.tmap_a, fb, kb * kBlockK, m0);
        tma_load_3d_pair(sb, &p.tmap_w, fb, 0, grow, wtile + kb);
        tma_load_3d_pair(sb + kAtomB / 2, &p.tmap_w, fb, 0, kPackBlockN + grow, wtile + kb);
        filled |= 1u << kb;
      }
      pdl_launch_dependents();
      // The even CTA's full barriers count both CTAs' bytes: once they
      // complete, every copy issued by the pair has landed.
      if (leader)
        for (int kb = 0; kb < num_kb; ++kb)
          if (filled & (1u << kb)) mbar_wait_drain(full0 + 8u * kb, 0, wc);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, 2 * kColsTile);
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(full0 + 8u * kb, 0, wc, kSiteMmaFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = s0 + kb * kAtom;
        const uint64_t adesc = smem_desc_sw128(sa);
        const uint64_t bdesc = smem_desc_sw128(sa + kAtomA);
#pragma unroll
        for (int k = 0; k < kBlockK / 16; ++k)
          mma_bf16_pair(tmem_base, adesc + 2u * k, bdesc + 2u * k, kIdesc, (kb | k) != 0 ? 1u : 0u);
      }
      if (ok) mma_commit_pair_multicast(tfull_bar, 0x3);  // the accumulator is ready in both CTAs
      mma_commit_pair_multicast(drain_bar, 0x1);
      mbar_wait_drain(drain_bar, 0, wc);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    // Warp w reads lane quarter q = w % 4: token rows 32 (q % 2) .. + 31 of
    // this CTA's 64, output columns 32 (q / 2) .. + 31 of the tile (gate in
    // tensor-memory columns 0-31, up in 32-63).
    const int q = warp & 3;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(tfull_bar, 0, wc, kSiteEpiTmemFull) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      uint32_t g[32], u[32];
      tmem_ld_x32(tacc, g);
      tmem_ld_x32(tacc + kColsTile / 2, u);
      tmem_wait_ld();
      reg_fence(g);
      reg_fence(u);
      // staging: slice 0's A region (its MMAs have completed), 2 KB per warp
      const uint32_t stg = s0 + q * (32 * 64);
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
        // 64-byte swizzle: 16-byte chunk j of row r lands at chunk j ^ ((r >> 1) & 3)
        st_shared_v4(row_addr + ((j ^ ((lane >> 1) & 3)) << 4), w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int row0 = mb * kTileM + static_cast<int>(rank) * kRowsA + 32 * (q & 1);
        const int col0 = nb * kColsTile + 32 * (q >> 1);
        if (col0 < p.N && row0 < p.M) tma_store_2d(&p.tmap_y, stg, col0, row0);
        bulk_commit();
        bulk_wait<0>();
      }
      __syncwarp();
    }
  }

  // Neither CTA leaves while the pair's MMAs may still read its shared memory
  // or the peer may still arrive on its barriers.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

int resident_pair_max_slices() { return kMaxSlices; }
int resident_pair_bn() { return kColsTile; }

cudaError_t configure_resident_pair() {
  return cudaFuncSetAttribute(fused_resident_pair_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmem));
}

cudaError_t launch_resident_pair(const LargeMParams& p, cudaStream_t stream) {
  const int num_kb = (p.K + kBlockK - 1) / kBlockK;
  if (num_kb < 1 || num_kb > kMaxSlices || p.bn != kColsTile || p.tiles_m < 1 || p.tiles_n < 1 ||
      p.grid != 2 * p.tiles_m * p.tiles_n || p.fp8 || p.down || p.mx)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_resident_pair_kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace swg
