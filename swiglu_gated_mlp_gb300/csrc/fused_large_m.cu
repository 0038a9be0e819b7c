// Large-M fused SwiGLU kernel: Y = SiLU(A W1) * (A W2) for 128-token tiles.
//
// The pages ("Tile-Level Activation Overlap for Efficient LLM Inference",
// gist.science, section "Methodology") fuse SwiGLU into the GEMM at tile level
// with two SM90 CUTLASS kernels: Kernel-1 overlaps the Swish of the Gate
// accumulator with the Up-tile loads, Kernel-2 runs one GEMM over a fused
// K x 2N weight and applies SiLU(gate) * up to column pairs in the epilogue,
// overlapping that arithmetic with the previous tile's TMA store. This kernel
// keeps the Kernel-2 idea (one packed weight stream, gate and up side by side
// in one accumulator, pairwise epilogue, store overlap) and re-does the rest
// for sm_103a:
//
//  * persistent CTAs (one per SM), warp-specialised: warp 0 issues TMA loads
//    into a STAGES-deep shared-memory ring, warp 1 (one thread) issues
//    tcgen05.mma, warps 2-5 run the epilogue;
//  * one MMA of M=128, N=2*BN, K=16 per step computes the gate columns and
//    the matching up columns of a 128 x BN output tile into tensor memory
//    (fp32), so Gate and Up never leave the SM;
//  * the two accumulators are double-buffered in TMEM: the epilogue of tile i
//    (tcgen05.ld -> SiLU * mul in fp32 registers -> bf16 -> swizzled shared
//    staging -> TMA store) overlaps the MMAs of tile i+1;
//  * every pipeline wait is bounded (see ptx.cuh); a stuck wait aborts the
//    CTA cleanly and is reported through the status word;
//  * before the grid-dependency wait an idle epilogue warp asks L2 to fetch
//    the first packed weight slices of the CTA's first tile and a share of
//    its A rows, so the first DRAM reads start under the previous grid's
//    tail: on long K loops (at least 4 ring-fulls) about 64 MB over the grid,
//    with 32-column tiles (small problems) the first 4 slices (more measured
//    slower there, as did staging right after the first ring-full);
//  * with 32-column tiles the producer and the MMA issuer hand over two K
//    slices per full/empty barrier exchange: small problems (the 0.5B shape,
//    14 slices in an 8-slot ring) wait on these hand-offs rather than on
//    bytes, and two per exchange took that shape from 7.39 to 6.94 us.
#include "kernels.h"
#include "ptx.cuh"

namespace swg {
namespace {

template <int BN>
struct LargeCfg {
  static constexpr int kABytes = kTileM * kBlockK * 2;   // 16 KB: 128 rows x 128 B
  static constexpr int kBBytes = 2 * BN * kBlockK * 2;   // BN gate rows + BN up rows
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (BN == 128) ? 4 : ((BN == 64) ? 6 : 8);
  // Ring slots handed over per full/empty barrier exchange: with 32-column
  // tiles (small problems, whose time goes to per-stage hand-offs rather than
  // to bytes) two 64-deep K slices at a time; deeper slices would leave the
  // shallower rings of the wider tiles too few exchanges in flight.
  static constexpr int kSlots = (BN == 32) ? 2 : 1;
  static_assert(kStages % kSlots == 0, "ring slots per exchange");
  static constexpr int kAccCols = 2 * BN;                // fp32 TMEM columns per accumulator
  static constexpr int kTmemCols = 2 * kAccCols;         // double buffered (128, 256 or 512)
  static constexpr int kStoreCols = 32;                  // output columns per TMA store
  static constexpr int kStgBytes = 32 * kStoreCols * 2;  // 32 rows x 64 B
  static constexpr int kNumStg = 8;                      // 4 epilogue warps x 2 buffers
  static constexpr int kBarBytes = 256;
  static constexpr size_t kSmem =
      1024 + size_t(kStages) * kStageBytes + size_t(kNumStg) * kStgBytes + kBarBytes;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kTmemCols <= 512, "tensor memory budget");
};

// Persistent tile order: groups of `group_m` row-tiles sweep all column tiles,
// so the CTAs running at the same time share both A rows and weight columns
// in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m, int& mb,
                                            int& nb) {
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int gm = min(tiles_m - first_m, group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    fused_large_m_kernel(const __grid_constant__ LargeMParams p) {
  using C = LargeCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem);
  const uint32_t sB = sA + C::kStages * C::kABytes;
  const uint32_t sStg = sB + C::kStages * C::kBBytes;
  uint8_t* bar_ptr = smem + size_t(C::kStages) * C::kStageBytes + C::kNumStg * C::kStgBytes;
  const uint32_t bar0 = smem_addr(bar_ptr);
  // barrier slots: full[S] | empty[S] | tmem_full[2] | tmem_empty[2] | drain
  const uint32_t full0 = bar0, empty0 = bar0 + 8u * C::kStages;
  const uint32_t tfull0 = bar0 + 16u * C::kStages, tempty0 = tfull0 + 16u;
  const uint32_t drain_bar = tempty0 + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * C::kStages + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.tiles_m * p.tiles_n;
  const int num_kb = (p.K + kBlockK - 1) / kBlockK;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_w);
    prefetch_tmap(&p.tmap_y);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8u * b, 1);
      mbar_init(tempty0 + 8u * b, 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // L2 staging of the first K slices before the grid-dependency wait: for long
  // K loops (at least 4 ring-fulls) p.l2_prefetch slices, and with 32-column
  // tiles (small problems) the first 4 (on the 0.5B shape 4 measured 2 %
  // faster than none; 8 and all 14 slower).
  const bool long_k = num_kb >= 4 * C::kStages;
  if (warp == 2 && lane == 0 && p.l2_prefetch > 0 && (long_k || BN == 32) &&
      static_cast<int>(blockIdx.x) < num_tiles) {
    // Inputs of the step, not products of the kernel before it in the stream;
    // L2 is coherent, so loads after the wait still see any write that kernel
    // made.
    int mb, nb;
    tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
    const int col0 = nb * BN;
    const int wtile = (col0 / kPackBlockN) * num_kb;
    const int wrow = col0 % kPackBlockN;
    const uint64_t pol = policy_evict_first();
    const int nw = min(long_k ? p.l2_prefetch : 4, num_kb);
    for (int kb = 0; kb < nw; ++kb) {
      tma_prefetch_l2_3d_hint(&p.tmap_w, 0, wrow, wtile + kb, pol);
      tma_prefetch_l2_3d_hint(&p.tmap_w, 0, wrow + kPackBlockN, wtile + kb, pol);
    }
    // A's rows are shared by the CTAs of a row tile: each takes every 8th slice
    for (int kb = static_cast<int>(blockIdx.x % 8u); kb < nw; kb += 8)
      tma_prefetch_l2_2d(&p.tmap_a, kb * kBlockK, mb * kTileM);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  pdl_wait();  // the set-up above overlaps the previous grid; memory traffic starts here

  if (warp == 0) {
    // ------------------------------------------------ TMA producer -----
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t filled = 0, fill_ph = 0;  // per stage: a fill was issued / parity of the last one
      bool skip_once = p.inject_stall != 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
        const int m0 = mb * kTileM;
        const int col0 = nb * BN;
        // packed tile index of (column block, K slice 0), and this tile's gate rows
        // inside the 256-row tile; the matching up rows follow 128 later
        const int wtile = (col0 / kPackBlockN) * num_kb;
        const int wrow = col0 % kPackBlockN;
        // kSlots consecutive slots (K slices) per exchange on slot s's barriers
        for (int kb = 0; kb < num_kb; kb += C::kSlots) {
          if (!mbar_wait(empty0 + 8u * s, ph ^ 1u, wc, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          if (skip_once) {
            skip_once = false;  // testing hook: leave this stage unfilled
          } else {
            const uint32_t fb = full0 + 8u * s;
            const int na = min(C::kSlots, num_kb - kb);
            mbar_arrive_expect_tx(fb, na * C::kStageBytes);
            for (int a = 0; a < na; ++a) {
              const int ss = s + a, k0 = (kb + a) * kBlockK;
              tma_load_2d(sA + ss * C::kABytes, &p.tmap_a, fb, k0, m0);
              tma_load_3d(sB + ss * C::kBBytes, &p.tmap_w, fb, 0, wrow, wtile + kb + a);
              tma_load_3d(sB + ss * C::kBBytes + BN * kBlockK * 2, &p.tmap_w, fb, 0,
                          wrow + kPackBlockN, wtile + kb + a);
            }
            filled |= 1u << s;
            fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
          }
          s += C::kSlots;
          if (s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      pdl_launch_dependents();
      // Copies still in flight must land before the CTA may exit.
      for (int i = 0; i < C::kStages; ++i)
        if (filled & (1u << i)) mbar_wait_drain(full0 + 8u * i, (fill_ph >> i) & 1u, wc);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer -------
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, 2 * BN);
      int s = 0;
      uint32_t ph = 0;
      int buf = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        if (!mbar_wait(tempty0 + 8u * buf, acc_ph ^ 1u, wc, kSiteMmaTmemEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * C::kAccCols;
        for (int kb = 0; kb < num_kb; kb += C::kSlots) {
          if (!mbar_wait(full0 + 8u * s, ph, wc, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int na = min(C::kSlots, num_kb - kb);
          for (int a = 0; a < na; ++a) {
            const uint64_t adesc = smem_desc_sw128(sA + (s + a) * C::kABytes);
            const uint64_t bdesc = smem_desc_sw128(sB + (s + a) * C::kBBytes);
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k)
              mma_bf16(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, ((kb + a) | k) != 0 ? 1u : 0u);
          }
          mma_commit(empty0 + 8u * s);  // frees the slots once these MMAs have read them
          s += C::kSlots;
          if (s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8u * buf);  // accumulator ready for the epilogue
        buf ^= 1;
        if (buf == 0) acc_ph ^= 1u;
      }
      // All MMAs issued by this thread must complete before TMEM is released.
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, wc);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue ---------
    const int q = warp & 3;  // the TMEM lane quarter this warp may read
    const int ew = warp - 2;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int buf = 0;
    uint32_t acc_ph = 0;
    int sbuf = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
      const int row0 = mb * kTileM + q * 32;
      const int col0 = nb * BN;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(tfull0 + 8u * buf, acc_ph, wc, kSiteEpiTmemFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + buf * C::kAccCols;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t g[32], u[32];
        tmem_ld_x32(tacc + c * 32, g);       // gate columns
        tmem_ld_x32(tacc + BN + c * 32, u);  // matching up columns
        tmem_wait_ld();
        reg_fence(g);
        reg_fence(u);
        if (c == BN / 32 - 1) {  // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty0 + 8u * buf);
        }
        if (lane == 0) bulk_wait_read<1>();  // this staging buffer's previous store has read it
        __syncwarp();
        const uint32_t stg = sStg + (ew * 2 + sbuf) * C::kStgBytes;
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
          const int ncol = col0 + c * 32;
          if (ncol < p.N && row0 < p.M) tma_store_2d(&p.tmap_y, stg, ncol, row0);
          bulk_commit();
        }
        sbuf ^= 1;
      }
      buf ^= 1;
      if (buf == 0) acc_ph ^= 1u;
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN>
cudaError_t configure_bn() {
  return cudaFuncSetAttribute(fused_large_m_kernel<BN>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(LargeCfg<BN>::kSmem));
}

template <int BN>
cudaError_t launch_bn(const LargeMParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LargeCfg<BN>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_large_m_kernel<BN>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int large_m_stages(int bn) {
  switch (bn) {
    case 128: return LargeCfg<128>::kStages;
    case 64: return LargeCfg<64>::kStages;
    case 32: return LargeCfg<32>::kStages;
    default: return 0;
  }
}

size_t large_m_smem_bytes(int bn) {
  switch (bn) {
    case 128: return LargeCfg<128>::kSmem;
    case 64: return LargeCfg<64>::kSmem;
    case 32: return LargeCfg<32>::kSmem;
    default: return 0;
  }
}

cudaError_t configure_large_m() {
  cudaError_t e = configure_bn<128>();
  if (e == cudaSuccess) e = configure_bn<64>();
  if (e == cudaSuccess) e = configure_bn<32>();
  return e;
}

cudaError_t launch_large_m(const LargeMParams& p, cudaStream_t stream) {
  switch (p.bn) {
    case 128: return launch_bn<128>(p, stream);
    case 64: return launch_bn<64>(p, stream);
    case 32: return launch_bn<32>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace swg
