// Sequential Gate -> Swish -> Up schedule (an ablation of the pages' Kernel-1
// on sm_103a): Y = SiLU(A W1) * (A W2) for 128 x 128 output tiles.
//
// The pages' Kernel-1 ("Tile-Level Activation Overlap for Efficient LLM
// Inference", gist.science, section "Methodology / Kernel-1") computes the
// Gate tile first, applies Swish to the register-resident Gate accumulator
// while the producer loads the Up weight tiles, then computes Up and lets the
// epilogue multiply and store. Here, per tile:
//
//  1. a first K loop runs MMAs (M=128, N=128) of A against the 128 gate rows of
//     the packed weight into TMEM columns [0, 128) of the tile's accumulator;
//  2. a second K loop runs A against the 128 up rows into columns [128, 256);
//     meanwhile the epilogue warps read the finished gate columns and compute
//     SiLU(gate) in registers (the overlap the pages exploit);
//  3. when the up loop completes, the epilogue multiplies, rounds to bf16 and
//     stores through swizzled staging + TMA, overlapping the next tile's loops
//     (double-buffered accumulator).
//
// Unlike the fused kernels, A is streamed twice per tile (once per K loop) and
// each MMA has N=128 instead of 256. It exists to measure that schedule on
// GB300 beside the single-pass kernels; every wait is bounded (ptx.cuh).
#include "kernels.h"
#include "ptx.cuh"

namespace swg {
namespace {

struct SeqCfg {
  static constexpr int kBN = 128;
  static constexpr int kABytes = kTileM * kBlockK * 2;   // 16 KB
  static constexpr int kBBytes = kBN * kBlockK * 2;      // 16 KB: gate rows or up rows
  static constexpr int kStageBytes = kABytes + kBBytes;  // 32 KB
  static constexpr int kStages = 6;
  static constexpr int kAccCols = 2 * kBN;               // gate | up
  static constexpr int kTmemCols = 2 * kAccCols;         // double buffered
  static constexpr int kStgBytes = 32 * 32 * 2;
  static constexpr int kNumStg = 8;
  static constexpr int kBarBytes = 256;
  static constexpr size_t kSmem =
      1024 + size_t(kStages) * kStageBytes + size_t(kNumStg) * kStgBytes + kBarBytes;
  static_assert(kSmem <= 232448, "shared memory budget");
};

__device__ __forceinline__ void seq_tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                                int& mb, int& nb) {
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int gm = min(tiles_m - first_m, group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

__global__ void __launch_bounds__(kThreads, 1)
    fused_sequential_kernel(const __grid_constant__ LargeMParams p) {
  using C = SeqCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem);
  const uint32_t sB = sA + C::kStages * C::kABytes;
  const uint32_t sStg = sB + C::kStages * C::kBBytes;
  uint8_t* bar_ptr = smem + size_t(C::kStages) * C::kStageBytes + C::kNumStg * C::kStgBytes;
  const uint32_t bar0 = smem_addr(bar_ptr);
  // barrier slots: full[S] | empty[S] | gate_full[2] | up_full[2] | tmem_empty[2] | drain
  const uint32_t full0 = bar0, empty0 = bar0 + 8u * C::kStages;
  const uint32_t gfull0 = bar0 + 16u * C::kStages, ufull0 = gfull0 + 16u;
  const uint32_t tempty0 = ufull0 + 16u, drain_bar = tempty0 + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * C::kStages + 7));
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
      mbar_init(gfull0 + 8u * b, 1);
      mbar_init(ufull0 + 8u * b, 1);
      mbar_init(tempty0 + 8u * b, 4);
    }
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

  if (warp == 0) {
    // ------------------------------------------------ TMA producer -----
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t filled = 0, fill_ph = 0;
      bool skip_once = p.inject_stall != 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        int mb, nb;
        seq_tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
        const int m0 = mb * kTileM;
        const int wtile = nb * num_kb;
        for (int pass = 0; ok && pass < 2; ++pass) {  // 0: gate rows, 1: up rows
          const int wrow = pass * kPackBlockN;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(empty0 + 8u * s, ph ^ 1u, wc, kSiteProducerEmpty)) {
              ok = false;
              break;
            }
            if (skip_once) {
              skip_once = false;  // testing hook: leave this stage unfilled
            } else {
              const uint32_t fb = full0 + 8u * s;
              mbar_arrive_expect_tx(fb, C::kStageBytes);
              tma_load_2d(sA + s * C::kABytes, &p.tmap_a, fb, kb * kBlockK, m0);
              tma_load_3d(sB + s * C::kBBytes, &p.tmap_w, fb, 0, wrow, wtile + kb);
              filled |= 1u << s;
              fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
            }
            if (++s == C::kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      }
      pdl_launch_dependents();
      for (int i = 0; i < C::kStages; ++i)
        if (filled & (1u << i)) mbar_wait_drain(full0 + 8u * i, (fill_ph >> i) & 1u, wc);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer -------
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, C::kBN);
      int s = 0;
      uint32_t ph = 0;
      int buf = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        if (!mbar_wait(tempty0 + 8u * buf, acc_ph ^ 1u, wc, kSiteMmaTmemEmpty)) break;
        tc_fence_after();
        for (int pass = 0; ok && pass < 2; ++pass) {
          const uint32_t d = tmem_base + buf * C::kAccCols + pass * C::kBN;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(full0 + 8u * s, ph, wc, kSiteMmaFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t adesc = smem_desc_sw128(sA + s * C::kABytes);
            const uint64_t bdesc = smem_desc_sw128(sB + s * C::kBBytes);
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k)
              mma_bf16(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, (kb | k) != 0 ? 1u : 0u);
            mma_commit(empty0 + 8u * s);
            if (++s == C::kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (ok) mma_commit((pass == 0 ? gfull0 : ufull0) + 8u * buf);
        }
        if (!ok) break;
        buf ^= 1;
        if (buf == 0) acc_ph ^= 1u;
      }
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, wc);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue ---------
    const int q = warp & 3;
    const int ew = warp - 2;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int buf = 0;
    uint32_t acc_ph = 0;
    int sbuf = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb;
      seq_tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
      const int row0 = mb * kTileM + q * 32;
      const int col0 = nb * C::kBN;
      const uint32_t tacc = tmem_base + lane_off + buf * C::kAccCols;
      // Swish on the finished gate accumulator while the up loop runs.
      int ok = 1;
      if (lane == 0) ok = mbar_wait(gfull0 + 8u * buf, acc_ph, wc, kSiteEpiTmemFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      float sg[C::kBN];
#pragma unroll
      for (int c = 0; c < C::kBN / 32; ++c) {
        uint32_t g[32];
        tmem_ld_x32(tacc + c * 32, g);
        tmem_wait_ld();
        reg_fence(g);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = __uint_as_float(g[j]);
          sg[c * 32 + j] = __fdividef(x, 1.0f + __expf(-x));
        }
      }
      if (lane == 0) ok = mbar_wait(ufull0 + 8u * buf, acc_ph, wc, kSiteEpiTmemFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C::kBN / 32; ++c) {
        uint32_t u[32];
        tmem_ld_x32(tacc + C::kBN + c * 32, u);
        tmem_wait_ld();
        reg_fence(u);
        if (c == C::kBN / 32 - 1) {  // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty0 + 8u * buf);
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
            w[e] = pack_bf16x2(sg[c * 32 + i0] * __uint_as_float(u[i0]),
                               sg[c * 32 + i0 + 1] * __uint_as_float(u[i0 + 1]));
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

}  // namespace

cudaError_t configure_sequential() {
  return cudaFuncSetAttribute(fused_sequential_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(SeqCfg::kSmem));
}

int sequential_stages() { return SeqCfg::kStages; }

cudaError_t launch_sequential(const LargeMParams& p, cudaStream_t stream) {
  if (p.bn != SeqCfg::kBN) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SeqCfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_sequential_kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace swg
