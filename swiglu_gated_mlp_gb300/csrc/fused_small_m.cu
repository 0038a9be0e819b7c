// Small-M (decode) fused SwiGLU kernel: Y = SiLU(A W1) * (A W2) for M <= 256.
//
// With few tokens the op is bound by streaming the weights from HBM once. The
// pages give small batches to Kernel-2 because its doubled threadblock count
// fills the SMs ("Tile-Level Activation Overlap for Efficient LLM Inference",
// gist.science, section "Methodology / Kernel-2", Optimization). Here the
// operands are swapped instead: each CTA owns one 128-column block of the
// packed weight (per 64-deep K slice, 128 gate rows + 128 up rows stored as
// one contiguous 32 KB tile) and streams it through a deep TMA ring, one tile
// per stage; the weight rows are the MMA's M side (128) and the
// tokens its N side (mt = M rounded up to 16), so
//   Gate^T[128 x mt] = W1_block^T * A^T   and   Up^T likewise,
// two tcgen05.mma per K step into two fp32 TMEM accumulators. The epilogue
// thread for weight column n reads gate and up for all tokens, applies
// SiLU(g) * u in fp32 and writes Y[m][n] (a warp writes 32 consecutive
// columns of one row at a time).
//
// When there are few column blocks for the SMs (small N), each block's K range
// is split over a cluster of `splits` CTAs: every CTA accumulates its K part in
// TMEM, writes the fp32 partial Gate and Up to its own shared memory, and after
// a cluster barrier each CTA sums, through distributed shared memory, all
// parts of its share of the block's columns, applies SiLU(g) * u and writes
// those outputs. No global scratch is used. With a caller workspace the K
// range can also be split across `gsplits` such clusters (more CTAs than
// clusters of 8 can hold): each cluster writes its summed shares to the
// workspace and counts itself in, and the last cluster of the block to arrive
// (one counter per cluster rank) adds all clusters' partials in cluster order,
// so the result does not depend on arrival order, and finishes the outputs.
//
// The same kernel computes the gated MLP's down-projection Out = Y x W3 + R
// (kDown): a packed tile then holds 256 consecutive output columns, the two
// accumulators are columns [0, 128) and [128, 256) of the block, and the
// epilogue adds the residual instead of applying SiLU(g) * u.
//
// With kMx (block-scaled E4M3, one power-of-two scale per 32 K values) each
// stage also brings the tile's two 512-byte weight-scale blocks (gate, up)
// and the activations' scale block for the same K slice; the MMA thread copies
// them into a per-stage slot of tensor memory (tcgen05.cp) and issues
// kind::mxf8f6f4 MMAs that apply both scales inside the tensor core.
#include "kernels.h"
#include "ptx.cuh"

namespace swg {
namespace {

constexpr int kWStageBytes = 2 * kPackBlockN * kBlockK * 2;  // 32 KB: 256 packed rows x 128 B

// Scratch of the allocation-free entry point (swiglu_forward_noalloc): the
// status record the kernel writes when a pipeline wait gives up, placed in a
// file-scope device array instead of library-allocated memory. Every GPU that
// loads the library holds these 256 bytes until the process exits; all calls
// of that entry point on a device share them.
static __device__ __align__(256) uint32_t g_static_scratch[kStaticScratchWords];

constexpr int kMaxStages = 8;
constexpr int kMaxClusters = 8;  // K split across at most this many clusters per unit
constexpr size_t kSmemLimit = 232448;
constexpr int kBarBytes = 256;

// The outputs of token m (of the group starting at m0), weight rows r .. r + 3
// of column block nblk, from the summed fp32 g and u: SiLU(g) * u (with the
// FP8 scales), or the two down-projection columns plus the residual.
template <bool kFp8, bool kDown>
__device__ __forceinline__ void finish_outputs(const SmallMParams& p, int m0, int nblk, int m,
                                               int r, float4 g, float4 u) {
  __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y);
  if constexpr (kDown) {  // columns n0 + r .. + 3 (g) and n0 + 128 + r .. + 3 (u)
    const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(p.residual);
    const int n_lo = nblk * 2 * kPackBlockN + r, n_hi = n_lo + kPackBlockN;
    const size_t row = static_cast<size_t>(m0 + m) * p.N;
    const float4 parts[2] = {g, u};
    const int cols[2] = {n_lo, n_hi};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (cols[h] >= p.N) continue;  // N % 8 == 0: cols[h] < N implies cols[h] + 3 < N
      float4 v = parts[h];
      if (res) {
        const uint2 rr = *reinterpret_cast<const uint2*>(res + row + cols[h]);
        const __nv_bfloat162 r0 = *reinterpret_cast<const __nv_bfloat162*>(&rr.x);
        const __nv_bfloat162 r1 = *reinterpret_cast<const __nv_bfloat162*>(&rr.y);
        v.x += __low2float(r0); v.y += __high2float(r0);
        v.z += __low2float(r1); v.w += __high2float(r1);
      }
      uint2 o;
      o.x = pack_bf16x2(v.x, v.y);
      o.y = pack_bf16x2(v.z, v.w);
      *reinterpret_cast<uint2*>(y + row + cols[h]) = o;
    }
  } else {
    const int n = nblk * kPackBlockN + r;  // N % 8 == 0: n < N implies n + 3 < N
    if (kFp8) {
      g.x *= p.scale_gate; g.y *= p.scale_gate; g.z *= p.scale_gate; g.w *= p.scale_gate;
      u.x *= p.scale_up; u.y *= p.scale_up; u.z *= p.scale_up; u.w *= p.scale_up;
    }
    if (n < p.N) {
      uint2 v;
      v.x = pack_bf16x2(silu_mul(g.x, u.x), silu_mul(g.y, u.y));
      v.y = pack_bf16x2(silu_mul(g.z, u.z), silu_mul(g.w, u.w));
      *reinterpret_cast<uint2*>(y + static_cast<size_t>(m0 + m) * p.N + n) = v;
    }
  }
}

// K split across clusters, after this CTA stored its cluster's sums of weight
// rows [part * R, part * R + R) (R = 128 / splits) in the workspace: count the
// CTA in on the (unit, rank) counter and, in the last cluster to arrive, add
// all clusters' sums in cluster order and finish the outputs. Out of line: it
// runs only with a workspace, and keeps the kernel body small otherwise.
template <bool kFp8, bool kDown>
__device__ __noinline__ void cross_cluster_finish(const SmallMParams& p, int unit, int part,
                                                  int splits, int gsplits, int mt, int mcount,
                                                  int m0, int nblk, volatile int* last_flag) {
  const int rows = kPackBlockN / splits;
  const int chunks = rows / 4;
  const size_t ws_stride = size_t(2) * mt * kPackBlockN;
  // Every CTA of every cluster counts itself in exactly once, whatever its
  // waits returned, so the counter is back at zero when the kernel ends.
  __syncthreads();  // all of this CTA's partial stores are issued
  if (threadIdx.x == 0) {
    __threadfence();  // (cumulative) they are visible before this CTA is counted
    uint32_t* counter = p.counters + size_t(unit) * splits + part;
    const uint32_t before = atomicAdd(counter, 1u);
    const bool last = before == static_cast<uint32_t>(gsplits - 1);
    if (last) {
      atomicExch(counter, 0u);  // every cluster of the unit has arrived
      __threadfence();          // and their partials are visible to this CTA
    }
    *last_flag = last ? 1 : 0;
  }
  __syncthreads();
  if (!*last_flag) return;
  // kSumBatch outputs per thread at a time, the loads of all clusters issued
  // before the sums (in cluster order: independent of arrival order)
  constexpr int kSumBatch = 4;
  const int items = mcount * chunks;
  for (int i0 = threadIdx.x; i0 < items; i0 += kSumBatch * blockDim.x) {
    float4 g[kSumBatch], u[kSumBatch];
#pragma unroll
    for (int b = 0; b < kSumBatch; ++b) g[b] = u[b] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kMaxClusters; ++c) {
      if (c < gsplits) {
        const float* src = p.ws + (size_t(unit) * gsplits + c) * ws_stride;
        float4 gs[kSumBatch], us[kSumBatch];
#pragma unroll
        for (int b = 0; b < kSumBatch; ++b) {
          const int idx = min(i0 + b * static_cast<int>(blockDim.x), items - 1);
          const int m = idx / chunks;
          const int r = part * rows + (idx % chunks) * 4;
          gs[b] = __ldcg(reinterpret_cast<const float4*>(src + size_t(m) * kPackBlockN + r));
          us[b] = __ldcg(reinterpret_cast<const float4*>(src + size_t(mt + m) * kPackBlockN + r));
        }
#pragma unroll
        for (int b = 0; b < kSumBatch; ++b) {
          g[b].x += gs[b].x; g[b].y += gs[b].y; g[b].z += gs[b].z; g[b].w += gs[b].w;
          u[b].x += us[b].x; u[b].y += us[b].y; u[b].z += us[b].z; u[b].w += us[b].w;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kSumBatch; ++b) {
      const int idx = i0 + b * static_cast<int>(blockDim.x);
      if (idx < items)
        finish_outputs<kFp8, kDown>(p, m0, nblk, idx / chunks, part * rows + (idx % chunks) * 4,
                                    g[b], u[b]);
    }
  }
}

template <bool kFp8, bool kDown, bool kMx>
__global__ void __launch_bounds__(kThreads, 1)
    fused_small_m_kernel(const __grid_constant__ SmallMParams p) {
  static_assert(!kMx || (kFp8 && !kDown), "block scales go with E4M3 gate/up inputs");
  // K values per stage: 64 bf16 or 128 E4M3, a 128-byte row either way
  constexpr int kBK = kFp8 ? kBlockK8 : kBlockK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int mt = p.mt;
  const int stages = p.stages;
  const uint32_t x_bytes = static_cast<uint32_t>(mt) * 128;
  const uint32_t stage_bytes = kWStageBytes + x_bytes;  // multiple of 1024 (mt % 8 == 0)
  const uint32_t s0 = smem_addr(smem);
  // block-scaled FP8: per stage 1.5 KB of scales (gate, up, activations) after the ring
  const uint32_t sf0 = s0 + stages * stage_bytes;
  uint8_t* bar_ptr = smem + size_t(stages) * stage_bytes + (kMx ? size_t(stages) * kSfStageBytes : 0);
  const uint32_t bar0 = smem_addr(bar_ptr);
  // barrier slots: full[8] | empty[8] | tmem_full | drain
  const uint32_t full0 = bar0, empty0 = bar0 + 8u * kMaxStages;
  const uint32_t tfull_bar = bar0 + 16u * kMaxStages, drain_bar = tfull_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * kMaxStages + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // accumulators: gate [0, mt), up [mt, 2 mt); then kSfTmemCols scale columns per stage
  const uint32_t sf_col = 2u * mt;
  uint32_t tmem_cols = 32;
  while (tmem_cols < sf_col + (kMx ? uint32_t(kSfTmemCols) * stages : 0u)) tmem_cols <<= 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_kb = (p.K + kBK - 1) / kBK;
  const int splits = p.splits > 1 ? p.splits : 1;
  const int gsplits = p.gsplits > 1 ? p.gsplits : 1;
  // CTA index = ((unit * gsplits) + cluster) * splits + rank in the cluster,
  // unit = column block * token groups + token group
  const int mgroups = p.mgroups > 1 ? p.mgroups : 1;
  const int part = blockIdx.x % splits;  // the CTA's rank in its cluster when splits > 1
  const int gpart = (blockIdx.x / splits) % gsplits;
  const int unit = blockIdx.x / (splits * gsplits);
  const int tgroup = unit % mgroups;
  const int nblk = unit / mgroups;
  const int m0 = tgroup * mt;                 // first token of this CTA's group
  const int mcount = min(mt, p.M - m0);       // tokens in the group
  const int kparts = splits * gsplits;        // K parts of the unit, in order
  const int kpart = gpart * splits + part;
  const int kb_begin = kpart * num_kb / kparts;
  const int kb_end = (kpart + 1) * num_kb / kparts;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    prefetch_tmap(&p.tmap_x);
    prefetch_tmap(&p.tmap_w);
    if constexpr (kMx) {
      prefetch_tmap(&p.tmap_sw);
      prefetch_tmap(&p.tmap_sa);
    }
    // The packed weight is an input of the decode step, not a product of the
    // kernel before it in the stream; fetching this CTA's first tiles into L2
    // before the grid-dependency wait overlaps their DRAM latency with the
    // previous grid's tail. L2 is coherent, so this is safe even when that
    // kernel did write the weight: the loads after the wait see its writes.
    const int npre = min(p.l2_prefetch, kb_end - kb_begin);
    const uint64_t pol = policy_evict_first();
    for (int i = 0; i < npre; ++i)
      tma_prefetch_l2_3d_hint(&p.tmap_w, 0, 0, nblk * num_kb + kb_begin + i, pol);
    for (int s = 0; s < stages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  pdl_wait();  // the set-up and L2 staging above overlap the previous grid; loads start here

  if (warp == 0) {
    // ------------------------------------------------ TMA producer -----
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();  // weights: read once
      const uint64_t pol_x = policy_evict_last();   // activations: re-read by every CTA
      const int wtile = nblk * num_kb;  // packed tile index of (this column block, K slice 0)
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
          const uint32_t sw = s0 + s * stage_bytes;
          const int k0 = kb * kBK;
          mbar_arrive_expect_tx(fb, stage_bytes + (kMx ? kSfStageBytes : 0));
          tma_load_3d_hint(sw, &p.tmap_w, fb, 0, 0, wtile + kb, pol_w);  // one contiguous 32 KB tile
          tma_load_2d_hint(sw + kWStageBytes, &p.tmap_x, fb, k0, m0, pol_x);
          if constexpr (kMx) {
            // 4 rows of 256 bytes: the tile's gate and up scale blocks; 2 rows: the
            // activations' block (128-row chunk m0 / 128, K slice kb)
            const uint32_t sf = sf0 + s * kSfStageBytes;
            tma_load_2d(sf, &p.tmap_sw, fb, 0, 4 * (wtile + kb));
            tma_load_2d(sf + 2 * kSfBlockBytes, &p.tmap_sa, fb, 0, 2 * ((m0 / 128) * num_kb + kb));
          }
          filled |= 1u << s;
          fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
        }
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      pdl_launch_dependents();
      for (int i = 0; i < stages; ++i)
        if (filled & (1u << i)) mbar_wait_drain(full0 + 8u * i, (fill_ph >> i) & 1u, wc);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer -------
    if (lane == 0) {
      const uint32_t idesc = kFp8 ? idesc_e4m3_f32(128, mt) : idesc_bf16_f32(128, mt);
      const uint32_t d_gate = tmem_base;
      const uint32_t d_up = tmem_base + static_cast<uint32_t>(mt);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        if (!mbar_wait(full0 + 8u * s, ph, wc, kSiteMmaFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sw = s0 + s * stage_bytes;
        const uint64_t gdesc = smem_desc_sw128(sw);                         // gate rows 0..127
        const uint64_t udesc = smem_desc_sw128(sw + kWStageBytes / 2);      // up rows 128..255
        const uint64_t xdesc = smem_desc_sw128(sw + kWStageBytes);          // tokens
        // scale slot of this stage: gate [0, 4), up [4, 8), tokens [8, 12)
        const uint32_t tsf = tmem_base + sf_col + uint32_t(s) * kSfTmemCols;
        if constexpr (kMx) {
          const uint32_t sf = sf0 + s * kSfStageBytes;
          tmem_cp_sf(tsf, smem_desc_sf(sf));
          tmem_cp_sf(tsf + 4, smem_desc_sf(sf + kSfBlockBytes));
          tmem_cp_sf(tsf + 8, smem_desc_sf(sf + 2 * kSfBlockBytes));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // four 32-byte K steps per 128-byte row
          const uint32_t acc = (kb != kb_begin || k != 0) ? 1u : 0u;
          if constexpr (kMx) {  // K step k consumes scale group k of the slice
            const uint32_t id = idesc_mx_e4m3(128, mt, k);
            mma_mx(d_gate, gdesc + 2u * k, xdesc + 2u * k, id, tsf, tsf + 8, acc);
            mma_mx(d_up, udesc + 2u * k, xdesc + 2u * k, id, tsf + 4, tsf + 8, acc);
          } else if constexpr (kFp8) {
            mma_e4m3(d_gate, gdesc + 2u * k, xdesc + 2u * k, idesc, acc);
            mma_e4m3(d_up, udesc + 2u * k, xdesc + 2u * k, idesc, acc);
          } else {
            mma_bf16(d_gate, gdesc + 2u * k, xdesc + 2u * k, idesc, acc);
            mma_bf16(d_up, udesc + 2u * k, xdesc + 2u * k, idesc, acc);
          }
        }
        mma_commit(empty0 + 8u * s);
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok) mma_commit(tfull_bar);
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, wc);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue ---------
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int n = nblk * kPackBlockN + q * 32 + lane;  // this thread's output column
    int ok = 1;
    if (lane == 0) ok = mbar_wait(tfull_bar, 0, wc, kSiteEpiTmemFull) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok && kparts > 1) {
      // K part only: fp32 partials to this CTA's shared memory (the ring is idle
      // now), as P[c][r] for accumulator column c (gate 0..mt-1, up mt..2mt-1)
      // and weight row r of the block.
      tc_fence_after();
      float* part_buf = reinterpret_cast<float*>(smem);
      const int r = q * 32 + lane;
#pragma unroll 1
      for (int mc = 0; mc < mt / 16; ++mc) {
        uint32_t g[16], u[16];
        tmem_ld_x16(tmem_base + lane_off + mc * 16, g);
        tmem_ld_x16(tmem_base + lane_off + mt + mc * 16, u);
        tmem_wait_ld();
        reg_fence(g);
        reg_fence(u);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          part_buf[(mc * 16 + j) * kPackBlockN + r] = __uint_as_float(g[j]);
          part_buf[(mt + mc * 16 + j) * kPackBlockN + r] = __uint_as_float(u[j]);
        }
      }
    } else if (ok && kDown) {
      // down-projection: thread r owns output columns n0 + r and n0 + 128 + r
      tc_fence_after();
      __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y);
      const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(p.residual);
      const int n_lo = nblk * 2 * kPackBlockN + q * 32 + lane, n_hi = n_lo + kPackBlockN;
#pragma unroll 1
      for (int mc = 0; mc < mt / 16; ++mc) {
        uint32_t g[16], u[16];
        tmem_ld_x16(tmem_base + lane_off + mc * 16, g);
        tmem_ld_x16(tmem_base + lane_off + mt + mc * 16, u);
        tmem_wait_ld();
        reg_fence(g);
        reg_fence(u);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = mc * 16 + j;
          if (m >= mcount) continue;
          const size_t row = static_cast<size_t>(m0 + m) * p.N;
          if (n_lo < p.N)
            y[row + n_lo] = __float2bfloat16_rn(
                __uint_as_float(g[j]) + (res ? __bfloat162float(res[row + n_lo]) : 0.0f));
          if (n_hi < p.N)
            y[row + n_hi] = __float2bfloat16_rn(
                __uint_as_float(u[j]) + (res ? __bfloat162float(res[row + n_hi]) : 0.0f));
        }
      }
    } else if (ok) {
      tc_fence_after();
      __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y);
      const float sg = kFp8 ? p.scale_gate : 1.0f, su = kFp8 ? p.scale_up : 1.0f;
#pragma unroll 1
      for (int mc = 0; mc < mt / 16; ++mc) {
        uint32_t g[16], u[16];
        tmem_ld_x16(tmem_base + lane_off + mc * 16, g);
        tmem_ld_x16(tmem_base + lane_off + mt + mc * 16, u);
        tmem_wait_ld();
        reg_fence(g);
        reg_fence(u);
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = mc * 16 + j;
            if (m < mcount)
              y[static_cast<size_t>(m0 + m) * p.N + n] = __float2bfloat16_rn(
                  silu_mul(sg * __uint_as_float(g[j]), su * __uint_as_float(u[j])));
          }
        }
      }
    }
    __syncwarp();
  }

  if (kparts > 1) {
    // every part's partials are in its CTA's shared memory
    if (splits > 1)
      cluster_sync();
    else
      __syncthreads();
    // This CTA finishes weight rows [part * R, part * R + R) of the block for
    // all tokens: sum the parts (fixed order), SiLU(g) * u, 4 columns per item.
    const int rows = kPackBlockN / splits;
    const int chunks = rows / 4;
    const uint32_t local = smem_addr(smem);
    if (gsplits == 1) {
      // one cluster per unit (splits > 1): sum the cluster's parts and finish
      for (int idx = threadIdx.x; idx < mcount * chunks; idx += blockDim.x) {
        const int m = idx / chunks;
        const int r = part * rows + (idx % chunks) * 4;
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
        for (int s = 0; s < splits; ++s) {
          const uint32_t base = mapa_shared(local, static_cast<uint32_t>(s));
          const float4 gs = ld_shared_cluster_v4(base + 4u * static_cast<uint32_t>(m * kPackBlockN + r));
          const float4 us =
              ld_shared_cluster_v4(base + 4u * static_cast<uint32_t>((mt + m) * kPackBlockN + r));
          g.x += gs.x; g.y += gs.y; g.z += gs.z; g.w += gs.w;
          u.x += us.x; u.y += us.y; u.z += us.z; u.w += us.w;
        }
        finish_outputs<kFp8, kDown>(p, m0, nblk, m, r, g, u);
      }
    } else {
      // K split across clusters: this cluster's sums to the workspace,
      // [g rows | u rows] x mt x 128 floats per (unit, cluster)
      float* mine = p.ws + (size_t(unit) * gsplits + gpart) * (size_t(2) * mt * kPackBlockN);
      for (int idx = threadIdx.x; idx < mcount * chunks; idx += blockDim.x) {
        const int m = idx / chunks;
        const int r = part * rows + (idx % chunks) * 4;
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
        for (int s = 0; s < splits; ++s) {
          float4 gs, us;
          if (splits > 1) {
            const uint32_t base = mapa_shared(local, static_cast<uint32_t>(s));
            gs = ld_shared_cluster_v4(base + 4u * static_cast<uint32_t>(m * kPackBlockN + r));
            us = ld_shared_cluster_v4(base + 4u * static_cast<uint32_t>((mt + m) * kPackBlockN + r));
          } else {
            const float* own = reinterpret_cast<const float*>(smem);
            gs = *reinterpret_cast<const float4*>(own + m * kPackBlockN + r);
            us = *reinterpret_cast<const float4*>(own + (mt + m) * kPackBlockN + r);
          }
          g.x += gs.x; g.y += gs.y; g.z += gs.z; g.w += gs.w;
          u.x += us.x; u.y += us.y; u.z += us.z; u.w += us.w;
        }
        *reinterpret_cast<float4*>(mine + size_t(m) * kPackBlockN + r) = g;
        *reinterpret_cast<float4*>(mine + size_t(mt + m) * kPackBlockN + r) = u;
      }
    }
    if (splits > 1) cluster_sync();  // no CTA leaves while a peer may still read its partials
    if (gsplits > 1)
      cross_cluster_finish<kFp8, kDown>(p, unit, part, splits, gsplits, mt, mcount, m0, nblk,
                                        abort_flag + 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace

int small_m_stages(int mt, int ctas_per_sm, int extra) {
  // Shared memory per SM is 228 KB, of which 1 KB per resident CTA is reserved.
  const size_t per_cta = ctas_per_sm <= 1 ? kSmemLimit : (233472 - 2048) / 2;
  const size_t stage = kWStageBytes + size_t(mt) * kBlockK * 2 + size_t(extra);
  size_t s = (per_cta - 1024 - kBarBytes) / stage;
  if (s > kMaxStages) s = kMaxStages;
  return static_cast<int>(s);
}

size_t small_m_smem_bytes(int mt, int stages, int extra) {
  return 1024 + size_t(stages) * (kWStageBytes + size_t(mt) * kBlockK * 2 + size_t(extra)) +
         kBarBytes;
}

template <bool kFp8, bool kDown, bool kMx>
cudaError_t configure_small_m_t() {
  cudaError_t e = cudaFuncSetAttribute(fused_small_m_kernel<kFp8, kDown, kMx>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemLimit));
  if (e == cudaSuccess)  // all of the unified L1/shared array as shared memory (2 CTAs may share an SM)
    e = cudaFuncSetAttribute(fused_small_m_kernel<kFp8, kDown, kMx>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}

cudaError_t configure_small_m() {
  cudaError_t e = configure_small_m_t<false, false, false>();
  if (e == cudaSuccess) e = configure_small_m_t<true, false, false>();
  if (e == cudaSuccess) e = configure_small_m_t<false, true, false>();
  if (e == cudaSuccess) e = configure_small_m_t<true, false, true>();
  return e;
}

cudaError_t static_scratch_address(uint32_t** out) {
  // The array's name is a host-side stand-in in host code; the device address
  // comes from the runtime, for the current device.
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<uint32_t*>(ptr);
  return cudaSuccess;
}

int small_m_max_clusters(int splits) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemLimit;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, fused_small_m_kernel<false, false, false>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

cudaError_t launch_small_m(const SmallMParams& p, cudaStream_t stream) {
  if (p.stages < 2 || p.stages > kMaxStages || p.mt < 16 || p.mt > 256 || (p.mt % 16) != 0)
    return cudaErrorInvalidValue;
  const int splits = p.splits > 1 ? p.splits : 1;
  const int gsplits = p.gsplits > 1 ? p.gsplits : 1;
  const int bk = p.fp8 ? kBlockK8 : kBlockK;
  const int num_kb = (p.K + bk - 1) / bk;
  if (splits * gsplits > 1 &&
      (splits > 8 || (kPackBlockN % (4 * splits)) != 0 || splits * gsplits > num_kb || p.mt > 128 ||
       size_t(2) * p.mt * kPackBlockN * 4 > size_t(p.stages) * (kWStageBytes + size_t(p.mt) * kBlockK * 2) ||
       (p.grid % (splits * gsplits)) != 0))
    return cudaErrorInvalidValue;
  if (gsplits > 1 && (gsplits > kMaxClusters || !p.ws || !p.counters ||
                      (reinterpret_cast<uintptr_t>(p.ws) & 15u) != 0))
    return cudaErrorInvalidValue;
  // block-scaled FP8: one 128-token group (the scale blocks cover 128 rows
  // from m0 = 0) and 2 mt accumulator columns + the scale slots within 512
  if (p.mx && (!p.fp8 || p.down || (p.mgroups > 1) || p.mt > 128 ||
               2 * p.mt + kSfTmemCols * p.stages > 512))
    return cudaErrorInvalidValue;
  const int extra = p.mx ? kSfStageBytes : 0;
  SmallMParams q = p;
  q.l2_prefetch = small_m_l2_prefetch(p.grid, p.splits);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = small_m_smem_bytes(p.mt, p.stages, extra);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = splits > 1 ? 2 : 1;
  if (p.fp8 && p.down) return cudaErrorInvalidValue;  // no FP8 down-projection
  const cudaError_t e =
      p.down  ? cudaLaunchKernelEx(&cfg, fused_small_m_kernel<false, true, false>, q)
      : p.mx  ? cudaLaunchKernelEx(&cfg, fused_small_m_kernel<true, false, true>, q)
      : p.fp8 ? cudaLaunchKernelEx(&cfg, fused_small_m_kernel<true, false, false>, q)
              : cudaLaunchKernelEx(&cfg, fused_small_m_kernel<false, false, false>, q);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace swg
