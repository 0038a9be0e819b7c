// Host-side launch interface of the device kernels (internal to libswiglu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace swg {

constexpr int kPackBlockN = 128;  // columns per gate/up block of the packed weight
constexpr int kBlockK = 64;       // K elements per pipeline stage (128 B rows, 128-B swizzle)
constexpr int kBlockK8 = 128;     // the same 128-byte rows for one-byte (FP8 E4M3) elements
constexpr int kTileM = 128;       // tokens per large-M tile (MMA M)
constexpr int kThreads = 192;     // 6 warps: TMA producer, MMA issuer, 4 epilogue warps
// Block-scaled FP8: one UE8M0 scale per 32 K values; a 128-row x 4-group
// scale block is 512 bytes. Per 128-deep K slice a packed weight tile has two
// blocks (gate, up) and an activation chunk of 128 rows has one.
constexpr int kMxGroup = 32;
constexpr int kSfBlockBytes = 512;
constexpr int kSfStageBytes = 3 * kSfBlockBytes;  // gate + up weight scales, activation scales
constexpr int kSfTmemCols = 16;                   // TMEM columns per stage of scales (12 used)

struct LargeMParams {
  CUtensorMap tmap_a;  // A  [M, K]       box {64, 128}, 128-B swizzle
  CUtensorMap tmap_w;  // Wp {64, 256, tiles} box {64, bn, 1}, 128-B swizzle
  CUtensorMap tmap_y;  // Y  [M, N]       box {32, 32},  64-B swizzle (store)
  void* y;             // Y [M, N] bf16 (split-K kernel: plain row stores)
  int M, K, N;
  int tiles_m, tiles_n, group_m;
  int bn;    // output columns per tile: 32, 64 or 128 (MMA N = 2 * bn)
  int grid;  // persistent CTAs
  int fp8;   // E4M3 inputs (pair kernel): gate and up accumulators are scaled by
  float scale_gate, scale_up;  // scale_a * scale_w1 and scale_a * scale_w2 in the epilogue
  int down;  // down-projection (pair kernel): tiles of 256 output columns, out = acc + residual
  const void* residual;  // [M, N] bf16 or null (down-projection only)
  int mx;    // block-scaled E4M3 (pair kernel): scales from tmap_sw / tmap_sa
  CUtensorMap tmap_sw;   // weight scales: uint8 rows of 256 bytes, 4 rows (1 KB) per packed tile
  CUtensorMap tmap_sa;   // activation scales: uint8 rows of 256 bytes, 2 rows per 512-byte block
  uint32_t* status;
  uint64_t timeout_ns;
  int inject_stall;
  int l2_prefetch;  // single-CTA kernel: K slices of its first tile each CTA stages in L2
};

struct SmallMParams {
  CUtensorMap tmap_x;  // A  [M, K]     box {64, mt}, 128-B swizzle
  CUtensorMap tmap_w;  // Wp {64, 256, tiles} box {64, 256, 1}, 128-B swizzle
  void* y;             // Y  [M, N] bf16
  int M, K, N;
  int mt;      // tokens rounded up to a multiple of 16 (MMA N), <= 256
  int stages;  // pipeline depth
  int grid;    // one CTA per 128-column block, token group and K part (splits x gsplits)
  int splits;  // K parts per column block (<= 1: none); > 1: clusters of `splits` CTAs
  int mgroups; // token groups of mt rows each (<= 1: one group holds all M tokens)
  int fp8;     // E4M3 inputs: accumulators are scaled by scale_gate / scale_up
  float scale_gate, scale_up;
  int down;    // down-projection: a block is 256 output columns (rows 0-127 and 128-255
               // of the packed tile), out = acc + residual instead of SiLU(g) * u
  const void* residual;  // [M, N] bf16 or null (down-projection only)
  int mx;      // block-scaled E4M3 (with fp8): per-stage scales from tmap_sw / tmap_sa
  CUtensorMap tmap_sw;   // weight scales: uint8 rows of 256 bytes, 4 rows (1 KB) per packed tile
  CUtensorMap tmap_sa;   // activation scales: uint8 rows of 256 bytes, 2 rows per 512-byte block
  uint32_t* status;
  uint64_t timeout_ns;
  int inject_stall;
  int l2_prefetch;  // packed tiles per CTA staged in L2 before the grid-dependency wait
  // K split across clusters (gsplits > 1): each cluster's reduced fp32 partials
  // go to ws, per (unit, cluster) 2 * mt * 128 floats; counters (one per unit
  // and cluster rank, zero before the launch and again after it) elect the
  // last cluster of a unit, which sums all partials in cluster order
  int gsplits;
  float* ws;
  uint32_t* counters;
};

// One-time per-device set-up (dynamic shared-memory limits of every instantiation).
cudaError_t configure_large_m();
cudaError_t configure_small_m();

int large_m_stages(int bn);
// K slices of its first tile a single-CTA kernel CTA stages in L2 before its
// grid-dependency wait: about 64 MB of packed weight over the grid
// (SWIGLU_L2_PREFETCH_LARGE=n forces n; 0 turns it off).
int large_m_l2_prefetch(int grid, int bn);
size_t large_m_smem_bytes(int bn);
cudaError_t launch_large_m(const LargeMParams& p, cudaStream_t stream);

// CTA-pair variant (bn = 128, 256-row tiles, grid = 2 x pairs): one-time set-up
// also reports how many pairs can be resident at once.
cudaError_t configure_large_m_pair(int* max_pairs);
size_t large_m_pair_smem_bytes();
int large_m_pair_stages(bool mx = false);
// Number of the pair kernel's tile-round pacing waits that ran out on the
// current device since the library was loaded (a testing counter).
cudaError_t large_m_pair_pace_run_out(unsigned long long* count);
cudaError_t launch_large_m_pair(const LargeMParams& p, cudaStream_t stream);

// K split over the two CTAs of a cluster, one 128 x 64 output tile per cluster
// (grid = 2 x tiles): single-wave problems whose tiles need more operand bytes
// than one SM's shared memory holds.
cudaError_t configure_split_k(int* max_clusters);
int split_k_bn();
int split_k_stages();
cudaError_t launch_split_k(const LargeMParams& p, cudaStream_t stream);

// Whole K range resident in shared memory (K <= 64 * resident_pair_max_slices()):
// one 128 x 64 output tile per CTA pair (grid = 2 x tiles), M = 128 MMAs.
int resident_pair_max_slices();
int resident_pair_bn();
cudaError_t configure_resident_pair();
cudaError_t launch_resident_pair(const LargeMParams& p, cudaStream_t stream);

// Sequential gate-then-up schedule (bn = 128, 128-row tiles), an ablation.
cudaError_t configure_sequential();
int sequential_stages();
cudaError_t launch_sequential(const LargeMParams& p, cudaStream_t stream);

// Words of the static scratch array behind swiglu_forward_noalloc (256 bytes);
// a call uses the first kStatusWords of them for its status record.
constexpr int kStaticScratchWords = 64;
constexpr int kStatusWords = 4;
// Device address of that array on the current device (no allocation).
cudaError_t static_scratch_address(uint32_t** out);

// Pipeline depth of the decode kernel when `ctas_per_sm` CTAs share an SM;
// `extra` bytes of scales per stage (block-scaled FP8).
int small_m_stages(int mt, int ctas_per_sm, int extra = 0);

// Programmatic dependent launch for the fused kernels (on unless the
// environment sets SWIGLU_PDL=0): a launch may begin while the previous grid
// in the stream drains; the kernel waits for it before touching memory.
bool pdl_enabled();
// Packed weight tiles each decode CTA stages in L2 ahead of its pipeline, for
// a grid of `grid` CTAs in clusters of `splits` (SWIGLU_L2_PREFETCH=n forces n).
int small_m_l2_prefetch(int grid, int splits);
size_t small_m_smem_bytes(int mt, int stages, int extra = 0);
cudaError_t launch_small_m(const SmallMParams& p, cudaStream_t stream);
// Clusters of `splits` decode CTAs (shared memory at the 1-CTA-per-SM limit)
// that can be resident at once; 0 if such clusters cannot be launched.
int small_m_max_clusters(int splits);

cudaError_t launch_pack(const void* w1, const void* w2, void* wp, int K, int N,
                        cudaStream_t stream);
cudaError_t launch_pack_fp8(const void* w1, const void* w2, void* wp, int K, int N,
                            cudaStream_t stream);
// Block-scaled FP8 scales: W1's and W2's [K/32, N] -> 1 KB per packed tile;
// A's [M, K/32] -> 512-byte blocks [ceil(M/128)][ceil(K/128)].
cudaError_t launch_pack_mx_weight_scales(const void* s1, const void* s2, void* out, int K, int N,
                                         cudaStream_t stream);
cudaError_t launch_tile_mx_act_scales(const void* sa, void* out, int M, int K,
                                      cudaStream_t stream);
// Down-projection weight W3 [N, H] -> tiles of 256 output columns x 64 K values.
cudaError_t launch_pack_down(const void* w3, void* wp, int N, int H, cudaStream_t stream);

}  // namespace swg
