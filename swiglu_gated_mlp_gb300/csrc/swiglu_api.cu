// libswiglu C ABI: argument checks, per-device set-up, TMA descriptor encoding,
// kernel choice and launch. Declarations and contracts are in include/swiglu.h.
#include "swiglu.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxKN = int64_t(1) << 21;
constexpr int64_t kMaxM = 2147483647;

struct DeviceState {
  std::atomic<bool> ready{false};
  swiglu_status_t init_status = SWIGLU_OK;
  int sm_count = 0;
  int max_pairs = 0;           // CTA pairs of the pair kernel resident at once
  int small_clusters[9] = {};  // decode-kernel clusters of s CTAs resident at once (s = 2, 4, 8)
  int split_clusters = 0;      // split-K kernel clusters (of 2) resident at once
  bool resident_pair = false;  // the whole-K-resident pair kernel is set up
  uint32_t* status = nullptr;  // uint32_t[4], see ptx.cuh
};

DeviceState g_dev[kMaxDevices];
std::mutex g_init_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<int> g_inject{0};
std::atomic<uint64_t> g_timeout_ns{1000000000ull};

int64_t env_int(const char* name, int64_t dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  const long long x = std::strtoll(v, &end, 10);
  return (end && *end == '\0') ? static_cast<int64_t>(x) : dflt;
}

// Row tiles (of 256 rows) per group in the CTA-pair kernels' tile order: the
// 76 pairs sweep a group's rows before moving to the next column blocks. 16
// rows tiles read the least DRAM in a sweep of 4 to 32 on the 72B gate/up
// shapes (bf16 and FP8) and on the down-projections (K = 18944 to 29568),
// where no grouping keeps a wave's A and W panels in L2; smaller shapes have
// at most 16 row tiles, one group. SWIGLU_PAIR_GROUP_M=g forces g.
int64_t pair_group_rows(int64_t row_tiles) {
  static const int64_t forced = env_int("SWIGLU_PAIR_GROUP_M", 0);
  const int64_t g = forced > 0 ? forced : 16;
  return std::max<int64_t>(1, std::min(g, row_tiles));
}

// Largest M for which AUTO picks the small-M (weights-as-MMA-M) kernel.
int64_t small_m_max() {
  static const int64_t v = env_int("SWIGLU_SMALL_M_MAX", 32);
  return v;
}

}  // namespace

namespace swg {
bool pdl_enabled() {
  static const bool on = env_int("SWIGLU_PDL", 1) != 0;
  return on;
}
// Decode-kernel L2 staging depth. About 64 MB over the whole grid: deeper
// staging measured slower (the staged lines start to displace one another).
// K-split clusters stage 4 tiles: their grids leave SMs idle, so the next grid
// starts early and deep staging competes with the current grid's tail.
int small_m_l2_prefetch(int grid, int splits) {
  static const int64_t forced = env_int("SWIGLU_L2_PREFETCH", -1);
  if (forced >= 0) return static_cast<int>(std::min<int64_t>(forced, 64));
  if (splits > 1) return 4;
  const int64_t budget = int64_t(64) << 20;
  const int64_t per_tile = 2 * int64_t(kPackBlockN) * 128;  // one packed tile: 32 KB
  return static_cast<int>(std::clamp<int64_t>(budget / (int64_t(std::max(grid, 1)) * per_tile), 2, 16));
}
int large_m_l2_prefetch(int grid, int bn) {
  static const int64_t forced = env_int("SWIGLU_L2_PREFETCH_LARGE", -1);
  if (forced >= 0) return static_cast<int>(std::min<int64_t>(forced, 1 << 20));
  const int64_t budget = int64_t(64) << 20;
  const int64_t per_slice = 2 * int64_t(bn) * 128;  // gate and up rows of one 64-deep K slice
  return static_cast<int>(budget / (int64_t(std::max(grid, 1)) * per_slice));
}
}  // namespace swg

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

int64_t padded_n(int64_t n) {
  return (n + swg::kPackBlockN - 1) / swg::kPackBlockN * swg::kPackBlockN;
}

int64_t k_slices(int64_t k) { return (k + swg::kBlockK - 1) / swg::kBlockK; }

swiglu_status_t init_device(int dev, DeviceState& d) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_NO_DEVICE;
  }
  if (major != 10 || minor != 3) return SWIGLU_ERR_UNSUPPORTED;  // built for sm_103a only
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      return SWIGLU_ERR_CUDA;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (cudaMalloc(&d.status, 4 * sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(d.status, 0, 4 * sizeof(uint32_t)) != cudaSuccess ||
      swg::configure_large_m() != cudaSuccess || swg::configure_small_m() != cudaSuccess ||
      swg::configure_sequential() != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  for (int s : {2, 4, 8}) d.small_clusters[s] = swg::small_m_max_clusters(s);
  // The CTA-pair and split-K kernels are optional: if a set-up fails, that variant is unavailable.
  if (swg::configure_large_m_pair(&d.max_pairs) != cudaSuccess) {
    cudaGetLastError();
    d.max_pairs = 0;
  }
  if (swg::configure_split_k(&d.split_clusters) != cudaSuccess) {
    cudaGetLastError();
    d.split_clusters = 0;
  }
  d.resident_pair = swg::configure_resident_pair() == cudaSuccess;
  if (!d.resident_pair) cudaGetLastError();
  return SWIGLU_OK;
}

swiglu_status_t device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return SWIGLU_ERR_UNSUPPORTED;
  DeviceState& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_init_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
      d.init_status = init_device(dev, d);
      d.ready.store(true, std::memory_order_release);
    }
  }
  *out = &d;
  return d.init_status;
}

// Tensor-map encoding with a small per-thread cache: a decode step calls the
// library with the same few buffers over and over, and encoding is a fixed
// host cost on every call. Entries are keyed on every encoded field.
struct TmapKey {
  const void* base;
  int dtype;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  int rank;
  int swizzle;
  bool operator==(const TmapKey& o) const { return std::memcmp(this, &o, sizeof(TmapKey)) == 0; }
};

constexpr int kTmapCacheSize = 16;
struct TmapCache {
  TmapKey key[kTmapCacheSize];
  CUtensorMap map[kTmapCacheSize];
  bool used[kTmapCacheSize] = {};
  int next = 0;
};
thread_local TmapCache t_tmap_cache;

bool encode_cached(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle,
                   CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  TmapKey k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.dtype = static_cast<int>(dtype);
  k.rank = rank;
  k.swizzle = static_cast<int>(swizzle);
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  TmapCache& c = t_tmap_cache;
  for (int i = 0; i < kTmapCacheSize; ++i) {
    if (c.used[i] && c.key[i] == k) {
      *map = c.map[i];
      return true;
    }
  }
  cuuint32_t estr[3] = {1, 1, 1};
  if (g_encode(map, dtype, rank, const_cast<void*>(base),
               const_cast<cuuint64_t*>(dims), const_cast<cuuint64_t*>(strides),
               const_cast<cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  c.key[c.next] = k;
  c.map[c.next] = *map;
  c.used[c.next] = true;
  c.next = (c.next + 1) % kTmapCacheSize;
  return true;
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return encode_cached(map, base, 2, dims, strides, box, swizzle, dtype);
}

// The packed weight as a 3-D tensor {64 K values, 256 rows, tiles}: every tile
// (one 128-column block x one 64-deep K slice, gate rows then up rows) is a
// contiguous 32 KB span; boxes of {64, rows, 1} are taken from one tile.
bool encode_packed_w(CUtensorMap* map, const void* base, int64_t K, int64_t N, uint32_t rows) {
  const int64_t tiles = (padded_n(N) / swg::kPackBlockN) * k_slices(K);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(swg::kBlockK), 2u * swg::kPackBlockN,
                              static_cast<cuuint64_t>(tiles)};
  const cuuint64_t strides[2] = {swg::kBlockK * 2, 2u * swg::kPackBlockN * swg::kBlockK * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(swg::kBlockK), rows, 1};
  return encode_cached(map, base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The packed down-projection weight: {64 K values, 256 output columns, tiles}.
int64_t padded_h(int64_t h) { return (h + 255) / 256 * 256; }

bool encode_packed_down(CUtensorMap* map, const void* base, int64_t N, int64_t H, uint32_t rows) {
  const int64_t tiles = (padded_h(H) / 256) * k_slices(N);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(swg::kBlockK), 256,
                              static_cast<cuuint64_t>(tiles)};
  const cuuint64_t strides[2] = {swg::kBlockK * 2, 256u * swg::kBlockK * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(swg::kBlockK), rows, 1};
  return encode_cached(map, base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The FP8 packed weight: {128 one-byte K values, 256 rows, tiles}, 32 KB tiles.
int64_t k_slices8(int64_t k) { return (k + swg::kBlockK8 - 1) / swg::kBlockK8; }

bool encode_packed_w8(CUtensorMap* map, const void* base, int64_t K, int64_t N, uint32_t rows) {
  const int64_t tiles = (padded_n(N) / swg::kPackBlockN) * k_slices8(K);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(swg::kBlockK8), 2u * swg::kPackBlockN,
                              static_cast<cuuint64_t>(tiles)};
  const cuuint64_t strides[2] = {swg::kBlockK8, 2u * swg::kPackBlockN * swg::kBlockK8};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(swg::kBlockK8), rows, 1};
  return encode_cached(map, base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

struct Plan {
  int variant = SWIGLU_VARIANT_AUTO;
  int bn = 0, stages = 0, tiles_m = 0, tiles_n = 0, group_m = 0, tiles = 0, grid = 0, mt = 0;
  int splits = 1;
  int mgroups = 1;
};

// Decode-kernel work split for `blocks` weight blocks and M tokens: token
// groups of mt rows, pipeline depth, and K parts per cluster. With few blocks
// for the SMs, more than 64 tokens go in 64-token groups (each group streams
// the same weights, the repeats coming from L2), and each (block, group) unit
// splits K over a cluster so that the units fill the SMs; all clusters must be
// resident at once.
void decode_split_plan(int64_t M, int64_t blocks, int64_t kslices, const DeviceState* d,
                       int* mt, int* mgroups, int* stages, int* splits) {
  const int sm_count = d ? d->sm_count : 0;
  *mt = static_cast<int>((M + 15) / 16 * 16);
  *mgroups = 1;
  if (d && M > 64 && blocks * 2 <= sm_count) {
    *mt = 64;
    *mgroups = static_cast<int>((M + 63) / 64);
  }
  const int64_t units = blocks * *mgroups;
  *stages = swg::small_m_stages(*mt, 1);
  if (sm_count > 0 && units > sm_count && swg::small_m_stages(*mt, 2) >= 3)
    *stages = swg::small_m_stages(*mt, 2);
  *splits = 1;
  const int64_t stage_bytes = 2 * swg::kPackBlockN * swg::kBlockK * 2 + int64_t(*mt) * 128;
  if (d && *mt <= 128 && int64_t(*mt) * 1024 <= *stages * stage_bytes) {
    for (int s : {8, 4, 2}) {
      if (units * s <= sm_count && s <= kslices && d->small_clusters[s] >= units) {
        *splits = s;
        break;
      }
    }
  }
}

struct DownPlan {
  bool decode = false;
  int mt = 0, mgroups = 1, stages = 0, splits = 1, grid = 0;  // splits: decode clusters
  int gsplits = 1;  // decode: clusters per unit (K split across clusters, caller workspace)
  int64_t blocks = 0, pm = 0, tiles = 0, group = 1;
};

// Decode-kernel K split across clusters, for a call with a workspace. It adds
// a tail to every launch (partial sums to the workspace, a fence and a counter,
// and the last cluster's final sum: about 3 us), so it is taken only where it
// raises the CTA count by at least 40 % over the plan without it, and with
// token tiles of at most 32 (the tail grows with the tile). Then the largest
// cluster size s and, for it, the most clusters g per unit (at most 8) with
// every CTA resident at once (one per SM; clusters of s must all fit). From a
// sweep of (s, g) on the 7B, 32B and 72B shapes at M = 1..64 and the 0.5B
// shape: 32B (20 blocks) at M <= 32 gains 6-10 % with (2, 3), 120 CTAs
// against 80; 7B (112 -> 140 CTAs), 72B (128) and 64-token tiles lose.
void down_cross_cluster_split(int64_t units, int64_t kslices, int mt, const DeviceState* d,
                              int* splits, int* gsplits) {
  const int sm_count = d->sm_count;
  // SWIGLU_DOWN_CLUSTER=s and SWIGLU_DOWN_CLUSTERS=g force the split (for measurements)
  static const int64_t forced_s = env_int("SWIGLU_DOWN_CLUSTER", 0);
  static const int64_t forced_g = env_int("SWIGLU_DOWN_CLUSTERS", 0);
  const auto fits = [&](int s, int g) {
    return g <= 8 && units * s * g <= sm_count && s * g <= kslices &&
           (s == 1 || d->small_clusters[s] >= units * g);
  };
  if (forced_s > 0 && forced_g > 0) {
    const int fs = static_cast<int>(forced_s), fg = static_cast<int>(forced_g);
    if ((fs == 1 || fs == 2 || fs == 4 || fs == 8) && fits(fs, fg)) {
      *splits = fs;
      *gsplits = fg;
    }
    return;
  }
  if (mt > 32) return;
  const int64_t base = units * *splits;
  for (int s : {8, 4, 2, 1}) {
    int g = 0;
    for (int c = 2; fits(s, c); ++c) g = c;
    if (g >= 2 && units * s * g * 10 >= base * 14) {
      *splits = s;
      *gsplits = g;
      return;
    }
  }
}

// Bytes of the decode down-projection's workspace for a plan: one counter per
// (unit, cluster rank), then 2 * mt * 128 fp32 partials per (unit, cluster).
size_t down_workspace_bytes(const DownPlan& dp) {
  if (!dp.decode || dp.gsplits <= 1) return 0;
  const size_t units = size_t(dp.blocks) * size_t(dp.mgroups);
  const size_t counters = (units * size_t(dp.splits) * 4 + 255) / 256 * 256;
  return counters + units * size_t(dp.gsplits) * 2 * size_t(dp.mt) * swg::kPackBlockN * 4;
}

// The down-projection's kernel and launch shape; `cross_cluster` allows the
// decode kernel's K split across clusters (the call has a workspace).
swiglu_status_t make_down_plan(int64_t M, int64_t N, int64_t H, const DeviceState* d,
                               DownPlan* dp, bool cross_cluster = false) {
  *dp = DownPlan{};
  dp->blocks = padded_h(H) / 256;  // 256 output columns per block
  const int64_t ks = k_slices(N);
  // decode kernel for few tokens, or up to 128 tokens when there are few output
  // blocks for the SMs (K then splits over clusters); CTA pairs otherwise
  if (M <= 64 || (M <= swg::kTileM && dp->blocks * 2 <= d->sm_count)) {
    dp->decode = true;
    decode_split_plan(M, dp->blocks, ks, d, &dp->mt, &dp->mgroups, &dp->stages, &dp->splits);
    const int64_t stage_bytes = 2 * swg::kPackBlockN * swg::kBlockK * 2 + int64_t(dp->mt) * 128;
    if (cross_cluster && dp->mt <= 128 && int64_t(dp->mt) * 1024 <= dp->stages * stage_bytes)
      down_cross_cluster_split(dp->blocks * dp->mgroups, ks, dp->mt, d, &dp->splits,
                               &dp->gsplits);
    dp->grid = static_cast<int>(dp->blocks * dp->mgroups * dp->splits * dp->gsplits);
    return SWIGLU_OK;
  }
  if (d->max_pairs < 1) return SWIGLU_ERR_UNSUPPORTED;
  dp->pm = (M + 2 * swg::kTileM - 1) / (2 * swg::kTileM);
  dp->tiles = dp->pm * dp->blocks;
  if (dp->tiles > 2147483647) return SWIGLU_ERR_UNSUPPORTED;
  dp->group = pair_group_rows(dp->pm);
  dp->grid = 2 * static_cast<int>(dp->tiles < d->max_pairs ? dp->tiles : d->max_pairs);
  return SWIGLU_OK;
}

// `d` may be null (allocation-free entry point): no SM count, no cluster data.
swiglu_status_t make_plan(int64_t M, int64_t K, int64_t N, int variant, const DeviceState* d,
                          Plan* pl, int elem_bytes = 2) {
  // 128-byte K slices: 64 bf16 or 128 E4M3 values
  const int64_t kslices = elem_bytes == 1 ? k_slices8(K) : k_slices(K);
  const int sm_count = d ? d->sm_count : 0;
  const int max_pairs = d ? d->max_pairs : 0;
  const int split_clusters = d ? d->split_clusters : 0;
  if (variant < SWIGLU_VARIANT_AUTO || variant > SWIGLU_VARIANT_RESIDENT_PAIR)
    return SWIGLU_ERR_INVALID_ARG;
  const int64_t split_bn = swg::split_k_bn();
  const int64_t split_tiles = ((M + swg::kTileM - 1) / swg::kTileM) * ((N + split_bn - 1) / split_bn);
  if (variant == SWIGLU_VARIANT_AUTO) {
    const int64_t nb = padded_n(N) / swg::kPackBlockN;
    const int64_t tiles128 = ((M + swg::kTileM - 1) / swg::kTileM) * nb;
    // From a sweep of M = 1..128 on the 7B and 32B shapes (every kernel, CUDA
    // events): the decode kernel up to 32 tokens, up to 64 on narrow N (K split
    // over clusters), up to 80 when the column blocks fill most SMs at one CTA
    // each; single CTAs up to 128 tokens; CTA pairs above when the 128-row
    // tiles fill the SMs.
    if (M <= small_m_max() && M <= 256) {
      variant = SWIGLU_VARIANT_SMALL_M;                  // decode: stream the weights once
    } else if (M <= 64 && sm_count > 0 && nb * 2 <= sm_count) {
      variant = SWIGLU_VARIANT_SMALL_M;                  // few column blocks: split K in clusters
    } else if (M <= 80 && sm_count > 0 && nb <= sm_count && nb * 2 > sm_count) {
      variant = SWIGLU_VARIANT_SMALL_M;                  // one resident CTA per column block
    } else if (M > swg::kTileM && max_pairs > 0 && tiles128 >= sm_count) {
      variant = SWIGLU_VARIANT_LARGE_M_PAIR;             // 256-row tiles on CTA pairs
    } else {
      variant = SWIGLU_VARIANT_LARGE_M;
    }
  }
  const int64_t np = padded_n(N);
  pl->variant = variant;
  if (variant == SWIGLU_VARIANT_SMALL_M) {
    if (M > 256) return SWIGLU_ERR_UNSUPPORTED;
    pl->tiles = static_cast<int>(np / swg::kPackBlockN);
    // One CTA per SM with the deepest ring, unless there are more (block, token
    // group) units than SMs: then two CTAs per SM (3+ stages each) keep the
    // whole grid resident; with few units, K splits over clusters.
    decode_split_plan(M, pl->tiles, kslices, d, &pl->mt, &pl->mgroups, &pl->stages, &pl->splits);
    pl->grid = pl->tiles * pl->mgroups * pl->splits;
    return SWIGLU_OK;
  }
  if (variant == SWIGLU_VARIANT_RESIDENT_PAIR) {
    // every K slice resident: 128 x 64 tiles, one per CTA pair
    if (!d || !d->resident_pair || elem_bytes != 2 || kslices > swg::resident_pair_max_slices())
      return SWIGLU_ERR_UNSUPPORTED;
    const int64_t bn = swg::resident_pair_bn();
    const int64_t tm = (M + swg::kTileM - 1) / swg::kTileM, tn = (N + bn - 1) / bn;
    if (tm * tn > 1073741823) return SWIGLU_ERR_UNSUPPORTED;
    pl->bn = static_cast<int>(bn);
    pl->tiles_m = static_cast<int>(tm);
    pl->tiles_n = static_cast<int>(tn);
    pl->group_m = 1;
    pl->tiles = static_cast<int>(tm * tn);
    pl->grid = 2 * pl->tiles;
    return SWIGLU_OK;
  }
  if (variant == SWIGLU_VARIANT_SPLIT_K) {
    if (split_clusters < 1 || elem_bytes != 2) return SWIGLU_ERR_UNSUPPORTED;
    if (split_tiles > 1073741823) return SWIGLU_ERR_UNSUPPORTED;
    pl->bn = static_cast<int>(split_bn);
    pl->stages = swg::split_k_stages();
    pl->tiles_m = static_cast<int>((M + swg::kTileM - 1) / swg::kTileM);
    pl->tiles_n = static_cast<int>((N + split_bn - 1) / split_bn);
    pl->group_m = 1;
    pl->tiles = static_cast<int>(split_tiles);
    pl->grid = 2 * pl->tiles;
    return SWIGLU_OK;
  }
  if (variant == SWIGLU_VARIANT_SEQUENTIAL) {
    const int64_t tm = (M + swg::kTileM - 1) / swg::kTileM;
    const int64_t tiles = tm * (np / swg::kPackBlockN);
    if (tiles > 2147483647) return SWIGLU_ERR_UNSUPPORTED;
    int64_t group = (48ll << 20) / (int64_t(swg::kTileM) * K * 2);
    if (group < 1) group = 1;
    if (group > tm) group = tm;
    const int sms = sm_count > 0 ? sm_count : 1;
    pl->bn = swg::kPackBlockN;
    pl->stages = swg::sequential_stages();
    pl->tiles_m = static_cast<int>(tm);
    pl->tiles_n = static_cast<int>(np / swg::kPackBlockN);
    pl->group_m = static_cast<int>(group);
    pl->tiles = static_cast<int>(tiles);
    pl->grid = static_cast<int>(tiles < sms ? tiles : sms);
    return SWIGLU_OK;
  }
  if (variant == SWIGLU_VARIANT_LARGE_M_PAIR) {
    if (max_pairs < 1) return SWIGLU_ERR_UNSUPPORTED;
    const int64_t pm = (M + 2 * swg::kTileM - 1) / (2 * swg::kTileM);  // 256-row tiles
    const int64_t ptiles = pm * (np / swg::kPackBlockN);
    if (ptiles > 2147483647) return SWIGLU_ERR_UNSUPPORTED;
    const int64_t group = pair_group_rows(pm);
    pl->bn = swg::kPackBlockN;
    pl->stages = swg::large_m_pair_stages();
    pl->tiles_m = static_cast<int>(pm);
    pl->tiles_n = static_cast<int>(np / swg::kPackBlockN);
    pl->group_m = static_cast<int>(group);
    pl->tiles = static_cast<int>(ptiles);
    pl->grid = 2 * static_cast<int>(ptiles < max_pairs ? ptiles : max_pairs);
    return SWIGLU_OK;
  }
  const int64_t tiles_m = (M + swg::kTileM - 1) / swg::kTileM;
  int bn = 32;
  for (int cand : {128, 64, 32}) {
    if (tiles_m * (np / cand) >= sm_count) {
      bn = cand;
      break;
    }
  }
  const int64_t tiles = tiles_m * (np / bn);
  if (tiles > 2147483647) return SWIGLU_ERR_UNSUPPORTED;
  pl->bn = bn;
  pl->stages = swg::large_m_stages(bn);
  pl->tiles_m = static_cast<int>(tiles_m);
  pl->tiles_n = static_cast<int>(np / bn);
  // Row tiles per group: as many as keep the group's A rows within about a
  // third of L2 (so W is read from HBM once per group, ideally once).
  const int64_t a_tile_bytes = int64_t(swg::kTileM) * K * 2;
  int64_t group = (48ll << 20) / (a_tile_bytes > 0 ? a_tile_bytes : 1);
  if (group < 1) group = 1;
  if (group > tiles_m) group = tiles_m;
  pl->group_m = static_cast<int>(group);
  pl->tiles = static_cast<int>(tiles);
  pl->grid = static_cast<int>(tiles < sm_count ? tiles : sm_count);
  return SWIGLU_OK;
}

swiglu_status_t check_shape(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || K <= 0 || N <= 0) return SWIGLU_ERR_INVALID_ARG;
  if ((K % 8) != 0 || (N % 8) != 0) return SWIGLU_ERR_UNSUPPORTED;  // 16-byte TMA row stride
  if (M > kMaxM || K > kMaxKN || N > kMaxKN) return SWIGLU_ERR_UNSUPPORTED;
  return SWIGLU_OK;
}

swiglu_status_t check_forward_args(const void* A, const void* Wp, const void* Y, int64_t M,
                                   int64_t K, int64_t N) {
  const swiglu_status_t st = check_shape(M, K, N);
  if (st != SWIGLU_OK || M == 0) return st;
  if (!A || !Wp || !Y) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Wp) || !aligned16(Y)) return SWIGLU_ERR_INVALID_ARG;
  const size_t a_bytes = size_t(M) * size_t(K) * 2, y_bytes = size_t(M) * size_t(N) * 2;
  const size_t w_bytes = swiglu_packed_weight_bytes(K, N);
  if (overlaps(Y, y_bytes, A, a_bytes) || overlaps(Y, y_bytes, Wp, w_bytes))
    return SWIGLU_ERR_INVALID_ARG;
  return SWIGLU_OK;
}

swiglu_status_t launch_forward(const void* A, const void* Wp, void* Y, int64_t M, int64_t K,
                               int64_t N, const Plan& pl, DeviceState& d, cudaStream_t stream) {
  const uint64_t timeout = g_timeout_ns.load();
  const int inject = g_inject.load();
  cudaError_t err;
  if (pl.variant == SWIGLU_VARIANT_SMALL_M) {
    swg::SmallMParams p{};
    if (!encode_2d(&p.tmap_x, A, K, M, K * 2, swg::kBlockK, pl.mt,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_packed_w(&p.tmap_w, Wp, K, N, 2 * swg::kPackBlockN))
      return SWIGLU_ERR_CUDA;
    p.y = Y;
    p.M = static_cast<int>(M);
    p.K = static_cast<int>(K);
    p.N = static_cast<int>(N);
    p.mt = pl.mt;
    p.stages = pl.stages;
    p.grid = pl.grid;
    p.splits = pl.splits;
    p.mgroups = pl.mgroups;
    p.status = d.status;
    p.timeout_ns = timeout;
    p.inject_stall = inject;
    err = swg::launch_small_m(p, stream);
  } else {
    swg::LargeMParams p{};
    // the whole-K-resident pair kernel: 64 A rows per CTA, 32 gate (up) rows per load
    const bool resident = pl.variant == SWIGLU_VARIANT_RESIDENT_PAIR;
    if (!encode_2d(&p.tmap_a, A, K, M, K * 2, swg::kBlockK, resident ? swg::kTileM / 2 : swg::kTileM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_packed_w(&p.tmap_w, Wp, K, N, resident ? pl.bn / 2 : pl.bn) ||
        !encode_2d(&p.tmap_y, Y, N, M, N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return SWIGLU_ERR_CUDA;
    p.y = Y;
    p.M = static_cast<int>(M);
    p.K = static_cast<int>(K);
    p.N = static_cast<int>(N);
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.group_m = pl.group_m;
    p.bn = pl.bn;
    p.grid = pl.grid;
    p.status = d.status;
    p.timeout_ns = timeout;
    p.inject_stall = inject;
    if (pl.variant == SWIGLU_VARIANT_LARGE_M) p.l2_prefetch = swg::large_m_l2_prefetch(pl.grid, pl.bn);
    err = pl.variant == SWIGLU_VARIANT_LARGE_M_PAIR ? swg::launch_large_m_pair(p, stream)
          : pl.variant == SWIGLU_VARIANT_SEQUENTIAL ? swg::launch_sequential(p, stream)
          : pl.variant == SWIGLU_VARIANT_SPLIT_K    ? swg::launch_split_k(p, stream)
          : resident                                ? swg::launch_resident_pair(p, stream)
                                                    : swg::launch_large_m(p, stream);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

// ---- set-up of the allocation-free entry point (swiglu_forward_noalloc) ----
// Per device: compute capability, the tensor-map encoder, the decode kernel's
// shared-memory limit and the device address of the static scratch array. No
// step allocates device memory.
struct NoAllocState {
  std::atomic<bool> ready{false};
  swiglu_status_t init_status = SWIGLU_OK;
  uint32_t* scratch = nullptr;
};
NoAllocState g_noalloc[kMaxDevices];

swiglu_status_t noalloc_init(NoAllocState& s) {
  int dev = -1, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_NO_DEVICE;
  }
  if (major != 10 || minor != 3) return SWIGLU_ERR_UNSUPPORTED;
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      return SWIGLU_ERR_CUDA;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (swg::configure_small_m() != cudaSuccess || swg::static_scratch_address(&s.scratch) != cudaSuccess ||
      s.scratch == nullptr) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

swiglu_status_t noalloc_state(NoAllocState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return SWIGLU_ERR_UNSUPPORTED;
  NoAllocState& s = g_noalloc[dev];
  if (!s.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_init_mu);
    if (!s.ready.load(std::memory_order_relaxed)) {
      s.init_status = noalloc_init(s);
      s.ready.store(true, std::memory_order_release);
    }
  }
  *out = &s;
  return s.init_status;
}

}  // namespace

namespace {
// Text form of a plan (swiglu_plan_string, swiglu_plan_string_fp8).
void format_plan(const Plan& pl, const DeviceState& d, const char* prefix, char* buf,
                 size_t buflen) {
  if (pl.variant == SWIGLU_VARIANT_SMALL_M)
    std::snprintf(buf, buflen,
                  "%ssmall_m mt=%d stages=%d tiles=%d groups=%d splits=%d grid=%d l2_prefetch=%d sms=%d",
                  prefix, pl.mt, pl.stages, pl.tiles, pl.mgroups, pl.splits, pl.grid,
                  swg::small_m_l2_prefetch(pl.grid, pl.splits), d.sm_count);
  else if (pl.variant == SWIGLU_VARIANT_SEQUENTIAL)
    std::snprintf(buf, buflen, "%ssequential bn=%d stages=%d tiles=%d grid=%d group_m=%d sms=%d",
                  prefix, pl.bn, pl.stages, pl.tiles, pl.grid, pl.group_m, d.sm_count);
  else if (pl.variant == SWIGLU_VARIANT_RESIDENT_PAIR)
    std::snprintf(buf, buflen, "%sresident_pair bn=%d tiles=%d grid=%d sms=%d", prefix, pl.bn,
                  pl.tiles, pl.grid, d.sm_count);
  else if (pl.variant == SWIGLU_VARIANT_SPLIT_K)
    std::snprintf(buf, buflen, "%ssplit_k bn=%d stages=%d tiles=%d grid=%d clusters=%d sms=%d",
                  prefix, pl.bn, pl.stages, pl.tiles, pl.grid, d.split_clusters, d.sm_count);
  else if (pl.variant == SWIGLU_VARIANT_LARGE_M_PAIR)
    std::snprintf(buf, buflen,
                  "%slarge_m_pair bn=%d stages=%d tiles=%d grid=%d group_m=%d max_pairs=%d sms=%d",
                  prefix, pl.bn, pl.stages, pl.tiles, pl.grid, pl.group_m, d.max_pairs, d.sm_count);
  else
    std::snprintf(buf, buflen, "%slarge_m bn=%d stages=%d tiles=%d grid=%d group_m=%d sms=%d",
                  prefix, pl.bn, pl.stages, pl.tiles, pl.grid, pl.group_m, d.sm_count);
}

// The FP8 entry point's kernel: as for bf16, the decode kernel up to 32 tokens,
// up to 64 on narrow N, up to 80 when the column blocks fill most SMs at one
// CTA each (there it beat the pair kernel by 4-11 % at M = 40-80 on the 7B
// shape); the CTA-pair kernel otherwise (there is no single-CTA FP8 kernel).
bool fp8_uses_decode(int64_t M, int64_t N, const DeviceState& d) {
  const int64_t nb = padded_n(N) / swg::kPackBlockN;
  return M <= 32 || (M <= 64 && nb * 2 <= d.sm_count) ||
         (M <= 80 && nb <= d.sm_count && nb * 2 > d.sm_count) || d.max_pairs < 1;
}

// Scale bytes of the block-scaled packed weight: 1 KB per (column block, K slice) tile.
size_t mx_weight_scale_bytes(int64_t K, int64_t N) {
  return size_t(padded_n(N) / swg::kPackBlockN) * size_t(k_slices8(K)) * 2 * swg::kSfBlockBytes;
}

// The block-scaled forward's kernel and launch shape: the decode kernel by the
// FP8 rule, with all tokens in one group (a scale block holds 128 rows from
// token 0, so M <= 128), the ring sized with the scales, two CTAs per SM when
// the column blocks outnumber the SMs, and K split over clusters on narrow N
// as for the other forms; CTA pairs otherwise.
swiglu_status_t make_mx_plan(int64_t M, int64_t K, int64_t N, const DeviceState& d, Plan* pl) {
  const int64_t kslices = k_slices8(K);
  if (M > 128 || !fp8_uses_decode(M, N, d)) {
    if (d.max_pairs < 1) return SWIGLU_ERR_UNSUPPORTED;
    const swiglu_status_t st = make_plan(M, K, N, SWIGLU_VARIANT_LARGE_M_PAIR, &d, pl, 1);
    pl->stages = swg::large_m_pair_stages(true);
    return st;
  }
  *pl = Plan{};
  pl->variant = SWIGLU_VARIANT_SMALL_M;
  pl->tiles = static_cast<int>(padded_n(N) / swg::kPackBlockN);
  pl->mt = static_cast<int>((M + 15) / 16 * 16);
  pl->mgroups = 1;
  pl->stages = swg::small_m_stages(pl->mt, 1, swg::kSfStageBytes);
  if (pl->tiles > d.sm_count) {
    // more column blocks than SMs: two CTAs per SM keep the whole grid
    // resident (3+ stages each; accumulators and scale slots in 256 columns)
    const int s2 = swg::small_m_stages(pl->mt, 2, swg::kSfStageBytes);
    if (s2 >= 3 && 2 * pl->mt + swg::kSfTmemCols * s2 <= 256) pl->stages = s2;
  }
  pl->splits = 1;
  const int64_t stage_bytes = 2 * swg::kPackBlockN * swg::kBlockK * 2 + int64_t(pl->mt) * 128;
  if (int64_t(pl->mt) * 1024 <= pl->stages * stage_bytes) {
    for (int s : {8, 4, 2}) {
      if (int64_t(pl->tiles) * s <= d.sm_count && s <= kslices && d.small_clusters[s] >= pl->tiles) {
        pl->splits = s;
        break;
      }
    }
  }
  pl->grid = pl->tiles * pl->splits;
  return SWIGLU_OK;
}
}  // namespace

extern "C" {

size_t swiglu_packed_weight_bytes(int64_t K, int64_t N) {
  if (K <= 0 || N <= 0 || K > kMaxKN || N > kMaxKN) return 0;
  return size_t(2) * size_t(padded_n(N)) * size_t(k_slices(K) * swg::kBlockK) * 2;
}

swiglu_status_t swiglu_pack_weights(const void* W1, const void* W2, void* Wpacked, int64_t K,
                                    int64_t N, swiglu_stream_t stream) {
  swiglu_status_t st = check_shape(0, K, N);
  if (st != SWIGLU_OK) return st;
  if (!W1 || !W2 || !Wpacked) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(W1) || !aligned16(W2) || !aligned16(Wpacked)) return SWIGLU_ERR_INVALID_ARG;
  const size_t w_bytes = size_t(K) * size_t(N) * 2;
  const size_t p_bytes = swiglu_packed_weight_bytes(K, N);
  if (overlaps(Wpacked, p_bytes, W1, w_bytes) || overlaps(Wpacked, p_bytes, W2, w_bytes))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  if (swg::launch_pack(W1, W2, Wpacked, static_cast<int>(K), static_cast<int>(N),
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

swiglu_status_t swiglu_forward_variant(const void* A, const void* Wpacked, void* Y, int64_t M,
                                       int64_t K, int64_t N, int variant,
                                       swiglu_stream_t stream) {
  swiglu_status_t st = check_forward_args(A, Wpacked, Y, M, K, N);
  if (st != SWIGLU_OK) return st;
  if (variant < SWIGLU_VARIANT_AUTO || variant > SWIGLU_VARIANT_RESIDENT_PAIR)
    return SWIGLU_ERR_INVALID_ARG;
  if (M == 0) return SWIGLU_OK;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  Plan pl;
  st = make_plan(M, K, N, variant, d, &pl);
  if (st != SWIGLU_OK) return st;
  return launch_forward(A, Wpacked, Y, M, K, N, pl, *d, reinterpret_cast<cudaStream_t>(stream));
}

swiglu_status_t swiglu_forward(const void* A, const void* Wpacked, void* Y, int64_t M, int64_t K,
                               int64_t N, swiglu_stream_t stream) {
  return swiglu_forward_variant(A, Wpacked, Y, M, K, N, SWIGLU_VARIANT_AUTO, stream);
}

swiglu_status_t swiglu_forward_from_host(const void* A_host, const void* Wpacked, void* Y_host,
                                         void* A_dev, void* Y_dev, int64_t M, int64_t K,
                                         int64_t N, swiglu_stream_t stream) {
  swiglu_status_t st = check_forward_args(A_dev, Wpacked, Y_dev, M, K, N);
  if (st != SWIGLU_OK) return st;
  if (M == 0) return SWIGLU_OK;
  if (!A_host || !Y_host) return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(A_dev, A_host, size_t(M) * size_t(K) * 2, cudaMemcpyHostToDevice, s) !=
      cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  Plan pl;
  st = make_plan(M, K, N, SWIGLU_VARIANT_AUTO, d, &pl);
  if (st != SWIGLU_OK) return st;
  st = launch_forward(A_dev, Wpacked, Y_dev, M, K, N, pl, *d, s);
  if (st != SWIGLU_OK) return st;
  if (cudaMemcpyAsync(Y_host, Y_dev, size_t(M) * size_t(N) * 2, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

swiglu_status_t swiglu_check_device_status(swiglu_stream_t stream) {
  DeviceState* d = nullptr;
  swiglu_status_t st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  uint32_t h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, d->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  if (h[0] == 0) return SWIGLU_OK;
  if (std::getenv("SWIGLU_VERBOSE"))
    std::fprintf(stderr, "libswiglu: device status %u (wait site %u, block %u, %u failures)\n",
                 h[0], h[1], h[2], h[3]);
  if (cudaMemset(d->status, 0, sizeof(h)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return h[0] == 4 ? SWIGLU_ERR_TIMEOUT : SWIGLU_ERR_CUDA;
}

const char* swiglu_status_string(swiglu_status_t status) {
  switch (status) {
    case SWIGLU_OK: return "SWIGLU_OK";
    case SWIGLU_ERR_INVALID_ARG: return "SWIGLU_ERR_INVALID_ARG: invalid argument";
    case SWIGLU_ERR_UNSUPPORTED: return "SWIGLU_ERR_UNSUPPORTED: unsupported shape or device";
    case SWIGLU_ERR_CUDA: return "SWIGLU_ERR_CUDA: CUDA call or kernel launch failed";
    case SWIGLU_ERR_TIMEOUT: return "SWIGLU_ERR_TIMEOUT: a kernel pipeline wait timed out";
    case SWIGLU_ERR_NO_DEVICE: return "SWIGLU_ERR_NO_DEVICE: no usable CUDA device";
    default: return "SWIGLU_ERR_UNKNOWN";
  }
}

swiglu_status_t swiglu_plan_string(int64_t M, int64_t K, int64_t N, int variant, char* buf,
                                   size_t buflen) {
  if (!buf || buflen == 0) return SWIGLU_ERR_INVALID_ARG;
  buf[0] = '\0';
  swiglu_status_t st = check_shape(M, K, N);
  if (st != SWIGLU_OK) return st;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  Plan pl;
  st = make_plan(M < 1 ? 1 : M, K, N, variant, d, &pl);
  if (st != SWIGLU_OK) return st;
  format_plan(pl, *d, "", buf, buflen);
  return SWIGLU_OK;
}

swiglu_status_t swiglu_plan_string_fp8(int64_t M, int64_t K, int64_t N, char* buf,
                                       size_t buflen) {
  if (!buf || buflen == 0) return SWIGLU_ERR_INVALID_ARG;
  buf[0] = '\0';
  swiglu_status_t st = check_shape(M, K, N);
  if (st != SWIGLU_OK) return st;
  if ((K % 16) != 0) return SWIGLU_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  const int64_t m = M < 1 ? 1 : M;
  Plan pl;
  st = make_plan(m, K, N,
                 fp8_uses_decode(m, N, *d) ? SWIGLU_VARIANT_SMALL_M : SWIGLU_VARIANT_LARGE_M_PAIR, d,
                 &pl, 1);
  if (st != SWIGLU_OK) return st;
  format_plan(pl, *d, "fp8 ", buf, buflen);
  return SWIGLU_OK;
}

swiglu_status_t swiglu_forward_noalloc(const void* A, const void* Wpacked, void* Y, int64_t M,
                                       int64_t K, int64_t N, uint32_t* status_out,
                                       swiglu_stream_t stream) {
  swiglu_status_t st = check_forward_args(A, Wpacked, Y, M, K, N);
  if (st != SWIGLU_OK) return st;
  if (M > 256) return SWIGLU_ERR_UNSUPPORTED;  // the decode kernel's limit
  if (swg::kStatusWords > swg::kStaticScratchWords) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0) {
    if (status_out) std::memset(status_out, 0, swg::kStatusWords * sizeof(uint32_t));
    return SWIGLU_OK;
  }
  NoAllocState* s = nullptr;
  st = noalloc_state(&s);
  if (st != SWIGLU_OK) return st;
  Plan pl;
  st = make_plan(M, K, N, SWIGLU_VARIANT_SMALL_M, nullptr, &pl);
  if (st != SWIGLU_OK) return st;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // The shared array keeps the previous call's record: the status must start at zero.
  if (cudaMemsetAsync(s->scratch, 0, swg::kStatusWords * sizeof(uint32_t), cs) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  swg::SmallMParams p{};
  if (!encode_2d(&p.tmap_x, A, K, M, K * 2, swg::kBlockK, pl.mt, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_packed_w(&p.tmap_w, Wpacked, K, N, 2 * swg::kPackBlockN))
    return SWIGLU_ERR_CUDA;
  p.y = Y;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.mt = pl.mt;
  p.stages = pl.stages;
  p.grid = pl.grid;
  p.splits = pl.splits;    // 1: no SM count, so no K split over clusters
  p.mgroups = pl.mgroups;  // 1: one CTA per column block holds all M tokens
  p.status = s->scratch;
  p.timeout_ns = g_timeout_ns.load();
  p.inject_stall = g_inject.load();
  if (swg::launch_small_m(p, cs) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  if (status_out && cudaMemcpyAsync(status_out, s->scratch, swg::kStatusWords * sizeof(uint32_t),
                                    cudaMemcpyDeviceToHost, cs) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

size_t swiglu_packed_weight_bytes_fp8(int64_t K, int64_t N) {
  if (K <= 0 || N <= 0 || K > kMaxKN || N > kMaxKN) return 0;
  return size_t(2) * size_t(padded_n(N)) * size_t(k_slices8(K) * swg::kBlockK8);
}

swiglu_status_t swiglu_pack_weights_fp8(const void* W1, const void* W2, void* Wpacked, int64_t K,
                                        int64_t N, swiglu_stream_t stream) {
  swiglu_status_t st = check_shape(0, K, N);
  if (st != SWIGLU_OK) return st;
  if ((K % 16) != 0) return SWIGLU_ERR_UNSUPPORTED;  // 16-byte rows of one-byte values
  if (!W1 || !W2 || !Wpacked) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(W1) || !aligned16(W2) || !aligned16(Wpacked)) return SWIGLU_ERR_INVALID_ARG;
  const size_t w_bytes = size_t(K) * size_t(N);
  const size_t p_bytes = swiglu_packed_weight_bytes_fp8(K, N);
  if (overlaps(Wpacked, p_bytes, W1, w_bytes) || overlaps(Wpacked, p_bytes, W2, w_bytes))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  if (swg::launch_pack_fp8(W1, W2, Wpacked, static_cast<int>(K), static_cast<int>(N),
                           reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

swiglu_status_t swiglu_forward_fp8(const void* A, const void* Wpacked, void* Y, int64_t M,
                                   int64_t K, int64_t N, float scale_a, float scale_w1,
                                   float scale_w2, swiglu_stream_t stream) {
  swiglu_status_t st = check_shape(M, K, N);
  if (st != SWIGLU_OK) return st;
  if ((K % 16) != 0) return SWIGLU_ERR_UNSUPPORTED;
  if (!std::isfinite(scale_a) || !std::isfinite(scale_w1) || !std::isfinite(scale_w2))
    return SWIGLU_ERR_INVALID_ARG;
  if (M == 0) return SWIGLU_OK;
  if (!A || !Wpacked || !Y) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Wpacked) || !aligned16(Y)) return SWIGLU_ERR_INVALID_ARG;
  const size_t a_bytes = size_t(M) * size_t(K), y_bytes = size_t(M) * size_t(N) * 2;
  if (overlaps(Y, y_bytes, A, a_bytes) ||
      overlaps(Y, y_bytes, Wpacked, swiglu_packed_weight_bytes_fp8(K, N)))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  // As for bf16: the decode kernel for up to 32 tokens, up to 64 on narrow N,
  // up to 80 when each column block has its own SM; CTA pairs otherwise (the
  // two FP8 kernels).
  Plan pl;
  const int64_t nb = padded_n(N) / swg::kPackBlockN;
  const bool small = fp8_uses_decode(M, N, *d);
  st = make_plan(M, K, N, small ? SWIGLU_VARIANT_SMALL_M : SWIGLU_VARIANT_LARGE_M_PAIR, d, &pl, 1);
  if (st != SWIGLU_OK) return st;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const float sg = scale_a * scale_w1, su = scale_a * scale_w2;
  cudaError_t err;
  if (small) {
    swg::SmallMParams p{};
    if (!encode_2d(&p.tmap_x, A, K, M, K, swg::kBlockK8, pl.mt, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
        !encode_packed_w8(&p.tmap_w, Wpacked, K, N, 2 * swg::kPackBlockN))
      return SWIGLU_ERR_CUDA;
    p.y = Y;
    p.M = static_cast<int>(M);
    p.K = static_cast<int>(K);
    p.N = static_cast<int>(N);
    p.mt = pl.mt;
    p.stages = pl.stages;
    p.grid = pl.grid;
    p.splits = pl.splits;
    p.mgroups = pl.mgroups;
    p.fp8 = 1;
    p.scale_gate = sg;
    p.scale_up = su;
    p.status = d->status;
    p.timeout_ns = g_timeout_ns.load();
    p.inject_stall = g_inject.load();
    err = swg::launch_small_m(p, cs);
  } else {
    swg::LargeMParams p{};
    if (!encode_2d(&p.tmap_a, A, K, M, K, swg::kBlockK8, swg::kTileM, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
        !encode_packed_w8(&p.tmap_w, Wpacked, K, N, pl.bn) ||
        !encode_2d(&p.tmap_y, Y, N, M, N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return SWIGLU_ERR_CUDA;
    p.M = static_cast<int>(M);
    p.K = static_cast<int>(K);
    p.N = static_cast<int>(N);
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.group_m = pl.group_m;
    p.bn = pl.bn;
    p.grid = pl.grid;
    p.fp8 = 1;
    p.scale_gate = sg;
    p.scale_up = su;
    p.status = d->status;
    p.timeout_ns = g_timeout_ns.load();
    p.inject_stall = g_inject.load();
    err = swg::launch_large_m_pair(p, cs);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

size_t swiglu_packed_weight_bytes_mxfp8(int64_t K, int64_t N) {
  const size_t values = swiglu_packed_weight_bytes_fp8(K, N);
  if (values == 0) return 0;
  return values + mx_weight_scale_bytes(K, N);
}

size_t swiglu_act_scale_bytes_mxfp8(int64_t M, int64_t K) {
  if (M < 0 || K <= 0 || M > kMaxM || K > kMaxKN) return 0;
  return size_t((M + 127) / 128) * size_t(k_slices8(K)) * swg::kSfBlockBytes;
}

swiglu_status_t swiglu_pack_weights_mxfp8(const void* W1, const void* S1, const void* W2,
                                          const void* S2, void* Wpacked, int64_t K, int64_t N,
                                          swiglu_stream_t stream) {
  swiglu_status_t st = check_shape(0, K, N);
  if (st != SWIGLU_OK) return st;
  if ((K % swg::kMxGroup) != 0) return SWIGLU_ERR_UNSUPPORTED;  // whole scale groups
  if (!W1 || !W2 || !S1 || !S2 || !Wpacked) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(W1) || !aligned16(W2) || !aligned16(Wpacked)) return SWIGLU_ERR_INVALID_ARG;
  const size_t w_bytes = size_t(K) * size_t(N), s_bytes = size_t(K / swg::kMxGroup) * size_t(N);
  const size_t p_bytes = swiglu_packed_weight_bytes_mxfp8(K, N);
  if (overlaps(Wpacked, p_bytes, W1, w_bytes) || overlaps(Wpacked, p_bytes, W2, w_bytes) ||
      overlaps(Wpacked, p_bytes, S1, s_bytes) || overlaps(Wpacked, p_bytes, S2, s_bytes))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* scales = static_cast<uint8_t*>(Wpacked) + swiglu_packed_weight_bytes_fp8(K, N);
  if (swg::launch_pack_fp8(W1, W2, Wpacked, static_cast<int>(K), static_cast<int>(N), cs) !=
          cudaSuccess ||
      swg::launch_pack_mx_weight_scales(S1, S2, scales, static_cast<int>(K), static_cast<int>(N),
                                        cs) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

swiglu_status_t swiglu_pack_act_scales_mxfp8(const void* SA, void* SAtiled, int64_t M, int64_t K,
                                             swiglu_stream_t stream) {
  swiglu_status_t st = check_shape(M, K, 8);
  if (st != SWIGLU_OK) return st;
  if ((K % swg::kMxGroup) != 0) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0) return SWIGLU_OK;
  if (!SA || !SAtiled || !aligned16(SAtiled)) return SWIGLU_ERR_INVALID_ARG;
  if (overlaps(SAtiled, swiglu_act_scale_bytes_mxfp8(M, K), SA,
               size_t(M) * size_t(K / swg::kMxGroup)))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  if (swg::launch_tile_mx_act_scales(SA, SAtiled, static_cast<int>(M), static_cast<int>(K),
                                     reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

swiglu_status_t swiglu_plan_string_mxfp8(int64_t M, int64_t K, int64_t N, char* buf,
                                         size_t buflen) {
  if (!buf || buflen == 0) return SWIGLU_ERR_INVALID_ARG;
  buf[0] = '\0';
  swiglu_status_t st = check_shape(M, K, N);
  if (st != SWIGLU_OK) return st;
  if ((K % swg::kMxGroup) != 0) return SWIGLU_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  Plan pl;
  st = make_mx_plan(M < 1 ? 1 : M, K, N, *d, &pl);
  if (st != SWIGLU_OK) return st;
  format_plan(pl, *d, "mxfp8 ", buf, buflen);
  return SWIGLU_OK;
}

swiglu_status_t swiglu_forward_mxfp8(const void* A, const void* SAtiled, const void* Wpacked,
                                     void* Y, int64_t M, int64_t K, int64_t N,
                                     swiglu_stream_t stream) {
  swiglu_status_t st = check_shape(M, K, N);
  if (st != SWIGLU_OK) return st;
  if ((K % swg::kMxGroup) != 0) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0) return SWIGLU_OK;
  if (!A || !SAtiled || !Wpacked || !Y) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(SAtiled) || !aligned16(Wpacked) || !aligned16(Y))
    return SWIGLU_ERR_INVALID_ARG;
  const size_t a_bytes = size_t(M) * size_t(K), y_bytes = size_t(M) * size_t(N) * 2;
  if (overlaps(Y, y_bytes, A, a_bytes) ||
      overlaps(Y, y_bytes, Wpacked, swiglu_packed_weight_bytes_mxfp8(K, N)) ||
      overlaps(Y, y_bytes, SAtiled, swiglu_act_scale_bytes_mxfp8(M, K)))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  Plan pl;
  st = make_mx_plan(M, K, N, *d, &pl);
  if (st != SWIGLU_OK) return st;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // scale tensors as rows of 256 bytes: 4 rows per packed weight tile, 2 rows
  // per activation block of 128 rows x one 128-deep K slice
  const uint8_t* wscales = static_cast<const uint8_t*>(Wpacked) + swiglu_packed_weight_bytes_fp8(K, N);
  const uint64_t w_rows = uint64_t(padded_n(N) / swg::kPackBlockN) * uint64_t(k_slices8(K)) * 4;
  const uint64_t a_rows = uint64_t((M + 127) / 128) * uint64_t(k_slices8(K)) * 2;
  CUtensorMap tmap_sw, tmap_sa;
  if (!encode_2d(&tmap_sw, wscales, 256, w_rows, 256, 256, 4, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
      !encode_2d(&tmap_sa, SAtiled, 256, a_rows, 256, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_DATA_TYPE_UINT8))
    return SWIGLU_ERR_CUDA;
  cudaError_t err;
  if (pl.variant == SWIGLU_VARIANT_SMALL_M) {
    swg::SmallMParams p{};
    if (!encode_2d(&p.tmap_x, A, K, M, K, swg::kBlockK8, pl.mt, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
        !encode_packed_w8(&p.tmap_w, Wpacked, K, N, 2 * swg::kPackBlockN))
      return SWIGLU_ERR_CUDA;
    p.tmap_sw = tmap_sw;
    p.tmap_sa = tmap_sa;
    p.y = Y;
    p.M = static_cast<int>(M);
    p.K = static_cast<int>(K);
    p.N = static_cast<int>(N);
    p.mt = pl.mt;
    p.stages = pl.stages;
    p.grid = pl.grid;
    p.splits = pl.splits;
    p.mgroups = pl.mgroups;
    p.fp8 = 1;
    p.mx = 1;
    p.scale_gate = 1.0f;  // the scales act inside the MMA
    p.scale_up = 1.0f;
    p.status = d->status;
    p.timeout_ns = g_timeout_ns.load();
    p.inject_stall = g_inject.load();
    err = swg::launch_small_m(p, cs);
  } else {
    swg::LargeMParams p{};
    if (!encode_2d(&p.tmap_a, A, K, M, K, swg::kBlockK8, swg::kTileM, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
        !encode_packed_w8(&p.tmap_w, Wpacked, K, N, pl.bn) ||
        !encode_2d(&p.tmap_y, Y, N, M, N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return SWIGLU_ERR_CUDA;
    p.tmap_sw = tmap_sw;
    p.tmap_sa = tmap_sa;
    p.M = static_cast<int>(M);
    p.K = static_cast<int>(K);
    p.N = static_cast<int>(N);
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.group_m = pl.group_m;
    p.bn = pl.bn;
    p.grid = pl.grid;
    p.fp8 = 1;
    p.mx = 1;
    p.scale_gate = 1.0f;
    p.scale_up = 1.0f;
    p.status = d->status;
    p.timeout_ns = g_timeout_ns.load();
    p.inject_stall = g_inject.load();
    err = swg::launch_large_m_pair(p, cs);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

size_t swiglu_down_packed_bytes(int64_t N, int64_t H) {
  if (N <= 0 || H <= 0 || N > kMaxKN || H > kMaxKN) return 0;
  return size_t(padded_h(H)) * size_t(k_slices(N) * swg::kBlockK) * 2;
}

swiglu_status_t swiglu_pack_down_weights(const void* W3, void* W3packed, int64_t N, int64_t H,
                                         swiglu_stream_t stream) {
  swiglu_status_t st = check_shape(0, N, H);
  if (st != SWIGLU_OK) return st;
  if (!W3 || !W3packed) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(W3) || !aligned16(W3packed)) return SWIGLU_ERR_INVALID_ARG;
  if (overlaps(W3packed, swiglu_down_packed_bytes(N, H), W3, size_t(N) * size_t(H) * 2))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  if (swg::launch_pack_down(W3, W3packed, static_cast<int>(N), static_cast<int>(H),
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

static swiglu_status_t down_plan_string(int64_t M, int64_t N, int64_t H, bool cross_cluster,
                                        char* buf, size_t buflen) {
  if (!buf || buflen == 0) return SWIGLU_ERR_INVALID_ARG;
  buf[0] = '\0';
  swiglu_status_t st = check_shape(M, N, H);
  if (st != SWIGLU_OK) return st;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  DownPlan dp;
  st = make_down_plan(M < 1 ? 1 : M, N, H, d, &dp, cross_cluster);
  if (st != SWIGLU_OK) return st;
  if (dp.decode)
    std::snprintf(buf, buflen,
                  "down small_m mt=%d stages=%d blocks=%lld groups=%d splits=%d clusters=%d grid=%d "
                  "sms=%d",
                  dp.mt, dp.stages, static_cast<long long>(dp.blocks), dp.mgroups, dp.splits,
                  dp.gsplits, dp.grid, d->sm_count);
  else
    std::snprintf(buf, buflen, "down large_m_pair tiles=%lld group_m=%lld grid=%d max_pairs=%d sms=%d",
                  static_cast<long long>(dp.tiles), static_cast<long long>(dp.group), dp.grid,
                  d->max_pairs, d->sm_count);
  return SWIGLU_OK;
}

swiglu_status_t swiglu_down_plan_string(int64_t M, int64_t N, int64_t H, char* buf,
                                        size_t buflen) {
  return down_plan_string(M, N, H, false, buf, buflen);
}

swiglu_status_t swiglu_down_plan_string_ws(int64_t M, int64_t N, int64_t H, char* buf,
                                           size_t buflen) {
  return down_plan_string(M, N, H, true, buf, buflen);
}

size_t swiglu_down_workspace_bytes(int64_t M, int64_t N, int64_t H) {
  if (check_shape(M, N, H) != SWIGLU_OK || M == 0) return 0;
  DeviceState* d = nullptr;
  if (device_state(&d) != SWIGLU_OK) return 0;
  DownPlan dp;
  if (make_down_plan(M, N, H, d, &dp, true) != SWIGLU_OK) return 0;
  return down_workspace_bytes(dp);
}

static swiglu_status_t down_forward(const void* Y, const void* W3packed, const void* R, void* Out,
                                    int64_t M, int64_t N, int64_t H, void* workspace,
                                    size_t workspace_bytes, swiglu_stream_t stream) {
  swiglu_status_t st = check_shape(M, N, H);
  if (st != SWIGLU_OK) return st;
  if (M == 0) return SWIGLU_OK;
  if (!Y || !W3packed || !Out) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(Y) || !aligned16(W3packed) || !aligned16(Out) || (R && !aligned16(R)))
    return SWIGLU_ERR_INVALID_ARG;
  const size_t y_bytes = size_t(M) * size_t(N) * 2, o_bytes = size_t(M) * size_t(H) * 2;
  if (overlaps(Out, o_bytes, Y, y_bytes) ||
      overlaps(Out, o_bytes, W3packed, swiglu_down_packed_bytes(N, H)) ||
      (R && R != Out && overlaps(Out, o_bytes, R, o_bytes)))  // Out == R (in place) is allowed
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  DownPlan dp;
  st = make_down_plan(M, N, H, d, &dp, workspace != nullptr);
  if (st != SWIGLU_OK) return st;
  const size_t ws_bytes = down_workspace_bytes(dp);
  if (ws_bytes > 0) {  // the plan splits K across clusters: the workspace must hold it
    if (workspace_bytes < ws_bytes || !aligned16(workspace) ||
        overlaps(workspace, ws_bytes, Out, size_t(M) * size_t(H) * 2) ||
        overlaps(workspace, ws_bytes, Y, size_t(M) * size_t(N) * 2) ||
        overlaps(workspace, ws_bytes, W3packed, swiglu_down_packed_bytes(N, H)) ||
        (R && overlaps(workspace, ws_bytes, R, size_t(M) * size_t(H) * 2)))
      return SWIGLU_ERR_INVALID_ARG;
  }
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (dp.decode) {
    // decode: weights as the MMA M side, K split over clusters when blocks are few
    swg::SmallMParams p{};
    p.mt = dp.mt;
    p.mgroups = dp.mgroups;
    p.stages = dp.stages;
    p.splits = dp.splits;
    p.gsplits = dp.gsplits;
    if (ws_bytes > 0) {  // counters first, then the partials (256-byte aligned)
      const size_t units = size_t(dp.blocks) * size_t(dp.mgroups);
      p.counters = static_cast<uint32_t*>(workspace);
      p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                      (units * size_t(dp.splits) * 4 + 255) / 256 * 256);
    }
    if (!encode_2d(&p.tmap_x, Y, N, M, N * 2, swg::kBlockK, p.mt, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_packed_down(&p.tmap_w, W3packed, N, H, 256))
      return SWIGLU_ERR_CUDA;
    p.y = Out;
    p.residual = R;
    p.down = 1;
    p.M = static_cast<int>(M);
    p.K = static_cast<int>(N);
    p.N = static_cast<int>(H);
    p.grid = dp.grid;
    p.status = d->status;
    p.timeout_ns = g_timeout_ns.load();
    p.inject_stall = g_inject.load();
    err = swg::launch_small_m(p, cs);
  } else {
    swg::LargeMParams p{};
    if (!encode_2d(&p.tmap_a, Y, N, M, N * 2, swg::kBlockK, swg::kTileM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_packed_down(&p.tmap_w, W3packed, N, H, swg::kPackBlockN) ||
        !encode_2d(&p.tmap_y, Out, H, M, H * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return SWIGLU_ERR_CUDA;
    p.M = static_cast<int>(M);
    p.K = static_cast<int>(N);
    p.N = static_cast<int>(H);
    p.tiles_m = static_cast<int>(dp.pm);
    p.tiles_n = static_cast<int>(dp.blocks);
    p.group_m = static_cast<int>(dp.group);
    p.bn = swg::kPackBlockN;
    p.grid = dp.grid;
    p.down = 1;
    p.residual = R;
    p.status = d->status;
    p.timeout_ns = g_timeout_ns.load();
    p.inject_stall = g_inject.load();
    err = swg::launch_large_m_pair(p, cs);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

swiglu_status_t swiglu_down_forward(const void* Y, const void* W3packed, const void* R, void* Out,
                                    int64_t M, int64_t N, int64_t H, swiglu_stream_t stream) {
  return down_forward(Y, W3packed, R, Out, M, N, H, nullptr, 0, stream);
}

swiglu_status_t swiglu_down_forward_ws(const void* Y, const void* W3packed, const void* R,
                                       void* Out, int64_t M, int64_t N, int64_t H,
                                       void* workspace, size_t workspace_bytes,
                                       swiglu_stream_t stream) {
  return down_forward(Y, W3packed, R, Out, M, N, H, workspace, workspace_bytes, stream);
}

void swiglu_testing_inject_stall(int enable, uint32_t timeout_ms) {
  g_inject.store(enable ? 1 : 0);
  if (timeout_ms) g_timeout_ns.store(uint64_t(timeout_ms) * 1000000ull);
}

swiglu_status_t swiglu_testing_pace_run_out(uint64_t* count) {
  if (!count) return SWIGLU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  swiglu_status_t st = device_state(&d);
  if (st != SWIGLU_OK) return st;
  unsigned long long v = 0;
  if (swg::large_m_pair_pace_run_out(&v) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  *count = static_cast<uint64_t>(v);
  return SWIGLU_OK;
}

}  // extern "C"
