// Packs W1, W2 [K, N] (N contiguous) into the tile-major, block-interleaved
// weight the fused kernels stream. For bf16 elements, viewed as
// [Np/128][Kp/64][256][64]; for FP8 (one byte) as [Np/128][Kp/128][256][128]:
//   Wp[j][b][i][t]       = W1[S b + t][128j + i]   (i < 128, gate)
//   Wp[j][b][128 + i][t] = W2[S b + t][128j + i]   (i < 128, up)
// with S = 64 or 128 values per K slice (a row is 128 bytes either way), zero
// where a column is >= N or a K index is >= K. Every [256][S] tile (32 KB)
// is contiguous, so each TMA box the kernels load is one contiguous span of
// memory. The pages fuse W1 and W2 into one K x 2N matrix ahead of time
// ("Tile-Level Activation Overlap for Efficient LLM Inference", gist.science,
// section "Methodology / Kernel-2"); this is that step, with 128-column blocks
// instead of single-column interleave. It runs once per weight set: one CTA
// per tile, a transpose through shared memory; the bits are copied unchanged.
#include "kernels.h"

namespace swg {
namespace {

constexpr int kTileRows = 2 * kPackBlockN;  // 256 packed rows: gate block, then up block

template <typename T, int S>
__global__ void __launch_bounds__(256)
    pack_kernel(const T* __restrict__ w1, const T* __restrict__ w2, T* __restrict__ wp, int K,
                int N, int k_slices) {
  // [t][i]; the padding keeps the column reads conflict-free
  __shared__ T tile[S][kTileRows + 4 / sizeof(T)];
  const int b = blockIdx.x;  // K slice
  const int j = blockIdx.y;  // column block
  const int k0 = b * S, n0 = j * kPackBlockN;
  // load: for each k, 128 consecutive columns of W1 then of W2 (coalesced)
  for (int idx = threadIdx.x; idx < S * kTileRows; idx += blockDim.x) {
    const int t = idx / kTileRows, i = idx % kTileRows;
    const int k = k0 + t, n = n0 + (i % kPackBlockN);
    const T* __restrict__ src = i < kPackBlockN ? w1 : w2;
    tile[t][i] = (k < K && n < N) ? src[static_cast<size_t>(k) * N + n] : T(0);
  }
  __syncthreads();
  // store: the tile's 256 rows of S K values, contiguous
  T* __restrict__ out =
      wp + (static_cast<size_t>(j) * k_slices + b) * (static_cast<size_t>(kTileRows) * S);
  for (int idx = threadIdx.x; idx < S * kTileRows; idx += blockDim.x) {
    const int i = idx / S, t = idx % S;
    out[idx] = tile[t][i];
  }
}

// Down-projection weight W3 [N, H] (H contiguous) -> [Hp/256][Np/64][256][64]:
// tile (j, b) row i is output column 256 j + i over K values 64 b .. 64 b + 63.
__global__ void __launch_bounds__(256)
    pack_down_kernel(const uint16_t* __restrict__ w3, uint16_t* __restrict__ wp, int N, int H,
                     int k_slices) {
  __shared__ uint16_t tile[kBlockK][kTileRows + 2];
  const int b = blockIdx.x;  // K slice (rows of W3)
  const int j = blockIdx.y;  // 256-column block of the output
  const int k0 = b * kBlockK, h0 = j * kTileRows;
  for (int idx = threadIdx.x; idx < kBlockK * kTileRows; idx += blockDim.x) {
    const int t = idx / kTileRows, i = idx % kTileRows;
    const int k = k0 + t, h = h0 + i;
    tile[t][i] = (k < N && h < H) ? w3[static_cast<size_t>(k) * H + h] : uint16_t(0);
  }
  __syncthreads();
  uint16_t* __restrict__ out =
      wp + (static_cast<size_t>(j) * k_slices + b) * (static_cast<size_t>(kTileRows) * kBlockK);
  for (int idx = threadIdx.x; idx < kBlockK * kTileRows; idx += blockDim.x) {
    const int i = idx / kBlockK, t = idx % kBlockK;
    out[idx] = tile[t][i];
  }
}

// Scales of block-scaled FP8 (one byte per 32 K values) in 512-byte blocks
// of 128 rows x 4 groups: row r, group g at (r % 32) * 16 + (r / 32) * 4 + g;
// 127 (a scale of 1) where no value exists.
__device__ __forceinline__ int sf_offset(int r, int g) { return (r & 31) * 16 + (r >> 5) * 4 + g; }

// W1's and W2's scales [groups, N] -> per packed tile (column block j, K slice
// b): W1's block for columns 128 j + r, groups 4 b + g, then W2's block.
__global__ void __launch_bounds__(256)
    pack_mx_weight_scales_kernel(const uint8_t* __restrict__ s1, const uint8_t* __restrict__ s2,
                                 uint8_t* __restrict__ out, int groups, int N, int k_slices) {
  const int b = blockIdx.x, j = blockIdx.y;
  uint8_t* __restrict__ dst = out + (static_cast<size_t>(j) * k_slices + b) * (2 * kSfBlockBytes);
  for (int idx = threadIdx.x; idx < 2 * kSfBlockBytes; idx += blockDim.x) {
    const int h = idx / kSfBlockBytes, r = (idx % kSfBlockBytes) >> 2, g = idx & 3;
    const int n = j * kPackBlockN + r, kg = b * 4 + g;
    const uint8_t* __restrict__ src = h ? s2 : s1;
    dst[h * kSfBlockBytes + sf_offset(r, g)] =
        (n < N && kg < groups) ? src[static_cast<size_t>(kg) * N + n] : uint8_t(127);
  }
}

// A's scales [M, groups] -> blocks [ceil(M/128)][k_slices]; grid (row blocks, K slices).
__global__ void __launch_bounds__(256)
    tile_mx_act_scales_kernel(const uint8_t* __restrict__ sa, uint8_t* __restrict__ out, int M,
                              int groups, int k_slices) {
  const int i = blockIdx.x, b = blockIdx.y;
  uint8_t* __restrict__ dst = out + (static_cast<size_t>(i) * k_slices + b) * kSfBlockBytes;
  for (int idx = threadIdx.x; idx < kSfBlockBytes; idx += blockDim.x) {
    const int r = idx >> 2, g = idx & 3;
    const int m = i * 128 + r, kg = b * 4 + g;
    dst[sf_offset(r, g)] =
        (m < M && kg < groups) ? sa[static_cast<size_t>(m) * groups + kg] : uint8_t(127);
  }
}

}  // namespace

cudaError_t launch_pack_down(const void* w3, void* wp, int N, int H, cudaStream_t stream) {
  const int blocks = (H + kTileRows - 1) / kTileRows;
  const int k_slices = (N + kBlockK - 1) / kBlockK;
  pack_down_kernel<<<dim3(k_slices, blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(w3), static_cast<uint16_t*>(wp), N, H, k_slices);
  return cudaGetLastError();
}

cudaError_t launch_pack(const void* w1, const void* w2, void* wp, int K, int N,
                        cudaStream_t stream) {
  const int n_blocks = (N + kPackBlockN - 1) / kPackBlockN;
  const int k_slices = (K + kBlockK - 1) / kBlockK;
  const dim3 grid(k_slices, n_blocks);
  pack_kernel<uint16_t, kBlockK><<<grid, 256, 0, stream>>>(
      static_cast<const uint16_t*>(w1), static_cast<const uint16_t*>(w2),
      static_cast<uint16_t*>(wp), K, N, k_slices);
  return cudaGetLastError();
}

cudaError_t launch_pack_fp8(const void* w1, const void* w2, void* wp, int K, int N,
                            cudaStream_t stream) {
  const int n_blocks = (N + kPackBlockN - 1) / kPackBlockN;
  const int k_slices = (K + kBlockK8 - 1) / kBlockK8;
  const dim3 grid(k_slices, n_blocks);
  pack_kernel<uint8_t, kBlockK8><<<grid, 256, 0, stream>>>(
      static_cast<const uint8_t*>(w1), static_cast<const uint8_t*>(w2),
      static_cast<uint8_t*>(wp), K, N, k_slices);
  return cudaGetLastError();
}

cudaError_t launch_pack_mx_weight_scales(const void* s1, const void* s2, void* out, int K, int N,
                                         cudaStream_t stream) {
  const int n_blocks = (N + kPackBlockN - 1) / kPackBlockN;
  const int k_slices = (K + kBlockK8 - 1) / kBlockK8;
  pack_mx_weight_scales_kernel<<<dim3(k_slices, n_blocks), 256, 0, stream>>>(
      static_cast<const uint8_t*>(s1), static_cast<const uint8_t*>(s2), static_cast<uint8_t*>(out),
      (K + kMxGroup - 1) / kMxGroup, N, k_slices);
  return cudaGetLastError();
}

cudaError_t launch_tile_mx_act_scales(const void* sa, void* out, int M, int K,
                                      cudaStream_t stream) {
  const int m_blocks = static_cast<int>((static_cast<int64_t>(M) + 127) / 128);  // M up to 2^31 - 1
  const int k_slices = (K + kBlockK8 - 1) / kBlockK8;
  tile_mx_act_scales_kernel<<<dim3(m_blocks, k_slices), 256, 0, stream>>>(
      static_cast<const uint8_t*>(sa), static_cast<uint8_t*>(out), M, (K + kMxGroup - 1) / kMxGroup,
      k_slices);
  return cudaGetLastError();
}

}  // namespace swg
