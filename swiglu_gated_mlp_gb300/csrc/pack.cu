// Packs W1, W2 [K, N] (N contiguous) into the tile-major, block-interleaved
// weight the fused kernels stream. Viewed as bf16 [Np/128][Kp/64][256][64]:
//   Wp[j][b][i][t]       = W1[64b + t][128j + i]   (i < 128, gate)
//   Wp[j][b][128 + i][t] = W2[64b + t][128j + i]   (i < 128, up)
// zero where a column is >= N or a K index is >= K. Every [256][64] tile (32 KB)
// is contiguous, so each TMA box the kernels load is one contiguous span of
// memory. The pages fuse W1 and W2 into one K x 2N matrix ahead of time
// ("Tile-Level Activation Overlap for Efficient LLM Inference", gist.science,
// section "Methodology / Kernel-2"); this is that step, with 128-column blocks
// instead of single-column interleave. It runs once per weight set: one CTA
// per tile, a transpose through shared memory.
#include "kernels.h"

namespace swg {
namespace {

constexpr int kTileRows = 2 * kPackBlockN;  // 256 packed rows: gate block, then up block

__global__ void __launch_bounds__(256)
    pack_kernel(const uint16_t* __restrict__ w1, const uint16_t* __restrict__ w2,
                uint16_t* __restrict__ wp, int K, int N, int k_slices) {
  __shared__ uint16_t tile[kBlockK][kTileRows + 2];  // [t][i]; +2 keeps the column reads conflict-free
  const int b = blockIdx.x;                           // K slice
  const int j = blockIdx.y;                           // column block
  const int k0 = b * kBlockK, n0 = j * kPackBlockN;
  // load: for each k, 128 consecutive columns of W1 then of W2 (coalesced)
  for (int idx = threadIdx.x; idx < kBlockK * kTileRows; idx += blockDim.x) {
    const int t = idx / kTileRows, i = idx % kTileRows;
    const int k = k0 + t, n = n0 + (i % kPackBlockN);
    const uint16_t* __restrict__ src = i < kPackBlockN ? w1 : w2;
    tile[t][i] = (k < K && n < N) ? src[static_cast<size_t>(k) * N + n] : uint16_t(0);
  }
  __syncthreads();
  // store: the tile's 256 rows of 64 K values, contiguous
  uint16_t* __restrict__ out =
      wp + (static_cast<size_t>(j) * k_slices + b) * (static_cast<size_t>(kTileRows) * kBlockK);
  for (int idx = threadIdx.x; idx < kBlockK * kTileRows; idx += blockDim.x) {
    const int i = idx / kBlockK, t = idx % kBlockK;
    out[idx] = tile[t][i];
  }
}

}  // namespace

cudaError_t launch_pack(const void* w1, const void* w2, void* wp, int K, int N,
                        cudaStream_t stream) {
  const int n_blocks = (N + kPackBlockN - 1) / kPackBlockN;
  const int k_slices = (K + kBlockK - 1) / kBlockK;
  const dim3 grid(k_slices, n_blocks);
  pack_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(w1),
                                        static_cast<const uint16_t*>(w2),
                                        static_cast<uint16_t*>(wp), K, N, k_slices);
  return cudaGetLastError();
}

}  // namespace swg
