// Packs W1, W2 [K, N] (N contiguous) into the K-contiguous block-interleaved
// weight the fused kernels stream:
//   Wp[j][i][k] = W1[k][j*128 + i],  Wp[j][128 + i][k] = W2[k][j*128 + i],
// zero for columns >= N. The pages fuse W1 and W2 into one K x 2N matrix ahead
// of time ("Tile-Level Activation Overlap for Efficient LLM Inference",
// gist.science, section "Methodology / Kernel-2"); this is that step, with
// 128-column blocks instead of single-column interleave. It runs once per
// weight set and is a plain tiled transpose through shared memory.
#include "kernels.h"

namespace swg {
namespace {

constexpr int kTile = 64;

__global__ void __launch_bounds__(256)
    pack_kernel(const uint16_t* __restrict__ w1, const uint16_t* __restrict__ w2,
                uint16_t* __restrict__ wp, int K, int N, int Np) {
  __shared__ uint16_t tile[kTile][kTile + 2];
  const int which = blockIdx.z;  // 0: W1 -> gate rows, 1: W2 -> up rows
  const uint16_t* __restrict__ w = which ? w2 : w1;
  const int k0 = blockIdx.x * kTile;
  const int n0 = blockIdx.y * kTile;
  const int tx = threadIdx.x & (kTile - 1);
  const int ty = threadIdx.x >> 6;  // 0..3
  for (int i = ty; i < kTile; i += 4) {
    const int k = k0 + i, n = n0 + tx;
    tile[i][tx] = (k < K && n < N) ? w[static_cast<size_t>(k) * N + n] : uint16_t(0);
  }
  __syncthreads();
  for (int i = ty; i < kTile; i += 4) {
    const int n = n0 + i, k = k0 + tx;
    if (k < K && n < Np) {
      const size_t row = static_cast<size_t>(n / kPackBlockN) * (2 * kPackBlockN) +
                         static_cast<size_t>(which) * kPackBlockN + (n % kPackBlockN);
      wp[row * K + k] = tile[tx][i];
    }
  }
}

}  // namespace

cudaError_t launch_pack(const void* w1, const void* w2, void* wp, int K, int N,
                        cudaStream_t stream) {
  const int np = (N + kPackBlockN - 1) / kPackBlockN * kPackBlockN;
  const dim3 grid((K + kTile - 1) / kTile, np / kTile, 2);
  pack_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(w1),
                                        static_cast<const uint16_t*>(w2),
                                        static_cast<uint16_t*>(wp), K, N, np);
  return cudaGetLastError();
}

}  // namespace swg
