// noreduce.cu -- the timing stand-in that domino_debug_skip_reduce puts in place of the shard-sum,
// so that a step without the reduction can be timed against the normal one.
#include "kernels.h"

namespace dm {

// Timing stand-in for the shard-sum (domino_debug_skip_reduce): the same grid, and no reduction.
// With a residual (layer stacks) the residual is copied into Y, so the layers after it still see
// activations of the usual size and the GEMMs draw their usual power; without one it returns at
// once and Y keeps whatever it held.
__global__ void __launch_bounds__(256) noreduce_kernel(uint32_t vecs_per_row, uint32_t total_vecs,
                                                       const uint16_t* __restrict__ res, int64_t ld_res,
                                                       uint16_t* __restrict__ Y, int64_t ld_y) {
  if (!res) return;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < total_vecs; v += stride) {
    const uint32_t r = v / vecs_per_row;
    const uint32_t c = (v - r * vecs_per_row) * 8u;
    *reinterpret_cast<uint4*>(Y + static_cast<int64_t>(r) * ld_y + c) =
        *reinterpret_cast<const uint4*>(res + static_cast<int64_t>(r) * ld_res + c);
  }
}

cudaError_t launch_noreduce(int64_t rows, int64_t cols, const uint16_t* res, int64_t ld_res, uint16_t* Y,
                            int64_t ld_y, int grid_cap, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const uint32_t vpr = static_cast<uint32_t>(cols / 8);
  const uint32_t total = static_cast<uint32_t>(rows) * vpr;
  const int threads = 256;
  int grid = static_cast<int>((total + threads - 1) / threads);
  if (grid > grid_cap) grid = grid_cap;
  noreduce_kernel<<<grid, threads, 0, st>>>(vpr, total, res, ld_res, Y, ld_y);
  return cudaGetLastError();
}

}  // namespace dm
