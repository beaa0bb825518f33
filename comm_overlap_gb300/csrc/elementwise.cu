// elementwise.cu -- HBM-bound kernels: the shard-sum that stands in for the AllReduce of the
// t row-parallel partials, and the pre-LN LayerNorm of the layer stack.
#include <cuda_bf16.h>

#include "actfn.cuh"
#include "kernels.h"

namespace dm {

// Y[r, c] = bf16( res[r, c] + (((P_0 + P_1) + P_2) + ... + P_{t-1})[r, c] ), fp32 sums in fixed
// shard order.  Each thread handles 8 consecutive columns: two 16-byte streaming loads per
// shard, one 16-byte store.  T > 0 fixes the shard count at compile time so that all t loads
// are in flight before the first add; T == 0 loops over a runtime count.
template <int T>
__global__ void __launch_bounds__(256) shard_sum_kernel(const float* __restrict__ P, int t,
                                                        uint32_t vecs_per_row, uint32_t total_vecs,
                                                        int64_t cols, int64_t slice,
                                                        const uint16_t* __restrict__ res,
                                                        int64_t ld_res, uint16_t* __restrict__ Y,
                                                        int64_t ld_y) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < total_vecs; v += stride) {
    const uint32_t r = v / vecs_per_row;
    const uint32_t c = (v - r * vecs_per_row) * 8u;
    const float4* p = reinterpret_cast<const float4*>(P + static_cast<int64_t>(r) * cols + c);
    const int64_t sl4 = slice / 4;
    float acc[8];
    if constexpr (T > 0) {
      float4 lo[T], hi[T];
#pragma unroll
      for (int i = 0; i < T; ++i) {
        lo[i] = __ldcs(p + i * sl4);
        hi[i] = __ldcs(p + i * sl4 + 1);
      }
      acc[0] = lo[0].x; acc[1] = lo[0].y; acc[2] = lo[0].z; acc[3] = lo[0].w;
      acc[4] = hi[0].x; acc[5] = hi[0].y; acc[6] = hi[0].z; acc[7] = hi[0].w;
#pragma unroll
      for (int i = 1; i < T; ++i) {
        acc[0] += lo[i].x; acc[1] += lo[i].y; acc[2] += lo[i].z; acc[3] += lo[i].w;
        acc[4] += hi[i].x; acc[5] += hi[i].y; acc[6] += hi[i].z; acc[7] += hi[i].w;
      }
    } else {
      float4 lo = __ldcs(p), hi = __ldcs(p + 1);
      acc[0] = lo.x; acc[1] = lo.y; acc[2] = lo.z; acc[3] = lo.w;
      acc[4] = hi.x; acc[5] = hi.y; acc[6] = hi.z; acc[7] = hi.w;
      for (int i = 1; i < t; ++i) {
        lo = __ldcs(p + i * sl4);
        hi = __ldcs(p + i * sl4 + 1);
        acc[0] += lo.x; acc[1] += lo.y; acc[2] += lo.z; acc[3] += lo.w;
        acc[4] += hi.x; acc[5] += hi.y; acc[6] += hi.z; acc[7] += hi.w;
      }
    }
    if (res) {
      const uint4 w = *reinterpret_cast<const uint4*>(res + static_cast<int64_t>(r) * ld_res + c);
      // residual first, then the reduced sum: res + sum (one rounding below)
      acc[0] = bf16lo(w.x) + acc[0]; acc[1] = bf16hi(w.x) + acc[1];
      acc[2] = bf16lo(w.y) + acc[2]; acc[3] = bf16hi(w.y) + acc[3];
      acc[4] = bf16lo(w.z) + acc[4]; acc[5] = bf16hi(w.z) + acc[5];
      acc[6] = bf16lo(w.w) + acc[6]; acc[7] = bf16hi(w.w) + acc[7];
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(Y + static_cast<int64_t>(r) * ld_y + c) = o;
  }
}

cudaError_t launch_shard_sum(const float* P, int t, int64_t rows, int64_t cols, const uint16_t* res,
                             int64_t ld_res, uint16_t* Y, int64_t ld_y, int grid_cap,
                             cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const uint32_t vpr = static_cast<uint32_t>(cols / 8);
  const uint32_t total = static_cast<uint32_t>(rows) * vpr;
  const int threads = 256;
  int grid = static_cast<int>((total + threads - 1) / threads);
  if (grid > grid_cap) grid = grid_cap;
  const int64_t slice = rows * cols;
#define DM_SS(TT) \
  shard_sum_kernel<TT><<<grid, threads, 0, st>>>(P, t, vpr, total, cols, slice, res, ld_res, Y, ld_y)
  switch (t) {
    case 1: DM_SS(1); break;
    case 2: DM_SS(2); break;
    case 3: DM_SS(3); break;
    case 4: DM_SS(4); break;
    case 8: DM_SS(8); break;
    default: DM_SS(0); break;
  }
#undef DM_SS
  return cudaGetLastError();
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// LayerNorm without affine parameters, one warp per row: fp32 mean, then fp32 biased
// variance of (z - mean), then (z - mean) * rsqrt(var + eps) rounded to bf16.
__global__ void __launch_bounds__(256) layernorm_kernel(const uint16_t* __restrict__ Z, int64_t rows,
                                                        int64_t h, float eps,
                                                        uint16_t* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (r >= rows) return;
  const uint4* z = reinterpret_cast<const uint4*>(Z + r * h);
  uint4* o = reinterpret_cast<uint4*>(out + r * h);
  const int nv = static_cast<int>(h / 8);
  float s = 0.0f;
  for (int v = lane; v < nv; v += 32) {
    const uint4 w = z[v];
    s += bf16lo(w.x) + bf16hi(w.x) + bf16lo(w.y) + bf16hi(w.y) + bf16lo(w.z) + bf16hi(w.z) +
         bf16lo(w.w) + bf16hi(w.w);
  }
  const float mean = warp_sum(s) / static_cast<float>(h);
  float ss = 0.0f;
  for (int v = lane; v < nv; v += 32) {
    const uint4 w = z[v];
    const float d[8] = {bf16lo(w.x) - mean, bf16hi(w.x) - mean, bf16lo(w.y) - mean,
                        bf16hi(w.y) - mean, bf16lo(w.z) - mean, bf16hi(w.z) - mean,
                        bf16lo(w.w) - mean, bf16hi(w.w) - mean};
#pragma unroll
    for (int e = 0; e < 8; ++e) ss += d[e] * d[e];
  }
  const float rstd = rsqrtf(warp_sum(ss) / static_cast<float>(h) + eps);
  for (int v = lane; v < nv; v += 32) {
    const uint4 w = z[v];
    uint4 y;
    y.x = pack_bf16x2((bf16lo(w.x) - mean) * rstd, (bf16hi(w.x) - mean) * rstd);
    y.y = pack_bf16x2((bf16lo(w.y) - mean) * rstd, (bf16hi(w.y) - mean) * rstd);
    y.z = pack_bf16x2((bf16lo(w.z) - mean) * rstd, (bf16hi(w.z) - mean) * rstd);
    y.w = pack_bf16x2((bf16lo(w.w) - mean) * rstd, (bf16hi(w.w) - mean) * rstd);
    o[v] = y;
  }
}

cudaError_t launch_layernorm(const uint16_t* Z, int64_t rows, int64_t h, float eps, uint16_t* out,
                             cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int grid = static_cast<int>((rows + 7) / 8);
  layernorm_kernel<<<grid, 256, 0, st>>>(Z, rows, h, eps, out);
  return cudaGetLastError();
}

}  // namespace dm
