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
                                                        uint16_t* __restrict__ out, float* __restrict__ rstd_out) {
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
  if (rstd_out && lane == 0) rstd_out[r] = rstd;
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

// The same LayerNorm with the row read from memory once: each lane keeps its (at most NPL) 16-byte
// pieces of the row in registers across the three passes.  Every sum takes the same terms in the
// same order as layernorm_kernel, so the results are the same bit for bit.
template <int NPL>
__global__ void __launch_bounds__(256) layernorm_reg_kernel(const uint16_t* __restrict__ Z, int64_t rows,
                                                            int64_t h, float eps, uint16_t* __restrict__ out,
                                                            float* __restrict__ rstd_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (r >= rows) return;
  const uint4* z = reinterpret_cast<const uint4*>(Z + r * h);
  uint4* o = reinterpret_cast<uint4*>(out + r * h);
  const int nv = static_cast<int>(h / 8);
  uint4 w[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) w[i] = (lane + 32 * i < nv) ? z[lane + 32 * i] : make_uint4(0u, 0u, 0u, 0u);
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < nv)
      s += bf16lo(w[i].x) + bf16hi(w[i].x) + bf16lo(w[i].y) + bf16hi(w[i].y) + bf16lo(w[i].z) + bf16hi(w[i].z) +
           bf16lo(w[i].w) + bf16hi(w[i].w);
  const float mean = warp_sum(s) / static_cast<float>(h);
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < nv) {
      const float d[8] = {bf16lo(w[i].x) - mean, bf16hi(w[i].x) - mean, bf16lo(w[i].y) - mean,
                          bf16hi(w[i].y) - mean, bf16lo(w[i].z) - mean, bf16hi(w[i].z) - mean,
                          bf16lo(w[i].w) - mean, bf16hi(w[i].w) - mean};
#pragma unroll
      for (int e = 0; e < 8; ++e) ss += d[e] * d[e];
    }
  const float rstd = rsqrtf(warp_sum(ss) / static_cast<float>(h) + eps);
  if (rstd_out && lane == 0) rstd_out[r] = rstd;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < nv) {
      uint4 y;
      y.x = pack_bf16x2((bf16lo(w[i].x) - mean) * rstd, (bf16hi(w[i].x) - mean) * rstd);
      y.y = pack_bf16x2((bf16lo(w[i].y) - mean) * rstd, (bf16hi(w[i].y) - mean) * rstd);
      y.z = pack_bf16x2((bf16lo(w[i].z) - mean) * rstd, (bf16hi(w[i].z) - mean) * rstd);
      y.w = pack_bf16x2((bf16lo(w[i].w) - mean) * rstd, (bf16hi(w[i].w) - mean) * rstd);
      o[lane + 32 * i] = y;
    }
}

cudaError_t launch_layernorm(const uint16_t* Z, int64_t rows, int64_t h, float eps, uint16_t* out,
                             float* rstd, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int grid = static_cast<int>((rows + 7) / 8);
  const int64_t per_lane = (h / 8 + 31) / 32;  // 16-byte pieces of a row per lane
  if (per_lane <= 8)
    layernorm_reg_kernel<8><<<grid, 256, 0, st>>>(Z, rows, h, eps, out, rstd);
  else if (per_lane <= 16)
    layernorm_reg_kernel<16><<<grid, 256, 0, st>>>(Z, rows, h, eps, out, rstd);
  else if (per_lane <= 32)
    layernorm_reg_kernel<32><<<grid, 256, 0, st>>>(Z, rows, h, eps, out, rstd);
  else
    layernorm_kernel<<<grid, 256, 0, st>>>(Z, rows, h, eps, out, rstd);
  return cudaGetLastError();
}

// Backward of LayerNorm without affine parameters, fused with the residual path, one warp per row:
//   out = bf16( res + r (gN - mean(gN) - N mean(gN N)) )
// gN: gradient at the LayerNorm output; N: the (bf16) LayerNorm output; r = 1/sqrt(var + eps) of
// the forward; res: the gradient arriving through the residual connection.  out may equal res.
__global__ void __launch_bounds__(256) layernorm_bwd_kernel(const uint16_t* __restrict__ gN,
                                                            const uint16_t* __restrict__ N,
                                                            const float* __restrict__ rstd,
                                                            const uint16_t* res, uint16_t* out, int64_t rows,
                                                            int64_t h) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (r >= rows) return;
  const uint4* g = reinterpret_cast<const uint4*>(gN + r * h);
  const uint4* n = reinterpret_cast<const uint4*>(N + r * h);
  const int nv = static_cast<int>(h / 8);
  float sg = 0.0f, sgn = 0.0f;
  for (int v = lane; v < nv; v += 32) {
    const uint4 gw = g[v], nw = n[v];
    const uint32_t ga[4] = {gw.x, gw.y, gw.z, gw.w}, na[4] = {nw.x, nw.y, nw.z, nw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float g0 = bf16lo(ga[e]), g1 = bf16hi(ga[e]);
      sg += g0 + g1;
      sgn += g0 * bf16lo(na[e]) + g1 * bf16hi(na[e]);
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  const float mg = warp_sum(sg) * inv_h, mgn = warp_sum(sgn) * inv_h;
  const float rs = rstd[r];
  const uint4* rr = reinterpret_cast<const uint4*>(res + r * h);
  uint4* o = reinterpret_cast<uint4*>(out + r * h);
  for (int v = lane; v < nv; v += 32) {
    const uint4 gw = g[v], nw = n[v], rw = rr[v];
    const uint32_t ga[4] = {gw.x, gw.y, gw.z, gw.w}, na[4] = {nw.x, nw.y, nw.z, nw.w},
                   ra[4] = {rw.x, rw.y, rw.z, rw.w};
    uint32_t oa[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float d0 = rs * (bf16lo(ga[e]) - mg - bf16lo(na[e]) * mgn);
      const float d1 = rs * (bf16hi(ga[e]) - mg - bf16hi(na[e]) * mgn);
      oa[e] = pack_bf16x2(bf16lo(ra[e]) + d0, bf16hi(ra[e]) + d1);
    }
    o[v] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  }
}

// The same backward with gN and N read from memory once (kept in registers across both passes;
// same sums in the same order as layernorm_bwd_kernel, so the same results bit for bit).
template <int NPL>
__global__ void __launch_bounds__(256) layernorm_bwd_reg_kernel(const uint16_t* __restrict__ gN,
                                                                const uint16_t* __restrict__ N,
                                                                const float* __restrict__ rstd,
                                                                const uint16_t* res, uint16_t* out, int64_t rows,
                                                                int64_t h) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (r >= rows) return;
  const uint4* g = reinterpret_cast<const uint4*>(gN + r * h);
  const uint4* n = reinterpret_cast<const uint4*>(N + r * h);
  const int nv = static_cast<int>(h / 8);
  uint4 gw[NPL], nw[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const bool in = lane + 32 * i < nv;
    gw[i] = in ? g[lane + 32 * i] : make_uint4(0u, 0u, 0u, 0u);
    nw[i] = in ? n[lane + 32 * i] : make_uint4(0u, 0u, 0u, 0u);
  }
  float sg = 0.0f, sgn = 0.0f;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < nv) {
      const uint32_t ga[4] = {gw[i].x, gw[i].y, gw[i].z, gw[i].w}, na[4] = {nw[i].x, nw[i].y, nw[i].z, nw[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float g0 = bf16lo(ga[e]), g1 = bf16hi(ga[e]);
        sg += g0 + g1;
        sgn += g0 * bf16lo(na[e]) + g1 * bf16hi(na[e]);
      }
    }
  const float inv_h = 1.0f / static_cast<float>(h);
  const float mg = warp_sum(sg) * inv_h, mgn = warp_sum(sgn) * inv_h;
  const float rs = rstd[r];
  const uint4* rr = reinterpret_cast<const uint4*>(res + r * h);
  uint4* o = reinterpret_cast<uint4*>(out + r * h);
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < nv) {
      const uint4 rw = rr[lane + 32 * i];
      const uint32_t ga[4] = {gw[i].x, gw[i].y, gw[i].z, gw[i].w}, na[4] = {nw[i].x, nw[i].y, nw[i].z, nw[i].w},
                     ra[4] = {rw.x, rw.y, rw.z, rw.w};
      uint32_t oa[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float d0 = rs * (bf16lo(ga[e]) - mg - bf16lo(na[e]) * mgn);
        const float d1 = rs * (bf16hi(ga[e]) - mg - bf16hi(na[e]) * mgn);
        oa[e] = pack_bf16x2(bf16lo(ra[e]) + d0, bf16hi(ra[e]) + d1);
      }
      o[lane + 32 * i] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    }
}

cudaError_t launch_layernorm_bwd(const uint16_t* gN, const uint16_t* N, const float* rstd, const uint16_t* res,
                                 uint16_t* out, int64_t rows, int64_t h, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int grid = static_cast<int>((rows + 7) / 8);
  const int64_t per_lane = (h / 8 + 31) / 32;  // 16-byte pieces of a row per lane
  if (per_lane <= 8)
    layernorm_bwd_reg_kernel<8><<<grid, 256, 0, st>>>(gN, N, rstd, res, out, rows, h);
  else if (per_lane <= 16)
    layernorm_bwd_reg_kernel<16><<<grid, 256, 0, st>>>(gN, N, rstd, res, out, rows, h);
  else
    layernorm_bwd_kernel<<<grid, 256, 0, st>>>(gN, N, rstd, res, out, rows, h);
  return cudaGetLastError();
}

// The epilogues' activation functions on a vector: non-gated out = act(a), da = act'(a); gated
// out = glu(a, b), da = d out / d a, db = d out / d b.
__global__ void act_eval_kernel(int act, const float* __restrict__ a, const float* __restrict__ b,
                                float* __restrict__ out, float* __restrict__ da, float* __restrict__ db, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    if (act == ACT_SWIGLU || act == ACT_BILINEAR) {
      float dg, du, hv;
      glu_bwd(act, a[i], b[i], 1.0f, dg, du, hv);
      out[i] = glu_fwd(act, a[i], b[i]);
      da[i] = dg;
      db[i] = du;
    } else {
      float hv, d;
      act_fwd_grad(act, a[i], hv, d);
      out[i] = act_fwd(act, a[i]);
      da[i] = d;
      if (db) db[i] = act_grad(act, a[i]) - d;  // 0 when the two code paths agree
    }
  }
}

cudaError_t launch_act_eval(int act, const float* a, const float* b, float* out, float* da, float* db, int64_t n,
                            cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int grid = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  act_eval_kernel<<<grid, 256, 0, st>>>(act, a, b, out, da, db, n);
  return cudaGetLastError();
}

}  // namespace dm
