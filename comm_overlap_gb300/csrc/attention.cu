// attention.cu -- causal multi-head self-attention of one row chunk, for the attention sublayer of
// the tensor-parallel Transformer block ("TP 的数据依赖：通信为何难以隐藏": for the attention layer of
// XAB=Y, A is the multi-head attention, B the output projection).  Heads are split over the t
// shards; shard i's query/key/value heads come from its own slice of the fused projection output.
//
// One CTA computes one (query block of 128 positions, head, sequence): O = softmax(Q K^T / sqrt(d)
// + causal mask) V with an online softmax over key/value blocks of 128 positions (the running
// maximum and sum are rescaled as blocks arrive, so the result equals the plain softmax up to
// rounding).  Warp roles:
//   warp 0 (one lane)  TMA producer: the Q tile once, then K and V tiles into two-deep rings.
//   warp 1 (one lane)  MMA issuer: S_j = Q K_j^T into one of two TMEM score buffers (issued one
//                      block ahead, so it overlaps the softmax of the previous block), then
//                      O += P_j V_j into the TMEM output accumulator.
//   warps 2-5          softmax, one query row per thread (TMEM lane quarter = warp % 4): scores
//                      from TMEM, running max / sum in fp32, O rescaled in TMEM when the maximum
//                      grows, P rounded to bf16 into shared memory (128-byte swizzled K-major
//                      layout of the MMA's A operand); at the end O / sum -> bf16 -> TMA store.
// Every wait is bounded (ptx.cuh); on expiry the CTA drains what it has in flight, frees TMEM and
// returns, leaving a code in this translation unit's error word.
#include <cuda_bf16.h>

#include "actfn.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dm {

static __device__ int g_attn_err;

constexpr int kAttnD = 128;                         // head dimension
constexpr int kAttnBlk = 128;                       // query rows / key-value positions per block
constexpr uint32_t kTile = kAttnBlk * kAttnD * 2;   // 32 KiB: one Q, K, V or P tile
constexpr uint32_t kHalf = kTile / 2;               // one 64-column (128-byte) swizzle panel
constexpr int kAttnThreads = 192;
constexpr int kAttnSmem = 1024 /* alignment slack */ + 1024 /* control */ + 6 * kTile;  // Q, K[2], V[2], P
constexpr uint32_t kAttnTmemCols = 512;             // S[2] (2 x 128) + O (128), rounded up
constexpr uint64_t kAttnDrainNs = 200000000ull;

// barrier indices
enum : int {
  B_Q_FULL = 0, B_K_FULL = 1, B_K_EMPTY = 3, B_V_FULL = 5, B_V_EMPTY = 7, B_S_FULL = 9, B_S_EMPTY = 11,
  B_P_FULL = 13, B_PV_DONE = 14, B_DRAIN = 15, B_COUNT = 16
};

__device__ __forceinline__ void attn_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kAttnDrainNs) return;
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmO,
                     const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 516);
  const uint32_t bar0 = smem_u32(smem);
  auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t sQ = smem_u32(smem + 1024), sK = sQ + kTile, sV = sQ + 3 * kTile, sP = sQ + 5 * kTile;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = a.n_qblk - 1 - static_cast<int>(blockIdx.x);  // longest (most key blocks) first
  const int hd = blockIdx.y, sq = blockIdx.z;
  const int shard = hd / a.nhi, jh = hd - shard * a.nhi;
  const int slot_q = (shard * 3 + 0) * a.nhi + jh, slot_k = (shard * 3 + 1) * a.nhi + jh,
            slot_v = (shard * 3 + 2) * a.nhi + jh;
  const int nkv = qb + 1;  // causal: key/value blocks 0 .. qb
  int* err = &g_attn_err;

  if (threadIdx.x == 0) {
    // the score buffers and P are released / filled by the four softmax warps
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(bar(i), (i == B_S_EMPTY || i == B_S_EMPTY + 1 || i == B_P_FULL) ? 4 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmQKV);
    tma_prefetch_map(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kAttnTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const int p0 = qb * kAttnBlk;
      mbar_arrive_expect_tx(bar(B_Q_FULL), kTile);
      tma_load_4d(sQ, &tmQKV, bar(B_Q_FULL), 0, slot_q, p0, sq);
      tma_load_4d(sQ + kHalf, &tmQKV, bar(B_Q_FULL), 64, slot_q, p0, sq);
      // armed[b]: parity of the last phase armed on K/V full barrier b (bit set = armed)
      uint32_t k_armed = 0, k_ph = 0, v_armed = 0, v_ph = 0;
      bool ok = true;
      for (int kv = 0; kv < nkv && ok; ++kv) {
        const int b = kv & 1;
        const uint32_t use = static_cast<uint32_t>(kv >> 1) & 1u;
        const int pos = kv * kAttnBlk;
        if (!mbar_wait(bar(B_K_EMPTY + b), use ^ 1u, abort_flag, err, a.err_site + 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(B_K_FULL + b), kTile);
        k_armed |= 1u << b;
        k_ph = (k_ph & ~(1u << b)) | (use << b);
        tma_load_4d(sK + b * kTile, &tmQKV, bar(B_K_FULL + b), 0, slot_k, pos, sq);
        tma_load_4d(sK + b * kTile + kHalf, &tmQKV, bar(B_K_FULL + b), 64, slot_k, pos, sq);
        if (!mbar_wait(bar(B_V_EMPTY + b), use ^ 1u, abort_flag, err, a.err_site + 2)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(B_V_FULL + b), kTile);
        v_armed |= 1u << b;
        v_ph = (v_ph & ~(1u << b)) | (use << b);
        tma_load_4d(sV + b * kTile, &tmQKV, bar(B_V_FULL + b), 0, slot_v, pos, sq);
        tma_load_4d(sV + b * kTile + kHalf, &tmQKV, bar(B_V_FULL + b), 64, slot_v, pos, sq);
      }
      if (!ok) {
        // let the copies still in flight land before the CTA leaves
        attn_wait_drain(bar(B_Q_FULL), 0);
        for (int b = 0; b < 2; ++b) {
          if ((k_armed >> b) & 1u) attn_wait_drain(bar(B_K_FULL + b), (k_ph >> b) & 1u);
          if ((v_armed >> b) & 1u) attn_wait_drain(bar(B_V_FULL + b), (v_ph >> b) & 1u);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t kIdQK = idesc_bf16_f32(kAttnBlk, kAttnBlk, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(kAttnBlk, kAttnD, false, true);
      const uint32_t tO = tmem_base + 256u;
      auto issue_qk = [&](int kv) -> bool {
        const int b = kv & 1;
        const uint32_t use = static_cast<uint32_t>(kv >> 1) & 1u;
        if (!mbar_wait(bar(B_K_FULL + b), use, abort_flag, err, a.err_site + 3)) return false;
        if (!mbar_wait(bar(B_S_EMPTY + b), use ^ 1u, abort_flag, err, a.err_site + 4)) return false;
        tc_fence_after();
        const uint32_t kb = sK + b * kTile;
#pragma unroll
        for (int kk = 0; kk < kAttnD / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>(kk >> 2) * kHalf + static_cast<uint32_t>(kk & 3) * 32u;
          umma_bf16(tmem_base + b * 128u, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), kIdQK,
                    static_cast<uint32_t>(kk != 0));
        }
        umma_commit(bar(B_K_EMPTY + b));
        umma_commit(bar(B_S_FULL + b));
        return true;
      };
      bool ok = mbar_wait(bar(B_Q_FULL), 0, abort_flag, err, a.err_site + 5);
      if (ok) ok = issue_qk(0);
      for (int kv = 0; kv < nkv && ok; ++kv) {
        if (kv + 1 < nkv && !issue_qk(kv + 1)) {
          ok = false;
          break;
        }
        const int b = kv & 1;
        const uint32_t use = static_cast<uint32_t>(kv >> 1) & 1u;
        if (!mbar_wait(bar(B_P_FULL), static_cast<uint32_t>(kv & 1), abort_flag, err, a.err_site + 6) ||
            !mbar_wait(bar(B_V_FULL + b), use, abort_flag, err, a.err_site + 7)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vb = sV + b * kTile;
#pragma unroll
        for (int kk = 0; kk < kAttnBlk / 16; ++kk) {
          const uint32_t aoff = static_cast<uint32_t>(kk >> 2) * kHalf + static_cast<uint32_t>(kk & 3) * 32u;
          // V is [position][d]: for the MMA's B operand (N = d, K = position) it is MN-major; the
          // two 64-column panels of d sit kHalf apart, 8-row groups of positions 1024 bytes apart
          umma_bf16(tO, sdesc_sw128(sP + aoff, 16, 1024), sdesc_sw128(vb + static_cast<uint32_t>(kk) * 2048u, kHalf, 1024),
                    kIdPV, static_cast<uint32_t>((kv | kk) != 0));
        }
        umma_commit(bar(B_V_EMPTY + b));
        umma_commit(bar(B_PV_DONE));
      }
      // every MMA this thread issued has completed once the drain barrier flips
      umma_commit(bar(B_DRAIN));
      attn_wait_drain(bar(B_DRAIN), 0);
    }
  } else {
    // ---------------- softmax warps: query row `row` of the block
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int q_pos = qb * kAttnBlk + row;
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    for (int kv = 0; kv < nkv; ++kv) {
      const int b = kv & 1;
      const uint32_t use = static_cast<uint32_t>(kv >> 1) & 1u;
      ok = mbar_wait(bar(B_S_FULL + b), use, abort_flag, err, a.err_site + 8);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(tq + b * 128u + 0u, r0);
      tmem_ld32(tq + b * 128u + 32u, r1);
      tmem_ld32(tq + b * 128u + 64u, r2);
      tmem_ld32(tq + b * 128u + 96u, r3);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_S_EMPTY + b));  // the score buffer may be overwritten
      float x[128];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        x[e] = __uint_as_float(r0[e]) * a.scale_log2;
        x[32 + e] = __uint_as_float(r1[e]) * a.scale_log2;
        x[64 + e] = __uint_as_float(r2[e]) * a.scale_log2;
        x[96 + e] = __uint_as_float(r3[e]) * a.scale_log2;
      }
      if (kv == qb) {  // diagonal block: key position kv*128 + c attends only if <= q_pos
        const int lim = q_pos - kv * kAttnBlk;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) x[c] = -INFINITY;
      }
      float mx = m_run;
#pragma unroll
      for (int c = 0; c < 128; ++c) mx = fmaxf(mx, x[c]);
      const float alpha = exp2f(m_run - mx);  // 0 on the first block (m_run = -inf)
      float sum = 0.0f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        x[c] = exp2f(x[c] - mx);
        sum += x[c];
      }
      l_run = l_run * alpha + sum;
      m_run = mx;
      if (kv > 0) {
        // P and O are free once the previous block's O += P V has completed
        ok = mbar_wait(bar(B_PV_DONE), static_cast<uint32_t>((kv - 1) & 1), abort_flag, err, a.err_site + 9);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tq + 256u + static_cast<uint32_t>(c * 32), o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tq + 256u + static_cast<uint32_t>(c * 32), o);
          }
          tmem_st_wait();
        }
      }
      // P row -> bf16, 16-byte unit u of panel (u >> 3) at position (u & 7) ^ (row & 7)
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t addr = sP + static_cast<uint32_t>(u >> 3) * kHalf + static_cast<uint32_t>(row) * 128u +
                              ((static_cast<uint32_t>(u & 7) ^ (static_cast<uint32_t>(row) & 7u)) << 4);
        st_shared_v4(addr, pack_bf16x2(x[8 * u], x[8 * u + 1]), pack_bf16x2(x[8 * u + 2], x[8 * u + 3]),
                     pack_bf16x2(x[8 * u + 4], x[8 * u + 5]), pack_bf16x2(x[8 * u + 6], x[8 * u + 7]));
      }
      fence_proxy_async_smem();  // P visible to the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_FULL));
    }
    if (ok) {
      ok = mbar_wait(bar(B_PV_DONE), static_cast<uint32_t>((nkv - 1) & 1), abort_flag, err, a.err_site + 10);
      if (__all_sync(0xFFFFFFFFu, ok)) {
        tc_fence_after();
        const float inv = 1.0f / l_run;
        // the P tile is free: each warp stages its 32 rows as two 32 x 64 boxes (128-byte swizzle)
        const uint32_t stage = sP + static_cast<uint32_t>(warp - 2) * 8192u;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tq + 256u + static_cast<uint32_t>(c * 32), o);
          tmem_ld_wait();
          const uint32_t box = stage + static_cast<uint32_t>(c >> 1) * 4096u + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t unit = static_cast<uint32_t>((c & 1) * 4 + k);
            st_shared_v4(box + ((unit ^ (static_cast<uint32_t>(lane) & 7u)) << 4),
                         pack_bf16x2(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                         pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                         pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                         pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int p0 = qb * kAttnBlk + quarter * 32;  // rows past the sequence end are clipped
        if (lane == 0 && p0 < a.seq) {
          tma_store_4d(&tmO, stage, 0, hd, p0, sq);
          tma_store_4d(&tmO, stage + 4096u, 64, hd, p0, sq);
          bulk_commit_group();
          bulk_wait_group_all();
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kAttnTmemCols);
  }
}

cudaError_t launch_attention(const CUtensorMap& tm_qkv, const CUtensorMap& tm_o, const AttnArgs& a, int nseq,
                             cudaStream_t st) {
  if (nseq == 0 || a.n_qblk == 0 || a.heads == 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attention_kernel<<<dim3(a.n_qblk, a.heads, nseq), kAttnThreads, kAttnSmem, st>>>(tm_qkv, tm_o, a);
  return cudaGetLastError();
}

cudaError_t take_attn_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_err, sizeof(int));
  if (e != cudaSuccess) return e;
  *code = v;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_attn_err, &zero, sizeof(int));
  }
  return e;
}

}  // namespace dm
