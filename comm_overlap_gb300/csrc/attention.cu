// attention.cu -- causal multi-head self-attention of one row chunk, for the attention sublayer of
// the tensor-parallel Transformer block ("TP 的数据依赖：通信为何难以隐藏": for the attention layer of
// XAB=Y, A is the multi-head attention, B the output projection).  Heads are split over the t
// shards; shard i's query/key/value heads come from its own slice of the fused projection output.
//
// One CTA computes two consecutive query blocks of 128 positions (tiles 0 and 1) of one head and
// sequence: O = softmax(Q K^T / sqrt(d) + causal mask) V, with an online softmax over key/value
// blocks of 128 positions (running maximum and sum rescaled as blocks arrive; equal to the plain
// softmax up to rounding).  Both tiles use the same K_j, V_j, and their work alternates on the
// tensor core so that one tile's softmax runs under the other tile's matrix products.
// Warp roles:
//   warp 0 (one lane)  TMA producer: both Q tiles once, then K and V tiles into two-deep rings.
//   warp 1 (one lane)  MMA issuer, per block j and tile x: O_x += P_x V_j as soon as the softmax
//                      handed P_x over, then S_x = Q_x K_{j+1}^T (in that order: P_x lives in the
//                      columns of S_x, and tensor-core operations of one thread run in order).
//   warps 2-5, 6-9     softmax of tile 0 and tile 1, one query row per thread (TMEM lane quarter =
//                      warp % 4): scores from TMEM, running max / sum in fp32, O_x rescaled in TMEM
//                      when a row maximum grew, P rounded to bf16 and stored into TMEM; at the end
//                      O / sum -> bf16 -> TMA store (staged in the tile's Q buffer).
// TMEM: S_0 = columns 0-127, S_1 = 128-255 (P_x in the first 64 columns of S_x as bf16 pairs),
// O_0 = 256-383, O_1 = 384-511.
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
constexpr uint32_t kTile = kAttnBlk * kAttnD * 2;   // 32 KiB: one Q, K or V tile
constexpr uint32_t kHalf = kTile / 2;               // one 64-column (128-byte) swizzle panel
constexpr int kAttnThreads = 320;
constexpr int kAttnSmem = 1024 /* alignment slack */ + 1024 /* control */ + 6 * kTile;  // Q[2], K[2], V[2]
constexpr uint32_t kAttnTmemCols = 512;
constexpr uint64_t kAttnDrainNs = 200000000ull;

// barrier indices
enum : int {
  B_Q_FULL = 0, B_K_FULL = 1, B_K_EMPTY = 3, B_V_FULL = 5, B_V_EMPTY = 7, B_S_FULL = 9, B_P_FULL = 11,
  B_PV_DONE = 13, B_DRAIN = 15, B_COUNT = 16
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
  const uint32_t sQ = smem_u32(smem + 1024), sK = sQ + 2 * kTile, sV = sQ + 4 * kTile;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_pairs = (a.n_qblk + 1) >> 1;
  const int q0 = 2 * (n_pairs - 1 - static_cast<int>(blockIdx.x));  // longest (most key blocks) first
  const int ntiles = (q0 + 1 < a.n_qblk) ? 2 : 1;
  const int hd = blockIdx.y, sq = blockIdx.z;
  const int shard = hd / a.nhi, jh = hd - shard * a.nhi;
  const int slot_q = (shard * 3 + 0) * a.nhi + jh, slot_k = (shard * 3 + 1) * a.nhi + jh,
            slot_v = (shard * 3 + 2) * a.nhi + jh;
  const int nblk = q0 + ntiles;  // key/value blocks 0 .. q0 + ntiles - 1 (tile x stops at q0 + x)
  int* err = &g_attn_err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), (i == B_P_FULL || i == B_P_FULL + 1) ? 4 : 1);
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
      mbar_arrive_expect_tx(bar(B_Q_FULL), kTile * static_cast<uint32_t>(ntiles));
      for (int x = 0; x < ntiles; ++x) {
        const int p0 = (q0 + x) * kAttnBlk;
        tma_load_4d(sQ + x * kTile, &tmQKV, bar(B_Q_FULL), 0, slot_q, p0, sq);
        tma_load_4d(sQ + x * kTile + kHalf, &tmQKV, bar(B_Q_FULL), 64, slot_q, p0, sq);
      }
      uint32_t k_armed = 0, k_ph = 0, v_armed = 0, v_ph = 0;
      bool ok = true;
      for (int j = 0; j < nblk && ok; ++j) {
        const int b = j & 1;
        const uint32_t use = static_cast<uint32_t>(j >> 1) & 1u;
        const int pos = j * kAttnBlk;
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
      const int last_tile = ntiles - 1;  // the tile with the most blocks: the last user of K_j, V_j
      // Shared-memory descriptors are built once; a K step adds its byte offset / 16 to the start
      // address field (bits 0-13: shared addresses below 256 KiB never carry out of it).
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024), dK0 = sdesc_sw128(sK, 16, 1024),
                     dV0 = sdesc_sw128(sV, kHalf, 1024);
      // S_x = Q_x K_j^T into TMEM columns 128 x
      auto issue_qk = [&](int x, int j) -> bool {
        const int b = j & 1;
        if (!mbar_wait(bar(B_K_FULL + b), static_cast<uint32_t>(j >> 1) & 1u, abort_flag, err, a.err_site + 3))
          return false;
        tc_fence_after();
        const uint64_t dq = dQ0 + ((static_cast<uint64_t>(x) * kTile) >> 4),
                       dk = dK0 + ((static_cast<uint64_t>(b) * kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kAttnD / 16; ++kk) {
          const uint64_t off = (static_cast<uint64_t>(kk >> 2) * kHalf + static_cast<uint64_t>(kk & 3) * 32u) >> 4;
          umma_bf16(tmem_base + 128u * x, dq + off, dk + off, kIdQK, static_cast<uint32_t>(kk != 0));
        }
        umma_commit(bar(B_S_FULL + x));
        if (x == last_tile) umma_commit(bar(B_K_EMPTY + b));
        return true;
      };
      bool ok = mbar_wait(bar(B_Q_FULL), 0, abort_flag, err, a.err_site + 5);
      for (int x = 0; x < ntiles && ok; ++x) ok = issue_qk(x, 0);
      for (int j = 0; j < nblk && ok; ++j) {
        const int b = j & 1;
        for (int x = 0; x < ntiles && ok; ++x) {
          if (j > q0 + x) continue;  // tile x is done
          if (!mbar_wait(bar(B_P_FULL + x), static_cast<uint32_t>(j & 1), abort_flag, err, a.err_site + 6) ||
              !mbar_wait(bar(B_V_FULL + b), static_cast<uint32_t>(j >> 1) & 1u, abort_flag, err, a.err_site + 7)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dv = dV0 + ((static_cast<uint64_t>(b) * kTile) >> 4);
#pragma unroll
          for (int kk = 0; kk < kAttnBlk / 16; ++kk)
            // A = P_x from TMEM (8 columns of bf16 pairs per K step of 16); B = V_j, MN-major: its
            // two 64-column panels of d sit kHalf apart, 8-row groups of positions 1024 bytes apart
            umma_bf16_tmem_a(tmem_base + 256u + 128u * x, tmem_base + 128u * x + 8u * kk,
                             dv + ((static_cast<uint64_t>(kk) * 2048u) >> 4), kIdPV, static_cast<uint32_t>((j | kk) != 0));
          umma_commit(bar(B_PV_DONE + x));
          if (x == last_tile) umma_commit(bar(B_V_EMPTY + b));
          if (j + 1 <= q0 + x && !issue_qk(x, j + 1)) ok = false;
        }
      }
      // every MMA this thread issued has completed once the drain barrier flips
      umma_commit(bar(B_DRAIN));
      attn_wait_drain(bar(B_DRAIN), 0);
    }
  } else {
    // ---------------- softmax warps: tile x, query row `row` of the tile
    const int x = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qblk = q0 + x;
    const int q_pos = qblk * kAttnBlk + row;
    const uint32_t lq = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + lq + 128u * x, tO = tmem_base + lq + 256u + 128u * x;
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = x < ntiles;
    for (int j = 0; ok && j <= qblk; ++j) {
      ok = mbar_wait(bar(B_S_FULL + x), static_cast<uint32_t>(j & 1), abort_flag, err, a.err_site + 8);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // raw scores stay in the registers of the TMEM loads; the reductions use 8 independent
      // accumulators each so that they are not one long dependency chain
      uint32_t sr[4][32];
#pragma unroll
      for (int i = 0; i < 4; ++i) tmem_ld32(tS + 32u * i, sr[i]);
      tmem_ld_wait();
      if (j == qblk) {  // diagonal block: key position j*128 + c attends only if <= q_pos
        const int lim = q_pos - j * kAttnBlk;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) m8[c & 7] = fmaxf(m8[c & 7], __uint_as_float(sr[c >> 5][c & 31]));
#pragma unroll
      for (int k = 4; k > 0; k >>= 1)
#pragma unroll
        for (int i = 0; i < k; ++i) m8[i] = fmaxf(m8[i], m8[i + k]);
      // Running maximum in the log2 domain (the scale log2(e) / sqrt(d) is positive).  It is raised
      // only when some row of the warp would exceed it by more than 8 (p <= 2^8 otherwise, harmless
      // in fp32 and bf16); O and the sum are then rescaled by alpha.  Numerator and denominator always
      // use the same maximum, so the result is unchanged.
      const float cand = fmaxf(m_run, m8[0] * a.scale_log2);
      const bool raise = __any_sync(0xFFFFFFFFu, cand > m_run + 8.0f) || j == 0;
      const float mx = raise ? cand : m_run;
      const float alpha = raise ? ex2_approx(m_run - mx) : 1.0f;  // 0 on the first block (m_run = -inf)
      const float nmx = -mx;
      float l8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) l8[k] = 0.0f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {  // p replaces the score in place
        const float pv = ex2_approx(fmaf(__uint_as_float(sr[c >> 5][c & 31]), a.scale_log2, nmx));
        sr[c >> 5][c & 31] = __float_as_uint(pv);
        l8[c & 7] += pv;
      }
#pragma unroll
      for (int k = 4; k > 0; k >>= 1)
#pragma unroll
        for (int i = 0; i < k; ++i) l8[i] += l8[i + k];
      l_run = l_run * alpha + l8[0];
      m_run = mx;
      if (j > 0) {
        // O_x and the P_x columns are free once the previous block's O_x += P_x V has completed
        ok = mbar_wait(bar(B_PV_DONE + x), static_cast<uint32_t>((j - 1) & 1), abort_flag, err, a.err_site + 9);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // P_x -> bf16 pairs into the first 64 columns of S_x (the scores are in registers)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e = 64 * h2 + 2 * c;
          pk[c] = pack_bf16x2(__uint_as_float(sr[e >> 5][e & 31]), __uint_as_float(sr[(e + 1) >> 5][(e + 1) & 31]));
        }
        tmem_st32(tS + 32u * h2, pk);
      }
      if (j > 0 && raise) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + static_cast<uint32_t>(c * 32), o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + static_cast<uint32_t>(c * 32), o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_FULL + x));
    }
    if (ok) {
      ok = mbar_wait(bar(B_PV_DONE + x), static_cast<uint32_t>(qblk & 1), abort_flag, err, a.err_site + 10);
      if (__all_sync(0xFFFFFFFFu, ok)) {
        tc_fence_after();
        const float inv = 1.0f / l_run;
        // the tile's Q buffer is free (its last product has completed): each warp stages its 32
        // rows as two 32 x 64 boxes (128-byte swizzle)
        const uint32_t stage = sQ + x * kTile + static_cast<uint32_t>(quarter) * 8192u;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + static_cast<uint32_t>(c * 32), o);
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
        const int p0 = qblk * kAttnBlk + quarter * 32;  // rows past the sequence end are clipped
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
  attention_kernel<<<dim3((a.n_qblk + 1) / 2, a.heads, nseq), kAttnThreads, kAttnSmem, st>>>(tm_qkv, tm_o, a);
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
