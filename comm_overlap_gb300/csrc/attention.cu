// attention.cu -- causal multi-head self-attention of one row chunk, for the attention sublayer of
// the tensor-parallel Transformer block ("TP 的数据依赖：通信为何难以隐藏": for the attention layer of
// XAB=Y, A is the multi-head attention, B the output projection).  Heads are split over the t
// shards; shard i's query/key/value heads come from its own slice of the fused projection output.
//
// Work item: two consecutive query blocks of 128 positions (tiles 0 and 1) of one head and
// sequence: O = softmax(Q K^T / sqrt(d) + causal mask) V, with an online softmax over key/value
// blocks of 128 positions (running maximum and sum rescaled as blocks arrive; equal to the plain
// softmax up to rounding).  Both tiles use the same K_j, V_j, and their work alternates on the
// tensor core so that one tile's softmax runs under the other tile's matrix products.
// The kernel is persistent: one CTA per SM walks a fixed list of units, a unit being the heaviest
// and the lightest remaining item of one (head, sequence), so that all units cost about the same;
// consecutive CTAs take consecutive units, which keeps the K/V of the heads in flight in L2.  The
// next item's Q tiles are loaded as soon as the current item's last Q K^T products have
// completed, and its first products start while the current item's O is being written out.
// Warp roles:
//   warp 0 (one lane)  TMA producer: each item's Q tiles, then its K and V tiles into two-deep rings
//                      (the rings run on across items).
//   warps 1, 10        MMA issuers of tile 0 and tile 1 (one lane each), per block j: O_x += P_x V_j
//   (one lane each)    as soon as the softmax handed P_x over, then S_x = Q_x K_{j+1}^T (in that
//                      order: P_x lives in the columns of S_x, and the tensor-core operations of
//                      one thread complete in order).  Issuing a 128 x 128 x 16 product takes a
//                      thread about as long as the tensor core takes to execute it, so a single
//                      issuer leaves the tensor core idle while it waits and commits.  The two issuers
//                      take turns (B_TURN) in the order one issuer would use -- per block tile 0's
//                      products, then tile 1's, so that neither tile's products are spread out by the
//                      other's -- and each waits for its data before its turn (the softmax hand-off
//                      last, polled: it is the critical path) and commits after it.
//   warps 2-5, 6-9     softmax of tile 0 and tile 1, one query row per thread (TMEM lane quarter =
//                      warp % 4): scores from TMEM, running max / sum in fp32, O_x rescaled in TMEM
//                      when a row maximum grew, P rounded to bf16 and stored into TMEM; at the end
//                      of an item O / sum -> bf16 -> TMA store through a per-warp staging box.
// TMEM: S_0 = columns 0-127, S_1 = 128-255 (P_x in the first 64 columns of S_x as bf16 pairs),
// O_0 = 256-383, O_1 = 384-511.
// Every wait is bounded (ptx.cuh); on expiry the CTA stops issuing work, lets what it has in
// flight drain, frees TMEM and returns, leaving a code in this translation unit's error word.
#include <cuda_bf16.h>

#include <atomic>

#include "actfn.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dm {

static __device__ int g_attn_err;

constexpr int kAttnD = 128;                         // head dimension
constexpr int kAttnBlk = 128;                       // query rows / key-value positions per block
constexpr uint32_t kTile = kAttnBlk * kAttnD * 2;   // 32 KiB: one Q, K or V tile
constexpr uint32_t kHalf = kTile / 2;               // one 64-column (128-byte) swizzle panel
constexpr uint32_t kOBox = 32 * 64 * 2;             // 4 KiB: one warp's 32 rows x 64 columns of O
constexpr int kAttnThreads = 352;
constexpr int kAttnIssuer1 = 10;  // the warp that issues tile 1's products (tile 0's: warp 1)
// alignment slack, control, Q[2], K[2], V[2], one O staging box per softmax warp
constexpr int kAttnSmem = 1024 + 1024 + 6 * static_cast<int>(kTile) + 8 * static_cast<int>(kOBox);
static_assert(kAttnSmem <= 232448, "shared memory beyond the per-CTA limit");
constexpr uint32_t kAttnTmemCols = 512;
constexpr uint64_t kAttnDrainNs = 200000000ull;

// barrier indices: pairs are per tile or per ring slot; the ring slots' releases are per tile and
// slot (B_K_EMPTY + 2 x + slot), since the two issuers' products complete independently
enum : int {
  B_Q_FULL = 0, B_Q_EMPTY = 2, B_K_FULL = 4, B_K_EMPTY = 6, B_V_FULL = 10, B_V_EMPTY = 12, B_S_FULL = 16,
  B_P_FULL = 18, B_PV_DONE = 20, B_O_FREE = 22, B_DRAIN = 24, B_TURN = 26, B_COUNT = 28
};
static_assert(8 * B_COUNT <= 512, "barriers overlap the TMEM slot");

// Two-lane fp32 arithmetic (sm_100 and later): each lane is an ordinary fp32 operation with round to
// nearest, so a pair computes exactly what two scalar operations would, in half the issue slots.  The
// softmax warps share their sub-partitions with the MMA issuer and the TMA producer; the fewer
// instructions they issue, the sooner the issuer's tensor-core instructions go out.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// the largest of three (no NaN reaches it: scores are finite or -inf)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}

// As mbar_wait, but polling with the non-blocking test_wait: the thread is never suspended, so it
// sees the phase complete sooner, at the cost of issue slots on its sub-partition while it spins.
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err_word,
                                          int site, uint64_t timeout_ns = kWaitTimeoutNs) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 1023u) == 1023u) {
      if (*abort_flag) return false;
      const uint64_t now = global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicCAS(err_word, 0, site);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void attn_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kAttnDrainNs) return;
  }
}

// The work list.  Items of one (head, sequence) group: query-block pairs ip = 0 .. n_pairs - 1
// (query blocks 2 ip and 2 ip + 1, key blocks 0 .. 2 ip + 1).  Unit k of a group holds item
// n_pairs - 1 - k and, if different, item k; groups are numbered head-fastest.
struct AttnWork {
  int n_pairs, upg, units;
  __device__ AttnWork(const AttnArgs& a, int nseq) {
    n_pairs = (a.n_qblk + 1) >> 1;
    upg = (n_pairs + 1) >> 1;
    units = upg * a.heads * nseq;
  }
};

struct AttnItem {
  int hd, sq, q0, ntiles, nblk;
};

__device__ __forceinline__ AttnItem attn_item(const AttnArgs& a, const AttnWork& w, int u, int half) {
  const int g = u / w.upg, k = u - g * w.upg;
  const int ip = half == 0 ? w.n_pairs - 1 - k : k;
  AttnItem it;
  it.hd = g % a.heads;
  it.sq = g / a.heads;
  it.q0 = 2 * ip;
  it.ntiles = (it.q0 + 1 < a.n_qblk) ? 2 : 1;
  it.nblk = it.q0 + it.ntiles;  // key/value blocks 0 .. nblk - 1 (tile x stops at q0 + x)
  return it;
}

// items in unit u: 2, or 1 when its heaviest and lightest item coincide
__device__ __forceinline__ int attn_unit_items(const AttnWork& w, int u) {
  const int k = u % w.upg;
  return (k < w.n_pairs - 1 - k) ? 2 : 1;
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmO,
                     const AttnArgs a, const int nseq) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 516);
  const uint32_t bar0 = smem_u32(smem);
  auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t sQ = smem_u32(smem + 1024), sK = sQ + 2 * kTile, sV = sQ + 4 * kTile, sO = sQ + 6 * kTile;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnWork w(a, nseq);
  int* err = &g_attn_err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(bar(i), (i == B_P_FULL || i == B_P_FULL + 1 || i == B_O_FREE || i == B_O_FREE + 1) ? 4 : 1);
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
      uint32_t gb = 0;          // ring position of the item's key block 0
      int nq[2] = {0, 0};       // items so far in which tile x took part
      // ring slot b's current block: bit 2 b + x set if tile x consumes it (cons); parity of the
      // blocks of slot b that tile x consumed so far (upar), i.e. of the releases it will have made
      uint32_t cons = 0, upar = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < w.units && ok; u += gridDim.x) {
        const int nit = attn_unit_items(w, u);
        for (int half = 0; half < nit && ok; ++half) {
          const AttnItem it = attn_item(a, w, u, half);
          const int slot_q = ((it.hd / a.nhi) * 3 + 0) * a.nhi + it.hd % a.nhi;
          for (int x = 0; x < it.ntiles; ++x) {
            // tile x's Q buffer is free once its previous item's last Q K^T has completed
            if (nq[x] > 0 && !mbar_wait(bar(B_Q_EMPTY + x), static_cast<uint32_t>(nq[x] - 1) & 1u, abort_flag, err,
                                        a.err_site + 11)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(B_Q_FULL + x), kTile);
            const int p0 = (it.q0 + x) * kAttnBlk;
            tma_load_4d(sQ + x * kTile, &tmQKV, bar(B_Q_FULL + x), 0, slot_q, p0, it.sq);
            tma_load_4d(sQ + x * kTile + kHalf, &tmQKV, bar(B_Q_FULL + x), 64, slot_q, p0, it.sq);
            ++nq[x];
          }
          const int slot_k = slot_q + a.nhi, slot_v = slot_q + 2 * a.nhi;
          for (int j = 0; j < it.nblk && ok; ++j) {
            const uint32_t r = gb + static_cast<uint32_t>(j);
            const int b = static_cast<int>(r & 1u);
            const int pos = j * kAttnBlk;
            // the slot is refilled once every tile that consumed its previous block has released it
            for (int x = 0; x < 2 && ok; ++x)
              if ((cons >> (2 * b + x)) & 1u)
                ok = mbar_wait(bar(B_K_EMPTY + 2 * x + b), ((upar >> (2 * b + x)) & 1u) ^ 1u, abort_flag, err,
                               a.err_site + 1);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(B_K_FULL + b), kTile);
            tma_load_4d(sK + b * kTile, &tmQKV, bar(B_K_FULL + b), 0, slot_k, pos, it.sq);
            tma_load_4d(sK + b * kTile + kHalf, &tmQKV, bar(B_K_FULL + b), 64, slot_k, pos, it.sq);
            for (int x = 0; x < 2 && ok; ++x)
              if ((cons >> (2 * b + x)) & 1u)
                ok = mbar_wait(bar(B_V_EMPTY + 2 * x + b), ((upar >> (2 * b + x)) & 1u) ^ 1u, abort_flag, err,
                               a.err_site + 2);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(B_V_FULL + b), kTile);
            tma_load_4d(sV + b * kTile, &tmQKV, bar(B_V_FULL + b), 0, slot_v, pos, it.sq);
            tma_load_4d(sV + b * kTile + kHalf, &tmQKV, bar(B_V_FULL + b), 64, slot_v, pos, it.sq);
            // tile 0 consumes key blocks 0 .. q0, tile 1 (if any) every block of the item
            const uint32_t users = (j <= it.q0 ? 1u : 0u) | (it.ntiles == 2 ? 2u : 0u);
            cons = (cons & ~(3u << (2 * b))) | (users << (2 * b));
            upar ^= users << (2 * b);
          }
          gb += static_cast<uint32_t>(it.nblk);
        }
      }
      if (!ok) {
        // let the copies still in flight land before the CTA leaves
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 100000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == kAttnIssuer1) {
    if (lane == 0) {
      // ---------------- MMA issuer of tile x
      const uint32_t x = warp == 1 ? 0u : 1u;
      constexpr uint32_t kIdQK = idesc_bf16_f32(kAttnBlk, kAttnBlk, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(kAttnBlk, kAttnD, false, true);
      // Shared-memory descriptors are built once; a K step adds its byte offset / 16 to the start
      // address field (bits 0-13: shared addresses below 256 KiB never carry out of it).
      const uint64_t dQ = sdesc_sw128(sQ + x * kTile, 16, 1024), dK0 = sdesc_sw128(sK, 16, 1024),
                     dV0 = sdesc_sw128(sV, kHalf, 1024);
      const uint32_t tS = tmem_base + 128u * x, tO = tmem_base + 256u + 128u * x;
      // S_x = Q_x K^T (K in ring slot kb) into TMEM columns 128 x
      auto qk = [=](uint32_t kb) {
        const uint64_t dk = dK0 + ((static_cast<uint64_t>(kb) * kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kAttnD / 16; ++kk) {
          const uint64_t off = (static_cast<uint64_t>(kk >> 2) * kHalf + static_cast<uint64_t>(kk & 3) * 32u) >> 4;
          umma_bf16(tS, dQ + off, dk + off, kIdQK, static_cast<uint32_t>(kk != 0));
        }
      };
      // O_x (+)= P_x V (V in ring slot vb); A = P_x from TMEM (8 columns of bf16 pairs per K step of
      // 16); B = V, MN-major: its two 64-column panels of d sit kHalf apart, 8-row groups of positions
      // 1024 bytes apart
      auto pv = [=](uint32_t vb, bool first) {
        const uint64_t dv = dV0 + ((static_cast<uint64_t>(vb) * kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kAttnBlk / 16; ++kk)
          umma_bf16_tmem_a(tO, tS + 8u * kk, dv + ((static_cast<uint64_t>(kk) * 2048u) >> 4), kIdPV,
                           static_cast<uint32_t>(!first || kk != 0));
      };
      uint32_t gb = 0;  // ring position of the item's key block 0
      // bit 0: parity of the items so far in which tile x took part; bit 1: there was one;
      // bit 2: parity of the key blocks handed over so far (phase of P_FULL); bit 3: parity of the
      // turns received (phase of B_TURN + x)
      uint32_t st = 0;
      int prev_nt = 0;  // tiles of the previous item
      bool ok = true;
      // this issuer's turn: wait for the other issuer to hand it over
      auto take_turn = [&](bool needed) -> bool {
        if (!needed) return true;
        if (!mbar_wait(bar(B_TURN + x), (st >> 3) & 1u, abort_flag, err, a.err_site + 13)) return false;
        st ^= 8u;
        return true;
      };
      for (int u = blockIdx.x; u < w.units && ok; u += gridDim.x) {
        const int nit = attn_unit_items(w, u);
        for (int half = 0; half < nit && ok; ++half) {
          const AttnItem it = attn_item(a, w, u, half);
          const int nt = it.ntiles;
          if (static_cast<int>(x) >= nt) {  // a last query block of its own: tile 0 only
            gb += static_cast<uint32_t>(it.nblk);
            prev_nt = nt;
            continue;
          }
          const int q0 = it.q0, qlast = q0 + static_cast<int>(x);  // tile x attends to key blocks 0 .. qlast
          // the item's first product S_x = Q_x K_0^T; tile 0 after the previous item's last products
          // (tile 1's if it had two tiles), tile 1 after tile 0's first product
          if (!mbar_wait(bar(B_Q_FULL + x), st & 1u, abort_flag, err, a.err_site + 5) ||
              !mbar_wait(bar(B_K_FULL + (gb & 1u)), (gb >> 1) & 1u, abort_flag, err, a.err_site + 3) ||
              !take_turn(x == 0 ? prev_nt == 2 : true)) {
            ok = false;
            break;
          }
          tc_fence_after();
          qk(gb & 1u);
          if (nt == 2) mbar_arrive(bar(B_TURN + (x ^ 1u)));
          umma_commit(bar(B_S_FULL + x));
          umma_commit(bar(B_K_EMPTY + 2 * x + (gb & 1u)));
          if (qlast == 0) umma_commit(bar(B_Q_EMPTY + x));
          for (int j = 0; j <= qlast && ok; ++j) {
            const uint32_t r = gb + static_cast<uint32_t>(j), r1 = r + 1u;
            // the waits that are usually over first, the softmax hand-off (the critical path) last
            if (!mbar_wait(bar(B_V_FULL + (r & 1u)), (r >> 1) & 1u, abort_flag, err, a.err_site + 7) ||
                (j < qlast &&
                 !mbar_wait(bar(B_K_FULL + (r1 & 1u)), (r1 >> 1) & 1u, abort_flag, err, a.err_site + 3)) ||
                // O_x is overwritten by the item's first product: the previous item's O_x must be read
                (j == 0 && (st & 2u) &&
                 !mbar_wait(bar(B_O_FREE + x), (st & 1u) ^ 1u, abort_flag, err, a.err_site + 12)) ||
                // tile 0 takes its turn in every block of a two-tile item, tile 1 in every block but
                // its last (which follows its own products of block q0)
                !take_turn(nt == 2 && (x == 0 || j <= q0)) ||
                // P_FULL completes once per key block the tile processes, in this order; it is the
                // critical path, so it is polled rather than waited on with a suspending try_wait
                !mbar_poll(bar(B_P_FULL + x), (st >> 2) & 1u, abort_flag, err, a.err_site + 6)) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv(r & 1u, j == 0);
            // S_x = Q_x K_{j+1}^T overwrites P_x only after the product above (issue order)
            if (j < qlast) qk(r1 & 1u);
            // hand the turn over, unless this issuer's own products of block q0 + 1 come next
            if (nt == 2 && (x == 0 || j != q0)) mbar_arrive(bar(B_TURN + (x ^ 1u)));
            umma_commit(bar(B_PV_DONE + x));
            umma_commit(bar(B_V_EMPTY + 2 * x + (r & 1u)));
            st ^= 4u;
            if (j < qlast) {
              umma_commit(bar(B_S_FULL + x));
              umma_commit(bar(B_K_EMPTY + 2 * x + (r1 & 1u)));
              if (j + 1 == qlast) umma_commit(bar(B_Q_EMPTY + x));  // its Q buffer is free
            }
          }
          st = (st ^ 1u) | 2u;
          gb += static_cast<uint32_t>(it.nblk);
          prev_nt = nt;
        }
      }
      // every MMA this thread issued has completed once its drain barrier flips
      umma_commit(bar(B_DRAIN + x));
      attn_wait_drain(bar(B_DRAIN + x), 0);
    }
    __syncwarp();
  } else {
    // ---------------- softmax warps: tile x, query row `row` of the tile
    const int x = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lq = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + lq + 128u * x, tO = tmem_base + lq + 256u + 128u * x;
    const uint32_t obox = sO + static_cast<uint32_t>(warp - 2) * kOBox;
    uint32_t cb = 0;  // key blocks this tile has processed (phase of S_FULL, P_FULL, PV_DONE)
    bool ok = true;
    for (int u = blockIdx.x; u < w.units && ok; u += gridDim.x) {
      const int nit = attn_unit_items(w, u);
      for (int half = 0; half < nit && ok; ++half) {
        const AttnItem it = attn_item(a, w, u, half);
        if (x >= it.ntiles) continue;
        const int qblk = it.q0 + x;
        const int q_pos = qblk * kAttnBlk + row;
        float m_run = -INFINITY, l_run = 0.0f;
        for (int j = 0; ok && j <= qblk; ++j, ++cb) {
          ok = mbar_wait(bar(B_S_FULL + x), cb & 1u, abort_flag, err, a.err_site + 8);
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
          for (int c = 0; c < 128; c += 2)
            m8[(c >> 1) & 7] = max3(m8[(c >> 1) & 7], __uint_as_float(sr[c >> 5][c & 31]),
                                    __uint_as_float(sr[c >> 5][(c & 31) + 1]));
#pragma unroll
          for (int k = 4; k > 0; k >>= 1)
#pragma unroll
            for (int i = 0; i < k; ++i) m8[i] = fmaxf(m8[i], m8[i + k]);
          // Running maximum in the log2 domain (the scale log2(e) / sqrt(d) is positive).  It is
          // raised only when some row of the warp would exceed it by more than 8 (p <= 2^8
          // otherwise, harmless in fp32 and bf16); O and the sum are then rescaled by alpha.
          // Numerator and denominator always use the same maximum, so the result is unchanged.
          const float cand = fmaxf(m_run, m8[0] * a.scale_log2);
          const bool raise = __any_sync(0xFFFFFFFFu, cand > m_run + 8.0f) || j == 0;
          const float mx = raise ? cand : m_run;
          const float alpha = raise ? ex2_approx(m_run - mx) : 1.0f;  // 0 on the first block (m_run = -inf)
          const float nmx = -mx;
          // p = 2^(s scale - max), summed in fp32 and rounded to bf16 pairs as it is produced, so
          // that only the 64 packed registers stay live across the wait below
          // (columns 2c, 2c + 1 as one pair: l8[k] sums the columns e with e % 8 = k, as four pairs)
          uint64_t l4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) l4[k] = f2(0.0f, 0.0f);
          const uint64_t sc2 = f2(a.scale_log2, a.scale_log2), nmx2 = f2(nmx, nmx);
          uint32_t pk[2][32];
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int e = 2 * c;
            float y0, y1;
            f2_split(fma_f2(f2(__uint_as_float(sr[e >> 5][e & 31]), __uint_as_float(sr[e >> 5][(e & 31) + 1])), sc2,
                            nmx2),
                     y0, y1);
            const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
            l4[c & 3] = add_f2(l4[c & 3], f2(p0, p1));
            pk[c >> 5][c & 31] = pack_bf16x2(p0, p1);
          }
          float l8[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) f2_split(l4[k], l8[2 * k], l8[2 * k + 1]);
#pragma unroll
          for (int k = 4; k > 0; k >>= 1)
#pragma unroll
            for (int i = 0; i < k; ++i) l8[i] += l8[i + k];
          l_run = l_run * alpha + l8[0];
          m_run = mx;
          // P_x -> the first 64 columns of S_x.  They and O_x are free: the previous block's
          // O_x += P_x V was issued before this block's S_x = Q_x K^T by the same thread, so it has
          // completed once S_FULL has (a commit arrives when all earlier operations of its thread have)
          tmem_st32(tS, pk[0]);
          tmem_st32(tS + 32u, pk[1]);
          if (j > 0 && raise) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + static_cast<uint32_t>(c * 32), o);
              tmem_ld_wait();
              const uint64_t al2 = f2(alpha, alpha);
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float v0, v1;
                f2_split(mul_f2(f2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), al2), v0, v1);
                o[e] = __float_as_uint(v0);
                o[e + 1] = __float_as_uint(v1);
              }
              tmem_st32(tO + static_cast<uint32_t>(c * 32), o);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_P_FULL + x));
        }
        if (!ok) break;
        // ---- end of the item: O_x / sum -> bf16, written out 64 columns at a time through this
        // warp's staging box (32 rows x 64 columns, 128-byte swizzle)
        ok = mbar_wait(bar(B_PV_DONE + x), (cb - 1u) & 1u, abort_flag, err, a.err_site + 10);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = 1.0f / l_run;
        const int p0 = qblk * kAttnBlk + quarter * 32;  // rows past the sequence end are clipped
        const int slot_o = it.hd;
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t o[2][32];
          tmem_ld32(tO + static_cast<uint32_t>(h2 * 64), o[0]);
          tmem_ld32(tO + static_cast<uint32_t>(h2 * 64 + 32), o[1]);
          tmem_ld_wait();
          if (h2 == 1) {
            // O_x is read: the next item's first product may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_O_FREE + x));
          }
          if (lane == 0) bulk_wait_group_read<0>();  // the box's previous store has read it
          __syncwarp();
          const uint32_t box = obox + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t unit = static_cast<uint32_t>(c * 4 + k);
              st_shared_v4(box + ((unit ^ (static_cast<uint32_t>(lane) & 7u)) << 4),
                           pack_bf16x2(__uint_as_float(o[c][8 * k]) * inv, __uint_as_float(o[c][8 * k + 1]) * inv),
                           pack_bf16x2(__uint_as_float(o[c][8 * k + 2]) * inv, __uint_as_float(o[c][8 * k + 3]) * inv),
                           pack_bf16x2(__uint_as_float(o[c][8 * k + 4]) * inv, __uint_as_float(o[c][8 * k + 5]) * inv),
                           pack_bf16x2(__uint_as_float(o[c][8 * k + 6]) * inv, __uint_as_float(o[c][8 * k + 7]) * inv));
            }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && p0 < a.seq) {
            tma_store_4d(&tmO, obox, h2 * 64, slot_o, p0, it.sq);
            bulk_commit_group();
          }
          __syncwarp();
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();  // every store of this warp has completed
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kAttnTmemCols);
  }
}

cudaError_t launch_attention(const CUtensorMap& tm_qkv, const CUtensorMap& tm_o, const AttnArgs& a, int nseq,
                             int max_ctas, cudaStream_t st) {
  if (nseq == 0 || a.n_qblk == 0 || a.heads == 0) return cudaSuccess;
  // per device: the shared-memory opt-in is an attribute of the kernel on one device (0 = not set up)
  static std::atomic<int> sms_of[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int sms = sms_of[dev].load(std::memory_order_acquire);
  if (sms == 0) {
    e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_of[dev].store(sms, std::memory_order_release);
  }
  const int n_pairs = (a.n_qblk + 1) / 2;
  const int64_t units = int64_t((n_pairs + 1) / 2) * a.heads * nseq;
  const int cap = max_ctas > 0 ? max_ctas : sms;
  const int grid = static_cast<int>(units < cap ? units : cap);
  attention_kernel<<<grid, kAttnThreads, kAttnSmem, st>>>(tm_qkv, tm_o, a, nseq);
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
