// Backward of the sparse MQA-mode attention over a fixed selection
// (freezhihu.org/question/1978819912970555965 §2.3.2: in the sparse training stage the main model
// is optimised through DSA, so the gradient flows through the attention over the selected rows).
//
// Forward, per token t and head h over its selected latent rows c_s (s in S_t):
//     z[h,s] = scale * q[h] . c_s,   p = softmax_s(z),   o[h] = sum_s p[h,s] c_s[0:512]
// Backward, given do = dL/do and the forward's lse:
//     p[h,s]  = exp(z[h,s] - lse[h])                 (recomputed)
//     dp[h,s] = do[h] . c_s[0:512],   D[h] = do[h] . o[h]
//     ds[h,s] = p[h,s] (dp[h,s] - D[h])
//     dq[h]   = scale * sum_s ds[h,s] c_s
//     dc_s   += scale * sum_h ds[h,s] q[h]  +  [sum_h p[h,s] do[h], 0]   (added over every token)
//
// Per token the operands are Q [128 x 576] and dO [128 x 512] (272 KB together, more than one SM's
// shared memory) and the dq accumulator is [128 x 576] fp32 (576 tensor-memory columns, more than
// one SM has).  So a token runs on a cluster of two CTAs, and the selected rows go in 32-key tiles:
//
//   rank 0 ("query" CTA): Q in shared memory; gathers the tiles' full 576-dim rows;
//     S = Q K^T (tensor cores) -> P = exp2(S scale log2e - lse log2e) by four row warps, written
//     straight into rank 1's shared memory; receives dS from rank 1; dq[:, 320:576] += dS K[:, 320:576];
//     dc^T[dims, keys] = Q^T dS for five 128-dim blocks (M = 128 dims, so every product keeps the
//     128-lane accumulator layout), drained by four epilogue warps into dkv with fp32 atomics.
//   rank 1 ("output-gradient" CTA): dO in shared memory; gathers the tiles' first 512 dims;
//     dP = dO V^T -> dS = P (dP - D) by four row warps (D per head from dO and the forward's O),
//     written into its own and rank 0's shared memory; dq[:, 0:320] += dS V[:, 0:320];
//     dv^T = dO^T P for four 128-dim blocks into dkv[:, 0:512].
//
// In each CTA one warp issues S (or dP) and the dq products and a second warp issues the dc^T (or
// dv^T) products, so that the two chains of tensor-core instructions are issued side by side.
//
// Persistent: one cluster per SM pair takes every (number of clusters)-th token.  Every wait is
// bounded (the kernel records DSA_ERR_DEVICE_TIMEOUT and leaves); an out-of-range position is
// skipped and reported as DSA_ERR_DEVICE_RANGE.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

using namespace attn;

constexpr int kKT = 32;                        // keys per tile
constexpr int kProdWarps = 8;                  // warps 1..8 gather
constexpr int kProducers = kProdWarps * 32;
constexpr int kRowWarp0 = 1 + kProdWarps;      // warps 9..12: one head row per thread
constexpr int kEpiWarp0 = kRowWarp0 + 4;       // warps 13..16: dc blocks and dq read-out
constexpr int kCreditWarp = kEpiWarp0 + 4;     // warp 17: Q / dO loads and slot credits
constexpr int kDcWarp = kCreditWarp + 1;       // warp 18: issues the dc^T / dv^T products
constexpr int kThreads = 32 * (kDcWarp + 1);
constexpr int kDL = 576, kDV = 512;
constexpr int kBox = 128 * 128;                // [128 rows x 64 dims] bf16, 128B-swizzled (TMA box)
constexpr int kBlk = kKT * 128;                // [32 rows x 64 dims] bf16, 128B-swizzled
constexpr int kKStage = 9 * kBlk, kVStage = 8 * kBlk;
constexpr int kSlot = 128 * kKT * 2;           // [128 heads x 32 keys] bf16, 64B-swizzled
constexpr int kStages = 2;
constexpr int kDqSplit = 320;                  // dq dims [0, 320) on rank 1, [320, 576) on rank 0
constexpr int kNDc0 = 5, kNDc1 = 4;            // 128-dim dc^T blocks per tile (576 -> 640 padded, 512)
// rank 0 shared memory
constexpr int kOffQ = 0, kOffK = 9 * kBox, kOffDs0 = kOffK + kStages * kKStage, kEnd0 = kOffDs0 + kSlot;
// rank 1 shared memory
constexpr int kOffDO = 0, kOffV = 8 * kBox, kOffP = kOffV + kStages * kVStage, kOffDs1 = kOffP + 2 * kSlot;
constexpr int kEnd1 = kOffDs1 + 2 * kSlot;
constexpr int kSmem = (kEnd0 > kEnd1 ? kEnd0 : kEnd1) + 1024;
// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDq0 = 64, kColDc0 = kColDq0 + (kDL - kDqSplit);   // rank 0: 480 used
constexpr uint32_t kColDp = 0, kColDq1 = 64, kColDc1 = kColDq1 + kDqSplit;           // rank 1: 512 used
static_assert(kColDc0 + kNDc0 * kKT <= kTmemCols && kColDc1 + kNDc1 * kKT <= kTmemCols, "TMEM budget");
static_assert(kSmem <= 227 * 1024 - 1024, "shared memory budget");
// The last rank-0 dc^T block covers dims 512..639 and so reads 64 rows past Q: those land in the K
// ring (inside this CTA's shared memory); their results are discarded.
static_assert(kOffQ + 10 * kBox <= kEnd0, "the padded Q^T block stays inside shared memory");

struct Bars {
  // rank 0
  uint64_t k_full[kStages], k_empty[kStages], s_full[2], s_empty[2], q_full, q_free;
  uint64_t p_empty[2];      // credit from rank 1: its P slot may be overwritten
  uint64_t ds_full;         // rank 1's bulk copy of dS into this CTA's slot landed (armed with its bytes)
  uint64_t ds_consumed;     // this CTA's products reading that slot completed
  // rank 1
  uint64_t v_full[kStages], v_empty[kStages], dp_full[2], dp_empty[2], do_full, do_free;
  uint64_t p_full[2];       // rank 0's 128 row threads wrote P into this slot
  uint64_t p_consumed[2];   // the row threads read it (128) and the products reading it completed (1)
  uint64_t dsl_full[2], dsl_empty[2];
  uint64_t ds_peer_empty;   // credit from rank 0: its dS slot may be overwritten
  // both
  uint64_t dc_full[kNDc0], dc_empty[kNDc0], dq_full, dq_free, mma_done;
};

__device__ __forceinline__ uint32_t baddr(const uint64_t& b) { return ptx::smem_addr(&b); }

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) break;
  }
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, const BwdArgs& a) {
  return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, a.status, a.limit_ns));
}
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  const BwdArgs& a) {
  return __all_sync(0xffffffffu, ptx::mbar_wait_cluster(bar, parity, abort_flag, a.status, a.limit_ns));
}

// Latent row of selection entry s (contiguous rows), or -1 for an empty or out-of-range slot.
__device__ __forceinline__ int64_t sel_row(const BwdArgs& a, int32_t s, bool* range_err) {
  if (s < 0) return -1;
  if (s >= a.n_kv_rows) {
    *range_err = true;
    return -1;
  }
  return s;
}

// 32-key tiles of token t's selection (valid slots come first), by the whole warp.
__device__ __forceinline__ int tiles_of(const BwdArgs& a, int t) {
  const int n = first_empty_slot(a.idx + static_cast<int64_t>(t) * a.k, a.k);
  return (n + kKT - 1) / kKT;
}

// Shared-memory descriptors (tcgen05 format).  K-major 128B-swizzled operands step 32 bytes per K16;
// MN-major ones step 16 rows.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) { return ptx::smem_desc(addr, 16, 1024, ptx::kLayoutSw128); }
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t addr, uint32_t lbo) {
  return ptx::smem_desc(addr, lbo, 1024, ptx::kLayoutSw128);
}
__device__ __forceinline__ uint64_t desc_sw64(uint32_t addr) { return ptx::smem_desc(addr, 16, 512, ptx::kLayoutSw64); }
__device__ __forceinline__ uint64_t desc_sw64_mn(uint32_t addr) { return ptx::smem_desc(addr, 8192, 512, ptx::kLayoutSw64); }

// Byte offset of 16-byte chunk c (0..3) of row r in a [rows x 64 B] 64B-swizzled slot.
__device__ __forceinline__ uint32_t slot_off(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }

// Selection entry of this lane's key in tile i of a row (-1 past the row's slots).
__device__ __forceinline__ int32_t sel_entry(const BwdArgs& a, const int32_t* idx_row, int i) {
  const int slot = i * kKT + (threadIdx.x & 31);
  return slot < a.k ? __ldg(idx_row + slot) : -1;
}

// Gather of a tile: NBLK 64-dim blocks of each of its 32 selected rows into a 128B-swizzled stage;
// lane l holds the selection entry s of key l.  Producer warp pw copies rows pw, pw + 8, pw + 16,
// pw + 24; an empty or out-of-range slot copies `fallback` (a row the token attends; its key is
// masked to P = 0 downstream).
template <int NBLK>
__device__ __forceinline__ void gather_tile(const BwdArgs& a, int32_t s, uint32_t dst, int pw, int lane,
                                            int64_t fallback) {
  constexpr int kChunks = NBLK * 8;
  bool unused = false;
  const int64_t pr = sel_row(a, s, &unused);
  const uint16_t* base = a.kv + (pr < 0 ? fallback : pr) * kDL;
  for (int r = pw; r < kKT; r += kProdWarps) {
    const uint16_t* src = reinterpret_cast<const uint16_t*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(base), r));
    const uint32_t drow = dst + r * 128;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int cc = lane + 32 * j;
      if (cc < kChunks) ptx::cp_async16_n<16>(drow + (cc >> 3) * kBlk + (((cc & 7) ^ (r & 7)) << 4), src + cc * 8);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_bwd_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap qmap,
                           const __grid_constant__ CUtensorMap domap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ Bars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag_s;

  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const int cl = blockIdx.x >> 1, n_cl = gridDim.x >> 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &abort_flag_s;
  const uint32_t sbase = ptx::smem_addr(smem);
  const float scale = a.scale;
  const float scale_log2 = a.scale * 1.4426950408889634f;

  if (tid == 0) {
    if (rank == 0) {
      for (int s = 0; s < kStages; ++s) {
        ptx::mbar_init(baddr(bars.k_full[s]), kProducers);
        ptx::mbar_init(baddr(bars.k_empty[s]), 1);
      }
      for (int b = 0; b < 2; ++b) {
        ptx::mbar_init(baddr(bars.s_full[b]), 1);
        ptx::mbar_init(baddr(bars.s_empty[b]), 128);
        ptx::mbar_init(baddr(bars.p_empty[b]), 1);
      }
      ptx::mbar_init(baddr(bars.q_full), 1);
      ptx::mbar_init(baddr(bars.q_free), 2);         // both MMA warps read Q
      ptx::mbar_init(baddr(bars.ds_full), 1);
      ptx::mbar_init(baddr(bars.ds_consumed), 2);    // the dq product and the dc^T products
      ptx::mbar_arrive_expect_tx(baddr(bars.ds_full), kSlot);  // armed for the first copy
    } else {
      for (int s = 0; s < kStages; ++s) {
        ptx::mbar_init(baddr(bars.v_full[s]), kProducers);
        ptx::mbar_init(baddr(bars.v_empty[s]), 1);
      }
      for (int b = 0; b < 2; ++b) {
        ptx::mbar_init(baddr(bars.dp_full[b]), 1);
        ptx::mbar_init(baddr(bars.dp_empty[b]), 128);
        ptx::mbar_init(baddr(bars.p_full[b]), 128);
        ptx::mbar_init(baddr(bars.p_consumed[b]), 129);
        ptx::mbar_init(baddr(bars.dsl_full[b]), 128);
        ptx::mbar_init(baddr(bars.dsl_empty[b]), 1);
      }
      ptx::mbar_init(baddr(bars.do_full), 1);
      ptx::mbar_init(baddr(bars.do_free), 2);        // both MMA warps read dO
      ptx::mbar_init(baddr(bars.ds_peer_empty), 1);
    }
    for (int j = 0; j < kNDc0; ++j) {
      ptx::mbar_init(baddr(bars.dc_full[j]), 1);
      ptx::mbar_init(baddr(bars.dc_empty[j]), 128);
    }
    ptx::mbar_init(baddr(bars.dq_full), 1);
    ptx::mbar_init(baddr(bars.dq_free), 128);
    ptx::mbar_init(baddr(bars.mma_done), 2);
    abort_flag_s = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_addr(&tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();  // both CTAs' barriers exist before any remote arrival or store
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t peer = rank ^ 1;

  if (warp == 0) {
    // ================================================================ MMA issue (one warp per CTA)
    int g = 0, nq = 0;
    bool ok = true;
    if (rank == 0) {
      constexpr uint32_t kIdS = ptx::instr_desc(128, kKT, 1, 1, 0, 0);
      constexpr uint32_t kIdDq = ptx::instr_desc(128, 256, 1, 1, 0, 1);
      const uint32_t q_s = sbase + kOffQ, ds_s = sbase + kOffDs0;
      for (int t = cl; ok && t < a.T; t += n_cl) {
        const int n = tiles_of(a, t);
        if (n == 0) continue;
        if (!warp_wait(baddr(bars.q_full), nq & 1, abort_flag, a)) break;
        ptx::tc_fence_after();
        // S(i) = Q K(i)^T into S buffer i % 2
        auto issue_s = [&](int i) -> bool {
          const int gi = g + i, st = gi % kStages, sb = gi & 1;
          if (!warp_wait(baddr(bars.k_full[st]), (gi / kStages) & 1, abort_flag, a) ||
              !warp_wait(baddr(bars.s_empty[sb]), ((gi >> 1) & 1) ^ 1, abort_flag, a))
            return false;
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint32_t kst = sbase + kOffK + st * kKStage;
#pragma unroll
          for (int f = 0; f < 36; ++f)
            ptx::mma_bf16_warp(tmem + kColS + sb * kKT, desc_sw128(q_s + (f >> 2) * kBox + (f & 3) * 32),
                               desc_sw128(kst + (f >> 2) * kBlk + (f & 3) * 32), kIdS, f > 0 ? 1u : 0u);
          ptx::mma_commit_warp(baddr(bars.s_full[sb]));
          return true;
        };
        if (!issue_s(0)) break;
        for (int i = 0; i < n; ++i) {
          const int gi = g + i, st = gi % kStages;
          if (i + 1 < n && !issue_s(i + 1)) {
            ok = false;
            break;
          }
          if (!warp_wait_cluster(baddr(bars.ds_full), gi & 1, abort_flag, a) ||
              (i == 0 && nq > 0 && !warp_wait(baddr(bars.dq_free), (nq - 1) & 1, abort_flag, a))) {
            ok = false;
            break;
          }
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          // dq[:, 320:576] += dS K(i)[:, 320:576]  (K rows read MN-major: dims 320.. = blocks 5..8)
          const uint32_t kst = sbase + kOffK + st * kKStage;
#pragma unroll
          for (int ks = 0; ks < kKT / 16; ++ks)
            ptx::mma_bf16_warp(tmem + kColDq0, desc_sw64(ds_s + ks * 32), desc_sw128_mn(kst + 5 * kBlk + ks * 16 * 128, kBlk),
                               kIdDq, (i > 0 || ks > 0) ? 1u : 0u);
          ptx::mma_commit_warp(baddr(bars.k_empty[st]));
          ptx::mma_commit_warp(baddr(bars.ds_consumed));  // (the dc^T products are the other warp's)
        }
        if (!ok) break;
        ptx::mma_commit_warp(baddr(bars.dq_full));
        ptx::mma_commit_warp(baddr(bars.q_free));
        g += n;
        ++nq;
      }
    } else {
      constexpr uint32_t kIdDp = ptx::instr_desc(128, kKT, 1, 1, 0, 0);
      constexpr uint32_t kIdDq256 = ptx::instr_desc(128, 256, 1, 1, 0, 1);
      constexpr uint32_t kIdDq64 = ptx::instr_desc(128, 64, 1, 1, 0, 1);
      const uint32_t do_s = sbase + kOffDO;
      for (int t = cl; ok && t < a.T; t += n_cl) {
        const int n = tiles_of(a, t);
        if (n == 0) continue;
        if (!warp_wait(baddr(bars.do_full), nq & 1, abort_flag, a)) break;
        ptx::tc_fence_after();
        // dP(i) = dO V(i)^T into dP buffer i % 2
        auto issue_dp = [&](int i) -> bool {
          const int gi = g + i, st = gi % kStages, pb = gi & 1;
          if (!warp_wait(baddr(bars.v_full[st]), (gi / kStages) & 1, abort_flag, a) ||
              !warp_wait(baddr(bars.dp_empty[pb]), ((gi >> 1) & 1) ^ 1, abort_flag, a))
            return false;
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint32_t vst = sbase + kOffV + st * kVStage;
#pragma unroll
          for (int f = 0; f < 32; ++f)
            ptx::mma_bf16_warp(tmem + kColDp + pb * kKT, desc_sw128(do_s + (f >> 2) * kBox + (f & 3) * 32),
                               desc_sw128(vst + (f >> 2) * kBlk + (f & 3) * 32), kIdDp, f > 0 ? 1u : 0u);
          ptx::mma_commit_warp(baddr(bars.dp_full[pb]));
          return true;
        };
        if (!issue_dp(0)) break;
        for (int i = 0; i < n; ++i) {
          const int gi = g + i, st = gi % kStages, ps = gi & 1;
          if (i + 1 < n && !issue_dp(i + 1)) {
            ok = false;
            break;
          }
          // dS(i) is in the local slot (its row threads had P(i) from rank 0 before writing it)
          if (!warp_wait(baddr(bars.dsl_full[ps]), (gi >> 1) & 1, abort_flag, a) ||
              (i == 0 && nq > 0 && !warp_wait(baddr(bars.dq_free), (nq - 1) & 1, abort_flag, a))) {
            ok = false;
            break;
          }
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint32_t vst = sbase + kOffV + st * kVStage, dsl = sbase + kOffDs1 + ps * kSlot;
          // dq[:, 0:320] += dS V(i)[:, 0:320]  (blocks 0..3 as one N = 256 product, block 4 as N = 64)
#pragma unroll
          for (int ks = 0; ks < kKT / 16; ++ks) {
            ptx::mma_bf16_warp(tmem + kColDq1, desc_sw64(dsl + ks * 32), desc_sw128_mn(vst + ks * 16 * 128, kBlk), kIdDq256,
                               (i > 0 || ks > 0) ? 1u : 0u);
            ptx::mma_bf16_warp(tmem + kColDq1 + 256, desc_sw64(dsl + ks * 32),
                               desc_sw128_mn(vst + 4 * kBlk + ks * 16 * 128, kBlk), kIdDq64, (i > 0 || ks > 0) ? 1u : 0u);
          }
          ptx::mma_commit_warp(baddr(bars.v_empty[st]));
          ptx::mma_commit_warp(baddr(bars.dsl_empty[ps]));  // (the dv^T products are the other warp's)
        }
        if (!ok) break;
        ptx::mma_commit_warp(baddr(bars.dq_full));
        ptx::mma_commit_warp(baddr(bars.do_free));
        g += n;
        ++nq;
      }
    }
    ptx::mma_commit_warp(baddr(bars.mma_done));
    drain_wait(baddr(bars.mma_done), 0, a.limit_ns);
  } else if (warp == kDcWarp) {
    // ================================================================ second MMA warp: the latent-row
    // gradient products, issued beside the S / dP and dq products of warp 0
    constexpr uint32_t kIdDc = ptx::instr_desc(128, kKT, 1, 1, 1, 1);
    int g = 0, nq = 0;
    bool ok = true;
    for (int t = cl; ok && t < a.T; t += n_cl) {
      const int n = tiles_of(a, t);
      if (n == 0) continue;
      if (!warp_wait(rank == 0 ? baddr(bars.q_full) : baddr(bars.do_full), nq & 1, abort_flag, a)) break;
      ptx::tc_fence_after();
      for (int i = 0; i < n; ++i) {
        const int gi = g + i, ps = gi & 1;
        // rank 0: dS(i) in this CTA's slot; rank 1: dS(i) in the local slot, written after P(i) arrived
        const bool got = rank == 0 ? warp_wait_cluster(baddr(bars.ds_full), gi & 1, abort_flag, a)
                                   : warp_wait(baddr(bars.dsl_full[ps]), (gi >> 1) & 1, abort_flag, a);
        if (!got) {
          ok = false;
          break;
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        const int nblk = rank == 0 ? kNDc0 : kNDc1;
        const uint32_t col = rank == 0 ? kColDc0 : kColDc1;
        const uint32_t lhs = sbase + (rank == 0 ? kOffQ : kOffDO);            // Q^T or dO^T, MN-major
        const uint32_t rhs = sbase + (rank == 0 ? kOffDs0 : kOffP + ps * kSlot);  // dS or P, MN-major
        for (int j = 0; j < nblk && ok; ++j) {
          // block j [dims 128j.., 32 keys]
          if (!warp_wait(baddr(bars.dc_empty[j]), (gi & 1) ^ 1, abort_flag, a)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            ptx::mma_bf16_warp(tmem + col + j * kKT, desc_sw128_mn(lhs + 2 * j * kBox + ks * 16 * 128, kBox),
                               desc_sw64_mn(rhs + ks * 16 * 64), kIdDc, ks > 0 ? 1u : 0u);
          ptx::mma_commit_warp(baddr(bars.dc_full[j]));
        }
        if (!ok) break;
        ptx::mma_commit_warp(rank == 0 ? baddr(bars.ds_consumed) : baddr(bars.p_consumed[ps]));
      }
      if (!ok) break;
      ptx::mma_commit_warp(rank == 0 ? baddr(bars.q_free) : baddr(bars.do_free));
      g += n;
      ++nq;
    }
    ptx::mma_commit_warp(baddr(bars.mma_done));
    drain_wait(baddr(bars.mma_done), 0, a.limit_ns);
  } else if (warp <= kProdWarps) {
    // ================================================================ row gathers
    const int pw = warp - 1;
    int g = 0;
    bool range_err = false;
    for (int t = cl; t < a.T; t += n_cl) {
      const int n = tiles_of(a, t);
      if (n == 0) continue;
      const int32_t* idx_row = a.idx + static_cast<int64_t>(t) * a.k;
      int64_t fallback = sel_row(a, __ldg(idx_row), &range_err);
      if (fallback < 0) fallback = 0;
      bool ok = true;
      int32_t s_next = sel_entry(a, idx_row, 0);  // each tile's entries are loaded a tile ahead
      for (int i = 0; i < n; ++i) {
        const int gi = g + i, st = gi % kStages;
        const int32_t s_cur = s_next;
        if (i + 1 < n) s_next = sel_entry(a, idx_row, i + 1);
        if (rank == 0) {
          if (!warp_wait(baddr(bars.k_empty[st]), ((gi / kStages) & 1) ^ 1, abort_flag, a)) {
            ok = false;
            break;
          }
          gather_tile<9>(a, s_cur, sbase + kOffK + st * kKStage, pw, lane, fallback);
          ptx::cp_async_arrive_noinc(baddr(bars.k_full[st]));
        } else {
          if (!warp_wait(baddr(bars.v_empty[st]), ((gi / kStages) & 1) ^ 1, abort_flag, a)) {
            ok = false;
            break;
          }
          gather_tile<8>(a, s_cur, sbase + kOffV + st * kVStage, pw, lane, fallback);
          ptx::cp_async_arrive_noinc(baddr(bars.v_full[st]));
        }
      }
      if (!ok) break;
      g += n;
    }
    ptx::cp_async_wait<0>();  // nothing of this thread's may still be in flight when the CTA exits
    (void)range_err;          // reported by the row warps, which see the same slots
  } else if (warp < kEpiWarp0) {
    // ================================================================ row warps: one head per thread
    const int h = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int g = 0, nq = 0;
    bool ok = true, range_err = false;
    if (rank == 0) {
      // ---- P = exp2(S scale log2e - lse log2e) over valid keys, into rank 1's P slot
      const uint32_t peer_p = ptx::map_to_rank(sbase + kOffP, peer);
      for (int t = cl; ok && t < a.T; t += n_cl) {
        const int n = tiles_of(a, t);
        if (n == 0) continue;
        const int32_t* idx_row = a.idx + static_cast<int64_t>(t) * a.k;
        const float lse2 = h < a.H ? a.lse[static_cast<int64_t>(t) * a.H + h] * 1.4426950408889634f : INFINITY;
        int32_t s_next = sel_entry(a, idx_row, 0);
        for (int i = 0; i < n; ++i) {
          const int gi = g + i, sb = gi & 1, ps = gi & 1;
          const int32_t sidx = s_next;
          if (i + 1 < n) s_next = sel_entry(a, idx_row, i + 1);
          if (!warp_wait(baddr(bars.s_full[sb]), (gi >> 1) & 1, abort_flag, a)) {
            ok = false;
            break;
          }
          uint32_t sv[32];
          ptx::tc_fence_after();
          ptx::tmem_ld32(tmem + kColS + sb * kKT + lane_base, sv);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          ptx::mbar_arrive(baddr(bars.s_empty[sb]));
          const uint32_t vm = __ballot_sync(0xffffffffu, sel_row(a, sidx, &range_err) >= 0);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = ((vm >> e) & 1u) ? fast_exp2(__uint_as_float(sv[e]) * scale_log2 - lse2) : 0.f;
            const float p1 = ((vm >> (e + 1)) & 1u) ? fast_exp2(__uint_as_float(sv[e + 1]) * scale_log2 - lse2) : 0.f;
            pk[e / 2] = pack_bf16(p0, p1);
          }
          if (!ptx::mbar_wait_cluster(baddr(bars.p_empty[ps]), ((gi >> 1) & 1) ^ 1, abort_flag, a.status, a.limit_ns)) {
            ok = false;
          }
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          const uint32_t dst = peer_p + ps * kSlot;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            ptx::st_cluster_v4(dst + slot_off(h, c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          ptx::fence_proxy_async_cluster();
          ptx::mbar_arrive_cluster(ptx::map_to_rank(baddr(bars.p_full[ps]), peer));
        }
        g += n;
        ++nq;
      }
    } else {
      // ---- dS = P (dP - D) into the local slot and rank 0's slot.  These 128 threads meet at named
      // barriers (unbounded), so they leave only together: a failed wait is voted on at the next
      // barrier instead of breaking out alone.
      const uint32_t peer_ds = ptx::map_to_rank(sbase + kOffDs0, peer);
      const uint8_t* dos = smem + kOffDO + h * 128;
      for (int t = cl; ok && t < a.T; t += n_cl) {
        const int n = tiles_of(a, t);
        if (n == 0) continue;
        // D = dO[h] . O[h] (dO from shared memory, the forward's O from global memory)
        const bool d_ok = warp_wait(baddr(bars.do_full), nq & 1, abort_flag, a);
        float D = 0.f;
        if (d_ok && h < a.H) {
          const uint4* orow = reinterpret_cast<const uint4*>(a.out + (static_cast<int64_t>(t) * a.H + h) * kDV);
#pragma unroll 2
          for (int b = 0; b < 8; ++b) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 x = *reinterpret_cast<const uint4*>(dos + b * kBox + ((c ^ (h & 7)) << 4));
              const uint4 y = __ldg(orow + b * 8 + c);
              const __nv_bfloat162* xv = reinterpret_cast<const __nv_bfloat162*>(&x);
              const __nv_bfloat162* yv = reinterpret_cast<const __nv_bfloat162*>(&y);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 xf = __bfloat1622float2(xv[e]), yf = __bfloat1622float2(yv[e]);
                D = fmaf(xf.x, yf.x, D);
                D = fmaf(xf.y, yf.y, D);
              }
            }
          }
        }
        for (int i = 0; i < n; ++i) {
          const int gi = g + i, pb = gi & 1, ps = gi & 1;
          bool fail = !d_ok;
          uint32_t dv[32];
          if (!fail && warp_wait(baddr(bars.dp_full[pb]), (gi >> 1) & 1, abort_flag, a)) {
            ptx::tc_fence_after();
            ptx::tmem_ld32(tmem + kColDp + pb * kKT + lane_base, dv);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(baddr(bars.dp_empty[pb]));
          } else {
            fail = true;
          }
          uint32_t pk[16];
          if (!fail && warp_wait_cluster(baddr(bars.p_full[ps]), (gi >> 1) & 1, abort_flag, a)) {
            const uint8_t* prow = smem + kOffP + ps * kSlot;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 x = *reinterpret_cast<const uint4*>(prow + slot_off(h, c));
              pk[4 * c] = x.x; pk[4 * c + 1] = x.y; pk[4 * c + 2] = x.z; pk[4 * c + 3] = x.w;
            }
            ptx::mbar_arrive(baddr(bars.p_consumed[ps]));
          } else {
            fail = true;
          }
          if (!fail) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[e]));
              pk[e] = pack_bf16(p.x * (__uint_as_float(dv[2 * e]) - D), p.y * (__uint_as_float(dv[2 * e + 1]) - D));
            }
          }
          // The local slot feeds this CTA's dq product; one bulk copy of it then feeds rank 0.  Before
          // the slot is rewritten, its products (dsl_empty) and the copy of two tiles ago (the
          // copying thread's bulk group) must have read it.
          if (!fail)
            fail = !ptx::mbar_wait(baddr(bars.dsl_empty[ps]), ((gi >> 1) & 1) ^ 1, abort_flag, a.status, a.limit_ns);
          if (h == 0) ptx::bulk_wait_read<1>();
          if (ptx::named_sync_or(1, 128, fail || *abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dsl = smem + kOffDs1 + ps * kSlot;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(dsl + slot_off(h, c)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive(baddr(bars.dsl_full[ps]));
          ptx::named_sync(2, 128);
          if (h == 0) {
            // a failed wait raises the abort flag, which the next vote picks up
            if (ptx::mbar_wait_cluster(baddr(bars.ds_peer_empty), (gi & 1) ^ 1, abort_flag, a.status, a.limit_ns)) {
              ptx::bulk_copy_to_cluster(peer_ds, ptx::smem_addr(dsl), kSlot, ptx::map_to_rank(baddr(bars.ds_full), peer));
              ptx::bulk_commit();
            }
          }
        }
        if (ok) {
          g += n;
          ++nq;
        }
      }
      if (h == 0) ptx::bulk_wait_all<0>();  // every copy has landed in rank 0 before either CTA exits
    }
    if (range_err) atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE);
  } else if (warp < kCreditWarp) {
    // ================================================================ epilogue: dc blocks, then dq
    const int q4 = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const int h = q4 * 32 + lane;
    const int nblk = rank == 0 ? kNDc0 : kNDc1;
    const uint32_t col_dc = rank == 0 ? kColDc0 : kColDc1;
    const float fac = rank == 0 ? scale : 1.f;        // key role carries the softmax scale
    const int dq0 = rank == 0 ? kDqSplit : 0, dqn = rank == 0 ? kDL - kDqSplit : kDqSplit;
    const uint32_t col_dq = rank == 0 ? kColDq0 : kColDq1;
    int g = 0, nq = 0;
    bool ok = true;
    for (int t = cl; ok && t < a.T; t += n_cl) {
      const int n = tiles_of(a, t);
      uint16_t* dq_row = a.dq + (static_cast<int64_t>(t) * a.H + h) * kDL + dq0;
      if (n == 0) {
        if (h < a.H)
          for (int c = 0; c < dqn; c += 8) *reinterpret_cast<uint4*>(dq_row + c) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int32_t* idx_row = a.idx + static_cast<int64_t>(t) * a.k;
      int32_t s_next = sel_entry(a, idx_row, 0);
      for (int i = 0; ok && i < n; ++i) {
        const int gi = g + i;
        bool unused = false;
        const int64_t my_row = sel_row(a, s_next, &unused);
        if (i + 1 < n) s_next = sel_entry(a, idx_row, i + 1);
        for (int j = 0; j < nblk; ++j) {
          if (!warp_wait(baddr(bars.dc_full[j]), gi & 1, abort_flag, a)) {
            ok = false;
            break;
          }
          uint32_t v[32];
          ptx::tc_fence_after();
          ptx::tmem_ld32(tmem + col_dc + j * kKT + lane_base, v);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          ptx::mbar_arrive(baddr(bars.dc_empty[j]));
          const int dim0 = j * 128 + q4 * 32;      // this warp's 32 dims (lane = dim)
          if (rank == 0 && dim0 >= kDL) continue;  // the padded rows of the last block (whole warps)
          // 4 x 4 transposes among groups of four lanes: afterwards lane 4g + r holds dims
          // dim0 + 4g .. + 3 of keys 4kk + r (kk = 0..7), so each key's 4 dims go in one vector add
          float x[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(v[c]) * fac;
          const int r4 = lane & 3;
#pragma unroll
          for (int sh = 2; sh >= 1; sh >>= 1) {
            const bool up = (r4 & sh) != 0;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (e & sh) continue;
                const float send = up ? x[4 * kk + e] : x[4 * kk + (e ^ sh)];
                const float recv = __shfl_xor_sync(0xffffffffu, send, sh);
                if (up) x[4 * kk + e] = recv;
                else x[4 * kk + (e ^ sh)] = recv;
              }
            }
          }
          const int dim = dim0 + (lane & ~3);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const long long r = __shfl_sync(0xffffffffu, static_cast<long long>(my_row), 4 * kk + r4);
            if (r >= 0)
              atomicAdd(reinterpret_cast<float4*>(a.dkv + r * kDL + dim),
                        make_float4(x[4 * kk], x[4 * kk + 1], x[4 * kk + 2], x[4 * kk + 3]));
          }
        }
      }
      if (!ok) break;
      // ---- dq of the token (this CTA's dims), scaled, bf16
      if (!warp_wait(baddr(bars.dq_full), nq & 1, abort_flag, a)) break;
      ptx::tc_fence_after();
      for (int c = 0; c < dqn / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld32(tmem + col_dq + c * 32 + lane_base, v);
        ptx::tmem_wait_ld();
        if (h < a.H) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint4*>(dq_row + c * 32 + e * 8) =
                make_uint4(pack_bf16(__uint_as_float(v[8 * e]) * scale, __uint_as_float(v[8 * e + 1]) * scale),
                           pack_bf16(__uint_as_float(v[8 * e + 2]) * scale, __uint_as_float(v[8 * e + 3]) * scale),
                           pack_bf16(__uint_as_float(v[8 * e + 4]) * scale, __uint_as_float(v[8 * e + 5]) * scale),
                           pack_bf16(__uint_as_float(v[8 * e + 6]) * scale, __uint_as_float(v[8 * e + 7]) * scale));
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(baddr(bars.dq_free));
      g += n;
      ++nq;
    }
  } else {
    // ================================================================ loads of Q / dO, and credits
    int g = 0, nq = 0, last = -1;
    bool ok = true;
    for (int t = cl; ok && t < a.T; t += n_cl) {
      const int n = tiles_of(a, t);
      if (n == 0) continue;
      // this token's Q (rank 0) or dO (rank 1), once the previous token's products are done with it
      const uint32_t full = rank == 0 ? baddr(bars.q_full) : baddr(bars.do_full);
      const uint32_t free_b = rank == 0 ? baddr(bars.q_free) : baddr(bars.do_free);
      if (nq > 0 && !warp_wait(free_b, (nq - 1) & 1, abort_flag, a)) break;
      if (lane == 0) {
        const int nb = rank == 0 ? 9 : 8;
        ptx::mbar_arrive_expect_tx(full, nb * kBox);
#pragma unroll 1
        for (int b = 0; b < nb; ++b)
          ptx::tma_load_2d(sbase + (rank == 0 ? kOffQ : kOffDO) + b * kBox, rank == 0 ? &qmap : &domap, full, b * 64,
                           t * a.H);
      }
      __syncwarp();
      last = nq;
      // slot credits to the peer: rank 0's dS slot after its products; rank 1's P slots after theirs
      for (int i = 0; i < n; ++i) {
        const int gi = g + i;
        if (rank == 0) {
          if (!warp_wait(baddr(bars.ds_consumed), gi & 1, abort_flag, a)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(baddr(bars.ds_full), kSlot);  // armed for the next copy
            ptx::mbar_arrive_cluster(ptx::map_to_rank(baddr(bars.ds_peer_empty), peer));
          }
        } else {
          const int ps = gi & 1;
          if (!warp_wait(baddr(bars.p_consumed[ps]), (gi >> 1) & 1, abort_flag, a)) {
            ok = false;
            break;
          }
          if (lane == 0) ptx::mbar_arrive_cluster(ptx::map_to_rank(baddr(bars.p_empty[ps]), peer));
        }
        __syncwarp();
      }
      g += n;
      ++nq;
    }
    // after an abort the last Q / dO load may still be landing: let it finish
    if (*abort_flag && last >= 0) drain_wait(rank == 0 ? baddr(bars.q_full) : baddr(bars.do_full), last & 1, a.limit_ns);
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();  // no remote store or arrival into either CTA after this point
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_sparse_attn_bwd(const BwdArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  CUtensorMap qmap, domap;
  const uint64_t rows = static_cast<uint64_t>(a.T) * a.H;
  if (!encode_tmap_2d(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kDL, rows, kDL * 2, 64, 128) ||
      !encode_tmap_2d(&domap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.dout, kDV, rows, kDV * 2, 64, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int clusters = a.T < sms / 2 ? a.T : sms / 2;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_attn_bwd_kernel, a, qmap, domap);
}

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_sparse_attn_backward(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows,
                                                 const int32_t* idx, int T, int H, int k, float scale,
                                                 const uint16_t* out, const uint16_t* dout, const float* lse,
                                                 uint16_t* dq, float* dkv, int32_t* dev_status, dsa_stream_t stream) {
  dsa_status_t st = check_attn_args(q, kv, n_kv_rows, nullptr, 0, 0, idx, T, H, k, out);
  if (st != DSA_OK) return st;
  if (!dout || !lse || !dq || !dkv) return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dout) & 15u) || (reinterpret_cast<uintptr_t>(dq) & 15u) ||
      (reinterpret_cast<uintptr_t>(dkv) & 15u))
    return DSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * H > (1ll << 31) - 1) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  int* status = status_target(dev_status);
  if (!status) return DSA_ERR_CUDA;
  BwdArgs a{};
  a.q = q; a.kv = kv; a.n_kv_rows = n_kv_rows; a.idx = idx; a.T = T; a.H = H; a.k = k; a.scale = scale;
  a.out = out; a.dout = dout; a.lse = lse; a.dq = dq; a.dkv = dkv; a.status = status; a.limit_ns = wait_limit_ns();
  return launch_sparse_attn_bwd(a, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
