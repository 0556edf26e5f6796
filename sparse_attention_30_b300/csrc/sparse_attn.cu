// Sparse attention over the selected latent rows, MQA mode of MLA
// (freezhihu.org/question/1978819912970555965, §2.1.2 output equation and §2.2):
//     o[t,h,:] = sum_{s in S_t} softmax_s(scale * q[t,h,:] . c_s) * c_s[0:512]
// Every head of token t sees the same rows c_s, so per token this is a dense
// [H x 576] x [576 x |S_t|] product followed by [H x |S_t|] x [|S_t| x 512].
//
// A cluster of two CTAs with different jobs works through a list of work items (a token, or with
// a key split one share of a token's selected tiles), one after another, and data flows one way:
//
//   rank 0, "score" CTA: Q [128 x 576] bf16 sits in TMEM (A operand of the MMA read straight
//     from tensor memory); S = Q K^T is computed 64 keys at a time (N = 64) into two TMEM
//     buffers from K rows that twelve cp.async warps gather into a 2-stage ring; four warps
//     (one head row per thread) run the online softmax.  Each 64-key tile of P (bf16) plus
//     per-row rescale factors is pushed into rank 1's shared memory with an asynchronous bulk
//     copy, and an item's final row statistics follow its last tile.
//   rank 1, "value" CTA: O [128 x 512] fp32 fills its whole TMEM; twelve warps gather the value
//     part (first 512 latent dims) of the same rows into a 2-stage ring and O += P V runs as soon
//     as a P tile lands.  When rank 0 moved a row's running max (lazily: only when it grows by
//     more than 2^8), the factor travels with P and O is rescaled before that tile's PV.  Ring
//     slots are handed back to rank 0 by a credit warp, off the critical path.
//
// Items follow each other without a pause in either pipeline: rank 0 loads the next item's Q
// into its K ring as soon as the last S product of the previous item has completed (twelve
// warps move it into TMEM), while rank 1 still finishes that item's PV products and writes its
// output; rank 1's next PV product waits only until O has been read out.  A scheduler warp in
// each CTA finds every item's tile count (the first empty slot of its index row) ahead of time
// and hands items to the other warps through a small ring.  MMAs are issued warp-uniformly (one
// elected lane), and tiles are 64 keys wide, because narrow or single-thread-issued tcgen05.mma
// chains are issue-bound rather than tensor-bound.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

using namespace attn;

constexpr int kProdWarps = 12;                 // warps 1..12 gather
constexpr int kProducers = kProdWarps * 32;
constexpr int kRowWarp0 = 1 + kProdWarps;      // warps 13..16: one head row per thread (TMEM lane)
constexpr int kCreditWarp = kRowWarp0 + 4;     // warp 17 (rank 1): slot credits
constexpr int kSchedWarp = kCreditWarp + 1;    // warp 18: work items
constexpr int kThreads = 32 * (kSchedWarp + 1);
constexpr int kKT = 64;                        // keys per tile
constexpr int kDL = 576, kDV = 512;
constexpr int kKStages = 2, kVStages = 2, kSlots = 4, kSBufs = 2, kSched = 4;
constexpr int kBlockBytes = kKT * 128;         // 64 rows x 64 bf16
constexpr int kKStageBytes = 9 * kBlockBytes;  // 72 KB: all 576 dims
constexpr int kVStageBytes = 8 * kBlockBytes;  // 64 KB: value dims 0..511
// P slot: P [128 x 64] bf16 (128B-swizzled) | 128 fp32 factors | 4 int flags (one per row warp)
constexpr int kSlotP = 128 * kKT * 2;
constexpr int kSlotFac = kSlotP;
constexpr int kSlotFlag = kSlotFac + 128 * 4;
constexpr int kSlotBytes = kSlotFlag + 16;     // bytes moved per tile
constexpr int kSlotStride = 17408;
constexpr int kStatsBytes = 1024;              // l[128], m[128]
constexpr int kQBoxBytes = 128 * 128;          // Q box: 128 rows x 128 bytes, 128B-swizzled
constexpr int kQBytes = 9 * kQBoxBytes;        // Q [128 x 576] bf16
// rank 0 layout
constexpr int kOffK = 0;
constexpr int kOffStage = kOffK + kKStages * kKStageBytes;  // two P staging buffers
constexpr int kOffStatStage = kOffStage + 2 * kSlotStride;  // statistics staging
constexpr int kEnd0 = kOffStatStage + kStatsBytes;
// rank 1 layout
constexpr int kOffV = 0;
constexpr int kOffSlots = kOffV + kVStages * kVStageBytes;
constexpr int kOffStats = kOffSlots + kSlots * kSlotStride;  // two statistics buffers
constexpr int kEnd1 = kOffStats + 2 * kStatsBytes;
constexpr int kSmem = (kEnd0 > kEnd1 ? kEnd0 : kEnd1) + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 288;                // rank 0: Q in columns 0..287, S buffers after it
constexpr float kRescaleThreshold = 8.0f;      // log2 units
// warps that take work items from the scheduler: rank 0 MMA + producers + row warps, rank 1 also
// the credit warp
constexpr int kItemReaders0 = 1 + kProdWarps + 4, kItemReaders1 = kItemReaders0 + 1;
static_assert(kColS + kSBufs * kKT <= kTmemCols, "rank 0 TMEM budget");
static_assert(kQBytes <= kKStages * kKStageBytes, "Q is staged in rank 0's K ring");
static_assert(kSmem <= 227 * 1024, "shared memory budget");

// Physical latent row of position s for row t, or -1 if the slot is empty or out of range.
__device__ __forceinline__ int64_t latent_row(const AttnArgs& a, int t, int32_t s, bool* range_err) {
  if (s < 0) return -1;
  if (a.block_table == nullptr) {
    if (s >= a.n_kv_rows) { *range_err = true; return -1; }
    return s;
  }
  if (s / a.page_size >= a.bt_stride) { *range_err = true; return -1; }
  const int32_t page = a.block_table[static_cast<int64_t>(t) * a.bt_stride + s / a.page_size];
  const int64_t r = static_cast<int64_t>(page) * a.page_size + s % a.page_size;
  if (page < 0 || r >= a.n_kv_rows) { *range_err = true; return -1; }
  return r;
}

// A work item: tiles [tile0, tile0 + n_tiles) of token t's selection, written as partial result
// sp (t < 0: no more items); nt is the token of this cluster's next item (-1: none).
struct Item {
  int t, sp, tile0, n_tiles, nt;
};

struct Bars {
  // rank 0
  uint64_t k_full[kKStages], k_empty[kKStages], s_full[kSBufs], s_empty[kSBufs], q_full, q_ready, q_free;
  uint64_t p_empty[kSlots], stats_empty[2];
  // rank 1
  uint64_t v_full[kVStages], v_empty[kVStages], p_full[kSlots], ready[kSlots], slot_free[kSlots];
  uint64_t stats_full[2], o_full, o_free;
  // both
  uint64_t sched_full[kSched], sched_empty[kSched], mma_done;
};

__device__ __forceinline__ uint32_t baddr(const uint64_t& b) { return ptx::smem_addr(&b); }

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) break;
  }
}

// Warp-uniform bounded wait (all lanes agree on the outcome).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, const AttnArgs& a) {
  return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, a.status, a.limit_ns));
}

// Work item j of this warp's CTA, from the scheduler ring (the warp's lane 0 releases the slot).
__device__ __forceinline__ bool read_item(Bars& bars, const Item* sched, int j, Item* it, volatile int* abort_flag,
                                          const AttnArgs& a) {
  const int slot = j % kSched;
  if (!warp_wait(baddr(bars.sched_full[slot]), (j / kSched) & 1, abort_flag, a)) return false;
  const volatile Item* e = sched + slot;
  it->t = e->t;
  it->sp = e->sp;
  it->tile0 = e->tile0;
  it->n_tiles = e->n_tiles;
  it->nt = e->nt;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(baddr(bars.sched_empty[slot]));
  return true;
}

// Gather of tile i: `nblk` 64-dim blocks (from latent dim 0) of each of the 64 selected rows into
// a 128B-swizzled stage.  Producer warp pw copies whole rows pw, pw + 12, ...: the tile's positions
// are read once (two per lane) and row addresses are broadcast with shuffles.  An empty or
// out-of-range slot copies `fallback_row` instead (the token's first selected row, which is always
// attended) so every copy is a plain 16-byte copy; the softmax masks that key to P = 0, so the
// substitute never contributes.  The loop is kept minimal: the producers are issue-bound.
template <int NBLK>
__device__ __forceinline__ void gather_rows(const AttnArgs& a, int t, const int32_t* idx_row, int i, uint32_t dst,
                                            int pw, int lane, int64_t fallback_row, bool* range_err) {
  constexpr int kChunks = NBLK * 8;
  const uint16_t* base[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int slot = i * kKT + h * 32 + lane;
    const int32_t s = slot < a.k ? __ldg(idx_row + slot) : -1;
    const int64_t pr = latent_row(a, t, s, range_err);
    base[h] = a.kv + (pr < 0 ? fallback_row : pr) * kDL;
  }
  for (int r = pw; r < kKT; r += kProdWarps) {
    const uint16_t* src = reinterpret_cast<const uint16_t*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(r >> 5 ? base[1] : base[0]), r & 31));
    const uint32_t drow = dst + r * 128;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int cc = lane + 32 * j;
      if (cc < kChunks)
        ptx::cp_async16_n<16>(drow + (cc >> 3) * kBlockBytes + (((cc & 7) ^ (r & 7)) << 4), src + cc * 8);
    }
  }
}

// One item's tiles through a producer ring of `stages` stages; g = tiles of earlier items.
// Completion of a stage is tracked by the hardware (each producer thread's cp.async copies arrive
// on the stage's barrier when they land), so producers never wait for their own copies.  The
// consumer issues fence.proxy.async after the barrier before the tensor core reads the stage.
template <int NBLK>
__device__ __forceinline__ bool produce_item(const AttnArgs& a, const Item& it, int g, uint32_t ring, int stage_bytes,
                                             int stages, uint64_t* full, uint64_t* empty, volatile int* abort_flag,
                                             bool* range_err) {
  const int pw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int32_t* idx_row = a.idx + static_cast<int64_t>(it.t) * a.k;
  // the first slot is valid whenever there is a tile (valid slots come first)
  int64_t fallback_row = latent_row(a, it.t, __ldg(idx_row), range_err);
  if (fallback_row < 0) {  // first position out of range: nothing safe to substitute
    atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE);
    fallback_row = 0;
  }
  for (int i = 0; i < it.n_tiles; ++i) {
    const int gi = g + i, st = gi % stages;
    if (!warp_wait(baddr(empty[st]), ((gi / stages) & 1) ^ 1, abort_flag, a)) return false;
    gather_rows<NBLK>(a, it.t, idx_row, it.tile0 + i, ring + st * stage_bytes, pw, lane, fallback_row, range_err);
    ptx::cp_async_arrive_noinc(baddr(full[st]));
  }
  return true;
}

// Dense causal mode: tile i of an item covers the 64 consecutive latent rows from
// (tile0 + i) * 64, so lane 0 of one warp moves it with NBLK tensor-map box loads ([64 rows x 64
// dims] each, 128B-swizzled, the same layout the gathers write); rows past the tensor read as zero
// and the softmax masks every key after the token's own position.  *issued counts the tiles whose
// loads were started, for the drain after an abort.
template <int NBLK>
__device__ __forceinline__ bool produce_item_dense(const AttnArgs& a, const CUtensorMap* kvmap, const Item& it, int g,
                                                   uint32_t ring, int stage_bytes, int stages, uint64_t* full,
                                                   uint64_t* empty, volatile int* abort_flag, int* issued) {
  for (int i = 0; i < it.n_tiles; ++i) {
    const int gi = g + i, st = gi % stages;
    if (!warp_wait(baddr(empty[st]), ((gi / stages) & 1) ^ 1, abort_flag, a)) return false;
    if ((threadIdx.x & 31) == 0) {
      ptx::mbar_arrive_expect_tx(baddr(full[st]), NBLK * kBlockBytes);
#pragma unroll 1
      for (int b = 0; b < NBLK; ++b)
        ptx::tma_load_2d(ring + st * stage_bytes + b * kBlockBytes, kvmap, baddr(full[st]), b * 64,
                         (it.tile0 + i) * kKT);
    }
    __syncwarp();
    *issued = gi + 1;
  }
  return true;
}

// After an abort, the tensor-map loads of the last `stages` tiles may still be landing in the ring:
// wait (bounded) until they have, so that no copy writes into the CTA's shared memory after exit.
__device__ __forceinline__ void drain_dense(uint64_t* full, int stages, int issued, uint64_t limit_ns) {
  for (int gi = issued > stages ? issued - stages : 0; gi < issued; ++gi)
    drain_wait(baddr(full[gi % stages]), (gi / stages) & 1, limit_ns);
}


// Indexer-loss mode: the four row warps of a score CTA (one head row per thread).  For every key s
// of token t's set, u_s = sum over heads of that head's attention probability
// 2^(S[h,s] * scale * log2(e) - lse[h] * log2(e)), with the forward's own normalisers lse.  Each warp
// sums its 32 heads with a butterfly that leaves keys 2*lane and 2*lane+1 on each lane, the four
// warps meet in shared memory, and threads h < 64 then own key h of every tile: they decide whether
// the key is in the set and accumulate, per token, U = sum u, A = sum u ln u, B = sum u I and the
// log-sum-exp Z of I over the set.  At the token's end, with p = u / U and q = softmax(I):
//     KL(p || q) = (A - B) / U - ln U + Z.
// A key owner's position (from the selection) and indexer score arrive by asynchronous copies into
// shared memory, the position two tiles and the score one tile ahead of use.
template <bool kDense>
__device__ __forceinline__ void loss_row_warps(const AttnArgs& a, Bars& bars, const Item* sched, uint8_t* smem,
                                               uint32_t tmem, volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = (warp & 3) * 32 + lane;
  const bool owner = h < kKT;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  float* red = reinterpret_cast<float*>(smem + kOffStage);             // [2 tiles][4 warps][64 keys]
  double* fin = reinterpret_cast<double*>(smem + kOffStage + 2048);    // [2 warps][5] partials, then 1/U
  double* acc = reinterpret_cast<double*>(smem + kOffStage + 4096) + h * 4;       // owner's U, A, B, sum e^(I-max)
  float* acc_max = reinterpret_cast<float*>(smem + kOffStage + 6144) + h;        // owner's running max of I
  int32_t* posb = reinterpret_cast<int32_t*>(smem + kOffStage + 6400);           // [2][64] selected positions
  float* scb = reinterpret_cast<float*>(smem + kOffStage + 6912);                // [2][64] their scores
  const uint32_t posb_s = ptx::smem_addr(posb + h), scb_s = ptx::smem_addr(scb + h);
  int g = 0;
  bool ok = true, range_err = false;
  for (int j = 0; ok; ++j) {
    Item it;
    if (!read_item(bars, sched, j, &it, abort_flag, a) || it.t < 0) break;
    const int t = it.t;
    const int32_t* idx_row = kDense ? nullptr : a.idx + static_cast<int64_t>(t) * a.k;
    const float* score_row = a.scores + static_cast<int64_t>(t) * a.ld;
    const float lse2 = h < a.H ? a.lse_in[static_cast<int64_t>(t) * a.H + h] * 1.4426950408889634f : 0.f;
    // key h of tile i: its slot, and (once its selection entry has landed) its position or -1
    auto slot_of = [&](int i) { return (it.tile0 + i) * kKT + h; };
    auto issue_idx = [&](int i) {  // selection entry of tile i -> posb[i & 1]
      if (!kDense && i < it.n_tiles && slot_of(i) < a.k) ptx::cp_async4(posb_s + (i & 1) * kKT * 4, idx_row + slot_of(i));
    };
    auto position = [&](int i) -> int {
      if (i >= it.n_tiles) return -1;
      const int slot = slot_of(i);
      if constexpr (kDense) {
        return slot <= a.q_pos0 + t ? slot : -1;
      } else {
        const int32_t sidx = slot < a.k ? posb[(i & 1) * kKT + h] : -1;
        return latent_row(a, t, sidx, &range_err) >= 0 ? sidx : -1;
      }
    };
    auto issue_score = [&](int i, int pos) {  // score of tile i's key -> scb[i & 1]
      if (pos >= 0 && pos < a.ld) ptx::cp_async4(scb_s + (i & 1) * kKT * 4, score_row + pos);
    };
    int pos = -1;
    if (owner) {
      acc[0] = acc[1] = acc[2] = acc[3] = 0.0;
      *acc_max = -INFINITY;
      issue_idx(0);
      issue_idx(1);
      ptx::cp_async_commit();
      ptx::cp_async_wait<0>();
      pos = position(0);
      issue_score(0, pos);
      ptx::cp_async_commit();
    }
    for (int i = 0; i < it.n_tiles; ++i) {
      const int gi = g + i, sb = gi % kSBufs;
      const bool got = warp_wait(baddr(bars.s_full[sb]), (gi / kSBufs) & 1, abort_flag, a);
      uint32_t s0[32], s1[32];
      if (got) {
        ptx::tc_fence_after();
        ptx::tmem_ld32(tmem + kColS + sb * kKT + lane_base, s0);
        ptx::tmem_ld32(tmem + kColS + sb * kKT + 32 + lane_base, s1);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(baddr(bars.s_empty[sb]));
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) s0[e] = s1[e] = 0;
      }
      // every key of the tile (keys outside the set are dropped by their owners below)
      float v[kKT];
#pragma unroll
      for (int e = 0; e < kKT; ++e) {
        const uint32_t raw = e < 32 ? s0[e] : s1[e - 32];
        v[e] = h < a.H ? fast_exp2(__uint_as_float(raw) * a.scale_log2 - lse2) : 0.f;
      }
      // sum over the warp's 32 heads; after the stage exchanging across lane bit sh, each lane keeps
      // the half of its remaining keys selected by that bit
#pragma unroll
      for (int n = kKT; n > 2; n >>= 1) {
        const int sh = n >> 2;  // n = 64, 32, 16, 8, 4 -> lane bit 16, 8, 4, 2, 1
        const bool up = (lane & sh) != 0;
#pragma unroll
        for (int e = 0; e < n / 2; ++e) {
          const float send = up ? v[e] : v[e + n / 2];
          const float recv = __shfl_xor_sync(0xffffffffu, send, sh);
          v[e] = (up ? v[e + n / 2] : v[e]) + recv;
        }
      }
      float* rb = red + (gi & 1) * (4 * kKT);
      *reinterpret_cast<float2*>(rb + (warp & 3) * kKT + 2 * lane) = make_float2(v[0], v[1]);
      if (ptx::named_sync_or(1, 128, !got || *abort_flag)) {
        ok = false;
        break;
      }
      if (owner) {
        ptx::cp_async_wait<0>();  // this tile's score and the next tile's selection entry
        const int slot = slot_of(i);
        if (pos >= 0 && pos < a.ld) {
          const float u = rb[h] + rb[kKT + h] + rb[2 * kKT + h] + rb[3 * kKT + h];
          const float I = scb[(i & 1) * kKT + h];
          acc[0] += u;
          if (u > 0.f) acc[1] += static_cast<double>(u) * logf(u);
          acc[2] += static_cast<double>(u) * I;
          const float zmax = *acc_max;
          if (I > zmax) {
            acc[3] = acc[3] * (zmax == -INFINITY ? 0.0 : static_cast<double>(expf(zmax - I))) + 1.0;
            *acc_max = I;
          } else {
            acc[3] += expf(I - zmax);
          }
          if (!kDense && a.p_out) a.p_out[static_cast<int64_t>(t) * a.k + slot] = u;
        } else {
          if (pos >= a.ld) range_err = true;
          if (!kDense && a.p_out && slot < a.k) a.p_out[static_cast<int64_t>(t) * a.k + slot] = 0.f;
        }
        pos = position(i + 1);
        issue_score(i + 1, pos);
        issue_idx(i + 2);
        ptx::cp_async_commit();
      }
    }
    if (owner) ptx::cp_async_wait<0>();  // nothing in flight into the buffers the next token reuses
    // ---- the token's totals: owners h < 64 are warps (h / 32) = 0 and 1 of the four
    if (owner) {
      double U = acc[0], A = acc[1], B = acc[2], zsum = acc[3];
      float zmax = *acc_max;
#pragma unroll
      for (int sh = 16; sh >= 1; sh >>= 1) {
        U += __shfl_xor_sync(0xffffffffu, U, sh);
        A += __shfl_xor_sync(0xffffffffu, A, sh);
        B += __shfl_xor_sync(0xffffffffu, B, sh);
        const float om = __shfl_xor_sync(0xffffffffu, zmax, sh);
        const double os = __shfl_xor_sync(0xffffffffu, zsum, sh);
        const float m = fmaxf(zmax, om);
        zsum = (zmax == -INFINITY ? 0.0 : zsum * expf(zmax - m)) + (om == -INFINITY ? 0.0 : os * expf(om - m));
        zmax = m;
      }
      if (lane == 0) {
        double* f = fin + (h >> 5) * 5;
        f[0] = U; f[1] = A; f[2] = B; f[3] = zmax; f[4] = zsum;
      }
    }
    ptx::named_sync(2, 128);
    if (h == 0) {
      double Ut = 0.0, At = 0.0, Bt = 0.0, zs = 0.0;
      float zm = -INFINITY;
      for (int w = 0; w < 2; ++w) {
        const double* f = fin + w * 5;
        Ut += f[0]; At += f[1]; Bt += f[2];
        const float m = fmaxf(zm, static_cast<float>(f[3]));
        zs = (zm == -INFINITY ? 0.0 : zs * exp(static_cast<double>(zm - m))) +
             (f[3] == -INFINITY ? 0.0 : f[4] * exp(f[3] - m));
        zm = m;
      }
      const bool has = ok && it.n_tiles > 0 && Ut > 0.0;
      const double kl = has ? (At - Bt) / Ut - log(Ut) + (zm + log(zs)) : 0.0;
      if (ok) {
        if (a.kl_out) a.kl_out[t] = static_cast<float>(kl);
        if (a.loss_acc) atomicAdd(a.loss_acc, kl);
      }
      fin[10] = has ? 1.0 / Ut : 0.0;
    }
    ptx::named_sync(2, 128);
    if (ok && !kDense && a.p_out && owner) {
      // normalise the row's target (the entries this thread wrote) and clear the slots past its tiles
      const float inv = static_cast<float>(fin[10]);
      float* prow = a.p_out + static_cast<int64_t>(t) * a.k;
      for (int slot = it.tile0 * kKT + h; slot < (it.tile0 + it.n_tiles) * kKT && slot < a.k; slot += kKT)
        prow[slot] *= inv;
      for (int slot = (it.tile0 + it.n_tiles) * kKT + h; slot < a.k; slot += kKT) prow[slot] = 0.f;
    }
    ptx::named_sync(2, 128);  // fin is reused by the next token
    g += it.n_tiles;
  }
  if (range_err) atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE);
}

// kMode bit 0: dense causal (no selection; row t attends latent rows 0 .. q_pos0 + t).
// kMode bit 1: indexer loss (no value pass; every CTA is an independent score CTA, launched without
// clusters).  Attention modes run as clusters of two.
// kMode bit 2: the balanced partition of AttnArgs::bal_tiles (a kernel instance of its own, so that
// the other modes carry none of its scheduling code).
template <int kMode>
__device__ __forceinline__ void attn_body(const AttnArgs& a, const CUtensorMap* qmap, const CUtensorMap* kvmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ Bars bars;
  __shared__ Item sched[kSched];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag_s;

  constexpr bool kDense = (kMode & 1) != 0, kLoss = (kMode & 2) != 0, kBal = (kMode & 4) != 0;
  const int rank = kLoss ? 0 : static_cast<int>(ptx::cluster_ctarank());
  const int cl = kLoss ? blockIdx.x : blockIdx.x >> 1, n_cl = kLoss ? gridDim.x : gridDim.x >> 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &abort_flag_s;
  const uint32_t sbase = ptx::smem_addr(smem);
  constexpr bool dense = kDense;
  const uint32_t fill = dense ? 1u : static_cast<uint32_t>(kProducers);  // arrivals per ring stage

  if (tid == 0) {
    if (rank == 0) {
      for (int s = 0; s < kKStages; ++s) {
        ptx::mbar_init(baddr(bars.k_full[s]), fill);
        ptx::mbar_init(baddr(bars.k_empty[s]), 1);
      }
      for (int b = 0; b < kSBufs; ++b) {
        ptx::mbar_init(baddr(bars.s_full[b]), 1);
        ptx::mbar_init(baddr(bars.s_empty[b]), 128);
      }
      ptx::mbar_init(baddr(bars.q_full), 1);
      ptx::mbar_init(baddr(bars.q_ready), kProducers);
      ptx::mbar_init(baddr(bars.q_free), 1);
      for (int s = 0; s < kSlots; ++s) ptx::mbar_init(baddr(bars.p_empty[s]), 1);
      for (int b = 0; b < 2; ++b) ptx::mbar_init(baddr(bars.stats_empty[b]), 1);
    } else {
      for (int s = 0; s < kVStages; ++s) {
        ptx::mbar_init(baddr(bars.v_full[s]), fill);
        ptx::mbar_init(baddr(bars.v_empty[s]), 1);
      }
      for (int s = 0; s < kSlots; ++s) {
        ptx::mbar_init(baddr(bars.p_full[s]), 1);
        ptx::mbar_init(baddr(bars.ready[s]), 128);
        ptx::mbar_init(baddr(bars.slot_free[s]), 1);
      }
      for (int b = 0; b < 2; ++b) ptx::mbar_init(baddr(bars.stats_full[b]), 1);
      ptx::mbar_init(baddr(bars.o_full), 1);
      ptx::mbar_init(baddr(bars.o_free), 128);
      // arm the first use of every P slot and statistics buffer for rank 0's bulk copies
      for (int s = 0; s < kSlots; ++s) ptx::mbar_arrive_expect_tx(baddr(bars.p_full[s]), kSlotBytes);
      for (int b = 0; b < 2; ++b) ptx::mbar_arrive_expect_tx(baddr(bars.stats_full[b]), kStatsBytes);
    }
    for (int s = 0; s < kSched; ++s) {
      ptx::mbar_init(baddr(bars.sched_full[s]), 1);
      ptx::mbar_init(baddr(bars.sched_empty[s]), rank == 0 ? kItemReaders0 : kItemReaders1);
    }
    ptx::mbar_init(baddr(bars.mma_done), 1);
    abort_flag_s = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_addr(&tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();  // both CTAs' barriers exist (and are armed) before any remote traffic
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kSchedWarp) {
    // ================================================================ scheduler (both CTAs)
    const int n_items = a.T * a.n_split;  // (the loss modes run without a key split)
    for (int j = 0;; ++j) {
      const int slot = j % kSched;
      // the ring runs items ahead: this wait is never urgent, so it sleeps between polls
      if (!__all_sync(0xffffffffu, ptx::mbar_wait_sleep(baddr(bars.sched_empty[slot]), ((j / kSched) & 1) ^ 1,
                                                        abort_flag, a.status, a.limit_ns, 1000)))
        break;
      Item it{-1, 0, 0, 0, -1};
      if constexpr (kBal) {
        // balanced: this cluster's contiguous range of the rows' virtual tiles, row by row
        const int tpr = a.bal_tiles;
        const int64_t G = static_cast<int64_t>(a.T) * tpr;
        const int64_t lo = bal_bound(cl, G, n_cl), hi = bal_bound(cl + 1, G, n_cl);
        const int t = static_cast<int>(lo / tpr) + j;
        const int64_t g0 = static_cast<int64_t>(t) * tpr;
        if (lo < hi && g0 < hi) {
          it.t = t;
          it.sp = cl - bal_cluster(g0, G, n_cl);
          const int v0 = static_cast<int>((lo > g0 ? lo : g0) - g0);
          const int v1 = static_cast<int>((hi < g0 + tpr ? hi : g0 + tpr) - g0);
          const int real = (first_empty_slot(a.idx + static_cast<int64_t>(t) * a.k, a.k) + kKT - 1) / kKT;
          it.tile0 = v0;
          it.n_tiles = max(0, min(v1, real) - v0);
          it.nt = g0 + tpr < hi ? t + 1 : -1;
        }
      } else {
        const int id = cl + j * n_cl;
        if (id < n_items) {
          it.t = id / a.n_split;
          it.sp = id % a.n_split;
          const int64_t n_keys = dense ? a.q_pos0 + it.t + 1 : first_empty_slot(a.idx + static_cast<int64_t>(it.t) * a.k, a.k);
          const int all_tiles = static_cast<int>((n_keys + kKT - 1) / kKT);
          const int per = (all_tiles + a.n_split - 1) / a.n_split;
          it.tile0 = it.sp * per;
          it.n_tiles = max(0, min(per, all_tiles - it.sp * per));
          const int next_id = id + n_cl;
          it.nt = next_id < n_items ? next_id / a.n_split : -1;
        }
      }
      if (lane == 0) {
        volatile Item* e = sched + slot;
        e->t = it.t;
        e->sp = it.sp;
        e->tile0 = it.tile0;
        e->n_tiles = it.n_tiles;
        e->nt = it.nt;
        ptx::mbar_arrive(baddr(bars.sched_full[slot]));
      }
      if (it.t < 0) break;
    }
  } else if (rank == 0) {
    // ================================================================ score CTA
    if (warp == 0) {
      // ---- per item: Q -> ring (TMA), then S = Q K^T tile after tile, issued by the whole warp
      constexpr uint32_t kIdescS = ptx::instr_desc(128, kKT, 1, 1, 0, 0);
      int g = 0, nq = 0;
      bool ok = true;
      int q_last = -1;  // phase of the last Q load issued
      for (int j = 0; ok; ++j) {
        Item it;
        if (!read_item(bars, sched, j, &it, abort_flag, a) || it.t < 0) break;
        if (it.n_tiles == 0) continue;
        // the ring and Q's TMEM columns are free once the previous item's products completed
        if (nq > 0 && !warp_wait(baddr(bars.q_free), (nq - 1) & 1, abort_flag, a)) break;
        if (lane == 0) {
          // Q [128 x 576] of the token as nine 128B-swizzled [128 x 64] boxes (rows past the tensor
          // read as zero; rows of the next token, when H < 128, are never used)
          ptx::mbar_arrive_expect_tx(baddr(bars.q_full), kQBytes);
#pragma unroll 1
          for (int b = 0; b < 9; ++b)
            ptx::tma_load_2d_hint(sbase + kOffK + b * kQBoxBytes, qmap, baddr(bars.q_full), b * 64, it.t * a.H,
                                  ptx::l2_evict_first_policy());  // Q and O stream: keep L2 for latent rows
          // the next item's Q into L2, so that its load after this item's last product is an L2 hit
          if (it.nt >= 0 && it.nt != it.t) {
#pragma unroll 1
            for (int b = 0; b < 9; ++b) ptx::tma_prefetch_2d(qmap, b * 64, it.nt * a.H);
          }
        }
        __syncwarp();
        q_last = nq;
        if (!warp_wait(baddr(bars.q_ready), nq & 1, abort_flag, a)) break;
        ptx::tc_fence_after();
        for (int i = 0; i < it.n_tiles; ++i) {
          const int gi = g + i, st = gi % kKStages, sb = gi % kSBufs;
          if (!warp_wait(baddr(bars.k_full[st]), (gi / kKStages) & 1, abort_flag, a) ||
              !warp_wait(baddr(bars.s_empty[sb]), ((gi / kSBufs) & 1) ^ 1, abort_flag, a)) {
            ok = false;
            break;
          }
          ptx::fence_proxy_async_smem();  // gathered rows (generic-proxy writes) -> tensor-core reads
          ptx::tc_fence_after();
          const uint64_t db0 = ptx::smem_desc(sbase + kOffK + st * kKStageBytes, 16, 1024, ptx::kLayoutSw128);
          const uint32_t d = tmem + kColS + sb * kKT;
#pragma unroll
          for (int f = 0; f < 36; ++f)  // K = 576 = 36 x 16; A step = 8 TMEM columns, B step = 32 bytes
            ptx::mma_bf16_ts_warp(d, tmem + f * 8, db0 + (f >> 2) * (kBlockBytes >> 4) + 2 * (f & 3), kIdescS,
                                  f > 0 ? 1u : 0u);
          ptx::mma_commit_warp(baddr(bars.k_empty[st]));
          ptx::mma_commit_warp(baddr(bars.s_full[sb]));
        }
        ptx::mma_commit_warp(baddr(bars.q_free));
        g += it.n_tiles;
        ++nq;
      }
      // after an abort, the last Q load may still be landing in the ring: let it finish
      if (*abort_flag && q_last >= 0) drain_wait(baddr(bars.q_full), q_last & 1, a.limit_ns);
      ptx::mma_commit_warp(baddr(bars.mma_done));
      drain_wait(baddr(bars.mma_done), 0, a.limit_ns);
    } else if (warp <= kProdWarps) {
      // ---- per item: move Q from the ring into TMEM (three warps per lane quarter, three boxes
      // each), then gather the item's K tiles
      const int quarter = warp & 3, bsel = (warp - 1) >> 2;
      const int h = quarter * 32 + lane;
      const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
      int g = 0, nq = 0, issued = 0;
      bool range_err = false;
      for (int j = 0;; ++j) {
        Item it;
        if (!read_item(bars, sched, j, &it, abort_flag, a) || it.t < 0) break;
        if (it.n_tiles == 0) continue;
        const bool got = warp_wait(baddr(bars.q_full), nq & 1, abort_flag, a);
        // row h of box b sits at b * 16 KB + h * 128 B with its 16-byte chunks XOR-swizzled by h & 7
        const uint8_t* qs = smem + kOffK + h * 128;
#pragma unroll 1
        for (int b = bsel; b < 9; b += 3) {
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 x = (got && h < a.H) ? *reinterpret_cast<const uint4*>(qs + b * kQBoxBytes + ((c ^ (h & 7)) << 4))
                                             : make_uint4(0, 0, 0, 0);
            v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
          }
          ptx::tmem_st32(tmem + lane_base + b * 32, v);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(baddr(bars.q_ready));
        // every producer has read Q out of the ring before any of them overwrites it
        if (!got || !warp_wait(baddr(bars.q_ready), nq & 1, abort_flag, a)) break;
        if constexpr (dense) {
          if (warp == 1 && !produce_item_dense<9>(a, kvmap, it, g, sbase + kOffK, kKStageBytes, kKStages, bars.k_full,
                                                  bars.k_empty, abort_flag, &issued))
            break;
        } else if (!produce_item<9>(a, it, g, sbase + kOffK, kKStageBytes, kKStages, bars.k_full, bars.k_empty,
                                    abort_flag, &range_err)) {
          break;
        }
        g += it.n_tiles;
        ++nq;
      }
      if (dense && warp == 1 && *abort_flag) drain_dense(bars.k_full, kKStages, issued, a.limit_ns);
      ptx::cp_async_wait<0>();  // nothing of this thread's may still be in flight when the CTA exits
      if (range_err) atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE);
    } else if (warp < kCreditWarp && kLoss) {
      loss_row_warps<kDense>(a, bars, sched, smem, tmem, abort_flag);
    } else if (warp < kCreditWarp) {
      // ---- online softmax, one head row per thread
      const int h = (warp & 3) * 32 + lane;
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t peer_slots = ptx::map_to_rank(sbase + kOffSlots, 1);
      uint8_t* stage = smem + kOffStage;
      int g = 0, nq = 0;
      bool ok = true, range_err = false;
      for (int j = 0; ok; ++j) {
        Item it;
        if (!read_item(bars, sched, j, &it, abort_flag, a) || it.t < 0) break;
        const int t = it.t;
        const int32_t* idx_row = dense ? nullptr : a.idx + static_cast<int64_t>(t) * a.k;
        float m_used = -INFINITY, l = 0.f;
        for (int i = 0; i < it.n_tiles; ++i) {
          const int gi = g + i, sb = gi % kSBufs;
          // exits are taken by all 128 threads together (named barriers below are unbounded):
          // a failed wait is voted on at the next barrier instead of breaking out alone
          const bool got = warp_wait(baddr(bars.s_full[sb]), (gi / kSBufs) & 1, abort_flag, a);
          uint32_t s0[32], s1[32];
          if (got) {
            ptx::tc_fence_after();
            ptx::tmem_ld32(tmem + kColS + sb * kKT + lane_base, s0);
            ptx::tmem_ld32(tmem + kColS + sb * kKT + 32 + lane_base, s1);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(baddr(bars.s_empty[sb]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) s0[e] = s1[e] = 0;
          }
          // which of the 64 keys are real (empty / out-of-range slots are masked)
          uint32_t vm[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int slot = (it.tile0 + i) * kKT + hh * 32 + lane;
            if constexpr (dense) {
              vm[hh] = __ballot_sync(0xffffffffu, slot <= a.q_pos0 + t);
            } else {
              const int32_t sidx = slot < a.k ? __ldg(idx_row + slot) : -1;
              vm[hh] = __ballot_sync(0xffffffffu, latent_row(a, t, sidx, &range_err) >= 0);
            }
          }
          float x[kKT];
          float mt = -INFINITY;
#pragma unroll
          for (int e = 0; e < kKT; ++e) {
            const uint32_t raw = e < 32 ? s0[e] : s1[e - 32];
            x[e] = ((vm[e >> 5] >> (e & 31)) & 1u) ? __uint_as_float(raw) * a.scale_log2 : -INFINITY;
            mt = fmaxf(mt, x[e]);
          }
          const float m_new = fmaxf(m_used, mt);
          const bool need = (i == 0) || (m_new > m_used + kRescaleThreshold);
          const bool moved = __any_sync(0xffffffffu, need);
          float fac = 1.f;
          if (moved) {
            fac = (i == 0) ? 0.f : fast_exp2(m_used - m_new);
            l *= fac;
            m_used = m_new;
          }
          float psum = 0.f;
          uint32_t packed[kKT / 2];
#pragma unroll
          for (int e = 0; e < kKT; e += 2) {
            const float p0 = fast_exp2(x[e] - m_used), p1 = fast_exp2(x[e + 1] - m_used);
            psum += p0 + p1;
            packed[e / 2] = pack_bf16(p0, p1);
          }
          l += psum;
          // staging buffer gi % 2 is free once the bulk copy of tile gi - 2 has read it
          const int sbuf = gi & 1;
          if (h == 0) ptx::bulk_wait_read<1>();
          if (ptx::named_sync_or(1, 128, !got || *abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sp = stage + sbuf * kSlotStride;
          // P row h: 128 bytes = 8 chunks of 16 B, 128B swizzle (chunk c lands at c ^ (h & 7))
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sp + h * 128 + ((c ^ (h & 7)) << 4)) =
                make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
          reinterpret_cast<float*>(sp + kSlotFac)[h] = (moved && i > 0) ? fac : 1.f;
          if (lane == 0) reinterpret_cast<int*>(sp + kSlotFlag)[warp & 3] = (moved && i > 0) ? 1 : 0;
          ptx::fence_proxy_async_smem();
          ptx::named_sync(2, 128);
          // a failed wait here raises the abort flag, which the next vote picks up (`ok` stays
          // uniform over the 128 threads)
          if (h == 0) {
            const int ps = gi % kSlots;
            if (ptx::mbar_wait(baddr(bars.p_empty[ps]), ((gi / kSlots) & 1) ^ 1, abort_flag, a.status, a.limit_ns)) {
              ptx::bulk_copy_to_cluster(peer_slots + ps * kSlotStride, ptx::smem_addr(sp), kSlotBytes,
                                        ptx::map_to_rank(baddr(bars.p_full[ps]), 1));
              ptx::bulk_commit();
            }
          }
        }
        if (it.n_tiles > 0) {
          // the item's row statistics for rank 1's normalisation, into its buffer nq % 2
          float* st = reinterpret_cast<float*>(smem + kOffStatStage);
          if (h == 0) ptx::bulk_wait_read<0>();  // the previous statistics copy has read the staging
          if (ptx::named_sync_or(1, 128, !ok || *abort_flag)) ok = false;
          if (ok) {
            st[h] = l;
            st[128 + h] = m_used;
            ptx::fence_proxy_async_smem();
            ptx::named_sync(2, 128);
            if (h == 0) {
              const int b = nq & 1;
              if (ptx::mbar_wait(baddr(bars.stats_empty[b]), ((nq >> 1) & 1) ^ 1, abort_flag, a.status,
                                 a.limit_ns)) {
                ptx::bulk_copy_to_cluster(ptx::map_to_rank(sbase + kOffStats + b * kStatsBytes, 1),
                                          ptx::smem_addr(st), kStatsBytes,
                                          ptx::map_to_rank(baddr(bars.stats_full[b]), 1));
                ptx::bulk_commit();
              }
            }
          }
        }
        const bool has = ok && it.n_tiles > 0;
        if (a.n_split > 1) {
          if (h < a.H) {
            float* ml = a.part_ml + ((static_cast<int64_t>(t) * a.n_split + it.sp) * a.H + h) * 2;
            ml[0] = has ? m_used : -INFINITY;
            ml[1] = has ? l : 0.f;
          }
        } else if (a.lse != nullptr && h < a.H) {
          a.lse[static_cast<int64_t>(t) * a.H + h] = has ? (m_used + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
        }
        g += it.n_tiles;
        if (it.n_tiles > 0) ++nq;
      }
      if (h == 0) ptx::bulk_wait_read<0>();  // no copy may still read this CTA's staging at exit
      if (range_err) atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE);
    }
  } else {
    // ================================================================ value CTA
    if (warp == 0) {
      // ---- per item: O = sum of P V over its tiles (two N = 256 halves), issued by the whole warp
      constexpr uint32_t kIdescPV = ptx::instr_desc(128, 256, 1, 1, 0, 1);
      int g = 0, nq = 0;
      bool ok = true;
      for (int j = 0; ok; ++j) {
        Item it;
        if (!read_item(bars, sched, j, &it, abort_flag, a) || it.t < 0) break;
        if (it.n_tiles == 0) continue;
        // the previous item's O has been read out before this item's first product overwrites it
        if (nq > 0 && !warp_wait(baddr(bars.o_free), (nq - 1) & 1, abort_flag, a)) break;
        for (int i = 0; i < it.n_tiles; ++i) {
          const int gi = g + i, vs = gi % kVStages, ps = gi % kSlots;
          if (!warp_wait(baddr(bars.v_full[vs]), (gi / kVStages) & 1, abort_flag, a) ||
              !warp_wait(baddr(bars.ready[ps]), (gi / kSlots) & 1, abort_flag, a)) {
            ok = false;
            break;
          }
          ptx::fence_proxy_async_smem();  // gathered rows (generic-proxy writes) -> tensor-core reads
          ptx::tc_fence_after();
          const uint32_t vst = sbase + kOffV + vs * kVStageBytes;
          const uint64_t da = ptx::smem_desc(sbase + kOffSlots + ps * kSlotStride, 16, 1024, ptx::kLayoutSw128);
#pragma unroll
          for (int ks = 0; ks < kKT / 16; ++ks) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              // V rows ks*16 .. ks*16+15 of blocks 4*half .. 4*half+3, read MN-major
              const uint64_t db =
                  ptx::smem_desc(vst + half * 4 * kBlockBytes + ks * 16 * 128, kBlockBytes, 1024, ptx::kLayoutSw128);
              ptx::mma_bf16_warp(tmem + half * 256, da + 2 * ks, db, kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit_warp(baddr(bars.v_empty[vs]));
          ptx::mma_commit_warp(baddr(bars.slot_free[ps]));
        }
        ptx::mma_commit_warp(baddr(bars.o_full));
        g += it.n_tiles;
        ++nq;
      }
      ptx::mma_commit_warp(baddr(bars.mma_done));
      drain_wait(baddr(bars.mma_done), 0, a.limit_ns);
    } else if (warp <= kProdWarps) {
      int g = 0, issued = 0;
      bool range_err = false;
      for (int j = 0;; ++j) {
        Item it;
        if (!read_item(bars, sched, j, &it, abort_flag, a) || it.t < 0) break;
        if (it.n_tiles == 0) continue;
        if constexpr (dense) {
          if (warp == 1 && !produce_item_dense<8>(a, kvmap, it, g, sbase + kOffV, kVStageBytes, kVStages, bars.v_full,
                                                  bars.v_empty, abort_flag, &issued))
            break;
        } else if (!produce_item<8>(a, it, g, sbase + kOffV, kVStageBytes, kVStages, bars.v_full, bars.v_empty,
                                    abort_flag, &range_err)) {
          break;
        }
        g += it.n_tiles;
      }
      if (dense && warp == 1 && *abort_flag) drain_dense(bars.v_full, kVStages, issued, a.limit_ns);
      ptx::cp_async_wait<0>();
      if (range_err) atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE);
    } else if (warp < kCreditWarp) {
      // ---- per item: rescale O when rank 0 moved a row's max, then the epilogue: O / l in bf16
      // (or, with a key split, the fp32 partial), one row per thread, straight from TMEM
      const int h = (warp & 3) * 32 + lane;
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint64_t policy = ptx::l2_evict_first_policy();  // written once, read by the next stage
      int g = 0, nq = 0;
      bool ok = true;
      for (int j = 0; ok; ++j) {
        Item it;
        if (!read_item(bars, sched, j, &it, abort_flag, a) || it.t < 0) break;
        for (int i = 0; ok && i < it.n_tiles; ++i) {
          const int gi = g + i, ps = gi % kSlots;
          if (!warp_wait(baddr(bars.p_full[ps]), (gi / kSlots) & 1, abort_flag, a)) {
            ok = false;
            break;
          }
          const uint8_t* sp = smem + kOffSlots + ps * kSlotStride;
          if (reinterpret_cast<const volatile int*>(sp + kSlotFlag)[warp & 3]) {
            // rank 0 moved this warp's running max: O must include PV(gi - 1) before it is rescaled
            const int pj = gi - 1;
            if (!warp_wait(baddr(bars.slot_free[pj % kSlots]), (pj / kSlots) & 1, abort_flag, a)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const float f = reinterpret_cast<const float*>(sp + kSlotFac)[h];
#pragma unroll 1
            for (int c = 0; c < 16; ++c) {
              uint32_t o[32];
              ptx::tmem_ld32(tmem + lane_base + c * 32, o);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
              ptx::tmem_st32(tmem + lane_base + c * 32, o);
            }
            ptx::tmem_wait_st();
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(baddr(bars.ready[ps]));
        }
        // ---- epilogue of the item (the four warps decide together: named barriers are unbounded)
        float inv_l = 0.f;
        if (ok && it.n_tiles > 0) {
          const int b = nq & 1;
          ok = warp_wait(baddr(bars.o_full), nq & 1, abort_flag, a) &&
               warp_wait(baddr(bars.stats_full[b]), (nq >> 1) & 1, abort_flag, a);
          const float l = ok ? reinterpret_cast<const float*>(smem + kOffStats + b * kStatsBytes)[h] : 0.f;
          inv_l = l > 0.f ? 1.f / l : 0.f;
        }
        if (ptx::named_sync_or(1, 128, !ok)) ok = false;
        if (ok && it.n_tiles > 0 && h == 0) {
          // the statistics buffer is free again: arm its next use and tell rank 0
          const int b = nq & 1;
          ptx::mbar_arrive_expect_tx(baddr(bars.stats_full[b]), kStatsBytes);
          ptx::mbar_arrive_cluster(ptx::map_to_rank(baddr(bars.stats_empty[b]), 0));
        }
        ptx::tc_fence_after();
        // Each 32-column block of O is transposed among groups of lanes so that a store instruction
        // writes whole row segments: bf16 rows (64 bytes per block) by 4 lanes, fp32 partial rows
        // (128 bytes) by 8 lanes.
        const bool split = a.n_split > 1;
        const bool has = ok && it.n_tiles > 0;
        const int64_t row0 = split ? (static_cast<int64_t>(it.t) * a.n_split + it.sp) * a.H : static_cast<int64_t>(it.t) * a.H;
        const int wrow = (warp & 3) * 32;  // this warp's first head row
#pragma unroll 1
        for (int c = 0; c < 16; ++c) {
          uint32_t o[32];
          if (has) {
            ptx::tmem_ld32(tmem + lane_base + c * 32, o);
            ptx::tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;  // an item without keys (or a failed one) writes zeros
          }
          if (split) {
            uint4 v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              v[e] = make_uint4(__float_as_uint(__uint_as_float(o[4 * e]) * inv_l),
                                __float_as_uint(__uint_as_float(o[4 * e + 1]) * inv_l),
                                __float_as_uint(__uint_as_float(o[4 * e + 2]) * inv_l),
                                __float_as_uint(__uint_as_float(o[4 * e + 3]) * inv_l));
            transpose_chunks<8>(v);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int hr = wrow + (lane & ~7) + k;
              if (hr < a.H)
                ptx::st_global_v4_hint(a.part_o + (row0 + hr) * kDV + c * 32 + (lane & 7) * 4, v[k], policy);
            }
          } else {
            uint4 v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              v[e] = make_uint4(pack_bf16(__uint_as_float(o[8 * e]) * inv_l, __uint_as_float(o[8 * e + 1]) * inv_l),
                                pack_bf16(__uint_as_float(o[8 * e + 2]) * inv_l, __uint_as_float(o[8 * e + 3]) * inv_l),
                                pack_bf16(__uint_as_float(o[8 * e + 4]) * inv_l, __uint_as_float(o[8 * e + 5]) * inv_l),
                                pack_bf16(__uint_as_float(o[8 * e + 6]) * inv_l, __uint_as_float(o[8 * e + 7]) * inv_l));
            transpose_chunks<4>(v);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int hr = wrow + (lane & ~3) + k;
              if (hr < a.H)
                ptx::st_global_v4_hint(a.out + (row0 + hr) * kDV + c * 32 + (lane & 3) * 8, v[k], policy);
            }
          }
        }
        if (it.n_tiles > 0) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(baddr(bars.o_free));  // O has been read: the next item may overwrite it
          g += it.n_tiles;
          ++nq;
        }
      }
    } else if (warp == kCreditWarp) {
      // ---- slot credits back to rank 0: slot ps is re-armed for tile gi + kSlots once tile gi's
      // products completed (a re-armed slot that no tile reaches is never waited on)
      int g = 0;
      bool ok = true;
      for (int j = 0; ok; ++j) {
        Item it;
        if (!read_item(bars, sched, j, &it, abort_flag, a) || it.t < 0) break;
        if (lane == 0) {
          for (int i = 0; i < it.n_tiles; ++i) {
            const int gi = g + i, ps = gi % kSlots;
            if (!ptx::mbar_wait(baddr(bars.slot_free[ps]), (gi / kSlots) & 1, abort_flag, a.status, a.limit_ns)) {
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx(baddr(bars.p_full[ps]), kSlotBytes);
            ptx::mbar_arrive_cluster(ptx::map_to_rank(baddr(bars.p_empty[ps]), 0));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        g += it.n_tiles;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();  // no remote access into either CTA's shared memory after this point
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kvmap) {
  attn_body<kMode>(a, &qmap, &kvmap);
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_loss_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap kvmap) {
  attn_body<kMode | 2>(a, &qmap, &kvmap);
}

// Merges the partial results of one (token, head) row: with per-part running max m_s (log2 domain),
// sum l_s and normalised output O_s, the row's softmax weights over the union of the parts give
// O = sum_s l_s 2^(m_s - m) O_s / sum_s l_s 2^(m_s - m), m = max_s m_s.  The parts of a row are
// n_split (key split), or, in the balanced partition, the clusters its tiles were spread over.
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnArgs a) {
  const int t = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int np = a.bal_tiles > 0
                     ? bal_parts(t, a.bal_tiles, static_cast<int64_t>(a.T) * a.bal_tiles, a.n_clusters)
                     : a.n_split;
  const int64_t base = static_cast<int64_t>(t) * a.n_split * a.H + h;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
  float m = -INFINITY;
  for (int s = 0; s < np; ++s) m = fmaxf(m, ml[base + static_cast<int64_t>(s) * a.H].x);
  float wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // loads of a few parts are issued before they are used (one memory round trip per group)
  for (int s0 = 0; s0 < np; s0 += 4) {
    float4 o[4];
    float2 p[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (s0 + u < np) {
        const int64_t r = base + static_cast<int64_t>(s0 + u) * a.H;
        p[u] = ml[r];
        o[u] = reinterpret_cast<const float4*>(a.part_o + r * kDV)[threadIdx.x];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (s0 + u < np) {
        const float wt = (p[u].y > 0.f && m > -INFINITY) ? p[u].y * fast_exp2(p[u].x - m) : 0.f;
        acc.x += wt * o[u].x; acc.y += wt * o[u].y; acc.z += wt * o[u].z; acc.w += wt * o[u].w;
        wsum += wt;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint2 pk;
  pk.x = pack_bf16(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(a.out + (static_cast<int64_t>(t) * a.H + h) * kDV)[threadIdx.x] = pk;
  if (threadIdx.x == 0 && a.lse != nullptr)
    a.lse[static_cast<int64_t>(t) * a.H + h] = wsum > 0.f ? (m + __log2f(wsum)) * 0.69314718055994530942f : -INFINITY;
}

}  // namespace

namespace {
template <int kMode>
cudaError_t launch_mode(const AttnArgs& a, const CUtensorMap& qmap, const CUtensorMap& kvmap, int ctas,
                        cudaStream_t stream) {
  auto kernel = (kMode & 2) ? indexer_loss_kernel<kMode & 1> : sparse_attn_kernel<kMode & 5>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (kMode & 2) ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, qmap, kvmap);
}
}  // namespace

cudaError_t launch_sparse_attn(const AttnArgs& a0, cudaStream_t stream) {
  if (a0.T <= 0) return cudaSuccess;
  AttnArgs a = a0;
  const bool loss = a.lse_in != nullptr;
  if (loss || a.n_split < 1 || a.part_o == nullptr || a.part_ml == nullptr) a.n_split = 1;
  if (loss || a.idx == nullptr || a.n_clusters < 1) a.bal_tiles = 0;  // (the host splits no row without buffers)
  // Q viewed as [T*H, 576] bf16, box 64 x 128 (rows past the tensor read as zero)
  CUtensorMap qmap;
  const uint64_t rows = static_cast<uint64_t>(a.T) * a.H;
  if (!encode_tmap_2d(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kDL, rows, kDL * 2, 64, 128))
    return cudaErrorInvalidValue;
  // the latent rows as [n_kv_rows, 576] bf16, box 64 x 64: the dense causal modes' tile loads
  CUtensorMap kvmap;
  if (!encode_tmap_2d(&kvmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.kv, kDL, static_cast<uint64_t>(a.n_kv_rows), kDL * 2,
                      64, kKT))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t items = static_cast<int64_t>(a.T) * a.n_split;
  const bool dense = a.idx == nullptr;
  cudaError_t e;
  if (loss) {
    // one independent score CTA per SM, each taking every gridDim-th token
    const int ctas = static_cast<int>(items < sms ? items : sms);
    e = dense ? launch_mode<3>(a, qmap, kvmap, ctas, stream) : launch_mode<2>(a, qmap, kvmap, ctas, stream);
    return e;
  }
  // one cluster per SM pair, each taking every n_clusters-th work item (balanced: the clusters the
  // partition was cut for)
  const int clusters = a.bal_tiles > 0 ? a.n_clusters : static_cast<int>(items < sms / 2 ? items : sms / 2);
  e = dense ? launch_mode<1>(a, qmap, kvmap, 2 * clusters, stream)
            : a.bal_tiles > 0 ? launch_mode<4>(a, qmap, kvmap, 2 * clusters, stream)
                              : launch_mode<0>(a, qmap, kvmap, 2 * clusters, stream);
  if (e != cudaSuccess || a.n_split == 1) return e;
  return launch_attn_combine(a, stream);
}

cudaError_t launch_attn_combine(const AttnArgs& a, cudaStream_t stream) {
  attn_combine_kernel<<<a.T * a.H, kDV / 4, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
