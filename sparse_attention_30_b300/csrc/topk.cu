// Fine-grained token selection (freezhihu.org/question/1978819912970555965, §2.1.2):
// for each query row keep the k positions with the largest indexer scores.
//
// One CTA per row; scores become order-preserving 32-bit keys and the selection is exact.
//   n <= k         every position is selected.
//   n <= kCandCap  the row is loaded into shared memory once and selected there.
//   otherwise      (sample and filter) a sample of kSample keys (kSample / 4 groups of four
//                  neighbours at evenly spread positions, one 16-byte load each, so the sample
//                  touches a quarter of the row's cache lines) gives a lower bound tau that the
//                  k-th largest key clears with overwhelming probability: the sample's rank-r
//                  key, r = the expected sample rank of the k-th largest key + 6 standard
//                  deviations + 2 (the extra margin covers neighbours whose scores correlate).  One pass over the row compacts the keys >= tau
//                  into shared memory; when between k and kCandCap of them were found, the
//                  exact selection runs on those.  Otherwise (a sample that missed, or heavy
//                  ties at tau) the row falls back to a radix select that re-reads it.
// The selection in shared memory is a three-level radix select (12 + 12 + 8 key bits); each
// level finds its bin with a block suffix scan built from warp shuffles.  Output slots are
// filled in no particular order.
#include <math.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;
constexpr int kCandCap = 6144;
constexpr int kSample = 4096;  // held in cand_key until the filter pass starts
constexpr int kUnroll = 8;     // float4 loads in flight per thread in the filter pass
static_assert(kSample <= kCandCap, "the sample is staged in the candidate buffer");
static_assert(kSample % (4 * kThreads) == 0 && kSample <= kCandCap + 1, "sample groups per thread; rows sampled are longer");

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkSmem {
  uint32_t hist[kBins];
  uint32_t cand_key[kCandCap];
  int32_t cand_pos[kCandCap];
  uint32_t warp_sum[kWarps];
  uint32_t n_out, n_cand, n_eq;
  uint32_t sel_bin, sel_above;
};

// Finds the largest bin b with (number of keys in bins >= b) >= kk, over nbins bins.
// Returns b in s.sel_bin and the count in bins > b in s.sel_above.
__device__ void select_bin(TopkSmem& s, int nbins, uint32_t kk) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (nbins + kThreads - 1) / kThreads;
  const int b0 = tid * per;
  uint32_t local = 0;
  for (int b = b0; b < b0 + per && b < nbins; ++b) local += s.hist[b];
  // suffix sum across the warp: incl = sum of local over lanes >= lane
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += v;
  }
  if (lane == 0) s.warp_sum[wid] = incl;
  __syncthreads();
  uint32_t above_warps = 0;
  for (int w = wid + 1; w < kWarps; ++w) above_warps += s.warp_sum[w];
  const uint32_t excl = above_warps + incl - local;  // keys in bins owned by higher threads
  if (excl < kk && excl + local >= kk) {
    uint32_t run = excl;
    for (int b = min(b0 + per, nbins) - 1; b >= b0; --b) {
      const uint32_t c = s.hist[b];
      if (run + c >= kk) {
        s.sel_bin = b;
        s.sel_above = run;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
}

// Three-level radix select over keys visited by `each(f)` (f(key) per key): returns a key thr and
// a count n_equal such that the top `rank` are the keys > thr plus n_equal of the keys == thr
// (thr is the rank-th largest key, or, when a coarser bin already splits the set exactly, the key
// just below that bin with n_equal = 0).
// With kLevels == 2 the last 8 key bits are left open: thr is the lowest key of the 24-bit prefix
// that holds the rank-th largest key (a lower bound of it) and n_equal is not set.
template <int kLevels = 3, class Each>
__device__ void radix_threshold(TopkSmem& s, uint32_t rank, Each&& each, uint32_t* thr, uint32_t* n_equal) {
  const int tid = threadIdx.x;
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0;
  __syncthreads();
  each([&](uint32_t key) { atomicAdd(&s.hist[key >> 20], 1u); });
  __syncthreads();
  select_bin(s, kBins, rank);
  const uint32_t top = s.sel_bin;
  uint32_t need = rank - s.sel_above;
  const uint32_t in_top = s.hist[top];
  __syncthreads();
  // Exact selection: when the bin that holds the rank-th key holds exactly the keys still needed,
  // every key of it is selected and no finer level is needed (thr just below the bin, no ties).
  // (Block-uniform: every thread read the same counts.)
  if constexpr (kLevels == 3) {
    if (in_top == need && top != 0) {
      *thr = (top << 20) - 1;
      *n_equal = 0;
      return;
    }
  }
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0;
  __syncthreads();
  each([&](uint32_t key) {
    if ((key >> 20) == top) atomicAdd(&s.hist[(key >> 8) & 0xFFFu], 1u);
  });
  __syncthreads();
  select_bin(s, kBins, need);
  const uint32_t pre24 = (top << 12) | s.sel_bin;
  need -= s.sel_above;
  const uint32_t in_pre24 = s.hist[s.sel_bin];
  __syncthreads();
  if constexpr (kLevels == 2) {
    *thr = pre24 << 8;
  } else {
    if (in_pre24 == need && pre24 != 0) {
      *thr = (pre24 << 8) - 1;
      *n_equal = 0;
      return;
    }
    for (int b = tid; b < 256; b += kThreads) s.hist[b] = 0;
    __syncthreads();
    each([&](uint32_t key) {
      if ((key >> 8) == pre24) atomicAdd(&s.hist[key & 0xFFu], 1u);
    });
    __syncthreads();
    select_bin(s, 256, need);
    *thr = (pre24 << 8) | s.sel_bin;
    *n_equal = need - s.sel_above;
    __syncthreads();
  }
}

// Appends, warp-aggregated, the positions whose predicate holds to out[] through counter *n.
__device__ __forceinline__ void append(uint32_t* n, int32_t* out, uint32_t cap, bool take, int pos,
                                       uint32_t key, uint32_t* keys) {
  const uint32_t active = __activemask();
  const uint32_t m = __ballot_sync(active, take);
  if (!m) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(active) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(n, static_cast<uint32_t>(__popc(m)));
  base = __shfl_sync(active, base, leader);
  if (take) {
    const uint32_t c = base + __popc(m & ((1u << lane) - 1u));
    if (c < cap) {
      out[c] = pos;
      if (keys) keys[c] = key;
    }
  }
}

// Emits the top k of the `count` candidates in shared memory (k <= count).
__device__ void select_from_candidates(TopkSmem& s, uint32_t count, uint32_t k, int32_t* out) {
  uint32_t thr, n_equal;
  radix_threshold(
      s, k,
      [&](auto&& f) {
        for (uint32_t i = threadIdx.x; i < count; i += kThreads) f(s.cand_key[i]);
      },
      &thr, &n_equal);
  for (uint32_t i = threadIdx.x; i < count; i += kThreads) {
    const uint32_t key = s.cand_key[i];
    bool take = key > thr;
    if (key == thr) take = atomicAdd(&s.n_eq, 1u) < n_equal;
    append(&s.n_out, out, k, take, s.cand_pos[i], 0, nullptr);
  }
}

// Row t's length (columns that take part in the selection).
__device__ __forceinline__ int row_length(const TopkArgs& a, int t) {
  int64_t n64 = a.row_lens ? static_cast<int64_t>(a.row_lens[t]) : a.q_pos0 + t + 1;
  if (!a.row_lens && n64 > a.n_cols) n64 = a.n_cols;
  if (n64 > a.ld) n64 = a.ld;
  if (n64 < 0) n64 = 0;
  return static_cast<int>(n64);
}

// Rows with n <= kCandCap: every position (n <= k), or one read into shared memory and the exact
// selection there.
__device__ void short_row(TopkSmem& s, const float* row, int n, uint32_t k, int32_t* out, int k_slots) {
  const int tid = threadIdx.x;
  if (static_cast<uint32_t>(n) <= k) {
    for (int i = tid; i < k_slots; i += kThreads) out[i] = i < n ? i : -1;
    return;
  }
  if (tid == 0) { s.n_out = 0; s.n_cand = 0; s.n_eq = 0; }
  for (int i = tid; i < n; i += kThreads) {
    s.cand_key[i] = order_key(row[i]);
    s.cand_pos[i] = i;
  }
  __syncthreads();
  select_from_candidates(s, n, k, out);
}

// The sample's lower bound: kSample keys in groups of four neighbours at evenly spread positions,
// tau = the sample's rank-r key, returned as a float bound.  {x >= tau_f} is a prefix of the key
// order for non-NaN x (it takes both zeros or neither), so it holds the row's top k whenever it
// has k members.  Needs n >= kSample.
__device__ float sample_bound(TopkSmem& s, const float* row, int n, uint32_t k) {
  const int tid = threadIdx.x;
  {
    constexpr int kGroups = kSample / 4, kPer = kGroups / kThreads;
    const float4* row4 = reinterpret_cast<const float4*>(row);
    const int64_t n4 = n >> 2;
    float4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) v[u] = row4[static_cast<int64_t>(tid + u * kThreads) * n4 / kGroups];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      uint32_t* d = s.cand_key + 4 * (tid + u * kThreads);
      d[0] = order_key(v[u].x);
      d[1] = order_key(v[u].y);
      d[2] = order_key(v[u].z);
      d[3] = order_key(v[u].w);
    }
  }
  __syncthreads();
  const float mu = static_cast<float>(k) * kSample / n;  // expected sample keys >= the k-th largest
  uint32_t r = static_cast<uint32_t>(mu + 6.f * sqrtf(mu) + 2.f);
  if (r > kSample) r = kSample;
  uint32_t tau, unused;
  radix_threshold<2>(
      s, r,
      [&](auto&& f) {
        for (int i = tid; i < kSample; i += kThreads) f(s.cand_key[i]);
      },
      &tau, &unused);
  return __uint_as_float((tau & 0x80000000u) ? (tau & 0x7FFFFFFFu) : ~tau);
}

// Compacts the positions p in [p0, p1) (p0 a multiple of 4) with row[p] >= tau_f into the
// candidate buffer; s.n_cand counts them all, including those beyond its capacity.
__device__ void filter_range(TopkSmem& s, const float* row, int p0, int p1, float tau_f) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int q0 = p0 >> 2, q1 = p1 >> 2;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  for (int b = q0; b < q1; b += kThreads * kUnroll) {  // block-uniform trip count
    const int i0 = b + tid;
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kThreads;
      v[u] = i < q1 ? __ldg(row4 + i) : make_float4(NAN, NAN, NAN, NAN);  // NaN never passes
    }
    uint32_t mask = 0;  // bit 4u + c: element c of v[u]
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      mask |= (v[u].x >= tau_f ? 1u : 0u) << (4 * u);
      mask |= (v[u].y >= tau_f ? 2u : 0u) << (4 * u);
      mask |= (v[u].z >= tau_f ? 4u : 0u) << (4 * u);
      mask |= (v[u].w >= tau_f ? 8u : 0u) << (4 * u);
    }
    if (!__any_sync(0xffffffffu, mask != 0)) continue;
    const uint32_t cnt = __popc(mask);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    uint32_t base = 0;
    if (lane == 31) base = atomicAdd(&s.n_cand, incl);
    base = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
    while (mask) {
      const int bit = __ffs(mask) - 1;
      mask &= mask - 1;
      const int pos = 4 * (i0 + (bit >> 2) * kThreads) + (bit & 3);
      if (base < static_cast<uint32_t>(kCandCap)) {
        s.cand_key[base] = order_key(row[pos]);  // an L1 hit: the loads above were cached
        s.cand_pos[base] = pos;
      }
      ++base;
    }
  }
  for (int i = (q1 << 2) + tid; i < p1; i += kThreads) {
    const float x = row[i];
    append(&s.n_cand, s.cand_pos, kCandCap, x >= tau_f, i, order_key(x), s.cand_key);
  }
}

// Radix select over the whole row, re-read from global memory (the general fallback).
__device__ void full_row_select(TopkSmem& s, const float* row, int n, uint32_t k, int32_t* out) {
  const int tid = threadIdx.x;
  if (tid == 0) { s.n_out = 0; s.n_eq = 0; }
  uint32_t thr, n_equal;
  radix_threshold(
      s, k,
      [&](auto&& f) {
        for (int i = tid; i < n; i += kThreads) f(order_key(row[i]));
      },
      &thr, &n_equal);
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t key = order_key(row[i]);
    bool take = key > thr;
    if (key == thr) take = atomicAdd(&s.n_eq, 1u) < n_equal;
    append(&s.n_out, out, k, take, i, 0, nullptr);
  }
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TopkSmem& s = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int t = blockIdx.x;
  const int n = row_length(a, t);
  const uint32_t k = static_cast<uint32_t>(a.k);
  int32_t* out = a.idx + static_cast<int64_t>(t) * a.k;
  const float* row = a.scores + static_cast<int64_t>(t) * a.ld;  // 16-byte aligned rows
  if (n <= kCandCap) {
    short_row(s, row, n, k, out, a.k);
    return;
  }
  if (threadIdx.x == 0) { s.n_out = 0; s.n_cand = 0; s.n_eq = 0; }
  const float tau_f = sample_bound(s, row, n, k);
  filter_range(s, row, 0, n, tau_f);
  __syncthreads();
  const uint32_t found = s.n_cand;
  if (found >= k && found <= static_cast<uint32_t>(kCandCap)) select_from_candidates(s, found, k, out);
  else full_row_select(s, row, n, k, out);
}

// Few long rows (decode): a cluster of `cluster` CTAs per row.  Every CTA derives the same bound
// from the same sample and filters its 1/cluster of the row into its own candidate buffer; rank 0
// gathers the candidates through distributed shared memory and selects.  A rank-0 fallback (the
// whole row) covers a sample that missed or overflowing candidates.
__global__ void __launch_bounds__(kThreads) topk_cluster_kernel(const TopkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TopkSmem& s = *reinterpret_cast<TopkSmem*>(smem_raw);
  const uint32_t rank = ptx::cluster_ctarank();
  uint32_t csize;
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
  const int t = blockIdx.x / csize;
  const int n = row_length(a, t);
  const uint32_t k = static_cast<uint32_t>(a.k);
  int32_t* out = a.idx + static_cast<int64_t>(t) * a.k;
  const float* row = a.scores + static_cast<int64_t>(t) * a.ld;
  if (n <= kCandCap) {  // uniform over the cluster: rank 0 alone, no cluster barrier
    if (rank == 0) short_row(s, row, n, k, out, a.k);
    return;
  }
  if (threadIdx.x == 0) { s.n_out = 0; s.n_cand = 0; s.n_eq = 0; }
  const float tau_f = sample_bound(s, row, n, k);
  const int seg = ((n + 4 * static_cast<int>(csize) - 1) / (4 * static_cast<int>(csize))) * 4;
  const int p0 = min(n, static_cast<int>(rank) * seg), p1 = min(n, p0 + seg);
  filter_range(s, row, p0, p1, tau_f);
  __syncthreads();
  ptx::cluster_sync_all();  // every rank's candidates are complete and visible to the cluster
  __shared__ uint32_t base_of[8], total_s;
  __shared__ int overflow_s;
  if (rank == 0 && threadIdx.x == 0) {
    uint32_t total = 0;
    int overflow = 0;
    for (uint32_t r = 0; r < csize; ++r) {
      const uint32_t c = r == 0 ? s.n_cand : ld_cluster_u32(ptx::map_to_rank(ptx::smem_addr(&s.n_cand), r));
      if (c > static_cast<uint32_t>(kCandCap)) overflow = 1;
      base_of[r] = total;
      total += c;
    }
    total_s = total;
    overflow_s = overflow || total > static_cast<uint32_t>(kCandCap) || total < k;
  }
  __syncthreads();
  if (rank == 0 && !overflow_s) {
    // append the other ranks' candidates after rank 0's own
    for (uint32_t r = 1; r < csize; ++r) {
      const uint32_t b = base_of[r], c = (r + 1 < csize ? base_of[r + 1] : total_s) - b;
      const uint32_t kr = ptx::map_to_rank(ptx::smem_addr(s.cand_key), r);
      const uint32_t pr = ptx::map_to_rank(ptx::smem_addr(s.cand_pos), r);
      for (uint32_t i = threadIdx.x; i < c; i += kThreads) {
        s.cand_key[b + i] = ld_cluster_u32(kr + 4 * i);
        s.cand_pos[b + i] = static_cast<int32_t>(ld_cluster_u32(pr + 4 * i));
      }
    }
  }
  __syncthreads();
  ptx::cluster_sync_all();  // the other ranks' shared memory is no longer read after this point
  if (rank != 0) return;
  if (!overflow_s) select_from_candidates(s, total_s, k, out);
  else full_row_select(s, row, n, k, out);
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(TopkSmem));
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // rows spread over clusters when there are too few rows to fill the GPU (decode)
  int csize = 1;
  while (csize < 8 && a.T * csize * 2 <= sms) csize *= 2;
  if (csize == 1 || a.ld <= kCandCap) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    topk_kernel<<<a.T, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.T * csize);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, a);
}

}  // namespace dsa
