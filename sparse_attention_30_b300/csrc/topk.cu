// Fine-grained token selection (freezhihu.org/question/1978819912970555965, §2.1.2):
// for each query row keep the k positions with the largest indexer scores.
//
// One CTA per row runs an exact radix select on order-preserving 32-bit keys:
//   pass 1  (reads the row)   histogram of the top 12 key bits in shared memory;
//                             a block suffix-scan (warp shuffles) finds the bin B that
//                             holds the k-th largest key;
//   pass 2  (reads the row)   positions in bins above B go straight to the output; keys
//                             in bin B are kept as (key, position) candidates in shared
//                             memory (if more than kCandCap, the next levels re-read the
//                             row from global memory instead);
//   levels 2, 3               12-bit and 8-bit histograms of the candidates pin the exact
//                             32-bit threshold key and how many keys equal to it to take;
//   final                     candidates above the threshold, then the needed number of
//                             equal ones, are appended to the output.
// Output slots are filled in no particular order; rows with n <= k select everything.
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;
constexpr int kCandCap = 6144;

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

// Visits the keys of bin `top` (top 12 bits) either from the candidate buffer or, if it
// overflowed, by re-reading the row.  f(key, pos) is called for each.
template <class F>
__device__ __forceinline__ void for_each_candidate(const TopkSmem& s, bool in_smem, uint32_t ncand,
                                                   const float* row, int n, uint32_t top, F&& f) {
  if (in_smem) {
    for (uint32_t i = threadIdx.x; i < ncand; i += kThreads) f(s.cand_key[i], s.cand_pos[i]);
  } else {
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = order_key(row[i]);
      if ((key >> 20) == top) f(key, i);
    }
  }
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TopkSmem& s = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  int64_t n64 = a.row_lens ? static_cast<int64_t>(a.row_lens[t]) : a.q_pos0 + t + 1;
  if (!a.row_lens && n64 > a.n_cols) n64 = a.n_cols;
  if (n64 > a.ld) n64 = a.ld;
  if (n64 < 0) n64 = 0;
  const int n = static_cast<int>(n64);
  const int k = a.k;
  int32_t* out = a.idx + static_cast<int64_t>(t) * k;
  const float* row = a.scores + static_cast<int64_t>(t) * a.ld;

  if (n <= k) {
    for (int i = tid; i < k; i += kThreads) out[i] = i < n ? i : -1;
    return;
  }

  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0;
  if (tid == 0) { s.n_out = 0; s.n_cand = 0; s.n_eq = 0; }
  __syncthreads();

  // ---- pass 1: top-12-bit histogram (rows are 16-byte aligned: ld % 4 == 0)
  const int n4 = n >> 2;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  for (int i = tid; i < n4; i += kThreads) {
    const float4 v = row4[i];
    atomicAdd(&s.hist[order_key(v.x) >> 20], 1u);
    atomicAdd(&s.hist[order_key(v.y) >> 20], 1u);
    atomicAdd(&s.hist[order_key(v.z) >> 20], 1u);
    atomicAdd(&s.hist[order_key(v.w) >> 20], 1u);
  }
  for (int i = (n4 << 2) + tid; i < n; i += kThreads) atomicAdd(&s.hist[order_key(row[i]) >> 20], 1u);
  __syncthreads();
  select_bin(s, kBins, static_cast<uint32_t>(k));
  const uint32_t top = s.sel_bin;
  uint32_t need = static_cast<uint32_t>(k) - s.sel_above;  // keys still to take from bin `top`
  const uint32_t ncand = s.hist[top];
  const bool in_smem = ncand <= static_cast<uint32_t>(kCandCap);
  __syncthreads();

  // ---- pass 2: emit bins above `top`, collect bin `top`
  auto visit = [&](uint32_t key, int pos) {
    const uint32_t b = key >> 20;
    if (b > top) {
      out[atomicAdd(&s.n_out, 1u)] = pos;
    } else if (b == top && in_smem) {
      const uint32_t c = atomicAdd(&s.n_cand, 1u);
      s.cand_key[c] = key;
      s.cand_pos[c] = pos;
    }
  };
  for (int i = tid; i < n4; i += kThreads) {
    const float4 v = row4[i];
    visit(order_key(v.x), 4 * i);
    visit(order_key(v.y), 4 * i + 1);
    visit(order_key(v.z), 4 * i + 2);
    visit(order_key(v.w), 4 * i + 3);
  }
  for (int i = (n4 << 2) + tid; i < n; i += kThreads) visit(order_key(row[i]), i);
  __syncthreads();

  // ---- level 2: bits 19..8 of the keys in bin `top`
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0;
  __syncthreads();
  for_each_candidate(s, in_smem, ncand, row, n, top,
                     [&](uint32_t key, int) { atomicAdd(&s.hist[(key >> 8) & 0xFFFu], 1u); });
  __syncthreads();
  select_bin(s, kBins, need);
  const uint32_t mid = s.sel_bin;
  need -= s.sel_above;
  __syncthreads();

  // ---- level 3: bits 7..0 of the keys with prefix (top, mid)
  for (int b = tid; b < 256; b += kThreads) s.hist[b] = 0;
  __syncthreads();
  const uint32_t pre24 = (top << 12) | mid;
  for_each_candidate(s, in_smem, ncand, row, n, top, [&](uint32_t key, int) {
    if ((key >> 8) == pre24) atomicAdd(&s.hist[key & 0xFFu], 1u);
  });
  __syncthreads();
  select_bin(s, 256, need);
  const uint32_t thr = (pre24 << 8) | s.sel_bin;
  const uint32_t n_equal = need - s.sel_above;  // keys equal to thr to take
  __syncthreads();

  // ---- final: candidates above the threshold, then n_equal of those equal to it
  for_each_candidate(s, in_smem, ncand, row, n, top, [&](uint32_t key, int pos) {
    if (key > thr) {
      out[atomicAdd(&s.n_out, 1u)] = pos;
    } else if (key == thr) {
      if (atomicAdd(&s.n_eq, 1u) < n_equal) out[atomicAdd(&s.n_out, 1u)] = pos;
    }
  });
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(TopkSmem));
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  topk_kernel<<<a.T, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
