// Small device helpers shared by the attention kernels (forward and backward).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace dsa {
namespace attn {

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// First empty slot of a selection row (valid slots come first), by the whole warp: each round
// probes 32 evenly spaced positions of the open interval, so k = 2048 takes three dependent loads.
__device__ inline int first_empty_slot(const int32_t* idx_row, int k) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = k;  // every slot below lo is valid; the first empty one is in [lo, hi]
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int p = lo + lane * step;
    const bool neg = p < hi && __ldg(idx_row + p) < 0;
    const unsigned m = __ballot_sync(0xffffffffu, neg);
    const int f = m ? __ffs(m) - 1 : 32;
    if (f == 0) return lo;
    const int nlo = lo + (f - 1) * step + 1;
    hi = f < 32 ? lo + f * step : hi;
    lo = nlo;
  }
  const int p = lo + lane;
  const unsigned m = __ballot_sync(0xffffffffu, p < hi && __ldg(idx_row + p) < 0);
  return m ? lo + __ffs(m) - 1 : hi;
}

// Transpose of N x N 16-byte chunks among N consecutive lanes: lane i's v[k] (chunk k of its
// row) becomes chunk i of lane k's row, so that N lanes then store one row's N chunks together.
template <int N>
__device__ __forceinline__ void transpose_chunks(uint4 (&v)[N]) {
  const int i = threadIdx.x & (N - 1);
#pragma unroll
  for (int sh = N / 2; sh >= 1; sh >>= 1) {
    const bool up = (i & sh) != 0;
#pragma unroll
    for (int k = 0; k < N; ++k) {
      if (k & sh) continue;
      const uint4 send = up ? v[k] : v[k ^ sh];
      uint4 recv;
      recv.x = __shfl_xor_sync(0xffffffffu, send.x, sh);
      recv.y = __shfl_xor_sync(0xffffffffu, send.y, sh);
      recv.z = __shfl_xor_sync(0xffffffffu, send.z, sh);
      recv.w = __shfl_xor_sync(0xffffffffu, send.w, sh);
      if (up) v[k] = recv;
      else v[k ^ sh] = recv;
    }
  }
}

}  // namespace attn
}  // namespace dsa
