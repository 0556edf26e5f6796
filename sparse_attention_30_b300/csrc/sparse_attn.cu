// Sparse attention over the selected latent rows, MQA mode of MLA
// (freezhihu.org/question/1978819912970555965, §2.1.2 output equation and §2.2):
//     o[t,h,:] = sum_{s in S_t} softmax_s(scale * q[t,h,:] . c_s) * c_s[0:512]
// Every head of token t sees the same rows c_s, so per token this is a dense
// [H x 576] x [576 x |S_t|] product followed by [H x |S_t|] x [|S_t| x 512].
//
// Layout on the chip (one CTA = one token x one half of the value dims):
//   TMEM (512 columns): O half [128 heads x 256] fp32 at columns 0..255,
//                       S tile [128 heads x 32 keys] fp32 at columns 256..287.
//   SMEM: Q [128 x 576] bf16 as 9 K-major 128B-swizzled blocks of 64 dims;
//         two buffers of 32 gathered latent rows in the same layout (the QK^T B operand,
//         and, read MN-major, the PV B operand); P [128 x 32] bf16, 64B-swizzled.
// The output does not fit TMEM for all 512 value dims next to S, so the two value halves
// run in two CTAs that both compute S (QK^T is recomputed once per half).
//
// Per 32-key tile: cp.async gather of the next tile overlaps the current tile's
// S = Q K^T (tcgen05.mma, 36 x K16), the softmax (thread = head = TMEM lane),
// and O += P V (2 x K16, N = 256).  The running max is only moved when it grows by more
// than 2^8 (log2 domain), which rescales O in TMEM; the final 1/l is applied on the way out.
#include <cuda_bf16.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 128;
constexpr int kKT = 32;                       // keys per tile
constexpr int kDL = 576, kDV = 512, kHalf = 256;
constexpr int kBlocks = kDL / 64;             // 9 swizzle blocks of 64 bf16 (128 B)
constexpr int kQBlockBytes = 128 * 128;       // 128 rows x 128 B
constexpr int kQBytes = kBlocks * kQBlockBytes;
constexpr int kKVBlockBytes = kKT * 128;
constexpr int kKVBytes = kBlocks * kKVBlockBytes;
constexpr int kPBytes = 128 * kKT * 2;
constexpr int kOffQ = 0;
constexpr int kOffKV = kQBytes;
constexpr int kOffP = kOffKV + 2 * kKVBytes;
constexpr int kSmem = kOffP + kPBytes + 1024;  // + alignment slack
constexpr int kChunksPerRow = kDL * 2 / 16;   // 72 16-byte chunks per latent row
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;
constexpr float kRescaleThreshold = 8.0f;     // log2 units

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Physical latent row of selected position s for token t, or -1 if the slot is empty or
// the position / page is out of range.
__device__ __forceinline__ int64_t latent_row(const AttnArgs& a, int t, int32_t s, bool* range_err) {
  if (s < 0) return -1;
  if (a.block_table == nullptr) {
    if (s >= a.n_kv_rows) { *range_err = true; return -1; }
    return s;
  }
  if (s / a.page_size >= a.bt_stride) { *range_err = true; return -1; }  // past this row of the table
  const int32_t page = a.block_table[static_cast<int64_t>(t) * a.bt_stride + s / a.page_size];
  const int64_t r = static_cast<int64_t>(page) * a.page_size + s % a.page_size;
  if (page < 0 || r >= a.n_kv_rows) { *range_err = true; return -1; }
  return r;
}

// Gathers the 32 latent rows of tile `tile` into KV buffer `dst` (9 swizzled blocks).
__device__ __forceinline__ void gather_tile(const AttnArgs& a, int t, int tile, uint32_t dst,
                                            int32_t* s_valid, bool* range_err) {
  const int32_t* idx = a.idx + static_cast<int64_t>(t) * a.k;
  for (int q = threadIdx.x; q < kKT * kChunksPerRow; q += kThreads) {
    const int r = q / kChunksPerRow, cc = q % kChunksPerRow;
    const int slot = tile * kKT + r;
    const int32_t s = slot < a.k ? __ldg(idx + slot) : -1;
    const int64_t pr = latent_row(a, t, s, range_err);
    const int blk = cc >> 3, c = cc & 7;
    const uint32_t d = dst + blk * kKVBlockBytes + r * 128 + ((c ^ (r & 7)) << 4);
    const uint16_t* src = a.kv + (pr < 0 ? 0 : pr * kDL) + cc * 8;
    ptx::cp_async16(d, src, pr >= 0);
    if (cc == 0) s_valid[r] = pr >= 0;
  }
}

__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag_s;
  __shared__ int32_t s_valid[2][kKT];

  const int t = blockIdx.x, v = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = tid;  // head row = TMEM lane
  volatile int* abort_flag = &abort_flag_s;

  const uint32_t sQ = ptx::smem_addr(smem + kOffQ);
  const uint32_t sKV0 = ptx::smem_addr(smem + kOffKV);
  const uint32_t sP = ptx::smem_addr(smem + kOffP);
  uint8_t* pP = smem + kOffP;
  const uint32_t bar_s = ptx::smem_addr(&bars[0]);
  const uint32_t bar_o = ptx::smem_addr(&bars[1]);

  if (tid == 0) {
    ptx::mbar_init(bar_s, 1);
    ptx::mbar_init(bar_o, 1);
    abort_flag_s = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_addr(&tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }

  // number of 32-key tiles: valid slots come first, so stop at the first tile whose
  // first slot is empty
  const int32_t* idx_row = a.idx + static_cast<int64_t>(t) * a.k;
  const int max_tiles = (a.k + kKT - 1) / kKT;

  // ---- Q (rows >= H are zero) and the first KV tile
  {
    const uint16_t* qrow = a.q + static_cast<int64_t>(t) * a.H * kDL;
    for (int q = tid; q < 128 * kChunksPerRow; q += kThreads) {
      const int r = q / kChunksPerRow, cc = q % kChunksPerRow;
      const int blk = cc >> 3, c = cc & 7;
      const uint32_t d = sQ + blk * kQBlockBytes + r * 128 + ((c ^ (r & 7)) << 4);
      const bool ok = r < a.H;
      ptx::cp_async16(d, qrow + (ok ? r * kDL + cc * 8 : 0), ok);
    }
  }
  bool range_err = false;
  int n_tiles = 0;
  if (max_tiles > 0 && idx_row[0] >= 0) {
    n_tiles = 1;
    gather_tile(a, t, 0, sKV0, s_valid[0], &range_err);
  }
  ptx::cp_async_commit();

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tS = tmem + kColS;
  const uint32_t tO = tmem;

  constexpr uint32_t kIdescS = ptx::instr_desc(128, kKT, 1, 1, 0, 0);
  constexpr uint32_t kIdescPV = ptx::instr_desc(128, kHalf, 1, 1, 0, 1);
  const uint64_t descQ = ptx::smem_desc(sQ, 16, 1024, ptx::kLayoutSw128);
  const uint64_t descP = ptx::smem_desc(sP, 16, 512, ptx::kLayoutSw64);

  float m_used = -INFINITY;  // running max (log2 domain) the exponentials are taken against
  float l = 0.f;             // running sum of exp2(x - m_used)
  uint32_t phase_s = 0, phase_o = 0;
  bool ok = true;

  for (int i = 0; ok && i < n_tiles; ++i) {
    const int buf = i & 1;
    const uint32_t sKV = sKV0 + buf * kKVBytes;
    // prefetch tile i+1 into the other buffer (its previous contents were last read by
    // the PV MMA of tile i-1, which completed before this iteration)
    if (i + 1 < max_tiles && idx_row[(i + 1) * kKT] >= 0) {
      n_tiles = i + 2;
      gather_tile(a, t, i + 1, sKV0 + (buf ^ 1) * kKVBytes, s_valid[buf ^ 1], &range_err);
    }
    ptx::cp_async_commit();
    ptx::cp_async_wait<1>();
    ptx::fence_proxy_async_smem();
    __syncthreads();

    // ---- S = Q K^T for 32 keys
    if (tid == 0) {
      ptx::tc_fence_after();
#pragma unroll 1
      for (int kb = 0; kb < kBlocks; ++kb) {
        const uint64_t da = descQ + ((kb * kQBlockBytes) >> 4);
        const uint64_t db = ptx::smem_desc(sKV + kb * kKVBlockBytes, 16, 1024, ptx::kLayoutSw128);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // 16 dims = 32 B = +2 in the descriptor
          ptx::mma_bf16(tS, da + 2 * ks, db + 2 * ks, kIdescS, (kb | ks) ? 1u : 0u);
      }
      ptx::mma_commit(bar_s);
    }
    if (!ptx::mbar_wait(bar_s, phase_s, abort_flag, a.status, a.limit_ns)) { ok = false; break; }
    phase_s ^= 1;
    ptx::tc_fence_after();

    // ---- softmax on this thread's head row
    uint32_t sr[32];
    ptx::tmem_ld32(tS + lane_base, sr);
    ptx::tmem_wait_ld();
    float x[kKT];
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < kKT; ++j) {
      x[j] = s_valid[buf][j] ? __uint_as_float(sr[j]) * a.scale_log2 : -INFINITY;
      mt = fmaxf(mt, x[j]);
    }
    const float m_new = fmaxf(m_used, mt);
    const bool need = (i == 0) || (m_new > m_used + kRescaleThreshold);
    if (__any_sync(0xffffffffu, need)) {
      // O and l are kept against m_used; move m_used up to m_new (O rescaled in TMEM)
      const float f = (i == 0) ? 0.f : fast_exp2(m_used - m_new);
      if (i > 0) {
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + lane_base + c * 32, o);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          ptx::tmem_st32(tO + lane_base + c * 32, o);
        }
        ptx::tmem_wait_st();
      }
      l *= f;
      m_used = m_new;
    }
    float psum = 0.f;
    uint32_t packed[kKT / 2];
#pragma unroll
    for (int j = 0; j < kKT; j += 2) {
      const float p0 = fast_exp2(x[j] - m_used), p1 = fast_exp2(x[j + 1] - m_used);
      psum += p0 + p1;
      packed[j / 2] = pack_bf16(p0, p1);
    }
    l += psum;
    // P row h: 64 bytes = 4 chunks of 16 B, 64B swizzle (chunk c lands at c ^ ((h >> 1) & 3))
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 val = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
      *reinterpret_cast<uint4*>(pP + h * 64 + ((c ^ ((h >> 1) & 3)) << 4)) = val;
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();

    // ---- O += P V over this value half (V read MN-major from the gathered rows)
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t vbase = sKV + (v * (kHalf / 64)) * kKVBlockBytes;
#pragma unroll
      for (int ks = 0; ks < kKT / 16; ++ks) {
        const uint64_t db = ptx::smem_desc(vbase + ks * 16 * 128, kKVBlockBytes, 1024, ptx::kLayoutSw128);
        ptx::mma_bf16(tO, descP + 2 * ks, db, kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
      }
      ptx::mma_commit(bar_o);
    }
    if (!ptx::mbar_wait(bar_o, phase_o, abort_flag, a.status, a.limit_ns)) { ok = false; break; }
    phase_o ^= 1;
    ptx::tc_fence_after();
  }
  ptx::cp_async_wait<0>();
  if (range_err) atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE);

  // ---- epilogue: O / l -> bf16
  const bool has_rows = n_tiles > 0 && ok;
  const float inv_l = (has_rows && l > 0.f) ? 1.f / l : 0.f;
  uint16_t* orow = a.out + (static_cast<int64_t>(t) * a.H + h) * kDV + v * kHalf;
#pragma unroll 1
  for (int c = 0; c < kHalf / 32; ++c) {
    uint32_t o[32];
    ptx::tmem_ld32(tO + lane_base + c * 32, o);
    ptx::tmem_wait_ld();
    if (h < a.H) {
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = has_rows ? pack_bf16(__uint_as_float(o[2 * j]) * inv_l, __uint_as_float(o[2 * j + 1]) * inv_l) : 0u;
      uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    }
  }
  if (v == 0 && a.lse != nullptr && h < a.H)
    a.lse[static_cast<int64_t>(t) * a.H + h] =
        has_rows ? (m_used + __log2f(l)) * 0.69314718055994530942f : -INFINITY;

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  sparse_attn_kernel<<<dim3(a.T, 2), kThreads, kSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
