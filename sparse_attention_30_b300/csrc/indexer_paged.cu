// Lightning indexer over a paged FP8 key cache, one new query token per sequence (decode)
// (freezhihu.org/question/1978819912970555965, §2.1.1 indexer equation):
//     I[b,s] = sum_j w[b,j] * ReLU(q^I[b,j] . k^I[s])   for s < seq_lens[b]
//
// One tensor-core tile is D[128 keys x H_I] = K8[128 x 128] * Q8[H_I x 128]^T for the 128 keys of
// two 64-token pages; keys sit on the TMEM lanes, so the head-weighted ReLU sum for a key runs
// down one thread's registers.
//
// Work distribution: the key tiles of all sequences form one list (sequence after sequence); each
// of about two CTAs per SM takes an equal contiguous share of it, so the batch's tiles are spread
// evenly whatever the mix of lengths, and each CTA pays its prologue once.  A share may span
// several sequences ("segments"): the producer loads each segment's query tile into one of two
// query buffers ahead of time, the MMA warp switches buffers at segment boundaries and each
// epilogue warp reloads its copy of the head weights.  Every role walks the tile list with a cursor.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: query tiles, key pages through a ring of stages
//   warp 1      owns TMEM and issues the FP8 MMAs (K = 128 as 4 x K32), one elected lane
//   warps 2..9  two epilogue groups of 4 warps; group g drains TMEM buffer g (tiles i = g mod 2):
//               ReLU, weight, sum over heads, key scale, store fp32 scores (-inf for a key whose
//               page entry is out of range).
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTileKeys = 128;
constexpr int kRowBytes = 128;  // d_I = 128 FP8 values per key
constexpr int kKeyTileBytes = kTileKeys * kRowBytes;
constexpr int kThreads = 320;
constexpr int kCtasPerSm = 2;
constexpr int kMaxPagesPerTile = kTileKeys / 8;  // pages of at least 8 tokens

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int HI>
struct PagedCfg {
  static constexpr int STAGES = HI <= 64 ? 5 : 4;  // two CTAs per SM
  static constexpr int Q_BYTES = HI * kRowBytes;
  static constexpr int Q_STRIDE = align_up(Q_BYTES, 1024);
  static constexpr int TMEM_COLS = 2 * HI <= 128 ? 128 : 256;
  static constexpr int OFF_Q = 0;  // two query buffers
  static constexpr int OFF_K = OFF_Q + 2 * Q_STRIDE;
  static constexpr int OFF_W = OFF_K + STAGES * kKeyTileBytes;  // per epilogue warp: HI weights
  static constexpr int N_BARS = 2 * STAGES + 2 + 2 + 2 + 2 + 1;
  static constexpr int OFF_INFO = OFF_W + 8 * HI * 4;  // producer look-ahead: 32 tiles
  static constexpr int OFF_BAR = align_up(OFF_INFO + 32 * (4 + kMaxPagesPerTile) * 4, 8);
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM = OFF_MISC + 32 + 1024;
};

// Tiles of sequence b (its length clamped to [0, max_seq_len]; out-of-range lengths are reported
// once by CTA 0).
__device__ __forceinline__ int seq_len_of(const IndexerArgs& a, int b) {
  const int len = a.seq_lens[b];
  return len < 0 ? 0 : (len > a.S ? a.S : len);
}

// Position in the tile list: tile j of sequence b, which has nt tiles (b == rows: past the end).
struct Cursor {
  int b, j, nt, len;
};

__device__ __forceinline__ void load_seq(const IndexerArgs& a, Cursor& c) {
  c.len = c.b < a.rows ? seq_len_of(a, c.b) : 0;
  c.nt = (c.len + kTileKeys - 1) / kTileKeys;
}

__device__ __forceinline__ void advance(const IndexerArgs& a, Cursor& c) {
  if (++c.j < c.nt) return;
  c.j = 0;
  do {
    ++c.b;
    load_seq(a, c);
  } while (c.b < a.rows && c.nt == 0);
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) break;
  }
}

template <int HI>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    indexer_paged_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                         const IndexerArgs a) {
  using C = PagedCfg<HI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t sQ = ptx::smem_addr(smem + C::OFF_Q);
  const uint32_t sK = ptx::smem_addr(smem + C::OFF_K);
  const uint32_t bar0 = ptx::smem_addr(smem + C::OFF_BAR);
  auto k_full = [&](int s) { return bar0 + 8u * s; };
  auto k_empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto t_full = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
  auto t_empty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 + b); };
  auto q_full = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 4 + b); };
  auto q_empty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 6 + b); };
  const uint32_t mma_done = bar0 + 8u * (2 * C::STAGES + 8);
  int* misc = reinterpret_cast<int*>(smem + C::OFF_MISC);  // tmem slot, abort flag, b0, j0, n_tiles
  volatile int* abort_flag = misc + 1;

  // ---- this CTA's share of the tile list (warp 0 counts, everyone reads the result)
  if (warp == 0) {
    long long total = 0;
    for (int b0 = 0; b0 < a.rows; b0 += 32) {
      int nt = 0;
      if (b0 + lane < a.rows) {
        const int len = a.seq_lens[b0 + lane];
        if ((len < 0 || len > a.S) && blockIdx.x == 0) atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE);
        nt = (seq_len_of(a, b0 + lane) + kTileKeys - 1) / kTileKeys;
      }
      total += __reduce_add_sync(0xffffffffu, nt);
    }
    const long long g0 = total * blockIdx.x / gridDim.x, g1 = total * (blockIdx.x + 1) / gridDim.x;
    // first sequence whose tiles reach past g0
    long long before = 0;
    int bs = a.rows, js = 0;
    for (int b0 = 0; b0 < a.rows; b0 += 32) {
      const int b = b0 + lane;
      const int nt = b < a.rows ? (seq_len_of(a, b) + kTileKeys - 1) / kTileKeys : 0;
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const long long end = before + incl;  // tiles up to and including sequence b
      const unsigned hit = __ballot_sync(0xffffffffu, nt > 0 && end > g0);
      if (hit) {
        const int l = __ffs(hit) - 1;
        const long long start_l = __shfl_sync(0xffffffffu, end, l) - __shfl_sync(0xffffffffu, nt, l);
        bs = b0 + l;
        js = static_cast<int>(g0 - start_l);
        break;
      }
      before += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      misc[2] = bs;
      misc[3] = js;
      misc[4] = static_cast<int>(g1 - g0);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(k_full(s), 1);
      ptx::mbar_init(k_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(t_full(b), 1);
      ptx::mbar_init(t_empty(b), 4);
      ptx::mbar_init(q_full(b), 1);
      ptx::mbar_init(q_empty(b), 1);
    }
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&qmap);
    ptx::prefetch_tensormap(&kmap);
  }
  __syncthreads();
  const int n_tiles = misc[4];
  if (n_tiles <= 0) return;  // uniform over the CTA, before any allocation
  Cursor start{misc[2], misc[3], 0, 0};
  load_seq(a, start);
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(misc), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    // The lanes look up 32 tiles at a time (lane l: tile i0 + l; its sequence position and the
    // block-table entries of its pages) so those dependent loads overlap; lane 0 then issues the
    // tiles in order: the segment's query tile when the sequence changes, then the key pages.
    int* info = reinterpret_cast<int*>(smem + C::OFF_INFO);  // [32][4]: b, j, len, bytes
    int* pages = info + 32 * 4;                               // [32][kMaxPagesPerTile]
    const int pg = a.page_size, per = kTileKeys / pg;
    Cursor c = start;
    for (int k = 0; k < lane; ++k) advance(a, c);
    int seg = -1, cur_b = -1, issued = 0;
    bool ok = true;
    for (int i0 = 0; ok && i0 < n_tiles; i0 += 32) {
      if (i0 + lane < n_tiles) {
        const int s0 = c.j * kTileKeys;
        const int32_t* bt = a.block_table + static_cast<int64_t>(c.b) * a.bt_stride;
        int nbytes = 0;
        for (int u = 0; u < per; ++u) {
          const int p = s0 / pg + u;
          int32_t phys = -1;
          if (p * pg < c.len) {
            phys = bt[p];
            if (phys >= 0 && phys < a.n_pages) nbytes += pg * kRowBytes;
            else { atomicCAS(a.status, 0, DSA_ERR_DEVICE_RANGE); phys = -1; }
          }
          pages[lane * kMaxPagesPerTile + u] = phys;
        }
        info[lane * 4] = c.b;
        info[lane * 4 + 1] = c.j;
        info[lane * 4 + 2] = c.len;
        info[lane * 4 + 3] = nbytes;
      }
      for (int k = 0; k < 32; ++k) advance(a, c);  // this lane's tile of the next round
      __syncwarp();
      if (lane == 0) {
        for (int k = 0; k < 32 && i0 + k < n_tiles; ++k) {
          const int i = i0 + k, b = info[k * 4];
          if (b != cur_b) {  // new segment: its query tile into the next buffer
            const int ns = seg + 1, qb = ns & 1;
            if (!ptx::mbar_wait(q_empty(qb), ((ns >> 1) & 1) ^ 1, abort_flag, a.status, a.limit_ns)) {
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx(q_full(qb), C::Q_BYTES);
            ptx::tma_load_2d(sQ + qb * C::Q_STRIDE, &qmap, q_full(qb), 0, b * HI);
            seg = ns;
            cur_b = b;
          }
          const int st = i % C::STAGES;
          if (!ptx::mbar_wait(k_empty(st), ((i / C::STAGES) & 1) ^ 1, abort_flag, a.status, a.limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t dst = sK + st * kKeyTileBytes;
          ptx::mbar_arrive_expect_tx(k_full(st), static_cast<uint32_t>(info[k * 4 + 3]));
          for (int u = 0; u < per; ++u) {
            const int32_t phys = pages[k * kMaxPagesPerTile + u];
            if (phys >= 0) ptx::tma_load_2d(dst + u * pg * kRowBytes, &kmap, k_full(st), 0, phys * pg);
          }
          ++issued;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();
    }
    if (lane == 0 && *abort_flag) {
      // let every copy already issued land before the CTA exits
      for (int i = (issued > C::STAGES ? issued - C::STAGES : 0); i < issued; ++i)
        drain_wait(k_full(i % C::STAGES), (i / C::STAGES) & 1, a.limit_ns);
      for (int qb = 0; qb < 2 && qb <= seg; ++qb) drain_wait(q_full(qb), ((seg - qb) >> 1) & 1, a.limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp, one elected lane)
    constexpr uint32_t kIdesc = ptx::instr_desc(kTileKeys, HI, 0, 0, 0, 0);
    auto wwait = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, a.status, a.limit_ns));
    };
    Cursor c = start;
    int seg = -1, cur_b = -1;
    uint64_t bdesc = 0;
    for (int i = 0; i < n_tiles; ++i) {
      if (c.b != cur_b) {
        if (seg >= 0) ptx::mma_commit_warp(q_empty(seg & 1));  // the previous query tile is free once read
        ++seg;
        cur_b = c.b;
        if (!wwait(q_full(seg & 1), (seg >> 1) & 1)) break;
        bdesc = ptx::smem_desc(sQ + (seg & 1) * C::Q_STRIDE, 16, 1024, ptx::kLayoutSw128);
      }
      const int st = i % C::STAGES;
      const int buf = i & 1;
      if (!wwait(k_full(st), (i / C::STAGES) & 1)) break;
      if (!wwait(t_empty(buf), ((i >> 1) & 1) ^ 1)) break;
      ptx::tc_fence_after();
      const uint64_t adesc = ptx::smem_desc(sK + st * kKeyTileBytes, 16, 1024, ptx::kLayoutSw128);
      const uint32_t d = tmem + buf * HI;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // K = 128 bytes = 4 x 32 FP8 values; +32 B = +2 in the descriptor
        ptx::mma_f8_warp(d, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
      ptx::mma_commit_warp(k_empty(st));
      ptx::mma_commit_warp(t_full(buf));
      advance(a, c);
    }
    ptx::mma_commit_warp(mma_done);
    drain_wait(mma_done, 0, a.limit_ns);
  } else {
    // ------------------------------------------------ epilogue
    const int g = (warp - 2) >> 2;  // tiles i = g mod 2 use TMEM buffer g
    const int sub = warp & 3;       // this warp may touch TMEM lanes [32*sub, 32*sub + 32)
    const int row = sub * 32 + lane;
    float* sW = reinterpret_cast<float*>(smem + C::OFF_W) + (warp - 2) * HI;  // this warp's copy
    // Cursors at tiles i, i + 2, i + 4 of this group.  A key's page entry is fetched four tiles
    // ahead and its scale two tiles ahead, so neither dependent load stalls the tile being finished.
    auto advance2 = [&](Cursor& c) {
      advance(a, c);
      advance(a, c);
    };
    auto page_of = [&](int i, const Cursor& c) -> int32_t {  // physical page of this thread's key, or -1
      const int s = c.j * kTileKeys + row;
      if (i >= n_tiles || s >= c.len) return -1;
      const int32_t phys = a.block_table[static_cast<int64_t>(c.b) * a.bt_stride + s / a.page_size];
      return (phys >= 0 && phys < a.n_pages) ? phys : -1;
    };
    auto scale_of = [&](int i, const Cursor& c, int32_t phys) -> float {
      const int s = c.j * kTileKeys + row;
      if (i >= n_tiles || s >= c.len || phys < 0) return 0.f;
      return a.k_scale[static_cast<int64_t>(phys) * a.page_size + s % a.page_size];
    };
    Cursor ca = start;
    if (g) advance(a, ca);
    Cursor cb = ca, cc = ca;
    advance2(cb);
    cc = cb;
    advance2(cc);
    int32_t page_a = page_of(g, ca), page_b = page_of(g + 2, cb);
    float sk_next = scale_of(g, ca, page_a);
    int cur_b = -1;
    for (int i = g; i < n_tiles; i += 2) {
      if (ca.b != cur_b) {
        // this warp's head weights for the new sequence: w' = w * q_scale (ReLU is positively
        // homogeneous, so the query scale folds into the weight)
        cur_b = ca.b;
        __syncwarp();  // every lane is done with the old weights
        for (int j = lane; j < HI; j += 32) {
          const int64_t o = static_cast<int64_t>(cur_b) * HI + j;
          sW[j] = a.w[o] * a.q_scale[o];
        }
        __syncwarp();
      }
      const float sk = sk_next;
      const int s = ca.j * kTileKeys + row;
      const bool kvalid = s < ca.len && page_a >= 0;
      const int32_t page_c = page_of(i + 4, cc);
      sk_next = scale_of(i + 2, cb, page_b);
      page_a = page_b;
      page_b = page_c;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(t_full(g), (i >> 1) & 1, abort_flag, a.status, a.limit_ns))) break;
      ptx::tc_fence_after();
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t taddr = tmem + (static_cast<uint32_t>(sub * 32) << 16) + g * HI;
#pragma unroll
      for (int cq = 0; cq < HI / 32; ++cq) {
        uint32_t v[32];
        ptx::tmem_ld32(taddr + cq * 32, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 w4 = reinterpret_cast<const float4*>(sW)[cq * 8 + j4];
          const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] = fmaf(fmaxf(__uint_as_float(v[j4 * 4 + e]), 0.f), wv[e], acc[e]);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(t_empty(g));
      if (s < ca.len)
        a.scores[static_cast<int64_t>(ca.b) * a.ld + s] = kvalid ? ((acc[0] + acc[1]) + (acc[2] + acc[3])) * sk : -INFINITY;
      ca = cb;
      cb = cc;
      advance2(cc);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

static_assert(PagedCfg<32>::SMEM <= 113 * 1024 && PagedCfg<64>::SMEM <= 113 * 1024 &&
                  PagedCfg<128>::SMEM <= 113 * 1024,
              "two CTAs per SM");

template <int HI>
cudaError_t launch_paged_t(const CUtensorMap& qm, const CUtensorMap& km, int max_keys, const IndexerArgs& a,
                           cudaStream_t stream) {
  using C = PagedCfg<HI>;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t upper = static_cast<int64_t>(a.rows) * ((max_keys + kTileKeys - 1) / kTileKeys);
  const int grid = static_cast<int>(upper < kCtasPerSm * sms ? upper : kCtasPerSm * sms);
  if (grid <= 0) return cudaSuccess;
  auto kern = indexer_paged_kernel<HI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, C::SMEM, stream>>>(qm, km, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_paged(const CUtensorMap& qm, const CUtensorMap& km, int H_I, int max_keys,
                                 const IndexerArgs& a, cudaStream_t stream) {
  switch (H_I) {
    case 32: return launch_paged_t<32>(qm, km, max_keys, a, stream);
    case 64: return launch_paged_t<64>(qm, km, max_keys, a, stream);
    case 128: return launch_paged_t<128>(qm, km, max_keys, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
