// Lightning indexer (freezhihu.org/question/1978819912970555965, §2.1.1 indexer equation):
//     I[t,s] = sum_j w[t,j] * ReLU(q^I[t,j] . k^I[s])
// on FP8 e4m3 inputs with per-token scales, over the preceding keys s <= t.
//
// One tensor-core tile is D[128 keys x 256] = K8[128 x 128] * Q8[256 x 128]^T, where the 256
// columns are (token, head) pairs: 256 / H_I tokens x H_I heads.  Keys sit on the TMEM lanes,
// so the head-weighted ReLU sum for a (token, key) pair runs down one thread's registers with no
// cross-thread reduction.  (The decode indexer over a paged cache is in indexer_paged.cu.)
//
// Warp roles (64 + 128 x NSPLIT threads: 576 for up to 64 heads, 320 for 128):
//   warp 0      TMA producer: the query tile once, then key tiles through a ring of stages
//   warp 1      owns TMEM and issues the FP8 MMAs (K = 128 as 4 x K32), one elected lane
//   warps 2..   epilogue: every tile's TMEM buffer is drained by all of them, the NSPLIT warps
//               that share a lane quarter (w mod 4) splitting its columns; head weights in
//               registers; ReLU, weight, sum over heads, key scale, causal mask, store fp32 scores.
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTileKeys = 128;
constexpr int kRowBytes = 128;  // d_I = 128 FP8 values per row
constexpr int kKeyTileBytes = kTileKeys * kRowBytes;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
__host__ __device__ constexpr int pow2_cols(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

template <int HI>
struct IdxCfg {
  static constexpr int NCOL = 256;
  static constexpr int TT = NCOL / HI;
  static constexpr int NACC = (TT >= 32) ? 1 : ((32 / TT) < 4 ? (32 / TT) : 4);
  // The epilogue splits the columns among NSPLIT warps per TMEM lane quarter: quarters of 64
  // columns (whole tokens up to 64 heads), halves for 128 heads (a quarter would split a token).
  static constexpr int NSPLIT = HI == 128 ? 2 : 4;
  static constexpr int SPLIT = NCOL / NSPLIT;  // columns per epilogue thread
  static constexpr int TS = TT / NSPLIT;       // tokens per split
  static constexpr int THREADS = 64 + 128 * NSPLIT;
  static constexpr int STAGES = 6;
  static constexpr int Q_BYTES = NCOL * kRowBytes;
  static constexpr int TMEM_COLS = pow2_cols(2 * NCOL);
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = align_up(Q_BYTES, 1024);
  static constexpr int OFF_W = OFF_K + STAGES * kKeyTileBytes;
  static constexpr int N_BARS = 1 + 2 * STAGES + 4 + 1;
  static constexpr int OFF_BAR = align_up(OFF_W + NCOL * 4, 8);
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
};

// Bounded wait that ignores the abort flag: used only to drain copies and MMAs already
// in flight before the CTA releases its shared and tensor memory.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) break;
  }
}

template <int HI>
__global__ void __launch_bounds__(IdxCfg<HI>::THREADS, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const IndexerArgs a) {
  using C = IdxCfg<HI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- this CTA's work: query rows [row0, row0 + TT) x key tiles [tb, te)
  const int row0 = blockIdx.x * C::TT;
  const int rlast = min(a.rows, row0 + C::TT) - 1;
  const int64_t e = a.q_pos0 + rlast + 1;
  const int key_end = static_cast<int>(e < a.S ? e : a.S);
  const int n_tiles_all = (key_end + kTileKeys - 1) / kTileKeys;
  const int tb = blockIdx.y * a.tiles_per_cta;
  const int te = min(n_tiles_all, tb + a.tiles_per_cta);
  if (tb >= te) return;  // uniform over the CTA, before any barrier or allocation
  const int n_tiles = te - tb;

  const uint32_t sQ = ptx::smem_addr(smem + C::OFF_Q);
  const uint32_t sK = ptx::smem_addr(smem + C::OFF_K);
  float* sW = reinterpret_cast<float*>(smem + C::OFF_W);
  const uint32_t bar0 = ptx::smem_addr(smem + C::OFF_BAR);
  auto q_full = [&]() { return bar0; };
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + C::STAGES + s); };
  auto t_full = [&](int b) { return bar0 + 8u * (1 + 2 * C::STAGES + b); };
  auto t_empty = [&](int b) { return bar0 + 8u * (3 + 2 * C::STAGES + b); };
  const uint32_t mma_done = bar0 + 8u * (5 + 2 * C::STAGES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full(), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(k_full(s), 1);
      ptx::mbar_init(k_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(t_full(b), 1);
      ptx::mbar_init(t_empty(b), 4 * C::NSPLIT);  // every epilogue warp drains every buffer
    }
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&qmap);
    ptx::prefetch_tensormap(&kmap);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp >= 2) {
    // w'[tt, j] = w[t, j] * q_scale[t, j]: ReLU is positively homogeneous, so the query
    // scale moves outside the ReLU and folds into the head weight.
    for (int i = threadIdx.x - 64; i < C::NCOL; i += C::THREADS - 64) {
      const int tt = i / HI, j = i % HI;
      const int r = row0 + tt;
      float v = 0.f;
      if (r < a.rows) {
        const int64_t o = static_cast<int64_t>(r) * HI + j;
        v = a.w[o] * a.q_scale[o];
      }
      sW[i] = v;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      ptx::mbar_arrive_expect_tx(q_full(), C::Q_BYTES);
      ptx::tma_load_2d(sQ, &qmap, q_full(), 0, row0 * HI);
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % C::STAGES;
        const uint32_t ph = (i / C::STAGES) & 1;
        if (!ptx::mbar_wait(k_empty(st), ph ^ 1, abort_flag, a.status, a.limit_ns)) break;
        const int s0 = (tb + i) * kTileKeys;
        const uint32_t dst = sK + st * kKeyTileBytes;
        ptx::mbar_arrive_expect_tx(k_full(st), kKeyTileBytes);
        ptx::tma_load_2d(dst, &kmap, k_full(st), 0, s0);
        ++issued;
      }
      if (*abort_flag) {
        // let every copy already issued land before the CTA exits
        for (int i = (issued > C::STAGES ? issued - C::STAGES : 0); i < issued; ++i)
          drain_wait(k_full(i % C::STAGES), (i / C::STAGES) & 1, a.limit_ns);
        drain_wait(q_full(), 0, a.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp, one elected lane)
    constexpr uint32_t kIdesc = ptx::instr_desc(kTileKeys, C::NCOL, 0, 0, 0, 0);
    const uint64_t bdesc = ptx::smem_desc(sQ, 16, 1024, ptx::kLayoutSw128);
    auto wwait = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, a.status, a.limit_ns));
    };
    if (wwait(q_full(), 0)) {
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % C::STAGES;
        const uint32_t ph = (i / C::STAGES) & 1;
        const int buf = i & 1;
        const uint32_t bph = (i >> 1) & 1;
        if (!wwait(k_full(st), ph)) break;
        if (!wwait(t_empty(buf), bph ^ 1)) break;
        ptx::tc_fence_after();
        const uint64_t adesc = ptx::smem_desc(sK + st * kKeyTileBytes, 16, 1024, ptx::kLayoutSw128);
        const uint32_t d = tmem + buf * C::NCOL;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // K = 128 bytes = 4 x 32 FP8 values; +32 B = +2 in the descriptor
          ptx::mma_f8_warp(d, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
        ptx::mma_commit_warp(k_empty(st));
        ptx::mma_commit_warp(t_full(buf));
      }
    }
    ptx::mma_commit_warp(mma_done);
    drain_wait(mma_done, 0, a.limit_ns);
  } else {
    // ------------------------------------------------ epilogue
    // The NSPLIT warps that share TMEM lanes [32*sub, 32*sub + 32) (sub = w mod 4) split the
    // columns: split h takes the (token, head) columns [SPLIT*h, SPLIT*h + SPLIT) of every tile, so
    // each thread keeps the head weights of its columns in registers for the whole block.  Read
    // from shared memory for every tile instead (1 KB per thread per tile), the weights kept the
    // L1 data pipe 82% busy and set the kernel's time.  TMEM is read 16 columns at a time so that
    // the weights, the columns and the sums fit the registers a thread has.
    constexpr int HALF = C::SPLIT;
    constexpr int TH = C::TS;  // tokens per split
    const int h = (warp - 2) >> 2;
    const int sub = warp & 3;
    const int row = sub * 32 + lane;
    float wr[HALF];
#pragma unroll
    for (int c = 0; c < HALF; ++c) wr[c] = sW[h * HALF + c];
    // the key scale of a tile is loaded one tile ahead so its latency does not land on the tile
    // being finished
    auto key_of = [&](int i) { return (tb + i) * kTileKeys + row; };
    auto scale_of = [&](int i) -> float {  // 0 for a key past the range
      const int s = key_of(i);
      return (i < n_tiles && s < key_end) ? a.k_scale[s] : 0.f;
    };
    float sk_next = scale_of(0);
    for (int i = 0; i < n_tiles; ++i) {
      const float sk = sk_next;
      sk_next = scale_of(i + 1);
      const int s = key_of(i);
      const bool kvalid = s < key_end;
      const int buf = i & 1;
      const uint32_t bph = (i >> 1) & 1;
      if (!ptx::mbar_wait(t_full(buf), bph, abort_flag, a.status, a.limit_ns)) break;
      ptx::tc_fence_after();
      float acc[TH][C::NACC];
#pragma unroll
      for (int tt = 0; tt < TH; ++tt)
#pragma unroll
        for (int e = 0; e < C::NACC; ++e) acc[tt][e] = 0.f;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(sub * 32) << 16) + buf * C::NCOL + h * HALF;
#pragma unroll
      for (int cc = 0; cc < HALF / 16; ++cc) {
        uint32_t v[16];
        ptx::tmem_ld16(taddr + cc * 16, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = cc * 16 + j;
          const int tt = col / HI, hj = col % HI;
          acc[tt][hj % C::NACC] = fmaf(fmaxf(__uint_as_float(v[j]), 0.f), wr[col], acc[tt][hj % C::NACC]);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(t_empty(buf));
#pragma unroll
      for (int tt = 0; tt < TH; ++tt) {
        float sum = acc[tt][0];
#pragma unroll
        for (int e = 1; e < C::NACC; ++e) sum += acc[tt][e];
        const int r = row0 + h * TH + tt;
        if (kvalid && r < a.rows && s <= a.q_pos0 + r) {
          a.scores[static_cast<int64_t>(r) * a.ld + s] = sum * sk;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int HI>
cudaError_t launch_t(const CUtensorMap& qm, const CUtensorMap& km, int max_keys, const IndexerArgs& a0,
                     cudaStream_t stream) {
  using C = IdxCfg<HI>;
  IndexerArgs a = a0;
  const int n_key_tiles = (max_keys + kTileKeys - 1) / kTileKeys;
  const int gx = (a.rows + C::TT - 1) / C::TT;
  // long key ranges per CTA amortise its prologue (TMEM allocation, weights, the query tile and
  // the pipeline fill: one CTA per SM); keep at least about four CTAs per SM for balance
  const int64_t total = static_cast<int64_t>(gx) * n_key_tiles;
  const int64_t tpc = total / (4 * 148);
  a.tiles_per_cta = static_cast<int>(tpc < 32 ? 32 : (tpc > 256 ? 256 : tpc));
  const int gy = (n_key_tiles + a.tiles_per_cta - 1) / a.tiles_per_cta;
  if (gx == 0 || gy == 0) return cudaSuccess;
  auto kern = indexer_kernel<HI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(gx, gy), C::THREADS, C::SMEM, stream>>>(qm, km, a);
  return cudaGetLastError();
}

}  // namespace

int indexer_supported_heads(int H_I, bool paged) {
  // prefill tiles always have 256 (token, head) columns; a decode tile has one token's
  // H_I columns and the epilogue drains them 32 at a time
  switch (H_I) {
    case 4: case 8: case 16: return paged ? 0 : 1;
    case 32: case 64: case 128: return 1;
    default: return 0;
  }
}

bool encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                       uint32_t box_rows);

cudaError_t launch_indexer(const uint8_t* q8, const uint8_t* k8, int64_t n_key_rows, int H_I, bool paged,
                           int max_keys, const IndexerArgs& a, cudaStream_t stream) {
  CUtensorMap qm, km;
  const uint32_t ncol = paged ? H_I : 256;
  if (!encode_tmap_2d_u8(&qm, q8, kRowBytes, static_cast<uint64_t>(a.rows) * H_I, kRowBytes, ncol))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d_u8(&km, k8, kRowBytes, n_key_rows, kRowBytes, paged ? a.page_size : kTileKeys))
    return cudaErrorInvalidValue;
  if (!indexer_supported_heads(H_I, paged)) return cudaErrorInvalidValue;
  if (paged) return launch_indexer_paged(qm, km, H_I, max_keys, a, stream);
  switch (H_I) {
    case 64: return launch_t<64>(qm, km, max_keys, a, stream);
    case 128: return launch_t<128>(qm, km, max_keys, a, stream);
    case 4: return launch_t<4>(qm, km, max_keys, a, stream);
    case 8: return launch_t<8>(qm, km, max_keys, a, stream);
    case 16: return launch_t<16>(qm, km, max_keys, a, stream);
    case 32: return launch_t<32>(qm, km, max_keys, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
