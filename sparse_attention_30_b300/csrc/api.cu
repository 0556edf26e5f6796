// C-ABI entry points of libdsa.so (declared in include/dsa.h): argument checks on the
// host, kernel launches on the caller's stream, the chunked forward driver, and the
// per-device status word the kernels report into.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {

__device__ int g_status;  // per-device: DSA_OK or the first device-side error recorded

namespace {

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
std::mutex g_mu;

// Address of this device's status word (looked up once per device).
int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

__global__ void wait_timeout_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // nobody arrives: the bounded wait must give up, record the timeout and return
  ptx::mbar_wait(ptx::smem_addr(&bar), 0, &abort_flag, status, limit_ns);
  __syncthreads();
}

}  // namespace

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                       uint32_t box_rows) {
  return encode_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, inner, rows, inner, box_inner, box_rows);
}

uint64_t wait_limit_ns() {
  static const uint64_t limit = []() -> uint64_t {
    const char* e = std::getenv("DSA_WAIT_LIMIT_MS");
    if (e == nullptr) return kWaitLimitNs;
    char* end = nullptr;
    const long long ms = std::strtoll(e, &end, 10);
    if (end == e || *end != '\0' || ms <= 0 || ms > 3600000) return kWaitLimitNs;
    return static_cast<uint64_t>(ms) * 1000000ull;
  }();
  return limit;
}

cudaError_t launch_wait_timeout_selftest(int* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace dsa

using namespace dsa;

namespace dsa {

dsa_status_t check_index_args(const uint8_t* q8, const float* q_scale, const float* w, const uint8_t* k8,
                              const float* k_scale, int T, int S, int H_I, int64_t q_pos0, const float* scores,
                              int64_t ld) {
  if (T < 0 || S < 1 || q_pos0 < 0) return DSA_ERR_INVALID_ARG;
  if (!q8 || !q_scale || !w || !k8 || !k_scale || !scores) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(scores)) return DSA_ERR_INVALID_ARG;
  if (ld % 4 != 0 || ld < std::min<int64_t>(S, q_pos0 + T)) return DSA_ERR_INVALID_ARG;
  if (!pow2(H_I) || H_I > 128) return DSA_ERR_INVALID_ARG;
  if (!indexer_supported_heads(H_I, false)) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * H_I > (1ll << 31) - 1 || q_pos0 + T > (1ll << 31) - 1) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

dsa_status_t check_paged_index_args(const uint8_t* q8, const float* q_scale, const float* w, const uint8_t* k8c,
                                    const float* ksc, int64_t n_pages, const int32_t* bt, int64_t bt_stride,
                                    const int32_t* lens, int B, int H_I, int page, int max_len, const float* scores,
                                    int64_t ld) {
  if (B < 0 || n_pages < 1 || max_len < 1 || bt_stride < 1) return DSA_ERR_INVALID_ARG;
  if (!q8 || !q_scale || !w || !k8c || !ksc || !bt || !lens || !scores) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8c) || !aligned16(scores)) return DSA_ERR_INVALID_ARG;
  if (ld % 4 != 0 || ld < max_len) return DSA_ERR_INVALID_ARG;
  if (page < 8 || page > 128 || 128 % page != 0) return DSA_ERR_INVALID_ARG;
  if (bt_stride < (max_len + page - 1) / page) return DSA_ERR_INVALID_ARG;
  if (!pow2(H_I) || H_I > 128) return DSA_ERR_INVALID_ARG;
  if (!indexer_supported_heads(H_I, true)) return DSA_ERR_UNSUPPORTED;
  if (n_pages * page > (1ll << 31) - 1) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

dsa_status_t check_topk_args(const float* scores, int64_t ld, int T, int64_t n_cols, int64_t q_pos0, int k,
                             const int32_t* idx, const int32_t* row_lens) {
  if (T < 0 || k < 1 || k > 65536 || q_pos0 < 0) return DSA_ERR_INVALID_ARG;
  if (!scores || !idx) return DSA_ERR_INVALID_ARG;
  if (!aligned16(scores) || ld % 4 != 0 || ld < 1) return DSA_ERR_INVALID_ARG;
  if (!row_lens && (n_cols < 1 || n_cols > ld)) return DSA_ERR_INVALID_ARG;
  if (ld > (1ll << 31) - 1) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

dsa_status_t check_attn_args(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows, const int32_t* bt,
                             int64_t bt_stride, int page, const int32_t* idx, int T, int H, int k,
                             const uint16_t* out) {
  if (T < 0 || H < 1 || k < 1 || k > 65536 || n_kv_rows < 1) return DSA_ERR_INVALID_ARG;
  if (!q || !kv || !idx || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  if (bt && (page < 1 || bt_stride < 1)) return DSA_ERR_INVALID_ARG;
  if (H > 128) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int* status_target(int32_t* dev_status) { return dev_status ? dev_status : status_ptr(); }

}  // namespace dsa

namespace {

dsa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// Every workspace starts with a 256-byte head whose first word is the status word of the calls
// that use it (read and cleared by dsa_status).
constexpr size_t kStatusHead = 256;

// Workspace layout of dsa_forward: [status head] [scores block (fp32)] [selection (int32), if not
// caller-owned] [key-split partial results (decode with few sequences)]
struct FwdPlan {
  int rows;          // query rows in total
  int chunk;         // rows scored per indexer / top-k launch
  int64_t ld;        // score row pitch (floats)
  int n_split;       // decode: partial results per sequence in the attention (1 = none)
  int bal_tiles;     // decode: virtual 64-key tiles per sequence of the balanced partition
  int n_clusters;    // decode: clusters the partition is cut for
  size_t scores_bytes, idx_bytes, part_o_bytes, part_ml_bytes, total;
};

// Decode attention runs one 2-SM cluster per sequence; with few sequences each one's selected
// keys are split over several clusters so that the 74 cluster slots of the GPU fill up.  (The
// balanced partition below spreads every pair's share evenly, but each extra work item costs a Q
// load and an fp32 partial epilogue: it measured slower for 32 and 64 sequences, 72.4 vs 68.4 us
// and 112.7 vs 93.8 us, so the decode forward keeps this split.)
int decode_split(int B) {
  if (B <= 0 || B >= 74) return 1;
  return std::max(1, std::min(4, 74 / B));
}

// Balanced partition of the attention (dsa_sparse_attn_split with n_split = 0): the rows' tiles,
// end to end, cut into equal contiguous ranges, one per 2-SM cluster (74 on a B300); a row spread
// over several clusters leaves one partial result per cluster.
struct BalPlan {
  int tpr, n_clusters, parts;
};
BalPlan plan_balanced(int rows, int tiles_per_row) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  BalPlan b{std::max(1, tiles_per_row), 1, 1};
  const int64_t G = static_cast<int64_t>(rows) * b.tpr;
  b.n_clusters = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms / 2, G)));
  for (int t = 0; t < rows; ++t) b.parts = std::max(b.parts, bal_parts(t, b.tpr, G, b.n_clusters));
  return b;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

dsa_status_t plan_forward(const dsa_forward_args* a, FwdPlan* p) {
  if (!a) return DSA_ERR_INVALID_ARG;
  if (a->H_I < 1 || a->H < 1 || a->k < 1 || a->k > 65536) return DSA_ERR_INVALID_ARG;
  if (a->mode == DSA_MODE_PREFILL) {
    if (a->T < 0 || a->S < 1 || a->q_pos0 < 0 || a->q_pos0 + a->T > a->S) return DSA_ERR_INVALID_ARG;
    p->rows = a->T;
    p->ld = (static_cast<int64_t>(a->S) + 3) & ~3ll;
    int chunk = a->chunk_rows > 0 ? a->chunk_rows : 0;
    if (chunk == 0) {
      // keep the fp32 score block near 1 GiB
      const int64_t c = (1ll << 28) / p->ld;
      chunk = static_cast<int>(std::max<int64_t>(256, std::min<int64_t>(c, 8192)));
    }
    p->chunk = std::max(1, std::min(chunk, std::max(1, a->T)));
  } else if (a->mode == DSA_MODE_DECODE) {
    if (a->B < 0 || a->max_seq_len < 1) return DSA_ERR_INVALID_ARG;
    p->rows = a->B;
    p->ld = (static_cast<int64_t>(a->max_seq_len) + 3) & ~3ll;
    p->chunk = std::max(1, a->B);
  } else {
    return DSA_ERR_INVALID_ARG;
  }
  p->n_split = a->mode == DSA_MODE_DECODE ? decode_split(a->B) : 1;
  p->bal_tiles = 0;
  p->n_clusters = 0;
  p->scores_bytes = align256(static_cast<size_t>(p->chunk) * p->ld * sizeof(float));
  p->idx_bytes = a->idx ? 0 : align256(static_cast<size_t>(std::max(1, p->rows)) * a->k * sizeof(int32_t));
  p->part_o_bytes = p->n_split > 1 ? align256(static_cast<size_t>(p->rows) * p->n_split * a->H * 512 * 4) : 0;
  p->part_ml_bytes = p->n_split > 1 ? align256(static_cast<size_t>(p->rows) * p->n_split * a->H * 2 * 4) : 0;
  // (same layout as dsa_sparse_attn_split's workspace: partial outputs, then partial max / sum)
  p->total = kStatusHead + p->scores_bytes + p->idx_bytes + p->part_o_bytes + p->part_ml_bytes;
  return DSA_OK;
}

// Device workspace of dsa_prefill_host: the status head, the keys once, then two slots of query-row
// chunk inputs and outputs (so that the copies of one chunk overlap the kernels of the other), and
// one score block.
struct HostPlan {
  FwdPlan f;
  size_t k8, k_scale, kv;                  // keys
  size_t q8, q_scale, w, q, idx, out, lse; // one slot (chunk rows)
  size_t slot, scores, total;
};

dsa_status_t plan_prefill_host(const dsa_forward_args* a, HostPlan* h) {
  if (!a || a->mode != DSA_MODE_PREFILL) return DSA_ERR_INVALID_ARG;
  dsa_status_t st = plan_forward(a, &h->f);
  if (st != DSA_OK) return st;
  const size_t C = static_cast<size_t>(h->f.chunk), S = static_cast<size_t>(a->S);
  h->k8 = align256(S * 128);
  h->k_scale = align256(S * 4);
  h->kv = align256(S * 576 * 2);
  h->q8 = align256(C * a->H_I * 128);
  h->q_scale = align256(C * a->H_I * 4);
  h->w = align256(C * a->H_I * 4);
  h->q = align256(C * a->H * 576 * 2);
  h->idx = align256(C * a->k * 4);
  h->out = align256(C * a->H * 512 * 2);
  h->lse = align256(C * a->H * 4);
  h->slot = h->q8 + h->q_scale + h->w + h->q + h->idx + h->out + h->lse;
  h->scores = h->f.scores_bytes;
  h->total = kStatusHead + h->k8 + h->k_scale + h->kv + 2 * h->slot + h->scores;
  return DSA_OK;
}

// Two non-blocking streams per device for the host pipeline's copies (created on first use).
bool copy_streams(cudaStream_t* in, cudaStream_t* out) {
  static cudaStream_t s_in[kMaxDevices], s_out[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!s_in[dev] && (cudaStreamCreateWithFlags(&s_in[dev], cudaStreamNonBlocking) != cudaSuccess ||
                     cudaStreamCreateWithFlags(&s_out[dev], cudaStreamNonBlocking) != cudaSuccess))
    return false;
  *in = s_in[dev];
  *out = s_out[dev];
  return true;
}

}  // namespace

extern "C" {

uint64_t dsa_wait_limit_ns(void) { return wait_limit_ns(); }

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_TIMEOUT: return "DSA_ERR_DEVICE_TIMEOUT";
    case DSA_ERR_DEVICE_RANGE: return "DSA_ERR_DEVICE_RANGE";
  }
  return "DSA_ERR_UNKNOWN";
}

int dsa_version(void) { return (2 << 16) | 0; }

dsa_status_t dsa_index(const uint8_t* q8, const float* q_scale, const float* w, const uint8_t* k8,
                       const float* k_scale, int T, int S, int H_I, int64_t q_pos0, float* scores, int64_t ld,
                       int32_t* dev_status, dsa_stream_t stream) {
  dsa_status_t st = check_index_args(q8, q_scale, w, k8, k_scale, T, S, H_I, q_pos0, scores, ld);
  if (st != DSA_OK || T == 0) return st;
  int* status = status_target(dev_status);
  if (!status) return DSA_ERR_CUDA;
  IndexerArgs a{};
  a.q_scale = q_scale; a.w = w; a.k_scale = k_scale;
  a.scores = scores; a.ld = ld; a.rows = T; a.S = S; a.q_pos0 = q_pos0;
  a.status = status; a.limit_ns = wait_limit_ns();
  const int max_keys = static_cast<int>(std::min<int64_t>(S, q_pos0 + T));
  return from_cuda(launch_indexer(q8, k8, S, H_I, false, max_keys, a, stream));
}

dsa_status_t dsa_index_paged(const uint8_t* q8, const float* q_scale, const float* w, const uint8_t* k8_cache,
                             const float* k_scale_cache, int64_t n_pages, const int32_t* block_table,
                             int64_t bt_stride, const int32_t* seq_lens, int B, int H_I, int page_size,
                             int max_seq_len, float* scores, int64_t ld, int32_t* dev_status, dsa_stream_t stream) {
  dsa_status_t st = check_paged_index_args(q8, q_scale, w, k8_cache, k_scale_cache, n_pages, block_table, bt_stride,
                                           seq_lens, B, H_I, page_size, max_seq_len, scores, ld);
  if (st != DSA_OK || B == 0) return st;
  int* status = status_target(dev_status);
  if (!status) return DSA_ERR_CUDA;
  IndexerArgs a{};
  a.q_scale = q_scale; a.w = w; a.k_scale = k_scale_cache;
  a.block_table = block_table; a.bt_stride = bt_stride; a.seq_lens = seq_lens; a.n_pages = n_pages;
  a.scores = scores; a.ld = ld; a.rows = B; a.S = max_seq_len; a.page_size = page_size;
  a.status = status; a.limit_ns = wait_limit_ns();
  return from_cuda(launch_indexer(q8, k8_cache, n_pages * page_size, H_I, true, max_seq_len, a, stream));
}

dsa_status_t dsa_topk(const float* scores, int64_t ld, int T, const int32_t* row_lens, int64_t n_cols,
                      int64_t q_pos0, int k, int32_t* idx, dsa_stream_t stream) {
  dsa_status_t st = check_topk_args(scores, ld, T, n_cols, q_pos0, k, idx, row_lens);
  if (st != DSA_OK || T == 0) return st;
  TopkArgs a{scores, ld, T, row_lens, n_cols, q_pos0, k, idx};
  return from_cuda(launch_topk(a, stream));
}

namespace {
dsa_status_t sparse_attn_split(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows, const int32_t* block_table,
                               int64_t bt_stride, int page_size, const int32_t* idx, int T, int H, int k, float scale,
                               uint16_t* out, float* lse, int n_split, float* part_o, float* part_ml,
                               int32_t* dev_status, cudaStream_t stream, int bal_tiles = 0, int n_clusters = 0) {
  dsa_status_t st = check_attn_args(q, kv, n_kv_rows, block_table, bt_stride, page_size, idx, T, H, k, out);
  if (st != DSA_OK || T == 0) return st;
  int* status = status_target(dev_status);
  if (!status) return DSA_ERR_CUDA;
  AttnArgs a{};
  a.q = q; a.kv = kv; a.n_kv_rows = n_kv_rows; a.block_table = block_table; a.bt_stride = bt_stride;
  a.page_size = page_size; a.idx = idx; a.T = T; a.H = H; a.k = k;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out; a.lse = lse; a.status = status; a.limit_ns = wait_limit_ns();
  a.n_split = n_split; a.part_o = part_o; a.part_ml = part_ml;
  a.bal_tiles = bal_tiles; a.n_clusters = n_clusters;
  return from_cuda(launch_sparse_attn(a, stream));
}
}  // namespace

size_t split_part_o_bytes(int T, int H, int n_split) {
  return align256(static_cast<size_t>(T) * n_split * H * 512 * 4);
}
size_t split_part_ml_bytes(int T, int H, int n_split) {
  return align256(static_cast<size_t>(T) * n_split * H * 2 * 4);
}

extern "C" size_t dsa_sparse_attn_split_workspace_size(int T, int H, int n_split) {
  if (T < 0 || H < 1 || H > 128 || n_split < 1 || n_split > 8) return 0;
  if (n_split == 1) return 0;
  return split_part_o_bytes(T, H, n_split) + split_part_ml_bytes(T, H, n_split);
}

extern "C" size_t dsa_sparse_attn_balanced_workspace_size(int T, int H, int k) {
  if (T < 1 || H < 1 || H > 128 || k < 1 || k > 65536) return 0;
  const BalPlan b = plan_balanced(T, (k + 63) / 64);
  if (b.parts == 1) return 0;
  return split_part_o_bytes(T, H, b.parts) + split_part_ml_bytes(T, H, b.parts);
}

extern "C" dsa_status_t dsa_sparse_attn_split(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows,
                                              const int32_t* block_table, int64_t bt_stride, int page_size,
                                              const int32_t* idx, int T, int H, int k, float scale, uint16_t* out,
                                              float* lse, int n_split, void* ws, size_t ws_bytes,
                                              int32_t* dev_status, dsa_stream_t stream) {
  if (n_split == 0) {  // balanced partition over every SM pair
    dsa_status_t st = check_attn_args(q, kv, n_kv_rows, block_table, bt_stride, page_size, idx, T, H, k, out);
    if (st != DSA_OK || T == 0) return st;
    const BalPlan b = plan_balanced(T, (k + 63) / 64);
    const size_t need = dsa_sparse_attn_balanced_workspace_size(T, H, k);
    if (need > 0 && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))) return DSA_ERR_WORKSPACE;
    char* w = static_cast<char*>(ws);
    return sparse_attn_split(q, kv, n_kv_rows, block_table, bt_stride, page_size, idx, T, H, k, scale, out, lse,
                             b.parts, b.parts > 1 ? reinterpret_cast<float*>(w) : nullptr,
                             b.parts > 1 ? reinterpret_cast<float*>(w + split_part_o_bytes(T, H, b.parts)) : nullptr,
                             dev_status, stream, b.tpr, b.n_clusters);
  }
  if (n_split < 1 || n_split > 8) return DSA_ERR_INVALID_ARG;
  if (n_split == 1)
    return sparse_attn_split(q, kv, n_kv_rows, block_table, bt_stride, page_size, idx, T, H, k, scale, out, lse, 1,
                             nullptr, nullptr, dev_status, stream);
  dsa_status_t st = check_attn_args(q, kv, n_kv_rows, block_table, bt_stride, page_size, idx, T, H, k, out);
  if (st != DSA_OK || T == 0) return st;
  const size_t need = dsa_sparse_attn_split_workspace_size(T, H, n_split);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DSA_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  return sparse_attn_split(q, kv, n_kv_rows, block_table, bt_stride, page_size, idx, T, H, k, scale, out, lse, n_split,
                           reinterpret_cast<float*>(w), reinterpret_cast<float*>(w + split_part_o_bytes(T, H, n_split)),
                           dev_status, stream);
}

extern "C" dsa_status_t dsa_sparse_attn(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows,
                                        const int32_t* block_table, int64_t bt_stride, int page_size,
                                        const int32_t* idx, int T, int H, int k, float scale, uint16_t* out,
                                        float* lse, int32_t* dev_status, dsa_stream_t stream) {
  return sparse_attn_split(q, kv, n_kv_rows, block_table, bt_stride, page_size, idx, T, H, k, scale, out, lse, 1,
                           nullptr, nullptr, dev_status, stream);
}

extern "C" dsa_status_t dsa_dense_causal_attn(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows, int T, int H,
                                              int64_t q_pos0, float scale, uint16_t* out, float* lse,
                                              int32_t* dev_status, dsa_stream_t stream) {
  if (T < 0 || H < 1 || q_pos0 < 0 || n_kv_rows < 1 || n_kv_rows > INT32_MAX) return DSA_ERR_INVALID_ARG;
  if (q_pos0 + static_cast<int64_t>(T) > n_kv_rows) return DSA_ERR_INVALID_ARG;
  if (!q || !kv || !out || !aligned16(q) || !aligned16(kv) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  if (H > 128) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  int* status = status_target(dev_status);
  if (!status) return DSA_ERR_CUDA;
  AttnArgs a{};
  a.q = q; a.kv = kv; a.n_kv_rows = n_kv_rows; a.idx = nullptr; a.T = T; a.H = H; a.k = 0; a.q_pos0 = q_pos0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out; a.lse = lse; a.status = status; a.limit_ns = wait_limit_ns(); a.n_split = 1;
  return from_cuda(launch_sparse_attn(a, stream));
}

extern "C" dsa_status_t dsa_indexer_loss(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows, const int32_t* idx,
                                         int T, int H, int k, int64_t q_pos0, float scale, const float* lse,
                                         const float* scores, int64_t ld, float* p, float* kl, double* loss_acc,
                                         int32_t* dev_status, dsa_stream_t stream) {
  if (T < 0 || H < 1 || n_kv_rows < 1 || n_kv_rows > INT32_MAX || ld < 1) return DSA_ERR_INVALID_ARG;
  if (!q || !kv || !lse || !scores || !aligned16(q) || !aligned16(kv)) return DSA_ERR_INVALID_ARG;
  if (idx) {
    if (k < 1 || k > 65536) return DSA_ERR_INVALID_ARG;
  } else {
    // dense warm-up: every position up to the row's own, so the rows must fit the keys and scores
    if (p || q_pos0 < 0 || q_pos0 + static_cast<int64_t>(T) > n_kv_rows || q_pos0 + static_cast<int64_t>(T) > ld)
      return DSA_ERR_INVALID_ARG;
  }
  if (H > 128) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  int* status = status_target(dev_status);
  if (!status) return DSA_ERR_CUDA;
  AttnArgs a{};
  a.q = q; a.kv = kv; a.n_kv_rows = n_kv_rows; a.idx = idx; a.T = T; a.H = H; a.k = idx ? k : 0;
  a.q_pos0 = idx ? 0 : q_pos0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status; a.limit_ns = wait_limit_ns(); a.n_split = 1;
  a.lse_in = lse; a.scores = scores; a.ld = ld; a.p_out = p; a.kl_out = kl; a.loss_acc = loss_acc;
  return from_cuda(launch_sparse_attn(a, stream));
}

size_t dsa_forward_workspace_size(const dsa_forward_args* args) {
  FwdPlan p;
  if (plan_forward(args, &p) != DSA_OK) return 0;
  return p.total;
}

dsa_status_t dsa_forward(const dsa_forward_args* a, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  FwdPlan p;
  dsa_status_t st = plan_forward(a, &p);
  if (st != DSA_OK) return st;
  if (!a->q8 || !a->q_scale || !a->w || !a->k8 || !a->k_scale || !a->q || !a->kv || !a->out)
    return DSA_ERR_INVALID_ARG;
  if (p.rows == 0) return DSA_OK;
  if (!ws || ws_bytes < p.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DSA_ERR_WORKSPACE;
  int32_t* wst = static_cast<int32_t*>(ws);
  char* body = static_cast<char*>(ws) + kStatusHead;
  float* scores = reinterpret_cast<float*>(body);
  int32_t* idx = a->idx ? a->idx : reinterpret_cast<int32_t*>(body + p.scores_bytes);
  cudaStream_t s = stream;

  if (a->mode == DSA_MODE_PREFILL) {
    st = check_index_args(a->q8, a->q_scale, a->w, a->k8, a->k_scale, a->T, a->S, a->H_I, a->q_pos0, scores, p.ld);
    if (st != DSA_OK) return st;
    st = check_attn_args(a->q, a->kv, a->S, nullptr, 0, 0, idx, a->T, a->H, a->k, a->out);
    if (st != DSA_OK) return st;
    for (int r0 = 0; r0 < a->T; r0 += p.chunk) {
      const int rows = std::min(p.chunk, a->T - r0);
      const int64_t pos0 = a->q_pos0 + r0;
      st = dsa_index(a->q8 + static_cast<int64_t>(r0) * a->H_I * 128, a->q_scale + static_cast<int64_t>(r0) * a->H_I,
                     a->w + static_cast<int64_t>(r0) * a->H_I, a->k8, a->k_scale, rows, a->S, a->H_I, pos0, scores,
                     p.ld, wst, s);
      if (st != DSA_OK) return st;
      st = dsa_topk(scores, p.ld, rows, nullptr, a->S, pos0, a->k, idx + static_cast<int64_t>(r0) * a->k, s);
      if (st != DSA_OK) return st;
    }
    return dsa_sparse_attn(a->q, a->kv, a->S, nullptr, 0, 0, idx, a->T, a->H, a->k, a->scale, a->out, a->lse, wst,
                           s);
  }
  // decode
  st = check_paged_index_args(a->q8, a->q_scale, a->w, a->k8, a->k_scale, a->n_pages, a->block_table, a->bt_stride,
                              a->seq_lens, a->B, a->H_I, a->page_size, a->max_seq_len, scores, p.ld);
  if (st != DSA_OK) return st;
  st = check_attn_args(a->q, a->kv, a->n_pages * a->page_size, a->block_table, a->bt_stride, a->page_size, idx, a->B,
                       a->H, a->k, a->out);
  if (st != DSA_OK) return st;
  st = dsa_index_paged(a->q8, a->q_scale, a->w, a->k8, a->k_scale, a->n_pages, a->block_table, a->bt_stride,
                       a->seq_lens, a->B, a->H_I, a->page_size, a->max_seq_len, scores, p.ld, wst, s);
  if (st != DSA_OK) return st;
  st = dsa_topk(scores, p.ld, a->B, a->seq_lens, p.ld, 0, a->k, idx, s);
  if (st != DSA_OK) return st;
  char* part = body + p.scores_bytes + p.idx_bytes;
  return sparse_attn_split(a->q, a->kv, a->n_pages * a->page_size, a->block_table, a->bt_stride, a->page_size, idx,
                           a->B, a->H, a->k, a->scale, a->out, a->lse, p.n_split,
                           p.n_split > 1 ? reinterpret_cast<float*>(part) : nullptr,
                           p.n_split > 1 ? reinterpret_cast<float*>(part + p.part_o_bytes) : nullptr, wst, s,
                           p.bal_tiles, p.n_clusters);
}

size_t dsa_forward_loss_workspace_size(const dsa_forward_args* args, int stage) {
  FwdPlan p;
  if (!args || args->mode != DSA_MODE_PREFILL || (stage != DSA_LOSS_SPARSE && stage != DSA_LOSS_DENSE_WARMUP) ||
      plan_forward(args, &p) != DSA_OK)
    return 0;
  return stage == DSA_LOSS_SPARSE ? p.total : kStatusHead + p.scores_bytes;
}

dsa_status_t dsa_forward_loss(const dsa_forward_args* a, int stage, float* kl, double* loss_acc, void* ws,
                              size_t ws_bytes, dsa_stream_t stream) {
  if (!a || a->mode != DSA_MODE_PREFILL || (stage != DSA_LOSS_SPARSE && stage != DSA_LOSS_DENSE_WARMUP))
    return DSA_ERR_INVALID_ARG;
  FwdPlan p;
  dsa_status_t st = plan_forward(a, &p);
  if (st != DSA_OK) return st;
  if (!a->q8 || !a->q_scale || !a->w || !a->k8 || !a->k_scale || !a->q || !a->kv || !a->out || !a->lse)
    return DSA_ERR_INVALID_ARG;
  if (p.rows == 0) return DSA_OK;
  const bool sparse = stage == DSA_LOSS_SPARSE;
  const size_t need = sparse ? p.total : kStatusHead + p.scores_bytes;
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DSA_ERR_WORKSPACE;
  int32_t* wst = static_cast<int32_t*>(ws);
  char* body = static_cast<char*>(ws) + kStatusHead;
  float* scores = reinterpret_cast<float*>(body);
  int32_t* idx = !sparse ? nullptr : a->idx ? a->idx : reinterpret_cast<int32_t*>(body + p.scores_bytes);
  st = check_index_args(a->q8, a->q_scale, a->w, a->k8, a->k_scale, a->T, a->S, a->H_I, a->q_pos0, scores, p.ld);
  if (st != DSA_OK) return st;
  if (sparse) {
    st = check_attn_args(a->q, a->kv, a->S, nullptr, 0, 0, idx, a->T, a->H, a->k, a->out);
    if (st != DSA_OK) return st;
  }
  cudaStream_t s = stream;
  for (int r0 = 0; r0 < a->T; r0 += p.chunk) {
    const int rows = std::min(p.chunk, a->T - r0);
    const int64_t pos0 = a->q_pos0 + r0;
    const uint16_t* q = a->q + static_cast<int64_t>(r0) * a->H * 576;
    uint16_t* out = a->out + static_cast<int64_t>(r0) * a->H * 512;
    float* lse = a->lse + static_cast<int64_t>(r0) * a->H;
    float* kl_c = kl ? kl + r0 : nullptr;
    st = dsa_index(a->q8 + static_cast<int64_t>(r0) * a->H_I * 128, a->q_scale + static_cast<int64_t>(r0) * a->H_I,
                   a->w + static_cast<int64_t>(r0) * a->H_I, a->k8, a->k_scale, rows, a->S, a->H_I, pos0, scores,
                   p.ld, wst, s);
    if (st != DSA_OK) return st;
    if (sparse) {
      int32_t* idx_c = idx + static_cast<int64_t>(r0) * a->k;
      st = dsa_topk(scores, p.ld, rows, nullptr, a->S, pos0, a->k, idx_c, s);
      if (st != DSA_OK) return st;
      st = dsa_sparse_attn(q, a->kv, a->S, nullptr, 0, 0, idx_c, rows, a->H, a->k, a->scale, out, lse, wst, s);
      if (st != DSA_OK) return st;
      st = dsa_indexer_loss(q, a->kv, a->S, idx_c, rows, a->H, a->k, 0, a->scale, lse, scores, p.ld, nullptr, kl_c,
                            loss_acc, wst, s);
    } else {
      st = dsa_dense_causal_attn(q, a->kv, a->S, rows, a->H, pos0, a->scale, out, lse, wst, s);
      if (st != DSA_OK) return st;
      st = dsa_indexer_loss(q, a->kv, a->S, nullptr, rows, a->H, 0, pos0, a->scale, lse, scores, p.ld, nullptr, kl_c,
                            loss_acc, wst, s);
    }
    if (st != DSA_OK) return st;
  }
  return DSA_OK;
}

size_t dsa_prefill_host_workspace_size(const dsa_forward_args* args) {
  HostPlan h;
  if (plan_prefill_host(args, &h) != DSA_OK) return 0;
  return h.total;
}

dsa_status_t dsa_prefill_host(const dsa_forward_args* a, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  HostPlan hp;
  dsa_status_t st = plan_prefill_host(a, &hp);
  if (st != DSA_OK) return st;
  if (!a->q8 || !a->q_scale || !a->w || !a->k8 || !a->k_scale || !a->q || !a->kv || !a->out)
    return DSA_ERR_INVALID_ARG;
  if (a->T == 0) return DSA_OK;
  if (!ws || ws_bytes < hp.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DSA_ERR_WORKSPACE;
  const int C = hp.f.chunk, H_I = a->H_I, H = a->H, K = a->k;
  int32_t* wst = static_cast<int32_t*>(ws);
  char* p = static_cast<char*>(ws) + kStatusHead;
  uint8_t* k8 = reinterpret_cast<uint8_t*>(p);
  float* k_scale = reinterpret_cast<float*>(p + hp.k8);
  uint16_t* kv = reinterpret_cast<uint16_t*>(p + hp.k8 + hp.k_scale);
  char* slots = p + hp.k8 + hp.k_scale + hp.kv;
  float* scores = reinterpret_cast<float*>(slots + 2 * hp.slot);
  struct Slot {
    uint8_t* q8; float* q_scale; float* w; uint16_t* q; int32_t* idx; uint16_t* out; float* lse;
  } sl[2];
  for (int b = 0; b < 2; ++b) {
    char* c = slots + b * hp.slot;
    sl[b].q8 = reinterpret_cast<uint8_t*>(c);
    sl[b].q_scale = reinterpret_cast<float*>(c += hp.q8);
    sl[b].w = reinterpret_cast<float*>(c += hp.q_scale);
    sl[b].q = reinterpret_cast<uint16_t*>(c += hp.w);
    sl[b].idx = reinterpret_cast<int32_t*>(c += hp.q);
    sl[b].out = reinterpret_cast<uint16_t*>(c += hp.idx);
    sl[b].lse = reinterpret_cast<float*>(c += hp.out);
  }
  cudaStream_t s_in, s_out, s = stream;
  if (!copy_streams(&s_in, &s_out)) return DSA_ERR_CUDA;
  // events: start (the workspace is free of earlier work on `stream`), keys copied, and per slot:
  // inputs copied, kernels done, outputs copied
  cudaEvent_t ev[8];
  for (int i = 0; i < 8; ++i)
    if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
      return DSA_ERR_CUDA;
    }
  cudaEvent_t start = ev[0], keys = ev[1], in_done[2] = {ev[2], ev[3]}, comp_done[2] = {ev[4], ev[5]},
              out_done[2] = {ev[6], ev[7]};
  auto H2D = cudaMemcpyHostToDevice;
  auto D2H = cudaMemcpyDeviceToHost;
  bool ok = cudaEventRecord(start, s) == cudaSuccess && cudaStreamWaitEvent(s_in, start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(s_out, start, 0) == cudaSuccess &&
            cudaMemcpyAsync(k8, a->k8, static_cast<size_t>(a->S) * 128, H2D, s_in) == cudaSuccess &&
            cudaMemcpyAsync(k_scale, a->k_scale, static_cast<size_t>(a->S) * 4, H2D, s_in) == cudaSuccess &&
            cudaMemcpyAsync(kv, a->kv, static_cast<size_t>(a->S) * 576 * 2, H2D, s_in) == cudaSuccess &&
            cudaEventRecord(keys, s_in) == cudaSuccess && cudaStreamWaitEvent(s, keys, 0) == cudaSuccess;
  const int n_chunks = (a->T + C - 1) / C;
  for (int c = 0; ok && c < n_chunks; ++c) {
    const int b = c & 1, r0 = c * C, rows = std::min(C, a->T - r0);
    const Slot& q = sl[b];
    // inputs of chunk c into slot b, once chunk c - 2's kernels are done with it
    if (c >= 2) ok = ok && cudaStreamWaitEvent(s_in, comp_done[b], 0) == cudaSuccess;
    ok = ok &&
         cudaMemcpyAsync(q.q8, a->q8 + static_cast<size_t>(r0) * H_I * 128, static_cast<size_t>(rows) * H_I * 128, H2D,
                         s_in) == cudaSuccess &&
         cudaMemcpyAsync(q.q_scale, a->q_scale + static_cast<size_t>(r0) * H_I, static_cast<size_t>(rows) * H_I * 4,
                         H2D, s_in) == cudaSuccess &&
         cudaMemcpyAsync(q.w, a->w + static_cast<size_t>(r0) * H_I, static_cast<size_t>(rows) * H_I * 4, H2D, s_in) ==
             cudaSuccess &&
         cudaMemcpyAsync(q.q, a->q + static_cast<size_t>(r0) * H * 576, static_cast<size_t>(rows) * H * 576 * 2, H2D,
                         s_in) == cudaSuccess &&
         cudaEventRecord(in_done[b], s_in) == cudaSuccess;
    if (!ok) break;
    // kernels of chunk c on the caller's stream, once its inputs landed and chunk c - 2's outputs left
    ok = cudaStreamWaitEvent(s, in_done[b], 0) == cudaSuccess &&
         (c < 2 || cudaStreamWaitEvent(s, out_done[b], 0) == cudaSuccess);
    if (!ok) break;
    const int64_t pos0 = a->q_pos0 + r0;
    st = dsa_index(q.q8, q.q_scale, q.w, k8, k_scale, rows, a->S, H_I, pos0, scores, hp.f.ld, wst, s);
    if (st == DSA_OK) st = dsa_topk(scores, hp.f.ld, rows, nullptr, a->S, pos0, K, q.idx, s);
    if (st == DSA_OK)
      st = dsa_sparse_attn(q.q, kv, a->S, nullptr, 0, 0, q.idx, rows, H, K, a->scale, q.out, q.lse, wst, s);
    if (st != DSA_OK) break;
    ok = cudaEventRecord(comp_done[b], s) == cudaSuccess;
    // outputs of chunk c back to the host
    ok = ok && cudaStreamWaitEvent(s_out, comp_done[b], 0) == cudaSuccess &&
         cudaMemcpyAsync(a->out + static_cast<size_t>(r0) * H * 512, q.out, static_cast<size_t>(rows) * H * 512 * 2,
                         D2H, s_out) == cudaSuccess &&
         (!a->lse || cudaMemcpyAsync(a->lse + static_cast<size_t>(r0) * H, q.lse, static_cast<size_t>(rows) * H * 4,
                                     D2H, s_out) == cudaSuccess) &&
         (!a->idx || cudaMemcpyAsync(a->idx + static_cast<size_t>(r0) * K, q.idx, static_cast<size_t>(rows) * K * 4,
                                     D2H, s_out) == cudaSuccess) &&
         cudaEventRecord(out_done[b], s_out) == cudaSuccess;
  }
  // the caller's stream covers the whole call: it waits for the last copies out
  if (ok) {
    for (int b = 0; b < 2 && b < n_chunks; ++b) ok = ok && cudaStreamWaitEvent(s, out_done[b], 0) == cudaSuccess;
  }
  for (int i = 0; i < 8; ++i) cudaEventDestroy(ev[i]);  // released once their work completes
  if (st != DSA_OK) return st;
  return ok ? DSA_OK : DSA_ERR_CUDA;
}

// Reads a device status word after the work already on `stream`, and clears it on the same stream
// (so that no later work of that stream can record into it between the read and the clear).
static dsa_status_t read_and_clear(int32_t* word, cudaStream_t stream) {
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSA_ERR_CUDA;
  if (v != 0 && cudaMemsetAsync(word, 0, sizeof(v), stream) != cudaSuccess) return DSA_ERR_CUDA;
  return static_cast<dsa_status_t>(v);
}

dsa_status_t dsa_status(void* status_word, dsa_stream_t stream) {
  if (!status_word || (reinterpret_cast<uintptr_t>(status_word) & 3u)) return DSA_ERR_INVALID_ARG;
  return read_and_clear(static_cast<int32_t*>(status_word), stream);
}

dsa_status_t dsa_device_status(dsa_stream_t stream) {
  int* p = status_ptr();
  if (!p) return DSA_ERR_CUDA;
  return read_and_clear(p, stream);
}

dsa_status_t dsa_selftest_wait_timeout(int timeout_us, int32_t* dev_status, dsa_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 10000000) return DSA_ERR_INVALID_ARG;
  int* p = status_target(dev_status);
  if (!p) return DSA_ERR_CUDA;
  return from_cuda(launch_wait_timeout_selftest(p, static_cast<uint64_t>(timeout_us) * 1000ull, stream));
}

}  // extern "C"
