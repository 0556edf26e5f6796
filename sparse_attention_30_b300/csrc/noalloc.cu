// dsa_decode_noalloc: the decode forward for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc themselves: a plugin inside a serving
// engine that hands out all device memory up front, or a decode loop that cannot afford
// the implicit device-wide synchronisation an allocation may cause.  For them the decode
// forward here takes its scratch (the fp32 score rows and the selected positions) from a
// fixed array in the library's own device memory instead of a caller-supplied workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds
// it until the process exits.  Host code cannot use its name as a device address; the
// address is looked up once per device with cudaGetSymbolAddress, on the first call made
// while that device is current, and that first call should therefore come before any
// stream capture.  All calls share the array and it keeps whatever the previous call left
// in it; nothing in it needs to start at zero (every score a call reads was written by the
// same call, and the selection is fully rewritten).  Calls whose work overlaps on the GPU
// (two streams, or two host threads) race on the array and must be ordered by the caller.
#include <mutex>

#include "dsa_internal.h"

namespace dsa {
namespace {

// Scratch capacity: enough for 32 sequences of 131072 tokens (or 64 of 32768) with k = 2048.
constexpr size_t kNoAllocBytes = 20ull << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_decode_noalloc_capacity(void) { return kNoAllocBytes; }

extern "C" dsa_status_t dsa_decode_noalloc(const dsa_forward_args* a, dsa_stream_t stream) {
  if (!a || a->mode != DSA_MODE_DECODE) return DSA_ERR_INVALID_ARG;
  if (a->B < 0 || a->max_seq_len < 1 || a->k < 1 || a->k > 65536) return DSA_ERR_INVALID_ARG;
  if (a->B == 0) return DSA_OK;
  // scratch needed: [B, round4(max_seq_len)] fp32 scores, then [B, k] int32 positions
  // unless the caller passed its own idx buffer
  const int64_t ld = (static_cast<int64_t>(a->max_seq_len) + 3) & ~3ll;
  const size_t score_bytes = round256(static_cast<size_t>(a->B) * ld * sizeof(float));
  const size_t idx_bytes = a->idx ? 0 : round256(static_cast<size_t>(a->B) * a->k * sizeof(int32_t));
  if (score_bytes + idx_bytes > kNoAllocBytes) return DSA_ERR_WORKSPACE;

  // Every argument of the three stages is checked before anything else, so that a rejected call
  // leaves the caller's buffers (idx included) untouched.  The checks of the scratch pointers look
  // only at null and alignment; the array is non-null and 256-byte aligned, which the stand-in
  // address below shares.
  {
    float* scores_standin = reinterpret_cast<float*>(static_cast<uintptr_t>(256));
    int32_t* idx_standin = a->idx ? a->idx : reinterpret_cast<int32_t*>(static_cast<uintptr_t>(256));
    if (!a->q || !a->kv || !a->out) return DSA_ERR_INVALID_ARG;
    dsa_status_t st = check_paged_index_args(a->q8, a->q_scale, a->w, a->k8, a->k_scale, a->n_pages, a->block_table,
                                             a->bt_stride, a->seq_lens, a->B, a->H_I, a->page_size, a->max_seq_len,
                                             scores_standin, ld);
    if (st != DSA_OK) return st;
    st = check_topk_args(scores_standin, ld, a->B, ld, 0, a->k, idx_standin, a->seq_lens);
    if (st != DSA_OK) return st;
    st = check_attn_args(a->q, a->kv, a->n_pages * a->page_size, a->block_table, a->bt_stride, a->page_size,
                         idx_standin, a->B, a->H, a->k, a->out);
    if (st != DSA_OK) return st;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    base = g_scratch_ptr[dev];
  }
  float* scores = static_cast<float*>(base);
  int32_t* idx = a->idx ? a->idx : reinterpret_cast<int32_t*>(static_cast<char*>(base) + score_bytes);

  // the kernels report into the per-device status word (dsa_device_status)
  dsa_status_t st = dsa_index_paged(a->q8, a->q_scale, a->w, a->k8, a->k_scale, a->n_pages, a->block_table,
                                    a->bt_stride, a->seq_lens, a->B, a->H_I, a->page_size, a->max_seq_len, scores,
                                    ld, nullptr, stream);
  if (st != DSA_OK) return st;
  st = dsa_topk(scores, ld, a->B, a->seq_lens, ld, 0, a->k, idx, stream);
  if (st != DSA_OK) return st;
  return dsa_sparse_attn(a->q, a->kv, a->n_pages * a->page_size, a->block_table, a->bt_stride, a->page_size, idx,
                         a->B, a->H, a->k, a->scale, a->out, a->lse, nullptr, stream);
}
