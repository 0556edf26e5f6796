// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsa.h"

namespace dsa {

// Bounded waits give up after this long (about one second).
constexpr uint64_t kWaitLimitNs = 1ull << 30;
// The limit the kernels are given: kWaitLimitNs, or DSA_WAIT_LIMIT_MS milliseconds when that
// environment variable holds a positive integer (read once; for tools that slow kernels down).
uint64_t wait_limit_ns();

// 2-D tensor map over a row-major matrix [rows, inner] with the given row pitch, 128-byte swizzle,
// box [box_inner, box_rows]; false if the driver rejects it.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows);

// ---------------------------------------------------------------- indexer

struct IndexerArgs {
  const float* q_scale;       // [rows, H_I]
  const float* w;             // [rows, H_I]
  const float* k_scale;       // prefill [S]; paged [n_pages * page_size]
  const int32_t* block_table; // paged only
  int64_t bt_stride;
  const int32_t* seq_lens;    // paged only
  int64_t n_pages;
  float* scores;
  int64_t ld;
  int rows;                   // prefill: T query rows; paged: B sequences
  int S;                      // prefill: number of keys; paged: max_seq_len
  int64_t q_pos0;
  int page_size;
  int tiles_per_cta;          // 128-key tiles handled by one CTA
  int* status;
  uint64_t limit_ns;
};

// q8 viewed as [rows * H_I, 128] bytes, k8 as [n_keys, 128] bytes (paged: n_pages * page_size).
cudaError_t launch_indexer(const uint8_t* q8, const uint8_t* k8, int64_t n_key_rows, int H_I, bool paged,
                           int max_keys, const IndexerArgs& a, cudaStream_t stream);
int indexer_supported_heads(int H_I, bool paged);
// The decode (paged) kernel: q8 as [rows * H_I, 128] (box H_I rows), the key cache as
// [n_pages * page_size, 128] (box page_size rows).
cudaError_t launch_indexer_paged(const CUtensorMap& qm, const CUtensorMap& km, int H_I, int max_keys,
                                 const IndexerArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- top-k

struct TopkArgs {
  const float* scores;
  int64_t ld;
  int T;
  const int32_t* row_lens;
  int64_t n_cols;
  int64_t q_pos0;
  int k;
  int32_t* idx;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- sparse attention

struct AttnArgs {
  const uint16_t* q;          // [T, H, 576] bf16
  const uint16_t* kv;         // [n_kv_rows, 576] bf16
  int64_t n_kv_rows;
  const int32_t* block_table; // NULL: contiguous
  int64_t bt_stride;
  int page_size;
  const int32_t* idx;         // [T, k]; NULL selects the dense causal mode
  int T, H, k;
  int64_t q_pos0;             // dense causal mode (idx NULL): row t attends latent rows 0 .. q_pos0 + t
  float scale_log2;           // softmax scale * log2(e)
  uint16_t* out;              // [T, H, 512] bf16
  float* lse;                 // [T, H] or NULL
  int* status;
  uint64_t limit_ns;
  // key split (decode with few sequences): n_split > 1 gives each token n_split clusters, each
  // over a contiguous share of its selected tiles, writing partial results that
  // launch_attn_combine merges into out / lse
  int n_split;
  float* part_o;              // [T, n_split, H, 512] fp32, each normalised by its own sum
  float* part_ml;             // [T, n_split, H, 2] fp32: running max (log2 domain) and sum
  // balanced partition (bal_tiles > 0): the T rows' bal_tiles virtual 64-key tiles each, end to end,
  // cut into n_clusters equal contiguous ranges (one per cluster); a row spread over several
  // clusters leaves one partial result per cluster, at part index (cluster - the row's first
  // cluster) < n_split, and launch_attn_combine merges them
  int bal_tiles;
  int n_clusters;
  // indexer-loss mode (lse_in non-NULL): no attention output; the head-summed attention target
  // over each row's set and its KL divergence from the softmax of the indexer scores
  const float* lse_in;        // [T, H] natural-log normalisers of the forward over the same sets
  const float* scores;        // [T, ld] indexer scores, column = key position
  int64_t ld;
  float* p_out;               // [T, k] L1-normalised target per slot (0 for empty slots), or NULL
  float* kl_out;              // [T] KL(p || softmax(I)) per row, or NULL
  double* loss_acc;           // sum over rows added here, or NULL
};
cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream);

// Balanced partition of G = rows x tiles-per-row virtual tiles over n_cl clusters: cluster c covers
// [bal_bound(c), bal_bound(c + 1)); bal_cluster(g) is the cluster whose range holds tile g (n_cl <= G).
__host__ __device__ inline int64_t bal_bound(int64_t c, int64_t G, int n_cl) { return c * G / n_cl; }
__host__ __device__ inline int bal_cluster(int64_t g, int64_t G, int n_cl) {
  return static_cast<int>(((g + 1) * n_cl - 1) / G);
}
// Number of clusters (partial results) row t is spread over.
__host__ __device__ inline int bal_parts(int t, int tpr, int64_t G, int n_cl) {
  const int64_t g0 = static_cast<int64_t>(t) * tpr;
  return bal_cluster(g0 + tpr - 1, G, n_cl) - bal_cluster(g0, G, n_cl) + 1;
}
cudaError_t launch_attn_combine(const AttnArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- sparse attention backward

struct BwdArgs {
  const uint16_t* q;          // [T, H, 576] bf16
  const uint16_t* kv;         // [n_kv_rows, 576] bf16
  int64_t n_kv_rows;
  const int32_t* idx;         // [T, k]
  int T, H, k;
  float scale;                // softmax scale
  const uint16_t* out;        // [T, H, 512] bf16: the forward's output
  const uint16_t* dout;       // [T, H, 512] bf16: gradient of the output
  const float* lse;           // [T, H] natural-log normalisers of the forward
  uint16_t* dq;               // [T, H, 576] bf16
  float* dkv;                 // [n_kv_rows, 576] fp32, added to
  int* status;
  uint64_t limit_ns;
};
cudaError_t launch_sparse_attn_bwd(const BwdArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- host-side argument checks (api.cu)

// Each returns DSA_OK, or the status the public call returns before launching anything.
dsa_status_t check_index_args(const uint8_t* q8, const float* q_scale, const float* w, const uint8_t* k8,
                              const float* k_scale, int T, int S, int H_I, int64_t q_pos0, const float* scores,
                              int64_t ld);
dsa_status_t check_paged_index_args(const uint8_t* q8, const float* q_scale, const float* w, const uint8_t* k8c,
                                    const float* ksc, int64_t n_pages, const int32_t* bt, int64_t bt_stride,
                                    const int32_t* lens, int B, int H_I, int page, int max_len, const float* scores,
                                    int64_t ld);
dsa_status_t check_topk_args(const float* scores, int64_t ld, int T, int64_t n_cols, int64_t q_pos0, int k,
                             const int32_t* idx, const int32_t* row_lens);
dsa_status_t check_attn_args(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows, const int32_t* bt,
                             int64_t bt_stride, int page, const int32_t* idx, int T, int H, int k,
                             const uint16_t* out);
// The device word a call reports into: the caller's (non-NULL) or this device's shared word.
int* status_target(int32_t* dev_status);

// ---------------------------------------------------------------- self test

cudaError_t launch_wait_timeout_selftest(int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace dsa
