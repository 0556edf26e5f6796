/*
 * dsa.h — C ABI of libdsa.so: DeepSeek Sparse Attention (DSA) forward on one
 * NVIDIA B300 (sm_103a).
 *
 * The method (freezhihu.org/question/1978819912970555965, §2.1–§2.2):
 *   1. lightning indexer   I[t,s] = sum_j w[t,j] * ReLU(q^I[t,j] . k^I[s])   (§2.1.1 equation)
 *      over the preceding tokens s <= t, with FP8 indexer inputs (§2.1.1);
 *   2. fine-grained token selection: the k positions with the largest I[t,s] (§2.1.2);
 *   3. attention of token t over only the selected latent rows c_s (§2.1.2 output
 *      equation), in the MQA mode of MLA: each 576-dim latent row is shared by all
 *      query heads and its first 512 dims are the value (§2.2).
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller owns every
 *     buffer and the library never allocates device memory.
 *   - Tensors are dense, row-major, contiguous unless a leading dimension is given.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - FP8 tensors are e4m3 ("fn": no infinities) bytes; every FP8 scale is a positive,
 *     finite fp32 (the score uses ReLU(sq*sk*x) = sq*sk*ReLU(x), which needs sq, sk > 0).
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).  Argument
 *     errors are detected on the host and returned before anything is launched;
 *     a failed launch returns DSA_ERR_CUDA.
 *   - Device-side faults the kernels detect themselves (a wait that timed out, an index
 *     out of range) are recorded in a device status word (int32, 0 = DSA_OK; the first
 *     error recorded stays until the word is cleared):
 *       * calls that take a workspace (dsa_forward, dsa_forward_loss, dsa_prefill_host)
 *         use the word at the start of their workspace; dsa_status(ws, stream) reads and
 *         clears it.  That word must hold 0 before the workspace's first use (allocate it
 *         zeroed, or clear its first 4 bytes);
 *       * the per-stage calls take `dev_status`: a caller-owned device int32 (4-byte
 *         aligned, zeroed before first use, read and cleared by dsa_status), or NULL for a
 *         word shared by every call on the device (read and cleared by dsa_device_status).
 *     So calls that may run at the same time on different streams or host threads each
 *     report into their own word; only calls given NULL share one.
 *   - Every wait inside a kernel is bounded: after about one second it gives up, the
 *     kernel records DSA_ERR_DEVICE_TIMEOUT and returns.  The environment variable
 *     DSA_WAIT_LIMIT_MS (a positive integer, read once per process) sets another limit,
 *     for profilers that slow kernels down by orders of magnitude.
 *   - No C++ exception crosses this boundary.  The functions are thread-safe as long
 *     as calls that share output buffers are ordered by the caller.
 *   - Pointers to FP8 / bf16 row data must be 16-byte aligned (the kernels move rows
 *     with 16-byte copies and the tensor-memory accelerator).
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* identical to cudaStream_t */

/* The bound, in nanoseconds, that every wait inside the kernels is given (host-only query). */
uint64_t dsa_wait_limit_ns(void);

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,    /* a null pointer, a bad size or a misaligned pointer */
  DSA_ERR_UNSUPPORTED = 2,    /* a shape the kernels are not built for (e.g. d_I != 128) */
  DSA_ERR_WORKSPACE = 3,      /* the workspace is missing or smaller than required */
  DSA_ERR_CUDA = 4,           /* a CUDA runtime call or a kernel launch failed */
  DSA_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up on a bounded wait (see dsa_device_status) */
  DSA_ERR_DEVICE_RANGE = 6    /* a kernel met an index or page number out of range and skipped it */
} dsa_status_t;

/* Human-readable name of a status code (static storage; never NULL). */
const char* dsa_status_string(dsa_status_t status);

/* Library ABI version: (major << 16) | minor. */
int dsa_version(void);

/*
 * dsa_index — lightning-indexer scores for a block of prefill query rows
 * (freezhihu.org/question/1978819912970555965 §2.1.1, indexer equation).
 *
 * Row t (0 <= t < T) is the query at absolute position q_pos0 + t; keys are the
 * positions 0 .. S-1.  For every s <= min(q_pos0 + t, S - 1) it writes
 *     scores[t * ld + s] = k_scale[s] * sum_j (w[t,j] * q_scale[t,j]) * ReLU(q8[t,j,:] . k8[s,:])
 * with the FP8 products accumulated in fp32 on the tensor cores and the head sum in fp32.
 * Entries with s > q_pos0 + t are not written.
 *
 *   q8       [T, H_I, 128]  e4m3, 16-byte aligned
 *   q_scale  [T, H_I]       fp32 per (token, head) dequantisation scale
 *   w        [T, H_I]       fp32 head weights w^I
 *   k8       [S, 128]       e4m3, 16-byte aligned
 *   k_scale  [S]            fp32 per-key scale
 *   scores   [T, ld]        fp32 output, ld >= min(S, q_pos0 + T), ld % 4 == 0, 16-byte aligned
 *   dev_status  device status word (see the conventions above), or NULL
 *   H_I must be a power of two in [4, 128] (other powers of two up to 128 return
 *   DSA_ERR_UNSUPPORTED, anything else DSA_ERR_INVALID_ARG); T, S >= 1 (T = 0 is a no-op);
 *   q_pos0 >= 0.
 */
dsa_status_t dsa_index(const uint8_t* q8, const float* q_scale, const float* w,
                       const uint8_t* k8, const float* k_scale,
                       int T, int S, int H_I, int64_t q_pos0,
                       float* scores, int64_t ld, int32_t* dev_status, dsa_stream_t stream);

/*
 * dsa_index_paged — indexer scores of one new query token per sequence against a
 * paged FP8 key cache (decode).  Sequence b holds seq_lens[b] tokens, the new one
 * included (it sits at position seq_lens[b] - 1 and scores itself too).  Logical
 * position p of sequence b lives in page block_table[b * bt_stride + p / page_size],
 * slot p % page_size.  Writes scores[b * ld + p] for 0 <= p < seq_lens[b].
 *
 *   q8 [B, H_I, 128], q_scale [B, H_I], w [B, H_I]   as in dsa_index, one token per sequence
 *   k8_cache      [n_pages, page_size, 128] e4m3, 16-byte aligned
 *   k_scale_cache [n_pages, page_size]      fp32
 *   block_table   [B, bt_stride] int32 page numbers (entries past a sequence's last page are not read)
 *   seq_lens      [B] int32, each in [1, max_seq_len]
 *   scores        [B, ld] fp32, ld >= max_seq_len, ld % 4 == 0
 *   page_size must divide 128 and be a multiple of 8; n_pages bounds the page numbers
 *   (an out-of-range page number is skipped and reported as DSA_ERR_DEVICE_RANGE).
 *   H_I must be 32, 64 or 128 (other head counts return DSA_ERR_UNSUPPORTED).
 *   dev_status    device status word, or NULL
 */
dsa_status_t dsa_index_paged(const uint8_t* q8, const float* q_scale, const float* w,
                             const uint8_t* k8_cache, const float* k_scale_cache, int64_t n_pages,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* seq_lens, int B, int H_I, int page_size, int max_seq_len,
                             float* scores, int64_t ld, int32_t* dev_status, dsa_stream_t stream);

/*
 * dsa_topk — fine-grained token selection
 * (freezhihu.org/question/1978819912970555965 §2.1.2; k = 2048 in §2.3.2).
 *
 * For each row t it selects the min(k, n_t) positions with the largest scores among
 * scores[t * ld + 0 .. n_t - 1], where n_t = row_lens[t] if row_lens is not NULL,
 * else min(n_cols, q_pos0 + t + 1) (the causal prefix of a prefill row).
 * idx[t * k + i] receives the selected positions in slots 0 .. min(k, n_t) - 1 (in no
 * particular order) and -1 in the remaining slots.  Equal scores at the boundary are
 * broken arbitrarily; selection compares fp32 scores exactly (order-preserving integer
 * keys), so NaN scores are not supported.
 *
 *   scores [T, ld] fp32 (16-byte aligned, ld % 4 == 0), idx [T, k] int32,
 *   row_lens [T] int32 or NULL, 1 <= k <= 65536, every n_t <= ld.
 */
dsa_status_t dsa_topk(const float* scores, int64_t ld, int T, const int32_t* row_lens,
                      int64_t n_cols, int64_t q_pos0, int k, int32_t* idx, dsa_stream_t stream);

/*
 * dsa_sparse_attn — MQA-mode MLA attention over the selected latent rows
 * (freezhihu.org/question/1978819912970555965 §2.1.2 output equation, §2.2).
 *
 * For every row t and head h:
 *     o[t,h,:] = sum_{s in S_t} softmax_s(scale * q[t,h,:] . c_s) * c_s[0:512]
 * where S_t = { idx[t*k + i] : idx[t*k + i] >= 0 } (valid slots must come first) and
 * c_s is latent row s: kv[s * 576 ...] if block_table is NULL, else slot s % page_size
 * of page block_table[t * bt_stride + s / page_size] in kv viewed as
 * [n_pages, page_size, 576].  QK^T and PV run on the tensor cores with bf16 inputs
 * and fp32 accumulation; the softmax is in fp32.  A row with no valid slot yields
 * zeros and lse = -inf.
 *
 *   q   [T, H, 576] bf16, 16-byte aligned, 1 <= H <= 128
 *   kv  [n_kv_rows, 576] bf16 (n_kv_rows = n_pages * page_size when paged), 16-byte aligned
 *   block_table [T, bt_stride] int32 (bt_stride >= 1) or NULL; page_size >= 1 when paged
 *   idx [T, k] int32 (positions; an index >= n_kv_rows, a position whose page index is
 *       >= bt_stride, or a page number out of range is treated as an empty slot and
 *       reported as DSA_ERR_DEVICE_RANGE)
 *   out [T, H, 512] bf16, 16-byte aligned
 *   lse [T, H] fp32 natural-log sum-exp of the scaled logits, or NULL
 *   dev_status  device status word, or NULL
 */
dsa_status_t dsa_sparse_attn(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows,
                             const int32_t* block_table, int64_t bt_stride, int page_size,
                             const int32_t* idx, int T, int H, int k, float scale,
                             uint16_t* out, float* lse, int32_t* dev_status, dsa_stream_t stream);

/*
 * dsa_sparse_attn_split — dsa_sparse_attn with the rows' selected keys spread over partial
 * attentions that a second kernel merges exactly (log-sum-exp weights).  Same inputs, outputs and
 * rules as dsa_sparse_attn; this is how the decode forward fills the GPU when it has few sequences.
 *   n_split in [1, 8]: each row's slots in n_split equal shares; `ws` holds
 *       dsa_sparse_attn_split_workspace_size(T, H, n_split) bytes (n_split = 1: dsa_sparse_attn,
 *       no workspace).
 *   n_split = 0: balanced over every SM pair of the GPU: the rows' ceil(k / 64) tiles of 64 slots,
 *       end to end, are cut into equal contiguous ranges, one per pair (74 on a B300), so every pair
 *       gets the same number of tiles whatever T is; `ws` holds
 *       dsa_sparse_attn_balanced_workspace_size(T, H, k) bytes (0 when no row is split).  This is
 *       the decode forward's partition.
 * `ws` is a caller-owned device buffer, 256-byte aligned, holding the partial outputs.
 */
size_t dsa_sparse_attn_split_workspace_size(int T, int H, int n_split);
size_t dsa_sparse_attn_balanced_workspace_size(int T, int H, int k);
dsa_status_t dsa_sparse_attn_split(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows,
                                   const int32_t* block_table, int64_t bt_stride, int page_size,
                                   const int32_t* idx, int T, int H, int k, float scale,
                                   uint16_t* out, float* lse, int n_split, void* ws, size_t ws_bytes,
                                   int32_t* dev_status, dsa_stream_t stream);

/*
 * dsa_dense_causal_attn — dense causal attention in the same MQA mode of MLA: every row attends
 * to every latent row at or before its own position.  This is the computation DSA replaces
 * (vpshk.cn/20260227158.html: the dense V3.1 model's cost climbs with the text length while
 * V3.2's stays nearly flat; 10100.com/article/43188788 §1: about half the long-context cost),
 * provided as the baseline DSA is measured against.  It equals dsa_sparse_attn with the
 * selection {0, ..., q_pos0 + t} for row t.
 *
 * For every row t (absolute position q_pos0 + t) and head h:
 *     o[t,h,:] = sum_{s = 0 .. q_pos0 + t} softmax_s(scale * q[t,h,:] . c_s) * c_s[0:512]
 *
 *   q   [T, H, 576] bf16, 16-byte aligned, 1 <= H <= 128
 *   kv  [n_kv_rows, 576] bf16 latent rows of positions 0 .. n_kv_rows - 1, 16-byte aligned;
 *       q_pos0 >= 0, q_pos0 + T <= n_kv_rows < 2^31
 *   out [T, H, 512] bf16, 16-byte aligned
 *   lse [T, H] fp32 natural-log sum-exp of the scaled logits, or NULL
 * Same arithmetic as dsa_sparse_attn (bf16 tensor-core products, fp32 accumulation and softmax);
 * the latent rows are read as contiguous 64-row tiles.  Errors: DSA_ERR_INVALID_ARG /
 * DSA_ERR_UNSUPPORTED before any launch; DSA_ERR_CUDA if the launch fails; device timeouts in
 * `dev_status` (or, when it is NULL, the shared word read by dsa_device_status).
 */
dsa_status_t dsa_dense_causal_attn(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows, int T, int H,
                                   int64_t q_pos0, float scale, uint16_t* out, float* lse,
                                   int32_t* dev_status, dsa_stream_t stream);

/*
 * dsa_indexer_loss — the lightning indexer's training objective
 * (freezhihu.org/question/1978819912970555965 §2.3.1 dense warm-up, §2.3.2 sparse training):
 *     L^I = sum_t KL(p_t || Softmax(I[t, S_t]))
 * where the target p_t is the main attention of all heads summed and L1-normalised over the
 * keys of S_t (read here as the per-head softmax probabilities, so p_t is their head average).
 *
 *   idx non-NULL: sparse stage, S_t = the valid slots of idx [T, k] (as in dsa_sparse_attn).
 *   idx NULL:     dense warm-up, S_t = every position 0 .. q_pos0 + t (q_pos0 >= 0,
 *                 q_pos0 + T <= n_kv_rows and <= ld; p must be NULL; k and the slot layout unused).
 *
 *   q, kv, T, H, scale: as in dsa_sparse_attn (contiguous kv [n_kv_rows, 576], n_kv_rows < 2^31)
 *   lse    [T, H] fp32: the natural-log softmax normalisers of the forward over the same sets
 *          (the lse output of dsa_sparse_attn / dsa_dense_causal_attn); the head probabilities
 *          are recomputed from q and kv as exp(scale * q . c_s - lse)
 *   scores [T, ld] fp32 indexer scores I[t, s] at column s (dsa_index output); every position in
 *          a set must be < ld (a larger one is skipped and reported as DSA_ERR_DEVICE_RANGE)
 *   p      [T, k] fp32 target per slot (0 for empty slots), or NULL
 *   kl     [T] fp32 KL term per row (0 for a row with an empty set), or NULL
 *   loss_acc  one double: sum_t KL_t is ADDED to it (the caller zeroes it), or NULL
 * The scores QK^T are recomputed on the tensor cores (bf16 inputs, fp32 accumulation); the
 * head sums in fp32; the per-row sums in fp64.  Errors as in dsa_sparse_attn.
 */
dsa_status_t dsa_indexer_loss(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows, const int32_t* idx,
                              int T, int H, int k, int64_t q_pos0, float scale, const float* lse,
                              const float* scores, int64_t ld, float* p, float* kl, double* loss_acc,
                              int32_t* dev_status, dsa_stream_t stream);

/*
 * dsa_sparse_attn_backward — gradients of dsa_sparse_attn over a fixed selection
 * (freezhihu.org/question/1978819912970555965 §2.3.2: the sparse training stage optimises the
 * main model through the attention over the selected rows S_t).
 *
 * With z[h,s] = scale * q[t,h,:] . c_s, p = softmax_s(z) over S_t and o = sum_s p c_s[0:512] (the
 * forward), and do = dL/do:
 *     ds[h,s] = p[h,s] * (do[t,h,:] . c_s[0:512] - do[t,h,:] . o[t,h,:])
 *     dq[t,h,:]  = scale * sum_{s in S_t} ds[h,s] c_s
 *     dkv[s,:]  += scale * sum_h ds[h,s] q[t,h,:]  +  [sum_h p[h,s] do[t,h,:], 0]   for every t with s in S_t
 * p is recomputed from q, kv and the forward's lse; products on the tensor cores with bf16 inputs
 * (p and ds are rounded to bf16 before their products) and fp32 accumulation.
 *
 *   q, kv, n_kv_rows, idx, T, H, k, scale: as in dsa_sparse_attn (contiguous kv only)
 *   out   [T, H, 512] bf16: the forward's output (for do . o), 16-byte aligned
 *   dout  [T, H, 512] bf16: gradient of the output, 16-byte aligned
 *   lse   [T, H] fp32: the forward's lse output
 *   dq    [T, H, 576] bf16 output, 16-byte aligned (rows of a token with no valid slot are zero)
 *   dkv   [n_kv_rows, 576] fp32, 16-byte aligned: the latent-row gradients are ADDED to it (the
 *         caller zeroes it), with atomic adds, so the summation order over tokens is not fixed
 *   dev_status  device status word, or NULL
 * Errors as dsa_sparse_attn (an out-of-range position is skipped and reported as
 * DSA_ERR_DEVICE_RANGE).
 */
dsa_status_t dsa_sparse_attn_backward(const uint16_t* q, const uint16_t* kv, int64_t n_kv_rows,
                                      const int32_t* idx, int T, int H, int k, float scale,
                                      const uint16_t* out, const uint16_t* dout, const float* lse,
                                      uint16_t* dq, float* dkv, int32_t* dev_status, dsa_stream_t stream);

/* Forward modes. */
enum { DSA_MODE_PREFILL = 0, DSA_MODE_DECODE = 1 };

/*
 * Arguments of the fused forward (indexer -> top-k -> sparse attention).
 *
 * PREFILL: one sequence with S keys (positions 0 .. S-1) and T query rows at positions
 *   q_pos0 .. q_pos0 + T - 1 (q_pos0 + T <= S).  q8/q_scale/w/q hold the T query rows,
 *   k8 [S,128] / k_scale [S] / kv [S,576] the keys.  The library scores the rows in
 *   chunks of chunk_rows (0 = library choice) so the fp32 score block stays bounded.
 * DECODE: B sequences, one new token each, with paged caches k8 [n_pages,page,128],
 *   k_scale [n_pages,page], kv [n_pages,page,576], block_table [B, bt_stride], seq_lens [B]
 *   (each in [1, max_seq_len]); q8/q_scale/w/q hold the B query tokens.
 *
 * Outputs: out [rows, H, 512] bf16; lse [rows, H] fp32 or NULL; idx [rows, k] int32 or
 * NULL (when NULL the selection lives in the workspace only).
 */
typedef struct {
  int mode;           /* DSA_MODE_PREFILL or DSA_MODE_DECODE */
  int H_I;            /* indexer heads: prefill 4..128 (powers of two), decode 32, 64 or 128 */
  int H;              /* attention heads (1..128) */
  int k;              /* tokens selected per query (1..65536) */
  float scale;        /* softmax scale */
  /* prefill */
  int T;
  int S;
  int64_t q_pos0;
  int chunk_rows;
  /* decode */
  int B;
  int page_size;
  int64_t n_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* seq_lens;
  int max_seq_len;
  /* inputs */
  const uint8_t* q8;
  const float* q_scale;
  const float* w;
  const uint8_t* k8;
  const float* k_scale;
  const uint16_t* q;
  const uint16_t* kv;
  /* outputs */
  uint16_t* out;
  float* lse;
  int32_t* idx;
} dsa_forward_args;

/* Bytes of device workspace dsa_forward needs for these arguments (0 on invalid args): a 256-byte
 * head whose first word is the call's status word, then the fp32 score block, the selection (when
 * args->idx is NULL) and, for decode with fewer than 74 sequences, the key-split partial results. */
size_t dsa_forward_workspace_size(const dsa_forward_args* args);

/*
 * dsa_forward — the whole hot path: scores (dsa_index / dsa_index_paged), selection
 * (dsa_topk) and attention (dsa_sparse_attn), asynchronously on `stream`.
 * `ws` is a caller-owned device buffer of at least dsa_forward_workspace_size(args)
 * bytes, 256-byte aligned; its first word is the status word the kernels of this call report
 * into (zero before the first use; dsa_status(ws, stream) reads and clears it), the rest holds
 * the fp32 score block and the selection.
 */
dsa_status_t dsa_forward(const dsa_forward_args* args, void* ws, size_t ws_bytes,
                         dsa_stream_t stream);

/* Stages of the indexer's training loss (freezhihu.org/question/1978819912970555965 §2.3). */
enum { DSA_LOSS_SPARSE = 0, DSA_LOSS_DENSE_WARMUP = 1 };

/* Bytes of device workspace dsa_forward_loss needs (0 on invalid args). */
size_t dsa_forward_loss_workspace_size(const dsa_forward_args* args, int stage);

/*
 * dsa_forward_loss — the training-side prefill forward with the indexer's loss
 * (§2.3.2 sparse stage, §2.3.1 dense warm-up).  args as for dsa_forward with
 * mode = DSA_MODE_PREFILL; args->lse is required (it feeds the loss).  For each chunk of
 * chunk_rows query rows (0 = library choice):
 *   DSA_LOSS_SPARSE:       dsa_index, dsa_topk, dsa_sparse_attn over the chunk's selection,
 *                          then dsa_indexer_loss over the same selection;
 *   DSA_LOSS_DENSE_WARMUP: dsa_index, dsa_dense_causal_attn (every preceding key), then
 *                          dsa_indexer_loss over every preceding key (args->idx and k unused
 *                          beyond validation).
 * Outputs: out, lse, idx (sparse stage, when non-NULL) as for dsa_forward; kl [T] per-row KL
 * terms (device, or NULL); *loss_acc (one device double, or NULL) has sum_t KL_t ADDED to it.
 * `ws`: dsa_forward_loss_workspace_size(args, stage) bytes, 256-byte aligned (the status word
 * head as in dsa_forward, the fp32 score block of one chunk, and the selection when args->idx is
 * NULL).  Errors as dsa_forward.
 */
dsa_status_t dsa_forward_loss(const dsa_forward_args* args, int stage, float* kl, double* loss_acc, void* ws,
                              size_t ws_bytes, dsa_stream_t stream);

/*
 * dsa_prefill_host — the prefill forward (mode DSA_MODE_PREFILL of dsa_forward) with every
 * tensor in HOST memory: args->q8, q_scale, w, k8, k_scale, q, kv and the outputs out, lse
 * (or NULL) and idx (or NULL) are host pointers, laid out as for dsa_forward.  The keys are
 * copied to the device once; then the query rows move in chunks of chunk_rows (0 = library
 * choice) through two device slots, so that one chunk's copies in and out run while the other
 * chunk's kernels run (the same kernels as dsa_forward, the same results).  Copies are
 * asynchronous only from page-locked (pinned) host memory; pageable memory works but
 * serialises them.
 * `ws` is a caller-owned device buffer of at least dsa_prefill_host_workspace_size(args) bytes,
 * 256-byte aligned, starting with the status word head of dsa_forward.  The call only enqueues work: the kernels run on `stream` and the copies on
 * two streams the library keeps per device, ordered after the work already on `stream`; the
 * outputs are in host memory once `stream` reaches the point after this call (synchronise it
 * before reading them, and do not touch the host buffers before then).  Errors as dsa_forward;
 * a failed copy or event returns DSA_ERR_CUDA.
 */
size_t dsa_prefill_host_workspace_size(const dsa_forward_args* args);
dsa_status_t dsa_prefill_host(const dsa_forward_args* args, void* ws, size_t ws_bytes,
                              dsa_stream_t stream);

/*
 * dsa_status — the device-side status of the calls that reported into `status_word`: a
 * workspace of dsa_forward / dsa_forward_loss / dsa_prefill_host (its first word), or a
 * caller-owned int32 passed as `dev_status` to the per-stage calls.  Reads the word after the
 * work already enqueued on `stream` (the host waits for that work), returns it (DSA_OK if
 * nothing was recorded) and clears it on the same stream, so that later work on `stream`
 * records into a clean word.  DSA_ERR_INVALID_ARG for a NULL or misaligned pointer,
 * DSA_ERR_CUDA if the copy or the synchronisation fails.  Calls on other streams that report
 * into the same word must be ordered by the caller.
 */
dsa_status_t dsa_status(void* status_word, dsa_stream_t stream);

/*
 * dsa_device_status — dsa_status for the word shared by every call on the current device that
 * was given no status word of its own (dev_status NULL, and dsa_decode_noalloc).  Every stream
 * records into this one word, so with concurrent streams an error may be read by the wrong
 * caller: give such calls their own words.
 */
dsa_status_t dsa_device_status(dsa_stream_t stream);

/*
 * dsa_selftest_wait_timeout — launches one block that waits on a barrier nobody
 * arrives at, with a limit of timeout_us microseconds; the kernel then records
 * DSA_ERR_DEVICE_TIMEOUT into dev_status (or the shared word when NULL) and returns.
 * Used to test the bounded-wait path without a hang.  Follow with dsa_status() /
 * dsa_device_status().
 */
dsa_status_t dsa_selftest_wait_timeout(int timeout_us, int32_t* dev_status, dsa_stream_t stream);

/*
 * dsa_decode_noalloc — the decode forward (mode DSA_MODE_DECODE of dsa_forward) for callers
 * that cannot allocate device memory.  The paper has no counterpart: this is a deployment
 * convenience.  Some callers may not call cudaMalloc themselves (a plugin inside a serving
 * engine that owns all device memory, a decode loop that cannot afford an allocation's
 * implicit synchronisation); instead of a caller-supplied workspace this call takes its
 * scratch (fp32 scores and, if args->idx is NULL, the selection) from a fixed array of
 * dsa_decode_noalloc_capacity() bytes (20 MiB) that the library keeps in the device memory
 * of every GPU that loads it, until the process exits.
 *   - Needs B * round4(max_seq_len) * 4 + B * k * 4 bytes (each rounded up to 256); a
 *     larger request returns DSA_ERR_WORKSPACE without launching anything.
 *   - The first call on a device (with that device current) looks up the array's address;
 *     make that first call before any stream capture.
 *   - Every call shares the array: calls whose work overlaps on the GPU race on it and
 *     must be ordered by the caller.  Nothing in it needs clearing between calls.
 *   - Every argument is checked before the first launch.  Device-side errors go to the
 *     shared word of dsa_device_status (there is no workspace to hold a word of its own).
 *   - Runs the same indexer, top-k and attention kernels as dsa_forward in decode mode, but
 *     without the key split dsa_forward uses for fewer than 74 sequences (the split's partial
 *     results would need more scratch): with few sequences it occupies fewer SMs and is slower,
 *     and its outputs agree with dsa_forward's to rounding rather than bit for bit.  It
 *     allocates nothing and calls no allocating routine.
 */
dsa_status_t dsa_decode_noalloc(const dsa_forward_args* args, dsa_stream_t stream);

/* Size in bytes of the fixed scratch array dsa_decode_noalloc uses. */
size_t dsa_decode_noalloc_capacity(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
