"""Plain float64 CPU oracle for DeepSeek Sparse Attention (DSA).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
CPU-baseline / reference arm may import this package.  The CUDA library never
imports, links or calls it, and it shares no code with the CUDA path.

What it computes, and the passage each step follows (pages are named by
address; sections are the pages' own numbering):

  * indexer score  I[t,s] = sum_j w[t,j] * ReLU(q^I[t,j] . k^I[s])
      freezhihu.org/question/1978819912970555965, §2.1.1 (lightning indexer
      equation); the scores of FP8 inputs are taken on the decoded values,
      times the per-token scales (§2.1.1: "can be implemented in FP8").
  * causal candidate set: query t scores the preceding tokens s <= t
      (same page, §2.1.1, "preceding tokens"; reading: t sees itself).
  * fine-grained top-k: the k positions with the largest I[t,s]
      (same page, §2.1.2); k = 2048 (same page, §2.3.2).
  * sparse attention u_t = Attn(h_t, {c_s : s in Top-k(I[t,:])})
      (same page, §2.1.2 output equation), MQA mode of MLA: one latent row
      c_s per token shared by every query head (same page, §2.2).  The value
      is the first 512 dims of the 576-dim latent, softmax scale 1/sqrt(192).
  * indexer training loss: target p = head-summed attention probabilities over
      the set, L1-normalised, and KL(p || Softmax(I)) (same page, §2.3.1 over all
      s <= t in the dense warm-up, §2.3.2 over the selected set S_t).
  * backward of the sparse attention over a fixed selection (dq, and the latent-row
      gradient summed over every token that selected the row): the sparse training
      stage optimises the main model through DSA (same page, §2.3.2).
  * dense causal attention over every row s <= t: the computation DSA replaces,
      which vpshk.cn/20260227158.html and 10100.com/article/43188788 §1 compare
      DSA's cost against.

Every step is the plain definition: exact decode of the FP8 / bf16 inputs to
float64, dot products in float64 (exact for FP8 inputs), a stable full sort for
top-k (ties go to the lower position), and a max-subtracted softmax.

Parity status: every function here is pinned by tests/test_oracle.py against
library routines (torch's float8 / bf16 casts, torch SDPA, matmul identities),
brute-force enumeration and closed forms.
"""
from .dsa import (  # noqa: F401
    e4m3_to_f64, bf16_bits_to_f64, indexer_row, indexer_scores, topk_row, topk_rows,
    attention_row, dense_causal_row, indexer_kl_row, indexer_loss_prefill_row, prefill_row, prefill_rows, decode_row, decode_gather,
    selected_pairs, causal_pairs, index_sets_match, attention_error, attention_row_backward,
    sparse_attention_backward,
)
