"""Python binding of libdsa.so: DeepSeek Sparse Attention forward on one B300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA kernels of
libdsa.so (see include/dsa.h for the exact contract of each call).  PyTorch supplies
device memory and the current stream.  Importing this module (re)builds libdsa.so if a
source is newer than it, loads it, and raises if either step fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libdsa.so")

DSA_OK = 0
STATUS_NAMES = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_WORKSPACE",
                4: "DSA_ERR_CUDA", 5: "DSA_ERR_DEVICE_TIMEOUT", 6: "DSA_ERR_DEVICE_RANGE"}
MODE_PREFILL, MODE_DECODE = 0, 1

# Names of every function include/dsa.h declares.
EXPORTS = ("dsa_status_string", "dsa_version", "dsa_index", "dsa_index_paged", "dsa_topk", "dsa_sparse_attn",
           "dsa_forward_workspace_size", "dsa_forward", "dsa_device_status", "dsa_selftest_wait_timeout",
           "dsa_decode_noalloc", "dsa_decode_noalloc_capacity", "dsa_sparse_attn_split_workspace_size",
           "dsa_sparse_attn_split", "dsa_prefill_host_workspace_size", "dsa_prefill_host",
           "dsa_dense_causal_attn", "dsa_indexer_loss", "dsa_wait_limit_ns", "dsa_forward_loss_workspace_size",
           "dsa_forward_loss", "dsa_status", "dsa_sparse_attn_backward", "dsa_sparse_attn_balanced_workspace_size")


class DSAError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")
        self.code = code


class ForwardArgs(ctypes.Structure):
    """Mirror of dsa_forward_args in include/dsa.h (same field order and types)."""
    _fields_ = [
        ("mode", ctypes.c_int), ("H_I", ctypes.c_int), ("H", ctypes.c_int), ("k", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("T", ctypes.c_int), ("S", ctypes.c_int), ("q_pos0", ctypes.c_int64), ("chunk_rows", ctypes.c_int),
        ("B", ctypes.c_int), ("page_size", ctypes.c_int), ("n_pages", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int64), ("seq_lens", ctypes.c_void_p),
        ("max_seq_len", ctypes.c_int),
        ("q8", ctypes.c_void_p), ("q_scale", ctypes.c_void_p), ("w", ctypes.c_void_p),
        ("k8", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("q", ctypes.c_void_p), ("kv", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("idx", ctypes.c_void_p),
    ]


def _load():
    from . import build as _build
    try:
        _build.build()  # compiles only when a source is newer than the library
    except Exception as e:  # no silent fallback: the package is unusable without its kernels
        raise ImportError(f"libdsa.so could not be built: {e}") from e
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libdsa.so is missing ({LIB_PATH})")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    sig = {
        "dsa_status_string": ([I], ctypes.c_char_p),
        "dsa_version": ([], I),
        "dsa_index": ([P, P, P, P, P, I, I, I, I64, P, I64, P, P], I),
        "dsa_index_paged": ([P, P, P, P, P, I64, P, I64, P, I, I, I, I, P, I64, P, P], I),
        "dsa_topk": ([P, I64, I, P, I64, I64, I, P, P], I),
        "dsa_sparse_attn": ([P, P, I64, P, I64, I, P, I, I, I, F, P, P, P, P], I),
        "dsa_forward_workspace_size": ([ctypes.POINTER(ForwardArgs)], ctypes.c_size_t),
        "dsa_forward": ([ctypes.POINTER(ForwardArgs), P, ctypes.c_size_t, P], I),
        "dsa_device_status": ([P], I),
        "dsa_status": ([P, P], I),
        "dsa_selftest_wait_timeout": ([I, P, P], I),
        "dsa_decode_noalloc": ([ctypes.POINTER(ForwardArgs), P], I),
        "dsa_decode_noalloc_capacity": ([], ctypes.c_size_t),
        "dsa_sparse_attn_split_workspace_size": ([I, I, I], ctypes.c_size_t),
        "dsa_sparse_attn_balanced_workspace_size": ([I, I, I], ctypes.c_size_t),
        "dsa_dense_causal_attn": ([P, P, I64, I, I, I64, F, P, P, P, P], I),
        "dsa_wait_limit_ns": ([], ctypes.c_uint64),
        "dsa_indexer_loss": ([P, P, I64, P, I, I, I, I64, F, P, P, I64, P, P, P, P, P], I),
        "dsa_sparse_attn_split": ([P, P, I64, P, I64, I, P, I, I, I, F, P, P, I, P, ctypes.c_size_t, P, P], I),
        "dsa_prefill_host_workspace_size": ([ctypes.POINTER(ForwardArgs)], ctypes.c_size_t),
        "dsa_forward_loss_workspace_size": ([ctypes.POINTER(ForwardArgs), I], ctypes.c_size_t),
        "dsa_forward_loss": ([ctypes.POINTER(ForwardArgs), I, P, P, P, ctypes.c_size_t, P], I),
        "dsa_prefill_host": ([ctypes.POINTER(ForwardArgs), P, ctypes.c_size_t, P], I),
        "dsa_sparse_attn_backward": ([P, P, I64, P, I, I, I, F, P, P, P, P, P, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    return lib


lib = _load()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(t=None):
    dev = t.device if t is not None and t.is_cuda else None
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _check(code, where):
    if code != DSA_OK:
        raise DSAError(code, where)


def _need(t, dtype, name, dims=None):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA {dtype} tensor")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name}: expected {dims} dims, got {tuple(t.shape)}")


def device_status(stream=None) -> int:
    """Status recorded in the device's shared word (calls given no status word of their own), read
    after the stream's work and cleared (dsa_device_status)."""
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream()
    return lib.dsa_device_status(s)


def status_word(device="cuda"):
    """A zeroed device int32 status word for the per-stage calls' `status` argument."""
    return torch.zeros((1,), dtype=torch.int32, device=device)


def read_status(word, stream=None) -> int:
    """Status recorded in `word` (a status_word() tensor or a workspace), read after the stream's work
    and cleared on that stream (dsa_status)."""
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(word)
    return lib.dsa_status(_ptr(word), s)


def index(q8, q_scale, w, k8, k_scale, q_pos0=0, scores=None, status=None):
    """Indexer scores of prefill rows (dsa_index). Returns scores [T, ld] fp32 (s <= pos written)."""
    _need(q8, torch.uint8, "q8", 3)
    _need(k8, torch.uint8, "k8", 2)
    for n, t in (("q_scale", q_scale), ("w", w), ("k_scale", k_scale)):
        _need(t, torch.float32, n)
    T, H_I, _ = q8.shape
    S = k8.shape[0]
    ld = (min(S, q_pos0 + T) + 3) // 4 * 4
    if scores is None:
        scores = torch.empty((T, ld), dtype=torch.float32, device=q8.device)
    _check(lib.dsa_index(_ptr(q8), _ptr(q_scale), _ptr(w), _ptr(k8), _ptr(k_scale), T, S, H_I, q_pos0,
                         _ptr(scores), scores.stride(0), _ptr(status), _stream(q8)), "dsa_index")
    return scores


def index_paged(q8, q_scale, w, k8_cache, k_scale_cache, block_table, seq_lens, max_seq_len, scores=None,
                status=None):
    """Decode indexer scores against a paged FP8 key cache (dsa_index_paged). Returns [B, ld] fp32."""
    _need(q8, torch.uint8, "q8", 3)
    _need(k8_cache, torch.uint8, "k8_cache", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, H_I, _ = q8.shape
    n_pages, page, _ = k8_cache.shape
    ld = (max_seq_len + 3) // 4 * 4
    if scores is None:
        scores = torch.empty((B, ld), dtype=torch.float32, device=q8.device)
    _check(lib.dsa_index_paged(_ptr(q8), _ptr(q_scale), _ptr(w), _ptr(k8_cache), _ptr(k_scale_cache), n_pages,
                               _ptr(block_table), block_table.stride(0), _ptr(seq_lens), B, H_I, page, max_seq_len,
                               _ptr(scores), scores.stride(0), _ptr(status), _stream(q8)), "dsa_index_paged")
    return scores


def topk(scores, k, q_pos0=0, n_cols=None, row_lens=None, idx=None):
    """Top-k positions per row (dsa_topk). Returns idx [T, k] int32, -1 padded, valid slots first."""
    _need(scores, torch.float32, "scores", 2)
    T, ld = scores.shape
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=scores.device)
    n_cols = ld if n_cols is None else n_cols
    _check(lib.dsa_topk(_ptr(scores), ld, T, _ptr(row_lens), n_cols, q_pos0, k, _ptr(idx), _stream(scores)),
           "dsa_topk")
    return idx


def sparse_attn(q, kv, idx, scale, block_table=None, page_size=0, out=None, lse=None, want_lse=True, status=None):
    """Attention over the selected latent rows (dsa_sparse_attn). Returns (out [T,H,512] bf16, lse [T,H] | None).

    kv is [S, 576] (contiguous) or [n_pages, page_size, 576] with block_table [T, P].
    """
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv")
    _need(idx, torch.int32, "idx", 2)
    T, H, _ = q.shape
    k = idx.shape[1]
    n_rows = kv.numel() // 576
    if block_table is not None:
        _need(block_table, torch.int32, "block_table", 2)
        page_size = kv.shape[1]
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    bt_stride = block_table.stride(0) if block_table is not None else 0
    _check(lib.dsa_sparse_attn(_ptr(q), _ptr(kv), n_rows, _ptr(block_table), bt_stride, page_size, _ptr(idx), T, H,
                               k, float(scale), _ptr(out), _ptr(lse), _ptr(status), _stream(q)), "dsa_sparse_attn")
    return out, lse


def dense_causal_attn(q, kv, scale, q_pos0=0, out=None, lse=None, want_lse=True, status=None):
    """Dense causal attention over every latent row up to each row's position (dsa_dense_causal_attn):
    the dense MLA baseline.  q [T, H, 576] holds rows at positions q_pos0 .. q_pos0 + T - 1, kv [S, 576].
    Returns (out [T,H,512] bf16, lse [T,H] | None)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv", 2)
    T, H, _ = q.shape
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    _check(lib.dsa_dense_causal_attn(_ptr(q), _ptr(kv), kv.shape[0], T, H, int(q_pos0), float(scale), _ptr(out),
                                     _ptr(lse), _ptr(status), _stream(q)), "dsa_dense_causal_attn")
    return out, lse


def indexer_loss(q, kv, lse, scores, scale, idx=None, q_pos0=0, p=None, kl=None, loss=None, want_p=True,
                 status=None):
    """The indexer's KL training loss (dsa_indexer_loss).  idx [T, k] selects the sparse stage (target
    over each row's selected set); idx=None is the dense warm-up over every position <= q_pos0 + t.
    lse [T, H] comes from the forward over the same sets, scores [T, ld] from the indexer.
    Returns (p [T, k] | None, kl [T], loss) with loss a float64 tensor of one element (summed over rows,
    added to `loss` when one is passed)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv", 2)
    _need(lse, torch.float32, "lse", 2)
    _need(scores, torch.float32, "scores", 2)
    T, H, _ = q.shape
    k = 0
    if idx is not None:
        _need(idx, torch.int32, "idx", 2)
        k = idx.shape[1]
        if p is None and want_p:
            p = torch.empty((T, k), dtype=torch.float32, device=q.device)
    if kl is None:
        kl = torch.empty((T,), dtype=torch.float32, device=q.device)
    if loss is None:
        loss = torch.zeros((1,), dtype=torch.float64, device=q.device)
    _check(lib.dsa_indexer_loss(_ptr(q), _ptr(kv), kv.shape[0], _ptr(idx), T, H, k, int(q_pos0), float(scale),
                                _ptr(lse), _ptr(scores), scores.stride(0), _ptr(p), _ptr(kl), _ptr(loss), _ptr(status),
                                _stream(q)),
           "dsa_indexer_loss")
    return p, kl, loss


def sparse_attn_backward(q, kv, idx, scale, out, dout, lse, dq=None, dkv=None, status=None):
    """Gradients of sparse_attn over the fixed selection idx (dsa_sparse_attn_backward).
    q [T, H, 576] / kv [S, 576] / out, dout [T, H, 512] bf16, lse [T, H] fp32 from the forward.
    Returns (dq [T, H, 576] bf16, dkv [S, 576] fp32); dkv is added to when passed (zeroed otherwise)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv", 2)
    _need(idx, torch.int32, "idx", 2)
    _need(out, torch.bfloat16, "out", 3)
    _need(dout, torch.bfloat16, "dout", 3)
    _need(lse, torch.float32, "lse", 2)
    T, H, _ = q.shape
    if dq is None:
        dq = torch.empty((T, H, 576), dtype=torch.bfloat16, device=q.device)
    if dkv is None:
        dkv = torch.zeros((kv.shape[0], 576), dtype=torch.float32, device=q.device)
    _check(lib.dsa_sparse_attn_backward(_ptr(q), _ptr(kv), kv.shape[0], _ptr(idx), T, H, idx.shape[1], float(scale),
                                        _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dkv), _ptr(status),
                                        _stream(q)), "dsa_sparse_attn_backward")
    return dq, dkv


def decode_split(B: int) -> int:
    """Key split the decode forward uses for B sequences (mirrors the library's choice)."""
    return 1 if B <= 0 or B >= 74 else max(1, min(4, 74 // B))


def sparse_attn_split(q, kv, idx, scale, n_split, block_table=None, out=None, lse=None, ws=None, status=None):
    """dsa_sparse_attn_split: attention with each row's keys spread over n_split partial passes
    (n_split = 0: the balanced partition over every SM pair that the decode forward uses)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv")
    _need(idx, torch.int32, "idx", 2)
    T, H, _ = q.shape
    page_size = kv.shape[1] if block_table is not None else 0
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    n = (lib.dsa_sparse_attn_balanced_workspace_size(T, H, idx.shape[1]) if n_split == 0
         else lib.dsa_sparse_attn_split_workspace_size(T, H, n_split))
    if ws is None and n:
        ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    bt_stride = block_table.stride(0) if block_table is not None else 0
    _check(lib.dsa_sparse_attn_split(_ptr(q), _ptr(kv), kv.numel() // 576, _ptr(block_table), bt_stride, page_size,
                                     _ptr(idx), T, H, idx.shape[1], float(scale), _ptr(out), _ptr(lse), n_split,
                                     _ptr(ws), 0 if ws is None else ws.numel(), _ptr(status), _stream(q)),
           "dsa_sparse_attn_split")
    return out, lse


class Forward:
    """Reusable fused forward (dsa_forward) for one set of shapes: owns the workspace.

    prefill: Forward.prefill(inputs, k, scale) with inputs = dict(q8, q_scale, w, k8, k_scale, q, kv)
    decode:  Forward.decode(inputs, k, scale) with inputs = dict(q8, q_scale, w, k8_cache, k_scale_cache,
             kv_cache, block_table, seq_lens, q) and max_seq_len.
    """

    def __init__(self, args: ForwardArgs, device, keep: dict):
        self.args = args
        self._keep = keep
        n = lib.dsa_forward_workspace_size(ctypes.byref(args))
        if n == 0:
            raise DSAError(1, "dsa_forward_workspace_size")
        self.ws = torch.zeros(n, dtype=torch.uint8, device=device)  # the status word at its head starts at 0

    @classmethod
    def prefill(cls, inp, k, scale, q_pos0=0, chunk_rows=0, out=None, lse=None, idx=None):
        q8, kv = inp["q8"], inp["kv"]
        T, H_I, _ = q8.shape
        H = inp["q"].shape[1]
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q8.device) if out is None else out
        a = ForwardArgs(mode=MODE_PREFILL, H_I=H_I, H=H, k=k, scale=scale, T=T, S=inp["k8"].shape[0],
                        q_pos0=q_pos0, chunk_rows=chunk_rows,
                        q8=_ptr(q8), q_scale=_ptr(inp["q_scale"]), w=_ptr(inp["w"]), k8=_ptr(inp["k8"]),
                        k_scale=_ptr(inp["k_scale"]), q=_ptr(inp["q"]), kv=_ptr(kv), out=_ptr(out),
                        lse=_ptr(lse), idx=_ptr(idx))
        f = cls(a, q8.device, dict(inp=inp, out=out, lse=lse, idx=idx))
        f.out, f.lse, f.idx = out, lse, idx
        return f

    @classmethod
    def decode(cls, inp, k, scale, max_seq_len, out=None, lse=None, idx=None):
        q8 = inp["q8"]
        B, H_I, _ = q8.shape
        H = inp["q"].shape[1]
        n_pages, page, _ = inp["k8_cache"].shape
        bt = inp["block_table"]
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q8.device) if out is None else out
        a = ForwardArgs(mode=MODE_DECODE, H_I=H_I, H=H, k=k, scale=scale, B=B, page_size=page, n_pages=n_pages,
                        block_table=_ptr(bt), bt_stride=bt.stride(0), seq_lens=_ptr(inp["seq_lens"]),
                        max_seq_len=max_seq_len, q8=_ptr(q8), q_scale=_ptr(inp["q_scale"]), w=_ptr(inp["w"]),
                        k8=_ptr(inp["k8_cache"]), k_scale=_ptr(inp["k_scale_cache"]), q=_ptr(inp["q"]),
                        kv=_ptr(inp["kv_cache"]), out=_ptr(out), lse=_ptr(lse), idx=_ptr(idx))
        f = cls(a, q8.device, dict(inp=inp, out=out, lse=lse, idx=idx))
        f.out, f.lse, f.idx = out, lse, idx
        return f

    def __call__(self, stream=None):
        s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(self.out)
        _check(lib.dsa_forward(ctypes.byref(self.args), _ptr(self.ws), self.ws.numel(), s), "dsa_forward")
        return self.out

    def status(self, stream=None) -> int:
        """Device-side status of the calls made with this workspace since the last read (dsa_status)."""
        return read_status(self.ws, stream)

    def capture(self):
        """One call captured into a CUDA graph (a torch.cuda.CUDAGraph): graph.replay() runs the same
        launches on the same buffers with no per-launch host work, as a serving loop runs its decode
        step.  The inputs are read when the graph replays, so a step writes its new tokens into the
        same tensors before replaying.  The status word keeps collecting the replays' errors."""
        dev = self.ws.device
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self()  # one call outside the capture (first-use kernel attributes are set here)
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self()
        return graph


LOSS_SPARSE, LOSS_DENSE_WARMUP = 0, 1


class ForwardLoss:
    """Training-side prefill forward with the indexer's KL loss (dsa_forward_loss): owns the workspace.

    ForwardLoss(inputs, k, scale, stage) with inputs = dict(q8, q_scale, w, k8, k_scale, q, kv) on the GPU and
    stage LOSS_SPARSE (selected sets) or LOSS_DENSE_WARMUP (every preceding key).  Calling it writes self.out,
    self.lse, self.kl (and self.idx in the sparse stage when given) and returns self.loss, a float64 tensor
    of one element holding sum_t KL_t of this call.
    """

    def __init__(self, inp, k, scale, stage=LOSS_SPARSE, q_pos0=0, chunk_rows=0, idx=None):
        q8 = inp["q8"]
        T, H_I, _ = q8.shape
        H = inp["q"].shape[1]
        dev = q8.device
        self.stage = stage
        self.out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.kl = torch.empty((T,), dtype=torch.float32, device=dev)
        self.loss = torch.zeros((1,), dtype=torch.float64, device=dev)
        self.idx = idx
        self.args = ForwardArgs(mode=MODE_PREFILL, H_I=H_I, H=H, k=k, scale=scale, T=T, S=inp["k8"].shape[0],
                                q_pos0=q_pos0, chunk_rows=chunk_rows,
                                q8=_ptr(q8), q_scale=_ptr(inp["q_scale"]), w=_ptr(inp["w"]), k8=_ptr(inp["k8"]),
                                k_scale=_ptr(inp["k_scale"]), q=_ptr(inp["q"]), kv=_ptr(inp["kv"]),
                                out=_ptr(self.out), lse=_ptr(self.lse), idx=_ptr(idx))
        self._keep = inp
        n = lib.dsa_forward_loss_workspace_size(ctypes.byref(self.args), stage)
        if n == 0:
            raise DSAError(1, "dsa_forward_loss_workspace_size")
        self.ws = torch.zeros(n, dtype=torch.uint8, device=dev)

    def __call__(self, stream=None):
        s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(self.out)
        self.loss.zero_()
        _check(lib.dsa_forward_loss(ctypes.byref(self.args), self.stage, _ptr(self.kl), _ptr(self.loss), _ptr(self.ws),
                                    self.ws.numel(), s), "dsa_forward_loss")
        return self.loss

    def status(self, stream=None) -> int:
        """Device-side status of the calls made with this workspace since the last read (dsa_status)."""
        return read_status(self.ws, stream)


class PrefillHost:
    """Prefill forward with inputs and outputs in host memory (dsa_prefill_host): owns the device workspace.

    PrefillHost(inputs, k, scale) with inputs = dict(q8, q_scale, w, k8, k_scale, q, kv) as CPU tensors
    (pinned for overlapped copies); calling it enqueues the chunked pipeline on the current stream of
    `device`; the outputs (self.out, and self.lse / self.idx if given) are valid after that stream is
    synchronised.
    """

    def __init__(self, inp, k, scale, q_pos0=0, chunk_rows=0, out=None, lse=None, idx=None, device="cuda"):
        q8 = inp["q8"]
        for n, t in inp.items():
            if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
                raise TypeError(f"{n}: expected a contiguous CPU tensor")
        T, H_I, _ = q8.shape
        H = inp["q"].shape[1]
        pin = q8.is_pinned()
        self.out = torch.empty((T, H, 512), dtype=torch.bfloat16, pin_memory=pin) if out is None else out
        self.lse, self.idx = lse, idx
        self.args = ForwardArgs(mode=MODE_PREFILL, H_I=H_I, H=H, k=k, scale=scale, T=T, S=inp["k8"].shape[0],
                                q_pos0=q_pos0, chunk_rows=chunk_rows,
                                q8=_ptr(q8), q_scale=_ptr(inp["q_scale"]), w=_ptr(inp["w"]), k8=_ptr(inp["k8"]),
                                k_scale=_ptr(inp["k_scale"]), q=_ptr(inp["q"]), kv=_ptr(inp["kv"]),
                                out=_ptr(self.out), lse=_ptr(lse), idx=_ptr(idx))
        self._keep = inp
        n = lib.dsa_prefill_host_workspace_size(ctypes.byref(self.args))
        if n == 0:
            raise DSAError(1, "dsa_prefill_host_workspace_size")
        self.device = torch.device(device)
        self.ws = torch.zeros(n, dtype=torch.uint8, device=self.device)

    def __call__(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        _check(lib.dsa_prefill_host(ctypes.byref(self.args), _ptr(self.ws), self.ws.numel(),
                                    ctypes.c_void_p(s.cuda_stream)), "dsa_prefill_host")
        return self.out

    def status(self, stream=None) -> int:
        """Device-side status of the calls made with this workspace since the last read (dsa_status)."""
        return read_status(self.ws, stream if stream is not None else torch.cuda.current_stream(self.device))


def selftest_wait_timeout(timeout_us=2000, status=None):
    """Runs the bounded-wait self-test kernel and returns the status it recorded (expects DSA_ERR_DEVICE_TIMEOUT)
    in `status` (a status_word() tensor) or, when None, in the device's shared word."""
    _check(lib.dsa_selftest_wait_timeout(timeout_us, _ptr(status), _stream()), "dsa_selftest_wait_timeout")
    return device_status() if status is None else read_status(status)
