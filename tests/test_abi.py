"""C-ABI checks that need no GPU: the library loads, exports every function include/dsa.h
declares, rejects bad arguments on the host before touching CUDA, and the Python mirror
of dsa_forward_args has the C layout."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def _lib():
    from sparse_attention_30_b300 import build
    build.build()
    import sparse_attention_30_b300 as dsa
    return dsa


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("dsa_index", "dsa_index_paged", "dsa_topk", "dsa_sparse_attn", "dsa_forward",
              "dsa_forward_workspace_size", "dsa_device_status", "dsa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    dsa = _lib()
    out = subprocess.run(["nm", "-D", "--defined-only", dsa.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (dsa_[a-z_]+)\b", out.stdout))
    for n in _declared_functions():
        assert n in exported, n
        assert hasattr(dsa.lib, n)
    assert set(dsa.EXPORTS) == set(_declared_functions())


def test_status_strings_and_version():
    dsa = _lib()
    for code, name in dsa.STATUS_NAMES.items():
        assert dsa.lib.dsa_status_string(code).decode() == name
    assert dsa.lib.dsa_status_string(99).decode() == "DSA_ERR_UNKNOWN"
    assert dsa.lib.dsa_version() >> 16 == 2


# Fake, 16-byte-aligned "device" addresses: validation must reject the call before any of
# them is dereferenced or any CUDA call is made.
A = 1 << 20


def test_index_rejects_bad_arguments_on_host():
    dsa = _lib()
    f = dsa.lib.dsa_index
    ok = dict(q8=A, qs=A, w=A, k8=A, ks=A, T=4, S=8, H=64, pos=0, sc=A, ld=8)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["q8"], a["qs"], a["w"], a["k8"], a["ks"], a["T"], a["S"], a["H"], a["pos"], a["sc"], a["ld"], None,
                 None)

    assert call(q8=None) == 1
    assert call(k8=A + 8) == 1          # misaligned
    assert call(ld=6) == 1              # ld % 4
    assert call(ld=4, T=8) == 1         # ld < min(S, pos + T)
    assert call(ld=4) == 4              # valid: with no GPU here it fails at the CUDA call
    assert call(H=48) == 1              # not a power of two
    assert call(H=2) == 2               # powers of two below 4 are not built
    assert call(H=1) == 2
    assert call(H=256) == 1
    assert call(S=0) == 1
    assert call(pos=-1) == 1
    assert call(T=0) == 0               # empty is a no-op with nothing launched


def test_paged_index_rejects_unsupported_heads_and_pages():
    dsa = _lib()
    f = dsa.lib.dsa_index_paged

    def call(H=64, page=64, bt_stride=2, max_len=128, ld=128, B=1):
        return f(A, A, A, A, A, 4, A, bt_stride, A, B, H, page, max_len, A, ld, None, None)

    assert call(H=16) == 2              # decode tiles need H_I of 32, 64 or 128
    assert call(H=8) == 2
    assert call(page=48) == 1
    assert call(page=256) == 1
    assert call(bt_stride=1) == 1       # fewer table entries than max_len needs
    assert call(ld=64) == 1
    assert call(B=0) == 0


def test_topk_and_attention_reject_bad_arguments_on_host():
    dsa = _lib()
    t = dsa.lib.dsa_topk
    assert t(A, 8, 2, None, 8, 0, 0, A, None) == 1        # k = 0
    assert t(A, 8, 2, None, 16, 0, 4, A, None) == 1       # n_cols > ld
    assert t(A, 6, 2, None, 6, 0, 4, A, None) == 1        # ld % 4
    assert t(None, 8, 2, None, 8, 0, 4, A, None) == 1
    assert t(A, 8, 0, None, 8, 0, 4, A, None) == 0
    s = dsa.lib.dsa_sparse_attn
    assert s(A, A, 10, None, 0, 0, A, 2, 129, 4, 0.1, A, None, None, None) == 2   # H > 128
    assert s(A, A + 2, 10, None, 0, 0, A, 2, 8, 4, 0.1, A, None, None, None) == 1
    assert s(A, A, 0, None, 0, 0, A, 2, 8, 4, 0.1, A, None, None, None) == 1
    assert s(A, A, 10, None, 0, 0, A, 0, 8, 4, 0.1, A, None, None, None) == 0
    d = dsa.lib.dsa_dense_causal_attn
    assert d(A, A, 10, 2, 129, 0, 0.1, A, None, None, None) == 2          # H > 128
    assert d(A, A, 10, 4, 8, 7, 0.1, A, None, None, None) == 1            # q_pos0 + T > n_kv_rows
    assert d(A, A, 10, 2, 8, -1, 0.1, A, None, None, None) == 1           # negative position
    assert d(A, A + 2, 10, 2, 8, 0, 0.1, A, None, None, None) == 1        # misaligned kv
    assert d(None, A, 10, 2, 8, 0, 0.1, A, None, None, None) == 1
    assert d(A, A, 1 << 31, 2, 8, 0, 0.1, A, None, None, None) == 1       # rows past int32
    assert d(A, A, 10, 0, 8, 3, 0.1, A, None, None, None) == 0            # nothing to do
    L = dsa.lib.dsa_indexer_loss
    #        q  kv  n   idx   T  H  k  pos0 scale lse scores ld  p     kl    loss  status stream
    assert L(A, A, 10, A, 2, 129, 4, 0, 0.1, A, A, 16, None, None, None, None, None) == 2     # H > 128
    assert L(A, A, 10, A, 2, 8, 0, 0, 0.1, A, A, 16, None, None, None, None, None) == 1       # k = 0
    assert L(A, A, 10, A, 2, 8, 4, 0, 0.1, None, A, 16, None, None, None, None, None) == 1    # no lse
    assert L(A, A, 10, A, 2, 8, 4, 0, 0.1, A, None, 16, None, None, None, None, None) == 1    # no scores
    assert L(A, A, 10, None, 4, 8, 0, 7, 0.1, A, A, 16, None, None, None, None, None) == 1    # dense: rows past keys
    assert L(A, A, 20, None, 4, 8, 0, 7, 0.1, A, A, 10, None, None, None, None, None) == 1    # dense: rows past ld
    assert L(A, A, 20, None, 4, 8, 0, 0, 0.1, A, A, 10, A, None, None, None, None) == 1  # dense: no per-slot target
    assert L(A, A + 2, 10, A, 2, 8, 4, 0, 0.1, A, A, 16, None, None, None, None, None) == 1   # misaligned kv
    assert L(A, A, 10, A, 0, 8, 4, 0, 0.1, A, A, 16, None, None, None, None, None) == 0       # nothing to do


def test_wait_limit_default_and_environment_override():
    import subprocess
    import sys
    code = "import sparse_attention_30_b300 as d; print(d.lib.dsa_wait_limit_ns())"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    def run(env_value):
        env = dict(os.environ)
        env.pop("DSA_WAIT_LIMIT_MS", None)
        if env_value is not None:
            env["DSA_WAIT_LIMIT_MS"] = env_value
        out = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, check=True)
        return int(out.stdout.strip().splitlines()[-1])
    assert run(None) == 1 << 30
    assert run("30000") == 30000 * 1000000
    for bad in ("0", "-5", "12ms", "", "99999999999"):
        assert run(bad) == 1 << 30


def test_forward_workspace_and_validation():
    dsa = _lib()
    a = dsa.ForwardArgs(mode=dsa.MODE_PREFILL, H_I=64, H=128, k=2048, scale=0.07, T=4096, S=4096, q_pos0=0,
                        chunk_rows=1024)
    n = dsa.lib.dsa_forward_workspace_size(ctypes.byref(a))
    # the 256-byte status head, one 1024-row fp32 score block and the int32 selection of all rows
    assert n == 256 + 1024 * 4096 * 4 + 4096 * 2048 * 4
    a.T = 5000                                        # q_pos0 + T > S
    assert dsa.lib.dsa_forward_workspace_size(ctypes.byref(a)) == 0
    d = dsa.ForwardArgs(mode=dsa.MODE_DECODE, H_I=64, H=128, k=2048, scale=0.07, B=64, page_size=64,
                        n_pages=32768, bt_stride=512, max_seq_len=32768)
    assert dsa.lib.dsa_forward_workspace_size(ctypes.byref(d)) == 256 + 64 * 32768 * 4 + 64 * 2048 * 4
    d.mode = 7
    assert dsa.lib.dsa_forward_workspace_size(ctypes.byref(d)) == 0
    d.mode = dsa.MODE_DECODE
    # null inputs are rejected before the workspace is even looked at
    assert dsa.lib.dsa_forward(ctypes.byref(d), None, 0, None) == 1


def test_forward_loss_workspace_and_validation():
    dsa = _lib()
    a = dsa.ForwardArgs(mode=dsa.MODE_PREFILL, H_I=64, H=128, k=2048, scale=0.07, T=4096, S=4096, q_pos0=0,
                        chunk_rows=1024)
    ws = dsa.lib.dsa_forward_loss_workspace_size
    # sparse stage: the status head, the score block of one chunk and the selection of all rows
    assert ws(ctypes.byref(a), dsa.LOSS_SPARSE) == 256 + 1024 * 4096 * 4 + 4096 * 2048 * 4
    # dense warm-up: the status head and the score block
    assert ws(ctypes.byref(a), dsa.LOSS_DENSE_WARMUP) == 256 + 1024 * 4096 * 4
    assert ws(ctypes.byref(a), 2) == 0                                   # no such stage
    d = dsa.ForwardArgs(mode=dsa.MODE_DECODE, H_I=64, H=128, k=2048, scale=0.07, B=64, page_size=64,
                        n_pages=32768, bt_stride=512, max_seq_len=32768)
    assert ws(ctypes.byref(d), dsa.LOSS_SPARSE) == 0                     # prefill only
    f = dsa.lib.dsa_forward_loss
    assert f(ctypes.byref(d), dsa.LOSS_SPARSE, None, None, None, 0, None) == 1
    assert f(ctypes.byref(a), 5, None, None, None, 0, None) == 1
    # every input and lse are required (lse feeds the loss), checked before the workspace
    assert f(ctypes.byref(a), dsa.LOSS_SPARSE, None, None, None, 0, None) == 1


def test_prefill_host_workspace_and_validation():
    dsa = _lib()
    a = dsa.ForwardArgs(mode=dsa.MODE_PREFILL, H_I=64, H=128, k=2048, scale=0.07, T=4096, S=4096, q_pos0=0,
                        chunk_rows=1024)
    n = dsa.lib.dsa_prefill_host_workspace_size(ctypes.byref(a))
    keys = 4096 * 128 + 4096 * 4 + 4096 * 576 * 2
    slot = 1024 * (64 * 128 + 64 * 4 + 64 * 4 + 128 * 576 * 2 + 2048 * 4 + 128 * 512 * 2 + 128 * 4)
    assert n == 256 + keys + 2 * slot + 1024 * 4096 * 4
    a.mode = dsa.MODE_DECODE                          # prefill only
    assert dsa.lib.dsa_prefill_host_workspace_size(ctypes.byref(a)) == 0
    assert dsa.lib.dsa_prefill_host(ctypes.byref(a), None, 0, None) == 1
    a.mode = dsa.MODE_PREFILL
    assert dsa.lib.dsa_prefill_host(ctypes.byref(a), None, 0, None) == 1       # null inputs
    buf = ctypes.create_string_buffer(64)
    P = ctypes.cast(buf, ctypes.c_void_p).value
    for f in ("q8", "q_scale", "w", "k8", "k_scale", "q", "kv", "out"):
        setattr(a, f, P)
    assert dsa.lib.dsa_prefill_host(ctypes.byref(a), None, 0, None) == 3       # no workspace
    assert dsa.lib.dsa_prefill_host(ctypes.byref(a), P + 1, n, None) == 3      # misaligned / too small


def test_forward_args_layout_matches_c():
    dsa = _lib()
    fields = [f for f, _ in dsa.ForwardArgs._fields_]
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"dsa.h\"\nint main(void){\n"
    src += 'printf("%zu\\n", sizeof(dsa_forward_args));\n'
    for f in fields:
        src += f'printf("%zu\\n", offsetof(dsa_forward_args, {f}));\n'
    src += "return 0;}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        vals = [int(x) for x in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(dsa.ForwardArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(dsa.ForwardArgs, f).offset == off, f


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_attention_30_b300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), fn
                assert "oracle/" not in text, fn


def _bal_parts(rows, tpr, n_cl):
    """Most clusters any row is spread over when rows x tpr tiles are cut into n_cl equal ranges
    (cluster c covers tiles [c G / n_cl, (c + 1) G / n_cl))."""
    G = rows * tpr
    cl = lambda g: ((g + 1) * n_cl - 1) // G
    return max(cl(t * tpr + tpr - 1) - cl(t * tpr) + 1 for t in range(rows))


def test_decode_split_mirror_matches_library_workspace():
    # the binding's decode_split mirrors the library's key-split choice; the library's decode
    # workspace holds the fp32 partial outputs exactly when it splits, so the sizes must agree
    dsa = _lib()
    H, k, max_len = 128, 2048, 4096
    r256 = lambda x: (x + 255) // 256 * 256
    for B in [1, 2, 5, 18, 19, 36, 37, 73, 74, 75, 200]:
        d = dsa.ForwardArgs(mode=dsa.MODE_DECODE, H_I=64, H=H, k=k, scale=0.07, B=B, page_size=64,
                            n_pages=B * 64, bt_stride=64, max_seq_len=max_len)
        n = dsa.lib.dsa_forward_workspace_size(ctypes.byref(d))
        split = dsa.decode_split(B)
        want = 256 + r256(B * max_len * 4) + r256(B * k * 4)
        if split > 1:
            want += r256(B * split * H * 512 * 4) + r256(B * split * H * 2 * 4)
        assert n == want, (B, split, n, want)
        assert split == (1 if B >= 74 else max(1, min(4, 74 // B)))


def test_balanced_partition_workspace():
    # dsa_sparse_attn_split with n_split = 0 cuts the rows' ceil(k / 64) tiles each, end to end, into
    # equal contiguous ranges, one per SM pair (74 here: with no GPU the library assumes a B300's
    # 148 SMs); its workspace holds one fp32 partial result per cluster a row is spread over
    dsa = _lib()
    H, k = 128, 2048
    r256 = lambda x: (x + 255) // 256 * 256
    for B in [1, 2, 5, 18, 32, 37, 64, 74, 75, 148, 200]:
        tpr = k // 64
        n_cl = min(74, B * tpr)
        parts = _bal_parts(B, tpr, n_cl)
        bal = dsa.lib.dsa_sparse_attn_balanced_workspace_size(B, H, k)
        assert bal == (0 if parts == 1 else r256(B * parts * H * 512 * 4) + r256(B * parts * H * 2 * 4)), B
        G = B * tpr
        sizes = [(c + 1) * G // n_cl - c * G // n_cl for c in range(n_cl)]
        assert max(sizes) - min(sizes) <= 1 and sum(sizes) == G          # equal shares, within one tile
    assert _bal_parts(64, 32, 74) == 3 and _bal_parts(1, 32, 32) == 32
    assert dsa.lib.dsa_sparse_attn_balanced_workspace_size(0, H, k) == 0


def test_default_prefill_chunk_keeps_the_score_block_near_one_gib():
    # chunk_rows = 0 lets the library choose: about 1 GiB of fp32 scores, 256..8192 rows, at most T
    dsa = _lib()
    for S, T, want_chunk in [(131072, 131072, 2048), (4096, 4096, 4096), (65536, 100, 100), (1 << 22, 8192, 256)]:
        a = dsa.ForwardArgs(mode=dsa.MODE_PREFILL, H_I=64, H=128, k=2048, scale=0.07, T=T, S=S, q_pos0=S - T,
                            chunk_rows=0)
        ld = (S + 3) // 4 * 4
        r256 = lambda x: (x + 255) // 256 * 256
        assert dsa.lib.dsa_forward_workspace_size(ctypes.byref(a)) == 256 + r256(want_chunk * ld * 4) + r256(T * 2048 * 4)


def test_status_reads_reject_bad_words_on_host():
    dsa = _lib()
    assert dsa.lib.dsa_status(None, None) == 1                # no word
    assert dsa.lib.dsa_status(A + 2, None) == 1               # misaligned word
    assert dsa.lib.dsa_selftest_wait_timeout(0, None, None) == 1


def test_noalloc_decode_checks_every_argument_before_launching():
    # a bad attention argument (misaligned output) is refused before the indexer and top-k are
    # queued, so nothing touches the caller's buffers
    dsa = _lib()
    a = dsa.ForwardArgs(mode=dsa.MODE_DECODE, H_I=64, H=128, k=2048, scale=0.07, B=4, page_size=64, n_pages=64,
                        bt_stride=16, max_seq_len=1024, block_table=A, seq_lens=A, q8=A, q_scale=A, w=A, k8=A,
                        k_scale=A, q=A, kv=A, out=A + 8, idx=A)
    assert dsa.lib.dsa_decode_noalloc(ctypes.byref(a), None) == 1
    a.out, a.H = A, 200                                       # too many heads: unsupported
    assert dsa.lib.dsa_decode_noalloc(ctypes.byref(a), None) == 2
    a.H, a.kv = 128, None
    assert dsa.lib.dsa_decode_noalloc(ctypes.byref(a), None) == 1
