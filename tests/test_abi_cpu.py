"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and rejects bad arguments before touching the GPU (no GPU here)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")

DSA_OK, INVALID, UNSUPPORTED, OOM, BAD_BLOCK, CUDA, TIMEOUT, WORKSPACE = range(8)


def declared_functions():
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(dsa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("dsa_index_scores", "dsa_topk_select", "dsa_kv_gather", "dsa_sparse_attn_decode",
              "dsa_sparse_attn_prefill", "dsa_kv_write", "dsa_kv_alloc_create", "dsa_decode_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from dynamic_sparse_attention_indexer_gb300 import _abi
    names = declared_functions()
    assert len(names) >= 18
    raw = C.CDLL(_abi._build.LIB)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in dsa.h but not exported"
        assert n in _abi.SIGNATURES, f"{n} has no ctypes signature"
    assert lib.dsa_abi_version() == 4
    assert lib.dsa_status_string(OOM) == b"DSA_ERR_OOM"


def test_block_allocator(lib):
    from dynamic_sparse_attention_indexer_gb300 import BlockAllocator, DSAError
    a = BlockAllocator(10)
    assert a.num_free == 10
    assert a.alloc(3) == [0, 1, 2]
    assert a.alloc(2) == [3, 4]
    a.free([1, 3])
    assert a.num_free == 7
    assert a.alloc(3) == [1, 3, 5]          # lowest free ids first
    with pytest.raises(DSAError) as e:
        a.alloc(6)                            # 4 free: OOM takes none
    assert e.value.status == OOM and a.num_free == 4
    with pytest.raises(DSAError):
        a.free([2, 2])                        # duplicate in one call
    with pytest.raises(DSAError):
        a.free([9])                           # never allocated
    with pytest.raises(DSAError):
        a.free([0, 42])                       # out of range: nothing freed
    assert a.num_free == 4
    a.free([0, 1, 2, 3, 4, 5])
    assert a.num_free == 10


def _kv(**over):
    from dynamic_sparse_attention_indexer_gb300 import _abi
    f = dict(k_cache=0x10000, v_cache=0x20000, idx_cache=0x30000, block_table=0x40000, context_lens=0x50000,
             num_blocks=16, block_size=64, num_kv_heads=2, head_dim=128, idx_dim=64, max_blocks_per_seq=8,
             batch=2, max_context_len=500)
    f.update(over)
    return _abi.PagedKV(**f)


def _qs(mode=0, n_q=2, seq=0, pos0=0):
    from dynamic_sparse_attention_indexer_gb300 import _abi
    return _abi.QuerySet(mode, n_q, seq, pos0)


@pytest.mark.parametrize("over,status", [
    (dict(block_size=32), UNSUPPORTED),
    (dict(head_dim=64), UNSUPPORTED),
    (dict(idx_dim=128), UNSUPPORTED),
    (dict(num_kv_heads=3), UNSUPPORTED),
    (dict(num_kv_heads=16), UNSUPPORTED),
    (dict(k_cache=0), INVALID),
    (dict(v_cache=0x20008), INVALID),         # misaligned
    (dict(max_context_len=8 * 64 + 1), INVALID),
    (dict(batch=0), INVALID),
    (dict(kv_row_stride=2 * 128 - 8), INVALID),   # below the row of two KV heads
    (dict(kv_row_stride=2 * 2 * 128 + 4), INVALID),  # rows not 16-byte aligned
])
def test_index_scores_rejects_bad_cache(lib, over, status):
    kv = _kv(**over)
    qs = _qs(n_q=kv.batch)
    st = lib.dsa_index_scores(C.byref(kv), C.byref(qs), 0x60000, 0, 0x70000, 512, None, 0, None)
    assert st == status
    assert lib.dsa_last_error_message()


def test_kv_row_stride_layouts_accepted(lib):
    """0 (separate arrays), the separate and the adjacent strides pass the cache
    checks (the call then reaches the CUDA runtime, absent here)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for stride, v in ((0, 0x20000), (2 * 128, 0x20000), (2 * 2 * 128, 0x10000 + 2 * 128 * 2)):
        kv = _kv(kv_row_stride=stride, v_cache=v)
        qs = _qs(n_q=kv.batch)
        assert lib.dsa_index_scores(C.byref(kv), C.byref(qs), 0x60000, 0, 0x70000, 512, None, 0, None) == CUDA


def test_argument_checks(lib):
    kv = _kv()
    qs = _qs()
    # ld too small, ld not a multiple of 4, misaligned scores
    assert lib.dsa_index_scores(C.byref(kv), C.byref(qs), 0x60000, 0, 0x70000, 496, None, 0, None) == INVALID
    assert lib.dsa_index_scores(C.byref(kv), C.byref(qs), 0x60000, 0, 0x70000, 514, None, 0, None) == INVALID
    assert lib.dsa_index_scores(C.byref(kv), C.byref(qs), 0x60000, 0, 0x70004, 512, None, 0, None) == INVALID
    # decode query set must cover the batch; prefill positions must fit the table
    assert lib.dsa_index_scores(C.byref(kv), C.byref(_qs(n_q=3)), 0x60000, 0, 0x70000, 512, None, 0,
                                None) == INVALID
    assert lib.dsa_index_scores(C.byref(kv), C.byref(_qs(1, 100, 0, 500)), 0x60000, 0, 0x70000, 1024, None,
                                0, None) == INVALID
    assert lib.dsa_index_scores(C.byref(kv), C.byref(_qs(1, 10, 2, 0)), 0x60000, 0, 0x70000, 512, None, 0,
                                None) == INVALID
    # top-k: k >= 1, prefix >= 0, workspace large enough
    args = (C.byref(kv), C.byref(qs), 0x70000, 512)
    assert lib.dsa_topk_select(*args, 0, 0, 0x80000, 0x90000, 0xA0000, 1 << 30, None) == INVALID
    assert lib.dsa_topk_select(*args, -1, 8, 0x80000, 0x90000, 0xA0000, 1 << 30, None) == INVALID
    assert lib.dsa_topk_select(*args, 0, 8, 0x80000, 0x90000, None, 0, None) == WORKSPACE
    assert lib.dsa_topk_select(*args, 0, 8, 0x80000, 0x90000, 0xA0000, 16, None) == WORKSPACE
    # attention: heads must be a multiple of the KV heads, group <= 16, known out dtype
    a = (C.byref(kv), 0x60000)
    assert lib.dsa_sparse_attn_decode(*a, 3, 0x80000, 0x90000, 8, 0, 0.1, 0xB0000, 0, None, 0xA0000,
                                      1 << 30, None) == INVALID
    assert lib.dsa_sparse_attn_decode(*a, 34, 0x80000, 0x90000, 8, 0, 0.1, 0xB0000, 0, None, 0xA0000,
                                      1 << 30, None) == UNSUPPORTED
    assert lib.dsa_sparse_attn_decode(*a, 8, 0x80000, 0x90000, 8, 0, 0.1, 0xB0000, 7, None, 0xA0000,
                                      1 << 30, None) == INVALID
    assert lib.dsa_sparse_attn_decode(*a, 8, 0x80000, 0x90000, 8, 0, float("nan"), 0xB0000, 0, None,
                                      0xA0000, 1 << 30, None) == INVALID
    # more than 64 query heads: the attention kernels stage one query's Q (all
    # heads) in a 64-head shared-memory slot, so the host refuses Hq = 128 even
    # with a valid group (Hkv = 8, G = 16), on every call that reaches them
    kv8 = _kv(num_kv_heads=8)
    assert lib.dsa_sparse_attn_decode(C.byref(kv8), 0x60000, 128, 0x80000, 0x90000, 8, 0, 0.1, 0xB0000, 0, None,
                                      0xA0000, 1 << 30, None) == UNSUPPORTED
    assert b"64" in lib.dsa_last_error_message()
    assert lib.dsa_sparse_attn_prefill(C.byref(kv8), C.byref(_qs(1, 10, 0, 0)), 0x60000, 128, 0x80000, 0x90000, 8,
                                       0, 0.1, 0xB0000, 0, None, 0xA0000, 1 << 30, None) == UNSUPPORTED
    assert lib.dsa_decode_step(C.byref(kv8), 0x60000, 0x68000, 128, 0, 8, 0.1, 0x70000, 512, 0x80000, 0x90000,
                               0xB0000, 0, None, 0xA0000, 1 << 30, None) == UNSUPPORTED
    assert lib.dsa_workspace_size(3, C.byref(kv8), C.byref(qs), 8, 128, 0) == 0
    # 64 heads with Hkv = 8 pass the head check (the call then reaches the
    # workspace check, which a tiny workspace fails)
    assert lib.dsa_sparse_attn_decode(C.byref(kv8), 0x60000, 64, 0x80000, 0x90000, 8, 0, 0.1, 0xB0000, 0, None,
                                      0xA0000, 16, None) == WORKSPACE
    # the split form: n_dense outside [-1, n_q]
    qs10 = _qs(1, 10, 0, 0)
    for n in (-2, 11):
        assert lib.dsa_sparse_attn_prefill_split(C.byref(kv), C.byref(qs10), 0x60000, 8, 0x80000, 0x90000, 8, 0,
                                                 0.1, n, 0xB0000, 0, None, 0xA0000, 1 << 30, None) == INVALID
    assert lib.dsa_prefill_dense_queries(C.byref(kv), C.byref(qs), 8, 8, 0) == -1   # a decode query set
    # fused prefill selection: a prefill query set, k >= 1, aligned q_idx, outputs present
    assert lib.dsa_prefill_select(C.byref(kv), C.byref(qs), 0x60000, 0, 8, 0x80000, 0x90000, None) == INVALID
    assert lib.dsa_prefill_select(C.byref(kv), C.byref(qs10), 0x60000, 0, 0, 0x80000, 0x90000, None) == INVALID
    assert lib.dsa_prefill_select(C.byref(kv), C.byref(qs10), 0x60004, 0, 8, 0x80000, 0x90000, None) == INVALID
    assert lib.dsa_prefill_select(C.byref(kv), C.byref(qs10), 0x60000, 0, 8, None, 0x90000, None) == INVALID
    # window attention: window >= 1, a prefill query set for the prefill form,
    # at most 64 query heads, a large enough workspace
    assert lib.dsa_window_attn_decode(C.byref(kv), 0x60000, 8, 0, 0.1, 0xB0000, 0, None, 0xA0000, 1 << 30,
                                      None) == INVALID
    assert lib.dsa_window_attn_decode(C.byref(kv8), 0x60000, 128, 16, 0.1, 0xB0000, 0, None, 0xA0000, 1 << 30,
                                      None) == UNSUPPORTED
    assert lib.dsa_window_attn_decode(C.byref(kv), 0x60000, 8, 16, 0.1, 0xB0000, 0, None, 0xA0000, 16,
                                      None) == WORKSPACE
    assert lib.dsa_window_attn_decode(C.byref(kv), 0x60008, 8, 16, 0.1, 0xB0000, 0, None, 0xA0000, 1 << 30,
                                      None) == INVALID
    assert lib.dsa_window_workspace_size(C.byref(kv), 8, 16) >= 2 * 16 * 4
    assert lib.dsa_window_workspace_size(C.byref(kv), 8, 0) == 0
    assert lib.dsa_window_attn_prefill(C.byref(kv), C.byref(qs), 0x60000, 8, 16, 0.1, 0xB0000, 0, None,
                                       None) == INVALID
    assert lib.dsa_window_attn_prefill(C.byref(kv), C.byref(qs10), 0x60000, 8, -3, 0.1, 0xB0000, 0, None,
                                       None) == INVALID
    assert lib.dsa_window_attn_prefill(C.byref(kv), C.byref(qs10), 0x60000, 8, 16, float("nan"), 0xB0000, 0,
                                       None, None) == INVALID
    # the prefill step: a prefill query set, aligned q_idx, outputs present
    assert lib.dsa_prefill_step(C.byref(kv), C.byref(qs), 0x60000, 0x70000, 8, 0, 8, 0.1, 0x80000, 512, 0x90000,
                                0xA0000, 0xB0000, 0, None, None, 0, None) == INVALID   # decode query set
    assert lib.dsa_prefill_step(C.byref(kv), C.byref(qs10), 0x60000, 0x70004, 8, 0, 8, 0.1, 0x80000, 512,
                                0x90000, 0xA0000, 0xB0000, 0, None, None, 0, None) == INVALID   # misaligned q_idx
    assert lib.dsa_prefill_step(C.byref(kv), C.byref(qs10), 0x60000, 0x70000, 8, 0, 8, 0.1, 0x80000, 512,
                                None, 0xA0000, 0xB0000, 0, None, None, 0, None) == INVALID      # no idx
    assert lib.dsa_prefill_step(C.byref(kv), C.byref(qs10), 0x60000, 0x70000, 8, 0, 8, 0.1, 0x80000, 512,
                                0x90000, 0xA0000, 0xB0000, 0, None, 0xC0000, 16, None) == WORKSPACE
    # prefill attention refuses a decode query set
    assert lib.dsa_sparse_attn_prefill(C.byref(kv), C.byref(qs), 0x60000, 8, 0x80000, 0x90000, 8, 0, 0.1,
                                       0xB0000, 0, None, None, 0, None) == INVALID
    # kv_write: negative count, misaligned source
    assert lib.dsa_kv_write(C.byref(kv), 0x1000, -1, 0x2000, 0x3000, 0x4000, None) == INVALID
    assert lib.dsa_kv_write(C.byref(kv), 0x1000, 4, 0x2008, 0x3000, 0x4000, None) == INVALID
    assert lib.dsa_kv_write(C.byref(kv), 0x1000, 0, 0x2008, 0x3000, 0x4000, None) == DSA_OK  # nothing to do
    # per-head write: negative count, misaligned slots or sources, missing pointers
    assert lib.dsa_kv_write_heads(C.byref(kv), 0x1000, -1, 0x2000, 0x3000, 0x4000, None) == INVALID
    assert lib.dsa_kv_write_heads(C.byref(kv), 0x1002, 4, 0x2000, 0x3000, 0x4000, None) == INVALID
    assert lib.dsa_kv_write_heads(C.byref(kv), 0x1000, 4, 0x2000, 0x3008, 0x4000, None) == INVALID
    assert lib.dsa_kv_write_heads(C.byref(kv), 0x1000, 4, 0x2000, 0x3000, None, None) == INVALID
    assert lib.dsa_kv_write_heads(C.byref(kv), 0x1000, 0, 0x2008, 0x3000, 0x4000, None) == DSA_OK


def test_valid_call_without_gpu_reports_cuda_error(lib):
    """With every argument valid the call reaches the CUDA runtime, which has
    no device here: a DSA_ERR_CUDA status, never a crash or a host fallback."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    kv = _kv()
    qs = _qs()
    assert lib.dsa_index_scores(C.byref(kv), C.byref(qs), 0x60000, 0, 0x70000, 512, None, 0, None) == CUDA


def test_workspace_sizes(lib):
    kv = _kv()
    qs = _qs()
    size = lambda op, k=8, hq=8, p=0: lib.dsa_workspace_size(op, C.byref(kv), C.byref(qs), k, hq, p)
    assert size(0) == 0                       # index_scores needs none
    topk, step = size(1), size(3)
    assert topk >= 2 * 1024 * 4                # a coarse histogram per sequence
    assert step > topk and step == size(2)     # plus the selected slots and the attention partials
    # the 128K decode workload: 8 sequences, 64/8 heads, prefix 1024, k 2048
    kv3 = _kv(num_blocks=16384, num_kv_heads=8, max_blocks_per_seq=2048, batch=8, max_context_len=131072)
    qs3 = _qs(n_q=8)
    s3 = lib.dsa_workspace_size(3, C.byref(kv3), C.byref(qs3), 2048, 64, 1024)
    assert 8 * 2048 * 4 <= s3 < 64 << 20      # selected slots + attention partials, well under 64 MB
    assert lib.dsa_workspace_size(3, C.byref(kv3), C.byref(qs3), 0, 64, 1024) == 0   # invalid k
    # the 16K prefill chunk: the automatic split sends every query to the dense
    # pass, whose workspace is the attended-position bitmap (8 B per query and
    # 64 positions), prefix or not
    kv4 = _kv(num_blocks=256, num_kv_heads=4, max_blocks_per_seq=256, batch=1, max_context_len=16384)
    qs4 = _qs(1, 16384, 0, 0)
    assert lib.dsa_prefill_dense_queries(C.byref(kv4), C.byref(qs4), 2048, 32, 576) == 16384
    bitmap = 16384 * 256 * 8
    assert lib.dsa_workspace_size(4, C.byref(kv4), C.byref(qs4), 2048, 32, 576) == bitmap
    assert lib.dsa_workspace_size(4, C.byref(kv4), C.byref(qs4), 2048, 32, 0) == bitmap
    wsz = lambda p, n: lib.dsa_prefill_attn_workspace_size(C.byref(kv4), C.byref(qs4), 2048, 32, p, n)
    assert wsz(576, -1) == bitmap
    # every query gathered: with a prefix the prefix part of every (query, head), 520 B each
    assert wsz(576, 0) - wsz(0, 0) >= 16384 * 32 * 520
    assert wsz(0, 0) < 16 << 20                # no per-query selection state in prefill
    # a split: the bitmap of the dense queries plus the gathered part's state
    assert wsz(576, 8192) >= 8192 * 128 * 8 + 8192 * 32 * 520
    assert wsz(576, 16385) == 0                # more dense queries than the set has
    # deep into a long sequence the automatic split gathers everything
    kv5 = _kv(num_blocks=4096, num_kv_heads=4, max_blocks_per_seq=4096, batch=1, max_context_len=262144)
    assert lib.dsa_prefill_dense_queries(C.byref(kv5), C.byref(_qs(1, 4096, 0, 200000)), 2048, 32, 576) == 0
    # and near its start takes a whole number of dense tile pairs (2 x 16 queries at group 8)
    n = lib.dsa_prefill_dense_queries(C.byref(kv5), C.byref(_qs(1, 4096, 0, 24000)), 2048, 32, 576)
    assert n == (10 * (576 + 2048) - 24000) // 32 * 32


def test_no_alloc_topk_refuses_batches_beyond_the_static_scratch(lib):
    """The allocation-free decode top-k keeps exactly 4096 bytes of scratch per
    sequence in its 4 MiB static array: batch 1024 fits, batch 1025 is refused
    on the host before anything touches the GPU (fake pointers, no GPU here:
    an accepted call goes on to the CUDA runtime and reports DSA_ERR_CUDA)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: an accepted call would launch on these fake pointers")
    fn = lib.dsa_topk_select_decode_noalloc
    for batch, want in ((1024, CUDA), (1025, UNSUPPORTED), (2048, UNSUPPORTED)):
        kv = _kv(batch=batch, max_context_len=500)
        st = fn(C.byref(kv), 0x70000, 512, 64, 64, 0x80000, 0x90000, None)
        assert st == want, (batch, st, lib.dsa_last_error_message())
        if want == UNSUPPORTED:
            assert b"static" in lib.dsa_last_error_message()


def test_per_head_decode_checks(lib):
    """The per-KV-head decode step runs one selection per (sequence, KV head):
    batch x num_kv_heads is held to the decode selection's 2048 rows, the
    scores matrix has one row per (sequence, KV head), and the usual pointer,
    dtype and workspace checks apply before anything reaches the GPU."""
    import torch
    fn = lib.dsa_decode_step_heads
    kv = _kv()                                    # 2 sequences, 2 KV heads, contexts up to 500
    ws = lib.dsa_heads_workspace_size(C.byref(kv), 8, 16, 0)
    # the virtual block table (one row per (sequence, KV head)) comes first
    assert ws >= 2 * 2 * 8 * 4 > 0
    assert lib.dsa_heads_workspace_size(C.byref(_kv(batch=4)), 8, 16, 0) > ws
    assert lib.dsa_heads_workspace_size(C.byref(kv), 8, 0, 0) == 0       # invalid k
    assert lib.dsa_heads_workspace_size(C.byref(kv), 5, 16, 0) == 0      # heads not a multiple of Hkv
    call = lambda kv=kv, q=0x60000, qi=0x70000, hq=8, k=16, ld=512, ws_bytes=ws, odt=0, scale=0.1, bth=None: fn(
        C.byref(kv), q, qi, bth, hq, 0, k, scale, 0x80000, ld, 0x90000, 0xA0000, 0xB0000, odt, None, 0xC0000,
        ws_bytes, None)
    assert call(qi=0x70004) == INVALID            # misaligned indexer query
    assert call(bth=0x50002) == INVALID           # misaligned per-head block tables
    assert call(qi=None) == INVALID
    assert call(q=0x60008) == INVALID             # misaligned query
    assert call(odt=5) == INVALID
    assert call(scale=float("inf")) == INVALID
    assert call(ld=100) == INVALID                # a score row shorter than the longest context
    assert call(ws_bytes=ws - 1) == WORKSPACE
    assert call(hq=128) == UNSUPPORTED            # more than 64 query heads
    big = _kv(batch=1025, max_context_len=500)    # 1025 x 2 (sequence, head) rows
    assert call(kv=big, ws_bytes=1 << 40) == UNSUPPORTED
    assert lib.dsa_heads_workspace_size(C.byref(big), 8, 16, 0) == 0
    if not torch.cuda.is_available():
        assert call() == CUDA                     # every argument valid: the call reaches the runtime
        assert call(bth=0x50000) == CUDA          # with per-head block tables as well


def test_copy_async_checks(lib):
    """The staging copy refuses NULL, misaligned and odd-sized arguments on the
    host, does nothing for zero bytes, and never launches for pointers the
    runtime cannot vouch for (here: no device at all)."""
    fn = lib.dsa_copy_async
    assert fn(None, 0x1000, 16, None) == INVALID
    assert fn(0x1000, None, 16, None) == INVALID
    assert fn(0x1008, 0x2000, 16, None) == INVALID
    assert fn(0x1000, 0x2008, 16, None) == INVALID
    assert fn(0x1000, 0x2000, 24, None) == INVALID
    assert fn(0x1000, 0x2000, 0, None) == DSA_OK
    import torch
    if not torch.cuda.is_available():
        assert fn(0x1000, 0x2000, 16, None) != DSA_OK
