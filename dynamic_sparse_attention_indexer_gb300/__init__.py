"""Dynamic sparse attention (DSA) hot path for GB300 (sm_103a).

A thin Python face on the C ABI of ``include/dsa.h``: it only marshals torch
tensors (device memory) and the current CUDA stream into the library's calls.
Every step runs in the library's CUDA kernels; there is no Python or CPU
fallback, and an op raises if the library cannot be loaded.

The method is the one of the article
"国产AI芯片完成前沿大模型Day-0适配:稀疏注意力与混合精度推理全解析", section 2:
an int8 indexer scores every causal key (§2.1), a top-k picks positions with a
vision prefix always attended (§2.1, §2.4), the rows come from a paged KV
cache (§2.2), and GQA attention runs over them only (§2.3).
"""
from __future__ import annotations

import ctypes as C
import math

import torch

from . import _abi

MODE_DECODE, MODE_PREFILL = 0, 1
OUT_BF16, OUT_F32 = 0, 1
OP_INDEX_SCORES, OP_TOPK_SELECT, OP_SPARSE_ATTN, OP_DECODE_STEP, OP_PREFILL_STEP = range(5)
BLOCK_SIZE, HEAD_DIM, IDX_DIM = 64, 128, 64


class DSAError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{status_string(status)}: {message}")


def lib():
    return _abi.load()


def status_string(s: int) -> str:
    return lib().dsa_status_string(s).decode()


def _check(status: int):
    if status != 0:
        raise DSAError(status, lib().dsa_last_error_message().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device=None):
    # The raw handle of the current stream without building a Stream object
    # (a few microseconds less per call); the public accessor where it is missing.
    if _raw_stream is not None:
        idx = None if device is None else torch.device(device).index
        return C.c_void_p(_raw_stream(torch.cuda.current_device() if idx is None else idx))
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def kv_cache_adjacent(num_blocks: int, num_kv_heads: int, device):
    """An uninitialised paged K/V cache in the adjacent layout: one bf16 array
    [num_blocks][64][2][Hkv][128] (the K and V of a slot one contiguous piece);
    returns the (k_cache, v_cache) views [num_blocks][64][Hkv][128] of it."""
    kv = torch.empty((num_blocks, BLOCK_SIZE, 2, num_kv_heads, HEAD_DIM), dtype=torch.bfloat16, device=device)
    return kv[:, :, 0], kv[:, :, 1]


class PagedKV:
    """The paged cache: k_cache/v_cache bf16 [num_blocks][64][Hkv][128] (two
    arrays, or the two views of kv_cache_adjacent), idx_cache int8
    [num_blocks][64][64], block_table int32 [B][max_blocks], context_lens int32
    [B] (all on one CUDA device)."""

    def __init__(self, k_cache, v_cache, idx_cache, block_table, context_lens, max_context_len=None):
        self.k_cache, self.v_cache, self.idx_cache = k_cache, v_cache, idx_cache
        self.block_table, self.context_lens = block_table, context_lens
        if max_context_len is None:
            max_context_len = int(context_lens.max().item())
        self.max_context_len = int(max_context_len)
        self.num_kv_heads = int(k_cache.shape[2])
        self.batch = int(block_table.shape[0])
        # Rows of consecutive slots are kv_row_stride values apart in both arrays.
        row = int(k_cache.stride(1))
        for t in (k_cache, v_cache):
            if t.stride(3) != 1 or t.stride(2) != HEAD_DIM or t.stride(1) != row or t.stride(0) != BLOCK_SIZE * row:
                raise ValueError("k_cache / v_cache: each slot's row must hold its KV heads contiguously, "
                                 "slots evenly spaced and the same in both arrays")
        self.struct = _abi.PagedKV(
            _ptr(k_cache), _ptr(v_cache), _ptr(idx_cache), _ptr(block_table), _ptr(context_lens),
            int(k_cache.shape[0]), int(k_cache.shape[1]), self.num_kv_heads, int(k_cache.shape[3]),
            int(idx_cache.shape[-1]), int(block_table.shape[1]), self.batch, self.max_context_len, row)

    @property
    def ref(self):
        return C.byref(self.struct)


def query_set(mode: int, n_q: int, seq: int = 0, pos0: int = 0):
    return _abi.QuerySet(mode, n_q, seq, pos0)


def decode_queries(kv: PagedKV):
    return query_set(MODE_DECODE, kv.batch)


def workspace_size(op: int, kv: PagedKV, qs, k: int, num_q_heads: int, prefix_len: int) -> int:
    return int(lib().dsa_workspace_size(op, kv.ref, C.byref(qs), k, num_q_heads, prefix_len))


def make_workspace(nbytes: int, device) -> torch.Tensor | None:
    """A zeroed workspace buffer (None when no workspace is needed)."""
    if nbytes == 0:
        return None
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _check(lib().dsa_workspace_init(_ptr(ws), nbytes, _stream(ws.device)))
    return ws


def _ws(ws):
    return (_ptr(ws), 0 if ws is None else ws.numel())


def copy_async(dst, src):
    """Staging copy by a kernel on the current stream of the CUDA side: dst and
    src contiguous tensors of the same byte size, each a CUDA tensor or a
    pinned CPU tensor (see dsa_copy_async)."""
    nb = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nb or not dst.is_contiguous() or not src.is_contiguous():
        raise ValueError("copy_async: dst and src must be contiguous and of the same size in bytes")
    device = dst.device if dst.is_cuda else src.device
    if not device.type == "cuda":
        raise ValueError("copy_async: one side must be a CUDA tensor")
    _check(lib().dsa_copy_async(_ptr(dst), _ptr(src), nb, _stream(device)))


def kv_write(kv: PagedKV, slot_mapping, k, v, idx_k):
    _check(lib().dsa_kv_write(kv.ref, _ptr(slot_mapping), int(slot_mapping.numel()), _ptr(k), _ptr(v),
                              _ptr(idx_k), _stream(kv.k_cache.device)))


def kv_write_heads(kv: PagedKV, slot_mapping_heads, k, v, idx_k):
    """Per-head cache write: slot_mapping_heads int32 [ntok][Hkv], k / v bf16
    [ntok][Hkv][128], idx_k int8 [ntok][Hkv][64] (indexer cache
    [blocks][Hkv][64][64])."""
    _check(lib().dsa_kv_write_heads(kv.ref, _ptr(slot_mapping_heads), int(slot_mapping_heads.shape[0]), _ptr(k),
                                    _ptr(v), _ptr(idx_k), _stream(kv.k_cache.device)))


def index_scores(kv: PagedKV, qs, q_idx, prefix_len: int, scores, ws=None):
    p, n = _ws(ws)
    _check(lib().dsa_index_scores(kv.ref, C.byref(qs), _ptr(q_idx), prefix_len, _ptr(scores),
                                  int(scores.stride(0)), p, n, _stream(scores.device)))


def topk_select(kv: PagedKV, qs, scores, prefix_len: int, k: int, idx, n_sel, ws=None):
    p, n = _ws(ws)
    _check(lib().dsa_topk_select(kv.ref, C.byref(qs), _ptr(scores), int(scores.stride(0)), prefix_len, k,
                                 _ptr(idx), _ptr(n_sel), p, n, _stream(scores.device)))


def kv_gather(kv: PagedKV, qs, idx, n_sel, k: int, prefix_len: int, k_out, v_out):
    _check(lib().dsa_kv_gather(kv.ref, C.byref(qs), _ptr(idx), _ptr(n_sel), k, prefix_len, _ptr(k_out),
                               _ptr(v_out), _stream(k_out.device)))


def _out_dtype(out):
    return OUT_F32 if out.dtype == torch.float32 else OUT_BF16


def sparse_attn_decode(kv: PagedKV, q, idx, n_sel, k: int, prefix_len: int, out, lse=None, ws=None,
                       softmax_scale: float | None = None):
    scale = 1.0 / math.sqrt(HEAD_DIM) if softmax_scale is None else softmax_scale
    p, n = _ws(ws)
    _check(lib().dsa_sparse_attn_decode(kv.ref, _ptr(q), int(q.shape[1]), _ptr(idx), _ptr(n_sel), k, prefix_len,
                                        scale, _ptr(out), _out_dtype(out), _ptr(lse), p, n, _stream(q.device)))


def sparse_attn_prefill(kv: PagedKV, qs, q, idx, n_sel, k: int, prefix_len: int, out, lse=None, ws=None,
                        softmax_scale: float | None = None, n_dense: int | None = None):
    """Prefill attention.  n_dense: queries [0, n_dense) by the dense masked
    pass, the rest gathered; None takes the library's automatic split."""
    scale = 1.0 / math.sqrt(HEAD_DIM) if softmax_scale is None else softmax_scale
    p, n = _ws(ws)
    if n_dense is None:
        _check(lib().dsa_sparse_attn_prefill(kv.ref, C.byref(qs), _ptr(q), int(q.shape[1]), _ptr(idx), _ptr(n_sel),
                                             k, prefix_len, scale, _ptr(out), _out_dtype(out), _ptr(lse), p, n,
                                             _stream(q.device)))
    else:
        _check(lib().dsa_sparse_attn_prefill_split(kv.ref, C.byref(qs), _ptr(q), int(q.shape[1]), _ptr(idx),
                                                   _ptr(n_sel), k, prefix_len, scale, int(n_dense), _ptr(out),
                                                   _out_dtype(out), _ptr(lse), p, n, _stream(q.device)))


def prefill_dense_queries(kv: PagedKV, qs, k: int, num_q_heads: int, prefix_len: int) -> int:
    """The automatic split: how many leading queries of qs go to the dense pass."""
    return int(lib().dsa_prefill_dense_queries(kv.ref, C.byref(qs), k, num_q_heads, prefix_len))


def prefill_attn_workspace_size(kv: PagedKV, qs, k: int, num_q_heads: int, prefix_len: int, n_dense: int) -> int:
    return int(lib().dsa_prefill_attn_workspace_size(kv.ref, C.byref(qs), k, num_q_heads, prefix_len, n_dense))


def heads_workspace_size(kv: PagedKV, num_q_heads: int, k: int, prefix_len: int) -> int:
    return int(lib().dsa_heads_workspace_size(kv.ref, num_q_heads, k, prefix_len))


def prefill_step(kv: PagedKV, qs, q, q_idx, prefix_len: int, k: int, scores, idx, n_sel, out, lse=None, ws=None,
                 softmax_scale: float | None = None):
    """Scores, top-k and attention of one prefill chunk in one call (the
    automatic dense / gathered split); ws: prefill_attn_workspace_size(kv, qs,
    k, num_q_heads, prefix_len) bytes."""
    scale = 1.0 / math.sqrt(HEAD_DIM) if softmax_scale is None else softmax_scale
    p, n = _ws(ws)
    _check(lib().dsa_prefill_step(kv.ref, C.byref(qs), _ptr(q), _ptr(q_idx), int(q.shape[1]), prefix_len, k, scale,
                                  _ptr(scores), int(scores.stride(0)), _ptr(idx), _ptr(n_sel), _ptr(out),
                                  _out_dtype(out), _ptr(lse), p, n, _stream(q.device)))


def decode_step_heads(kv: PagedKV, q, q_idx, prefix_len: int, k: int, scores, idx, n_sel, out, lse=None, ws=None,
                      softmax_scale: float | None = None, block_table_heads=None):
    """The decode step with one indexer head per KV head: q_idx [B][Hkv][64],
    the indexer cache [blocks][Hkv][64][64], scores [B * Hkv][ld], idx
    [B][Hkv][k], n_sel [B][Hkv]; block_table_heads: int32 [Hkv][B][max_blocks],
    one block table per KV head, or None for the shared one."""
    scale = 1.0 / math.sqrt(HEAD_DIM) if softmax_scale is None else softmax_scale
    p, n = _ws(ws)
    if block_table_heads is not None:
        hkv, B, mb = kv.num_kv_heads, kv.batch, int(kv.block_table.shape[1])
        if (tuple(block_table_heads.shape) != (hkv, B, mb) or block_table_heads.dtype != kv.block_table.dtype
                or not block_table_heads.is_contiguous() or block_table_heads.device != kv.block_table.device):
            raise ValueError("block_table_heads must be a contiguous int32 [num_kv_heads][batch][max_blocks] tensor "
                             "on the cache's device")
    _check(lib().dsa_decode_step_heads(kv.ref, _ptr(q), _ptr(q_idx), _ptr(block_table_heads), int(q.shape[1]),
                                       prefix_len, k, scale,
                                       _ptr(scores), int(scores.stride(0)), _ptr(idx), _ptr(n_sel), _ptr(out),
                                       _out_dtype(out), _ptr(lse), p, n, _stream(q.device)))


def prefill_select(kv: PagedKV, qs, q_idx, prefix_len: int, k: int, idx, n_sel):
    """Prefill scores and top-k in one call, the scores never materialised."""
    _check(lib().dsa_prefill_select(kv.ref, C.byref(qs), _ptr(q_idx), prefix_len, k, _ptr(idx), _ptr(n_sel),
                                    _stream(q_idx.device)))


def window_workspace_size(kv: PagedKV, num_q_heads: int, window: int) -> int:
    return int(lib().dsa_window_workspace_size(kv.ref, num_q_heads, window))


def window_attn_decode(kv: PagedKV, q, window: int, out, lse=None, ws=None, softmax_scale: float | None = None):
    """Local sliding-window attention of each sequence's newest token over its
    last `window` positions."""
    scale = 1.0 / math.sqrt(HEAD_DIM) if softmax_scale is None else softmax_scale
    p, n = _ws(ws)
    _check(lib().dsa_window_attn_decode(kv.ref, _ptr(q), int(q.shape[1]), int(window), scale, _ptr(out),
                                        _out_dtype(out), _ptr(lse), p, n, _stream(q.device)))


def window_attn_prefill(kv: PagedKV, qs, q, window: int, out, lse=None, softmax_scale: float | None = None):
    """Local sliding-window attention of the prefill queries of qs."""
    scale = 1.0 / math.sqrt(HEAD_DIM) if softmax_scale is None else softmax_scale
    _check(lib().dsa_window_attn_prefill(kv.ref, C.byref(qs), _ptr(q), int(q.shape[1]), int(window), scale,
                                         _ptr(out), _out_dtype(out), _ptr(lse), _stream(q.device)))


def decode_step(kv: PagedKV, q, q_idx, prefix_len: int, k: int, scores, idx, n_sel, out, lse=None, ws=None,
                softmax_scale: float | None = None):
    scale = 1.0 / math.sqrt(HEAD_DIM) if softmax_scale is None else softmax_scale
    p, n = _ws(ws)
    _check(lib().dsa_decode_step(kv.ref, _ptr(q), _ptr(q_idx), int(q.shape[1]), prefix_len, k, scale,
                                 _ptr(scores), int(scores.stride(0)), _ptr(idx), _ptr(n_sel), _ptr(out),
                                 _out_dtype(out), _ptr(lse), p, n, _stream(q.device)))


def check_device_status(device=None) -> int:
    """Synchronise and read-and-clear the device status word (0 = OK)."""
    code = C.c_int32(0)
    _check(lib().dsa_check_device_status(_stream(device), C.byref(code)))
    return int(code.value)


class BlockAllocator:
    """Host free list of KV block ids (lowest first)."""

    def __init__(self, num_blocks: int):
        h = C.c_void_p()
        _check(lib().dsa_kv_alloc_create(num_blocks, C.byref(h)))
        self._h = h

    def alloc(self, n: int) -> list[int]:
        buf = (C.c_int32 * max(n, 1))()
        _check(lib().dsa_kv_alloc_blocks(self._h, n, buf))
        return list(buf[:n])

    def free(self, ids):
        buf = (C.c_int32 * max(len(ids), 1))(*ids)
        _check(lib().dsa_kv_free_blocks(self._h, buf, len(ids)))

    @property
    def num_free(self) -> int:
        return int(lib().dsa_kv_alloc_num_free(self._h))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib().dsa_kv_alloc_destroy(h)
            self._h = None
