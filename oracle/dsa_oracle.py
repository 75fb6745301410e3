"""Plain CPU oracle for the dynamic sparse attention (DSA) hot path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline / reference legs of ``bench.py`` may
import this module.  The CUDA library never calls it and shares no code with
it: no kernels, headers, helpers or tables.

Every function is the slow, obviously correct definition of one step, in
float64 / int64 numpy.  The method follows the article
"国产AI芯片完成前沿大模型Day-0适配:稀疏注意力与混合精度推理全解析"
(ruibaoantu.com), section 2 ("稀疏注意力DSA适配的四大攻坚点"); section numbers
below refer to that article.  Where the article leaves a step open, the
reading taken is stated in the function that takes it.

Data layout (shared with the CUDA path only through the seeded generator):
  k_cache, v_cache : [num_blocks][64][Hkv][d]   (blocks of 64 consecutive positions;
                     within a block, position-major, the KV heads of a position adjacent)
  idx_cache        : [num_blocks][64][D]        int8 indexer keys
  block_table      : [B][max_blocks]            int32, block id of positions [64j, 64j+64)

Pins (tests/test_oracle_pins.py): closed forms for the scores, all-tie and
monotone-score top-k cases, brute-force subset enumeration of the top-k,
the vision-prefix invariant, dense causal attention against PyTorch's
scaled_dot_product_attention when k covers the whole context, and
single-row / constant-V / identical-key attention closed forms.
"""
from __future__ import annotations

import numpy as np

BLOCK = 64  # positions per KV block (section 2.2: fixed-size blocks, e.g. 64 x 128)


# --------------------------------------------------------------------------
# Row fetch through the block table (section 2.2)
# --------------------------------------------------------------------------
def fetch_rows(cache: np.ndarray, bt_row: np.ndarray, positions: np.ndarray,
               head: int | None = None) -> np.ndarray:
    """Rows of a paged cache at absolute ``positions`` of one sequence.

    Section 2.2: the cache is cut into fixed blocks, each holding the values
    of consecutive positions; position t lives in block ``bt_row[t // 64]``
    at row ``t % 64``.  With ``head`` given the cache is [blk][64][Hkv][d]
    (K or V: one block row holds every KV head of its position), otherwise
    [blk][64][D] (indexer keys).
    """
    positions = np.asarray(positions, dtype=np.int64)
    blocks = np.asarray(bt_row, dtype=np.int64)[positions // BLOCK]
    rows = positions % BLOCK
    if head is None:
        return cache[blocks, rows]
    return cache[blocks, rows, head]


# --------------------------------------------------------------------------
# Step 1: index scores (section 2.1)
# --------------------------------------------------------------------------
def candidate_positions(prefix_len: int, pos: int) -> np.ndarray:
    """Causal key positions that take part in index selection: [P, pos].

    Section 2.4: the vision prefix [0, P) never takes part in selection.
    Causality: a query at position ``pos`` sees keys 0..pos inclusive.
    """
    return np.arange(prefix_len, pos + 1, dtype=np.int64)


def index_scores(q_idx: np.ndarray, idx_cache: np.ndarray, bt_row: np.ndarray,
                 prefix_len: int, pos: int) -> tuple[np.ndarray, np.ndarray]:
    """Indexer score of every candidate key of one query.

    Section 2.1 scores query against key before attention ("初步相似度打分").
    Reading: the plain integer dot product of the int8 indexer query with the
    int8 indexer key, exact in int64 (no activation, no weights, no scale).
    Returns (positions, scores).
    """
    ts = candidate_positions(prefix_len, pos)
    keys = fetch_rows(idx_cache, bt_row, ts).astype(np.int64)
    return ts, keys @ np.asarray(q_idx, dtype=np.int64)


# --------------------------------------------------------------------------
# Step 2: top-k selection with the vision prefix forced in (sections 2.1, 2.4)
# --------------------------------------------------------------------------
def topk_select(ts: np.ndarray, scores: np.ndarray, k: int) -> tuple[np.ndarray, int]:
    """The k best candidates, ascending by position, padded with -1 to length k.

    Order: higher score first, and among equal scores the lower position
    first; the first k of that order are kept (all of them when there are at
    most k).  Returns (idx[k], n_sel).  A full sort, on purpose: the GPU
    takes a different route (histogram threshold + ordered compaction).
    """
    ts = np.asarray(ts, dtype=np.int64)
    scores = np.asarray(scores, dtype=np.int64)
    if ts.size <= k:
        chosen = ts
    else:
        order = np.lexsort((ts, -scores))  # primary: -score, secondary: position
        chosen = ts[order[:k]]
    chosen = np.sort(chosen)
    out = np.full(k, -1, dtype=np.int64)
    out[:chosen.size] = chosen
    return out, int(chosen.size)


def attended_positions(prefix_len: int, pos: int, idx: np.ndarray, n_sel: int) -> np.ndarray:
    """The attended set S: the causal part of the prefix, then the selection.

    Section 2.4: the vision prefix is always fully attended.  Reading: only
    its causal part [0, min(P, pos+1)) is, and it does not use the k budget.
    """
    prefix = np.arange(min(prefix_len, pos + 1), dtype=np.int64)
    return np.concatenate([prefix, np.asarray(idx[:n_sel], dtype=np.int64)])


# --------------------------------------------------------------------------
# Step 3: gather (section 2.2, "先收集、后计算")
# --------------------------------------------------------------------------
def kv_gather(k_cache, v_cache, bt_row, positions, num_kv_heads, rows_out):
    """K and V rows of ``positions`` copied into contiguous [Hkv][rows_out][d]
    buffers, in the order given; rows past ``len(positions)`` are zero."""
    d = k_cache.shape[-1]
    ko = np.zeros((num_kv_heads, rows_out, d), dtype=k_cache.dtype)
    vo = np.zeros((num_kv_heads, rows_out, d), dtype=v_cache.dtype)
    for g in range(num_kv_heads):
        ko[g, :len(positions)] = fetch_rows(k_cache, bt_row, positions, head=g)
        vo[g, :len(positions)] = fetch_rows(v_cache, bt_row, positions, head=g)
    return ko, vo


# --------------------------------------------------------------------------
# Step 4: attention over the attended set (section 2.3)
# --------------------------------------------------------------------------
def softmax_attention(q: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray,
                      scale: float) -> tuple[np.ndarray, np.ndarray]:
    """softmax(scale * q k^T) v for a group of query heads sharing one K/V set.

    q: [G][d], k_rows/v_rows: [R][d] (R >= 1).  Returns (out [G][d], lse [G])
    with lse the natural log of the softmax denominator including the max.
    """
    q = np.asarray(q, dtype=np.float64)
    kr = np.asarray(k_rows, dtype=np.float64)
    vr = np.asarray(v_rows, dtype=np.float64)
    z = scale * (q @ kr.T)
    m = z.max(axis=1, keepdims=True)
    w = np.exp(z - m)
    l = w.sum(axis=1)
    out = (w @ vr) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return out, lse


def sparse_gqa_attention(q_heads: np.ndarray, k_cache, v_cache, bt_row,
                         positions: np.ndarray, num_kv_heads: int,
                         scale: float) -> tuple[np.ndarray, np.ndarray]:
    """GQA attention of one query token over the attended set.

    q_heads: [Hq][d].  Query head h reads KV head h // (Hq / Hkv); all heads
    share the one selection made for the token.
    """
    hq, d = q_heads.shape
    group = hq // num_kv_heads
    out = np.zeros((hq, d), dtype=np.float64)
    lse = np.zeros(hq, dtype=np.float64)
    for g in range(num_kv_heads):
        kr = fetch_rows(k_cache, bt_row, positions, head=g)
        vr = fetch_rows(v_cache, bt_row, positions, head=g)
        o, s = softmax_attention(q_heads[g * group:(g + 1) * group], kr, vr, scale)
        out[g * group:(g + 1) * group] = o
        lse[g * group:(g + 1) * group] = s
    return out, lse


# --------------------------------------------------------------------------
# One query token, all four steps
# --------------------------------------------------------------------------
def dsa_query(q_heads, q_idx, k_cache, v_cache, idx_cache, bt_row, pos: int,
              prefix_len: int, k: int, num_kv_heads: int, scale: float) -> dict:
    """Index, select, gather and attend for one query token at ``pos``."""
    ts, s = index_scores(q_idx, idx_cache, bt_row, prefix_len, pos)
    idx, n_sel = topk_select(ts, s, k)
    positions = attended_positions(prefix_len, pos, idx, n_sel)
    out, lse = sparse_gqa_attention(q_heads, k_cache, v_cache, bt_row, positions,
                                    num_kv_heads, scale)
    return {"positions": ts, "scores": s, "idx": idx, "n_sel": n_sel,
            "attended": positions, "out": out, "lse": lse}


def decode_query(w: dict, b: int, scale: float | None = None) -> dict:
    """Decode: sequence b's newest token sits at pos = L_b - 1 (its own K/V
    and indexer key are already in the cache)."""
    d = w["k_cache"].shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    pos = int(w["context_lens"][b]) - 1
    return dsa_query(w["q"][b], w["q_idx"][b], w["k_cache"], w["v_cache"], w["idx_cache"],
                     w["block_table"][b], pos, int(w["prefix_len"]), int(w["k"]),
                     int(w["num_kv_heads"]), scale)


def prefill_query(w: dict, i: int, scale: float | None = None) -> dict:
    """Prefill: query i of sequence ``seq`` sits at pos = pos0 + i and sees
    keys [0, pos] (causal, also inside the prefix)."""
    d = w["k_cache"].shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    seq = int(w["seq"])
    pos = int(w["pos0"]) + i
    return dsa_query(w["q"][i], w["q_idx"][i], w["k_cache"], w["v_cache"], w["idx_cache"],
                     w["block_table"][seq], pos, int(w["prefix_len"]), int(w["k"]),
                     int(w["num_kv_heads"]), scale)


# --------------------------------------------------------------------------
# Per-KV-head indexer (section 2.4, "per head" state; the next row of the scope)
# --------------------------------------------------------------------------
def decode_query_heads(w: dict, b: int, scale: float | None = None) -> dict:
    """Decode with one indexer head per KV head.  Reading taken (the article
    keeps the KV state per head, section 2.4, and does not say whether the
    selection is per head): KV head g has its own indexer query q_idx[b][g] and
    keys idx_cache[block][g][row], scores, selects its own top-k, and the query
    heads of group g attend the prefix plus that selection.

    w["idx_cache"]: [num_blocks][Hkv][64][D]; w["q_idx"]: [B][Hkv][D].

    With w["block_table_heads"] ([Hkv][B][max_blocks], the per-head block
    bitmaps of the KV allocator, section 2.4) head g finds its positions
    through its own table: its indexer keys, K and V rows are the head-g
    slices of the blocks that table names, so a physical block can hold
    different positions for different heads."""
    d = w["k_cache"].shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    hkv = int(w["num_kv_heads"])
    q_heads = w["q"][b]
    group = q_heads.shape[0] // hkv
    pos = int(w["context_lens"][b]) - 1
    tables = w.get("block_table_heads")
    P, k = int(w["prefix_len"]), int(w["k"])
    res = {"idx": [], "n_sel": [], "scores": [], "attended": [],
           "out": np.zeros(q_heads.shape, dtype=np.float64), "lse": np.zeros(q_heads.shape[0], dtype=np.float64)}
    for g in range(hkv):
        bt_row = w["block_table"][b] if tables is None else tables[g][b]
        ts, s = index_scores(w["q_idx"][b][g], w["idx_cache"][:, g], bt_row, P, pos)
        idx, n_sel = topk_select(ts, s, k)
        positions = attended_positions(P, pos, idx, n_sel)
        kr = fetch_rows(w["k_cache"], bt_row, positions, head=g)
        vr = fetch_rows(w["v_cache"], bt_row, positions, head=g)
        o, l = softmax_attention(q_heads[g * group:(g + 1) * group], kr, vr, scale)
        res["out"][g * group:(g + 1) * group] = o
        res["lse"][g * group:(g + 1) * group] = l
        res["idx"].append(idx)
        res["n_sel"].append(n_sel)
        res["scores"].append(s)
        res["attended"].append(positions)
    return res


# --------------------------------------------------------------------------
# Local sliding-window attention, the hybrid attention's local sibling
# ("Qwen3.5在摩尔线程MTT S5000上的原生推理优化实践", section 2.3)
# --------------------------------------------------------------------------
def window_positions(pos: int, window: int) -> np.ndarray:
    """Reading taken (the page names the sub-module, "局部滑动窗口注意力", and
    gives no definition): a causal window of ``window`` positions ending at the
    query's own, [max(0, pos - window + 1), pos]; no prefix, no selection."""
    return np.arange(max(0, pos - window + 1), pos + 1, dtype=np.int64)


def window_query(w: dict, pos: int, q_heads: np.ndarray, seq: int, window: int,
                 scale: float | None = None) -> dict:
    """Window attention of one query token at ``pos`` of sequence ``seq``."""
    d = w["k_cache"].shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    positions = window_positions(pos, window)
    out, lse = sparse_gqa_attention(q_heads, w["k_cache"], w["v_cache"], w["block_table"][seq],
                                    positions, int(w["num_kv_heads"]), scale)
    return {"attended": positions, "out": out, "lse": lse}


# --------------------------------------------------------------------------
# Cache write and block allocation (section 2.4, KDA)
# --------------------------------------------------------------------------
def kv_write_heads(k_cache, v_cache, idx_cache, slot_mapping_heads, k_new, v_new, idx_new):
    """Cache write with one slot per (token, KV head), the write side of the
    per-head block bitmaps (section 2.4: heads must not overwrite one
    another's blocks): token j's head-h K, V and indexer key go to the head-h
    slice of slot slot_mapping_heads[j][h] only.  k_new, v_new: [ntok][Hkv][d];
    idx_new: [ntok][Hkv][D]; idx_cache: [num_blocks][Hkv][64][D].  Returns
    updated copies (inputs untouched)."""
    kc, vc, ic = k_cache.copy(), v_cache.copy(), idx_cache.copy()
    slots = np.asarray(slot_mapping_heads, dtype=np.int64)
    for j in range(slots.shape[0]):
        for h in range(slots.shape[1]):
            blk, row = divmod(int(slots[j, h]), BLOCK)
            kc[blk, row, h] = k_new[j, h]
            vc[blk, row, h] = v_new[j, h]
            ic[blk, h, row] = idx_new[j, h]
    return kc, vc, ic


def kv_write(k_cache, v_cache, idx_cache, slot_mapping, k_new, v_new, idx_new):
    """Scatter new tokens into their slots; slot = block_id * 64 + row.
    k_new, v_new: [ntok][Hkv][d]; idx_new: [ntok][D].  Returns updated copies
    (inputs untouched)."""
    kc, vc, ic = k_cache.copy(), v_cache.copy(), idx_cache.copy()
    for j, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        blk, row = divmod(int(slot), BLOCK)
        kc[blk, row] = k_new[j]
        vc[blk, row] = v_new[j]
        ic[blk, row] = idx_new[j]
    return kc, vc, ic
