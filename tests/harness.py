"""GPU-vs-oracle plumbing for the parity tests: run the library on a seeded
workload, run the oracle on the same inputs, compare.  Data movement only
(copies, block remapping); all arithmetic is in the library or the oracle."""
from __future__ import annotations

import numpy as np
import torch

import dynamic_sparse_attention_indexer_gb300 as dsa
import oracle.dsa_oracle as O
import synth

# Attention outputs: elementwise |gpu - ref| <= ATOL + RTOL * |ref|
# (bf16 inputs, fp32 accumulation, P rounded to bf16 for the P.V product).
ATOL, RTOL = 2e-3, 1e-2


def on(w: dict, device) -> dict:
    """The workload on `device`; an adjacent-layout cache moves as its one
    array and gets its k_cache / v_cache views back."""
    out = {k: (v.to(device) if isinstance(v, torch.Tensor) and k not in ("k_cache", "v_cache") else v)
           for k, v in w.items()}
    if "kv" in w:
        out["k_cache"], out["v_cache"] = out["kv"][:, :, 0], out["kv"][:, :, 1]
    else:
        out["k_cache"], out["v_cache"] = w["k_cache"].to(device), w["v_cache"].to(device)
    return out


def paged_kv(w: dict) -> dsa.PagedKV:
    return dsa.PagedKV(w["k_cache"], w["v_cache"], w["idx_cache"], w["block_table"], w["context_lens"],
                       w["max_context_len"])


def round4(x: int) -> int:
    return (x + 3) // 4 * 4


def run_decode_step(w: dict, out_dtype=torch.bfloat16, split_api=False) -> dict:
    """The fused decode step (or the four separate calls) on device tensors."""
    dev = w["q"].device
    kv = paged_kv(w)
    B, k, P, hq = kv.batch, int(w["k"]), int(w["prefix_len"]), int(w["num_q_heads"])
    ld = round4(int(w["max_context_len"]))
    scores = torch.zeros((B, ld), dtype=torch.int32, device=dev)
    idx = torch.empty((B, k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, hq, 128), dtype=out_dtype, device=dev)
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev)
    qs = dsa.decode_queries(kv)
    ws = dsa.make_workspace(dsa.workspace_size(dsa.OP_DECODE_STEP, kv, qs, k, hq, P), dev)
    if split_api:
        dsa.index_scores(kv, qs, w["q_idx"], P, scores)
        dsa.topk_select(kv, qs, scores, P, k, idx, n_sel, ws)
        dsa.sparse_attn_decode(kv, w["q"], idx, n_sel, k, P, out, lse, ws)
    else:
        dsa.decode_step(kv, w["q"], w["q_idx"], P, k, scores, idx, n_sel, out, lse, ws)
    status = dsa.check_device_status(dev)
    assert status == 0, f"device status {status}"
    return {"scores": scores, "idx": idx, "n_sel": n_sel, "out": out, "lse": lse, "ws": ws}


def assert_close(gpu, ref, what: str):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; max abs err "
                           f"{err.max():.3e}, worst at ref={ref.flat[np.argmax(err - bound)]:.4f}")


def check_decode_against_oracle(wn: dict, res: dict, seqs=None, check_scores=True):
    """Compare every sequence (or `seqs`) of a small decode workload with the
    full oracle.  wn: numpy workload; res: run_decode_step output."""
    P = int(wn["prefix_len"])
    B = int(wn["spec"].batch)
    idx = res["idx"].cpu().numpy()
    n_sel = res["n_sel"].cpu().numpy()
    out = res["out"].float().cpu().numpy()
    lse = res["lse"].cpu().numpy()
    scores = res["scores"].cpu().numpy()
    for b in (range(B) if seqs is None else seqs):
        r = O.decode_query(wn, b)
        L = int(wn["context_lens"][b])
        if check_scores:
            assert np.array_equal(scores[b, P:L], r["scores"]), f"scores of sequence {b}"
        assert int(n_sel[b]) == r["n_sel"], f"n_sel of sequence {b}: {n_sel[b]} vs {r['n_sel']}"
        assert np.array_equal(idx[b], r["idx"]), f"idx of sequence {b}"
        assert_close(out[b], r["out"], f"out of sequence {b}")
        assert_close(lse[b], r["lse"], f"lse of sequence {b}")


# ------------------------------------------------- full-size, sampled parity ---
def _compact_blocks(w: dict, b: int, positions: np.ndarray, cache: str, head=None):
    """Copy the blocks holding `positions` of sequence b into a small CPU cache
    with its own block table (same positions, fewer blocks)."""
    bt = w["block_table"][b].cpu().numpy().astype(np.int64)
    jblocks = np.unique(positions // O.BLOCK)
    ids = torch.as_tensor(bt[jblocks], device=w[cache].device)
    src = w[cache].index_select(0, ids)
    if head is not None:
        src = src[:, :, head:head + 1]  # [blk][64][Hkv][d]: keep one KV head
    local_bt = np.full(bt.shape, -1, dtype=np.int64)
    local_bt[jblocks] = np.arange(len(jblocks))
    t = src.cpu()
    arr = t.to(torch.float64).numpy() if t.dtype == torch.bfloat16 else t.numpy().astype(np.int64)
    return arr, local_bt


def oracle_decode_sampled(w: dict, b: int, heads_kv, k: int, P: int):
    """Oracle result of decode sequence b of a device-resident workload, for
    the KV heads in `heads_kv` only."""
    L = int(w["context_lens"][b].item())
    pos = L - 1
    cand = O.candidate_positions(P, pos)
    icache, ibt = _compact_blocks(w, b, cand, "idx_cache")
    q_idx = w["q_idx"][b].cpu().numpy().astype(np.int64)
    ts, s = O.index_scores(q_idx, icache, ibt, P, pos)
    idx, n_sel = O.topk_select(ts, s, k)
    att = O.attended_positions(P, pos, idx, n_sel)
    hq, hkv = int(w["num_q_heads"]), int(w["num_kv_heads"])
    G = hq // hkv
    scale = 1.0 / np.sqrt(128)
    heads = {}
    for g in heads_kv:
        kc, kbt = _compact_blocks(w, b, att, "k_cache", head=g)
        vc, _ = _compact_blocks(w, b, att, "v_cache", head=g)
        q = w["q"][b, g * G:(g + 1) * G].cpu().to(torch.float64).numpy()
        out, lse = O.sparse_gqa_attention(q, kc, vc, kbt, att, 1, scale)
        heads[g] = (out, lse)
    return {"scores": s, "idx": idx, "n_sel": n_sel, "heads": heads}


def oracle_indices_all(w: dict, k: int, P: int, rows=None):
    """Oracle scores and selection of every decode sequence (or, with `rows`,
    of those prefill query rows) of a device-resident workload: the indexer
    cache, block table and indexer queries are read back once."""
    icache = w["idx_cache"].cpu().numpy()  # int8; the oracle widens the rows it reads
    bt = w["block_table"].cpu().numpy().astype(np.int64)
    q_idx = w["q_idx"].cpu().numpy().astype(np.int64)
    res = {}
    if rows is None:  # decode: sequence b's newest token
        lens = w["context_lens"].cpu().numpy()
        items = [(b, b, int(lens[b]) - 1) for b in range(len(lens))]
    else:             # prefill: query row i of sequence w["seq"]
        items = [(int(i), int(w["seq"]), int(w["pos0"]) + int(i)) for i in rows]
    for key, seq, pos in items:
        ts, s = O.index_scores(q_idx[key], icache, bt[seq], P, pos)
        idx, n_sel = O.topk_select(ts, s, k)
        res[key] = {"scores": s, "idx": idx, "n_sel": n_sel, "pos": pos}
    return res


def run_prefill(w: dict, out_dtype=torch.bfloat16, n_dense=None) -> dict:
    """index_scores -> topk_select -> sparse_attn_prefill for the queries of
    sequence w["seq"] at positions pos0 .. pos0 + T - 1.  n_dense: queries
    [0, n_dense) by the dense masked pass, the rest gathered (None: the
    library's automatic split)."""
    dev = w["q"].device
    kv = paged_kv(w)
    T, k, P, hq = int(w["num_queries"]), int(w["k"]), int(w["prefix_len"]), int(w["num_q_heads"])
    qs = dsa.query_set(dsa.MODE_PREFILL, T, int(w["seq"]), int(w["pos0"]))
    ld = round4(int(w["pos0"]) + T)
    scores = torch.zeros((T, ld), dtype=torch.int32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(T, dtype=torch.int32, device=dev)
    out = torch.empty((T, hq, 128), dtype=out_dtype, device=dev)
    lse = torch.empty((T, hq), dtype=torch.float32, device=dev)
    if n_dense is None:
        nbytes = dsa.workspace_size(dsa.OP_PREFILL_STEP, kv, qs, k, hq, P)
    else:
        nbytes = dsa.prefill_attn_workspace_size(kv, qs, k, hq, P, n_dense)
    ws = dsa.make_workspace(nbytes, dev)
    dsa.index_scores(kv, qs, w["q_idx"], P, scores)
    dsa.topk_select(kv, qs, scores, P, k, idx, n_sel, ws)
    dsa.sparse_attn_prefill(kv, qs, w["q"], idx, n_sel, k, P, out, lse, ws, n_dense=n_dense)
    status = dsa.check_device_status(dev)
    assert status == 0, f"device status {status}"
    return {"scores": scores, "idx": idx, "n_sel": n_sel, "out": out, "lse": lse}


def run_prefill_step(w: dict, out_dtype=torch.bfloat16) -> dict:
    """The same chunk through the one-call prefill step (scores, top-k with
    the dense pass's bitmap, attention with the automatic split)."""
    dev = w["q"].device
    kv = paged_kv(w)
    T, k, P, hq = int(w["num_queries"]), int(w["k"]), int(w["prefix_len"]), int(w["num_q_heads"])
    qs = dsa.query_set(dsa.MODE_PREFILL, T, int(w["seq"]), int(w["pos0"]))
    ld = round4(int(w["pos0"]) + T)
    scores = torch.zeros((T, ld), dtype=torch.int32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(T, dtype=torch.int32, device=dev)
    out = torch.empty((T, hq, 128), dtype=out_dtype, device=dev)
    lse = torch.empty((T, hq), dtype=torch.float32, device=dev)
    ws = dsa.make_workspace(dsa.prefill_attn_workspace_size(kv, qs, k, hq, P, -1), dev)
    dsa.prefill_step(kv, qs, w["q"], w["q_idx"], P, k, scores, idx, n_sel, out, lse, ws)
    status = dsa.check_device_status(dev)
    assert status == 0, f"device status {status}"
    return {"scores": scores, "idx": idx, "n_sel": n_sel, "out": out, "lse": lse}


def check_prefill_against_oracle(wn: dict, res: dict, rows=None):
    P = int(wn["prefix_len"])
    pos0 = int(wn["pos0"])
    T = int(wn["num_queries"])
    idx = res["idx"].cpu().numpy()
    n_sel = res["n_sel"].cpu().numpy()
    out = res["out"].float().cpu().numpy()
    lse = res["lse"].cpu().numpy()
    scores = res["scores"].cpu().numpy()
    for i in (range(T) if rows is None else rows):
        r = O.prefill_query(wn, i)
        pos = pos0 + i
        if pos >= P:
            assert np.array_equal(scores[i, P:pos + 1], r["scores"]), f"scores of query {i}"
        assert int(n_sel[i]) == r["n_sel"], f"n_sel of query {i}"
        assert np.array_equal(idx[i], r["idx"]), f"idx of query {i}"
        assert_close(out[i], r["out"], f"out of query {i}")
        assert_close(lse[i], r["lse"], f"lse of query {i}")


def oracle_prefill_sampled(w: dict, i: int, heads_kv, k: int, P: int):
    """Oracle result of prefill query i of a device-resident workload."""
    seq = int(w["seq"])
    pos = int(w["pos0"]) + i
    cand = O.candidate_positions(P, pos)
    wv = dict(w)
    wv["block_table"] = w["block_table"][seq:seq + 1]
    q_idx = w["q_idx"][i].cpu().numpy().astype(np.int64)
    if cand.size:
        icache, ibt = _compact_blocks(wv, 0, cand, "idx_cache")
        ts, s = O.index_scores(q_idx, icache, ibt, P, pos)
    else:
        ts, s = cand, np.zeros(0, dtype=np.int64)
    idx, n_sel = O.topk_select(ts, s, k)
    att = O.attended_positions(P, pos, idx, n_sel)
    hq, hkv = int(w["num_q_heads"]), int(w["num_kv_heads"])
    G = hq // hkv
    heads = {}
    for g in heads_kv:
        kc, kbt = _compact_blocks(wv, 0, att, "k_cache", head=g)
        vc, _ = _compact_blocks(wv, 0, att, "v_cache", head=g)
        q = w["q"][i, g * G:(g + 1) * G].cpu().to(torch.float64).numpy()
        out, lse = O.sparse_gqa_attention(q, kc, vc, kbt, att, 1, 1.0 / np.sqrt(128))
        heads[g] = (out, lse)
    return {"scores": s, "idx": idx, "n_sel": n_sel, "heads": heads}
