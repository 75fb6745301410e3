"""Pins of the CPU oracle to facts outside itself (no GPU).

Each check below ties one oracle step to something the article or the
mathematics fixes: closed forms, brute-force enumeration, special cases that
reduce to a library routine (PyTorch's scaled_dot_product_attention), and
invariants.  test_oracle_mutants.py re-runs these checks against planted
mistakes to show that each one is caught.

Section numbers refer to the article
"国产AI芯片完成前沿大模型Day-0适配:稀疏注意力与混合精度推理全解析".
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    """Parse a golden fixture: '#' comments, 'key: v1 v2 ...' lines."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            out.setdefault(key.strip(), []).append([float(x) for x in vals.split()])
    return out


# ---------------------------------------------------------------- helpers ---
def _tiny_idx_cache(rows_by_pos, nblk, D, bt_row):
    """Indexer cache with the given rows placed at their positions."""
    cache = np.zeros((nblk, O.BLOCK, D), dtype=np.int64)
    for t, row in rows_by_pos.items():
        cache[bt_row[t // O.BLOCK], t % O.BLOCK] = row
    return cache


def _encoded_kv(nblk, hkv, d):
    """K/V cache [blk][64][Hkv][d] whose value encodes (block, head, row, col) exactly."""
    blk, r, g, c = np.meshgrid(np.arange(nblk), np.arange(O.BLOCK), np.arange(hkv),
                               np.arange(d), indexing="ij")
    return (blk * 1_000_000 + g * 100_000 + r * 1000 + c).astype(np.float64)


# ------------------------------------------------------------- row fetch ----
def check_fetch(mod=O):
    bt = np.array([5, 2, 7, 0], dtype=np.int64)
    cache = _encoded_kv(8, 2, 4)
    pos = np.array([0, 63, 64, 130, 255])
    got = mod.fetch_rows(cache, bt, pos, head=1)
    want = np.stack([bt[t // 64] * 1_000_000 + 100_000 + (t % 64) * 1000 + np.arange(4) for t in pos])
    return np.array_equal(got, want)


def test_fetch_rows_closed_form():
    """Section 2.2: position t is row t % 64 of block table[t // 64]."""
    assert check_fetch()


# ---------------------------------------------------------------- scores ----
def check_scores_closed_forms(mod=O):
    rng = np.random.default_rng(1)
    D, P, pos = 64, 64, 64 * 3 + 10
    bt = np.array([3, 0, 2, 1], dtype=np.int64)
    cache = rng.integers(-8, 9, size=(4, O.BLOCK, D))
    ok = True
    # q = unit vector e_j  ->  s(t) = key_t[j]
    for j in (0, 17, 63):
        q = np.zeros(D, dtype=np.int64)
        q[j] = 1
        ts, s = mod.index_scores(q, cache, bt, P, pos)
        ok &= np.array_equal(ts, np.arange(P, pos + 1))
        ok &= np.array_equal(s, [cache[bt[t // 64], t % 64, j] for t in ts])
    # linearity: s(q1 + q2) = s(q1) + s(q2)
    q1, q2 = rng.integers(-8, 9, size=D), rng.integers(-8, 9, size=D)
    _, s1 = mod.index_scores(q1, cache, bt, P, pos)
    _, s2 = mod.index_scores(q2, cache, bt, P, pos)
    _, s12 = mod.index_scores(q1 + q2, cache, bt, P, pos)
    ok &= np.array_equal(s12, s1 + s2)
    # causality at the edge: pos == P has exactly one candidate, pos < P none
    ts, _ = mod.index_scores(q1, cache, bt, P, P)
    ok &= list(ts) == [P]
    ts, _ = mod.index_scores(q1, cache, bt, P, P - 1)
    ok &= ts.size == 0
    return bool(ok)


def test_scores_closed_forms():
    """Section 2.1 scores: unit-vector queries read one key component; the
    score is linear in the query; candidates are [P, pos] inclusive."""
    assert check_scores_closed_forms()


def check_scores_golden(mod=O):
    g = _read_golden("index_scores_small.txt")
    q = np.array(g["q"][0], dtype=np.int64)
    keys = [np.array(r, dtype=np.int64) for r in g["key"]]
    want = [int(v) for v in g["score"][0]]
    P = int(g["prefix_len"][0][0])
    bt = np.array([1, 0], dtype=np.int64)
    rows = {P + i: k for i, k in enumerate(keys)}
    cache = _tiny_idx_cache(rows, 2, len(q), bt)
    ts, s = mod.index_scores(q, cache, bt, P, P + len(keys) - 1)
    return list(s) == want and list(ts) == [P + i for i in range(len(keys))]


def test_scores_golden_hand_computed():
    assert check_scores_golden()


# ----------------------------------------------------------------- top-k ----
def check_topk_special_cases(mod=O):
    ok = True
    ts = np.arange(100, 400)
    # all ties -> the lowest k positions
    idx, n = mod.topk_select(ts, np.zeros(300, dtype=np.int64), 37)
    ok &= n == 37 and np.array_equal(idx, np.arange(100, 137))
    # strictly increasing scores -> the last k positions
    idx, n = mod.topk_select(ts, np.arange(300), 50)
    ok &= n == 50 and np.array_equal(idx, np.arange(350, 400))
    # strictly decreasing -> the first k positions
    idx, n = mod.topk_select(ts, -np.arange(300), 50)
    ok &= n == 50 and np.array_equal(idx, np.arange(100, 150))
    # k >= number of candidates -> all, padded with -1
    idx, n = mod.topk_select(ts[:10], np.arange(10)[::-1].copy(), 16)
    ok &= n == 10 and np.array_equal(idx[:10], ts[:10]) and np.all(idx[10:] == -1)
    # empty candidate set
    idx, n = mod.topk_select(ts[:0], np.zeros(0, dtype=np.int64), 4)
    ok &= n == 0 and np.all(idx == -1)
    return bool(ok)


def test_topk_special_cases():
    """Ties go to the lower position; output ascending, -1 padded."""
    assert check_topk_special_cases()


def _brute_topk(ts, s, k):
    """Among all k-subsets: maximal score sum, then lexicographically
    smallest ascending position tuple (= ties to the lower position)."""
    best = None
    for comb in itertools.combinations(range(len(ts)), k):
        key = (-sum(int(s[i]) for i in comb), tuple(int(ts[i]) for i in comb))
        if best is None or key < best:
            best = key
    return list(best[1])


def check_topk_brute_force(mod=O, trials=60):
    rng = np.random.default_rng(7)
    for _ in range(trials):
        n = int(rng.integers(1, 10))
        k = int(rng.integers(1, 8))
        ts = np.sort(rng.choice(np.arange(64, 200), size=n, replace=False))
        s = rng.integers(-2, 3, size=n)  # heavy ties
        idx, nsel = mod.topk_select(ts, s, k)
        want = list(ts) if n <= k else _brute_topk(ts, s, k)
        if nsel != len(want) or list(idx[:nsel]) != want or np.any(idx[nsel:] != -1):
            return False
    return True


def test_topk_brute_force_subsets():
    assert check_topk_brute_force()


def check_topk_rank_definition(mod=O):
    """t is selected iff fewer than k candidates beat it (higher score, or
    equal score at a lower position)."""
    rng = np.random.default_rng(11)
    ts = np.arange(500, 900)
    s = rng.integers(-6, 7, size=ts.size)
    k = 57
    idx, n = mod.topk_select(ts, s, k)
    sel = set(idx[:n].tolist())
    for i, t in enumerate(ts):
        beats = int(np.sum((s > s[i]) | ((s == s[i]) & (ts < t))))
        if (beats < k) != (int(t) in sel):
            return False
    return n == k


def test_topk_rank_definition():
    assert check_topk_rank_definition()


# ------------------------------------------------------ prefix invariant -----
def _small_workload(seed=3, **kw):
    spec = synth.small_spec(**kw)
    return synth.to_numpy(synth.make_workload(spec, seed, "cpu"))


def check_prefix_invariant(mod=O):
    w = _small_workload(lens=(40, 64, 65, 300), batch=4, prefix_len=64, hq=4, hkv=2, k=16)
    for b in range(4):
        r = mod.decode_query(w, b)
        pos = int(w["context_lens"][b]) - 1
        P = int(w["prefix_len"])
        n_prefix = min(P, pos + 1)
        att = r["attended"]
        if not set(range(n_prefix)).issubset(set(att.tolist())):
            return False
        if len(att) != n_prefix + min(16, max(0, pos + 1 - P)):
            return False
        if np.any(r["idx"][: r["n_sel"]] < P):  # the prefix is never scored
            return False
    return True


def test_prefix_always_attended():
    """Section 2.4: the vision prefix is always attended and never selected."""
    assert check_prefix_invariant()


# ------------------------------------------------------------- attention ----
def check_attention_closed_forms(mod=O):
    rng = np.random.default_rng(5)
    ok = True
    q = rng.standard_normal((4, 16))
    v = rng.standard_normal((1, 16))
    kk = rng.standard_normal((1, 16))
    out, lse = mod.softmax_attention(q, kk, v, 0.25)
    ok &= np.allclose(out, np.repeat(v, 4, 0), rtol=0, atol=1e-15)
    ok &= np.allclose(lse, 0.25 * q @ kk[0], atol=1e-12)
    # identical keys -> mean of V, lse = z + ln R
    kk = np.repeat(rng.standard_normal((1, 16)), 9, 0)
    v = rng.standard_normal((9, 16))
    out, lse = mod.softmax_attention(q, kk, v, 0.3)
    ok &= np.allclose(out, np.repeat(v.mean(0, keepdims=True), 4, 0), atol=1e-12)
    ok &= np.allclose(lse, 0.3 * q @ kk[0] + math.log(9), atol=1e-12)
    # constant V -> that constant
    kk = rng.standard_normal((13, 16))
    v = np.full((13, 16), 0.625)
    out, _ = mod.softmax_attention(q, kk, v, 0.1)
    ok &= np.allclose(out, 0.625, atol=1e-13)
    return bool(ok)


def test_attention_closed_forms():
    assert check_attention_closed_forms()


def check_attention_golden(mod=O):
    g = _read_golden("attention_two_rows.txt")
    q = np.array(g["q"], dtype=np.float64)
    kk = np.array(g["k"], dtype=np.float64)
    v = np.array(g["v"], dtype=np.float64)
    scale = g["scale"][0][0]
    out, lse = mod.softmax_attention(q, kk, v, scale)
    return (np.allclose(out, np.array(g["out"]), atol=1e-12)
            and np.allclose(lse, np.array(g["lse"][0]), atol=1e-12))


def test_attention_golden_two_rows():
    assert check_attention_golden()


def _sdpa_dense(q, k_rows, v_rows, scale, causal):
    """PyTorch's scaled_dot_product_attention in float64 on the CPU."""
    qt = torch.from_numpy(q)[None]            # [1, H, Lq, d]
    kt = torch.from_numpy(k_rows)[None]
    vt = torch.from_numpy(v_rows)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    return o[0].numpy()


def check_dense_decode_equals_sdpa(mod=O):
    """k >= L: sparse attention of the last token is dense attention over
    all L keys (the prefix plus every candidate)."""
    w = _small_workload(lens=(300, 190), batch=2, prefix_len=64, hq=8, hkv=2, k=4096)
    for b in range(2):
        r = mod.decode_query(w, b)
        L = int(w["context_lens"][b])
        if not np.array_equal(r["attended"], np.arange(L)):
            return False
        G = 4
        for g in range(2):
            kr = mod.fetch_rows(w["k_cache"], w["block_table"][b], np.arange(L), head=g)
            vr = mod.fetch_rows(w["v_cache"], w["block_table"][b], np.arange(L), head=g)
            q = w["q"][b][g * G:(g + 1) * G][:, None, :]   # [G, 1, d]
            ref = _sdpa_dense(q, np.repeat(kr[None], G, 0), np.repeat(vr[None], G, 0),
                              1 / math.sqrt(128), causal=False)[:, 0]
            if not np.allclose(r["out"][g * G:(g + 1) * G], ref, rtol=0, atol=1e-12):
                return False
    return True


def test_dense_limit_decode_equals_sdpa():
    assert check_dense_decode_equals_sdpa()


def check_dense_prefill_equals_sdpa(mod=O):
    """Prefill with k >= T: every query attends causally to [0, pos],
    which is PyTorch's causal SDPA."""
    spec = synth.Spec("p", "prefill", 1, (150,), 40, 4, 2, 4096, num_queries=150, pos0=0)
    w = synth.to_numpy(synth.make_workload(spec, 9, "cpu"))
    T = 150
    for g in range(2):
        kr = mod.fetch_rows(w["k_cache"], w["block_table"][0], np.arange(T), head=g)
        vr = mod.fetch_rows(w["v_cache"], w["block_table"][0], np.arange(T), head=g)
        q = np.transpose(w["q"][:, 2 * g:2 * g + 2, :], (1, 0, 2))   # [2, T, d]
        ref = _sdpa_dense(q, np.repeat(kr[None], 2, 0), np.repeat(vr[None], 2, 0),
                          1 / math.sqrt(128), causal=True)
        for i in (0, 1, 39, 40, 41, 99, 149):
            r = mod.prefill_query(w, i)
            if not np.allclose(r["out"][2 * g:2 * g + 2], ref[:, i], rtol=0, atol=1e-12):
                return False
    return True


def test_dense_limit_prefill_equals_causal_sdpa():
    assert check_dense_prefill_equals_sdpa()


def check_window_equals_banded_sdpa(mod=O):
    """Local sliding-window attention: every query attends [pos - W + 1, pos],
    which is PyTorch's SDPA with a banded boolean mask; with W >= T it is the
    causal SDPA."""
    spec = synth.Spec("p", "prefill", 1, (150,), 0, 4, 2, 8, num_queries=150, pos0=0)
    w = synth.to_numpy(synth.make_workload(spec, 9, "cpu"))
    T = 150
    i_idx = np.arange(T)[:, None]
    j_idx = np.arange(T)[None, :]
    for W in (37, 64, 150, 500):
        band = torch.from_numpy((j_idx <= i_idx) & (j_idx > i_idx - W))
        for g in range(2):
            kr = mod.fetch_rows(w["k_cache"], w["block_table"][0], np.arange(T), head=g)
            vr = mod.fetch_rows(w["v_cache"], w["block_table"][0], np.arange(T), head=g)
            q = np.transpose(w["q"][:, 2 * g:2 * g + 2, :], (1, 0, 2))   # [2, T, d]
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q)[None], torch.from_numpy(np.repeat(kr[None], 2, 0))[None],
                torch.from_numpy(np.repeat(vr[None], 2, 0))[None], attn_mask=band,
                scale=1 / math.sqrt(128))[0].numpy()
            for i in (0, 1, 36, 37, 38, 63, 64, 65, 149):
                r = mod.window_query(w, i, w["q"][i], 0, W)
                if len(r["attended"]) != min(W, i + 1):
                    return False
                if not np.allclose(r["out"][2 * g:2 * g + 2], ref[:, i], rtol=0, atol=1e-12):
                    return False
    return True


def test_window_equals_banded_sdpa():
    assert check_window_equals_banded_sdpa()


def check_window_of_one(mod=O):
    """W = 1: every head's output is the query's own V row and its log-sum-exp
    is its own scaled score."""
    w = _small_workload(lens=(300,), batch=1, prefix_len=0, hq=4, hkv=2, k=8)
    for pos in (0, 63, 64, 299):
        r = mod.window_query(w, pos, w["q"][0], 0, 1)
        for h in range(4):
            g = h // 2
            v = mod.fetch_rows(w["v_cache"], w["block_table"][0], np.array([pos]), head=g)[0]
            kk = mod.fetch_rows(w["k_cache"], w["block_table"][0], np.array([pos]), head=g)[0]
            if not np.allclose(r["out"][h], v, rtol=0, atol=1e-12):
                return False
            if not np.isclose(r["lse"][h], float(w["q"][0][h] @ kk) / math.sqrt(128), rtol=0, atol=1e-10):
                return False
    return True


def test_window_of_one():
    assert check_window_of_one()


def _heads_workload(**kw):
    spec = synth.small_spec(lens=(300, 190, 777), batch=3, prefix_len=64, hq=8, hkv=2, k=40, idx_heads=2, **kw)
    return synth.to_numpy(synth.make_workload(spec, 3, "cpu"))


def check_heads_with_equal_indexers_share_the_selection(mod=O):
    """Per-head indexer whose heads all carry the same keys and query: every
    head selects what the shared indexer selects, and the outputs equal the
    shared path's (the per-head reading reduces to the pinned shared one)."""
    w = _heads_workload()
    w_shared = dict(w)
    w_shared["idx_cache"] = w["idx_cache"][:, 0]
    w_shared["q_idx"] = w["q_idx"][:, 0]
    w_heads = dict(w)
    w_heads["idx_cache"] = np.repeat(w["idx_cache"][:, :1], 2, axis=1)
    w_heads["q_idx"] = np.repeat(w["q_idx"][:, :1], 2, axis=1)
    for b in range(3):
        r1 = mod.decode_query(w_shared, b)
        r2 = mod.decode_query_heads(w_heads, b)
        for g in range(2):
            if not (np.array_equal(r2["idx"][g], r1["idx"]) and r2["n_sel"][g] == r1["n_sel"]):
                return False
        if not (np.allclose(r2["out"], r1["out"], rtol=0, atol=1e-12) and np.allclose(r2["lse"], r1["lse"], rtol=0, atol=1e-12)):
            return False
    return True


def test_heads_with_equal_indexers_share_the_selection():
    assert check_heads_with_equal_indexers_share_the_selection()


def check_heads_are_independent(mod=O):
    """Head 1's indexer query zero: all its scores tie, so it selects the k
    lowest candidate positions, while head 0 keeps its own top-k; swapping the
    two KV heads (caches, indexers and query heads) swaps the results."""
    w = _heads_workload()
    w["q_idx"] = w["q_idx"].copy()
    w["q_idx"][:, 1] = 0
    for b in range(3):
        r = mod.decode_query_heads(w, b)
        pos = int(w["context_lens"][b]) - 1
        n = min(40, pos + 1 - 64)
        if not (r["n_sel"][1] == n and np.array_equal(r["idx"][1][:n], np.arange(64, 64 + n))):
            return False
        ts, s = mod.index_scores(w["q_idx"][b][0], w["idx_cache"][:, 0], w["block_table"][b], 64, pos)
        idx0, _ = mod.topk_select(ts, s, 40)
        if not np.array_equal(r["idx"][0], idx0):
            return False
        sw = dict(w)
        for name in ("k_cache", "v_cache"):
            sw[name] = w[name][:, :, ::-1]
        sw["idx_cache"] = w["idx_cache"][:, ::-1]
        sw["q_idx"] = w["q_idx"][:, ::-1]
        sw["q"] = np.concatenate([w["q"][:, 4:], w["q"][:, :4]], axis=1)
        r2 = mod.decode_query_heads(sw, b)
        if not (np.array_equal(r2["idx"][0], r["idx"][1]) and np.array_equal(r2["idx"][1], r["idx"][0])):
            return False
        if not np.allclose(np.concatenate([r2["out"][4:], r2["out"][:4]]), r["out"], rtol=0, atol=1e-12):
            return False
    return True


def test_heads_are_independent():
    assert check_heads_are_independent()


def relocate_heads(w, seed=5):
    """The same per-head workload re-laid out with one block table per KV head:
    head g's slices of every block (K, V and indexer keys) move to block
    perm_g[old id], a different permutation for each head, and head g's table
    names the new ids.  Each physical block then holds, in its head-g slice,
    positions that other heads keep elsewhere."""
    nb = w["k_cache"].shape[0]
    hkv = int(w["num_kv_heads"])
    rng = np.random.default_rng(seed)
    w2 = dict(w)
    k2, v2, i2 = np.empty_like(w["k_cache"]), np.empty_like(w["v_cache"]), np.empty_like(w["idx_cache"])
    tables = []
    for g in range(hkv):
        perm = rng.permutation(nb)  # old block id -> this head's new id
        k2[perm, :, g] = w["k_cache"][:, :, g]
        v2[perm, :, g] = w["v_cache"][:, :, g]
        i2[perm, g] = w["idx_cache"][:, g]
        bt = w["block_table"].copy()
        bt[bt >= 0] = perm[bt[bt >= 0]]
        tables.append(bt)
    w2["k_cache"], w2["v_cache"], w2["idx_cache"] = k2, v2, i2
    w2["block_table_heads"] = np.stack(tables)
    return w2


def check_heads_per_head_block_tables(mod=O):
    """Per-head block tables (the allocator's per-head block bitmaps): each KV
    head's data moved under its own permutation of the pool, each head reading
    through its own table, gives the same selections and outputs as the
    shared table over the original layout."""
    w = _heads_workload()
    w2 = relocate_heads(w)
    if all(np.array_equal(w2["block_table_heads"][g], w["block_table"]) for g in range(2)):
        return False  # the relocation must move something
    for b in range(3):
        r1, r2 = mod.decode_query_heads(w, b), mod.decode_query_heads(w2, b)
        for g in range(2):
            if not (np.array_equal(r1["idx"][g], r2["idx"][g]) and r1["n_sel"][g] == r2["n_sel"][g]
                    and np.array_equal(r1["scores"][g], r2["scores"][g])):
                return False
        if not (np.array_equal(r1["out"], r2["out"]) and np.array_equal(r1["lse"], r2["lse"])):
            return False
    return True


def test_heads_per_head_block_tables():
    assert check_heads_per_head_block_tables()


def check_block_table_permutation(mod=O):
    """Re-laying the cache under another block permutation changes nothing."""
    w = _small_workload(lens=(777,), batch=1, prefix_len=64, hq=8, hkv=2, k=100)
    r1 = mod.decode_query(w, 0)
    nb = w["k_cache"].shape[0]
    perm = np.random.default_rng(2).permutation(nb)   # old block id -> new id
    w2 = dict(w)
    for name in ("k_cache", "v_cache", "idx_cache"):
        new = np.empty_like(w[name])
        new[perm] = w[name]
        w2[name] = new
    bt = w["block_table"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    w2["block_table"] = bt
    r2 = mod.decode_query(w2, 0)
    return (np.array_equal(r1["idx"], r2["idx"]) and np.array_equal(r1["out"], r2["out"])
            and np.array_equal(r1["lse"], r2["lse"]))


def test_block_table_permutation_invariance():
    assert check_block_table_permutation()


# ------------------------------------------------------- gather / write -----
def check_gather(mod=O):
    bt = np.array([3, 1, 0, 2], dtype=np.int64)
    kc = _encoded_kv(4, 2, 8)
    vc = -_encoded_kv(4, 2, 8)
    pos = np.array([0, 1, 70, 200])
    ko, vo = mod.kv_gather(kc, vc, bt, pos, 2, 6)
    ok = True
    for g in range(2):
        for r, t in enumerate(pos):
            want = bt[t // 64] * 1_000_000 + g * 100_000 + (t % 64) * 1000 + np.arange(8)
            ok &= np.array_equal(ko[g, r], want) and np.array_equal(vo[g, r], -want)
        ok &= np.all(ko[g, 4:] == 0) and np.all(vo[g, 4:] == 0)
    return bool(ok)


def test_gather_closed_form():
    assert check_gather()


def check_kv_write(mod=O):
    rng = np.random.default_rng(4)
    kc = np.zeros((3, 64, 2, 8))
    vc = np.zeros((3, 64, 2, 8))
    ic = np.zeros((3, 64, 4), dtype=np.int64)
    slots = np.array([5, 64 * 2 + 63, 64 + 1])
    kn = rng.standard_normal((3, 2, 8))
    vn = rng.standard_normal((3, 2, 8))
    inn = rng.integers(-8, 9, size=(3, 4))
    k2, v2, i2 = mod.kv_write(kc, vc, ic, slots, kn, vn, inn)
    ok = np.array_equal(k2[0, 5], kn[0]) and np.array_equal(k2[2, 63], kn[1])
    ok &= np.array_equal(v2[1, 1], vn[2]) and np.array_equal(i2[2, 63], inn[1])
    ok &= np.count_nonzero(k2) == kn.size and np.count_nonzero(kc) == 0
    return bool(ok)


def test_kv_write_scatter():
    assert check_kv_write()


def check_kv_write_heads(mod=O):
    """Per-head write: each head's values land in its own slice of its own
    slot, nothing else changes, and two heads given the same block keep both
    their values (no write conflict between heads)."""
    rng = np.random.default_rng(6)
    kc = np.zeros((3, 64, 2, 8))
    vc = np.zeros((3, 64, 2, 8))
    ic = np.zeros((3, 2, 64, 4), dtype=np.int64)
    slots = np.array([[5, 5], [64 * 2 + 63, 64 + 7], [64 + 1, 3]])  # token 0: both heads in slot 5
    kn = rng.standard_normal((3, 2, 8)) + 10.0  # nonzero everywhere
    vn = rng.standard_normal((3, 2, 8)) + 10.0
    inn = rng.integers(1, 9, size=(3, 2, 4))
    k2, v2, i2 = mod.kv_write_heads(kc, vc, ic, slots, kn, vn, inn)
    ok = True
    for j in range(3):
        for h in range(2):
            blk, row = divmod(int(slots[j, h]), 64)
            ok &= np.array_equal(k2[blk, row, h], kn[j, h]) and np.array_equal(v2[blk, row, h], vn[j, h])
            ok &= np.array_equal(i2[blk, h, row], inn[j, h])
    ok &= np.count_nonzero(k2) == kn.size and np.count_nonzero(v2) == vn.size and np.count_nonzero(i2) == inn.size
    ok &= np.count_nonzero(kc) == 0
    return bool(ok)


def test_kv_write_heads():
    assert check_kv_write_heads()
