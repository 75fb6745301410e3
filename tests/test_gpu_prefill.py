"""Prefill path on the GPU against the CPU oracle: causal int8 indexer GEMM,
per-row top-k, and sparse GQA attention over each query's own selection."""
import dataclasses

import numpy as np
import pytest
import torch

import harness as H
import oracle.dsa_oracle as O
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _prefill_spec(T, pos0=0, P=64, k=100, hq=8, hkv=2, batch_lens=None, seq=0, **kw):
    lens = batch_lens or (pos0 + T,)
    return synth.Spec("prefill-small", "prefill", len(lens), tuple(lens), P, hq, hkv, k, num_queries=T,
                      pos0=pos0, **kw)


# How the attention splits the chunk: the library's automatic split (every
# query of these small chunks goes to the dense masked pass), every query
# gathered, and a split inside a dense tile pair (both parts in one call).
SPLITS = ["auto", "gather", "split"]


def _n_dense(split, T):
    return {"auto": None, "gather": 0, "split": T // 2 + 1}[split]


def _run(spec, seed=5, seq=0, out_dtype=torch.bfloat16, split="auto"):
    w_cpu = synth.make_workload(spec, seed, "cpu")
    w_cpu["seq"] = seq
    w = H.on(w_cpu, DEV)
    res = H.run_prefill(w, out_dtype=out_dtype, n_dense=_n_dense(split, spec.num_queries))
    H.check_prefill_against_oracle(synth.to_numpy(w_cpu), res)
    return res


@pytest.mark.parametrize("split", SPLITS)
def test_prefill_small_from_position_zero(lib, split):
    """Queries inside the prefix, at its edge, and with fewer / more than k candidates."""
    _run(_prefill_spec(T=400, pos0=0, P=64, k=100), split=split)


@pytest.mark.parametrize("split", SPLITS)
def test_prefill_continuation_chunk(lib, split):
    """A chunk of queries that starts deep into the sequence (pos0 > 0)."""
    _run(_prefill_spec(T=200, pos0=1000, P=100, k=256, hq=16, hkv=2), split=split)


def test_prefill_second_sequence_of_the_table(lib):
    spec = _prefill_spec(T=150, pos0=50, P=64, k=64, batch_lens=(700, 200))
    _run(spec, seq=1)


@pytest.mark.parametrize("split", SPLITS)
def test_prefill_group_16_and_fp32(lib, split):
    _run(_prefill_spec(T=130, pos0=200, P=32, k=50, hq=32, hkv=2), out_dtype=torch.float32, split=split)


def test_prefill_full_int8_range(lib):
    _run(_prefill_spec(T=150, pos0=300, P=64, k=90, idx_lo=-128, idx_hi=127))


@pytest.mark.parametrize("split", SPLITS)
def test_prefill_separate_kv_arrays(lib, split):
    """The same path with K and V in two arrays (two copies per attended row)."""
    _run(_prefill_spec(T=200, pos0=100, P=64, k=100, hq=16, hkv=4, kv_layout="separate"), split=split)


@pytest.mark.parametrize("split", SPLITS)
def test_prefill_prefix_tiles_ragged(lib, split):
    """Tiles of a group of 3 heads (42 queries per 128-row tile, two rows
    unused), a prefix of 130 (three 64-key chunks, the last with 2 keys) and
    queries before, inside and past it."""
    _run(_prefill_spec(T=300, pos0=10, P=130, k=80, hq=24, hkv=8), split=split)


@pytest.mark.parametrize("split", SPLITS)
def test_prefill_without_prefix(lib, split):
    _run(_prefill_spec(T=100, pos0=0, P=0, k=40), split=split)


def test_prefill_group_1(lib):
    """One query head per KV head: 128 queries per dense tile."""
    _run(_prefill_spec(T=300, pos0=40, P=20, k=60, hq=4, hkv=4))


def test_prefill_automatic_split_at_the_crossover(lib):
    """A chunk whose later queries lie past the dense pass's range: the
    automatic split runs a whole number of dense tile pairs and gathers the rest."""
    spec = _prefill_spec(T=400, pos0=300, P=16, k=24)
    w_cpu = synth.make_workload(spec, 5, "cpu")
    w_cpu["seq"] = 0
    w = H.on(w_cpu, DEV)
    kv = H.paged_kv(w)
    qs = H.dsa.query_set(H.dsa.MODE_PREFILL, spec.num_queries, 0, spec.pos0)
    n = H.dsa.prefill_dense_queries(kv, qs, spec.k, spec.num_q_heads, spec.prefix_len)
    pair = 2 * (128 // (spec.num_q_heads // spec.num_kv_heads))
    lim = 10 * (spec.prefix_len + spec.k) - spec.pos0
    assert 0 < n < spec.num_queries and n % pair == 0 and n <= lim < n + pair
    res = H.run_prefill(w)
    H.check_prefill_against_oracle(synth.to_numpy(w_cpu), res)


def test_prefill_dense_ignores_unwritten_slots(lib):
    """Slots of the last block past the chunk's last position hold NaN (never
    written): the dense pass reads them with its 64-position blocks but gives
    them zero weight, so every output stays finite and matches the oracle."""
    spec = _prefill_spec(T=100, pos0=37, P=16, k=40)
    w_cpu = synth.make_workload(spec, 5, "cpu")
    w_cpu["seq"] = 0
    last = spec.pos0 + spec.num_queries - 1
    blk = int(w_cpu["block_table"][0, last // 64])
    w_cpu["kv"][blk, last % 64 + 1:] = float("nan")  # [block][row][K/V][head][128]
    w = H.on(w_cpu, DEV)
    res = H.run_prefill(w, n_dense=spec.num_queries)
    assert torch.isfinite(res["out"].float()).all() and torch.isfinite(res["lse"]).all()
    H.check_prefill_against_oracle(synth.to_numpy(w_cpu), res)


def test_prefill_dense_bad_selected_position_sets_status(lib):
    """A selected position past the query's own one is left out by the dense
    pass and reported through the status word, without a fault."""
    spec = _prefill_spec(T=64, pos0=100, P=16, k=40)
    w = H.on(synth.make_workload(spec, 5, "cpu") | {"seq": 0}, DEV)
    res = H.run_prefill(w, n_dense=spec.num_queries)
    kv = H.paged_kv(w)
    qs = H.dsa.query_set(H.dsa.MODE_PREFILL, spec.num_queries, 0, spec.pos0)
    idx = res["idx"].clone()
    idx[3, 0] = spec.pos0 + 3 + 5
    ws = H.dsa.make_workspace(H.dsa.prefill_attn_workspace_size(kv, qs, spec.k, spec.num_q_heads,
                                                                  spec.prefix_len, spec.num_queries), DEV)
    out = torch.empty_like(res["out"])
    H.dsa.sparse_attn_prefill(kv, qs, w["q"], idx, res["n_sel"], spec.k, spec.prefix_len, out, None, ws,
                              n_dense=spec.num_queries)
    assert H.dsa.check_device_status() == 4
    assert H.dsa.check_device_status() == 0


def test_full_prefill_16k(lib):
    """The full 16K chunk: scores and indices bit-exact against the oracle on
    256 seeded-random query rows plus the edge rows (inside the prefix, at its
    edge, at the k-candidate edge, the last row); attention on sampled rows and
    KV heads; counts, order, range and padding checked on every row."""
    spec = synth.CONFIGS[4]
    w = synth.make_workload(spec, 1004, DEV)
    res = H.run_prefill(w)
    P, k = spec.prefix_len, spec.k
    idx = res["idx"].cpu().numpy()
    n_sel = res["n_sel"].cpu().numpy()
    scores = res["scores"].cpu().numpy()
    out = res["out"].float().cpu().numpy()
    lse = res["lse"].cpu().numpy()
    G = spec.num_q_heads // spec.num_kv_heads
    edge = [0, 1, P - 1, P, P + 1, P + k - 1, P + k, P + k + 1, spec.num_queries - 1]
    rows = sorted(set(edge) | set(np.random.default_rng(16).integers(0, spec.num_queries, 256).tolist()))
    ref = H.oracle_indices_all(w, k, P, rows=rows)
    for i in rows:
        r = ref[i]
        if i >= P:
            assert np.array_equal(scores[i, P:i + 1], r["scores"]), f"scores row {i}"
        assert int(n_sel[i]) == r["n_sel"], f"n_sel row {i}"
        assert np.array_equal(idx[i], r["idx"]), f"idx row {i}"
    for i in (0, 575, 576, 577, P + k - 1, P + k, 9000, spec.num_queries - 1):
        r = H.oracle_prefill_sampled(w, i, [0, 3], k, P)
        for g, (o, s) in r["heads"].items():
            H.assert_close(out[i, g * G:(g + 1) * G], o, f"out row {i} kv head {g}")
            H.assert_close(lse[i, g * G:(g + 1) * G], s, f"lse row {i} kv head {g}")
    # every row: the count, ascending order, causal range, -1 padding
    pos = np.arange(spec.num_queries)
    want = np.minimum(k, np.maximum(0, pos + 1 - P))
    assert np.array_equal(n_sel, want)
    valid = np.arange(k)[None, :] < n_sel[:, None]
    assert np.all(idx[~valid] == -1)
    sel = np.where(valid, idx, 0)
    assert np.all(np.where(valid, (sel >= P) & (sel <= pos[:, None]), True))
    d = np.diff(np.where(valid, idx, np.iinfo(np.int32).max), axis=1)
    assert np.all(d[valid[:, 1:]] > 0)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


# ----------------------------------------------- scores + top-k in one kernel
def _fused_select(spec, seed=5, q_idx_fill=None):
    w_cpu = synth.make_workload(spec, seed, "cpu")
    w_cpu["seq"] = 0
    if q_idx_fill is not None:
        w_cpu["q_idx"].fill_(q_idx_fill)
    w = H.on(w_cpu, DEV)
    kv = H.paged_kv(w)
    T, k, P = spec.num_queries, spec.k, spec.prefix_len
    qs = H.dsa.query_set(H.dsa.MODE_PREFILL, T, 0, spec.pos0)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    n_sel = torch.full((T,), -7, dtype=torch.int32, device=DEV)
    H.dsa.prefill_select(kv, qs, w["q_idx"], P, k, idx, n_sel)
    assert H.dsa.check_device_status() == 0
    return w_cpu, idx.cpu().numpy(), n_sel.cpu().numpy()


def _check_fused_against_oracle(w_cpu, idx, n_sel, rows=None):
    wn = synth.to_numpy(w_cpu)
    T = int(wn["num_queries"])
    for i in (range(T) if rows is None else rows):
        r = O.prefill_query(wn, i)
        assert int(n_sel[i]) == r["n_sel"], f"n_sel of query {i}"
        assert np.array_equal(idx[i], r["idx"]), f"idx of query {i}"


@pytest.mark.parametrize("case", ["from_zero", "continuation", "no_prefix", "group_of_3_rows"])
def test_fused_select_matches_oracle(lib, case):
    """Queries with fewer candidates than k (all taken), at the edge, and with
    a real selection in the same 128-query CTA; pass-1 window path."""
    spec = {"from_zero": _prefill_spec(T=400, pos0=0, P=64, k=100),
            "continuation": _prefill_spec(T=300, pos0=1000, P=100, k=256),
            "no_prefix": _prefill_spec(T=260, pos0=0, P=0, k=40),
            "group_of_3_rows": _prefill_spec(T=129, pos0=700, P=130, k=80, hq=24, hkv=8)}[case]
    _check_fused_against_oracle(*_fused_select(spec))


@pytest.mark.parametrize("lo,hi", [(-128, 127), (-16, 16), (-1, 1)])
def test_fused_select_value_ranges(lib, lo, hi):
    """Full int8 (f16 products, scores past the pass-1 window: the three-level
    radix path), [-16, 16] (e4m3 products, scores up to 16384: radix path),
    [-1, 1] (scores in [-64, 64]: heavy ties at the threshold)."""
    spec = _prefill_spec(T=300, pos0=400, P=64, k=90, idx_lo=lo, idx_hi=hi)
    _check_fused_against_oracle(*_fused_select(spec))


def test_fused_select_all_ties(lib):
    """A zero indexer query: every score 0, the k lowest candidate positions."""
    spec = _prefill_spec(T=200, pos0=300, P=32, k=64)
    w_cpu, idx, n_sel = _fused_select(spec, q_idx_fill=0)
    for i in range(200):
        pos = 300 + i
        n = min(64, pos + 1 - 32)
        assert int(n_sel[i]) == n
        assert np.array_equal(idx[i][:n], np.arange(32, 32 + n)) and np.all(idx[i][n:] == -1)
    _check_fused_against_oracle(w_cpu, idx, n_sel, rows=[0, 31, 199])


def test_fused_select_full_16k_equals_separate_steps(lib):
    """The 16K chunk: the fused kernel's indices and counts equal, bit for bit
    and on every row, those of dsa_index_scores + dsa_topk_select (checked
    against the oracle in test_full_prefill_16k), and the oracle on sampled rows."""
    spec = synth.CONFIGS[4]
    w = synth.make_workload(spec, 1004, DEV)
    res = H.run_prefill(w)
    kv = H.paged_kv(w)
    T, k, P = spec.num_queries, spec.k, spec.prefix_len
    qs = H.dsa.query_set(H.dsa.MODE_PREFILL, T, 0, 0)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    n_sel = torch.full((T,), -7, dtype=torch.int32, device=DEV)
    H.dsa.prefill_select(kv, qs, w["q_idx"], P, k, idx, n_sel)
    assert H.dsa.check_device_status() == 0
    assert torch.equal(n_sel, res["n_sel"])
    assert torch.equal(idx, res["idx"])
    rows = sorted(set(np.random.default_rng(11).integers(0, T, size=24).tolist()) | {0, P, P + k, T - 1})
    ref = H.oracle_indices_all(w, k, P, rows=rows)
    idx_h, n_h = idx.cpu().numpy(), n_sel.cpu().numpy()
    for i in rows:
        assert int(n_h[i]) == ref[i]["n_sel"] and np.array_equal(idx_h[i], ref[i]["idx"]), f"query {i}"


@pytest.mark.parametrize("T,pos0,P,k,hq,hkv,out_dtype", [
    (400, 0, 64, 100, 8, 2, torch.bfloat16),     # from position 0: every query dense (automatic split)
    (400, 300, 16, 24, 8, 2, torch.bfloat16),    # past the dense range: dense tile pairs, then gathered
    (260, 90, 64, 100, 32, 2, torch.float32),    # group 16, fp32 out
])
def test_prefill_step_one_call(lib, T, pos0, P, k, hq, hkv, out_dtype):
    """The one-call prefill step (its top-k writes the dense pass's bitmap)
    against the oracle, and against the three calls in sequence: the same
    scores and selections bit for bit, outputs within tolerance."""
    spec = _prefill_spec(T=T, pos0=pos0, P=P, k=k, hq=hq, hkv=hkv)
    w_cpu = synth.make_workload(spec, 5, "cpu")
    w_cpu["seq"] = 0
    w = H.on(w_cpu, DEV)
    one = H.run_prefill_step(w, out_dtype=out_dtype)
    H.check_prefill_against_oracle(synth.to_numpy(w_cpu), one)
    three = H.run_prefill(w, out_dtype=out_dtype)
    assert torch.equal(one["scores"], three["scores"])
    assert torch.equal(one["idx"], three["idx"]) and torch.equal(one["n_sel"], three["n_sel"])
    H.assert_close(one["out"].float().cpu().numpy(), three["out"].float().cpu().numpy(), "step vs three calls")
