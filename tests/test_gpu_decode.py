"""Decode path on the GPU against the CPU oracle (bit-exact indices and
scores; attention within atol 2e-3 + rtol 1e-2 * |ref|)."""
import numpy as np
import pytest
import torch

import harness as H
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run(spec, seed=11, out_dtype=torch.bfloat16, split_api=False, mutate=None):
    w_cpu = synth.make_workload(spec, seed, "cpu")
    if mutate:
        mutate(w_cpu)
    w = H.on(w_cpu, DEV)
    res = H.run_decode_step(w, out_dtype=out_dtype, split_api=split_api)
    H.check_decode_against_oracle(synth.to_numpy(w_cpu), res)
    return res


@pytest.mark.parametrize("layout", ["adjacent", "separate"])
def test_decode_small_fused(lib, layout):
    """K and V of a slot in one row (one copy per attended position) or in two
    arrays (two copies)."""
    _run(synth.small_spec(kv_layout=layout))


def test_decode_small_split_calls_match_fused(lib):
    """The separate calls and the fused step select the same positions; their
    outputs agree within the attention tolerance (the fused step walks the
    prefix rows in a pass of their own, so its partial states are merged in
    another order)."""
    spec = synth.small_spec(lens=(3000, 513, 4100), k=300, hq=16, hkv=4)
    a = _run(spec, split_api=True)
    w = H.on(synth.make_workload(spec, 11, "cpu"), DEV)
    b = H.run_decode_step(w)
    assert torch.equal(a["idx"], b["idx"]) and torch.equal(a["n_sel"], b["n_sel"])
    H.assert_close(b["out"].float().cpu().numpy(), a["out"].float().cpu().numpy(), "fused out vs separate calls")
    H.assert_close(b["lse"].cpu().numpy(), a["lse"].cpu().numpy(), "fused lse vs separate calls")


@pytest.mark.parametrize("lens,prefix,k", [
    ((40, 64, 65, 66), 64, 8),          # context inside the prefix, at its edge, one and two past it
    ((129, 200, 1000), 0, 7),           # no prefix
    ((128, 192, 4096), 64, 4096),       # k larger than every candidate set: take all
    ((4096 + 1, 64 * 37), 100, 1),      # k = 1, prefix not a multiple of the block size
    ((2048 * 3 + 5,), 64, 2048),        # several compaction chunks, ragged tail
])
def test_decode_edge_shapes(lib, lens, prefix, k):
    _run(synth.small_spec(batch=len(lens), lens=lens, prefix_len=prefix, k=k, hq=8, hkv=2))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (32, 2), (8, 8), (16, 1), (64, 8), (8, 1)])
@pytest.mark.parametrize("layout", ["adjacent", "separate"])
def test_decode_group_sizes(lib, hq, hkv, layout):
    _run(synth.small_spec(hq=hq, hkv=hkv, lens=(900, 1800), kv_layout=layout))


@pytest.mark.parametrize("hq,hkv,layout", [(64, 8, "adjacent"), (64, 8, "separate"), (16, 2, "adjacent")])
def test_decode_two_pass_mixed_contexts(lib, hq, hkv, layout):
    """A long context makes the selection take several CTAs per sequence, so
    the step walks every sequence's prefix rows in a pass of their own, before
    its wait on the selection; beside it, contexts inside the prefix, at its
    edge and just past it (the first two have all their rows in the second
    pass), and prefix segments of one tile."""
    _run(synth.small_spec(batch=5, lens=(20000, 40, 64, 65, 300), prefix_len=64, k=100, hq=hq, hkv=hkv,
                          kv_layout=layout))


@pytest.mark.parametrize("lens", [
    (12000, 16500),          # top-k cluster of 2 CTAs per sequence (longest context 16.5K)
    (30000, 9000, 21000),    # 4 CTAs per sequence
    (60000, 45001),          # 8 CTAs per sequence
])
def test_decode_selection_cluster_sizes(lib, lens):
    """Contexts that make the selection kernel use clusters of 2, 4 and 8 CTAs
    per sequence (parts exchange their counts through distributed shared memory)."""
    _run(synth.small_spec(lens=lens, prefix_len=128, k=1024, hq=8, hkv=2))


def _binary_keys(w):
    """Index keys of 0s and 1s and an all-ones query: scores are counts in
    [0, 64], so the k-th largest is shared by many positions in every part."""
    g = torch.Generator().manual_seed(3)
    w["idx_cache"].copy_(torch.randint(0, 2, tuple(w["idx_cache"].shape), generator=g).to(torch.int8))
    w["q_idx"].fill_(1)


def _zero_query(w):
    w["q_idx"].zero_()


@pytest.mark.parametrize("lens,k,mutate", [
    ((12000, 16500), 8000, _zero_query),       # all scores equal: the tie quota ends inside rank 1
    ((30000, 9000, 21000), 1024, _binary_keys),  # ties at the threshold in every part of 4
    ((60000, 45001), 4000, _binary_keys),        # ... of 8
])
def test_decode_ties_across_cluster_parts(lib, lens, k, mutate):
    """Ties at the k-th largest score spread over the CTAs of a selection
    cluster: each part keeps its ties only while their rank over the whole
    sequence is below the quota, so the lowest positions win."""
    _run(synth.small_spec(lens=lens, prefix_len=128, k=k, hq=8, hkv=2), mutate=mutate)


def test_decode_one_query_over_the_whole_grid(lib):
    """A single sequence whose attended rows are cut over every CTA of the
    persistent grid: over a hundred partials per head merged."""
    _run(synth.small_spec(lens=(9000,), prefix_len=1024, k=2048, hq=64, hkv=8))


def test_decode_fp32_output(lib):
    _run(synth.small_spec(lens=(1000, 2000)), out_dtype=torch.float32)


def test_decode_all_ties_take_lowest_positions(lib):
    """A zero indexer query makes every score 0: the k lowest candidates win."""
    def zero_q(w):
        w["q_idx"].zero_()
    res = _run(synth.small_spec(lens=(1500, 700)), mutate=zero_q)
    idx = res["idx"].cpu().numpy()
    assert np.array_equal(idx[0], np.arange(64, 64 + 256))


def test_decode_full_int8_range_uses_exact_fallback(lib):
    """Indexer values over the whole int8 range push scores far outside the
    1-wide histogram window; the exact radix fallback must take over."""
    _run(synth.small_spec(lens=(3000, 5000), idx_lo=-128, idx_hi=127))


def test_decode_extreme_scores_at_window_edge(lib):
    """All keys and the query at +8: every score is 4096, just outside the
    window (edge bin), with ties everywhere."""
    def extreme(w):
        w["q_idx"].fill_(8)
        w["idx_cache"].fill_(8)
    _run(synth.small_spec(lens=(700, 1300)), mutate=extreme)


def test_decode_outlier_keys(lib):
    _run(synth.small_spec(lens=(1500, 2500), outlier_frac=0.01))


def test_decode_deterministic(lib):
    spec = synth.small_spec(lens=(5000, 6000), k=512)
    w = H.on(synth.make_workload(spec, 5, "cpu"), DEV)
    a, b = H.run_decode_step(w), H.run_decode_step(w)
    for key in ("scores", "idx", "n_sel", "out", "lse"):
        assert torch.equal(a[key], b[key]), key


def test_workspace_left_clean_for_reuse(lib):
    """Calls leave their counters at zero: one workspace serves repeated calls."""
    import dynamic_sparse_attention_indexer_gb300 as dsa
    spec = synth.small_spec(lens=(3000, 4000))
    w_cpu = synth.make_workload(spec, 8, "cpu")
    w = H.on(w_cpu, DEV)
    res = H.run_decode_step(w)
    ws = res["ws"]
    kv = H.paged_kv(w)
    for _ in range(3):
        dsa.decode_step(kv, w["q"], w["q_idx"], 64, 256, res["scores"], res["idx"], res["n_sel"], res["out"],
                        res["lse"], ws)
    assert dsa.check_device_status() == 0
    H.check_decode_against_oracle(synth.to_numpy(w_cpu), res)


def test_kv_gather_bitwise(lib):
    import dynamic_sparse_attention_indexer_gb300 as dsa
    import oracle.dsa_oracle as O
    spec = synth.small_spec(lens=(900, 300), k=128)
    w_cpu = synth.make_workload(spec, 3, "cpu")
    w = H.on(w_cpu, DEV)
    res = H.run_decode_step(w)
    kv = H.paged_kv(w)
    rows = 64 + 128
    ko = torch.full((2, 2, rows, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    vo = torch.full_like(ko, 7.0)
    dsa.kv_gather(kv, dsa.decode_queries(kv), res["idx"], res["n_sel"], 128, 64, ko, vo)
    assert dsa.check_device_status() == 0
    wn = synth.to_numpy(w_cpu)
    for b in range(2):
        r = O.decode_query(wn, b)
        kr, vr = O.kv_gather(wn["k_cache"], wn["v_cache"], wn["block_table"][b], r["attended"], 2, rows)
        assert np.array_equal(ko[b].double().cpu().numpy(), kr)
        assert np.array_equal(vo[b].double().cpu().numpy(), vr)


def test_kv_write_scatter_bitwise(lib):
    import dynamic_sparse_attention_indexer_gb300 as dsa
    import oracle.dsa_oracle as O
    spec = synth.small_spec(lens=(500,), batch=1, spare_blocks=4)
    w_cpu = synth.make_workload(spec, 4, "cpu")
    w = H.on(w_cpu, DEV)
    kv = H.paged_kv(w)
    g = torch.Generator().manual_seed(0)
    n = 9
    nb = w_cpu["k_cache"].shape[0]
    slots = torch.randperm(nb * 64, generator=g)[:n].to(torch.int32)
    kn = torch.randn((n, 2, 128), generator=g).to(torch.bfloat16)
    vn = torch.randn((n, 2, 128), generator=g).to(torch.bfloat16)
    inn = torch.randint(-8, 9, (n, 64), generator=g, dtype=torch.int8)
    dsa.kv_write(kv, slots.to(DEV), kn.to(DEV), vn.to(DEV), inn.to(DEV))
    assert dsa.check_device_status() == 0
    wn = synth.to_numpy(w_cpu)
    kc, vc, ic = O.kv_write(wn["k_cache"], wn["v_cache"], wn["idx_cache"], slots.numpy(),
                            kn.double().numpy(), vn.double().numpy(), inn.numpy().astype(np.int64))
    assert np.array_equal(w["k_cache"].double().cpu().numpy(), kc)
    assert np.array_equal(w["v_cache"].double().cpu().numpy(), vc)
    assert np.array_equal(w["idx_cache"].cpu().numpy().astype(np.int64), ic)


def test_bad_block_table_sets_status_not_fault(lib):
    """A block id outside the pool is reported through the status word; the
    kernels read block 0 in its place and the context stays usable."""
    import dynamic_sparse_attention_indexer_gb300 as dsa
    spec = synth.small_spec(lens=(700, 900))
    w = H.on(synth.make_workload(spec, 2, "cpu"), DEV)
    w["block_table"][1, 3] = w["k_cache"].shape[0] + 5
    kv = H.paged_kv(w)
    scores = torch.zeros((2, 900), dtype=torch.int32, device=DEV)
    dsa.index_scores(kv, dsa.decode_queries(kv), w["q_idx"], 64, scores)
    assert dsa.check_device_status() == 4
    assert dsa.check_device_status() == 0    # read-and-clear
    torch.cuda.synchronize()


def test_bad_selected_position_sets_status_not_fault(lib):
    """The stand-alone attention call resolves the positions it is given: one
    outside the block table, or one whose block id lies outside the pool, is
    reported through the status word and read from block 0 instead."""
    import dynamic_sparse_attention_indexer_gb300 as dsa
    spec = synth.small_spec(lens=(700, 900))
    w = H.on(synth.make_workload(spec, 2, "cpu"), DEV)
    res = H.run_decode_step(w, split_api=True)
    kv = H.paged_kv(w)
    idx = res["idx"].clone()
    idx[0, 5] = 1 << 24                           # past max_blocks * 64
    dsa.sparse_attn_decode(kv, w["q"], idx, res["n_sel"], 256, 64, res["out"], res["lse"], res["ws"])
    assert dsa.check_device_status() == 4
    idx = res["idx"].clone()
    w["block_table"][1, int(idx[1, 0]) // 64] = w["k_cache"].shape[0] + 5
    dsa.sparse_attn_decode(kv, w["q"], idx, res["n_sel"], 256, 64, res["out"], res["lse"], res["ws"])
    assert dsa.check_device_status() == 4
    assert dsa.check_device_status() == 0
    torch.cuda.synchronize()


# ------------------------------------------------------- full-size workloads ---
def _full_size(cfg, sample_seqs, sample_heads):
    """The full workload in the launch configuration the bench times: scores
    and indices of EVERY sequence bit-exact against the oracle; attention
    output and lse against the oracle on sampled (sequence, KV head) pairs."""
    spec = synth.CONFIGS[cfg]
    w = synth.make_workload(spec, 1000 + cfg, DEV)
    res = H.run_decode_step(w)
    P, k = spec.prefix_len, spec.k
    idx = res["idx"].cpu().numpy()
    n_sel = res["n_sel"].cpu().numpy()
    scores = res["scores"].cpu().numpy()
    out = res["out"].float().cpu().numpy()
    lse = res["lse"].cpu().numpy()
    G = spec.num_q_heads // spec.num_kv_heads
    ref = H.oracle_indices_all(w, k, P)
    for b in range(spec.batch):
        r = ref[b]
        L = r["pos"] + 1
        assert np.array_equal(scores[b, P:L], r["scores"]), f"scores seq {b}"
        assert int(n_sel[b]) == r["n_sel"], f"n_sel seq {b}"
        assert np.array_equal(idx[b], r["idx"]), f"idx seq {b}"
    for b in sample_seqs:
        r = H.oracle_decode_sampled(w, b, sample_heads, k, P)
        for g, (o, s) in r["heads"].items():
            H.assert_close(out[b, g * G:(g + 1) * G], o, f"out seq {b} kv head {g}")
            H.assert_close(lse[b, g * G:(g + 1) * G], s, f"lse seq {b} kv head {g}")
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_full_decode_512(lib):
    _full_size(1, [0], [0])


def test_full_decode_8k(lib):
    _full_size(2, [0, 17, 31], [0, 3])


def test_full_decode_128k(lib):
    _full_size(3, [0, 5], [0, 7])


def test_full_decode_1m_ragged(lib):
    _full_size(5, [0, 3], [2])
