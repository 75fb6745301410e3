"""Decode with one indexer head per KV head on the GPU against the CPU oracle:
each KV head's scores and selection bit-exact, its query heads' attention
over the prefix plus that selection within tolerance."""
import numpy as np
import pytest
import torch

import harness as H
import oracle.dsa_oracle as O
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
dsa = H.dsa


def _run(spec, seed=5, out_dtype=torch.bfloat16, seqs=None):
    w_cpu = synth.make_workload(spec, seed, "cpu")
    w = H.on(w_cpu, DEV)
    wn = synth.to_numpy(w_cpu)
    kv = H.paged_kv(w)
    B, hq, hkv, k, P = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.k, spec.prefix_len
    ld = H.round4(int(max(w_cpu["context_lens"])))
    scores = torch.zeros((B * hkv, ld), dtype=torch.int32, device=DEV)
    idx = torch.full((B, hkv, k), -7, dtype=torch.int32, device=DEV)
    n_sel = torch.full((B, hkv), -7, dtype=torch.int32, device=DEV)
    out = torch.empty((B, hq, 128), dtype=out_dtype, device=DEV)
    lse = torch.empty((B, hq), dtype=torch.float32, device=DEV)
    ws = dsa.make_workspace(dsa.heads_workspace_size(kv, hq, k, P), DEV)
    dsa.decode_step_heads(kv, w["q"], w["q_idx"], P, k, scores, idx, n_sel, out, lse, ws,
                          block_table_heads=w.get("block_table_heads"))
    assert dsa.check_device_status() == 0
    sc, ix, ns = scores.cpu().numpy(), idx.cpu().numpy(), n_sel.cpu().numpy()
    o, ls = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in (range(B) if seqs is None else seqs):
        r = O.decode_query_heads(wn, b)
        pos = int(wn["context_lens"][b]) - 1
        for g in range(hkv):
            if pos >= P:
                assert np.array_equal(sc[b * hkv + g, P:pos + 1], r["scores"][g]), f"scores of sequence {b} head {g}"
            assert int(ns[b, g]) == r["n_sel"][g], f"n_sel of sequence {b} head {g}"
            assert np.array_equal(ix[b, g], r["idx"][g]), f"idx of sequence {b} head {g}"
        H.assert_close(o[b], r["out"], f"out of sequence {b}")
        H.assert_close(ls[b], r["lse"], f"lse of sequence {b}")


@pytest.mark.parametrize("hq,hkv", [(8, 2), (16, 4), (32, 2), (8, 8)])
def test_heads_small(lib, hq, hkv):
    """Contexts inside the prefix, at its edge, with fewer and more candidates
    than k, over groups of 4, 4, 16 and 1 query heads."""
    spec = synth.small_spec(lens=(40, 64, 65, 300, 777, 1500), batch=6, prefix_len=64, hq=hq, hkv=hkv, k=100,
                            idx_heads=hkv)
    _run(spec)


def test_heads_fp32_separate_arrays_full_int8(lib):
    spec = synth.small_spec(lens=(900, 2113), batch=2, prefix_len=32, hq=16, hkv=4, k=64, idx_heads=4,
                            kv_layout="separate", idx_lo=-128, idx_hi=127)
    _run(spec, out_dtype=torch.float32)


def test_heads_32k(lib):
    """B = 4 sequences of 32K positions, 8 KV heads: 32 (sequence, head)
    selections of k = 2048 from ~31.7K candidates each, every one bit-exact."""
    spec = synth.Spec("heads 32K", "decode", 4, (32768, 30000, 32768, 17000), 1024, 64, 8, 2048, idx_heads=8)
    _run(spec)


@pytest.mark.parametrize("hq,hkv,layout", [(8, 2, "adjacent"), (64, 8, "adjacent"), (16, 4, "separate")])
def test_heads_per_head_block_tables(lib, hq, hkv, layout):
    """One block table per KV head (the allocator's per-head block bitmaps):
    each head reads its indexer keys, K and V from the head slices of the blocks
    its own table names, which hold other sequences' positions for the other
    heads.  Contexts inside and at the edge of the prefix, and a long one."""
    spec = synth.small_spec(lens=(40, 64, 65, 777, 20000), batch=5, prefix_len=64, hq=hq, hkv=hkv, k=100,
                            idx_heads=hkv, head_tables=True, kv_layout=layout)
    _run(spec)


def test_kv_write_heads_bitwise(lib):
    """Per-head cache write against the oracle, bitwise: each head's K, V and
    indexer key in its own slot's head slice, with two heads of one token sent
    to the same slot and heads of different tokens sharing blocks."""
    spec = synth.small_spec(lens=(500,), batch=1, hkv=4, hq=16, idx_heads=4, spare_blocks=4)
    w_cpu = synth.make_workload(spec, 4, "cpu")
    w = H.on(w_cpu, DEV)
    kv = H.paged_kv(w)
    g = torch.Generator().manual_seed(1)
    n, hkv = 9, 4
    nb = w_cpu["k_cache"].shape[0]
    slots = torch.stack([torch.randperm(nb * 64, generator=g)[:n] for _ in range(hkv)], dim=1).to(torch.int32)
    slots[0, 1] = slots[0, 0]  # two heads of one token, one slot
    # within a head no slot repeats, so the order of the writes does not matter
    assert all(len(set(slots[:, h].tolist())) == n for h in range(hkv))
    kn = torch.randn((n, hkv, 128), generator=g).to(torch.bfloat16)
    vn = torch.randn((n, hkv, 128), generator=g).to(torch.bfloat16)
    inn = torch.randint(-8, 9, (n, hkv, 64), generator=g, dtype=torch.int8)
    dsa.kv_write_heads(kv, slots.to(DEV), kn.to(DEV), vn.to(DEV), inn.to(DEV))
    assert dsa.check_device_status() == 0
    wn = synth.to_numpy(w_cpu)
    kc, vc, ic = O.kv_write_heads(wn["k_cache"], wn["v_cache"], wn["idx_cache"], slots.numpy(),
                                  kn.double().numpy(), vn.double().numpy(), inn.numpy().astype(np.int64))
    assert np.array_equal(w["k_cache"].double().cpu().numpy(), kc)
    assert np.array_equal(w["v_cache"].double().cpu().numpy(), vc)
    assert np.array_equal(w["idx_cache"].cpu().numpy().astype(np.int64), ic)


def test_heads_bad_block_ids_set_status_not_fault(lib):
    """A block id outside the pool in a head's own block table, and a per-head
    write slot outside it, are reported through the status word: the kernels
    read block 0 in its place (or skip the write) and the context stays usable
    (a valid call right after gives results equal to the oracle's)."""
    spec = synth.small_spec(lens=(300, 900), batch=2, prefix_len=64, hq=8, hkv=2, k=40, idx_heads=2,
                            head_tables=True)
    w = H.on(synth.make_workload(spec, 3, "cpu"), DEV)
    kv = H.paged_kv(w)
    nb = w["k_cache"].shape[0]
    bad = w["block_table_heads"].clone()
    bad[1, 1, 5] = nb + 5  # head 1, sequence 1, block-table entry 5 (positions 320-383)
    ld = H.round4(int(w["max_context_len"]))
    scores = torch.zeros((2 * 2, ld), dtype=torch.int32, device=DEV)
    idx = torch.empty((2, 2, 40), dtype=torch.int32, device=DEV)
    n_sel = torch.empty((2, 2), dtype=torch.int32, device=DEV)
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device=DEV)
    ws = dsa.make_workspace(dsa.heads_workspace_size(kv, 8, 40, 64), DEV)
    dsa.decode_step_heads(kv, w["q"], w["q_idx"], 64, 40, scores, idx, n_sel, out, None, ws, block_table_heads=bad)
    assert dsa.check_device_status() == 4  # DSA_ERR_BAD_BLOCK_TABLE
    slots = torch.tensor([[nb * 64 + 3, 5]], dtype=torch.int32, device=DEV)  # head 0's slot outside the pool
    kn = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device=DEV)
    dsa.kv_write_heads(kv, slots, kn, kn, torch.zeros((1, 2, 64), dtype=torch.int8, device=DEV))
    assert dsa.check_device_status() == 4  # DSA_ERR_BAD_BLOCK_TABLE
    assert dsa.check_device_status() == 0  # read and cleared
    _run(spec, seed=3)  # the context is usable: a valid call matches the oracle
