"""The allocation-free decode top-k against the workspace version.

dsa_topk_select_decode_noalloc serves callers that cannot allocate device
memory (a plugin inside a process whose device memory belongs to the host
framework's pool, with no allocator handed to it; a path that cannot afford
cudaMalloc's synchronisation).  Its scratch is a static array inside the
library, shared by every call and keeping the last call's contents, so the
test makes calls back to back with different inputs and checks each result
against dsa_topk_select, bit for bit (indices admit no tolerance).

This file is named to be collected last; it must pass on its own in a fresh
process (the first call on the device sets the scratch up) and after the
other tests.
"""
import ctypes as C

import pytest
import torch

import harness as H
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _scores(spec, seed):
    import dynamic_sparse_attention_indexer_gb300 as dsa
    w = H.on(synth.make_workload(spec, seed, "cpu"), DEV)
    kv = H.paged_kv(w)
    ld = H.round4(w["max_context_len"])
    scores = torch.zeros((kv.batch, ld), dtype=torch.int32, device=DEV)
    dsa.index_scores(kv, dsa.decode_queries(kv), w["q_idx"], spec.prefix_len, scores)
    return w, kv, scores


def _with_workspace(kv, scores, spec):
    import dynamic_sparse_attention_indexer_gb300 as dsa
    qs = dsa.decode_queries(kv)
    ws = dsa.make_workspace(dsa.workspace_size(dsa.OP_TOPK_SELECT, kv, qs, spec.k, spec.num_q_heads,
                                               spec.prefix_len), DEV)
    idx = torch.empty((kv.batch, spec.k), dtype=torch.int32, device=DEV)
    n_sel = torch.empty(kv.batch, dtype=torch.int32, device=DEV)
    dsa.topk_select(kv, qs, scores, spec.prefix_len, spec.k, idx, n_sel, ws)
    return idx, n_sel


def _no_alloc(lib, kv, scores, spec):
    idx = torch.full((kv.batch, spec.k), 12345, dtype=torch.int32, device=DEV)
    n_sel = torch.full((kv.batch,), 12345, dtype=torch.int32, device=DEV)
    st = lib.dsa_topk_select_decode_noalloc(kv.ref, scores.data_ptr(), scores.stride(0), spec.prefix_len,
                                            spec.k, idx.data_ptr(), n_sel.data_ptr(),
                                            C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.dsa_last_error_message().decode()
    return idx, n_sel


def test_no_alloc_topk_matches_workspace_version(lib):
    import dynamic_sparse_attention_indexer_gb300 as dsa
    spec_a = synth.small_spec(lens=(20000, 700, 9000, 13000), prefix_len=64, k=512, hq=8, hkv=2)
    spec_b = synth.small_spec(lens=(5000, 30001), prefix_len=128, k=1000, hq=8, hkv=2)
    wa, kva, sa = _scores(spec_a, 21)
    wb, kvb, sb = _scores(spec_b, 22)
    ref_a = _with_workspace(kva, sa, spec_a)
    ref_b = _with_workspace(kvb, sb, spec_b)
    # Back-to-back calls on the shared static scratch, alternating inputs.
    for kv, s, spec, ref in ((kva, sa, spec_a, ref_a), (kvb, sb, spec_b, ref_b), (kva, sa, spec_a, ref_a)):
        idx, n_sel = _no_alloc(lib, kv, s, spec)
        torch.cuda.synchronize()
        assert torch.equal(n_sel, ref[1])
        assert torch.equal(idx, ref[0])
    assert dsa.check_device_status() == 0
