"""Local sliding-window attention (the hybrid attention's local sibling) on the
GPU against the CPU oracle: decode through the sparse attention kernels over
the window's positions, prefill through the masked dense tcgen05 pass with the
window as its mask."""
import numpy as np
import pytest
import torch

import harness as H
import oracle.dsa_oracle as O
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
dsa = H.dsa


def _decode(spec, window, out_dtype=torch.bfloat16, seed=7):
    w_cpu = synth.make_workload(spec, seed, "cpu")
    w = H.on(w_cpu, DEV)
    wn = synth.to_numpy(w_cpu)
    kv = H.paged_kv(w)
    B, hq = spec.batch, spec.num_q_heads
    out = torch.empty((B, hq, 128), dtype=out_dtype, device=DEV)
    lse = torch.empty((B, hq), dtype=torch.float32, device=DEV)
    ws = dsa.make_workspace(dsa.window_workspace_size(kv, hq, window), DEV)
    dsa.window_attn_decode(kv, w["q"], window, out, lse, ws)
    assert dsa.check_device_status() == 0
    out_h, lse_h = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        pos = int(wn["context_lens"][b]) - 1
        r = O.window_query(wn, pos, wn["q"][b], b, window)
        H.assert_close(out_h[b], r["out"], f"out of sequence {b}")
        H.assert_close(lse_h[b], r["lse"], f"lse of sequence {b}")


def _prefill(spec, window, out_dtype=torch.bfloat16, seed=7, rows=None, poison_tail=False):
    w_cpu = synth.make_workload(spec, seed, "cpu")
    w_cpu["seq"] = 0
    if poison_tail:  # slots of the last block past the chunk's last position hold NaN
        last = spec.pos0 + spec.num_queries - 1
        blk = int(w_cpu["block_table"][0, last // 64])
        w_cpu["kv"][blk, last % 64 + 1:] = float("nan")
    w = H.on(w_cpu, DEV)
    wn = synth.to_numpy(w_cpu)
    kv = H.paged_kv(w)
    T, hq = spec.num_queries, spec.num_q_heads
    qs = dsa.query_set(dsa.MODE_PREFILL, T, 0, spec.pos0)
    out = torch.empty((T, hq, 128), dtype=out_dtype, device=DEV)
    lse = torch.empty((T, hq), dtype=torch.float32, device=DEV)
    dsa.window_attn_prefill(kv, qs, w["q"], window, out, lse)
    assert dsa.check_device_status() == 0
    out_h, lse_h = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(out_h).all() and np.isfinite(lse_h).all()
    for i in (range(T) if rows is None else rows):
        r = O.window_query(wn, spec.pos0 + i, wn["q"][i], 0, window)
        H.assert_close(out_h[i], r["out"], f"out of query {i}")
        H.assert_close(lse_h[i], r["lse"], f"lse of query {i}")


@pytest.mark.parametrize("window", [1, 37, 64, 200, 5000])
def test_window_decode(lib, window):
    """Contexts shorter than, equal to and longer than the window."""
    spec = synth.small_spec(lens=(1, 37, 64, 65, 200, 777, 3000, 4999), batch=8, prefix_len=0, hq=8, hkv=2, k=8)
    _decode(spec, window)


def test_window_decode_group_16_fp32(lib):
    spec = synth.small_spec(lens=(500, 1300), batch=2, prefix_len=0, hq=32, hkv=2, k=8)
    _decode(spec, 300, out_dtype=torch.float32)


def _pspec(T, pos0, hq=8, hkv=2, **kw):
    return synth.Spec("window-prefill", "prefill", 1, (pos0 + T,), 0, hq, hkv, 8, num_queries=T, pos0=pos0, **kw)


@pytest.mark.parametrize("window", [1, 37, 128, 1000])
@pytest.mark.parametrize("pos0", [0, 500])
def test_window_prefill(lib, window, pos0):
    """Windows inside one block, across blocks, a whole step, and longer than
    the context; a chunk from position 0 and a continuation chunk."""
    _prefill(_pspec(300, pos0), window)


@pytest.mark.parametrize("hq,hkv", [(24, 8), (32, 2), (4, 4)])
def test_window_prefill_groups(lib, hq, hkv):
    """Tiles of 42 queries (group 3, two unused rows), 8 (group 16) and 128 (group 1)."""
    _prefill(_pspec(260, 70, hq=hq, hkv=hkv), 100)


def test_window_prefill_fp32_separate_arrays_unwritten_tail(lib):
    _prefill(_pspec(200, 33, kv_layout="adjacent"), 90, out_dtype=torch.float32, poison_tail=True)
    _prefill(_pspec(200, 33, kv_layout="separate"), 90)


def test_window_prefill_long_context(lib):
    """A 2048-query chunk deep into a 12K context with a 3000-position window
    (the dense pass starts each tile pair at its first window block), sampled
    rows plus the first and last."""
    rows = sorted(set(np.random.default_rng(3).integers(0, 2048, size=48).tolist()) | {0, 1, 2047})
    _prefill(_pspec(2048, 10000, hq=32, hkv=4), 3000, rows=rows)
