"""Run-to-run determinism: the same inputs give bit-identical outputs.

Every reduction of the hot path has a fixed order (the stream-K ranges and the
merge of their partial states are functions of the shapes only; the top-k's
compaction is ordered; the dense prefill pass walks fixed tiles), so two calls
on the same inputs must agree bit for bit, not only within the tolerance."""
import pytest
import torch

import harness as H
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _same(a: dict, b: dict, keys):
    for key in keys:
        assert torch.equal(a[key], b[key]), f"{key} differs between two identical calls"


@pytest.mark.parametrize("lens", [(300, 5000, 1, 2049), (9000, 9000, 9000, 9000)])
def test_decode_step_repeats_bitwise(lens):
    spec = synth.small_spec(lens=lens, batch=len(lens), prefix_len=64, hq=16, hkv=2, k=256)
    w = H.on(synth.make_workload(spec, 21, "cpu"), DEV)
    r1 = H.run_decode_step(w)
    r2 = H.run_decode_step(w)
    torch.cuda.synchronize()
    _same(r1, r2, ("scores", "idx", "n_sel", "out", "lse"))


def test_decode_split_calls_repeat_bitwise():
    spec = synth.small_spec(lens=(4000, 777, 12000), batch=3, prefix_len=128, hq=32, hkv=4, k=512)
    w = H.on(synth.make_workload(spec, 22, "cpu"), DEV)
    r1 = H.run_decode_step(w, split_api=True)
    r2 = H.run_decode_step(w, split_api=True)
    torch.cuda.synchronize()
    _same(r1, r2, ("scores", "idx", "n_sel", "out", "lse"))


def test_prefill_step_repeats_bitwise():
    spec = synth.Spec("prefill-det", "prefill", 1, (1500,), 128, 16, 2, 256, num_queries=700, pos0=800)
    w_cpu = synth.make_workload(spec, 23, "cpu")
    w_cpu["seq"] = 0
    w = H.on(w_cpu, DEV)
    r1 = H.run_prefill_step(w)
    r2 = H.run_prefill_step(w)
    torch.cuda.synchronize()
    keys = [k for k in ("scores", "idx", "n_sel", "out", "lse") if k in r1]
    _same(r1, r2, keys)
