"""DSA decode benchmark on GB300: tokens/s and achieved HBM bandwidth.

One step = one full DSA decode step of one attention layer over the batch:
indexer scores -> top-k (prefix forced in) -> fused gather + GQA attention,
for the decode workload B=8, context 131072, prefix 1024, 64/8 heads,
head_dim 128, int8 indexer dim 64, top-k 2048, 1% of K rows scaled x4.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Inputs are synthetic and seeded; they are resident in HBM before timing.
Consecutive steps rotate over 4 independent KV caches ("layers", 17.6 GB in
all), so no step finds its data in the 129 MB L2.  Multi-GPU runs (torchrun)
give every rank its own batch (weak scaling, no collective on the data path).
The same line also carries the 16K prefill chunk (scores, top-k, attention,
timed per call) with the peak rates it is compared against, measured in the
same run by the microbenchmarks of libdsa_probe.so.  The reference arm
(--impl reference) times the CPU oracle on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)

CONFIG_ID = 3
PREFILL_ID = 4
LAYERS = 4
METRIC = "DSA decode tokens/s & achieved HBM GB/s (% of roofline) at 128K ctx, 1xGB300"


# ------------------------------------------------------------ helpers ------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def algorithmic_bytes(spec, lens, n_sel):
    """Bytes the method must move per step (HBM): non-prefix indexer keys and
    their block-table entries, the indexer query, selected K and V rows (prefix
    + selection, every KV head), Q, the output, and the index list."""
    P, hkv, hq = spec.prefix_len, spec.num_kv_heads, spec.num_q_heads
    idx_bytes = sum(max(0, L - P) * 64 + math.ceil(L / 64) * 4 for L in lens) + 64 * len(lens)
    rows = sum(min(P, L) + int(n) for L, n in zip(lens, n_sel))
    kv_bytes = rows * hkv * 2 * 128 * 2
    qo_bytes = 2 * len(lens) * hq * 128 * 2 + len(lens) * hq * 4
    sel_bytes = len(lens) * spec.k * 4
    return {"indexer": idx_bytes, "attention": kv_bytes + qo_bytes + sel_bytes, "step":
            idx_bytes + kv_bytes + qo_bytes + sel_bytes}


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def code_digest(path):
    """sha256 of a source file's code: // comments and blank lines removed, so
    that comment edits do not count as a change of the kernel."""
    import hashlib
    import re
    lines = []
    for line in open(path).read().splitlines():
        code = re.sub(r"//.*$", "", line).rstrip()
        if code.strip():
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


WINDOW = 4096  # positions of the sliding-window sibling the bench times


def window_decode_line(spec, lens, ms, peak, peak_kind):
    """Decode window attention (each sequence's newest token over its last
    WINDOW positions) against the bytes it must move: the K and V rows of the
    window for every KV head, Q and the bf16 output."""
    rows = sum(min(WINDOW, int(L)) for L in lens)
    nbytes = rows * spec.num_kv_heads * 512 + 2 * len(lens) * spec.num_q_heads * 128 * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "dsa_window_attn_decode per call in a graph: sparse_attn_kernel (the window's rows "
                      "walked from each context's end) + attn_combine_kernel", "window": WINDOW, "ms": ms, "bound": "hbm", "achieved": gbs,
            "peak": peak, "unit": "GB/s", "frac": gbs / peak, "algorithmic_bytes": nbytes, "peak_kind": peak_kind}


def heads_decode_line(spec, lens, n_sel_heads, ms, peak, peak_kind):
    """The decode step with one indexer head per KV head against the bytes it
    must move: every KV head's non-prefix indexer keys and its indexer query,
    the block-table entries, each KV head's own K and V rows (prefix plus its
    selection), Q, the bf16 output and the index lists."""
    P, hkv, hq = spec.prefix_len, spec.num_kv_heads, spec.num_q_heads
    idx_bytes = sum(max(0, L - P) * 64 * hkv + math.ceil(L / 64) * 4 for L in lens) + 64 * hkv * len(lens)
    rows = sum(min(P, L) + int(n) for L, ns in zip(lens, n_sel_heads) for n in ns)
    nbytes = idx_bytes + rows * 512 + 2 * len(lens) * hq * 128 * 2 + len(lens) * hkv * spec.k * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "dsa_decode_step_heads per call in a graph: the scoring, selection, attention and merge "
                      "kernels over (sequence, KV head) rows", "ms": ms,
            "tokens_per_s": len(lens) / (ms * 1e-3), "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
            "frac": gbs / peak, "algorithmic_bytes": nbytes, "peak_kind": peak_kind}


def profiled_attention_traffic():
    """DRAM bytes per attention call from the committed ncu record
    (profiles/decode_128k_traffic.json), or None once the attention code has
    changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "decode_128k_traffic.json")
    src = os.path.join(ROOT, "dynamic_sparse_attention_indexer_gb300", "csrc", "k_attn.cu")
    try:
        with open(path) as f:
            rec = json.load(f)
        digest = code_digest(src)
    except (OSError, ValueError):
        return None
    if rec.get("code_sha256_k_attn") != digest:
        return None
    return int(rec["traffic_bytes_per_call"])


def reduce_over_ranks(values: dict, op: str):
    """Max ("max") or sum ("sum") of scalar values over all ranks (no-op
    without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return dict(values)
    keys = sorted(values)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(values[k]) for k in keys], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return {k: float(v) for k, v in zip(keys, t.cpu().tolist())}


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------- oracle timing -----
def oracle_sequence_inputs(w, b):
    """Per-sequence CPU copies (not timed): indexer, K and V blocks of seq b."""
    import numpy as np
    import torch
    L = int(w["context_lens"][b].item())
    nblk = math.ceil(L / 64)
    ids = w["block_table"][b, :nblk].long()
    local_bt = np.arange(nblk, dtype=np.int64)
    icache = w["idx_cache"].index_select(0, ids).cpu().numpy().astype(np.int64)
    kc = w["k_cache"].index_select(0, ids).cpu().to(torch.float32).numpy()
    vc = w["v_cache"].index_select(0, ids).cpu().to(torch.float32).numpy()
    return {"q": w["q"][b].cpu().to(torch.float64).numpy(), "q_idx": w["q_idx"][b].cpu().numpy().astype(np.int64),
            "idx_cache": icache, "k_cache": kc, "v_cache": vc, "bt": local_bt, "pos": L - 1}


def time_oracle(seq_inputs, spec):
    """Seconds the oracle takes for the given decode tokens (single thread)."""
    import oracle.dsa_oracle as O
    t0 = time.perf_counter()
    for d in seq_inputs:
        O.dsa_query(d["q"], d["q_idx"], d["k_cache"], d["v_cache"], d["idx_cache"], d["bt"], d["pos"],
                    spec.prefix_len, spec.k, spec.num_kv_heads, 1.0 / math.sqrt(128))
    return time.perf_counter() - t0


def cpu_threads_used():
    # numpy's BLAS is limited to one thread before numpy loads (see main); the
    # int64 scoring and the sort are single threaded in numpy anyway.
    return 1


def _export_sequence(w, b, d, tag):
    """Sequence b's oracle inputs as .npy files in directory d (not timed):
    query, indexer query, indexer blocks (int8), K and V blocks (bf16 bits)."""
    import numpy as np
    import torch
    L = int(w["context_lens"][b].item())
    nblk = math.ceil(L / 64)
    ids = w["block_table"][b, :nblk].long()
    paths = {}
    arrays = {"q": w["q"][b].cpu().to(torch.float64).numpy(),
              "q_idx": w["q_idx"][b].cpu().numpy().astype(np.int64),
              "idx_cache": w["idx_cache"].index_select(0, ids).cpu().numpy(),
              "k16": w["k_cache"].index_select(0, ids).view(torch.int16).cpu().numpy().view(np.uint16),
              "v16": w["v_cache"].index_select(0, ids).view(torch.int16).cpu().numpy().view(np.uint16)}
    for name, arr in arrays.items():
        paths[name] = os.path.join(d, f"{tag}_{name}.npy")
        np.save(paths[name], arr)
    paths["pos"] = L - 1
    paths["nblk"] = nblk
    return paths


def _oracle_worker(task):
    """One host process: loads one sequence's inputs, waits for the common
    start time, then runs the oracle on that decode token repeatedly for
    `seconds`.  Returns (tokens, seconds)."""
    import numpy as np
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import oracle.dsa_oracle as O
    paths, prefix, k, hkv, start_at, seconds = task
    q = np.load(paths["q"])
    q_idx = np.load(paths["q_idx"])
    idx = np.load(paths["idx_cache"], mmap_mode="r")
    kc = (np.load(paths["k16"]).astype(np.uint32) << 16).view(np.float32)   # bf16 -> fp32, exact
    vc = (np.load(paths["v16"]).astype(np.uint32) << 16).view(np.float32)
    bt = np.arange(paths["nblk"], dtype=np.int64)
    while time.time() < start_at:
        time.sleep(0.005)
    n, t0 = 0, time.perf_counter()
    while True:
        O.dsa_query(q, q_idx, kc, vc, idx, bt, paths["pos"], prefix, k, hkv, 1.0 / math.sqrt(128))
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return n, el


def cpu_baseline_all_cores(w, spec, seconds, n_seq=4):
    """The oracle as it stands on every host core at once: one process per
    core (spawned), each repeating one decode token of the workload (the
    sequences taken in turn).  Throughput = sum of the per-process rates over
    the same time window."""
    import multiprocessing as mp
    import shutil
    import tempfile
    base = "/dev/shm" if os.path.isdir("/dev/shm") else None
    d = tempfile.mkdtemp(prefix="dsa_oracle_", dir=base)
    try:
        seqs = [_export_sequence(w, b, d, f"s{b}") for b in range(min(n_seq, spec.batch))]
        cores = os.cpu_count() or 1
        start_at = time.time() + 4.0 + 0.2 * cores  # after every process has loaded its inputs
        tasks = [(seqs[i % len(seqs)], spec.prefix_len, spec.k, spec.num_kv_heads, start_at, seconds)
                 for i in range(cores)]
        with mp.get_context("spawn").Pool(cores) as pool:
            res = pool.map(_oracle_worker, tasks)
    finally:
        shutil.rmtree(d, ignore_errors=True)
    tokens = sum(n for n, _ in res)
    rate = sum(n / el for n, el in res)
    return {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes, one per host core, each repeating one decode token of the workload "
                      f"({len(seqs)} sequences in turn) for {seconds:.0f} s: {tokens} tokens"}


class Probes:
    """Peak-rate microbenchmarks (libdsa_probe.so), timed with CUDA events on
    the current stream."""

    def __init__(self, dev):
        import ctypes as C
        import torch
        from dynamic_sparse_attention_indexer_gb300 import _build
        _build.ensure_built()
        lib = C.CDLL(_build.PROBE_LIB)
        for fn in ("probe_mma_s8", "probe_mma_bf16"):
            getattr(lib, fn).restype = C.c_float
            getattr(lib, fn).argtypes = [C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        lib.probe_tc.restype = C.c_float
        lib.probe_tc.argtypes = [C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        lib.probe_gather.restype = C.c_float
        lib.probe_gather.argtypes = [C.c_void_p, C.c_ulonglong, C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                     C.c_void_p]
        self.lib, self.dev = lib, dev
        self.sink = torch.zeros(4, dtype=torch.int32, device=dev)
        self.sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def _stream(self):
        import ctypes as C
        import torch
        return C.c_void_p(torch.cuda.current_stream(self.dev).cuda_stream)

    def mma_tops(self, kind):
        """Best of 5: int8 TOPS (kind "s8", m16n8k32) or bf16 TFLOP/s ("bf16", m16n8k16) of mma.sync."""
        fn, ops = (self.lib.probe_mma_s8, 8192) if kind == "s8" else (self.lib.probe_mma_bf16, 4096)
        ctas, iters = 4 * self.sms, 20000
        fn(ctas, 200, self.sink.data_ptr(), self._stream())
        best = min(fn(ctas, iters, self.sink.data_ptr(), self._stream()) for _ in range(5))
        return ctas * 8 * iters * 8 * ops / (best * 1e-3) / 1e12

    def tc_tops(self, f8):
        """Best of 5: TOPS (e4m3, f8=True) or TFLOP/s (f16) of back-to-back
        tcgen05.mma 128 x 256 tiles, one CTA per SM."""
        k = 32 if f8 else 16
        iters = 20000
        self.lib.probe_tc(int(f8), self.sms, 200, self.sink.data_ptr(), self._stream())
        best = min(self.lib.probe_tc(int(f8), self.sms, iters, self.sink.data_ptr(), self._stream())
                   for _ in range(5))
        assert int(self.sink.sum().item()) == 0, "tensor-core probe wait ran out"
        return self.sms * iters * 2 * 128 * 256 * k / (best * 1e-3) / 1e12

    def gather_gbs(self, piece, region_bytes=32 << 20):
        """Best of 5: GB/s of random `piece`-byte bulk copies into shared memory
        from a buffer of region_bytes (L2-resident), four issuing warps and
        three 64 KB stages per SM."""
        import torch
        buf = torch.ones(region_bytes // 4, dtype=torch.int32, device=self.dev)
        n_pieces = region_bytes // piece
        iters = 400
        args = (buf.data_ptr(), n_pieces, piece, 3, self.sms, iters, self.sink.data_ptr(), self._stream())
        self.lib.probe_gather(*args)
        best = min(self.lib.probe_gather(*args) for _ in range(5))
        assert int(self.sink.sum().item()) == 0, "gather probe wait ran out"
        return self.sms * iters * 65536 / (best * 1e-3) / 1e9


def measure_prefill(dev, steps, warmup, probes, cpu_seconds):
    """The 16K prefill chunk (T = 16384 causal queries against the same 16384
    positions, 32/4 heads, prefix 576, k = 2048): scores, top-k and attention,
    each call timed with CUDA events on the stream it runs on, with clocks
    sampled during the timed calls; the peaks it is compared against, measured
    now; and the oracle on sampled query rows (one host thread)."""
    import numpy as np
    import torch
    import dynamic_sparse_attention_indexer_gb300 as dsa
    import harness as H
    import synth
    spec = synth.CONFIGS[PREFILL_ID]
    w = synth.make_workload(spec, 1000 + PREFILL_ID, dev)
    kv = H.paged_kv(w)
    T, k, P, hq, hkv = spec.num_queries, spec.k, spec.prefix_len, spec.num_q_heads, spec.num_kv_heads
    qs = dsa.query_set(dsa.MODE_PREFILL, T, 0, 0)
    ld = H.round4(T)
    scores = torch.zeros((T, ld), dtype=torch.int32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(T, dtype=torch.int32, device=dev)
    out = torch.empty((T, hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, hq), dtype=torch.float32, device=dev)
    ws = dsa.make_workspace(dsa.workspace_size(dsa.OP_PREFILL_STEP, kv, qs, k, hq, P), dev)
    n_dense = dsa.prefill_dense_queries(kv, qs, k, hq, P)
    ws_gather = dsa.make_workspace(dsa.prefill_attn_workspace_size(kv, qs, k, hq, P, 0), dev)
    out_g = torch.empty_like(out)
    calls = {"index": lambda: dsa.index_scores(kv, qs, w["q_idx"], P, scores),
             "topk": lambda: dsa.topk_select(kv, qs, scores, P, k, idx, n_sel, ws),
             "attention": lambda: dsa.sparse_attn_prefill(kv, qs, w["q"], idx, n_sel, k, P, out, lse, ws),
             # the same attention with every query gathered (the path the automatic split
             # keeps for positions past its range), for comparison; not part of the chunk
             "attention_gather_only": lambda: dsa.sparse_attn_prefill(kv, qs, w["q"], idx, n_sel, k, P, out_g,
                                                                      None, ws_gather, n_dense=0),
             # the local sliding-window sibling on the same chunk, not part of it
             "window": lambda: dsa.window_attn_prefill(kv, qs, w["q"], WINDOW, out_g),
             # scores + top-k in one kernel, the scores never written (same indices;
             # not part of the chunk, which takes the faster separate calls)
             "select_fused": lambda: dsa.prefill_select(kv, qs, w["q_idx"], P, k, idx_f, n_sel_f),
             # the whole chunk in one call: scores, top-k writing the dense pass's
             # bitmap, attention (the chunk's time)
             "step": lambda: dsa.prefill_step(kv, qs, w["q"], w["q_idx"], P, k, scores, idx, n_sel, out, lse,
                                              ws_step)}
    ws_step = dsa.make_workspace(dsa.prefill_attn_workspace_size(kv, qs, k, hq, P, -1), dev)
    idx_f = torch.empty_like(idx)
    n_sel_f = torch.empty_like(n_sel)
    st = torch.cuda.current_stream(dev)
    for _ in range(max(1, warmup)):
        for f in calls.values():
            f()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    ms = {}
    for name, f in calls.items():
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(steps):
            f()
        b.record(st)
        b.synchronize()
        ms[name] = a.elapsed_time(b) / steps
    clock_info = clocks.stop()
    assert dsa.check_device_status(dev) == 0
    total = ms["step"]  # the chunk: one prefill_step call (the separate calls sum to index + topk + attention)
    pos = np.arange(T)
    causal_pairs = int(np.maximum(0, pos + 1 - P).sum())          # scored (query, key) pairs
    n_sel_h = n_sel.cpu().numpy().astype(np.int64)
    gathered = int(n_sel_h.sum()) * hkv * 2 * 128 * 2                # selected K and V rows, every KV head
    s8 = probes.mma_tops("s8")
    bf16 = probes.mma_tops("bf16")
    f8 = probes.tc_tops(True)
    f16 = probes.tc_tops(False)
    gather = probes.gather_gbs(hkv * 128 * 2)
    idx_tops = 2 * 64 * causal_pairs / (ms["index"] * 1e-3) / 1e12
    # The indexer stores a 4-byte score per scored pair and reads the indexer
    # rows of the query and key tiles: it is bound by HBM, not by the tensor cores.
    idx_bytes = 4 * causal_pairs + T * 64 + (T * 64) * ((T + 127) // 128) // 2
    peak_hbm, peak_kind = measured_peaks()
    idx_gbs = idx_bytes / (ms["index"] * 1e-3) / 1e9
    gather_gbs = gathered / (ms["attention_gather_only"] * 1e-3) / 1e9
    # Tensor work of the dense masked pass as it runs: per KV head and pair of
    # query tiles (2 x floor(128 / G) queries), every 64-position block up to the
    # pair's last position, per tile S = Q K^T (128 x 64 x 128) and O += P V with
    # P as hi + lo (two 128 x 128 x 64 products): 3 x 2 x 128 x 64 x 128 flops.
    G = hq // hkv
    qt = 128 // G
    dense_flops = 0
    for q0 in range(0, n_dense, 2 * qt):
        last = min(q0 + 2 * qt, n_dense) - 1
        dense_flops += ((last // 64) + 1) * 2 * 3 * 2 * 128 * 64 * 128 * hkv
    dense_tflops = dense_flops / (ms["attention"] * 1e-3) / 1e12 if n_dense == T else None
    attended = int(n_sel_h.sum()) + int(np.minimum(pos + 1, P).sum())
    useful_flops = 4 * attended * 128 * hq                           # Q.K and P.V over the attended rows
    # the window form: each tile pair from the block of its first window position
    win_flops = 0
    for q0 in range(0, T, 2 * qt):
        last = min(q0 + 2 * qt, T) - 1
        c_begin = max(0, q0 - WINDOW + 1) // 64
        blocks = last // 64 + 1 - c_begin
        win_flops += ((blocks + 1) // 2) * 2 * 3 * 2 * 128 * 128 * 128 * hkv  # steps x tiles x products
    win_tflops = win_flops / (ms["window"] * 1e-3) / 1e12
    # oracle on sampled rows of the chunk (rows drawn uniformly, seeded)
    cpu = None
    if cpu_seconds > 0:
        import oracle.dsa_oracle as O
        wn = synth.to_numpy(w)
        rows = np.random.default_rng(4).integers(0, T, size=4096)
        n, t0 = 0, time.perf_counter()
        while n < len(rows) and (n < 4 or time.perf_counter() - t0 < cpu_seconds):
            O.prefill_query(wn, int(rows[n]))
            n += 1
        el = time.perf_counter() - t0
        cpu = {"value": n / el, "unit": "query rows/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} query rows of the chunk drawn uniformly at random (seed 4), full oracle per row, "
                         f"{el:.1f} s"}
    return {
        "workload": spec.name, "queries": T, "ms": {**ms, "total": total}, "tokens_per_s": T / (total * 1e-3),
        "indexer": {"kernel": "prefill_index_kernel (tcgen05.mma kind::f8f6f4, e4m3 operands, exact)",
                    "bound": "hbm", "achieved": idx_gbs, "peak": peak_hbm, "unit": "GB/s",
                    "frac": idx_gbs / peak_hbm, "bytes": idx_bytes, "peak_kind": peak_kind,
                    "tops": idx_tops, "ops": 2 * 64 * causal_pairs,
                    "tensor_peaks_tops": {"tcgen05_e4m3": f8, "tcgen05_f16": f16, "mma_sync_s8": s8},
                    "tensor_frac": {"tcgen05_e4m3": idx_tops / f8, "mma_sync_s8": idx_tops / s8},
                    "peak_note": "tensor peaks measured in this run by libdsa_probe.so microbenchmarks"},
        "attention": {"kernel": "dsa_sparse_attn_prefill per call: dense_mask_kernel + dense_attn_kernel "
                                "(masked dense pass on tcgen05.mma kind::f16, bf16 operands, fp32 in tensor "
                                f"memory) for the first {n_dense} of {T} queries (automatic split)",
                      "bound": "tensor", "achieved": dense_tflops, "peak": f16, "unit": "TFLOP/s",
                      "frac": dense_tflops / f16 if dense_tflops else None, "flops": dense_flops,
                      "attended_flops": useful_flops, "dense_queries": n_dense,
                      "peak_kind": "measured in this run: back-to-back tcgen05.mma kind::f16 128 x 256 tiles "
                                   "(libdsa_probe.so); bf16 runs at the f16 rate"},
        "attention_gather_only": {"kernel": "prefix_attn_kernel + sparse_attn_kernel + attn_combine_kernel, every "
                                            "query's attended rows gathered from L2", "ms": ms["attention_gather_only"],
                                  "bound": "l2", "achieved": gather_gbs, "peak": gather, "unit": "GB/s",
                                  "frac": gather_gbs / gather, "bytes": gathered,
                                  "peak_kind": f"measured in this run: random {hkv * 256}-byte bulk copies from an "
                                               f"L2-resident 32 MB buffer into shared memory (libdsa_probe.so)"},
        "window": {"kernel": "dsa_window_attn_prefill per call: dense_attn_kernel with the window as its mask",
                   "window": WINDOW, "ms": ms["window"], "bound": "tensor", "achieved": win_tflops, "peak": f16,
                   "unit": "TFLOP/s", "frac": win_tflops / f16, "flops": win_flops},
        "mma_sync_bf16_peak_tflops": bf16,
        "clocks": clock_info,
        "cpu_baseline": cpu,
    }


# --------------------------------------------------------------- arms ------
def run_reference(args, rank, world):
    """The CPU oracle, as it stands, on a bounded sample of the workload."""
    import torch
    import synth
    if rank != 0:
        return
    spec = synth.CONFIGS[CONFIG_ID]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = synth.make_workload(spec, 1000 + CONFIG_ID, dev)
    n = max(1, args.steps) + max(0, args.warmup)
    inputs = [oracle_sequence_inputs(w, i % spec.batch) for i in range(min(n, spec.batch))]
    del w
    for i in range(args.warmup):
        time_oracle([inputs[i % len(inputs)]], spec)
    secs = 0.0
    for i in range(args.steps):
        secs += time_oracle([inputs[(args.warmup + i) % len(inputs)]], spec)
    value = args.steps / secs
    sample = f"{args.steps} decode tokens (one sequence each) of the workload, full oracle per token"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_block(spec),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_block(spec, layers=LAYERS):
    return {"workload": spec.name, "batch": spec.batch, "context": 131072, "prefix": spec.prefix_len,
            "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads, "head_dim": 128, "idx_dim": 64,
            "top_k": spec.k, "block_size": 64, "seed": 1000 + CONFIG_ID,
            "l2": f"inputs larger than L2: steps rotate over {layers} independent KV caches (no flush)"}


def run_gpu(args, rank, world, local_rank):
    import torch
    import dynamic_sparse_attention_indexer_gb300 as dsa
    import harness as H
    import synth
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    spec = synth.CONFIGS[CONFIG_ID]
    P, k, hq = spec.prefix_len, spec.k, spec.num_q_heads

    # --- resident inputs: args.layers independent caches; one query batch per layer
    LAYERS = args.layers
    layers = []
    for l in range(LAYERS):
        w = synth.make_workload(spec, 1000 + CONFIG_ID + 7919 * l + 104729 * rank, dev)
        kv = H.paged_kv(w)
        B = kv.batch
        ld = H.round4(w["max_context_len"])
        bufs = {"scores": torch.empty((B, ld), dtype=torch.int32, device=dev),
                "idx": torch.empty((B, k), dtype=torch.int32, device=dev),
                "n_sel": torch.empty(B, dtype=torch.int32, device=dev),
                "out": torch.empty((B, hq, 128), dtype=torch.bfloat16, device=dev),
                "lse": torch.empty((B, hq), dtype=torch.float32, device=dev)}
        ws = dsa.make_workspace(dsa.workspace_size(dsa.OP_DECODE_STEP, kv, dsa.decode_queries(kv), k, hq, P), dev)
        layers.append((w, kv, bufs, ws))
    lens = [int(x) for x in layers[0][0]["context_lens"].tolist()]
    B = len(lens)

    def step(l):
        w, kv, b, ws = layers[l]
        dsa.decode_step(kv, w["q"], w["q_idx"], P, k, b["scores"], b["idx"], b["n_sel"], b["out"], b["lse"], ws)

    # eager warm-up (first call sets kernel attributes), then one graph per layer
    # and one graph of a whole pass over the layers (as a serving loop captures
    # one decode iteration of all its layers)
    for l in range(LAYERS):
        step(l)
    torch.cuda.synchronize()
    assert dsa.check_device_status(dev) == 0
    stream = torch.cuda.Stream(device=dev)
    graphs = []
    with torch.cuda.stream(stream):
        for l in range(LAYERS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(l)
            graphs.append(g)
        cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cycle, stream=stream):
            for l in range(LAYERS):
                step(l)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % LAYERS].replay()
        cycle.replay()
    torch.cuda.synchronize()

    # --- timed region: exactly K steps
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps // LAYERS):  # exactly args.steps steps
            cycle.replay()
        for l in range(args.steps % LAYERS):
            graphs[l].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clock_info = clocks.stop()
    local_ms = e0.elapsed_time(e1)
    n_sel = [int(x) for x in layers[0][2]["n_sel"].tolist()]
    assert dsa.check_device_status(dev) == 0

    # --- per-call breakdown on the launching stream: each call is captured once
    # per layer into a graph, replayed; time per launch = graph time / launches.
    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for l in range(LAYERS):
                    fn(l)
        return g

    def per_launch_ms(g, reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / (reps * LAYERS)

    def attn_call(l):
        w, kv, b, ws = layers[l]
        dsa.sparse_attn_decode(kv, w["q"], b["idx"], b["n_sel"], k, P, b["out"], b["lse"], ws)

    def index_call(l):
        w, kv, b, ws = layers[l]
        dsa.index_scores(kv, dsa.decode_queries(kv), w["q_idx"], P, b["scores"])

    reps = max(8, min(args.steps // LAYERS, 250))
    attn_ms = per_launch_ms(graph_of(attn_call), reps)
    index_ms = per_launch_ms(graph_of(index_call), reps)

    # the local sliding-window sibling over the same caches: each sequence's
    # newest token over its last WINDOW positions
    hq_d = spec.num_q_heads
    win_ws = [dsa.make_workspace(dsa.window_workspace_size(layers[l][1], hq_d, WINDOW), dev) for l in range(LAYERS)]
    win_out = torch.empty_like(layers[0][2]["out"])

    def win_call(l):
        w, kv, b, ws = layers[l]
        dsa.window_attn_decode(kv, w["q"], WINDOW, win_out, None, win_ws[l])

    win_ms = per_launch_ms(graph_of(win_call), reps)
    del win_ws

    # the per-KV-head indexer form on a workload of the same shapes whose
    # indexer keys and queries carry one head per KV head
    hkv_d = spec.num_kv_heads
    wh = synth.make_workload(dataclasses.replace(spec, idx_heads=hkv_d), 4241 + 104729 * rank, dev)
    kvh = H.paged_kv(wh)
    hb = {"scores": torch.empty((B * hkv_d, H.round4(wh["max_context_len"])), dtype=torch.int32, device=dev),
          "idx": torch.empty((B, hkv_d, k), dtype=torch.int32, device=dev),
          "n_sel": torch.empty((B, hkv_d), dtype=torch.int32, device=dev)}
    heads_ws = dsa.make_workspace(dsa.heads_workspace_size(kvh, hq_d, k, P), dev)

    def heads_call(l):
        dsa.decode_step_heads(kvh, wh["q"], wh["q_idx"], P, k, hb["scores"], hb["idx"], hb["n_sel"], win_out,
                              None, heads_ws)

    heads_call(0)
    torch.cuda.synchronize()
    assert dsa.check_device_status(dev) == 0
    heads_ms = per_launch_ms(graph_of(heads_call), reps)
    heads_lens = [int(x) for x in wh["context_lens"].tolist()]
    heads_nsel = hb["n_sel"].tolist()
    del wh, kvh, hb, heads_ws
    torch.cuda.empty_cache()
    step(0)
    torch.cuda.synchronize()

    # --- end to end through the public API with host buffers.  A step's inputs
    # (q, q_idx) sit back to back in one pinned staging buffer and one device
    # buffer, its outputs (out, lse) likewise, so that each step is one copy in
    # and one copy out (the API takes the device views); the copies are the
    # library's staging copy (dsa_copy_async: a kernel, chained to the step by
    # programmatic dependent launch, instead of the copy engines).
    w0, kv0, b0, ws0 = layers[0]
    q_nb, qi_nb = w0["q"].numel() * 2, w0["q_idx"].numel()
    out_nb, lse_nb = b0["out"].numel() * 2, b0["lse"].numel() * 4
    in_dev, out_dev, views = [], [], []
    for l in range(LAYERS):
        w, kv, b, ws = layers[l]
        bi = torch.empty(q_nb + qi_nb, dtype=torch.uint8, device=dev)
        bo = torch.empty(out_nb + lse_nb, dtype=torch.uint8, device=dev)
        qv = bi[:q_nb].view(torch.bfloat16).view(w["q"].shape)
        qiv = bi[q_nb:].view(torch.int8).view(w["q_idx"].shape)
        qv.copy_(w["q"])
        qiv.copy_(w["q_idx"])
        views.append((qv, qiv, bo[:out_nb].view(torch.bfloat16).view(b["out"].shape),
                      bo[out_nb:].view(torch.float32).view(b["lse"].shape)))
        in_dev.append(bi)
        out_dev.append(bo)
    in_host = [in_dev[l].cpu().pin_memory() for l in range(LAYERS)]
    out_host = torch.empty(out_nb + lse_nb, dtype=torch.uint8).pin_memory()
    n_e2e = max(8, min(args.steps, 500))

    def step_io(l):
        w, kv, b, ws = layers[l]
        qv, qiv, ov, lv = views[l]
        dsa.decode_step(kv, qv, qiv, P, k, b["scores"], b["idx"], b["n_sel"], ov, lv, ws)

    # One graph per layer holds the whole call sequence a serving loop makes for
    # a step: the host-to-device copies of the step's queries (pinned host
    # memory), the decode step, and the device-to-host copies of its output;
    # the host waits for the result before the next step.
    e2e_graphs = []
    with torch.cuda.stream(stream):
        for l in range(LAYERS):
            w, kv, b, ws = layers[l]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                dsa.copy_async(in_dev[l], in_host[l])
                step_io(l)
                dsa.copy_async(out_host, out_dev[l])
            e2e_graphs.append(g)
    torch.cuda.synchronize()

    def e2e_step(i):
        e2e_graphs[i % LAYERS].replay()
        stream.synchronize()

    with torch.cuda.stream(stream):
        for i in range(8):
            e2e_step(i)
        barrier()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        e2e_s = time.perf_counter() - t0
    h2d = in_host[0].numel()
    d2h = out_host.numel()

    # The same sequence without a graph: every step the Python API call
    # (argument checks and launches through the C ABI), the host-to-device
    # copies of the step's queries from pinned memory before it and the
    # device-to-host copies of its output after it, then the host waits.
    def e2e_api_step(i):
        l = i % LAYERS
        dsa.copy_async(in_dev[l], in_host[l])
        step_io(l)
        dsa.copy_async(out_host, out_dev[l])
        stream.synchronize()

    with torch.cuda.stream(stream):
        for i in range(8):
            e2e_api_step(i)
        barrier()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_api_step(i)
        e2e_api_s = time.perf_counter() - t0
    assert dsa.check_device_status(dev) == 0

    # --- aggregate over ranks (max time, summed tokens)
    agg = reduce_over_ranks({"ms": local_ms, "e2e_s": e2e_s, "e2e_api_s": e2e_api_s, "attn_ms": attn_ms,
                             "index_ms": index_ms, "win_ms": win_ms, "heads_ms": heads_ms}, "max")
    tokens = reduce_over_ranks({"tok": float(B * args.steps), "e2e_tok": float(B * n_e2e)}, "sum")

    # --- prefill chunk and its peaks (rank 0)
    prefill = None
    if rank == 0 and not args.no_prefill:
        del layers[1:]
        torch.cuda.empty_cache()
        prefill = measure_prefill(dev, args.prefill_steps, 3, Probes(dev),
                                  0.0 if args.no_cpu_baseline or world > 1 else args.cpu_seconds / 2)

    # --- CPU baseline (rank 0, N = 1 only): the oracle on a bounded sample,
    # on every host core at once, and on one thread
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_all_cores(w0, spec, args.cpu_seconds)
        n_seq = min(args.cpu_sample, B)
        inputs = [oracle_sequence_inputs(w0, b) for b in range(n_seq)]
        secs, passes = 0.0, 0
        while passes < 1 or (secs < args.cpu_seconds / 2 and passes < 200):
            secs += time_oracle(inputs, spec)
            passes += 1
        n_tok = n_seq * passes
        cpu["one_thread"] = {"value": n_tok / secs, "unit": "tokens/s", "cores": cpu_threads_used(),
                             "sample": f"{n_seq} of the {B} decode tokens of one step (full oracle per token), "
                                       f"{passes} passes: {n_tok} tokens in {secs:.1f} s"}

    if rank != 0:
        return
    ab = algorithmic_bytes(spec, lens, n_sel)
    peak, peak_kind = measured_peaks()
    ms_step = agg["ms"] / args.steps
    attn_gbs = ab["attention"] / (agg["attn_ms"] * 1e-3) / 1e9
    step_gbs = ab["step"] / (ms_step * 1e-3) / 1e9
    traffic = args.attn_traffic if args.attn_traffic > 0 else profiled_attention_traffic()
    launches_per_step = 4  # indexer (+ histogram), top-k selection, attention, partial merge
    line = {
        "metric": METRIC, "value": tokens["tok"] / (agg["ms"] * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(spec, LAYERS),
        "hbm": {"step_bytes": ab["step"], "achieved_gbs": step_gbs, "peak_gbs": peak,
                "frac": step_gbs / peak, "peak_kind": peak_kind},
        "roofline": {"kernel": "dsa_sparse_attn_decode per call in a graph: sparse_attn_kernel + "
                               "attn_combine_kernel",
                     "bound": "hbm", "achieved": attn_gbs, "peak": peak, "unit": "GB/s", "frac": attn_gbs / peak,
                     "traffic": traffic, "algorithmic_bytes": ab["attention"], "ms": agg["attn_ms"],
                     "peak_kind": peak_kind},
        "indexer": {"ms": agg["index_ms"], "achieved_gbs": ab["indexer"] / (agg["index_ms"] * 1e-3) / 1e9},
        "window_decode": window_decode_line(spec, lens, agg["win_ms"], peak, peak_kind),
        "heads_decode": heads_decode_line(spec, heads_lens, heads_nsel, agg["heads_ms"], peak, peak_kind),
        "clocks": clock_info,
        "e2e": {"value": tokens["e2e_tok"] / agg["e2e_s"], "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "graph replay: per step one captured graph of the host-to-device copy of the step's "
                       "queries (q and q_idx packed in one pinned buffer), the decode step and the "
                       "device-to-host copy of its output (out and lse packed), both copies by dsa_copy_async; "
                       "the host waits for each step"},
        "e2e_api": {"value": tokens["e2e_tok"] / agg["e2e_api_s"], "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "how": "no graph: per step the same two copies and the Python API call through the C "
                           "ABI (host argument checks and kernel launches included); the host waits for each "
                           "step"},
        "gpu_launches": launches_per_step * args.steps,
        "cpu_baseline": cpu,
        "prefill": prefill,
    }
    print(json.dumps(line), flush=True)


def run_prefill(args):
    """Only the 16K prefill chunk (one GPU), printed as its own JSON line: a
    small command for profiling the prefill kernels."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    res = measure_prefill(dev, args.steps, args.warmup, Probes(dev), 0.0)
    print(json.dumps({"metric": "DSA prefill tokens/s, 16K causal chunk, 1xGB300", "value": res["tokens_per_s"],
                      "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": res["ms"]["total"], "higher_is_better": True, "dtype": "bf16 / int8 indexer",
                      "data": "synthetic", "config": {"workload": res["workload"]}, "prefill": res}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--prefill", action="store_true",
                    help="time the 16K prefill path instead of the decode headline (one GPU)")
    ap.add_argument("--cpu-sample", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle time of the all-cores CPU baseline (the one-thread and prefill ones take half)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="leave the prefill chunk out of the headline line")
    ap.add_argument("--prefill-steps", type=int, default=5, help="timed calls of each prefill step")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="independent caches the steps rotate over (4 keeps every step out of L2; "
                         "1 gives a small case for ncu captures)")
    ap.add_argument("--attn-traffic", type=float, default=0.0,
                    help="DRAM bytes per attention launch from an ncu capture (0 = not measured)")
    args = ap.parse_args()
    assert args.warmup >= 0 and args.steps >= 1

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, rank, world)
        return
    if args.prefill:
        if rank == 0:
            run_prefill(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", init_method="env://")
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("MKL_NUM_THREADS", "1")
    main()
