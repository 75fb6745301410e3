"""Seeded synthetic workloads for the DSA hot path.

This module only draws random inputs (bf16 Q/K/V ~ N(0,1), int8 indexer
vectors uniform in [-lo, hi], a seeded random block table and optional
key-row outliers).  It holds none of the method's arithmetic; both the CPU
oracle and the CUDA library consume the tensors it returns.

A workload is defined by (spec, seed, device): every tensor is drawn from its
own ``torch.Generator`` seeded from (seed, tensor name), on the device the
workload is built on.  Small workloads are built on the CPU and copied to the
GPU; full-size ones are built on the GPU and the oracle reads back only the
rows it needs.
"""
from __future__ import annotations

import dataclasses
import math
import zlib

import numpy as np
import torch

BLOCK = 64
HEAD_DIM = 128
IDX_DIM = 64


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    mode: str                      # "decode" or "prefill"
    batch: int                     # decode: sequences; prefill: 1
    context_lens: tuple            # per sequence, or ("uniform", lo, hi)
    prefix_len: int
    num_q_heads: int
    num_kv_heads: int
    k: int
    outlier_frac: float = 0.0      # fraction of K rows scaled by outlier_scale
    outlier_scale: float = 4.0
    idx_lo: int = -8               # indexer values uniform in [idx_lo, idx_hi]
    idx_hi: int = 8
    num_queries: int = 0           # prefill: T
    pos0: int = 0                  # prefill: position of query 0
    spare_blocks: int = 0          # extra unused blocks in the pool
    kv_layout: str = "adjacent"    # "adjacent": K and V of a slot in one row; "separate": two arrays
    idx_heads: int = 1             # 1: one indexer key per position; num_kv_heads: one per (position, KV head)
    head_tables: bool = False      # per-head indexer: one block table per KV head (block_table_heads)


# The five workloads of the headline measurement plan.
DECODE_512 = Spec("decode B=1 L=512 P=64 Hq/Hkv=8/1 k=128", "decode", 1, (512,), 64, 8, 1, 128)
DECODE_8K = Spec("decode B=32 L=8192 P=256 Hq/Hkv=32/4 k=2048", "decode", 32, (8192,) * 32,
                 256, 32, 4, 2048)
DECODE_128K = Spec("decode B=8 L=131072 P=1024 Hq/Hkv=64/8 k=2048 1% K outliers x4", "decode", 8,
                   (131072,) * 8, 1024, 64, 8, 2048, outlier_frac=0.01)
PREFILL_16K = Spec("prefill T=L=16384 P=576 Hq/Hkv=32/4 k=2048", "prefill", 1, (16384,), 576,
                   32, 4, 2048, num_queries=16384, pos0=0)
DECODE_1M = Spec("decode B=4 L~U[262144,1048576] P=1024 Hq/Hkv=64/8 k=2048", "decode", 4,
                 ("uniform", 262144, 1048576), 1024, 64, 8, 2048)
CONFIGS = {1: DECODE_512, 2: DECODE_8K, 3: DECODE_128K, 4: PREFILL_16K, 5: DECODE_1M}


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(name.encode())) & ((1 << 62) - 1))
    return g


def context_lengths(spec: Spec, seed: int) -> list[int]:
    if spec.context_lens and spec.context_lens[0] == "uniform":
        _, lo, hi = spec.context_lens
        g = _gen(seed, "context_lens", "cpu")
        return [int(x) for x in torch.randint(lo, hi + 1, (spec.batch,), generator=g)]
    return [int(x) for x in spec.context_lens]


def _randn_bf16(shape, g, device, chunk_rows=1 << 14):
    """N(0,1) drawn in fp32 and rounded to bf16 (round-to-nearest-even),
    produced in slices along dim 0 to bound the fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    n0 = shape[0]
    per = max(1, chunk_rows)
    for s in range(0, n0, per):
        e = min(n0, s + per)
        out[s:e] = torch.randn((e - s,) + tuple(shape[1:]), generator=g, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
    return out


def make_workload(spec: Spec, seed: int, device="cpu") -> dict:
    """Draw every input of ``spec``.  Returns a dict of tensors on ``device``
    plus the scalar parameters."""
    device = torch.device(device)
    lens = context_lengths(spec, seed)
    nblk_seq = [math.ceil(L / BLOCK) for L in lens]
    pool = sum(nblk_seq) + spec.spare_blocks
    max_blocks = max(nblk_seq)

    # Block table: a seeded permutation of the pool dealt out in order.
    perm = torch.randperm(pool, generator=_gen(seed, "block_perm", "cpu")).to(torch.int32)
    bt = torch.full((spec.batch, max_blocks), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(nblk_seq):
        bt[b, :n] = perm[off:off + n]
        off += n
    # Per-head block tables (the per-head block bitmaps of the allocator): each
    # KV head deals its own seeded permutation of the pool in the same way, so a
    # physical block holds, in each head's slice, positions of another sequence.
    bt_heads = None
    if spec.head_tables:
        bt_heads = torch.full((spec.num_kv_heads, spec.batch, max_blocks), -1, dtype=torch.int32)
        for h in range(spec.num_kv_heads):
            ph = torch.randperm(pool, generator=_gen(seed, f"block_perm_head{h}", "cpu")).to(torch.int32)
            off = 0
            for b, n in enumerate(nblk_seq):
                bt_heads[h, b, :n] = ph[off:off + n]
                off += n

    hkv, hq = spec.num_kv_heads, spec.num_q_heads
    # The same values in either layout (each array drawn from its own stream).
    if spec.kv_layout == "adjacent":
        kv = torch.empty((pool, BLOCK, 2, hkv, HEAD_DIM), dtype=torch.bfloat16, device=device)
        k_cache, v_cache = kv[:, :, 0], kv[:, :, 1]
    else:
        k_cache = torch.empty((pool, BLOCK, hkv, HEAD_DIM), dtype=torch.bfloat16, device=device)
        v_cache = torch.empty_like(k_cache)
    rows = max(1, (1 << 24) // (hkv * BLOCK * HEAD_DIM))
    for name, dst in (("k_cache", k_cache), ("v_cache", v_cache)):
        g = _gen(seed, name, device)
        for s0 in range(0, pool, rows):
            e0 = min(pool, s0 + rows)
            dst[s0:e0] = torch.randn((e0 - s0, BLOCK, hkv, HEAD_DIM), generator=g, device=device,
                                     dtype=torch.float32).to(torch.bfloat16)
    if spec.outlier_frac > 0:
        # One independent Bernoulli draw per (block, row, kv head), i.e. per
        # (sequence, position, kv head); K only, before use (x4 is exact in bf16).
        mask = torch.rand((pool, BLOCK, hkv), generator=_gen(seed, "outliers", device),
                          device=device) < spec.outlier_frac
        k_cache[mask] = (k_cache[mask].float() * spec.outlier_scale).to(torch.bfloat16)
    # per-head indexer: [pool][Hkv][64][64] (a head's keys of a block contiguous) and q_idx [nq][Hkv][64]
    idx_shape = (pool, BLOCK, IDX_DIM) if spec.idx_heads == 1 else (pool, spec.idx_heads, BLOCK, IDX_DIM)
    idx_cache = torch.randint(spec.idx_lo, spec.idx_hi + 1, idx_shape,
                              generator=_gen(seed, "idx_cache", device), device=device,
                              dtype=torch.int8)
    nq = spec.batch if spec.mode == "decode" else spec.num_queries
    q = _randn_bf16((nq, hq, HEAD_DIM), _gen(seed, "q", device), device)
    q_shape = (nq, IDX_DIM) if spec.idx_heads == 1 else (nq, spec.idx_heads, IDX_DIM)
    q_idx = torch.randint(spec.idx_lo, spec.idx_hi + 1, q_shape,
                          generator=_gen(seed, "q_idx", device), device=device, dtype=torch.int8)
    out = {
        "spec": spec, "seed": seed, "mode": spec.mode,
        "k_cache": k_cache, "v_cache": v_cache, "idx_cache": idx_cache,
        "block_table": bt.to(device), "context_lens": torch.tensor(lens, dtype=torch.int32).to(device),
        "q": q, "q_idx": q_idx,
        "prefix_len": spec.prefix_len, "k": spec.k,
        "num_q_heads": hq, "num_kv_heads": hkv,
        "seq": 0, "pos0": spec.pos0, "num_queries": nq,
        "max_context_len": max(lens),
    }
    if spec.kv_layout == "adjacent":
        out["kv"] = kv  # the one array behind the k_cache / v_cache views
    if bt_heads is not None:
        out["block_table_heads"] = bt_heads.to(device)
    return out


def to_numpy(w: dict) -> dict:
    """CPU numpy view of a workload for the oracle: bf16 -> float64 (exact),
    integers -> int64."""
    out = {}
    for key, val in w.items():
        if key == "kv":
            continue  # the k_cache / v_cache views carry its values
        if isinstance(val, torch.Tensor):
            t = val.detach().cpu()
            if t.dtype == torch.bfloat16:
                out[key] = t.to(torch.float64).numpy()
            elif t.dtype == torch.int8:
                out[key] = t.numpy().astype(np.int64)
            else:
                out[key] = t.numpy()
        else:
            out[key] = val
    return out


def small_spec(name="small", mode="decode", batch=None, lens=(700, 1500, 2113), prefix_len=64,
               hq=16, hkv=2, k=256, **kw) -> Spec:
    """A workload the oracle finishes in seconds that still spans several
    blocks, chunks and tiles, with a ragged tail (batch = len(lens))."""
    assert batch is None or batch == len(lens)
    return Spec(name, mode, len(lens), tuple(lens), prefix_len, hq, hkv, k, **kw)
