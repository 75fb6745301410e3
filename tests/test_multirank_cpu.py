"""The N > 1 bench path on the CPU: two gloo ranks reduce their timings (max)
and token counts (sum) the way bench.py does under torchrun.  No GPU: decode
sequences are independent, so ranks share nothing but these reductions."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mx = bench.reduce_over_ranks({"ms": 10.0 + rank, "e2e_s": 2.0 - rank}, "max")
        sm = bench.reduce_over_ranks({"tok": 8.0 * (rank + 1)}, "sum")
        bench.barrier()
        q.put((rank, mx, sm))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, sm in out:
        assert mx == {"ms": 11.0, "e2e_s": 2.0}   # slowest rank's time
        assert sm == {"tok": 24.0}                # all ranks' tokens


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks({"ms": 3.0}, "max") == {"ms": 3.0}


def test_code_digest_ignores_comments(tmp_path):
    """The profiled traffic stays valid across comment edits, not code edits."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text("// header\nint f(int x) {  // why\n  return x + 1;\n}\n")
    b.write_text("// another header\n\nint f(int x) {\n  return x + 1;  // note\n}\n")
    c.write_text("// header\nint f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_digest(str(a)) == bench.code_digest(str(b))
    assert bench.code_digest(str(a)) != bench.code_digest(str(c))
