"""Multi-process host logic of bench.py on CPU (gloo, world_size 2).

The GDN core shards with no exchange (each rank runs its own replica), so the
only cross-rank steps are the timing barrier and the max over ranks of the
step time; the reference arm runs on rank 0 alone.
"""
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CHILD = textwrap.dedent("""
    import io, contextlib, os, sys
    sys.path.insert(0, {root!r})
    import bench
    world, rank, local = bench.dist_setup()
    assert world == 2 and rank in (0, 1)
    bench.barrier(world)
    ms = bench.max_over_ranks(1.0 + rank, world, "cpu")       # slowest rank wins
    assert ms == 2.0, ms
    value = world * 4096 / (ms * 1e-3)                           # whole-job tokens/s
    assert abs(value - 4096 * 1000) < 1e-6
    if rank == 1:                                                # reference arm: rank 0 only
        class A: steps = 1; warmup = 3
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(A, world, rank)
        assert buf.getvalue() == ""
    bench.barrier(world)
    import torch.distributed as dist
    dist.destroy_process_group()
    print("rank", rank, "ok")
""")


def test_two_rank_gloo_timing_logic():
    port = free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(r),
                   LOCAL_RANK=str(r), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = [p.communicate(timeout=240)[0] for p in procs]
    for r, (p, out) in enumerate(zip(procs, outs)):
        assert p.returncode == 0, out
        assert f"rank {r} ok" in out
