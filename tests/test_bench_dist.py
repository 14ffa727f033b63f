"""The bench's multi-rank path on the CPU (gloo, world size 2): rendezvous,
barrier and the max over ranks that sets the reported time, and the
reference arm's rule that only rank 0 runs and prints."""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(body: str, world: int = 2, timeout: int = 120):
    port = _free_port()
    script = textwrap.dedent(body)
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", script], cwd=ROOT, env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_dist_max_over_ranks_gloo():
    outs = _run_ranks("""
        import json, os, bench
        rank, world, local = bench.dist_setup()
        assert world == 2
        bench.barrier(world)
        got = bench.all_max(10.0 + rank, world)
        print(json.dumps({"rank": rank, "max": got}))
        import torch.distributed as dist
        dist.destroy_process_group()
    """)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in res) == [0, 1]
    assert all(r["max"] == 11.0 for r in res)


def test_reference_arm_rank0_only():
    outs = _run_ranks("""
        import bench
        from workload import CONFIGS
        class A: budget = 68; steps = 1; warmup = 0; gpus = 2
        import os
        line = bench.bench_reference(A, CONFIGS["tiny"], int(os.environ["RANK"]), 2)
        print("LINE" if line is not None else "NONE")
    """)
    assert [o.strip().splitlines()[-1] for o in outs] == ["LINE", "NONE"]
