"""The benchmark's multi-rank host logic on CPU: two gloo ranks launched the way the
benchmark is launched for N > 1 (torch.distributed.run, one process per rank).

Every rank owns whole sequences (replicas, no collective on the data path); the only
cross-rank steps are the barrier around the timed region and the maximum of the ranks'
times, and only rank 0 prints.
"""
import json
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


def torchrun(args, tmp_path, timeout=600):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), *args]
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""),
               OMP_NUM_THREADS="2")
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_slowest_rank_sets_the_job_time(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent('''
        import importlib.util, json, os, sys
        import torch.distributed as dist
        spec = importlib.util.spec_from_file_location("bench", os.path.join(os.getcwd(), "bench.py"))
        bench = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(bench)
        world, rank, local = bench.dist_setup()
        dist.init_process_group("gloo")
        dist.barrier()
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world)   # rank 1 is the slow one
        rate = bench.job_rate(32, world, ms)
        # one file per rank: the launcher merges the ranks' stdout, lines may interleave
        with open(os.path.join(sys.argv[1], f"rank{rank}.json"), "w") as f:
            json.dump({"rank": rank, "world": world, "ms": ms, "rate": rate}, f)
        dist.destroy_process_group()
    '''))
    r = torchrun([str(script), str(tmp_path)], tmp_path)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads((tmp_path / f"rank{i}.json").read_text()) for i in range(2)]
    assert sorted(d["rank"] for d in lines) == [0, 1]
    for d in lines:
        assert d["world"] == 2 and d["ms"] == 15.0
        assert abs(d["rate"] - 2 * 32 / 15e-3) < 1e-6


def test_reference_arm_under_two_ranks_prints_one_line(tmp_path):
    r = torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                  "--warmup", "3"], tmp_path)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
