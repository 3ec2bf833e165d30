"""Multi-process (gloo, world_size 2, CPU) checks of the benchmark's replica harness: rank
setup from the torchrun environment, barriers, max-over-ranks timing, whole-job throughput,
and that only rank 0 runs and prints the CPU reference arm."""
import io
import os
import socket
import sys
import contextlib

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    class A:
        pass

    w, r, loc = bench.dist_setup(A())
    assert (w, r, loc) == (world, rank, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    args = A()
    args.workload, args.ref_tokens, args.warmup, args.steps = "toy_T64", 2, 1, 1
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, w, r)
    dist.destroy_process_group()
    q.put((rank, m, buf.getvalue()))


def test_two_rank_harness():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [m for _, m, _ in res] == [15.0, 15.0]          # max over ranks on every rank
    assert '"impl": "reference"' in res[0][2]             # rank 0 prints the reference line
    assert res[1][2] == ""                                # rank 1 exits without work


def test_gpus_flag_spawns_the_ranks():
    """`bench.py --gpus 2` with no launcher environment starts its two rank processes itself
    (gloo on this CPU-only host) and rank 0 prints one line for the whole job."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
                                                           "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                          "--workload", "toy_T64", "--steps", "1", "--warmup", "3", "--ref-tokens", "2"],
                         capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
