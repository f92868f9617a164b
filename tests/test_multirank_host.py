"""The benchmark's multi-rank host logic on CPU ranks (gloo), no GPU:

* two ranks through bench.py's own setup: the timing taken is the slowest
  rank's, and the value counts every rank's units over it (weak scaling);
* the reference arm launched by torch.distributed.run with two ranks: rank 0
  alone prints one line, every rank exits 0.
"""
import json
import os
import socket
import subprocess
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _, pg = bench.dist_setup(None)
    ms = 10.0 + 3.0 * r  # rank 1 is the slow one
    m = bench.max_over_ranks(pg, ms, torch.device("cpu"))
    out.put((r, w, m, bench.aggregate_value(w, 32, 5, m)))
    pg.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_time():
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert all(x[2] == 13.0 for x in res)  # both ranks report the max
    assert all(abs(x[3] - 2 * 32 * 5 / 0.013) < 1e-6 for x in res)


def test_reference_arm_under_torchrun_prints_one_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference", "--gpus", "2",
           "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["value"] > 0
