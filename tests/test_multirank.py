"""The N > 1 path of bench.py on CPU with world size 2.

The path has no data exchange (each rank runs an independent replica); the
only cross-rank steps are the timing reduction (max over ranks) and rank 0
alone printing the JSON line.  Both are checked here over gloo, on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as tdist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0])
    thr = bench.job_throughput(world, 3.0, got[0])
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": got, "thr": thr}, f)
    tdist.barrier()
    tdist.destroy_process_group()


def test_timing_is_max_over_ranks_with_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d["max"] == [2.0, 10.0, 5.0]
        assert d["thr"] == 2 * 3.0 / 2.0


def test_reference_arm_prints_once_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--impl", "reference", "--workload", "tiny_1x1024", "--steps", "1", "--warmup", "0",
           "--ref-rows", "64"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
