"""The multi-rank host logic of bench.py on CPU with gloo (world size 2): the
slowest rank's time decides the whole-job throughput, and the reference arm
under torchrun prints one line from rank 0 while the other ranks exit cleanly."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms = bench.max_over_ranks(dist, 10.0 + 5.0 * rank)
    out[rank] = (ms, bench.job_throughput(world, 8192, ms))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        ms, thr = out[rank]
        assert ms == 15.0                               # the slowest rank's time
        assert abs(thr - 2 * 8192 / 0.015) < 1e-6


def test_reference_arm_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--workload", "tiny-4k", "--steps", "1",
           "--warmup", "1", "--cpu-layers", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_one_core_baseline_child():
    """The one-core oracle baseline runs in a child process limited to one BLAS
    thread and reports a positive throughput for one core; an unknown workload
    is reported as unavailable instead of failing the bench."""
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_meank_gb300 import configs
    d = bench.cpu_baseline_one_core(configs.TINY, 0, 2)
    assert d["cores"] == 1 and d["value"] > 0, d
    assert "2 of 2 layers" in d["sample"]
    bad = bench.cpu_baseline_one_core(configs.TINY.with_(name="no-such-workload"), 0, 1)
    assert bad["value"] is None and bad["unavailable"]
