"""The bench's multi-process path on CPU (gloo, world size 2): whole-job
aggregation (max time over ranks, tokens summed) and the reference arm under
torchrun (rank 0 alone works and prints one JSON line, the other rank exits 0)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    agg = bench.aggregate(ms_total=10.0 + rank, tokens=100 * (rank + 1), e2e_ms=5.0 * (rank + 1),
                          world=world, device=torch.device("cpu"))
    q.put((rank, agg))
    dist.destroy_process_group()


def test_aggregate_takes_max_time_and_sums_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert res[r] == {"ms_max": 11.0, "e2e_ms_max": 10.0, "tokens": 300.0}


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--config", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_launch_counts_match_the_measured_steps():
    """The bench's claimed launches per step, for the workloads whose counts were read
    off CUDA-graph runs on the GPU (gpu_launches / steps): decode 6 (bf16) and 5 (FP8),
    prefill 8 (chunked dispatch), decode with the split router GEMM 9."""
    sys.path.insert(0, ROOT)
    import bench
    # decode: 440 global rows, top-8, 256 experts / slots, cap 3520 + 64
    assert bench.launches_per_step(440, 8, 256, 256, 3584, 1) == 6
    assert bench.launches_per_step(440, 8, 256, 256, 3584, 1, fp8=True) == 5
    # FP8 with many rows per slot: MM1, the quantisation of h, MM2
    assert bench.launches_per_step(8192, 8, 256, 256, 65600, 1, fp8=True, fp8_pair=True) == 9
    assert bench.fp8_pair(65600, 256, 7168, 2048) and not bench.fp8_pair(3584, 256, 7168, 2048)
    assert not bench.fp8_pair(65600, 256, 7168, 2304)
    # a skewed FP8 layer (EPLB: 57 rows per slot): pair launches, then the one-launch kernel
    assert bench.fp8_split(16384, 288, 7168, 2048) and not bench.fp8_split(3584, 256, 7168, 2048)
    assert bench.launches_per_step(2048, 8, 256, 288, 16384, 1, fp8=True, fp8_split=True) == 10
    assert bench.launches_per_step(440, 8, 256, 256, 3584, 1, router_gemm=True) == 9
    # prefill: 8192 rows x 8 pairs take the chunked dispatch (histogram, scan, rank, copy)
    assert bench.launches_per_step(8192, 8, 256, 256, 65600, 1) == 8
    # the combine in the down projection's epilogue takes one launch off either step
    assert bench.launches_per_step(440, 8, 256, 256, 3584, 1, fused_combine=True) == 5
    assert bench.launches_per_step(8192, 8, 256, 256, 65600, 1, fused_combine=True) == 7
