"""Multi-process plumbing of bench.py on the CPU (gloo, world size 2).

The hot path shards by request with no collective: each rank runs its own
replica of the workload on its own GPU, and only the timing is reduced (max
over ranks).  These tests exercise that reduction and the whole-job
throughput with real gloo process groups, and check that the reference arm
runs on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    local_ms = [12.5, 20.0][rank]                      # the second rank is the slow one
    max_ms = bench.reduce_max(local_ms, dist, "cpu")
    gbs = bench.weak_scaling_gbs(world, 1e9, 10, max_ms)
    dist.barrier()
    q.put((rank, max_ms, gbs))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_with_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, max_ms, gbs in res:
        assert max_ms == 20.0
        # 2 replicas x 1 GB x 10 steps in 20 ms of the slowest rank
        assert abs(gbs - 2 * 1e9 * 10 / 0.020 / 1e9) < 1e-9


def test_reduce_without_process_group_is_identity():
    import bench
    assert bench.reduce_max(3.25) == 3.25
    assert bench.weak_scaling_gbs(1, 2e9, 4, 1000.0) == pytest.approx(8.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank0_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny_gqa", "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    if rank == 0:
        d = json.loads(lines[-1])
        assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
        assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
        assert d["n_gpus"] == 2
    else:
        assert lines == []


@pytest.mark.parametrize("workload,fused", [("tiny_gqa", False), ("qwen3_0p6b_prefill", False),
                                            ("qwen3_0p6b_prefill", True), ("encoder_merge", False)])
def test_reference_arm_prints_the_config_of_the_gpu_arm(workload, fused):
    """Both arms describe one workload with the same `config` object (built on the host),
    including how the multi-query step finds its pages (--fused: straight from req_to_token)."""
    import bench
    from paged_kv_cache_req_gb300.workloads import make_encoder_merge, make_extend_workload, make_workload
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          workload, "--steps", "1", "--warmup", "3", "--ref-key-heads", "2000000"] +
                         (["--fused"] if fused else []),
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    d = json.loads([l for l in out.stdout.splitlines() if l.strip()][-1])
    if workload == "encoder_merge":
        want = bench.merge_config(make_encoder_merge(seed=0), 1)
    elif workload in bench.EXTEND_WORKLOADS:
        want = bench.extend_config(make_extend_workload(workload, seed=0), 1, token_table=fused)
        assert want["pages"].startswith("read from req_to_token" if fused else "kv_indptr")
    else:
        want = bench.decode_config(make_workload(workload, seed=0), "paged", False, 1)
    assert d["config"] == json.loads(json.dumps(want))
