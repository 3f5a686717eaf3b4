"""The multi-rank (N > 1) path of bench.py on CPU with the gloo backend.

The hot path shards by sequence with no exchange step, so N GPUs run N
independent replicas: each rank draws its own sequences, the ranks meet at a
barrier around the timed region, the step time is the maximum over ranks, and
rank 0 alone prints the JSON line (the reference arm runs on rank 0 only and
the other ranks exit 0 without work). These tests run two ranks as CPU
processes, rendezvous on 127.0.0.1."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cpu_env():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    env["OMP_NUM_THREADS"] = "1"
    return env


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from cross_layer_kv_pool_b300 import synth
    import torch.distributed as dist

    ws, r, _ = bench.dist_init()
    assert (ws, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(ws)
    mx = bench.max_over_ranks(1.5 * (rank + 1), ws)
    # each replica prefills its own sequences (tokens seeded 1 + rank)
    s = synth.TINY_FP32
    tok = synth.make_tokens(s, 2, 16, seed=1 + rank)
    got = [torch.zeros_like(tok) for _ in range(ws)]
    dist.all_gather(got, tok)
    distinct = not torch.equal(got[0], got[1])
    bench.barrier(ws)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": mx, "distinct": distinct}, f)


def test_barrier_max_and_distinct_replicas(tmp_path):
    port = _free_port()
    old = os.environ.get("CUDA_VISIBLE_DEVICES")
    os.environ["CUDA_VISIBLE_DEVICES"] = ""
    try:
        mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                           start_method="spawn")
    finally:
        if old is None:
            os.environ.pop("CUDA_VISIBLE_DEVICES", None)
        else:
            os.environ["CUDA_VISIBLE_DEVICES"] = old
    for rank in range(2):
        res = json.loads((tmp_path / f"rank{rank}.json").read_text())
        assert res["max"] == 3.0        # every rank sees the slowest rank's time
        assert res["distinct"]          # replicas work on different sequences


def test_reference_arm_two_ranks_prints_one_line():
    """``bench.py --impl reference`` launched like the driver's N = 2 run:
    rank 0 times the oracle and prints one line, rank 1 exits 0 silently."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "1", "--workload", "tiny_fp32"]
    r = subprocess.run(cmd, cwd=ROOT, env=_cpu_env(), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["config"]["parallelism"] == "replicas x2"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
