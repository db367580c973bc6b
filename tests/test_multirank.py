"""The multi-rank host path of bench.py on CPU: two `gloo` ranks.

The operator shards over independent (batch, head) problems, so a job of N
ranks runs one batch per rank with no data-path collective; the only
communication is a barrier and a max over ranks of the timed durations.
These tests run that plumbing with world size 2 on the host, and the
reference arm under torchrun, where rank 0 alone works and prints.
"""

import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    try:
        import torch
        import bench
        from linear_attention_sequence_chunked_gb300 import workloads as W
        w, r, _ = bench.dist_env()
        dist = bench.init_dist(w, "gloo")
        cpu = torch.device("cpu")
        # each rank times a different duration; every rank must see the slowest
        t_max = bench.max_over_ranks(0.25 * (r + 1), w, cpu)
        bench.barrier(w)
        # each rank's batch is its own: gather a fingerprint of every rank's inputs
        wl = W.make_workload(2, B=1, T=70, H=2, d_k=64, d_v=64, seed=bench.rank_seed(r))
        fp = torch.tensor([float(np.sum(W.bf16_bits_to_f32(wl.k)[..., :3])), float(np.sum(wl.g))],
                          dtype=torch.float64)
        fps = [torch.zeros_like(fp) for _ in range(w)]
        dist.all_gather(fps, fp)
        dist.destroy_process_group()
        q.put((r, w, t_max, [f.tolist() for f in fps]))
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((rank, "error", repr(e), None))


def test_two_gloo_ranks_share_the_slowest_time_and_own_their_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort(key=lambda x: x[0])
    for r, w, t_max, fps in results:
        assert w == 2, t_max
        assert t_max == pytest.approx(0.5)
        assert fps == results[0][3]          # both ranks gathered the same list
    fp0, fp1 = results[0][3]
    assert fp0 != fp1                        # rank 1's problems are not rank 0's


def test_aggregate_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # two ranks of 1000 units each, the slower one took 0.5 s: 4000 units/s
    assert bench.aggregate_rate(2, 1000, 0.5) == pytest.approx(4000.0)
    assert bench.aggregate_rate(1, 1000, 0.5) == pytest.approx(2000.0)
    assert bench.rank_seed(0) != bench.rank_seed(1)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_our_arm_fails_loudly_without_a_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    r = subprocess.run([sys.executable, "bench.py", "--steps", "1"], cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode != 0
    assert "needs a CUDA device" in r.stderr
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
