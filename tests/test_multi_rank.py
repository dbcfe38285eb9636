"""The multi-process path of bench.py on the CPU (gloo, world size 2).

The layer partitions into independent sequences, so N GPUs run N replicas
with no data-path collective; the only cross-rank steps are the timing
barrier and the max-over-ranks reduction, and the reference arm runs on
rank 0 alone.  These tests run those steps as two gloo processes.
"""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from varlen_gated_delta_gb300 import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench._dist()
        # rank r timed (3 + r) ms for the layer and (10 - r) ms end to end
        ms, e2e = bench._max_over_ranks([3.0 + r, 10.0 - r], "cpu")
        wl = W.WORKLOADS["tiny"]
        d = W.make_inputs(wl, "cpu", seed=bench._replica_seed(wl, r))
        dist.barrier()
        out[r] = (w, r, ms, e2e, float(d["qkv"].double().sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_draw_distinct_batches():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in (0, 1):
        w, rank, ms, e2e, _ = res[r]
        assert (w, rank) == (2, r)
        assert ms == 4.0 and e2e == 10.0          # the slowest replica on every rank
    assert res[0][4] != res[1][4]                # replicas draw different batches


def test_whole_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._job_tokens_per_s(1, 64, 50, 2.5) == pytest.approx(64 * 50 / 2.5e-3)
    assert bench._job_tokens_per_s(4, 64, 50, 2.5) == pytest.approx(4 * 64 * 50 / 2.5e-3)
    # a single process: the reduction is the identity
    assert bench._max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """The driver's N > 1 launch of the reference arm: two ranks on the CPU,
    rank 0 times the oracle and prints the only JSON line, rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2",
           "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the JSON line carries every key of the benchmark contract
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["metric"] == "gated-delta layer tokens/s" and line["unit"] == "tokens/s"
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["config"]["workload"] == "tiny" and line["steps"] == 2
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["cores"] >= 1
