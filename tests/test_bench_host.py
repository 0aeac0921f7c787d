"""Host logic of bench.py's multi-rank path on CPU: two gloo ranks, max of the
times and sum of the work across ranks (the only cross-rank step; there is no
collective on the data path)."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        secs, units = bench.reduce_over_ranks(1.0 + rank, 100.0 * (rank + 1))
        bench.barrier()
        q.put((rank, secs, units))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, secs, units in got:
        assert secs == 2.0 and units == 300.0


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(1.5, 7.0) == (1.5, 7.0)


def test_reference_arm_runs_on_cpu(capsys):
    sys.path.insert(0, ROOT)
    import json
    import bench
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
                "--ref-step-seconds", "0.2"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cpu_model"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_step_budget_shrinks_with_steps(capsys):
    """The oracle time of the whole reference run stays near
    --ref-total-seconds: here 7 steps of 0.1 s are raised to the 0.25 s
    floor."""
    sys.path.insert(0, ROOT)
    import json
    import bench
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "4", "--warmup", "3",
                "--ref-total-seconds", "0.7"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert "~0.25 s" in line["config"]["sample"]
    assert 0 < line["ms_per_step"] < 1000


def test_oracle_inputs_fill_every_used_block():
    """Host inputs of the oracle arm: every block a sequence reaches holds
    drawn values (no all-zero block), blocks no sequence uses stay zero, and
    the values look N(0, 1)."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from paged_kv_cache_64_gb300 import workloads
    plan = workloads.make_plan("qwen", num_seqs=16)
    lay, q, k, v = bench.oracle_inputs(plan)
    B = plan.spec.block_size
    used = set()
    for s, L in enumerate(lay.seq_lens):
        used.update(lay.block_tables[s, :-(-int(L) // B)].tolist())
    used = np.array(sorted(used))
    unused = np.setdiff1d(np.arange(plan.num_blocks), used)
    for pool in (k, v):
        assert (pool[used].reshape(len(used), -1) != 0).any(axis=1).all()
        assert not pool[unused[:1000]].any()
    vals = k[used].view(np.float16).astype(np.float64)  # qwen pools are fp16
    assert abs(vals.mean()) < 0.01 and abs(vals.std() - 1) < 0.01
    assert q.shape == (16, 14, 64) and q.dtype == np.uint16


def test_cow_and_apc_arguments_are_checked():
    """--cow is the prefix workload's copy-on-write reading (forks only);
    --gpus N must match the ranks the launcher started (one process here)."""
    sys.path.insert(0, ROOT)
    import pytest
    import bench
    assert "WORLD_SIZE" not in os.environ
    for argv in (["--workload", "llama", "--cow"], ["--workload", "prefix", "--cow", "--apc"],
                 ["--workload", "qwen", "--apc"], ["--warmup", "2"], ["--gpus", "2"],
                 ["--impl", "reference", "--gpus", "4"], ["--steps", "0"]):
        with pytest.raises(SystemExit):
            bench.main(argv)
