"""The N > 1 host logic of bench.py on CPU: two gloo ranks (world size 2).

Each rank owns an independent shard of sequences (its own seed), there is no
data-path collective, and the ranks meet only in the barrier around the timed
region and the max / sum reductions that turn per-rank times and token counts
into the whole-job value."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
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
    import bench
    from mamba2_ssm_decode_gb300 import workloads as W
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    dev = torch.device("cpu")
    # each rank: its own shard (seed + rank) of the same workload shape
    case = W.tiny(seed=100 + rank)
    tokens, nbytes, _ = bench.accounting(case)
    bench.barrier(w)
    fake_ms = 10.0 + 5.0 * rank            # rank 1 is the slower one
    t_max = bench.max_over_ranks(fake_ms, w, dev)
    tok_all = bench.sum_over_ranks(tokens, w, dev)
    q.put((rank, t_max, tok_all, tokens, float(case.x.float().sum())))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(world))
    (r0, tmax0, all0, tok0, x0), (r1, tmax1, all1, tok1, x1) = res
    assert tmax0 == tmax1 == 15.0                   # max over ranks
    assert all0 == all1 == tok0 + tok1              # whole-job tokens
    assert x0 != x1                                 # distinct shards


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["RANK"], os.environ["WORLD_SIZE"] = "1", "2"
    try:
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    finally:
        os.environ.pop("RANK")
        os.environ.pop("WORLD_SIZE")
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("name", ["mamba2-2.7b-decode", "mtp-varlen"])
def test_accounting_matches_formula(name):
    """Algorithmic bytes of the default workloads against the closed-form count."""
    sys.path.insert(0, ROOT)
    import bench
    from mamba2_ssm_decode_gb300 import workloads as W
    case = W.WORKLOADS[name](device="cpu")
    tokens, nbytes, _ = bench.accounting(case)
    slots, H, P, N, G = case.dims
    block = H * P * N * case.state.element_size()
    if name == "mamba2-2.7b-decode":
        valid = int((case.state_batch_indices != case.pad_slot_id).sum())
        assert valid == 243 and tokens == 243
        rows_part = 256 * (H * P * 2 * 3 + H * 4 + 2 * G * N * 2)
        assert nbytes == 2 * valid * block + rows_part + 256 * 4
    else:
        rows = case.rows
        assert tokens == rows                      # no pad sequences in this workload
        rows_part = rows * (H * P * 2 * 3 + H * 4 + 2 * G * N * 2)
        meta = 2 * 128 * 4 * 4 + 129 * 4 + 128 * 4
        assert nbytes == (128 + rows) * block + rows_part + meta
