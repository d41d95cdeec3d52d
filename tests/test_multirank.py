"""Host logic of the multi-GPU launch, run as two gloo ranks on the CPU.

Every (b, h) problem of the mixer is independent, so N GPUs run N replicas, each on its
own seeded batch, with no collective on the data path.  What the ranks share is the
timing: the whole-job rate is all ranks' tokens over the slowest rank's step time.  These
tests check, with world_size 2 over gloo at 127.0.0.1, that the ranks draw different
batches, that the max-over-ranks reduction and the whole-job rate are right, and that a
rank that raises is reported instead of hanging the other.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out, fail_rank):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import datetime

    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    try:
        import bench
        import synth_inputs as si
        if rank == fail_rank:
            raise RuntimeError("injected failure on rank %d" % rank)
        inp = si.sequence_inputs(1, 2, 32, 16, 16, dtype="bf16", qkv_std=0.25, seed=bench.rank_seed(3, rank))
        step_ms = [4.0, 6.5][rank]
        mx = bench.max_over_ranks(step_ms, world, device="cpu")
        rate = bench.whole_job_rate(1000, world, mx)
        out.put((rank, float(inp["q"].float().sum()), mx, rate))
    except Exception as e:   # reported to the parent; the other rank's collective times out
        out.put((rank, "error", str(e), None))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:
            pass


def _run(world, fail_rank=-1):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out, fail_rank)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r = out.get(timeout=120)
        res[r[0]] = r[1:]
    for p in procs:
        p.join(timeout=60)
    return res


def test_two_ranks_distinct_batches_and_max_time():
    res = _run(2)
    (s0, mx0, rate0), (s1, mx1, rate1) = res[0], res[1]
    assert s0 != s1                                   # each rank draws its own batch
    assert mx0 == mx1 == 6.5                          # slowest rank's step time
    assert rate0 == rate1 == pytest.approx(2 * 1000 / 6.5e-3)


def test_failing_rank_is_reported_not_hung():
    res = _run(2, fail_rank=1)
    assert res[1][0] == "error" and "injected failure" in res[1][1]
    # rank 0 either finished its reduction with an error (peer gone) or reported one
    assert 0 in res
