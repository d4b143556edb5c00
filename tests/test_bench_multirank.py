"""Host logic of bench.py's multi-rank run, on CPU with the gloo backend (world size 2).

Every rank runs its own replica of the workload (weak scaling): the step time is the slowest rank's
(barrier + all-reduce MAX), the reported value counts the units of all ranks, and only rank 0 prints.
The reference arm runs on rank 0 alone; the other ranks return at once without work.
"""
import contextlib
import io
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_setup()
    # each rank times its own replica; rank 1 is the slow one
    ms_local = 2.0 if r == 0 else 3.0
    ms_max = bench.barrier_max(ms_local, w, "cpu")
    rate = bench.whole_job_rate(1000.0, w, ms_max)

    class Args:
        gpus, steps, warmup = world, 1, 3

    buf = io.StringIO()
    rc = None
    if r != 0:  # the reference arm on a rank other than 0: no work, no output
        with contextlib.redirect_stdout(buf):
            rc = bench.run_reference(Args)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "ms_max": ms_max, "rate": rate, "ref_rc": rc,
                   "ref_out": buf.getvalue()}, f)


def test_bench_two_ranks_gloo(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a gloo rank did not finish")
        assert p.exitcode == 0
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert (d["world"], d["rank"], d["local"]) == (world, r, r)
        assert d["ms_max"] == 3.0  # the slowest rank's time on every rank
        assert d["rate"] == pytest.approx(1000.0 * world / 3e-3)  # all ranks' units over the slowest time
    assert res[1]["ref_rc"] == 0 and res[1]["ref_out"] == ""


def test_whole_job_rate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.barrier_max(1.25, 1, "cpu") == 1.25
    assert bench.whole_job_rate(805306368, 1, 0.2) == pytest.approx(805306368 / 0.2e-3)
