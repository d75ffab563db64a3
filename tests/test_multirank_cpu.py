"""The N > 1 path of bench.py on CPU: two gloo ranks (no GPU).

Decode shards by sequence with no exchange step: rank r of N takes sequences
[r B, (r + 1) B) of an N x B job; the only collectives are the barrier and the
max over ranks of the timed region.  Checked here: the process-group setup the
bench uses (RANK / WORLD_SIZE / MASTER_* from the environment, 127.0.0.1), the
max-over-ranks reduction, that the shards cover the job exactly once and equal
the same rows of the whole job's inputs, that the oracle run on each shard
gives the same outputs as on the whole batch (sharding changes no value), and
the whole-job throughput formula.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from oracle.layer import OracleLayer
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), BENCH_BACKEND="gloo")
    import torch
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    # max over ranks of the timed region
    out[f"max{rank}"] = bench.max_over_ranks(10.0 + rank, w, "cpu")
    # this rank's shard of a small Mamba-2 job and of a GDN job
    results = []
    for kind, wl in (
        ("m2", configs.Mamba2Workload(LayerShape(MAMBA2, batch=world * 3, n_heads=4, n_groups=2, d_head=16,
                                                 d_state=16, ring_len=3), seed=31, s0_std=0.1)),
        ("gdn", configs.GdnWorkload(LayerShape(GDN, batch=world * 3, n_heads=4, n_groups=2, d_head=16, d_state=16,
                                               ring_len=3), seed=32, s0_std=0.05)),
    ):
        sh = bench.shard_of(wl, rank, w)
        lay = OracleLayer(sh.shape, list(range(sh.shape.batch)), sh.S0(), A=sh.A() if kind == "m2" else None)
        ys = [lay.decode(sh.step(t)) for t in range(5)]
        results.append((kind, sh.b0, sh.b1, np.stack(ys)))
    out[f"res{rank}"] = results
    dist.barrier()
    dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=180)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        return world, dict(out)


def test_max_over_ranks_with_gloo(two_ranks):
    world, out = two_ranks
    assert out["max0"] == out["max1"] == 10.0 + world - 1


def test_shards_cover_the_job_and_match_the_whole_batch(two_ranks):
    world, out = two_ranks
    for i, kind in enumerate(("m2", "gdn")):
        ranges = sorted((out[f"res{r}"][i][1], out[f"res{r}"][i][2]) for r in range(world))
        assert ranges == [(0, 3), (3, 6)]  # disjoint, contiguous, the whole job
        wl = (configs.Mamba2Workload(LayerShape(MAMBA2, batch=world * 3, n_heads=4, n_groups=2, d_head=16,
                                                d_state=16, ring_len=3), seed=31, s0_std=0.1) if kind == "m2"
              else configs.GdnWorkload(LayerShape(GDN, batch=world * 3, n_heads=4, n_groups=2, d_head=16, d_state=16,
                                                  ring_len=3), seed=32, s0_std=0.05))
        whole = OracleLayer(wl.shape, list(range(wl.shape.batch)), wl.S0(), A=wl.A() if kind == "m2" else None)
        ys = np.stack([whole.decode(wl.step(t)) for t in range(5)])
        for r in range(world):
            _, b0, b1, y_shard = out[f"res{r}"][i]
            np.testing.assert_array_equal(y_shard, ys[:, b0:b1])


def test_shard_inputs_are_rows_of_the_job():
    wl = configs.Mamba2Workload(configs.CONFIG0.with_batch(4), seed=33, s0_std=0.1)
    sh = bench.shard_of(wl, 1, 2)
    full = wl.step(7)
    part = sh.step(7)
    for k in full:
        np.testing.assert_array_equal(part[k], full[k][2:4])
    np.testing.assert_array_equal(sh.S0(), wl.S0()[2:4])
    with pytest.raises(ValueError):
        bench.shard_of(configs.Mamba2Workload(configs.CONFIG0.with_batch(3), seed=33, s0_std=0.1), 0, 2)


def test_job_value_counts_every_rank():
    # 4 ranks x 256 sequences x 100 steps in a slowest-rank time of 20 ms
    assert bench.job_value(4, 256, 100, 20.0) == pytest.approx(4 * 256 * 100 / 0.020)
