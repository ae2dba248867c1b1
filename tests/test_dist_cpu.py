"""The replicas path of bench.py on two CPU ranks (gloo): barrier, the reductions
over ranks, the whole-job rate (units of all ranks over the slowest rank's
time), and the reference arm running on rank 0 only.  No GPU is used."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.Dist()
    try:
        assert dist.world == world and dist.rank == rank
        assert dist.pg is not None and dist.pg.get_backend() == "gloo"
        dist.barrier()
        # rank r contributes 10 (r + 1)
        mx = dist.max(10.0 * (rank + 1))
        sm = dist.sum(10.0 * (rank + 1))
        # rank r processed 100 (r + 1) units in 50 (r + 1) ms
        rate, ms = bench.job_rate(dist, 100.0 * (rank + 1), 50.0 * (rank + 1))
        # the reference arm runs on rank 0 alone; other ranks return without work
        ref = bench.run_reference(None, dist) if rank != 0 else "skipped"
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{mx} {sm} {rate} {ms} {ref is None}\n")
    finally:
        dist.close()


@pytest.mark.timeout(180)
def test_replicas_two_gloo_ranks(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(150)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    expect_rate = (100.0 + 200.0) / (100.0 * 1e-3)   # 300 units over the slower 100 ms
    for r in range(world):
        mx, sm, rate, ms, ref_none = open(tmp_path / f"rank{r}.txt").read().split()
        assert float(mx) == 20.0 and float(sm) == 30.0
        assert float(ms) == 100.0
        assert abs(float(rate) - expect_rate) < 1e-9 * expect_rate
        if r != 0:
            assert ref_none == "True"
