"""The benchmark's multi-rank bookkeeping on CPU with two gloo ranks: the
max-over-ranks step time, the sum of the work over ranks, and rank 0 alone
printing (the reference arm exits without work on other ranks)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx = bench.dist_max(float(10 + rank))
    sm = bench.dist_sum(float(1 + rank))
    bench.barrier()
    r, w, l = bench.dist_env()
    results[rank] = (mx, sm, r, w, l)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
        res = dict(results)
    assert res[0][:2] == (11.0, 3.0) and res[1][:2] == (11.0, 3.0)
    assert res[0][2:] == (0, 2, 0) and res[1][2:] == (1, 2, 1)


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    import bench
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_warmup_floor():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
