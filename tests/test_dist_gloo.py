"""Multi-rank host logic of the benchmark, on CPU with the gloo backend (world size 2)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from state_space_sequence_trapezoidal_b300 import dist as d


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, _ = d.init("gloo")
    d.barrier()
    local_ms = 10.0 + 5.0 * r  # rank 1 is the slow one
    m = d.max_over_ranks(local_ms)
    out[r] = (r, w, m, d.rank_seed(100, r), d.aggregate_throughput(32768, w, m / 1e3))
    d.barrier()
    import torch.distributed as td

    td.destroy_process_group()


def test_two_ranks_take_the_max_time_and_distinct_seeds():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][1] == res[1][1] == 2
    assert res[0][2] == res[1][2] == pytest.approx(15.0)
    assert res[0][3] != res[1][3]
    assert res[0][4] == pytest.approx(32768 * 2 / 0.015)


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert d.env_rank() == (0, 1, 0)
    assert d.max_over_ranks(3.5) == 3.5
