"""The multi-GPU path of bench.py is replicas: each rank decodes its own
request batch, and the reported time is the max over ranks.  Its host logic
runs here as two gloo ranks on the CPU."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import synth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    u = synth.make_requests(4, 8, bench.request_seed(r))
    ms = 1.0 + r                      # ranks finish at different times
    bench.barrier(w)
    worst = bench.max_over_ranks(ms, w, "cpu")
    out[rank] = (r, w, local, worst, float(u[0, 0]))
    dist.destroy_process_group()


def test_two_rank_replicas():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, w, local, worst, u0) in res.items():
        assert r == rank and w == world and local == rank
        assert worst == 2.0                       # the slower rank's time
    assert res[0][4] != res[1][4]                 # each replica decodes its own requests


def test_single_process_defaults(monkeypatch):
    import bench
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.request_seed(0) != bench.request_seed(1)
    assert np.isfinite(bench.step_bytes(
        {"live_beams": 2, "index_bytes": 20, "legal_slots": 5, "unique_tokens": 5, "chunks": 2},
        __import__("synth").CONFIGS["tiny"], 2))
