"""The multi-process path of bench.py on CPU: two ranks over gloo (127.0.0.1),
as torchrun launches them on one node. Each rank draws its own rows (weak
scaling, no data-path collective), the timed region is closed by a barrier,
its time is the maximum over ranks, and the reported value is the whole job's
units over that time."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    from sparse_mla_attention_04_gb300 import inputs
    r, w, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    # a rank-dependent "elapsed time": every rank must see the slowest one
    ms_max = bench.max_over_ranks(2.0 + 3.0 * r, w, "cpu")
    # the rank's own rows: the decode workload's index sets, shrunk to a tiny pool
    wl = inputs.decode(n_seqs=4, ctx=4096, topk=128, name="decode_small")
    idx = inputs.make_indices(wl, seed=bench.rank_seed(0, 0, r))
    mine = torch.from_numpy(idx.astype(np.int64))
    gathered = [torch.empty_like(mine) for _ in range(w)]
    torch.distributed.all_gather(gathered, mine)   # test-side check only
    bench.barrier(w)
    out.put((r, w, ms_max, [g.numpy() for g in gathered]))
    torch.distributed.destroy_process_group()


def test_two_ranks_over_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = [out.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort(key=lambda x: x[0])
    for r, w, ms_max, gathered in res:
        assert w == 2
        assert ms_max == 5.0                      # the slower rank's time, on every rank
    a, b = res[0][3]
    assert a.shape == b.shape                     # same workload shape per rank
    assert not np.array_equal(a, b)               # but each rank has its own rows
    assert np.array_equal(res[0][3][1], res[1][3][1])


def test_job_rate_and_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks, 1e9 bytes each, slowest 10 ms -> 2e11 B/s for the job
    assert bench.job_rate(1e9, 2, 10.0) == pytest.approx(2e11)
    assert bench.job_rate(1e9, 1, 10.0) == pytest.approx(1e11)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5   # world 1: no collective
    bench.barrier(1)
    assert bench.rank_seed(7, 0, 0) != bench.rank_seed(7, 0, 1)
    assert bench.rank_seed(7, 1, 0) != bench.rank_seed(7, 0, 0)
