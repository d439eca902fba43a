"""The multi-rank bench path on CPU: two gloo ranks, independent batches, max-over-ranks time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    r = bench.Ranks(backend="gloo")
    t = 1.0 + rank  # rank 1 is the slow one
    units = 100 * (rank + 1)
    q.put((rank, r.max(t), r.sum(units), bench.rank_seed(4, rank)))
    r.barrier()
    r.close()


def test_two_gloo_ranks_reduce_time_and_units():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(i, world, port, q)) for i in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    assert all(g[1] == 2.0 for g in got)  # max over ranks
    assert all(g[2] == 300 for g in got)  # units summed over ranks
    assert got[0][3] != got[1][3]  # every rank verifies its own batch


def test_whole_job_value_and_subset():
    import bench
    from reject_row_vocab_gb300 import workload as wl
    assert bench.whole_job_value([100, 300], 2.0) == 200.0
    w = wl.ragged_block(batch=10, max_len=4, vocab=64, seed=3)
    s = bench.subset(w, 4)
    assert s.batch == 4 and s.rows == int(w.cu_seqlens[4]) and s.logits.shape[0] == s.rows
    t = wl.eagle2_tree(batch=3, topk=2, depth=2, keep=4, vocab=64, seed=4)
    st = bench.subset(t, 2)
    assert st.rows == 2 * t.nodes and st.tokens.shape == (2, t.nodes)
