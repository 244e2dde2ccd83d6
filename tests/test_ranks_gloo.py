"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank reports a different step time; both must agree on the maximum, the
aggregate throughput must count every rank's tokens over that maximum, and the
per-rank input seeds must differ (independent batches, weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from kimi_delta_attention_08_gb300 import ranks


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = ranks.world_info()
        ms = 10.0 + 5.0 * r                      # rank 1 is the slow one
        mx = ranks.max_over_ranks(ms, dist)
        dist.barrier()
        q.put((r, w, lr, mx, ranks.aggregate_tokens_per_s(32768, w, mx),
               ranks.rank_seed(0, r)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[3] == pytest.approx(15.0) for r in res)
    assert all(r[4] == pytest.approx(2 * 32768 / 15e-3) for r in res)
    assert res[0][5] != res[1][5]


def test_single_rank_is_identity():
    assert ranks.max_over_ranks(3.5) == 3.5
    assert ranks.aggregate_tokens_per_s(1000, 1, 2.0) == pytest.approx(5e5)


def test_spawn_world_brings_up_two_ranks(tmp_path):
    """The launcher bench.py uses for --gpus N when no launcher set WORLD_SIZE:
    two processes on 127.0.0.1, ranks 0 and 1 of a world of 2, one collective."""
    import json
    probe = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rank_probe.py")
    assert ranks.spawn_world(2, [probe, str(tmp_path)]) == 0
    recs = sorted((json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)),
                  key=lambda r: r["rank"])
    assert [r["rank"] for r in recs] == [0, 1] and [r["local"] for r in recs] == [0, 1]
    assert all(r["world"] == 2 and r["sum"] == 3.0 for r in recs)


def test_bench_rejects_world_size_mismatch():
    """Under a launcher whose WORLD_SIZE differs from --gpus, bench.py exits 2
    before touching a GPU."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="3", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 2 and "WORLD_SIZE is 3" in r.stderr


def _exchange_worker(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist
    from kimi_delta_attention_08_gb300 import shard, synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # this rank's piece: (M_r, B_r) of 3 states, seeded by rank
        piece = torch.from_numpy(np.stack([synth.normal_f32((3, 128, 128), 700 + rank, 1, 0.05),
                                           synth.normal_f32((3, 128, 128), 700 + rank, 2)]))
        pieces = shard.exchange(piece)
        q.put((rank, pieces.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_shard_exchange_orders_pieces_by_rank(world):
    """The sharded forward's exchange over gloo ranks: every rank receives every
    rank's (M, B) piece in rank order, so composing the first r pieces (here in
    fp64 numpy, in the test) gives each rank the same start state as the pieces
    drawn independently would."""
    import numpy as np
    from kimi_delta_attention_08_gb300 import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = [(synth.normal_f32((3, 128, 128), 700 + r, 1, 0.05),
               synth.normal_f32((3, 128, 128), 700 + r, 2)) for r in range(world)]
    for r in range(world):
        got = res[r]
        assert got.shape == (world, 2, 3, 128, 128)
        for s in range(world):
            assert np.array_equal(got[s, 0], expect[s][0]) and np.array_equal(got[s, 1], expect[s][1])
        # start state of rank r from the gathered pieces equals the independent fold
        X, Y = np.zeros((3, 128, 128)), np.zeros((3, 128, 128))
        for s in range(r):
            X = X @ got[s, 0].astype(np.float64) + got[s, 1]
            Y = Y @ expect[s][0].astype(np.float64) + expect[s][1]
        assert np.array_equal(X, Y)
