"""Data-parallel host logic with two gloo ranks on the CPU: sharding by
sequence and summing the d_rab gradients over ranks equals the single-process
result, and the timing aggregation takes the max time and the summed work."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from hstu_jagged_attention_02_gb300 import dp, synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    return synth.make_batch([5, 40, 17, 66, 3, 29], H=2, d_qk=8, d_v=8, dtype="fp32",
                            num_contexts=[1, 2, 0, 3, 0, 1], num_targets=[1, 4, 2, 6, 1, 3], seed=321)


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import oracle as O
        b = _batch()
        shards = dp.lpt_shard(dp.sequence_costs(b), world)
        mine = dp.gather_sequences(b, shards[rank])
        g = O.backward(mine)
        drp = torch.from_numpy(np.ascontiguousarray(g["d_rab_pos"]))
        drt = torch.from_numpy(np.ascontiguousarray(g["d_rab_time"]))
        dp.allreduce_sum_([drp, drt])
        ms, work = dp.reduce_step_time(10.0 + rank, float(dp.sequence_costs(mine).sum()))
        q.put((rank, shards, drp.numpy(), drt.numpy(), ms, work))
    finally:
        dist.destroy_process_group()


def test_lpt_shard_balances_and_covers():
    costs = [100, 90, 80, 70, 10, 5, 5, 1]
    sh = dp.lpt_shard(costs, 3)
    assert sorted(sum(sh, [])) == list(range(8))
    loads = [sum(costs[i] for i in s) for s in sh]
    assert max(loads) - min(loads) <= max(costs)


def test_two_gloo_ranks_match_single_process():
    from oracle import oracle as O
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=300) for _ in range(world)], key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    b = _batch()
    full = O.backward(b)
    shards = res[0][1]
    assert shards == res[1][1]
    assert sorted(shards[0] + shards[1]) == list(range(b.B))
    for r in res:
        np.testing.assert_allclose(r[2], full["d_rab_pos"], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(r[3], full["d_rab_time"], rtol=1e-10, atol=1e-12)
        assert r[4] == 11.0                                   # max over ranks
        assert r[5] == float(dp.sequence_costs(b).sum())      # summed work


def _layer_batch():
    r = np.random.default_rng(77)
    H, d = 2, 4
    D = H * d
    hist = np.array([5, 9, 14, 3, 11])
    nt = np.array([2, 3, 1, 2, 4], np.int32)
    lengths = hist + nt
    off = synth.offsets_from_lengths(lengths)
    T = int(off[-1])
    ts = np.concatenate([np.sort(r.integers(0, 4000, size=n)) for n in lengths]).astype(np.int64)
    empty = np.zeros((T, H, 0))
    return synth.Batch(name="layer", seed=77, dtype="fp32", B=5, H=H, d_qk=d, d_v=d, lengths=lengths,
                       offsets=off, num_targets=nt, num_contexts=None, timestamps=ts, q=empty, k=empty, v=empty,
                       u=None, dy=None, rab_pos=r.normal(0, 0.2, (H, 128)), rab_time=r.normal(0, 0.2, (H, 64)),
                       alpha=0.5, max_seq_len=int(lengths.max()), x=r.standard_normal((T, D)),
                       w1=r.normal(0, 0.3, (D, 4 * D)), w2=r.normal(0, 0.3, (D, D)),
                       dout=r.standard_normal((T, D)))


def _layer_worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import oracle as O
        b = _layer_batch()
        shards = dp.lpt_shard(dp.sequence_costs(b), world)
        g = O.layer_backward(dp.gather_sequences(b, shards[rank]))
        grads = [torch.from_numpy(np.ascontiguousarray(g[k])) for k in ("dw1", "dw2", "d_rab_pos", "d_rab_time")]
        dp.allreduce_sum_(grads)
        q.put((rank, [t.numpy() for t in grads]))
    finally:
        dist.destroy_process_group()


def test_layer_gradients_all_reduced_over_two_ranks_match_single_process():
    from oracle import oracle as O
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_layer_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full = O.layer_backward(_layer_batch())
    for _, grads in res:
        for got, key in zip(grads, ("dw1", "dw2", "d_rab_pos", "d_rab_time")):
            np.testing.assert_allclose(got, full[key], rtol=1e-9, atol=1e-12)
