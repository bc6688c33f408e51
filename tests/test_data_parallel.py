"""Data parallelism over ranks: the token-count exchange, run as two gloo
ranks on the CPU (the loss itself is the oracle's here; on the GPU the same
orchestration calls the library's kernels)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from ppo_policy_loss_gb300 import dist as rldist

B, T, V = 6, 7, 13


def _problem():
    rng = np.random.default_rng(80)
    z = rng.normal(0, 1.5, (B * T, V))
    ids = rng.integers(0, V, B * T)
    L = np.array([7, 2, 0, 5, 1, 6])
    mask = (np.arange(T)[None, :] < L[:, None]).astype(np.uint8).reshape(-1)
    adv = np.repeat(rng.normal(0, 1, B), T)
    _, logp0, _ = oracle.row_stats(z, "f64", V, ids, mask, threads=1)
    lo = logp0 + rng.normal(0, 0.1, B * T)
    return z, ids, mask, adv, lo


def _count_fn(mask, b, t):
    m = mask.numpy().reshape(b, t)
    return torch.tensor([oracle.count(m), int((m.sum(1) > 0).sum())], dtype=torch.int64)


def _loss_fn(logits, ids, mask, adv, b, t, counts, logp_old=None, agg="token_mean", **kw):
    z, i, m = logits.numpy(), ids.numpy(), mask.numpy()
    _, logp, ent = oracle.row_stats(z, "f64", z.shape[1], i, m, threads=1)
    o = oracle.loss_from_stats(logp, ent, m, adv.numpy(), logp_old.numpy(), None, 0.2, 0.0, 0.03,
                               agg=agg, T=t, global_counts=counts.tolist())
    return {"loss_share": torch.tensor([o["loss"]], dtype=torch.float64)}


def _rank_main(rank, world, port, agg, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    z, ids, mask, adv, lo = _problem()
    rows = slice(rank * (B // world) * T, (rank + 1) * (B // world) * T)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x[rows]))
    out = rldist.policy_loss_data_parallel(t(z), t(ids), t(mask), t(adv), B // world, T,
                                           count_fn=_count_fn, loss_fn=_loss_fn,
                                           logp_old=t(lo), agg=agg)
    q.put((rank, float(out["loss"][0]), out["global_counts"].tolist()))
    dist.barrier()
    dist.destroy_process_group()


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("agg", ["token_mean", "seq_mean_token_mean"])
def test_two_ranks_reproduce_the_single_process_loss(agg):
    z, ids, mask, adv, lo = _problem()
    _, logp, ent = oracle.row_stats(z, "f64", V, ids, mask, threads=1)
    whole = oracle.loss_from_stats(logp, ent, mask, adv, lo, None, 0.2, 0.0, 0.03, agg=agg, T=T)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, agg, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, loss, counts in res:
        assert counts == [int(mask.sum()), 5]
        assert abs(loss - whole["loss"]) < 1e-12, (rank, loss, whole["loss"])


def _vp_rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    R = 5

    def partials_fn(logits, ids, mask, adv, b, t, off, total, **kw):
        # stand-in for the first launch: each row's entry tags the shard and the row
        return torch.tensor([[float(rank), float(r), float(off), float(total)] for r in range(R)])

    def merge_fn(logits, ids, mask, adv, b, t, off, total, gathered, **kw):
        return {"gathered": gathered.clone()}

    off = [0, 7, 11][rank]
    out = rldist.policy_loss_vocab_parallel(None, None, None, None, 1, R, off, 13,
                                            partials_fn=partials_fn, merge_fn=merge_fn)
    q.put((rank, out["gathered"].tolist()))
    dist.barrier()
    dist.destroy_process_group()


def test_vocab_parallel_exchange_orders_the_shards():
    """Three gloo ranks: the all-gather between the two launches hands every
    rank every shard's partials, in rank (shard) order, row by row."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_vp_rank_main, args=(r, 3, port, q)) for r in range(3)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, g in res:
        assert len(g) == 3
        for k, shard in enumerate(g):
            assert [row[0] for row in shard] == [float(k)] * 5
            assert [row[1] for row in shard] == [0.0, 1.0, 2.0, 3.0, 4.0]
            assert shard[0][2] == [0, 7, 11][k] and shard[0][3] == 13
