"""Vocabulary tensor parallelism's host logic on CPU ranks (gloo), no GPU.

``vocab_parallel.linear_logprob_vocab_parallel`` gives rank r the W rows of shard r,
computes that shard's records, all-gathers every rank's records into rank order and
merges them in shard order ("vLLM RL-Kernel v0.1.0", boundary table: cross-rank LSE
merge, fixed rank reduction order).  Here the library's shard and merge calls are
replaced by the fp64 oracle's per-range record and merge (rounded to the 16-byte fp32
record on the way), so these tests check what the exchange itself must get right on
2 and 4 ranks: which rows each rank holds, that slot i of the gathered records is shard
i's, that every rank ends with the same result, and that it is the full-vocabulary
result.  A rank that fails before the exchange makes its peers' exchange fail with an
error instead of hanging.
"""
import datetime
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port, timeout_s=60):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))


def _case():
    from invariant_selected_token_gb300 import workloads as WL
    return WL.small_case(7, 32, 1000, seed=61, inactive_frac=0.3)


def _to_record(M, S, tl, owned):
    rec = np.zeros((M.shape[0], 4), dtype=np.int32)
    rec[:, 0] = M.astype(np.float32).view(np.int32)
    rec[:, 1] = S.astype(np.float32).view(np.int32)
    rec[:, 2] = tl.astype(np.float32).view(np.int32)
    rec[:, 3] = owned.astype(np.int32)
    return torch.from_numpy(rec)


def _rank_main(rank, world, port, out_q):
    _init(rank, world, port)
    try:
        from invariant_selected_token_gb300 import vocab_parallel as VP
        from oracle import linear_logprob as O
        w = _case()
        V = w.W.shape[0]
        L = O.logits(w.hidden, w.W)
        vb, ve = VP.local_vocab_range(V)
        W_local = torch.from_numpy(w.W[vb:ve].view(np.int16)).view(torch.bfloat16)
        seen = {}

        def shard_fn(hidden, W_shard, targets, active, V_total, n, r, workspace=None, status=None):
            assert (V_total, n, r) == (V, world, rank) and W_shard.shape[0] == ve - vb
            return _to_record(*O.shard_partial(L, vb, ve, w.targets))

        def merge_fn(parts, active, status=None):
            assert len(parts) == world
            ranges = O.shard_vocab_ranges(V, world)
            for i, p in enumerate(parts):   # slot i holds shard i's records
                want = _to_record(*O.shard_partial(L, ranges[i][0], ranges[i][1], w.targets))
                assert torch.equal(p, want), "slot %d" % i
            a = np.asarray([p.numpy() for p in parts])
            recs = [(a[i, :, 0].view(np.float32).astype(np.float64),
                     a[i, :, 1].view(np.float32).astype(np.float64),
                     a[i, :, 2].view(np.float32).astype(np.float64), a[i, :, 3])
                    for i in range(world)]
            lse, tl, owners = O.merge_partials(recs)
            seen["owners"] = owners
            act = np.asarray(active).astype(bool)
            return (torch.from_numpy(np.where(act, tl - lse, 0.0)),
                    torch.from_numpy(np.where(act, lse, 0.0)))

        act = torch.from_numpy(w.active)
        lp, lse = VP.linear_logprob_vocab_parallel(
            torch.zeros((w.T, 32), dtype=torch.bfloat16), W_local, torch.from_numpy(w.targets),
            act, V, shard_fn=shard_fn, merge_fn=merge_fn)
        assert np.all(seen["owners"] == 1)
        out_q.put((rank, (vb, ve), lp.numpy(), lse.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_vocab_parallel_exchange_on_gloo_ranks(world):
    from oracle import linear_logprob as O
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q), daemon=True) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = _case()
    ranges = O.shard_vocab_ranges(w.W.shape[0], world)
    assert [r[1] for r in res] == [tuple(x) for x in ranges]   # rank r holds shard r
    for r in res[1:]:                                           # every rank the same result
        assert np.array_equal(r[2], res[0][2]) and np.array_equal(r[3], res[0][3])
    ref_lp, ref_lse = O.selected_logprob(w.hidden, w.W, w.targets, w.active)
    assert np.abs(res[0][2] - ref_lp).max() <= 1e-5
    assert np.abs(res[0][3] - ref_lse).max() <= 1e-5 * np.abs(ref_lse).max()


def _gather_main(rank, world, port, out_q):
    _init(rank, world, port)
    try:
        from invariant_selected_token_gb300 import vocab_parallel as VP
        T = 5
        rec = (torch.arange(T * 4, dtype=torch.int32).view(T, 4) + 1000 * rank)
        parts = VP.gather_records(rec)
        out_q.put((rank, [p.clone() for p in parts]))
    finally:
        dist.destroy_process_group()


def test_gather_records_rank_order():
    world, port = 4, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gather_main, args=(r, world, port, q), daemon=True) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    base = torch.arange(20, dtype=torch.int32).view(5, 4)
    for _, parts in res:
        assert len(parts) == world
        for i, p in enumerate(parts):
            assert torch.equal(p, base + 1000 * i)


def _failing_main(rank, world, port, out_q):
    _init(rank, world, port, timeout_s=20)
    from invariant_selected_token_gb300 import vocab_parallel as VP
    if rank == 1:
        out_q.put((rank, "left before the exchange"))
        out_q.close()
        out_q.join_thread()   # the message is sent before the process goes
        os._exit(0)           # leaves between steps: nothing of its own in flight
    try:
        VP.gather_records(torch.zeros((3, 4), dtype=torch.int32))
        out_q.put((rank, "exchange completed"))
    except Exception as e:  # the peer is gone: gloo reports it
        out_q.put((rank, "error: %s" % type(e).__name__))


def test_rank_leaving_before_exchange_fails_the_peer_not_hangs():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_failing_main, args=(r, world, port, q), daemon=True) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    assert res[1] == "left before the exchange"
    assert res[0].startswith("error:"), res[0]


def _three_main(rank, world, port, out_q):
    _init(rank, world, port)
    try:
        from invariant_selected_token_gb300 import vocab_parallel as VP
        try:
            VP.local_vocab_range(1000)
            out_q.put((rank, "accepted"))
        except ValueError as e:
            out_q.put((rank, "refused: %s" % e))
    finally:
        dist.destroy_process_group()


def test_group_of_three_ranks_is_refused():
    """The shards are nodes of the tile tree, so a group must have 1, 2, 4 or 8 ranks."""
    world, port = 3, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_three_main, args=(r, world, port, q), daemon=True) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(v.startswith("refused") for v in res.values()), res
