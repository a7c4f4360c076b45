"""Vocabulary tensor parallelism through the library, one process per vocabulary rank.

Each rank is its own process holding only its shard's W rows; it calls
rlk_linear_logprob_shard, the ranks all-gather their 16-byte records (gloo, staged through
host memory), and every rank merges them in shard order with rlk_lse_merge ("vLLM
RL-Kernel v0.1.0", boundary table: cross-rank LSE merge in a fixed rank order).  Every
rank's logprob and lse must equal the unsharded rlk_linear_logprob bit for bit.

This machine gives the test one GPU, so the ranks share it: each process has its own
context, and no kernel waits on another rank's kernel -- the exchange happens on the host
between launches, after each rank's stream has finished its shard.
"""
import datetime
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from invariant_selected_token_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs(case, device):
    """(hidden, W, targets, active) on `device`, the same in every process."""
    if case == "small":
        w = WL.small_case(300, 256, 5000, seed=71, inactive_frac=0.2)
        d = WL.to_device(w, device)
        return d.hidden, d.W, d.targets, d.active
    W = WL.head_weights(device)
    T = 96
    hidden = WL.rms_hidden(T, W.shape[1], device, seed=72)
    rng = np.random.default_rng(72)
    targets = torch.from_numpy(rng.integers(0, W.shape[0], T).astype(np.int32)).to(device)
    active = torch.from_numpy((rng.random(T) > 0.1).astype(np.uint8)).to(device)
    return hidden, W, targets, active


def _rank_main(rank, world, port, case, out_q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=120))
    try:
        from invariant_selected_token_gb300 import binding, vocab_parallel as VP
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        hidden, W, targets, active = _inputs(case, dev)
        vb, ve = VP.local_vocab_range(_V(case))
        W_local = W[vb:ve].contiguous()
        del W
        status = binding.new_status(dev)
        lp, lse = VP.linear_logprob_vocab_parallel(hidden, W_local, targets, active, _V(case),
                                                   status=status)
        torch.cuda.synchronize()
        binding.raise_on_device_status(status)
        out_q.put((rank, (vb, ve), lp.cpu().numpy().view(np.int32),
                   lse.cpu().numpy().view(np.int32)))
    except Exception as e:  # reported to the parent, which fails the test
        out_q.put((rank, None, repr(e), None))
    finally:
        dist.destroy_process_group()


def _V(case):
    return 5000 if case == "small" else WL.V_QWEN3_8B


@pytest.mark.parametrize("case,world", [("small", 2), ("small", 8), ("qwen", 4)])
def test_vocab_ranks_match_the_unsharded_call(rlk, cuda_device, case, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, case, q), daemon=True) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=600) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
    for r in res:
        assert r[1] is not None, "rank %d failed: %s" % (r[0], r[2])
    hidden, W, targets, active = _inputs(case, cuda_device)
    assert [r[1] for r in res] == rlk.shard_ranges(W.shape[0], world)
    ref_lp, ref_lse = rlk.linear_logprob(hidden, W, targets, active, world)
    ref_lp = ref_lp.cpu().numpy().view(np.int32)
    ref_lse = ref_lse.cpu().numpy().view(np.int32)
    for r in res:
        assert int((r[2] != ref_lp).sum()) == 0, "rank %d logprob" % r[0]
        assert int((r[3] != ref_lse).sum()) == 0, "rank %d lse" % r[0]
    for p in procs:
        assert p.exitcode == 0
