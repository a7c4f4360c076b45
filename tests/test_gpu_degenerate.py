"""Degenerate batches: every row inactive, one active row among inactive ones,
the smallest vocabularies, one shard per tile.

Inactive rows get logprob = lse = +0 and zero gradients whatever their hidden
row holds, and their targets are never read (an out-of-range one raises no
status bit).  A lone active row gets the bits it gets alone.  The smallest
vocabularies follow the fp64 oracle like any other; with one column the
logprob is exactly 0 (lse = the target logit).
"""
import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL
from oracle import linear_logprob as O

pytestmark = pytest.mark.gpu

T, H, V = 300, 256, 1100  # 9 vocabulary tiles, the last one ragged


def bits(t):
    return t.contiguous().view(torch.int32)


def batch(cuda_device, seed):
    wl = WL.small_case(T, H, V, seed=seed)
    return wl, WL.to_device(wl, cuda_device)


@pytest.mark.parametrize("n_shards", [1, 2, 8])
def test_all_rows_inactive(rlk, cuda_device, n_shards):
    _, w = batch(cuda_device, 41)
    targets = torch.full((T,), -7, dtype=torch.int32, device=cuda_device)
    active = torch.zeros(T, dtype=torch.uint8, device=cuda_device)
    status = rlk.new_status(cuda_device)
    lp, lse = rlk.linear_logprob(w.hidden, w.W, targets, active, n_shards, status=status)
    L = rlk.debug_logits(w.hidden, w.W)
    lpm, lsem = rlk.logits_logprob(L, targets, active, n_shards, status=status)
    g = torch.ones(T, dtype=torch.float32, device=cuda_device)
    dh, dW = rlk.linear_logprob_backward(w.hidden, w.W, targets, g, lse, active, status=status)
    torch.cuda.synchronize()
    rlk.raise_on_device_status(status)
    for out in (lp, lse, lpm, lsem):
        assert torch.all(bits(out) == 0)  # +0.0
    assert torch.all(dh == 0) and torch.all(dW == 0)


def test_lone_active_row(rlk, cuda_device):
    _, w = batch(cuda_device, 43)
    r = 137
    active = torch.zeros(T, dtype=torch.uint8, device=cuda_device)
    active[r] = 1
    targets = torch.full((T,), 1 << 30, dtype=torch.int32, device=cuda_device)
    targets[r] = w.targets[r]
    status = rlk.new_status(cuda_device)
    lp, lse = rlk.linear_logprob(w.hidden, w.W, targets, active, 4, status=status)
    lp1, lse1 = rlk.linear_logprob(w.hidden[r:r + 1].contiguous(), w.W,
                                   w.targets[r:r + 1].contiguous(), None, 4)
    torch.cuda.synchronize()
    rlk.raise_on_device_status(status)
    assert torch.equal(bits(lp[r:r + 1]), bits(lp1)) and torch.equal(bits(lse[r:r + 1]), bits(lse1))
    others = torch.ones(T, dtype=torch.bool, device=cuda_device)
    others[r] = False
    assert torch.all(bits(lp[others]) == 0) and torch.all(bits(lse[others]) == 0)


@pytest.mark.parametrize("v,n_shards", [(1, 1), (2, 1), (127, 1), (128, 1), (129, 2), (256, 2),
                                        (257, 2), (1024, 8)])
def test_small_vocabularies(rlk, cuda_device, v, n_shards):
    wl = WL.small_case(37, 128, v, seed=50 + v)
    w = WL.to_device(wl, cuda_device)
    lp, lse = rlk.linear_logprob(w.hidden, w.W, w.targets, None, n_shards)
    ref_lp, ref_lse = O.selected_logprob(wl.hidden, wl.W, wl.targets)
    lp, lse = lp.cpu().numpy(), lse.cpu().numpy()
    assert np.abs(lp - ref_lp).max() <= 1e-4
    assert (np.abs(lse - ref_lse) / np.maximum(np.abs(ref_lse), 1e-30)).max() <= 2e-5
    if v == 1:
        assert np.all(lp == 0.0)
