"""Failure behaviour on the GPU, made without faulting anything.

Bad targets are detected by the kernels and reported through the device
status word (outputs NaN, other rows untouched); an unsupported device is
refused on the host before any launch (simulated through the documented
RLK_TEST_DEVICE_CC override); empty batches are no-ops.
"""
import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL
from oracle import linear_logprob as O

pytestmark = pytest.mark.gpu


def test_out_of_range_targets_flagged(rlk, cuda_device):
    w = WL.small_case(40, 128, 1000, seed=8)
    tg = w.targets.copy()
    tg[3], tg[17], tg[39] = -1, 1000, 2 ** 31 - 1
    dw = WL.to_device(w, cuda_device)
    dw.targets = torch.from_numpy(tg).to(cuda_device)
    status = rlk.new_status(cuda_device)
    lp, lse = rlk.linear_logprob(dw.hidden, dw.W, dw.targets, None, 2, status=status)
    with pytest.raises(rlk.RlkError) as e:
        rlk.raise_on_device_status(status)
    assert e.value.code == rlk.RLK_ERR_TARGET_RANGE
    lp, lse = lp.cpu().numpy(), lse.cpu().numpy()
    bad = np.zeros(40, bool)
    bad[[3, 17, 39]] = True
    assert np.all(np.isnan(lp[bad])) and np.all(np.isnan(lse[bad]))
    ref_lp, _ = O.selected_logprob(w.hidden, w.W, w.targets)
    assert np.abs(lp[~bad] - ref_lp[~bad]).max() <= 1e-4


def test_inactive_bad_targets_are_ignored(rlk, cuda_device):
    w = WL.small_case(16, 64, 300, seed=9)
    dw = WL.to_device(w, cuda_device)
    tg = dw.targets.clone()
    tg[::2] = -7
    act = torch.ones(16, dtype=torch.uint8, device=cuda_device)
    act[::2] = 0
    status = rlk.new_status(cuda_device)
    lp, lse = rlk.linear_logprob(dw.hidden, dw.W, tg, act, 1, status=status)
    rlk.raise_on_device_status(status)
    assert torch.all(lp[::2] == 0) and torch.all(torch.isfinite(lp[1::2]))


def test_merge_without_owner_flagged(rlk, cuda_device):
    w = WL.to_device(WL.small_case(8, 64, 1000, seed=10), cuda_device)
    vb, ve = rlk.shard_range(1000, 2, 0)
    p0 = rlk.linear_logprob_shard(w.hidden, w.W[vb:ve], w.targets, None, 1000, 2, 0)
    status = rlk.new_status(cuda_device)
    # shard 0 twice: targets in shard 1 have no owner, targets in shard 0 have two
    lp, lse = rlk.lse_merge([p0, p0], status=status)
    with pytest.raises(rlk.RlkError):
        rlk.raise_on_device_status(status)
    assert torch.all(torch.isnan(lp))


def test_unsupported_device_refused_before_launch(rlk, cuda_device, monkeypatch):
    w = WL.to_device(WL.small_case(4, 64, 100, seed=11), cuda_device)
    monkeypatch.setenv("RLK_TEST_DEVICE_CC", "100")
    with pytest.raises(rlk.RlkError) as e:
        rlk.linear_logprob(w.hidden, w.W, w.targets)
    assert e.value.code == 2
    monkeypatch.delenv("RLK_TEST_DEVICE_CC")
    lp, _ = rlk.linear_logprob(w.hidden, w.W, w.targets)
    assert torch.all(torch.isfinite(lp))


def test_empty_batch_is_noop(rlk, cuda_device):
    W = torch.zeros((100, 64), dtype=torch.bfloat16, device=cuda_device)
    h = torch.zeros((0, 64), dtype=torch.bfloat16, device=cuda_device)
    t = torch.zeros((0,), dtype=torch.int32, device=cuda_device)
    lp, lse = rlk.linear_logprob(h, W, t)
    assert lp.numel() == 0 and lse.numel() == 0


def test_unaligned_hidden_refused(rlk, cuda_device):
    buf = torch.zeros(8 * 64 + 1, dtype=torch.bfloat16, device=cuda_device)
    h = buf[1:].view(8, 64)  # 2-byte offset
    W = torch.zeros((100, 64), dtype=torch.bfloat16, device=cuda_device)
    t = torch.zeros(8, dtype=torch.int32, device=cuda_device)
    with pytest.raises(rlk.RlkError) as e:
        rlk.linear_logprob(h, W, t)
    assert e.value.code == 3


@pytest.mark.parametrize("T", [64, 120, 200, 300])
def test_pipeline_wait_gives_up_with_timeout_status(rlk, cuda_device, monkeypatch, T):
    """A pipeline stage that never fills: the bounded wait gives up, the kernel reports
    RLK_ERR_TIMEOUT and returns, and the context stays usable for the next call.  T = 64
    and T = 120 run the logits kernel's single ring with a shrunk hidden box (five and four
    stages), T = 200 its separate hidden and W rings (two token tiles), T = 300 its single
    ring of full boxes."""
    import time
    w = WL.small_case(T, 256, 1024, seed=12)
    dw = WL.to_device(w, cuda_device)
    monkeypatch.setenv("RLK_TEST_DROP_STAGE", "1")
    status = rlk.new_status(cuda_device)
    t0 = time.time()
    rlk.linear_logprob(dw.hidden, dw.W, dw.targets, None, 1, status=status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    monkeypatch.delenv("RLK_TEST_DROP_STAGE")
    with pytest.raises(rlk.RlkError) as e:
        rlk.raise_on_device_status(status)
    assert e.value.code == rlk.RLK_ERR_TIMEOUT
    assert elapsed < 30
    status2 = rlk.new_status(cuda_device)
    lp, _ = rlk.linear_logprob(dw.hidden, dw.W, dw.targets, None, 1, status=status2)
    torch.cuda.synchronize()
    rlk.raise_on_device_status(status2)
    ref_lp, _ = O.selected_logprob(w.hidden, w.W, w.targets)
    assert np.abs(lp.cpu().numpy() - ref_lp).max() <= 1e-4


def test_gemm_pipeline_wait_gives_up_with_timeout_status(rlk, cuda_device, monkeypatch):
    """The backward's grad_hidden GEMM with a pipeline stage that never fills: its bounded
    wait gives up, RLK_ERR_TIMEOUT is reported, the kernel returns, and the next backward
    on the same context gives the reference bits."""
    import time
    w = WL.small_case(256, 256, 3000, seed=13, w_std=0.05)
    dw = WL.to_device(w, cuda_device)
    _, lse = rlk.linear_logprob(dw.hidden, dw.W, dw.targets)
    g = torch.full((256,), 0.5, dtype=torch.float32, device=cuda_device)
    ref_dh, ref_dW = rlk.linear_logprob_backward(dw.hidden, dw.W, dw.targets, g, lse)
    torch.cuda.synchronize()
    monkeypatch.setenv("RLK_TEST_DROP_STAGE", "2")
    status = rlk.new_status(cuda_device)
    t0 = time.time()
    rlk.linear_logprob_backward(dw.hidden, dw.W, dw.targets, g, lse, status=status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    monkeypatch.delenv("RLK_TEST_DROP_STAGE")
    with pytest.raises(rlk.RlkError) as e:
        rlk.raise_on_device_status(status)
    assert e.value.code == rlk.RLK_ERR_TIMEOUT
    assert elapsed < 30
    status2 = rlk.new_status(cuda_device)
    dh, dW = rlk.linear_logprob_backward(dw.hidden, dw.W, dw.targets, g, lse, status=status2)
    torch.cuda.synchronize()
    rlk.raise_on_device_status(status2)
    assert torch.equal(dh.view(torch.int32), ref_dh.view(torch.int32))
    assert torch.equal(dW.view(torch.int32), ref_dW.view(torch.int32))
