"""Training pair that saves the forward's fp32 logits for the backward.

* rlk_linear_logprob_save_logits returns rlk_linear_logprob's logprob and
  lse bit for bit, and stores every row's fp32 logits equal, bit for bit, to
  the logits rlk_debug_logits dumps (the exact accumulators).
* rlk_linear_logprob_backward_from_logits, fed those logits, returns
  rlk_linear_logprob_backward's grad_hidden and grad_W bit for bit (same G,
  same GEMMs); with exact-grid inputs its G also equals the C emulator's.
* Bad strides and alignment are refused before any launch; an active row
  with an out-of-range target sets RLK_ERR_TARGET_RANGE as the recomputing
  backward does.
"""
import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL
from oracle import emulator as E
from oracle import linear_logprob as O

pytestmark = pytest.mark.gpu


def same(a, b, what):
    ai, bi = a.contiguous().view(torch.int32), b.contiguous().view(torch.int32)
    n = int((ai != bi).sum().item())
    assert n == 0, "%s: %d differing values" % (what, n)


def both_backwards(rlk, dw, g, ld=None):
    T, H = dw.hidden.shape
    V = dw.W.shape[0]
    dev = dw.hidden.device
    status = rlk.new_status(dev)
    lp, lse = rlk.linear_logprob(dw.hidden, dw.W, dw.targets, dw.active, 1, status=status)
    logits = None if ld is None else torch.full((T, ld), float("nan"), dtype=torch.float32,
                                                device=dev)
    lp_s, lse_s, logits = rlk.linear_logprob_save_logits(dw.hidden, dw.W, dw.targets, dw.active,
                                                         1, logits=logits, status=status)
    dh, dW = rlk.linear_logprob_backward(dw.hidden, dw.W, dw.targets, g, lse, dw.active,
                                         status=status)
    ws = torch.empty(rlk.backward_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
    dh_s, dW_s = rlk.linear_logprob_backward_from_logits(logits, dw.hidden, dw.W, dw.targets, g,
                                                         lse_s, dw.active, workspace=ws,
                                                         status=status)
    torch.cuda.synchronize()
    rlk.raise_on_device_status(status)
    return (lp, lse, dh, dW), (lp_s, lse_s, dh_s, dW_s), logits, ws


@pytest.mark.parametrize("T,H,V,seed,pad", [(64, 256, 1024, 0, 0), (37, 128, 1001, 1, 3),
                                            (130, 192, 2047, 2, 1), (300, 512, 5000, 4, 0),
                                            (1, 64, 300, 5, 4)])
def test_saved_logits_forward_and_backward_bits(rlk, cuda_device, T, H, V, seed, pad):
    w = WL.small_case(T, H, V, seed=seed + 70, w_std=0.05, inactive_frac=0.1 if T > 8 else 0.0)
    dw = WL.to_device(w, cuda_device)
    g = torch.from_numpy(np.random.default_rng(seed).standard_normal(T).astype(np.float32)
                         ).to(cuda_device)
    ld = (V + 3) // 4 * 4 + 4 * pad
    (lp, lse, dh, dW), (lp_s, lse_s, dh_s, dW_s), logits, _ = both_backwards(rlk, dw, g, ld)
    same(lp_s, lp, "logprob")
    same(lse_s, lse, "lse")
    same(logits[:, :V], rlk.debug_logits(dw.hidden, dw.W), "saved logits")
    assert torch.isnan(logits[:, V:]).all(), "columns past V were written"
    same(dh_s, dh, "grad_hidden")
    same(dW_s, dW, "grad_W")


def test_saved_logits_exact_inputs_grad_matches_emulator(rlk, cuda_device):
    T, H, V = 130, 192, 2047
    w = WL.exact_case(T, H, V, seed=77, inactive_frac=0.1)
    dw = WL.to_device(w, cuda_device)
    g_np = np.random.default_rng(3).standard_normal(T).astype(np.float32)
    g = torch.from_numpy(g_np).to(cuda_device)
    _, (_, lse_s, _, _), logits, ws = both_backwards(rlk, dw, g)
    L32 = E.exact_fp32_logits(O.logits(w.hidden, w.W))
    emu = E.linear_logprob(L32, w.targets, w.active, 1)
    assert np.array_equal(lse_s.cpu().numpy().view(np.uint32), emu["lse"].view(np.uint32))
    assert np.array_equal(logits[:, :V].cpu().numpy().view(np.uint32), L32.view(np.uint32))
    G_emu = E.grad_logits(L32, emu["lse"], w.targets, g_np, w.active)
    G_gpu = rlk.backward_grad_view(ws, T, V).contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(G_gpu, G_emu)


def test_saved_logits_qwen_shape(rlk, qwen):
    """The packed Qwen3-8B-shaped batch (T = 4096, V = 151936): forward outputs, the
    backward's two gradients bit for bit against the recomputing pair."""
    pk = qwen.packed
    dw = WL.DeviceWorkload("q", pk.hidden, qwen.W, pk.targets)
    T = pk.hidden.shape[0]
    g = torch.from_numpy(np.random.default_rng(11).standard_normal(T).astype(np.float32)
                         ).to(qwen.device)
    (lp, lse, dh, dW), (lp_s, lse_s, dh_s, dW_s), logits, _ = both_backwards(rlk, dw, g)
    same(lp_s, lp, "logprob")
    same(lse_s, lse, "lse")
    same(dh_s, dh, "grad_hidden")
    same(dW_s, dW, "grad_W")
    rows = torch.arange(0, T, 512, device=qwen.device)
    same(logits[rows, :151936], rlk.debug_logits(pk.hidden[rows].contiguous(), qwen.W),
         "saved logits (sampled rows)")
    del logits, dh, dW, dh_s, dW_s
    torch.cuda.empty_cache()


def test_saved_logits_argument_checks_and_target_status(rlk, cuda_device):
    T, H, V = 16, 64, 1000
    w = WL.small_case(T, H, V, seed=5)
    dw = WL.to_device(w, cuda_device)
    with pytest.raises(rlk.RlkError) as e:   # stride not a multiple of 4
        rlk.linear_logprob_save_logits(dw.hidden, dw.W, dw.targets,
                                       logits=torch.empty((T, 1002), dtype=torch.float32,
                                                          device=cuda_device))
    assert e.value.code == rlk.RLK_ERR_ALIGNMENT
    with pytest.raises(rlk.RlkError) as e:   # stride below V
        rlk.linear_logprob_save_logits(dw.hidden, dw.W, dw.targets,
                                       logits=torch.empty((T, 996), dtype=torch.float32,
                                                          device=cuda_device))
    assert e.value.code == rlk.RLK_ERR_INVALID_ARG
    _, lse, logits = rlk.linear_logprob_save_logits(dw.hidden, dw.W, dw.targets)
    bad = dw.targets.clone()
    bad[3] = V + 5
    g = torch.ones(T, dtype=torch.float32, device=cuda_device)
    st_a, st_b = rlk.new_status(cuda_device), rlk.new_status(cuda_device)
    dh_a, dW_a = rlk.linear_logprob_backward(dw.hidden, dw.W, bad, g, lse, status=st_a)
    dh_b, dW_b = rlk.linear_logprob_backward_from_logits(logits, dw.hidden, dw.W, bad, g, lse,
                                                         status=st_b)
    torch.cuda.synchronize()
    for st in (st_a, st_b):
        with pytest.raises(rlk.RlkError) as e:
            rlk.raise_on_device_status(st)
        assert e.value.code == rlk.RLK_ERR_TARGET_RANGE
    same(dh_b, dh_a, "grad_hidden, bad target")
    same(dW_b, dW_a, "grad_W, bad target")
