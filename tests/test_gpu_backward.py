"""Backward of sum_t g[t] * logprob[t] on the GPU.

* The bf16 logit gradient G the kernel forms equals the C emulator's, bit
  for bit, on exact-logit inputs (the forward's lse is itself bit-pinned).
* grad_hidden = G·W and grad_W = Gᵀ·h match fp64 products of the emulator's
  G within fp32 accumulation error, and the fp64 definition (oracle) within
  the bf16 rounding of G: |err| <= 2^-8 * (|G| @ |operand|) + 1e-6.
* A token's grad_hidden row is bit-identical whatever batch it is in;
  repeated runs give identical bits.
"""
import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL
from oracle import emulator as E
from oracle import linear_logprob as O

pytestmark = pytest.mark.gpu


def bf16_to_f64(bits):
    return WL.bf16_bits_to_f32(bits).astype(np.float64)


def run_backward(rlk, dw, g, n_shards=1):
    status = rlk.new_status(dw.hidden.device)
    lp, lse = rlk.linear_logprob(dw.hidden, dw.W, dw.targets, dw.active, n_shards, status=status)
    T, H = dw.hidden.shape
    V = dw.W.shape[0]
    ws = torch.empty(rlk.backward_workspace_size(T, H, V), dtype=torch.uint8, device=dw.hidden.device)
    dh, dW = rlk.linear_logprob_backward(dw.hidden, dw.W, dw.targets, g, lse, dw.active,
                                         workspace=ws, status=status)
    torch.cuda.synchronize()
    rlk.raise_on_device_status(status)
    return lse, dh, dW, ws


@pytest.mark.parametrize("T,H,V,seed", [(64, 256, 1024, 0), (37, 128, 1000, 1), (130, 192, 2047, 2),
                                        (5, 64, 300, 3), (300, 512, 5000, 4)])
def test_exact_inputs_grad_bits_and_products(rlk, cuda_device, T, H, V, seed):
    w = WL.exact_case(T, H, V, seed=seed + 30, inactive_frac=0.1 if T > 8 else 0.0)
    dw = WL.to_device(w, cuda_device)
    g_np = np.random.default_rng(seed).standard_normal(T).astype(np.float32)
    g = torch.from_numpy(g_np).to(cuda_device)
    lse, dh, dW, ws = run_backward(rlk, dw, g)
    L32 = E.exact_fp32_logits(O.logits(w.hidden, w.W))
    emu = E.linear_logprob(L32, w.targets, w.active, 1)
    assert np.array_equal(lse.cpu().numpy().view(np.uint32), emu["lse"].view(np.uint32))
    G_emu = E.grad_logits(L32, emu["lse"], w.targets, g_np, w.active)
    G_gpu = rlk.backward_grad_view(ws, T, V).contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    mism = np.flatnonzero(G_gpu != G_emu)
    assert mism.size == 0, "G: %d mismatching bf16 values" % mism.size
    # products of the (bit-pinned) G in fp64: only fp32 accumulation error remains
    Gd = bf16_to_f64(G_emu)
    h = bf16_to_f64(w.hidden)
    Wd = bf16_to_f64(w.W)
    ref_dh, ref_dW = Gd @ Wd, Gd.T @ h
    mag_dh, mag_dW = np.abs(Gd) @ np.abs(Wd), np.abs(Gd).T @ np.abs(h)
    assert np.all(np.abs(dh.cpu().numpy() - ref_dh) <= 2e-6 * mag_dh + 1e-7)
    assert np.all(np.abs(dW.cpu().numpy() - ref_dW) <= 2e-6 * mag_dW + 1e-7)
    # the fp64 definition, within the bf16 rounding of G
    d_dh, d_dW = O.backward(w.hidden, w.W, w.targets, g_np.astype(np.float64), w.active)
    assert np.all(np.abs(dh.cpu().numpy() - d_dh) <= 2.0 ** -8 * mag_dh + 1e-6)
    assert np.all(np.abs(dW.cpu().numpy() - d_dW) <= 2.0 ** -8 * mag_dW + 1e-6)
    if w.active is not None:
        assert np.all(dh.cpu().numpy()[w.active == 0] == 0)


@pytest.mark.parametrize("T,H,V", [(64, 256, 4000), (200, 1024, 3000)])
def test_realistic_inputs_vs_definition(rlk, cuda_device, T, H, V):
    w = WL.small_case(T, H, V, seed=T + H, w_std=0.05)
    dw = WL.to_device(w, cuda_device)
    g_np = np.random.default_rng(5).standard_normal(T).astype(np.float32)
    _, dh, dW, _ = run_backward(rlk, dw, torch.from_numpy(g_np).to(cuda_device))
    L = O.logits(w.hidden, w.W)
    G = O.grad_logits(L, w.targets, g_np.astype(np.float64))
    Wd, h = bf16_to_f64(w.W), bf16_to_f64(w.hidden)
    d_dh, d_dW = G @ Wd, G.T @ h
    assert np.all(np.abs(dh.cpu().numpy() - d_dh) <= 2.0 ** -8 * (np.abs(G) @ np.abs(Wd)) + 1e-6)
    assert np.all(np.abs(dW.cpu().numpy() - d_dW) <= 2.0 ** -8 * (np.abs(G).T @ np.abs(h)) + 1e-6)


def test_grad_hidden_rows_batch_invariant_and_runs_repeat(rlk, cuda_device):
    w = WL.to_device(WL.small_case(300, 256, 20000, seed=44, w_std=0.05), cuda_device)
    g = torch.randn(300, generator=torch.Generator(device=cuda_device).manual_seed(1),
                    device=cuda_device)
    _, dh, dW, _ = run_backward(rlk, w, g)
    _, dh2, dW2, _ = run_backward(rlk, w, g)
    assert torch.equal(dh.view(torch.int32), dh2.view(torch.int32))
    assert torch.equal(dW.view(torch.int32), dW2.view(torch.int32))
    for lo, hi in ((0, 1), (7, 71), (129, 300)):
        sub = WL.DeviceWorkload("sub", w.hidden[lo:hi].contiguous(), w.W,
                                w.targets[lo:hi].contiguous())
        _, dh_s, _, _ = run_backward(rlk, sub, g[lo:hi].contiguous())
        assert torch.equal(dh_s.view(torch.int32), dh[lo:hi].view(torch.int32)), (lo, hi)


def test_qwen_shape_backward_sampled(rlk, qwen):
    pk = qwen.packed
    idx = torch.arange(0, 4096, 16, device=qwen.device)  # 256 tokens
    h, tg = pk.hidden[idx].contiguous(), pk.targets[idx].contiguous()
    g_np = np.random.default_rng(9).standard_normal(256).astype(np.float32)
    dw = WL.DeviceWorkload("q", h, qwen.W, tg)
    _, dh, dW, _ = run_backward(rlk, dw, torch.from_numpy(g_np).to(qwen.device))
    h_bits = WL.bf16_tensor_bits(h)
    L = O.logits(h_bits, qwen.W_bits)
    G = O.grad_logits(L, tg.cpu().numpy(), g_np.astype(np.float64))
    Wd = O.decode_bf16(qwen.W_bits)
    hd = O.decode_bf16(h_bits)
    rows = np.arange(0, 256, 37)
    ref_dh = G[rows] @ Wd
    mag = np.abs(G[rows]) @ np.abs(Wd)
    assert np.all(np.abs(dh.cpu().numpy()[rows] - ref_dh) <= 2.0 ** -8 * mag + 1e-6)
    vocab = np.unique(np.concatenate([tg.cpu().numpy()[:8], np.arange(0, 151936, 9973)]))
    ref_dW = G[:, vocab].T @ hd
    magW = np.abs(G[:, vocab]).T @ np.abs(hd)
    assert np.all(np.abs(dW.cpu().numpy()[vocab] - ref_dW) <= 2.0 ** -8 * magW + 1e-6)


def test_grad_w_feature_bands(rlk, cuda_device):
    """T = 8192 with H = 2560: grad_W takes its 10 feature tiles in bands (8, then a ragged
    2), grad_hidden runs feature tiles fastest over 64 token tiles.  Both against the fp64
    definition within the bf16 rounding of G, and grad_hidden rows against a 300-row
    batch of the same tokens bit for bit."""
    T, H, V = 8192, 2560, 1000
    w = WL.small_case(T, H, V, seed=808, w_std=0.03)
    dw = WL.to_device(w, cuda_device)
    g_np = np.random.default_rng(8).standard_normal(T).astype(np.float32)
    _, dh, dW, _ = run_backward(rlk, dw, torch.from_numpy(g_np).to(cuda_device))
    L = O.logits(w.hidden, w.W)
    G = O.grad_logits(L, w.targets, g_np.astype(np.float64))
    Wd, h = bf16_to_f64(w.W), bf16_to_f64(w.hidden)
    assert np.all(np.abs(dW.cpu().numpy() - G.T @ h) <= 2.0 ** -8 * (np.abs(G).T @ np.abs(h)) + 1e-6)
    rows = np.arange(0, T, 97)
    assert np.all(np.abs(dh.cpu().numpy()[rows] - G[rows] @ Wd)
                  <= 2.0 ** -8 * (np.abs(G[rows]) @ np.abs(Wd)) + 1e-6)
    lo, hi = 4000, 4300
    sub = WL.DeviceWorkload("sub", dw.hidden[lo:hi].contiguous(), dw.W,
                            dw.targets[lo:hi].contiguous())
    _, dh_s, _, _ = run_backward(rlk, sub, torch.from_numpy(g_np[lo:hi]).to(cuda_device))
    assert torch.equal(dh_s.view(torch.int32), dh[lo:hi].view(torch.int32))
