"""Strict RMSNorm on the GPU: every output bit against the C emulator, the
fp64 definition within one bf16 rounding, and rows independent of the batch."""
import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL
from oracle import emulator as E
from oracle import rmsnorm as R

pytestmark = pytest.mark.gpu


def bf16_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


CASES = [(7, 64, False), (64, 4096, True), (33, 2560, True), (5, 8192, True), (300, 128, False),
         (1, 192, True), (129, 4096, False)]


@pytest.mark.parametrize("T,H,res", CASES)
def test_rmsnorm_bits_and_definition(rlk, cuda_device, T, H, res):
    rng = np.random.default_rng(T * H)
    x = WL.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32) * 4)
    r = WL.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)) if res else None
    g = WL.f32_to_bf16_bits((1 + 0.2 * rng.standard_normal(H)).astype(np.float32))
    eps = 1e-6
    out, r_out = rlk.rmsnorm(bf16_dev(x, cuda_device), bf16_dev(g, cuda_device), eps,
                             None if r is None else bf16_dev(r, cuda_device), want_residual_out=res)
    y_emu, xr_emu = E.rmsnorm(x, g, eps, r)
    assert np.array_equal(bits_of(out), y_emu)
    if res:
        assert np.array_equal(bits_of(r_out), xr_emu)
    y_ref, _ = R.rmsnorm(x, g, eps, r)
    y = WL.bf16_bits_to_f32(bits_of(out)).astype(np.float64)
    assert np.all(np.abs(y - y_ref) <= 2.0 ** -7 * np.abs(y_ref) + 1e-30)


def test_rmsnorm_rows_independent_of_batch(rlk, cuda_device):
    rng = np.random.default_rng(5)
    T, H = 300, 4096
    x = bf16_dev(WL.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)), cuda_device)
    g = bf16_dev(WL.f32_to_bf16_bits(np.ones(H, np.float32)), cuda_device)
    full, _ = rlk.rmsnorm(x, g)
    for lo, hi in ((0, 1), (5, 77), (128, 300)):
        part, _ = rlk.rmsnorm(x[lo:hi].contiguous(), g)
        assert torch.equal(part.view(torch.int16), full[lo:hi].view(torch.int16))


def test_rmsnorm_feeds_the_head(rlk, cuda_device):
    """Final norm then selected logprob: the normalised rows go straight into the head."""
    rng = np.random.default_rng(6)
    T, H, V = 64, 512, 3000
    x = bf16_dev(WL.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32) * 10), cuda_device)
    g = bf16_dev(WL.f32_to_bf16_bits(np.ones(H, np.float32)), cuda_device)
    hidden, _ = rlk.rmsnorm(x, g)
    w = WL.small_case(T, H, V, seed=6, w_std=0.05)
    dw = WL.to_device(w, cuda_device)
    lp, lse = rlk.linear_logprob(hidden, dw.W, dw.targets)
    from oracle import linear_logprob as O
    ref_lp, _ = O.selected_logprob(bits_of(hidden), w.W, w.targets)
    assert np.abs(lp.cpu().numpy() - ref_lp).max() <= 1e-4


@pytest.mark.parametrize("H", [4096, 8192, 320])
def test_rmsnorm_in_place(rlk, cuda_device, H):
    """out = x and residual_out = residual (the residual stream updated in place) give the
    out-of-place bits."""
    rng = np.random.default_rng(H + 11)
    T = 37
    x = bf16_dev(WL.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32) * 3), cuda_device)
    r = bf16_dev(WL.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)), cuda_device)
    g = bf16_dev(WL.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(H)).astype(np.float32)),
                 cuda_device)
    ref_out, ref_res = rlk.rmsnorm(x, g, 1e-6, r, want_residual_out=True)
    xi, ri = x.clone(), r.clone()
    out, r_out = rlk.rmsnorm(xi, g, 1e-6, ri, want_residual_out=True, out=xi, residual_out=ri)
    torch.cuda.synchronize()
    assert out.data_ptr() == xi.data_ptr() and r_out.data_ptr() == ri.data_ptr()
    assert torch.equal(xi.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(ri.view(torch.int16), ref_res.view(torch.int16))
