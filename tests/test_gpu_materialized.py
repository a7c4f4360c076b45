"""Selected logprob and log_softmax on materialised logits (fp32 / bf16 [T, V]).

The logits here are drawn on the CPU, so the C emulator can predict every
output bit from the very values the GPU reads: the tile pairs, the tree,
the shard records, lse, logprob and each log_softmax element must match it
exactly; against the fp64 oracle they must meet the usual tolerance.  Fed
the fused path's own logits, this path must return the fused path's bits.
"""
import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL
from oracle import emulator as E
from oracle import linear_logprob as O

pytestmark = pytest.mark.gpu


def u32(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def same_bits(a, b, what):
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    mism = np.flatnonzero(u32(a).ravel() != u32(b).ravel())
    assert mism.size == 0, "%s: %d mismatches (first %d: %r vs %r)" % (
        what, mism.size, mism[0], a.ravel()[mism[0]], b.ravel()[mism[0]])


def cpu_logits(T, V, seed, scale=2.0):
    rng = np.random.default_rng(seed)
    L = (rng.standard_normal((T, V)) * scale).astype(np.float32)
    tg = rng.integers(0, V, T).astype(np.int32)
    return L, tg


SHAPES = [(64, 1024, 0), (37, 1000, 1), (3, 151936, 2), (300, 5000, 3), (1, 1, 4), (9, 129, 5),
          (130, 262144, 6)]


@pytest.mark.parametrize("T,V,seed", SHAPES)
def test_fp32_logits_bits_and_parity(rlk, cuda_device, T, V, seed):
    L, tg = cpu_logits(T, V, seed)
    act = (np.random.default_rng(seed + 9).random(T) > 0.15).astype(np.uint8) if T > 4 else None
    dL = torch.from_numpy(L).to(cuda_device)
    dtg = torch.from_numpy(tg).to(cuda_device)
    dact = None if act is None else torch.from_numpy(act).to(cuda_device)
    nt = (V + 127) // 128
    for n in (1, 2, 4, 8):
        if n > nt:
            continue
        emu = E.linear_logprob(L, tg, act, n_shards=n)
        ws = rlk.new_workspace(T, V, n, cuda_device)
        lp, lse = rlk.logits_logprob(dL, dtg, dact, n, workspace=ws)
        same_bits(lp.cpu().numpy(), emu["logprob"], "logprob n=%d" % n)
        same_bits(lse.cpu().numpy(), emu["lse"], "lse n=%d" % n)
        rec = rlk.workspace_records(ws, T, V, n).cpu().numpy()
        same_bits(rec[..., 0].view(np.float32), emu["rec_m"], "record m")
        same_bits(rec[..., 1].view(np.float32), emu["rec_s"], "record s")
        same_bits(rec[..., 2].view(np.float32), emu["rec_tgt"], "record tgt")
    ref_lp, ref_lse = O.lse_and_logprob_from_logits(L.astype(np.float64), tg, act)
    assert np.abs(lp.cpu().numpy() - ref_lp).max() <= 1e-4
    assert (np.abs(lse.cpu().numpy() - ref_lse) / np.maximum(np.abs(ref_lse), 1)).max() <= 2e-5


@pytest.mark.parametrize("T,V,seed", [(64, 1024, 10), (17, 151936, 11), (200, 3000, 12)])
def test_bf16_logits_and_log_softmax(rlk, cuda_device, T, V, seed):
    L, tg = cpu_logits(T, V, seed, scale=3.0)
    Lb = WL.f32_to_bf16_bits(L)
    Lw = WL.bf16_bits_to_f32(Lb)  # the values the GPU reads, widened exactly
    dLb = torch.from_numpy(Lb.view(np.int16)).view(torch.bfloat16).to(cuda_device)
    dtg = torch.from_numpy(tg).to(cuda_device)
    emu = E.linear_logprob(Lw, tg, None, n_shards=1)
    lp, lse = rlk.logits_logprob(dLb, dtg)
    same_bits(lp.cpu().numpy(), emu["logprob"], "bf16 logprob")
    same_bits(lse.cpu().numpy(), emu["lse"], "bf16 lse")
    out, lse2 = rlk.log_softmax(dLb)
    e_out, e_lse = E.log_softmax(Lw)
    same_bits(lse2.cpu().numpy(), e_lse, "log_softmax lse")
    same_bits(out.cpu().numpy(), e_out, "log_softmax values")
    ref = O.log_softmax_from_logits(Lw.astype(np.float64))
    assert np.abs(out.cpu().numpy() - ref).max() <= 1e-4 * (1 + np.abs(ref).max() / 100)


def test_bf16_logits_wide_range_underflow(rlk, cuda_device):
    """bf16 tiles whose values reach below max - 86, where the contract's exp gives +0:
    such tiles take the exps with the underflow select, tiles within 86 of their max
    take them without it, and the bits must not depend on which.  Planted rows put a
    tile's smallest value at exactly max - 86 (no select needed), one bf16 step below
    it (select needed), at -inf, and at both signs of zero."""
    T, V = 40, 3000
    L, tg = cpu_logits(T, V, 31, scale=40.0)
    L[T // 2:] *= np.float32(0.075)  # the second half's tiles stay within 86 of their max
    L[0, :128] = 0.0
    L[0, 5] = -86.0
    L[1, :128] = 1.0
    L[1, 7] = -85.5            # RN(-85.5 - 1) = -86.5: below -86 by one bf16 step of 86
    L[2, 128:256] = -3.0
    L[2, 200] = -np.inf
    L[3, :128] = np.where(np.arange(128) % 2 == 0, 0.0, -0.0)
    L[4, 256:384] = 2.0
    L[4, 300] = -84.0          # RN(-84 - 2) = -86 exactly
    Lb = WL.f32_to_bf16_bits(L)
    Lw = WL.bf16_bits_to_f32(Lb)
    assert Lw[1, 7] == np.float32(-85.5) and Lw[0, 5] == np.float32(-86.0)
    dLb = torch.from_numpy(Lb.view(np.int16)).view(torch.bfloat16).to(cuda_device)
    dtg = torch.from_numpy(tg).to(cuda_device)
    for n in (1, 4):
        emu = E.linear_logprob(Lw, tg, None, n_shards=n)
        ws = rlk.new_workspace(T, V, n, cuda_device)
        lp, lse = rlk.logits_logprob(dLb, dtg, None, n, workspace=ws)
        same_bits(lp.cpu().numpy(), emu["logprob"], "wide bf16 logprob n=%d" % n)
        same_bits(lse.cpu().numpy(), emu["lse"], "wide bf16 lse n=%d" % n)
        rec = rlk.workspace_records(ws, T, V, n).cpu().numpy()
        same_bits(rec[..., 0].view(np.float32), emu["rec_m"], "wide record m")
        same_bits(rec[..., 1].view(np.float32), emu["rec_s"], "wide record s")
    out, lse2 = rlk.log_softmax(dLb)
    e_out, e_lse = E.log_softmax(Lw)
    same_bits(lse2.cpu().numpy(), e_lse, "wide log_softmax lse")
    same_bits(out.cpu().numpy(), e_out, "wide log_softmax values")
    ref_lp, ref_lse = O.lse_and_logprob_from_logits(Lw.astype(np.float64), tg, None)
    assert np.abs(lp.cpu().numpy() - ref_lp).max() <= 1e-4 * (1 + np.abs(ref_lp).max() / 100)


def test_fp32_log_softmax_masked_and_strided(rlk, cuda_device):
    T, V = 50, 1000
    L, _ = cpu_logits(T, V, 21)
    act = (np.arange(T) % 5 != 0).astype(np.uint8)
    padded = np.zeros((T, 1024), np.float32)
    padded[:, :V] = L
    dpad = torch.from_numpy(padded).to(cuda_device)
    out, lse = rlk.log_softmax(dpad[:, :V], torch.from_numpy(act).to(cuda_device))
    e_out, e_lse = E.log_softmax(L, act)
    same_bits(out.cpu().numpy(), e_out, "strided log_softmax")
    same_bits(lse.cpu().numpy(), e_lse, "strided lse")
    assert np.all(out.cpu().numpy()[act == 0] == 0)


def test_materialised_equals_fused(rlk, cuda_device):
    """The fused path's own logits through this path give the fused path's bits."""
    w = WL.to_device(WL.small_case(300, 512, 20000, seed=22, w_std=0.05, inactive_frac=0.1),
                     cuda_device)
    fused_lp, fused_lse = rlk.linear_logprob(w.hidden, w.W, w.targets, w.active, 4)
    L = rlk.debug_logits(w.hidden, w.W)
    lp, lse = rlk.logits_logprob(L, w.targets, w.active, 4)
    assert torch.equal(lp.view(torch.int32), fused_lp.view(torch.int32))
    assert torch.equal(lse.view(torch.int32), fused_lse.view(torch.int32))
    out, lse2 = rlk.log_softmax(L, w.active)
    assert torch.equal(lse2.view(torch.int32), fused_lse.view(torch.int32))


def test_materialised_equals_fused_qwen(rlk, qwen):
    pk = qwen.packed
    idx = torch.arange(0, 4096, 97, device=qwen.device)
    h, tg = pk.hidden[idx].contiguous(), pk.targets[idx].contiguous()
    fused_lp, fused_lse = rlk.linear_logprob(h, qwen.W, tg, None, 4)
    L = rlk.debug_logits(h, qwen.W)
    lp, lse = rlk.logits_logprob(L, tg, None, 4)
    assert torch.equal(lp.view(torch.int32), fused_lp.view(torch.int32))
    assert torch.equal(lse.view(torch.int32), fused_lse.view(torch.int32))
