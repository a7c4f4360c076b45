"""Bit-exact pins of the GPU path against the CPU contract emulator.

The inputs come from ``exact_case``: every logit is a multiple of 2^-9 far
below 2^24 ulps, so it is exact in fp32 whatever order any hardware sums
it in, and its value is known on the CPU (the fp64 oracle's logits, cast
exactly).  From those logits the emulator (plain C, written from the
contract text, sharing nothing with the CUDA sources) predicts every bit of
the tile tree, the shard records, the log-sum-exp and the logprob.  The
GPU must reproduce them exactly: mismatch_count = 0, max_abs_diff = 0.
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


def assert_bits_equal(got, want, what):
    g, w = u32(got), u32(want)
    mism = np.flatnonzero(g != w)
    assert mism.size == 0, "%s: %d mismatches, first at %d: %r vs %r" % (
        what, mism.size, mism[0], np.asarray(got).ravel()[mism[0]], np.asarray(want).ravel()[mism[0]])


def records_np(rec_int32):
    r = rec_int32.cpu().numpy()
    return r[..., 0].view(np.float32), r[..., 1].view(np.float32), r[..., 2].view(np.float32), \
        r[..., 3].view(np.uint32)


EXACT = [(64, 256, 1024, 0), (200, 128, 3000, 1), (1, 64, 1, 2), (130, 4096, 2047, 3),
         (257, 64, 129, 4), (96, 512, 40000, 5)]


@pytest.mark.parametrize("T,H,V,seed", EXACT)
def test_exact_logits_and_full_contract(rlk, cuda_device, T, H, V, seed):
    w = WL.exact_case(T, H, V, seed=seed, inactive_frac=0.1 if T > 4 else 0.0)
    dw = WL.to_device(w, cuda_device)
    L64 = O.logits(w.hidden, w.W)
    L32 = E.exact_fp32_logits(L64)
    # the GPU's fp32 logits are the exact values
    Lg = rlk.debug_logits(dw.hidden, dw.W).cpu().numpy()
    assert_bits_equal(Lg, L32, "logits")
    nt = (V + 127) // 128
    for n in (1, 2, 4, 8):
        if n > nt:
            continue
        emu = E.linear_logprob(L32, w.targets, w.active, n_shards=n)
        ws = rlk.new_workspace(T, V, n, cuda_device)
        status = rlk.new_status(cuda_device)
        lp, lse = rlk.linear_logprob(dw.hidden, dw.W, dw.targets, dw.active, n, workspace=ws,
                                     status=status)
        torch.cuda.synchronize()
        rlk.raise_on_device_status(status)
        assert_bits_equal(lp.cpu().numpy(), emu["logprob"], "logprob n=%d" % n)
        assert_bits_equal(lse.cpu().numpy(), emu["lse"], "lse n=%d" % n)
        m, s, tg, own = records_np(rlk.workspace_records(ws, T, V, n))
        assert_bits_equal(m, emu["rec_m"], "record m n=%d" % n)
        assert_bits_equal(s, emu["rec_s"], "record s n=%d" % n)
        assert_bits_equal(tg, emu["rec_tgt"], "record tgt n=%d" % n)
        assert np.array_equal(own, emu["rec_owned"])


@pytest.mark.parametrize("T,H,V,seed", EXACT[:4])
def test_exact_shard_api_records(rlk, cuda_device, T, H, V, seed):
    """One call per shard on that shard's W rows only, then the separate merge call."""
    w = WL.exact_case(T, H, V, seed=seed + 50)
    dw = WL.to_device(w, cuda_device)
    L32 = E.exact_fp32_logits(O.logits(w.hidden, w.W))
    nt = (V + 127) // 128
    for n in (1, 2, 4, 8):
        if n > nt:
            continue
        emu = E.linear_logprob(L32, w.targets, None, n_shards=n)
        parts = []
        for r in range(n):
            vb, ve = rlk.shard_range(V, n, r)
            parts.append(rlk.linear_logprob_shard(dw.hidden, dw.W[vb:ve], dw.targets, None, V, n, r))
        m = np.stack([records_np(p)[0] for p in parts])
        s = np.stack([records_np(p)[1] for p in parts])
        assert_bits_equal(m, emu["rec_m"], "shard m n=%d" % n)
        assert_bits_equal(s, emu["rec_s"], "shard s n=%d" % n)
        lp, lse = rlk.lse_merge(parts)
        assert_bits_equal(lp.cpu().numpy(), emu["logprob"], "merged logprob n=%d" % n)
        assert_bits_equal(lse.cpu().numpy(), emu["lse"], "merged lse n=%d" % n)


def test_exact_qwen_shape(rlk, cuda_device):
    """Exact grid at H=4096, V=151936: the full 1187-tile tree (depth 11), bit for bit."""
    dw = WL.exact_device_case(48, 4096, 151936, cuda_device, seed=77)
    hid_bits = WL.bf16_tensor_bits(dw.hidden)
    W_bits = WL.bf16_tensor_bits(dw.W)
    L32 = E.exact_fp32_logits(O.logits(hid_bits, W_bits))
    tg = dw.targets.cpu().numpy()
    Lg = rlk.debug_logits(dw.hidden, dw.W).cpu().numpy()
    assert_bits_equal(Lg, L32, "qwen logits")
    for n in (1, 4, 8):
        emu = E.linear_logprob(L32, tg, None, n_shards=n)
        ws = rlk.new_workspace(48, 151936, n, cuda_device)
        lp, lse = rlk.linear_logprob(dw.hidden, dw.W, dw.targets, None, n, workspace=ws)
        assert_bits_equal(lp.cpu().numpy(), emu["logprob"], "qwen logprob n=%d" % n)
        assert_bits_equal(lse.cpu().numpy(), emu["lse"], "qwen lse n=%d" % n)
        m, s, _, _ = records_np(rlk.workspace_records(ws, 48, 151936, n))
        assert_bits_equal(s, emu["rec_s"], "qwen records n=%d" % n)
