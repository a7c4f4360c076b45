"""GPU results against the fp64 oracle, element by element.

Tolerances: |logprob - oracle| <= 1e-4 and |lse - oracle| <= 2e-5 |lse|
(the bar the method's own target states for fp32 results against an fp64
reference).  Sizes run from one token and one vocabulary entry to the full
Qwen3-8B head, with ragged M tiles (T not a multiple of 128), ragged
vocabulary tiles (V not a multiple of 128 or 256) and masked rows.
"""
import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL
from oracle import linear_logprob as O

pytestmark = pytest.mark.gpu

TOL_LP = 1e-4
TOL_LSE_REL = 2e-5


def run(rlk, dw, n_shards):
    status = rlk.new_status(dw.hidden.device)
    lp, lse = rlk.linear_logprob(dw.hidden, dw.W, dw.targets, dw.active, n_shards, status=status)
    torch.cuda.synchronize()
    rlk.raise_on_device_status(status)
    return lp.cpu().numpy(), lse.cpu().numpy()


def assert_close(lp, lse, ref_lp, ref_lse, what=""):
    d_lp = np.abs(lp.astype(np.float64) - ref_lp)
    d_lse = np.abs(lse.astype(np.float64) - ref_lse) / np.maximum(np.abs(ref_lse), 1.0)
    assert np.all(np.isfinite(lp)) and np.all(np.isfinite(lse)), what
    assert d_lp.max() <= TOL_LP, (what, d_lp.max(), int(d_lp.argmax()))
    assert d_lse.max() <= TOL_LSE_REL, (what, d_lse.max(), int(d_lse.argmax()))


@pytest.mark.parametrize("n_shards", [1, 2, 4, 8])
def test_tiny_all_rows(rlk, cuda_device, n_shards):
    w = WL.tiny()
    lp, lse = run(rlk, WL.to_device(w, cuda_device), n_shards)
    ref_lp, ref_lse = O.selected_logprob(w.hidden, w.W, w.targets)
    assert_close(lp, lse, ref_lp, ref_lse, "tiny")


RAGGED = [
    (1, 64, 1, 1), (1, 64, 2, 1), (3, 64, 129, 1), (128, 128, 256, 2), (129, 192, 257, 2),
    (255, 256, 1000, 4), (257, 64, 1024, 8), (300, 128, 5000, 8), (37, 512, 2047, 4),
    (513, 64, 384, 2), (64, 1024, 12345, 4), (112, 256, 3000, 4), (120, 512, 9000, 2),
    # wide hidden sizes: 80, 128 and 1024 K blocks per logit
    (130, 5120, 700, 2), (129, 8192, 1500, 4), (3, 65536, 300, 1),
]


@pytest.mark.parametrize("T,H,V,n_shards", RAGGED)
def test_ragged_shapes(rlk, cuda_device, T, H, V, n_shards):
    w = WL.small_case(T, H, V, seed=T * 7 + V, n_shards=n_shards, inactive_frac=0.2 if T > 8 else 0)
    lp, lse = run(rlk, WL.to_device(w, cuda_device), n_shards)
    ref_lp, ref_lse = O.selected_logprob(w.hidden, w.W, w.targets, w.active)
    assert_close(lp, lse, ref_lp, ref_lse, (T, H, V))
    if w.active is not None:
        inact = w.active == 0
        assert np.all(lp[inact] == 0) and np.all(lse[inact] == 0)


def test_wide_logit_range(rlk, cuda_device):
    """Logits spread over ~+-60, so exps underflow inside tiles and merges."""
    w = WL.small_case(96, 256, 3000, seed=5, w_std=0.6)
    lp, lse = run(rlk, WL.to_device(w, cuda_device), 2)
    ref_lp, ref_lse = O.selected_logprob(w.hidden, w.W, w.targets)
    assert np.abs(ref_lp).max() > 50
    assert_close(lp, lse, ref_lp, ref_lse, "wide")


def test_debug_logits_match_oracle(rlk, cuda_device):
    w = WL.small_case(130, 4096, 700, seed=3, w_std=0.02)
    dw = WL.to_device(w, cuda_device)
    L = rlk.debug_logits(dw.hidden, dw.W).cpu().numpy().astype(np.float64)
    ref = O.logits(w.hidden, w.W)
    assert np.abs(L - ref).max() <= 1e-4 * (1 + np.abs(ref).max())


def test_qwen_packed_sampled_rows(rlk, qwen):
    """Packed 4096-token batch, 4 shards, the configuration the benchmark times."""
    pk = qwen.packed
    lp, lse = run(rlk, pk, 4)
    rows = np.unique(np.concatenate([[0, 127, 128, 4095], WL.permutation(4096, 99)[:44]]))
    hid_bits = WL.bf16_tensor_bits(pk.hidden[torch.from_numpy(rows).to(pk.hidden.device)])
    tg = pk.targets.cpu().numpy()[rows]
    ref_lp, ref_lse = O.selected_logprob(hid_bits, qwen.W_bits, tg)
    assert_close(lp[rows], lse[rows], ref_lp, ref_lse, "qwen packed")
    # the target recipe puts most targets near the top of the distribution
    assert np.median(ref_lp) > -9.0
    assert 10.0 < np.median(ref_lse) < 16.0


@pytest.mark.parametrize("n", [1, 64, 256])
def test_qwen_decode_rows_against_oracle(rlk, qwen, n):
    """Decode batches as the rollout side issues them (T = 1 and T = 64 rows of the packed
    batch: one token tile with a shrunk hidden box and a deeper ring; T = 256: two token
    tiles sharing each W tile), every row against the oracle directly -- not only through
    their bitwise equality with the packed rows."""
    pk = qwen.packed
    rows = WL.decode_rows(n)
    idx = torch.from_numpy(rows).to(qwen.device)
    dw = WL.DeviceWorkload("decode%d" % n, pk.hidden[idx].contiguous(), qwen.W,
                           pk.targets[idx].contiguous())
    lp, lse = run(rlk, dw, 4)
    ref_lp, ref_lse = O.selected_logprob(WL.bf16_tensor_bits(dw.hidden), qwen.W_bits,
                                         dw.targets.cpu().numpy())
    assert_close(lp, lse, ref_lp, ref_lse, "qwen decode T=%d" % n)


@pytest.mark.slow
def test_qwen_grpo_long_sampled(rlk, qwen):
    """Long-response GRPO batch (~221k rows, prompt rows masked) in 8192-row calls; a seeded
    2048-token subset of the active rows against the oracle."""
    g = WL.grpo_long(qwen.W, qwen.device)
    act = g.active.cpu().numpy()
    rng = np.random.default_rng(1235)
    n = g.hidden.shape[0]
    assert 200_000 < act.sum() < 260_000
    lp_all = np.empty(n, np.float32)
    lse_all = np.empty(n, np.float32)
    ws = rlk.new_workspace(8192, qwen.W.shape[0], 4, qwen.device)
    for r0, r1 in g.meta["chunks"]:
        lp, lse = rlk.linear_logprob(g.hidden[r0:r1], qwen.W, g.targets[r0:r1], g.active[r0:r1], 4,
                                     workspace=ws)
        lp_all[r0:r1] = lp.cpu().numpy()
        lse_all[r0:r1] = lse.cpu().numpy()
    assert np.all(lp_all[act == 0] == 0) and np.all(lse_all[act == 0] == 0)
    rows = np.sort(rng.choice(np.flatnonzero(act), 2048, replace=False))
    hid_bits = WL.bf16_tensor_bits(g.hidden[torch.from_numpy(rows).to(qwen.device)])
    ref_lp, ref_lse = O.selected_logprob(hid_bits, qwen.W_bits, g.targets.cpu().numpy()[rows])
    assert_close(lp_all[rows], lse_all[rows], ref_lp, ref_lse, "grpo")


def test_qwen_logit_accuracy(rlk, qwen):
    """fp32 tensor-core logits vs fp64 at K=4096: error far below the logprob tolerance."""
    pk = qwen.packed
    rows = np.arange(0, 4096, 257)
    hid = pk.hidden[torch.from_numpy(rows).to(qwen.device)].contiguous()
    L = rlk.debug_logits(hid, qwen.W).cpu().numpy().astype(np.float64)
    ref = O.logits(WL.bf16_tensor_bits(hid), qwen.W_bits)
    err = L - ref
    stats = "max|err|=%.3g mean err=%.3g max|logit|=%.3g" % (np.abs(err).max(), err.mean(),
                                                            np.abs(ref).max())
    print("qwen logits:", stats)
    assert np.abs(err).max() <= 2e-5 * (1 + np.abs(ref).max()), stats


def test_token_tile_bands_ragged(rlk, cuda_device):
    """T = 8322: 66 token tiles (the last one 2 rows), i.e. three bands of 32 tiles for the
    logits kernel's work order, the last band holding two tiles.  Every row against the
    oracle, and bit for bit against the same rows computed in batches of 4096 and of 130
    rows (one band, different band boundaries)."""
    T, H, V = 8322, 128, 3000
    w = WL.small_case(T, H, V, seed=77, n_shards=2)
    dw = WL.to_device(w, cuda_device)
    lp, lse = run(rlk, dw, 2)
    ref_lp, ref_lse = O.selected_logprob(w.hidden, w.W, w.targets)
    assert_close(lp, lse, ref_lp, ref_lse, "T=8322")
    for bsz in (4096, 130):
        for b0 in range(0, T, bsz):
            b1 = min(T, b0 + bsz)
            p_lp, p_lse = rlk.linear_logprob(dw.hidden[b0:b1].contiguous(), dw.W,
                                             dw.targets[b0:b1].contiguous(), None, 2)
            assert np.array_equal(p_lp.cpu().numpy().view(np.int32), lp[b0:b1].view(np.int32))
            assert np.array_equal(p_lse.cpu().numpy().view(np.int32), lse[b0:b1].view(np.int32))
