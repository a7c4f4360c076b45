"""Layout invariance on the GPU, compared bit for bit.

A token's logprob and lse must not depend on the batch it is computed in
(size, position, order), on the shard split of the vocabulary, on a decode
(few rows) versus a packed launch, or on the run.  Every comparison is on
the uint32 views: mismatch_count = 0 and max_abs_diff = 0.
"""
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL

pytestmark = pytest.mark.gpu


def bits(t):
    return t.contiguous().view(torch.int32)


def assert_same(a, b, what):
    ia, ib = bits(a), bits(b)
    mism = int((ia != ib).sum().item())
    maxdiff = float((a.double() - b.double()).abs().max().item()) if a.numel() else 0.0
    assert mism == 0 and maxdiff == 0.0, "%s: mismatch_count=%d max_abs_diff=%g" % (what, mism, maxdiff)


def in_batches(rlk, hidden, W, targets, active, bsz, n_shards=1, order=None):
    T = hidden.shape[0]
    order = torch.arange(T, device=hidden.device) if order is None else order
    lp = torch.empty(T, dtype=torch.float32, device=hidden.device)
    lse = torch.empty_like(lp)
    ws = rlk.new_workspace(min(bsz, T), W.shape[0], n_shards, hidden.device)
    for b0 in range(0, T, bsz):
        idx = order[b0:b0 + bsz]
        act = None if active is None else active[idx].contiguous()
        o_lp, o_lse = rlk.linear_logprob(hidden[idx].contiguous(), W, targets[idx].contiguous(), act,
                                         n_shards, workspace=ws)
        lp[idx] = o_lp
        lse[idx] = o_lse
    return lp, lse


def sharded(rlk, hidden, W, targets, active, n):
    V = W.shape[0]
    parts = []
    for r in range(n):
        vb, ve = rlk.shard_range(V, n, r)
        parts.append(rlk.linear_logprob_shard(hidden, W[vb:ve], targets, active, V, n, r))
    return rlk.lse_merge(parts, active)


@pytest.mark.parametrize("T,H,V", [(300, 256, 1000), (64, 256, 1024), (520, 512, 7777)])
def test_small_invariance(rlk, cuda_device, T, H, V):
    w = WL.to_device(WL.small_case(T, H, V, seed=T + V, inactive_frac=0.1), cuda_device)
    ref_lp, ref_lse = rlk.linear_logprob(w.hidden, w.W, w.targets, w.active, 1)
    for bsz in (1, 7, 64, 129):
        for seed in (0, 1):
            order = torch.from_numpy(WL.permutation(T, seed)).to(cuda_device)
            lp, lse = in_batches(rlk, w.hidden, w.W, w.targets, w.active, bsz, 1, order)
            assert_same(lp, ref_lp, "bsz=%d perm=%d" % (bsz, seed))
            assert_same(lse, ref_lse, "bsz=%d perm=%d lse" % (bsz, seed))
    nt = (V + 127) // 128
    for n in (2, 4, 8):
        if n > nt:
            continue
        lp, lse = rlk.linear_logprob(w.hidden, w.W, w.targets, w.active, n)
        assert_same(lp, ref_lp, "n_shards=%d" % n)
        lp, lse = sharded(rlk, w.hidden, w.W, w.targets, w.active, n)
        assert_same(lp, ref_lp, "shard API n=%d" % n)
        assert_same(lse, ref_lse, "shard API n=%d lse" % n)
    for _ in range(3):
        lp, lse = rlk.linear_logprob(w.hidden, w.W, w.targets, w.active, 1)
        assert_same(lp, ref_lp, "repeat")


def test_qwen_decode_rows_match_packed(rlk, qwen):
    """Rollout-style decode batches (T = 1, 8, 64, 256) vs the same rows inside the packed batch."""
    pk = qwen.packed
    full_lp, full_lse = rlk.linear_logprob(pk.hidden, qwen.W, pk.targets, None, 4)
    for T in (1, 8, 64, 256):
        idx = torch.from_numpy(WL.decode_rows(T)).to(qwen.device)
        lp, lse = rlk.linear_logprob(pk.hidden[idx].contiguous(), qwen.W,
                                     pk.targets[idx].contiguous(), None, 1)
        assert_same(lp, full_lp[idx], "decode T=%d" % T)
        assert_same(lse, full_lse[idx], "decode T=%d lse" % T)


def test_qwen_shard_api_matches_full(rlk, qwen):
    pk = qwen.packed
    full_lp, full_lse = rlk.linear_logprob(pk.hidden, qwen.W, pk.targets, None, 1)
    for n in (2, 4, 8):
        lp, lse = sharded(rlk, pk.hidden, qwen.W, pk.targets, None, n)
        assert_same(lp, full_lp, "qwen shard API n=%d" % n)
        assert_same(lse, full_lse, "qwen shard API n=%d lse" % n)
        lp, lse = rlk.linear_logprob(pk.hidden, qwen.W, pk.targets, None, n)
        assert_same(lp, full_lp, "qwen n_shards=%d" % n)


@pytest.mark.slow
def test_qwen_sweep_set(rlk, qwen):
    """Fixed 8192-token set: batch sizes {1,7,64,1024,8192} x row orders x shard counts."""
    sw = WL.sweep_set(qwen.W, qwen.device)
    T = sw.hidden.shape[0]
    ref_lp, ref_lse = rlk.linear_logprob(sw.hidden, qwen.W, sw.targets, None, 1)
    # b = 1 over the first 512 tokens (each call is one row; order is immaterial)
    lp, lse = in_batches(rlk, sw.hidden[:512], qwen.W, sw.targets[:512], None, 1)
    assert_same(lp, ref_lp[:512], "b=1")
    for bsz in (7, 64, 1024, 8192):
        for seed in (11, 12, 13):
            order = torch.from_numpy(WL.permutation(T, seed)).to(qwen.device)
            lp, lse = in_batches(rlk, sw.hidden, qwen.W, sw.targets, None, bsz, 1, order)
            assert_same(lp, ref_lp, "sweep b=%d perm=%d" % (bsz, seed))
            assert_same(lse, ref_lse, "sweep b=%d perm=%d lse" % (bsz, seed))
    for n in (2, 4, 8):
        lp, lse = in_batches(rlk, sw.hidden, qwen.W, sw.targets, None, 1024, n,
                             torch.from_numpy(WL.permutation(T, 20 + n)).to(qwen.device))
        assert_same(lp, ref_lp, "sweep shards=%d" % n)


def test_hidden_of_other_rows_cannot_leak(rlk, cuda_device):
    """Inactive rows full of huge values leave every active row's bits unchanged."""
    w = WL.to_device(WL.small_case(256, 256, 2000, seed=31), cuda_device)
    ref_lp, ref_lse = rlk.linear_logprob(w.hidden, w.W, w.targets, None, 1)
    hid = w.hidden.clone()
    act = torch.ones(256, dtype=torch.uint8, device=cuda_device)
    act[1::3] = 0
    hid[1::3] = 3.0e38
    tg = w.targets.clone()
    tg[1::3] = -5  # never read for inactive rows
    lp, lse = rlk.linear_logprob(hid, w.W, tg, act, 1)
    keep = act.bool()
    assert_same(lp[keep], ref_lp[keep], "active rows")
    assert torch.all(lp[~keep] == 0) and torch.all(lse[~keep] == 0)


@pytest.mark.parametrize("T,H,V", [(5, 128, 1000), (300, 256, 40000), (64, 512, 262144),
                                   (9, 64, 129)])
def test_tree_layouts_agree(rlk, cuda_device, monkeypatch, T, H, V):
    """One warp per token and one CTA per token evaluate the same tree: same bits, records too."""
    w = WL.to_device(WL.small_case(T, H, V, seed=T + 3, w_std=0.05, inactive_frac=0.2), cuda_device)
    nt = (V + 127) // 128
    for n in (1, 2, 4, 8):
        if n > nt:
            continue
        outs = []
        for threads in ("32", "256"):
            monkeypatch.setenv("RLK_TEST_TREE_THREADS", threads)
            ws = rlk.new_workspace(T, V, n, cuda_device)
            lp, lse = rlk.linear_logprob(w.hidden, w.W, w.targets, w.active, n, workspace=ws)
            vb, ve = rlk.shard_range(V, n, n - 1)
            part = rlk.linear_logprob_shard(w.hidden, w.W[vb:ve], w.targets, w.active, V, n, n - 1)
            outs.append((lp, lse, rlk.workspace_records(ws, T, V, n).clone(), part))
        monkeypatch.delenv("RLK_TEST_TREE_THREADS")
        (a_lp, a_lse, a_rec, a_part), (b_lp, b_lse, b_rec, b_part) = outs
        assert_same(a_lp, b_lp, "logprob n=%d" % n)
        assert_same(a_lse, b_lse, "lse n=%d" % n)
        assert torch.equal(a_rec, b_rec), "records n=%d" % n
        assert torch.equal(a_part, b_part), "shard record n=%d" % n


@pytest.mark.parametrize("T,H,V", [(1, 256, 5000), (300, 512, 20000)])
def test_inputs_written_just_before_each_call(rlk, cuda_device, T, H, V):
    """The logits and tile-tree kernels start early (programmatic dependent launch) and
    wait for the previous kernel before touching memory.  Rewriting the inputs with an
    ordinary kernel right before every call must still give each call the new inputs:
    alternate two batches through the same buffers and compare every result, bit for
    bit, with that batch's result computed alone."""
    batches = [WL.to_device(WL.small_case(T, H, V, seed=s), cuda_device) for s in (31, 32)]
    W = batches[0].W
    ref = [rlk.linear_logprob(b.hidden, W, b.targets, None, 2) for b in batches]
    ref_mat = [rlk.logits_logprob(rlk.debug_logits(b.hidden, W), b.targets, None, 2)
               for b in batches]
    g = torch.full((T,), 0.5, dtype=torch.float32, device=cuda_device)
    ref_bwd = [rlk.linear_logprob_backward(b.hidden, W, b.targets, g, r[1], want_W=False)[0]
               for b, r in zip(batches, ref)]
    hidden = torch.empty_like(batches[0].hidden)
    targets = torch.empty_like(batches[0].targets)
    logits = torch.empty((T, V), dtype=torch.float32, device=cuda_device)
    ws = rlk.new_workspace(T, V, 2, cuda_device)
    lp = torch.empty(T, dtype=torch.float32, device=cuda_device)
    lse = torch.empty_like(lp)
    for it in range(12):
        k = it % 2
        hidden.copy_(batches[k].hidden)   # ordinary kernels, immediately before the call
        targets.copy_(batches[k].targets)
        rlk.linear_logprob(hidden, W, targets, None, 2, lp, lse, ws)
        assert_same(lp, ref[k][0], "logprob, iteration %d" % it)
        assert_same(lse, ref[k][1], "lse, iteration %d" % it)
        logits.copy_(rlk.debug_logits(batches[k].hidden, W))
        m_lp, m_lse = rlk.logits_logprob(logits, targets, None, 2)
        assert_same(m_lp, ref_mat[k][0], "materialised logprob, iteration %d" % it)
        gh, _ = rlk.linear_logprob_backward(hidden, W, targets, g, ref[k][1], want_W=False)
        assert_same(gh, ref_bwd[k], "grad_hidden, iteration %d" % it)
