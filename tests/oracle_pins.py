"""Pins of the fp64 oracle, written as functions of the oracle module.

Each pin checks the oracle against something other than itself: exact
rational arithmetic on tiny inputs, closed forms, invariants of softmax, or
the hand-derived tile tree.  They take the oracle as an argument so that
``test_oracle_pins.py`` can also run them against oracles with a planted
mistake and show that every such mistake is caught.
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

from invariant_selected_token_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(x: np.ndarray) -> np.ndarray:
    return workloads.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def pin_bf16_decode(O):
    # bf16 is the upper half of an IEEE binary32: sign, 8 exponent bits, 7 fraction bits
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3E80: 0.25, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x8000: -0.0, 0xBF40: -0.75}
    bits = np.array(list(cases.keys()), dtype=np.uint16)
    got = O.decode_bf16(bits)
    for b, g in zip(cases, got):
        assert g == cases[b] and math.copysign(1, g) == math.copysign(1, cases[b]), hex(b)


def pin_brute_force_tiny(O):
    """Exact rational logits and 50-digit exp/log on T<=4, H<=16, V<=32."""
    getcontext().prec = 50
    for seed, (T, H, V) in enumerate([(1, 1, 2), (3, 7, 5), (4, 16, 32), (2, 16, 17)]):
        w = workloads.small_case(T, H, V, seed=100 + seed, w_std=0.7)
        lp, lse = O.selected_logprob(w.hidden, w.W, w.targets)
        hb = workloads.bf16_bits_to_f32(w.hidden).astype(np.float64)
        Wb = workloads.bf16_bits_to_f32(w.W).astype(np.float64)
        for t in range(T):
            ls = [sum((Fraction(float(hb[t, k])) * Fraction(float(Wb[v, k])) for k in range(H)),
                      Fraction(0)) for v in range(V)]
            M = max(ls)
            S = sum((Decimal((l - M).numerator) / Decimal((l - M).denominator)).exp() for l in ls)
            Md = Decimal(M.numerator) / Decimal(M.denominator)
            lse_x = Md + S.ln()
            lt = ls[int(w.targets[t])]
            lp_x = Decimal(lt.numerator) / Decimal(lt.denominator) - lse_x
            assert abs(float(lse_x) - lse[t]) <= 1e-14 * max(1.0, abs(float(lse_x))), (seed, t)
            assert abs(float(lp_x) - lp[t]) <= 1e-14 * max(1.0, abs(float(lp_x))), (seed, t)


def pin_constant_logits(O):
    """All W rows equal -> every class has probability 1/V -> logprob = -ln V."""
    g = _golden("closed_forms.json")["neg_log_V"]
    rng = np.random.default_rng(7)
    for V in (2, 1024, 151936):
        H = 64
        row = _bits(rng.standard_normal(H) * 0.1)
        W = np.broadcast_to(row, (V, H)).copy()
        hid = _bits(rng.standard_normal((3, H)))
        tg = np.array([0, V - 1, V // 2], dtype=np.int32)
        lp, lse = O.selected_logprob(hid, W, tg)
        assert np.all(np.abs(lp - g[str(V)]) <= 1e-12), (V, lp)


def pin_two_class_softplus(O):
    """V = 2: log p(class 0) = -log(1 + exp(l1 - l0)) (H = 1, so l = h * w exactly)."""
    g = _golden("closed_forms.json")["softplus"]
    for d_str, want in g.items():
        d = float(d_str)
        # h = 1, w0 = 0, w1 = d: l0 = 0, l1 = d, all exact in bf16 for these d
        hid = _bits(np.array([[1.0]]))
        W = _bits(np.array([[0.0], [d]]))
        assert workloads.bf16_bits_to_f32(W)[1, 0] == d
        lp, lse = O.selected_logprob(hid, W, np.array([0], dtype=np.int32))
        assert abs(lp[0] - want) <= 1e-12 * max(1.0, abs(want)), (d, lp[0], want)
        lp1, _ = O.selected_logprob(hid, W, np.array([1], dtype=np.int32))
        assert abs(lp1[0] - (want + d)) <= 1e-12 * max(1.0, abs(want + d)), d


def pin_probabilities_sum_to_one(O):
    """sum_v exp(logprob_v) = 1 for one row, every target in turn."""
    w = workloads.small_case(1, 128, 777, seed=11, w_std=0.3)
    V = w.V
    hid = np.repeat(w.hidden, V, axis=0)
    lp, _ = O.selected_logprob(hid, w.W, np.arange(V, dtype=np.int32))
    total = math.fsum(math.exp(x) for x in lp)
    assert abs(total - 1.0) <= 1e-12, total


def pin_shift_invariance(O):
    """Adding c to every logit (hidden[:, k0] = 1, W[:, k0] = c) keeps logprob, shifts lse by c."""
    w = workloads.small_case(6, 64, 300, seed=12)
    base_h = workloads.bf16_bits_to_f32(w.hidden).copy()
    base_W = workloads.bf16_bits_to_f32(w.W).copy()
    base_h[:, 0] = 1.0
    base_W[:, 0] = 0.0
    lp0, lse0 = O.selected_logprob(_bits(base_h), _bits(base_W), w.targets)
    for c in (3.5, -20.25, 96.0):
        Wc = base_W.copy()
        Wc[:, 0] = c
        lp1, lse1 = O.selected_logprob(_bits(base_h), _bits(Wc), w.targets)
        assert np.all(np.abs(lp1 - lp0) <= 1e-12 * 64), c
        assert np.all(np.abs((lse1 - lse0) - c) <= 1e-12 * 128), c


def pin_shard_merge(O):
    """fp64 merge of the tree-aligned shard records equals the full lse; one owner per target."""
    w = workloads.small_case(5, 64, 1000, seed=13)
    L = O.logits(w.hidden, w.W)
    _, lse_full = O.lse_and_logprob_from_logits(L, w.targets)
    for n in (1, 2, 4, 8):
        ranges = O.shard_vocab_ranges(w.V, n)
        assert ranges[0][0] == 0 and ranges[-1][1] == w.V
        assert all(ranges[i][1] == ranges[i + 1][0] for i in range(n - 1))
        parts = [O.shard_partial(L, a, b, w.targets) for a, b in ranges]
        lse, tl, owners = O.merge_partials(parts)
        assert np.all(owners == 1)
        assert np.all(np.abs(lse - lse_full) <= 1e-12 * np.abs(lse_full)), n
        assert np.array_equal(tl, L[np.arange(w.T), w.targets])


def pin_tile_tree(O):
    """Shard tile counts follow the hand-derived bisection of 1187 and 8 tiles."""
    g = _golden("tile_tree.json")
    for V_str, rec in g.items():
        if V_str.startswith("_"):
            continue
        V = int(V_str)
        assert O.n_vocab_tiles(V) == rec["n_tiles"]
        for n in (2, 4, 8):
            ranges = O.shard_vocab_ranges(V, n)
            tiles = [(b - a + 127) // 128 for a, b in ranges]
            assert tiles == rec[str(n)], (V, n, tiles)


def pin_vocab_permutation(O):
    w = workloads.small_case(4, 32, 257, seed=14)
    perm = np.random.default_rng(3).permutation(w.V)
    inv = np.argsort(perm)
    lp0, lse0 = O.selected_logprob(w.hidden, w.W, w.targets)
    lp1, lse1 = O.selected_logprob(w.hidden, w.W[perm], inv[w.targets].astype(np.int32))
    assert np.all(np.abs(lp1 - lp0) <= 1e-12) and np.all(np.abs(lse1 - lse0) <= 1e-12)


def pin_masks_and_bad_targets(O):
    w = workloads.small_case(4, 32, 100, seed=15)
    act = np.array([1, 0, 1, 0], dtype=np.uint8)
    lp, lse = O.selected_logprob(w.hidden, w.W, w.targets, active=act)
    assert lp[1] == 0.0 and lse[1] == 0.0 and lp[3] == 0.0 and lse[3] == 0.0
    assert lp[0] != 0.0 and lse[2] != 0.0
    bad = w.targets.copy()
    bad[0] = -1
    bad[2] = w.V
    lp, lse = O.selected_logprob(w.hidden, w.W, bad)
    assert np.isnan(lp[0]) and np.isnan(lp[2]) and np.isfinite(lp[1])


def pin_tiny_regression(O):
    """First rows of the tiny workload against the stored oracle values."""
    g = _golden("tiny_oracle.json")
    w = workloads.tiny()
    lp, lse = O.selected_logprob(w.hidden, w.W, w.targets, rows=range(8))
    assert w.targets[:8].tolist() == g["targets"]
    assert np.all(np.abs(lp - np.array(g["logprob"])) <= 1e-12)
    assert np.all(np.abs(lse - np.array(g["lse"])) <= 1e-12)


def pin_backward_finite_differences(O):
    """The analytic gradients against central differences of the oracle's own forward.

    Perturbing one bf16 input and re-running the forward is an independent
    route to the same derivative (the forward is pinned separately above).
    Inputs are bf16 grid values; perturbations are done on the fp64 level by
    evaluating the forward on exact fp64 inputs, so they need no bf16 step.
    """
    w = workloads.small_case(3, 8, 11, seed=16, w_std=0.5)
    g = np.array([0.7, -1.3, 2.0])
    h = O.decode_bf16(w.hidden)
    Wd = O.decode_bf16(w.W)

    def f(hh, WW):
        lp, _ = O.lse_and_logprob_from_logits(hh @ WW.T, w.targets)
        return float(np.dot(g, lp))

    dh, dW = O.backward(w.hidden, w.W, w.targets, g)
    eps = 1e-6
    for (t, k) in [(0, 0), (1, 5), (2, 7)]:
        hp, hm = h.copy(), h.copy()
        hp[t, k] += eps
        hm[t, k] -= eps
        fd = (f(hp, Wd) - f(hm, Wd)) / (2 * eps)
        assert abs(fd - dh[t, k]) <= 1e-6 * max(1.0, abs(fd)), (t, k, fd, dh[t, k])
    for (v, k) in [(0, 0), (w.targets[1], 3), (10, 7)]:
        Wp, Wm = Wd.copy(), Wd.copy()
        Wp[v, k] += eps
        Wm[v, k] -= eps
        fd = (f(h, Wp) - f(h, Wm)) / (2 * eps)
        assert abs(fd - dW[v, k]) <= 1e-6 * max(1.0, abs(fd)), (v, k, fd, dW[v, k])


def pin_backward_rows_sum_to_zero(O):
    """Each row of onehot - softmax sums to zero, so sum_v dlogit[t, v] = 0."""
    w = workloads.small_case(5, 16, 300, seed=17)
    L = O.logits(w.hidden, w.W)
    G = O.grad_logits(L, w.targets, np.linspace(-2, 2, 5))
    assert np.all(np.abs(G.sum(axis=1)) <= 1e-12)
    assert np.all(G[np.arange(5), w.targets] * np.linspace(-2, 2, 5) >= 0)


def pin_log_softmax_exact(O):
    """Full log_softmax of small fp64 logit rows against 50-digit Decimal exp and ln.

    Decimal(x) of a double is exact, so each expected value is l_v - ln(sum_u e^(l_u))
    with only the Decimal rounding at 50 digits; logits spread over +-40 exercise the max
    shift.  The outputs of an inactive row are 0."""
    getcontext().prec = 50
    rng = np.random.default_rng(21)
    for T, V in ((1, 1), (2, 2), (3, 17), (2, 130)):
        L = rng.uniform(-40.0, 40.0, size=(T, V))
        act = np.ones(T, dtype=np.uint8)
        act[-1] = 0 if T > 1 else 1
        out = O.log_softmax_from_logits(L, act)
        for t in range(T):
            if not act[t]:
                assert np.all(out[t] == 0.0), (T, V, t)
                continue
            ln_sum = sum(Decimal(float(x)).exp() for x in L[t]).ln()
            for v in range(V):
                want = float(Decimal(float(L[t, v])) - ln_sum)
                assert abs(out[t, v] - want) <= 1e-13 * max(1.0, abs(want)), (T, V, t, v)


def pin_log_softmax_normalised(O):
    """Every active row of exp(log_softmax) sums to 1, and a row of equal logits gives -ln V."""
    rng = np.random.default_rng(22)
    L = rng.standard_normal((4, 3000)) * 6.0 + 25.0    # max far from 0
    out = O.log_softmax_from_logits(L)
    for t in range(4):
        assert abs(math.fsum(math.exp(x) for x in out[t]) - 1.0) <= 1e-12, t
    g = _golden("closed_forms.json")["neg_log_V"]
    for V in (2, 1024, 151936):
        row = np.full((1, V), 3.75)
        assert np.all(np.abs(O.log_softmax_from_logits(row) - g[str(V)]) <= 1e-12), V


def pin_log_softmax_shift_and_selection(O):
    """Adding c to a row leaves its log_softmax unchanged, and the entry at a row's target is
    the selected-token logprob of the pinned (logprob, lse) oracle on the same logits."""
    rng = np.random.default_rng(23)
    L = rng.standard_normal((5, 777)) * 4.0
    base = O.log_softmax_from_logits(L)
    for c in (-70.5, 3.25, 96.0):
        assert np.all(np.abs(O.log_softmax_from_logits(L + c) - base) <= 1e-12 * (1 + abs(c))), c
    tg = rng.integers(0, 777, 5)
    lp, _ = O.lse_and_logprob_from_logits(L, tg)
    assert np.all(np.abs(base[np.arange(5), tg] - lp) <= 1e-13 * np.maximum(1.0, np.abs(lp)))


ALL_PINS = [pin_bf16_decode, pin_brute_force_tiny, pin_constant_logits, pin_two_class_softplus,
            pin_probabilities_sum_to_one, pin_shift_invariance, pin_shard_merge, pin_tile_tree,
            pin_vocab_permutation, pin_masks_and_bad_targets, pin_backward_finite_differences,
            pin_backward_rows_sum_to_zero, pin_log_softmax_exact, pin_log_softmax_normalised,
            pin_log_softmax_shift_and_selection]
