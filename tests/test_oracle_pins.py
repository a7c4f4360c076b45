"""The fp64 oracle against its pins, and planted mistakes against the same pins.

The second half copies the oracle module, plants one plausible mistake in
the copy (on the CPU) and checks that at least one pin fails for it.
"""
import importlib.util

import numpy as np
import pytest

from oracle import linear_logprob as O
import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS + [pins.pin_tiny_regression], ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(O)


def _fresh_copy():
    spec = importlib.util.spec_from_file_location("oracle_mutant", O.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_decode_shift(m):
    def decode_bf16(bits):
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        return (b.astype(np.uint32) << 15).view(np.float32).astype(np.float64)
    m.decode_bf16 = decode_bf16


def _mut_k_reversed(m):
    orig = m.logits
    def logits(hidden_bits, W_bits, rows=None, vocab_chunk=16384):
        return orig(hidden_bits, np.ascontiguousarray(W_bits[:, ::-1]), rows, vocab_chunk)
    m.logits = logits


def _patch_lse(m, fn):
    m.lse_and_logprob_from_logits = fn


def _mut_drop_max(m):
    def f(L, targets, active=None):
        M = L.max(axis=1)
        S = np.exp(L - M[:, None]).sum(axis=1)
        lse = np.log(S)
        lp = L[np.arange(L.shape[0]), targets] - lse
        return lp, lse
    _patch_lse(m, f)


def _mut_target_off_by_one(m):
    def f(L, targets, active=None):
        M = L.max(axis=1)
        lse = M + np.log(np.exp(L - M[:, None]).sum(axis=1))
        t = np.minimum(np.asarray(targets) + 1, L.shape[1] - 1)
        return L[np.arange(L.shape[0]), t] - lse, lse
    _patch_lse(m, f)


def _mut_wrong_sign(m):
    def f(L, targets, active=None):
        M = L.max(axis=1)
        lse = M + np.log(np.exp(L - M[:, None]).sum(axis=1))
        return lse - L[np.arange(L.shape[0]), targets], lse
    _patch_lse(m, f)


def _mut_exp_sign(m):
    def f(L, targets, active=None):
        M = L.max(axis=1)
        lse = M + np.log(np.exp(M[:, None] - L).sum(axis=1))
        return L[np.arange(L.shape[0]), targets] - lse, lse
    _patch_lse(m, f)


def _mut_dropped_term(m):
    def f(L, targets, active=None):  # the sum misses the last vocabulary column
        M = L.max(axis=1)
        lse = M + np.log(np.exp(L[:, :-1] - M[:, None]).sum(axis=1))
        lp = L[np.arange(L.shape[0]), targets] - lse
        if active is not None:
            lp = np.where(active.astype(bool), lp, 0.0)
            lse = np.where(active.astype(bool), lse, 0.0)
        return lp, lse
    _patch_lse(m, f)


def _mut_mask_ignored(m):
    orig = m.lse_and_logprob_from_logits
    m.lse_and_logprob_from_logits = lambda L, targets, active=None: orig(L, targets, None)


def _mut_floor_split(m):
    def tile_tree_nodes(n_tiles, depth):
        nodes = [(0, n_tiles)]
        for _ in range(depth):
            nxt = []
            for a, b in nodes:
                mid = a + (b - a) // 2
                nxt += [(a, mid), (mid, b)]
            nodes = nxt
        return nodes
    m.tile_tree_nodes = tile_tree_nodes


def _mut_merge_unweighted(m):
    def merge_partials(parts):
        M = np.stack([p[0] for p in parts]).max(axis=0)
        S = np.stack([p[1] for p in parts]).sum(axis=0)
        tl = np.stack([p[2] for p in parts]).sum(axis=0)
        own = np.stack([p[3] for p in parts]).astype(np.int64).sum(axis=0)
        return M + np.log(S), tl, own
    m.merge_partials = merge_partials


def _mut_grad_sign(m):
    orig = m.grad_logits
    m.grad_logits = lambda L, targets, g, active=None: -orig(L, targets, g, active)


def _mut_grad_unscaled(m):
    orig = m.grad_logits
    m.grad_logits = lambda L, targets, g, active=None: orig(L, targets, np.ones_like(g), active)


def _mut_grad_transposed(m):
    def backward(hidden_bits, W_bits, targets, grad_logprob, active=None):
        h = m.decode_bf16(hidden_bits)
        Wd = m.decode_bf16(W_bits)
        G = m.grad_logits(h @ Wd.T, targets, grad_logprob, active)
        return G @ Wd, (G.T @ h)[::-1]          # rows of grad_W in the wrong order
    m.backward = backward


def _patch_log_softmax(m, fn):
    m.log_softmax_from_logits = fn


def _mut_log_softmax_drop_max(m):
    def f(L, active=None):  # lse without the max it was shifted by
        M = L.max(axis=1)
        return L - np.log(np.exp(L - M[:, None]).sum(axis=1))[:, None]
    _patch_log_softmax(m, f)


def _mut_log_softmax_sign(m):
    def f(L, active=None):
        M = L.max(axis=1)
        return (M + np.log(np.exp(L - M[:, None]).sum(axis=1)))[:, None] - L
    _patch_log_softmax(m, f)


def _mut_log_softmax_dropped_column(m):
    def f(L, active=None):  # the sum misses the last vocabulary column
        M = L.max(axis=1)
        with np.errstate(divide="ignore"):  # a one-column row leaves an empty sum
            out = L - (M + np.log(np.exp(L[:, :-1] - M[:, None]).sum(axis=1)))[:, None]
        if active is not None:
            out = np.where(np.asarray(active).astype(bool)[:, None], out, 0.0)
        return out
    _patch_log_softmax(m, f)


def _mut_log_softmax_mask_ignored(m):
    orig = m.log_softmax_from_logits
    m.log_softmax_from_logits = lambda L, active=None: orig(L, None)


MUTANTS = [_mut_decode_shift, _mut_k_reversed, _mut_drop_max, _mut_target_off_by_one,
           _mut_wrong_sign, _mut_exp_sign, _mut_dropped_term, _mut_mask_ignored,
           _mut_floor_split, _mut_merge_unweighted, _mut_grad_sign, _mut_grad_unscaled,
           _mut_grad_transposed, _mut_log_softmax_drop_max, _mut_log_softmax_sign,
           _mut_log_softmax_dropped_column, _mut_log_softmax_mask_ignored]


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutate):
    mod = _fresh_copy()
    mutate(mod)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # AssertionError, or a crash the mistake causes
            caught.append((pin.__name__, type(e).__name__))
    assert caught, "no pin caught " + mutate.__name__
