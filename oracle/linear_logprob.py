"""fp64 oracle of the selected-token logprob over the full vocabulary.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): nothing on the
product path imports this module.

What it computes, and where the pages say so:

* "vLLM RL-Kernel v0.1.0: ROCm 上でのビット単位のトレーニング-ロールアウト一貫性",
  strict-path boundary table, row "Linear logprob": the result covers the
  actual vocabulary range, the target's owner, a local reduction and a
  cross-rank log-sum-exp merge.
* Bitwise-consistency blog on RL-Kernel + vime on AMD, section 3.1: a
  token's logprob is log_softmax over the logits, read at the target; its
  max and sum reductions are what decide the last bits.

So for each active row t, with logits l[t, v] = sum_k h[t, k] * W[v, k]:

    M = max_v l[t, v]
    S = sum_v exp(l[t, v] - M)
    lse = M + log(S)
    logprob = l[t, target[t]] - lse

Inactive rows give (0, 0).  Everything is fp64: bf16 inputs widen exactly,
each product of two bf16 values is exact in fp64, and the dot products use a
library matmul (the logits are independent of one another, so the matmul is
only cut into vocabulary chunks to bound memory).  The exp sum is numpy's
pairwise sum, whose relative error is below ~2e-15 at V = 151936.

Also here, for the shard-merge invariant (the same boundary-table row's
"cross-rank LSE merge"): the vocabulary ranges of the canonical tile tree
(recursive bisection of the 128-wide tiles, larger half first) and the fp64
merge of per-range (M, S) records.  This oracle ignores the fp32 contract
entirely; ``contract_emulator.c`` covers that.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

VOCAB_TILE = 128


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (bf16 is the top half of fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def logits(hidden_bits: np.ndarray, W_bits: np.ndarray, rows: Optional[Sequence[int]] = None,
           vocab_chunk: int = 16384) -> np.ndarray:
    """l[t, v] = sum_k h[t, k] W[v, k] in fp64 for the selected rows -> [len(rows), V]."""
    h = decode_bf16(hidden_bits if rows is None else hidden_bits[np.asarray(rows)])
    V = W_bits.shape[0]
    out = np.empty((h.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, vocab_chunk):
        v1 = min(V, v0 + vocab_chunk)
        out[:, v0:v1] = h @ decode_bf16(W_bits[v0:v1]).T
    return out


def lse_and_logprob_from_logits(L: np.ndarray, targets: np.ndarray,
                                active: Optional[np.ndarray] = None
                                ) -> Tuple[np.ndarray, np.ndarray]:
    """(logprob, lse) per row from fp64 logits [T, V]; inactive rows -> (0, 0).

    An active row whose target lies outside [0, V) gets NaN (no owner).
    """
    T, V = L.shape
    M = L.max(axis=1)
    S = np.exp(L - M[:, None]).sum(axis=1)
    lse = M + np.log(S)
    tg = np.asarray(targets, dtype=np.int64)
    ok = (tg >= 0) & (tg < V)
    tl = np.where(ok, L[np.arange(T), np.clip(tg, 0, V - 1)], np.nan)
    lp = tl - lse
    if active is not None:
        act = np.asarray(active).astype(bool)
        lp = np.where(act, lp, 0.0)
        lse = np.where(act, lse, 0.0)
    return lp, lse


def log_softmax_from_logits(L: np.ndarray, active: Optional[np.ndarray] = None) -> np.ndarray:
    """fp64 log_softmax l - lse of logits [T, V]; inactive rows -> 0."""
    M = L.max(axis=1)
    lse = M + np.log(np.exp(L - M[:, None]).sum(axis=1))
    out = L - lse[:, None]
    if active is not None:
        out = np.where(np.asarray(active).astype(bool)[:, None], out, 0.0)
    return out


def selected_logprob(hidden_bits: np.ndarray, W_bits: np.ndarray, targets: np.ndarray,
                     active: Optional[np.ndarray] = None, rows: Optional[Sequence[int]] = None,
                     row_batch_bytes: int = 1 << 30) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 (logprob, lse) for every row (or the listed ``rows``) of one batch."""
    T = hidden_bits.shape[0]
    idx = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    V = W_bits.shape[0]
    per_batch = max(1, row_batch_bytes // (8 * V))
    lp = np.empty(idx.shape[0], dtype=np.float64)
    lse = np.empty(idx.shape[0], dtype=np.float64)
    tg = np.asarray(targets)[idx]
    act = None if active is None else np.asarray(active)[idx]
    for b0 in range(0, idx.shape[0], per_batch):
        b1 = min(idx.shape[0], b0 + per_batch)
        L = logits(hidden_bits, W_bits, rows=idx[b0:b1])
        lp[b0:b1], lse[b0:b1] = lse_and_logprob_from_logits(
            L, tg[b0:b1], None if act is None else act[b0:b1])
    return lp, lse


# --------------------------------------------------------------------------
# vocabulary shards of the canonical tile tree, and the fp64 cross-shard merge
# --------------------------------------------------------------------------
def n_vocab_tiles(V: int) -> int:
    return (V + VOCAB_TILE - 1) // VOCAB_TILE


def tile_tree_nodes(n_tiles: int, depth: int) -> List[Tuple[int, int]]:
    """Tile ranges [a, b) of the nodes at ``depth`` of the recursive bisection.

    A node [a, b) with more than one tile splits at a + ceil((b - a) / 2), the
    left (lower-vocabulary) half taking the extra tile.
    """
    nodes = [(0, n_tiles)]
    for _ in range(depth):
        nxt = []
        for a, b in nodes:
            if b - a < 2:
                raise ValueError("tree too shallow for this many shards")
            mid = a + (b - a + 1) // 2
            nxt += [(a, mid), (mid, b)]
        nodes = nxt
    return nodes


def shard_vocab_ranges(V: int, n_shards: int) -> List[Tuple[int, int]]:
    """Vocabulary ranges [v0, v1) of the n_shards (a power of two) tree-aligned shards."""
    depth = int(round(math.log2(n_shards)))
    if 1 << depth != n_shards:
        raise ValueError("n_shards must be a power of two")
    return [(a * VOCAB_TILE, min(V, b * VOCAB_TILE))
            for a, b in tile_tree_nodes(n_vocab_tiles(V), depth)]


def shard_partial(L: np.ndarray, v0: int, v1: int, targets: np.ndarray):
    """fp64 (M_r, S_r, target logit or 0, owned) for the vocabulary range [v0, v1)."""
    part = L[:, v0:v1]
    M = part.max(axis=1)
    S = np.exp(part - M[:, None]).sum(axis=1)
    tg = np.asarray(targets, dtype=np.int64)
    owned = (tg >= v0) & (tg < v1)
    tl = np.where(owned, L[np.arange(L.shape[0]), np.clip(tg, v0, v1 - 1)], 0.0)
    return M, S, tl, owned


def merge_partials(parts) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """fp64 merge of per-shard records -> (lse, target logit, owner count)."""
    Ms = np.stack([p[0] for p in parts])
    Ss = np.stack([p[1] for p in parts])
    M = Ms.max(axis=0)
    S = (Ss * np.exp(Ms - M[None, :])).sum(axis=0)
    tl = np.stack([p[2] for p in parts]).sum(axis=0)
    owners = np.stack([p[3] for p in parts]).astype(np.int64).sum(axis=0)
    return M + np.log(S), tl, owners


# --------------------------------------------------------------------------
# backward: gradients of sum_t g[t] * logprob[t]
# --------------------------------------------------------------------------
def grad_logits(L: np.ndarray, targets: np.ndarray, grad_logprob: np.ndarray,
                active: Optional[np.ndarray] = None) -> np.ndarray:
    """d/dl[t, v] of sum_t g[t] logprob[t] = g[t] (onehot(v = target[t]) - softmax(l[t])[v]).

    The blog on bitwise consistency (sections 3.3, 4.2) asks the kernel for a
    backward with the same numeric discipline as its forward; this is the
    fp64 definition it is checked against.  Inactive rows give 0.
    """
    T, V = L.shape
    M = L.max(axis=1)
    lse = M + np.log(np.exp(L - M[:, None]).sum(axis=1))
    P = np.exp(L - lse[:, None])
    G = -P
    tg = np.asarray(targets, dtype=np.int64)
    ok = (tg >= 0) & (tg < V)
    G[np.arange(T)[ok], tg[ok]] += 1.0
    G *= np.asarray(grad_logprob, dtype=np.float64)[:, None]
    if active is not None:
        G[~np.asarray(active).astype(bool)] = 0.0
    return G


def backward(hidden_bits: np.ndarray, W_bits: np.ndarray, targets: np.ndarray,
             grad_logprob: np.ndarray, active: Optional[np.ndarray] = None):
    """fp64 (grad_hidden [T, H], grad_W [V, H]) of sum_t g[t] * logprob[t]."""
    h = decode_bf16(hidden_bits)
    Wd = decode_bf16(W_bits)
    G = grad_logits(h @ Wd.T, targets, grad_logprob, active)
    return G @ Wd, G.T @ h
