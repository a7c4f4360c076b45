"""The tile-tree kernels' evaluation order, replayed on the CPU.

``k_tile_tree`` (a warp per token) and ``k_tile_tree_cta`` (256 threads per
token) spread a token's perfect tree of 2^depth slots over their threads and
merge each thread's node in a fixed schedule (``merge_run`` in
``csrc/rlk_merge.cu``): every even slot of a node holds a tile, an odd slot
2i+1 holds one exactly when the bit reversal of i is below count - L/2, and
level 1 merges a pair only where its odd slot is held; the levels above run
as a binary counter; then the threads' nodes merge pairwise, lower thread on
the left, and an empty side leaves the other unchanged.  This test replays
that schedule symbolically for every tile count the library accepts and
checks that it builds exactly the contract's recursive-bisection tree (the
oracle's ``tile_tree_nodes`` split rule), including the shard nodes.
"""
import math

import pytest

from oracle import linear_logprob as O

MAX_TILES = 262144 // 128


def bisection(a, b):
    """The contract's tree over tiles [a, b) as nested pairs (oracle split rule)."""
    if b - a == 1:
        return a
    (l0, l1), (r0, r1) = O.tile_tree_nodes(b - a, 1)
    return (bisection(a + l0, a + l1), bisection(a + r0, a + r1))


def depth_of(n):
    return 0 if n <= 1 else math.ceil(math.log2(n))


def slot_run(u, log_p, depth, n_tiles):
    """Mirror of the kernels' slot_run: thread u's node (first tile, tile count)."""
    first, count = 0, n_tiles
    levels = log_p
    if depth < log_p:
        if u >= (1 << depth):
            return 0, 0
        levels = depth
    for b in range(levels - 1, -1, -1):
        left = (count + 1) >> 1
        if (u >> b) & 1:
            first += left
            count -= left
        else:
            count = left
    return first, count


def brev(i, bits):
    return int(format(i, "0%db" % bits)[::-1], 2) if bits else 0


def merge_run(first, count, log_l):
    """Mirror of merge_run: the node's expression, or None when it holds no tile."""
    if log_l == 0:
        return first if count > 0 else None
    pairs = 1 << (log_l - 1)
    assert pairs <= count <= 2 * pairs, (first, count, log_l)
    odd_limit = count - pairs
    pend = [None] * log_l
    rel = 0
    x = None
    for i in range(pairs):
        x = first + rel
        rel += 1
        if brev(i, log_l - 1) < odd_limit:
            x = (x, first + rel)
            rel += 1
        level = 0
        while level < log_l - 1 and (i >> level) & 1:
            x = (pend[level], x)
            level += 1
        if level < log_l - 1:
            pend[level] = x
    assert rel == count
    return x


def join(left, right):
    if left is None:
        return right
    if right is None:
        return left
    return (left, right)


@pytest.mark.parametrize("log_p", [5, 8])
def test_schedule_builds_the_bisection_tree(log_p):
    sizes = range(1, MAX_TILES + 1) if log_p == 5 else \
        sorted(set(list(range(1, 700)) + list(range(700, MAX_TILES + 1, 13)) +
                   [1023, 1024, 1025, 1187, 1536, 2047, 2048]))
    for n in sizes:
        depth = depth_of(n)
        log_l = max(depth - log_p, 0)
        nodes = [merge_run(*slot_run(u, log_p, depth, n), log_l) for u in range(1 << log_p)]
        shard_nodes = {}
        level_nodes = nodes
        for lv in range(log_p):
            shard_nodes[lv] = level_nodes
            level_nodes = [join(level_nodes[2 * i], level_nodes[2 * i + 1])
                           for i in range(len(level_nodes) // 2)]
        shard_nodes[log_p] = level_nodes
        assert level_nodes[0] == bisection(0, n), n
        # shard r of 2^d is the thread group r << shard_level after shard_level levels
        for d in range(0, 4):
            if (1 << d) > n:
                break
            shard_level = min(depth, log_p) - d
            if shard_level < 0:
                continue
            got = shard_nodes[shard_level][: 1 << d]
            want = [bisection(a, b) for a, b in O.tile_tree_nodes(n, d)]
            assert got == want, (n, d)
