"""Host model of the tensor-core K-min's chained splits (no GPU).

The K-min kernel at 32 <= D <= 62 splits a row's points j into ranges, one block each.  A
block's list starts from the row's shared list (its distances enter as stand-ins that rank
after any point of equal distance and are never reported), screens each tile's points with an
approximate distance (within a margin of the true one) against its list's K-th distance or the
shared one, takes the true distance of every passing point, and writes its list into the shared
one, slot by slot, after a tile where it became better.  Blocks run in any interleaving, so a
block may read the shared list while another block is half way through rewriting it.

This model runs that scheme on random interleavings, with torn reads and screen errors up to
the margin, on distances drawn from a few integers (so that exact ties are everywhere), and
checks that merging the blocks' reported lists gives the K smallest (distance, index) pairs,
the lower index first on equal distances: the definition of the K-min reduction, computed here
by sorting.
"""
import math

import numpy as np
import pytest

INF = math.inf
EMPTY = (INF, INF, -1)  # (distance, tie key, index); index -1: an empty slot


def _insert(lst, entry):
    """Sorted insertion by (distance, tie key) into a fixed-length list; the last entry falls
    off.  A point's tie key is its index j; a stand-in's is +inf (it ranks after any point of
    equal distance), or -1 in the deliberately wrong variant the last test runs."""
    for k in range(len(lst)):
        if entry[:2] < lst[k][:2]:
            lst.insert(k, entry)
            lst.pop()
            return


class Block:
    def __init__(self, j_lo, j_hi, K, KP):
        self.j_lo, self.j_hi, self.K = j_lo, j_hi, K
        self.lst = [EMPTY] * KP
        self.started = False
        self.next_j = j_lo
        self.pub = INF

    def kth(self):
        return self.lst[self.K - 1]


def _run_row(d, K, KP, S, tile, margin, rng, stand_in_tie=INF, reread=False):
    N = len(d)
    chunk = -(-(-(-N // S)) // tile) * tile
    blocks = [Block(lo, min(N, lo + chunk), K, KP) for lo in range(0, N, chunk)]
    shared = [INF] * KP
    pending = []  # (slot, value) writes not yet landed
    live = list(range(len(blocks)))
    while live or pending:
        # one scheduler step: land one pending slot write, or advance one block by one tile
        if pending and (not live or rng.random() < 0.5):
            slot, value = pending.pop(int(rng.integers(len(pending))))
            shared[slot] = value
            continue
        bi = live[int(rng.integers(len(live)))]
        b = blocks[bi]
        if not b.started:
            b.started = True
            for v in list(shared):  # the whole shared list, as it stands (possibly torn)
                if v < INF:
                    _insert(b.lst, (v, stand_in_tie, -2))  # index -2: a stand-in
            b.pub = b.kth()[0]
            continue
        if reread:  # deliberately wrong: the whole shared list again, which may hold this block's points
            for v in list(shared):
                if v < INF:
                    _insert(b.lst, (v, stand_in_tie, -2))
        gth = shared[K - 1]  # the shared K-th slot, read once a tile
        thr = min(b.kth()[0], gth) + margin
        j_end = min(b.j_hi, b.next_j + tile)
        for j in range(b.next_j, j_end):
            screened = d[j] + rng.uniform(-margin, margin)
            if screened > thr:
                continue
            entry = (d[j], j, j)
            if entry[:2] < b.kth()[:2]:
                _insert(b.lst, entry)
                thr = min(b.kth()[0], gth) + margin
        b.next_j = j_end
        kth = b.kth()[0]
        if kth < b.pub and kth < gth:  # share the list, slot by slot
            pending.extend((k, e[0]) for k, e in enumerate(b.lst))
            b.pub = kth
        if b.next_j >= b.j_hi:
            live.remove(bi)
    # each block reports its own points among its first K entries, in order; a merge by
    # (distance, index) takes the first K of the union
    reported = sorted((e[0], e[2]) for b in blocks for e in b.lst[:K] if e[2] >= 0)
    return reported[:K]


@pytest.mark.parametrize("K,KP", [(1, 1), (3, 4), (10, 10), (7, 16), (32, 32)])
def test_chained_splits_give_the_k_min(K, KP):
    rng = np.random.default_rng(1000 + 7 * K + KP)
    for trial in range(60):
        N = int(rng.integers(1, 400))
        S = int(rng.integers(1, 9))
        levels = int(rng.integers(1, 12))
        d = rng.integers(0, levels, size=N).astype(float)  # exact ties everywhere
        margin = float(rng.choice([0.0, 0.4, 1.5]))
        got = _run_row(d, K, KP, S, tile=16, margin=margin, rng=rng)
        order = sorted(range(N), key=lambda j: (d[j], j))[:K]
        want = [(d[j], j) for j in order]
        assert got == want, (trial, N, S, margin)


def test_model_catches_a_stand_in_that_wins_ties():
    """The model is sharp: with stand-ins ranking before points of equal distance, a tie
    between a stand-in and the point of a split whose index should win drops that point, and
    some interleaving shows it."""
    rng = np.random.default_rng(5)
    failures = 0
    for _ in range(200):
        N = 64
        d = rng.integers(0, 3, size=N).astype(float)
        got = _run_row(d, 4, 4, 4, tile=8, margin=0.0, rng=rng, stand_in_tie=-1)
        order = sorted(range(N), key=lambda j: (d[j], j))[:4]
        if got != [(d[j], j) for j in order]:
            failures += 1
    assert failures > 0


def test_model_catches_a_block_that_rereads_its_own_points():
    """The model is sharp the other way too: a block that takes the whole shared list again
    after it has shared its own, holds its own points twice (once as stand-ins), and some
    interleaving then turns away a point of the K smallest."""
    rng = np.random.default_rng(6)
    failures = 0
    for _ in range(200):
        N = 96
        d = rng.permutation(N).astype(float)  # distinct distances: only the rereading can fail
        got = _run_row(d, 4, 4, 3, tile=8, margin=0.0, rng=rng, reread=True)
        order = sorted(range(N), key=lambda j: (d[j], j))[:4]
        if got != [(d[j], j) for j in order]:
            failures += 1
    assert failures > 0
