"""Dense Max/Min's branch-free scan, replayed on the CPU.

The kernel keeps, per row, the running maximum (fmax over each block of steps) and the
start of the last block whose maximum strictly exceeded it; after each tile it recomputes that
block and takes the first point equal to the maximum.  That must give the value and the
lowest index of a plain argmax over the whole row, for any values: ties inside a block,
between blocks, between tiles, NaN padding (which never wins) and -inf.  Here the same
procedure runs on random value arrays with many exact ties and is compared with NumPy's
argmax (first occurrence)."""
import numpy as np
import pytest


def _scan(v, tile, block):
    """v: values of one row in j order.  Returns (max, index) as the kernel derives them."""
    hi, bj = -np.inf, -1
    for t0 in range(0, len(v), tile):
        tv = v[t0:t0 + tile]
        pad = (-len(tv)) % block
        tv = np.concatenate([tv, np.full(pad, np.nan)])   # padding points carry NaN
        last = -1
        for b0 in range(0, len(tv), block):
            bm = np.nanmax(tv[b0:b0 + block]) if not np.all(np.isnan(tv[b0:b0 + block])) else -np.inf
            if bm > hi:                                    # strictly greater raises it
                last = b0
            hi = max(hi, bm)
        if last >= 0:                                      # first point of that block equal to it
            blk = tv[last:last + block]
            bj = t0 + last + int(np.nonzero(blk == hi)[0][0])
    return hi, bj


@pytest.mark.parametrize("tile,block", [(512, 8), (64, 8), (16, 4), (8, 8)])
@pytest.mark.parametrize("seed", range(6))
def test_block_scan_matches_first_argmax(tile, block, seed):
    r = np.random.Generator(np.random.PCG64(seed))
    for n in (1, 7, 8, 9, 100, 1000):
        v = r.integers(-5, 6, size=n).astype(np.float64)   # few distinct values: many exact ties
        if seed % 2:
            v[r.random(n) < 0.3] = -np.inf
        hi, bj = _scan(v, tile, block)
        if np.all(v == -np.inf):
            assert hi == -np.inf and bj == -1
            continue
        assert hi == v.max() and bj == int(np.argmax(v)), (n, tile, block)
