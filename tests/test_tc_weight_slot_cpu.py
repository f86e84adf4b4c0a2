"""The tensor-core LogSumExp carries the log-weight relative to its tile's largest,
v = max(w' - F, -1024) in [-1024, 0], as a split fp16 pair (hi = fp16(v), lo = fp16(v - hi)),
multiplied by A's slot of 1 in the product: the accumulator receives hi + lo.  The prepass's
split is replayed here with NumPy's fp16 rounding and the pair is checked to carry v to within
2^-21 of its size (plus fp16's subnormal spacing for tiny v).  In the tile's frame, where the
largest term is 2^0 = 1, a term 2^(t + v) then moves by at most max_v |v| 2^v 2^-21 ln 2 < 2e-7
of that largest term (its own relative error grows with |v|, its weight falls faster)."""
import numpy as np


def _split(v32):
    hi = v32.astype(np.float16)
    lo = (v32 - hi.astype(np.float32)).astype(np.float16)
    return hi.astype(np.float32), lo.astype(np.float32)


def test_pair_carries_the_weight():
    r = np.random.Generator(np.random.PCG64(61))
    v = np.concatenate([-r.uniform(0, 1024, 200_000), -10.0 ** r.uniform(-12, 3, 200_000), [0.0, -1024.0]])
    v32 = np.maximum(v, -1024.0).astype(np.float32)
    hi, lo = _split(v32)
    got = hi.astype(np.float64) + lo.astype(np.float64)
    err = np.abs(got - v32.astype(np.float64))
    assert np.all(err <= 2.0 ** -21 * np.abs(v32) + 2.0 ** -24)
    # each term's error in the tile's frame (its largest term is 2^0 = 1): 2^v (2^err - 1)
    assert np.all(np.exp2(v32.astype(np.float64)) * np.expm1(err * np.log(2.0)) < 2e-7)


def test_clamp_makes_empty_weights_vanish():
    """-1024 (an empty weight, or one below 2^-1024 of the tile's largest) is exact in fp16 and
    gives a term 2^(t - 1024) that underflows to 0 for any t <= 0 the norm guard admits."""
    hi, lo = _split(np.array([-1024.0], np.float32))
    assert hi[0] == -1024.0 and lo[0] == 0.0
    assert np.float32(2.0) ** np.float32(-1024.0 - 0.0) == 0.0
