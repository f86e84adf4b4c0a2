"""bench.py's parity statistics (the JSON line's "parity" object), on CPU: the oracle's own
outputs in fp32 pass, and a result moved past a tolerance fails."""
import numpy as np

import bench


def _ref(orc):
    r = np.random.Generator(np.random.PCG64(9))
    x = r.standard_normal((40, 3)).astype(np.float32)
    y = r.standard_normal((700, 3)).astype(np.float32)
    b = r.standard_normal((700, 1)).astype(np.float32)
    g = r.standard_normal((40, 1)).astype(np.float32)
    inp = {"x": x, "y": y, "b": b, "g": g}
    return bench._oracle_step(orc, inp, 0.5, np.arange(40))


def _as_gpu(ref):
    i, d, _ = ref["knn"]
    return (ref["sum"][0].astype(np.float32), ref["lse"].astype(np.float32), ref["grad"][0].astype(np.float32),
            i.astype(np.int32), d.astype(np.float32))


def test_oracle_outputs_pass(orc):
    ref = _ref(orc)
    p = bench.parity_stats(ref, *_as_gpu(ref))
    assert p["ok"] and p["rows"] == 40 and p["knn_separated_mismatches"] == 0


def test_each_gate_fails_past_its_tolerance(orc):
    ref = _ref(orc)
    for k, bump in ((0, lambda a: a + 2e-4 * ref["sum"][1].astype(np.float32)),
                    (1, lambda L: L + np.float32(3e-4)),
                    (2, lambda g: g + 2e-4 * ref["grad"][1].astype(np.float32))):
        out = list(_as_gpu(ref))
        out[k] = bump(out[k])
        assert not bench.parity_stats(ref, *out)["ok"], k
    out = list(_as_gpu(ref))
    i = out[3].copy()
    sep = np.argwhere(np.diff(ref["knn"][1], axis=1) > 1e-3)   # two well-separated neighbours
    rr, kk = sep[0]
    i[rr, kk], i[rr, kk + 1] = i[rr, kk + 1], i[rr, kk]
    out[3] = i
    p = bench.parity_stats(ref, *out)
    assert not p["ok"] and p["knn_separated_mismatches"] >= 1
