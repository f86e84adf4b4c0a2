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


def test_roofline_peaks():
    """The pipe-count peaks the bench reports (152 SMs, 2070 MHz; FP32 128, ALU 64 lanes per
    clock and SM; ex2 32, sqrt/rcp/rsqrt 16): Sum at D = 3 is FP32-bound at 7 operations a pair,
    the K-min's direct count is 6 FP32 + 1 ALU (its screen's 3 + 1), the Laplace Sum is bound by
    its two XU operations (sqrt at 16 lanes, ex2 at 32)."""
    xu = {"ex2": 32.0, "rcp": 16.0, "rsqrt": 16.0, "sqrt": 16.0}
    clk = 152 * 2070e6
    s = bench.roofline("sum", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, "k")
    assert abs(s["peak"] - clk * 128 / 7) < 1 and s["limiting_pipe"] == "fp32"
    assert abs(s["frac"] - 1e12 / s["peak"]) < 1e-12
    k = bench.roofline("knn", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, "k")
    assert abs(k["peak"] - clk * 128 / 6) < 1 and abs(k["screen"]["peak"] - clk * 128 / 3) < 1
    lp = bench.roofline("sum", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, "k", kind="laplace")
    assert abs(lp["peak"] - clk / (1 / 16 + 1 / 32)) < 1 and lp["limiting_pipe"] == "xu"
    # traffic only for a captured kernel, and only while its sources are the captured ones
    name = "grad_kernel[D=3,E=1]"
    fresh = bench.TRAFFIC[name]["source_hash"] == bench._kernel_source_hash()
    t = bench.roofline("grad", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, name)["traffic"]
    assert t == (bench.TRAFFIC[name]["bytes_per_launch"] if fresh else None)
    assert bench.roofline("grad", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, "other")["traffic"] is None


def test_max_reports_both_bounds():
    """Max / Min with one column are measured against the method's count (k b formed per pair:
    2D + 1 FP32, the kernel's XU operation, one compare) and, beside it, against the key
    scan's own count (Gaussian 2D FP32 + 1 compare; Cauchy 2D + 1 FP32 + 1 compare, no XU;
    Laplace 2D + 1 FP32, one sqrt, 1 compare); wider signals carry only the method's."""
    xu = {"ex2": 32.0, "rcp": 16.0, "rsqrt": 16.0, "sqrt": 16.0}
    clk = 152 * 2070e6
    m = bench.roofline("max", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, "k")
    assert m["ops_per_pair"] == {"fp32": 7, "xu": {"ex2": 1}, "cmp": 1}
    assert abs(m["peak"] - clk * 128 / 7) < 1
    assert m["own_bound"]["ops_per_pair"] == {"fp32": 6, "xu": {}, "cmp": 1}
    assert abs(m["own_bound"]["peak"] - clk * 128 / 6) < 1
    assert m["own_bound"]["frac"] < m["frac"]
    assert "own_bound" in bench.roofline("min", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, "k")
    c = bench.roofline("max", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, "k", kind="cauchy")
    assert c["ops_per_pair"]["xu"] == {"rcp": 1} and abs(c["peak"] - clk * 16) < 1   # rcp-bound
    assert c["own_bound"]["ops_per_pair"] == {"fp32": 7, "xu": {}, "cmp": 1}
    assert abs(c["own_bound"]["peak"] - clk * 128 / 7) < 1
    lp = bench.roofline("max", 3, 1, 1e-3, 1e9, 152, 2070.0, xu, "k", kind="laplace")
    assert lp["own_bound"]["ops_per_pair"] == {"fp32": 7, "xu": {"sqrt": 1}, "cmp": 1}
    assert abs(lp["own_bound"]["peak"] - clk * 16) < 1   # sqrt-bound
    assert "own_bound" not in bench.roofline("max", 3, 4, 1e-3, 1e9, 152, 2070.0, xu, "k")
