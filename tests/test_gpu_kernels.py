"""Laplace, Cauchy and inverse-multiquadric Sums and the Max / Min reductions (with
their Arg) for every kernel, CUDA path vs the fp64 oracle through the C ABI.

Sum tolerance as for the Gaussian: |a_gpu - a| <= 1e-4 sum_j |k_ij b_je|.  Max / Min:
see parity.check_maxmin (value within 1e-4 relative; index exact unless the oracle's
extreme and runner-up are within 1e-5, where any attaining index is accepted).
"""
import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr
from symbolic_matrix_reductions_gb300 import workloads as W

from parity import check_maxmin, check_sum

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KINDS = ["gaussian", "laplace", "cauchy", "imq"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from symbolic_matrix_reductions_gb300 import build
    build.build()
    kr.load_library()


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.load()


def _dev(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in arrs]


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _case(seed, M, N, D, E):
    r = np.random.Generator(np.random.PCG64(seed))
    x = r.standard_normal((M, D)).astype(np.float32)
    y = r.standard_normal((N, D)).astype(np.float32)
    b = r.standard_normal((N, E)).astype(np.float32)
    return x, y, b


# (M, N, D, E, sigma, split): ragged row blocks and tiles, padded coordinates (5 -> 8,
# 20 -> 32, 70 -> 128) and columns, the scalar instance (D = 128) and split-j.
SHAPES = [
    (1, 1, 3, 1, 1.0, 0), (513, 1537, 3, 1, 0.5, 0), (1100, 2049, 3, 1, 0.9, 5), (700, 3000, 1, 1, 0.3, 0),
    (257, 1000, 2, 2, 1.5, 3), (300, 1001, 5, 3, 1.2, 0), (129, 600, 16, 1, 2.0, 2), (150, 300, 20, 5, 2.5, 0),
    (100, 300, 50, 1, 3.0, 4), (40, 100, 70, 4, 5.0, 0), (40, 65, 128, 16, 6.0, 2),
]


@pytest.mark.parametrize("kernel", ["laplace", "cauchy", "imq"])
@pytest.mark.parametrize("M,N,D,E,sigma,split", SHAPES)
def test_kernel_sum(orc, kernel, M, N, D, E, sigma, split):
    x, y, b = _case(M * 7 + N + D + len(kernel), M, N, D, E)
    a = kr.kernel_reduce(*_dev(x, y, b), sigma, "sum", split=split, kernel=kernel)
    a_ref, S_ref = orc.kernel_sum(x, y, b, sigma, kernel)
    check_sum(_np(a), a_ref, S_ref, f"{kernel} {M}x{N} D{D} E{E} S{split}")


@pytest.mark.parametrize("kernel", KINDS)
@pytest.mark.parametrize("M,N,D,E,sigma,split", SHAPES)
def test_maxmin(orc, kernel, M, N, D, E, sigma, split):
    x, y, b = _case(M * 3 + N + D + len(kernel), M, N, D, E)
    xt, yt, bt = _dev(x, y, b)
    for red in ("max", "min"):
        idx, val = kr.kernel_reduce_arg(xt, yt, bt, sigma, red, split=split, kernel=kernel)
        v_ref, i_ref, s_ref = orc.kernel_maxmin(x, y, b, sigma, kernel, red)
        check_maxmin(_np(val), _np(idx), x, y, b, sigma, kernel, v_ref, i_ref, s_ref,
                     f"{kernel} {red} {M}x{N} D{D} E{E} S{split}")
        # the value-only call gives the same values
        v2 = kr.kernel_reduce(xt, yt, bt, sigma, red, split=split, kernel=kernel)
        assert np.array_equal(_np(v2), _np(val))


def test_maxmin_ties_lowest_index(orc):
    """Every point of y is one of 60 distinct points, repeated: duplicates have bitwise
    equal kernel values, so each extreme is attained by a group of indices and every
    split count must return the lowest of them.  With b = 1 Max is the nearest point."""
    r = np.random.Generator(np.random.PCG64(31))
    x = r.standard_normal((400, 3)).astype(np.float32)
    y = r.standard_normal((60, 3)).astype(np.float32)[r.integers(0, 60, size=3000)]
    b = np.ones((3000, 1), np.float32)
    i1, _, _ = orc.knn(x, y, 1)
    for kernel in KINDS:
        for red in ("max", "min"):
            v_ref, i_ref, s_ref = orc.kernel_maxmin(x, y, b, 0.8, kernel, red)
            if red == "max":
                assert np.array_equal(i_ref[:, 0], i1[:, 0])
            for split in (0, 1, 7):
                idx, val = kr.kernel_reduce_arg(*_dev(x, y, b), 0.8, red, split=split, kernel=kernel)
                assert np.array_equal(_np(idx), i_ref), (kernel, red, split)


@pytest.mark.parametrize("kernel", KINDS)
def test_maxmin_key_scan_modes(orc, kernel):
    """Max / Min with one signal column scan a key that falls as |k v| rises (v = b for Max,
    -b for Min; Gaussian q - log2|v|, Laplace sqrt(q) - log2|v|, Cauchy (1 + q) / |v|,
    inverse multiquadric (1 + q) / v^2) in a mode fixed by the signs of v over a block's
    column chunk: some positive (the smallest key over them), all negative (the largest), or
    zeros without positives (the value scan).  Each case against the oracle, unsplit and
    with splits whose chunks take different modes; with rows of infinite or NaN coordinates
    (their blocks go back to the value scan) and without; and signals spanning 1e-30 to 1e30,
    outside the range where the Cauchy and inverse-multiquadric keys are exact (value scan)."""
    r = np.random.Generator(np.random.PCG64(77))
    M, N, D = 1500, 2600, 3
    x = r.standard_normal((M, D)).astype(np.float32)
    y = r.standard_normal((N, D)).astype(np.float32)
    x_bad = x.copy()
    x_bad[5, 0] = np.inf     # every distance infinite: value 0 at the first index
    x_bad[1300, 1] = np.nan  # every value NaN: -inf (Max) / +inf (Min), index -1
    pos = (np.abs(r.standard_normal((N, 1))) + 0.05).astype(np.float32)
    j = np.arange(N)[:, None]
    cases = {
        "positive": pos,
        "negative": -pos,
        "zeros and negatives": np.where(j % 7 == 0, 0.0, -pos).astype(np.float32),
        "positive then negative": np.where(j < N // 2, pos, -pos).astype(np.float32),
        "mixed": r.standard_normal((N, 1)).astype(np.float32),
        "wide range": (pos * 10.0 ** r.integers(-30, 31, size=(N, 1))).astype(np.float32),
    }
    for xs, xname in ((x, "finite rows"), (x_bad, "inf and NaN rows")):
        for name, b in cases.items():
            for red in ("max", "min"):
                v_ref, i_ref, s_ref = orc.kernel_maxmin(xs, y, b, 0.9, kernel, red)
                for split in (0, 1, 2, 5):
                    idx, val = kr.kernel_reduce_arg(*_dev(xs, y, b), 0.9, red, split=split, kernel=kernel)
                    check_maxmin(_np(val), _np(idx), xs, y, b, 0.9, kernel, v_ref, i_ref, s_ref,
                                 f"{kernel}: {xname}, {name}, {red}, split {split}")


def test_maxmin_empty_and_degenerate(orc):
    x, y, b = _case(3, 50, 0, 3, 2)
    xt, yt, bt = _dev(x, np.zeros((0, 3), np.float32), np.zeros((0, 2), np.float32))
    idx, val = kr.kernel_reduce_arg(xt, yt, bt, 1.0, "max")
    assert (_np(idx) == -1).all() and np.isneginf(_np(val)).all()
    idx, val = kr.kernel_reduce_arg(xt, yt, bt, 1.0, "min", kernel="cauchy")
    assert (_np(idx) == -1).all() and np.isposinf(_np(val)).all()
    # M = 0 is a no-op
    e = torch.empty((0, 3), device=DEV)
    kr.kernel_reduce_arg(e, *_dev(*_case(4, 1, 10, 3, 1)[1:]), 1.0, "max")


def test_kernel_sum_host_buffers(orc):
    x, y, b = _case(8, 300, 500, 4, 2)
    host = kr.kernel_reduce(*(torch.from_numpy(a) for a in (x, y, b)), 0.8, "sum", kernel="cauchy").numpy()
    dev = _np(kr.kernel_reduce(*_dev(x, y, b), 0.8, "sum", kernel="cauchy"))
    assert np.array_equal(host, dev)


def test_grad_b_other_kernel(orc):
    """The transposed product takes the kernel option like the Sum."""
    x, y, _ = _case(9, 700, 300, 3, 2)
    g = np.random.Generator(np.random.PCG64(10)).standard_normal((700, 2)).astype(np.float32)
    gb = kr.kernel_reduce_grad_b(*_dev(x, y, g), 0.6, kernel="laplace")
    ref, S = orc.kernel_sum(y, x, g, 0.6, "laplace")
    check_sum(_np(gb), ref, S, "grad-b laplace")


def test_workload_gauss_d3_maxmin_and_kernels(orc):
    """The gauss_d3 batch (M = N = 1e5) at full size; a seeded row subset with the full N."""
    inp = W.generate("gauss_d3")
    s = inp["sigma"]
    xt, yt, bt = _dev(inp["x"], inp["y"], inp["b"])
    rows = W.row_subset(inp["x"].shape[0], 1024, 13)
    for kernel in KINDS:
        idx, val = kr.kernel_reduce_arg(xt, yt, bt, s, "max", kernel=kernel)
        v_ref, i_ref, s_ref = orc.kernel_maxmin(inp["x"][rows], inp["y"], inp["b"], s, kernel, "max")
        check_maxmin(_np(val)[rows], _np(idx)[rows], inp["x"][rows], inp["y"], inp["b"], s, kernel,
                     v_ref, i_ref, s_ref, f"gauss_d3 max {kernel}")
        if kernel != "gaussian":
            a = _np(kr.kernel_reduce(xt, yt, bt, s, "sum", kernel=kernel))
            a_ref, S_ref = orc.kernel_sum(inp["x"][rows], inp["y"], inp["b"], s, kernel)
            check_sum(a[rows], a_ref, S_ref, f"gauss_d3 sum {kernel}")
