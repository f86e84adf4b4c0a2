"""Large index ranges and run-to-run determinism, through the C ABI.

* N = 2^28 + 12345 points (D = 1): indices far above 2^24 must come out exact, the
  split-j partial layout must not overflow, and ties between a low and a very high
  index must keep the low one.
* N*D above 2^31 elements (N = 1.4e8 points in D = 16, y = 9 GB): rows planted as exact
  copies of points beyond element 2^31 must find them (K-min, ArgMax) and their Sum must
  see them.
* Every kernel family run twice on the same inputs gives bitwise-equal results (split-j
  partials are combined in a fixed order; nothing depends on scheduling)."""
import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr
from symbolic_matrix_reductions_gb300 import workloads as W

from parity import check_knn, check_maxmin, check_sum

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


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


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def test_elements_beyond_2_31():
    M, D, N = 64, 16, 140_000_000                       # N*D = 2.24e9 > 2^31
    g = torch.Generator(device=DEV).manual_seed(2031)
    y = torch.randn((N, D), device=DEV, generator=g)
    first = (1 << 31) // D + 1                          # first point whose elements lie past 2^31
    jh = np.linspace(first, N - 1, M).round().astype(np.int64)   # fp64 and integer: in range
    assert jh.min() >= first and jh.max() <= N - 1
    j = torch.from_numpy(jh).to(DEV)
    x = y[j].clone()                                    # row k is an exact copy of point j_k
    b = torch.zeros((N, 1), device=DEV)
    b[j] = 1.0
    idx, dist = kr.kernel_knn(x, y, 2)
    assert np.array_equal(_np(idx)[:, 0], jh) and (_np(dist)[:, 0] == 0).all()
    am, vm = kr.kernel_reduce_arg(x, y, b, 0.5, "max")
    assert np.array_equal(_np(am)[:, 0], jh) and (_np(vm)[:, 0] == 1.0).all()
    # Sum: only the planted points carry weight; the exact value from those points alone
    a = _np(kr.kernel_reduce(x, y, b, 0.5, "sum"))[:, 0]
    xp = x.double().cpu().numpy()
    ref = np.exp(-((xp[:, None, :] - xp[None, :, :]) ** 2).sum(-1) / 0.25).sum(1)
    assert np.all(np.abs(a - ref) <= 1e-4 * ref)
    del y, b


def test_large_n_index_range(orc):
    M, N = 64, (1 << 28) + 12345
    r = np.random.Generator(np.random.PCG64(2028))
    # rows far outside the N(0,1) cloud (values no random point takes), each planted in y
    x = (50.0 + 0.25 * np.arange(M, dtype=np.float32))[:, None]
    y = r.standard_normal((N, 1)).astype(np.float32)
    y[N - 1 - np.arange(M), 0] = x[:, 0]          # each row's exact match sits near the end ...
    y[1000 + np.arange(0, M, 2), 0] = x[::2, 0]    # ... and even rows also have one at a low index
    b = np.ones((N, 1), np.float32)
    xt, yt, bt = (torch.from_numpy(a).to(DEV) for a in (x, y, b))
    idx, dist = kr.kernel_knn(xt, yt, 3)
    i_ref, d_ref, n_ref = orc.knn(x, y, 3)
    check_knn(_np(idx), _np(dist), x, y, i_ref, d_ref, n_ref, "N = 2^28 + 12345")
    idx0 = _np(idx)[:, 0]
    assert (idx0[::2] == 1000 + np.arange(0, M, 2)).all()      # the tie keeps the low index
    assert (idx0[1::2] == N - 1 - np.arange(1, M, 2)).all()    # indices above 2^28 exact
    am, vm = kr.kernel_reduce_arg(xt, yt, bt, 0.1, "max")
    assert np.array_equal(_np(am)[:, 0], idx0)                 # b = 1: ArgMax is the nearest point
    rows = np.arange(0, M, 8)
    a = _np(kr.kernel_reduce(xt, yt, bt, 0.1, "sum"))
    a_ref, S_ref = orc.gauss_sum(x[rows], y, b, 0.1)
    check_sum(a[rows], a_ref, S_ref, "N = 2^28 + 12345")


def _twice(fn):
    first = [_np(t).copy() for t in fn()]
    second = [_np(t) for t in fn()]
    return all(np.array_equal(p, q, equal_nan=True) for p, q in zip(first, second))


def test_determinism_every_family():
    inp = W.generate("gauss_d3", M=20_000, N=60_000)
    x, y, b, g = (torch.from_numpy(inp[k]).to(DEV) for k in ("x", "y", "b", "g"))
    s = inp["sigma"]
    f50 = W.generate("falkon_d50", M=3000, N=100_000)
    x5, y5, b5 = (torch.from_numpy(f50[k]).to(DEV) for k in ("x", "y", "b"))
    xb, yb, bb = (t[:18_000].reshape(3, 6000, -1).contiguous() for t in (x, y, b))
    order = np.argsort(inp["y"][:, 0])
    ri, si, rj = np.array([[0, 10_000], [10_000, 20_000]]), np.array([2, 3]), np.array([[0, 30_000], [45_000, 60_000], [0, 60_000]])
    cases = {
        "sum": lambda: [kr.kernel_reduce(x, y, b, s, "sum")],
        "lse": lambda: [kr.kernel_reduce(x, y, b, s, "lse")],
        "grad-x": lambda: [kr.kernel_reduce_grad_x(x, y, b, g, s)],
        "grad-y": lambda: [kr.kernel_reduce_grad_y(x, y, b, g, s)],
        "knn": lambda: list(kr.kernel_knn(x, y, 10)),
        "cauchy sum": lambda: [kr.kernel_reduce(x, y, b, s, "sum", kernel="cauchy")],
        "laplace argmin": lambda: list(kr.kernel_reduce_arg(x, y, b, s, "min", kernel="laplace")),
        "tensor sum": lambda: [kr.kernel_reduce(x5, y5, b5, 1.0, "sum")],
        "tensor lse": lambda: [kr.kernel_reduce(x5, y5, b5, 1.0, "lse")],
        "batched sum": lambda: [kr.kernel_reduce(xb, yb, bb, s, "sum")],
        "block-sparse max": lambda: list(kr.kernel_reduce_ranges(x, y[order].contiguous(), b[order].contiguous(), s,
                                                                  "max", ri, si, rj, want_index=True)),
    }
    for name, fn in cases.items():
        assert _twice(fn), name
