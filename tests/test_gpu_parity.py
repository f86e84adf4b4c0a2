"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small cases span several tiles and row blocks with ragged tails, every kernel
family and the split-j combine; the workload cases run the full configuration
on the GPU (the launch the benchmark times) and check a seeded row subset with
the full N against the oracle.
"""
import os

import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr
from symbolic_matrix_reductions_gb300 import workloads as W

from parity import check_grad, check_knn, check_lse, check_sum

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


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _dev(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in arrs]


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _case(seed, M, N, D, E, scale=1.0):
    r = _rng(seed)
    x = (r.standard_normal((M, D)) * scale).astype(np.float32)
    y = (r.standard_normal((N, D)) * scale).astype(np.float32)
    b = r.standard_normal((N, E)).astype(np.float32)
    g = r.standard_normal((M, E)).astype(np.float32)
    return x, y, b, g


# (M, N, D, E, sigma, split): tails around the 512-row block and the tile sizes,
# padded coordinate counts (5 -> 8, 20 -> 32, 70 -> 128), padded signal columns.
SMALL = [
    (1, 1, 3, 1, 1.0, 0), (33, 7, 3, 1, 0.7, 0), (513, 1537, 3, 1, 0.5, 0), (1100, 2049, 3, 1, 0.9, 1),
    (1100, 2049, 3, 1, 0.9, 5), (700, 3000, 1, 1, 0.3, 0), (257, 1000, 2, 2, 1.5, 0), (300, 777, 4, 3, 1.0, 3),
    (300, 1001, 5, 1, 1.2, 0), (129, 600, 16, 1, 2.0, 0), (200, 513, 16, 4, 3.0, 2), (150, 300, 20, 5, 2.5, 0),
    (100, 257, 50, 1, 3.0, 0), (100, 300, 50, 1, 3.0, 4), (64, 200, 64, 2, 4.0, 0), (40, 100, 70, 1, 5.0, 0),
    (40, 65, 128, 16, 6.0, 2), (90, 130, 8, 16, 1.5, 0),
]


@pytest.mark.parametrize("M,N,D,E,sigma,split", SMALL)
def test_sum_small(orc, M, N, D, E, sigma, split):
    x, y, b, _ = _case(M * 7 + N + D, M, N, D, E)
    a = kr.kernel_reduce(*_dev(x, y, b), sigma, "sum", split=split)
    a_ref, S_ref = orc.gauss_sum(x, y, b, sigma)
    check_sum(_np(a), a_ref, S_ref, f"{M}x{N} D{D} E{E} S{split}")


@pytest.mark.parametrize("M,N,D,E,sigma,split", SMALL)
def test_lse_small(orc, M, N, D, E, sigma, split):
    x, y, w, _ = _case(M * 5 + N + D, M, N, D, E)
    L = kr.kernel_reduce(*_dev(x, y, w), sigma, "lse", split=split)
    check_lse(_np(L), orc.gauss_lse(x, y, w, sigma), f"{M}x{N} D{D} E{E} S{split}")


@pytest.mark.parametrize("M,N,D,E,sigma,split", SMALL)
def test_grad_small(orc, M, N, D, E, sigma, split):
    x, y, b, g = _case(M * 3 + N + D, M, N, D, E)
    gx = kr.kernel_reduce_grad_x(*_dev(x, y, b, g), sigma, split=split)
    gx_ref, G_ref = orc.gauss_grad_x(x, y, b, g, sigma)
    check_grad(_np(gx), gx_ref, G_ref, f"{M}x{N} D{D} E{E} S{split}")


KNN_SMALL = [
    (1, 1, 3, 1, 0), (33, 7, 3, 10, 0), (513, 1537, 3, 10, 0), (513, 1537, 3, 10, 6), (300, 2000, 16, 10, 0),
    (300, 2000, 16, 10, 3), (200, 900, 1, 4, 0), (100, 700, 5, 3, 0), (90, 1000, 50, 16, 2), (70, 300, 128, 32, 0),
    (64, 100, 8, 1, 0), (64, 100, 8, 1, 4), (50, 20, 2, 32, 0),   # K > N
    (300, 2000, 16, 32, 0), (200, 1500, 8, 32, 3), (300, 2000, 16, 16, 2), (250, 1800, 3, 32, 2),
    (260, 1700, 4, 16, 0),   # two rows a thread with 16- and 32-entry lists
]


@pytest.mark.parametrize("M,N,D,K,split", KNN_SMALL)
def test_knn_small(orc, M, N, D, K, split):
    x, y, _, _ = _case(M + 11 * N + D, M, N, D, 1)
    idx, dist = kr.kernel_knn(*_dev(x, y), K, split=split)
    i_ref, d_ref, n_ref = orc.knn(x, y, K)
    check_knn(_np(idx), _np(dist), x, y, i_ref, d_ref, n_ref, f"{M}x{N} D{D} K{K} S{split}")


def test_knn_ties_lowest_index(orc):
    """Integer grid points with many exact duplicates: ties must keep the lowest index."""
    r = _rng(5)
    y = r.integers(-3, 4, size=(3000, 3)).astype(np.float32)
    x = r.integers(-3, 4, size=(400, 3)).astype(np.float32)
    for split in (0, 1, 7):
        idx, dist = kr.kernel_knn(*_dev(x, y), 10, split=split)
        i_ref, d_ref, _ = orc.knn(x, y, 10)
        assert np.array_equal(_np(idx), i_ref), f"split {split}"   # integer distances are exact
        assert np.array_equal(_np(dist), d_ref.astype(np.float32))


def test_lse_far_rows_and_extreme_weights(orc):
    """Rows far from every point (all kernel values underflow in the tile frame),
    weights shifted by +-1000, and zero weights (log-weight -inf)."""
    r = _rng(6)
    y = r.standard_normal((2000, 3)).astype(np.float32)
    x = np.concatenate([r.standard_normal((200, 3)), 40 + r.standard_normal((100, 3))]).astype(np.float32)
    w = r.standard_normal((2000, 2)).astype(np.float32)
    for shift in (0.0, 1000.0, -1000.0):
        ws = (w + shift).astype(np.float32)
        L = kr.kernel_reduce(*_dev(x, y, ws), 0.5, "lse")
        check_lse(_np(L), orc.gauss_lse(x, y, ws, 0.5), f"shift {shift}")
    w2 = w.copy()
    w2[::3, 0] = -np.inf
    w2[:, 1] = -np.inf
    w2[1500:1600, 1] = 0.0
    L = kr.kernel_reduce(*_dev(x, y, w2), 0.8, "lse", split=3)
    check_lse(_np(L), orc.gauss_lse(x, y, w2, 0.8), "zero weights")


def test_empty_and_degenerate(orc):
    x, y, b, g = _case(9, 50, 0, 3, 2)
    xt, yt, bt, gt = _dev(x, y, b, g)
    assert (_np(kr.kernel_reduce(xt, yt, bt, 1.0, "sum")) == 0).all()
    assert np.isneginf(_np(kr.kernel_reduce(xt, yt, bt, 1.0, "lse"))).all()
    assert (_np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, 1.0)) == 0).all()
    idx, dist = kr.kernel_knn(xt, yt, 4)
    assert (_np(idx) == -1).all() and np.isinf(_np(dist)).all()
    e = torch.empty((0, 3), device=DEV)
    assert kr.kernel_reduce(e, yt, bt, 1.0).shape == (0, 2)
    # x_i = y_j, N = 1: a = b exactly (k = 2^0 = 1)
    p = _rng(1).standard_normal((1, 3)).astype(np.float32)
    bb = np.array([[1.25, -3.5]], dtype=np.float32)
    a = _np(kr.kernel_reduce(*_dev(p, p, bb), 0.7, "sum"))
    assert np.array_equal(a, bb)


def test_split_and_determinism(orc):
    x, y, b, g = _case(12, 3000, 20000, 3, 1)
    xt, yt, bt, gt = _dev(x, y, b, g)

    def run(split):
        return [_np(kr.kernel_reduce(xt, yt, bt, 0.6, "sum", split=split)),
                _np(kr.kernel_reduce(xt, yt, bt, 0.6, "lse", split=split)),
                _np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, 0.6, split=split)),
                _np(kr.kernel_knn(xt, yt, 10, split=split)[0])]

    outs = {}
    for split in (1, 9):
        outs[split] = run(split)
        for u, v in zip(outs[split], run(split)):
            assert np.array_equal(u, v), "run-to-run results differ"
    # K-min selection is unique under the (d, j) order, so the split does not change it
    assert np.array_equal(outs[1][3], outs[9][3])
    a_ref, S_ref = orc.gauss_sum(x[:300], y, b, 0.6)
    for split in (1, 9):
        check_sum(outs[split][0][:300], a_ref, S_ref, f"split {split}")


def test_host_buffers_match_device(orc):
    """CPU tensors go through the library's staging path and give the same bits."""
    x, y, b, g = _case(13, 1000, 5000, 3, 1)
    xt, yt, bt, gt = _dev(x, y, b, g)
    xc, yc, bc, gc = (torch.from_numpy(a) for a in (x, y, b, g))
    assert np.array_equal(kr.kernel_reduce(xc, yc, bc, 0.8, "sum").numpy(),
                          _np(kr.kernel_reduce(xt, yt, bt, 0.8, "sum")))
    assert np.array_equal(kr.kernel_reduce_grad_x(xc, yc, bc, gc, 0.8).numpy(),
                          _np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, 0.8)))
    pinned = [t.pin_memory() for t in (xc, yc)]
    i_host, d_host = kr.kernel_knn(*pinned, 5)
    i_dev, d_dev = kr.kernel_knn(xt, yt, 5)
    assert np.array_equal(i_host.numpy(), _np(i_dev)) and np.array_equal(d_host.numpy(), _np(d_dev))


def test_workspace_allocation_failure_leaves_output_untouched():
    x, y, b, _ = _case(14, 500, 4000, 3, 1)
    xt, yt, bt = _dev(x, y, b)
    out = torch.full((500, 1), 7.0, device=DEV)
    os.environ["KREDUCE_FAIL_ALLOC"] = "1"
    try:
        with pytest.raises(kr.KrError) as ei:
            kr.kernel_reduce(xt, yt, bt, 1.0, "sum", out=out, split=4)
        assert ei.value.status == kr.KR_ERR_ALLOC
    finally:
        del os.environ["KREDUCE_FAIL_ALLOC"]
    assert (_np(out) == 7.0).all()
    kr.kernel_reduce(xt, yt, bt, 1.0, "sum", out=out, split=4)   # works again
    assert not (_np(out) == 7.0).all()


def test_autograd_readme_example(orc):
    """KeOps README usage example: a = K.sum(dim=1), grad of sum(a^2) wrt x."""
    inp = W.generate("gauss_small")
    x = torch.from_numpy(inp["x"]).to(DEV).requires_grad_(True)
    y, b = _dev(inp["y"], inp["b"])
    a = kr.GaussianSum.apply(x, y, b, inp["sigma"])
    (gx,) = torch.autograd.grad((a ** 2).sum(), [x])
    a_ref, S_ref = orc.gauss_sum(inp["x"], inp["y"], inp["b"], inp["sigma"])
    check_sum(_np(a.detach()), a_ref, S_ref, "gauss_small")
    gx_ref, G_ref = orc.gauss_grad_x(inp["x"], inp["y"], inp["b"], 2 * _np(a.detach()), inp["sigma"])
    check_grad(_np(gx), gx_ref, G_ref, "gauss_small grad of sum(a^2)")


# ---------------------------------------------------------------------------
# full-size workloads: the GPU runs every row, the oracle a seeded subset
# ---------------------------------------------------------------------------
def test_workload_gauss_d3(orc):
    inp = W.generate("gauss_d3")
    s = inp["sigma"]
    xt, yt, bt, gt = _dev(inp["x"], inp["y"], inp["b"], inp["g"])
    a = _np(kr.kernel_reduce(xt, yt, bt, s, "sum"))
    gx = _np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, s))
    rows = W.row_subset(inp["x"].shape[0], 2048, 7)
    a_ref, S_ref = orc.gauss_sum(inp["x"][rows], inp["y"], inp["b"], s)
    check_sum(a[rows], a_ref, S_ref, "gauss_d3")
    gx_ref, G_ref = orc.gauss_grad_x(inp["x"][rows], inp["y"], inp["b"], inp["g"][rows], s)
    check_grad(gx[rows], gx_ref, G_ref, "gauss_d3")


def test_workload_gauss_d3_grad_of_sum_of_squares(orc):
    """The gradient the README differentiates, at the full M = N = 1e5: a = Sum, then the
    x-gradient of sum_i a_i^2, i.e. the upstream g = 2a (computed by the GPU for every
    row).  The oracle checks a and the gradient on 4096 seeded rows with the full N; its
    gradient takes the same upstream values the GPU used, so the gate is the kernel's."""
    inp = W.generate("gauss_d3")
    s = inp["sigma"]
    xt, yt, bt = _dev(inp["x"], inp["y"], inp["b"])
    a = kr.kernel_reduce(xt, yt, bt, s, "sum")
    gx = _np(kr.kernel_reduce_grad_x(xt, yt, bt, 2.0 * a, s))
    a = _np(a)
    rows = W.row_subset(inp["x"].shape[0], 4096, 11)
    a_ref, S_ref = orc.gauss_sum(inp["x"][rows], inp["y"], inp["b"], s)
    worst_sum = check_sum(a[rows], a_ref, S_ref, "gauss_d3 a")
    gx_ref, G_ref = orc.gauss_grad_x(inp["x"][rows], inp["y"], inp["b"], 2.0 * a[rows], s)
    worst_grad = check_grad(gx[rows], gx_ref, G_ref, "gauss_d3 grad of sum(a^2)")
    print(f"gauss_d3 grad of sum(a^2), {rows.size} rows: a err/S {worst_sum:.2e}, grad err/G {worst_grad:.2e}")


def test_workload_gauss_d3_unit(orc):
    inp = W.generate("gauss_d3_unit")
    s = inp["sigma"]
    xt, yt, bt, wt = _dev(inp["x"], inp["y"], inp["b"], inp["w_log"])
    a = _np(kr.kernel_reduce(xt, yt, bt, s, "sum"))
    L = _np(kr.kernel_reduce(xt, yt, wt, s, "lse"))
    # a seeded subset of 4096 rows with the full N = 1e6 (rows are independent)
    rows = W.row_subset(inp["x"].shape[0], 4096, 8)
    a_ref, S_ref = orc.gauss_sum(inp["x"][rows], inp["y"], inp["b"], s)
    worst_sum = check_sum(a[rows], a_ref, S_ref, "gauss_d3_unit")
    worst_lse = check_lse(L[rows], orc.gauss_lse(inp["x"][rows], inp["y"], inp["w_log"], s), "gauss_d3_unit")
    # LogSumExp of log b equals log of the Sum of b (b > 0)
    assert np.max(np.abs(L[rows] - np.log(a_ref))) < 1e-4
    print(f"gauss_d3_unit, {rows.size} rows: Sum err/S {worst_sum:.2e}, LSE abs err {worst_lse:.2e}")


def test_workload_falkon_d50(orc):
    inp = W.generate("falkon_d50")
    s = inp["sigma"]
    xt, yt, bt = _dev(inp["x"], inp["y"], inp["b"])
    a = _np(kr.kernel_reduce(xt, yt, bt, s, "sum"))
    p = kr.plan_device(kr.OP_SUM, inp["x"].shape[0], inp["y"].shape[0], 50, 1)
    assert p.split > 1, "the tall product must run in split-j mode"
    rows = W.row_subset(inp["x"].shape[0], 1000, 9)
    a_ref, S_ref = orc.gauss_sum(inp["x"][rows], inp["y"], inp["b"], s)
    check_sum(a[rows], a_ref, S_ref, "falkon_d50")
    # the LogSumExp of the same product (b as log-weights) on the tensor cores too
    assert kr.plan_device(kr.OP_LSE, inp["x"].shape[0], inp["y"].shape[0], 50, 1).path == kr.KR_PATH_TENSOR_CORES
    L = _np(kr.kernel_reduce(xt, yt, bt, s, "lse"))
    rows = W.row_subset(inp["x"].shape[0], 256, 10)
    check_lse(L[rows], orc.gauss_lse(inp["x"][rows], inp["y"], inp["b"], s), "falkon_d50 lse")
    # the x-gradient of the same product (g ~ N(0,1)) on the tensor cores
    assert kr.plan_device(kr.OP_GRAD, inp["x"].shape[0], inp["y"].shape[0], 50, 1).path == kr.KR_PATH_TENSOR_CORES
    gt = _dev(inp["g"])[0]
    gx = _np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, s))
    rows = W.row_subset(inp["x"].shape[0], 32, 12)   # the fp64 gradient costs ~1 s a row at N = 1e7
    gx_ref, G_ref = orc.gauss_grad_x(inp["x"][rows], inp["y"], inp["b"], inp["g"][rows], s)
    worst = check_grad(gx[rows], gx_ref, G_ref, "falkon_d50 grad")
    print(f"falkon_d50 grad, {rows.size} rows: err/G {worst:.2e}")
    # the K-min (K = 10) of the same clouds: the tensor-core screen, its splits chained
    # through the rows' shared lists
    assert kr.plan_device(kr.OP_KNN, inp["x"].shape[0], inp["y"].shape[0], 50, 10).path == kr.KR_PATH_TENSOR_CORES
    idx, dist = (_np(v) for v in kr.kernel_knn(xt, yt, 10))
    rows = W.row_subset(inp["x"].shape[0], 64, 13)
    i_ref, d_ref, n_ref = orc.knn(inp["x"][rows], inp["y"], 10)
    ties = check_knn(idx[rows], dist[rows], inp["x"][rows], inp["y"], i_ref, d_ref, n_ref, "falkon_d50 knn")
    print(f"falkon_d50 knn, {rows.size} rows: {ties} near-tie positions")


def test_workload_knn_d16(orc):
    inp = W.generate("knn_d16")
    xt, yt = _dev(inp["x"], inp["y"])
    idx, dist = kr.kernel_knn(xt, yt, inp["K"])
    # a seeded subset of 4096 rows with the full N = 1e6 (rows are independent)
    rows = W.row_subset(inp["x"].shape[0], 4096, 10)
    i_ref, d_ref, n_ref = orc.knn(inp["x"][rows], inp["y"], inp["K"])
    ties = check_knn(_np(idx)[rows], _np(dist)[rows], inp["x"][rows], inp["y"], i_ref, d_ref, n_ref, "knn_d16")
    print(f"knn_d16, {rows.size} rows: {ties} near-tie positions of {i_ref.size}")


# ---------------------------------------------------------------------------
# tensor-core Sum (tcgen05, split fp16 expansion): 32 <= D <= 62, E = 1
# ---------------------------------------------------------------------------
TC_CASES = [
    (1, 1, 32, 0.9, 0), (127, 129, 50, 1.0, 0), (300, 1000, 50, 1.0, 0), (300, 1000, 50, 1.0, 3),
    (513, 2000, 62, 1.3, 0), (256, 4096, 32, 0.8, 5), (1000, 300, 40, 1.1, 0),
    (130, 20001, 50, 1.0, 1),   # one split: 79 tiles per block (the gradient: 157), the rings wrap many times
]


@pytest.mark.parametrize("M,N,D,sigma,split", TC_CASES)
def test_tensor_core_sum(orc, M, N, D, sigma, split):
    r = _rng(M + N + D)
    x = (r.standard_normal((M, D)) / np.sqrt(D)).astype(np.float32)
    y = (r.standard_normal((N, D)) / np.sqrt(D)).astype(np.float32)
    b = r.standard_normal((N, 1)).astype(np.float32)
    assert kr.plan_device(kr.OP_SUM, M, N, D, 1).path == kr.KR_PATH_TENSOR_CORES
    a = kr.kernel_reduce(*_dev(x, y, b), sigma, "sum", split=split, path=kr.KR_PATH_TENSOR_CORES)
    a_ref, S_ref = orc.gauss_sum(x, y, b, sigma)
    check_sum(_np(a), a_ref, S_ref, f"tc {M}x{N} D{D} S{split}")


@pytest.mark.parametrize("M,N,D,sigma,split", TC_CASES + [(200, 3000, 61, 1.2, 2)])
def test_tensor_core_lse(orc, M, N, D, sigma, split):
    """The LogSumExp on the tensor cores (the weight relative to its tile's frame is one more
    operand slot, so D <= 61; D = 62 takes the CUDA cores), with weights spread over many
    orders of magnitude, some -inf (weight 0) and some so small that they leave the
    operand's range (clamped to 2^-1024 of the tile's largest)."""
    r = _rng(M + 3 * N + D)
    x = (r.standard_normal((M, D)) / np.sqrt(D)).astype(np.float32)
    y = (r.standard_normal((N, D)) / np.sqrt(D)).astype(np.float32)
    w = (4.0 * r.standard_normal((N, 1))).astype(np.float32)
    w[r.random((N, 1)) < 0.05] = -np.inf
    w[r.random((N, 1)) < 0.02] = -3000.0
    tc = D <= 61
    assert (kr.plan_device(kr.OP_LSE, M, N, D, 1).path == kr.KR_PATH_TENSOR_CORES) == tc
    L = kr.kernel_reduce(*_dev(x, y, w), sigma, "lse", split=split, path=kr.KR_PATH_TENSOR_CORES)
    check_lse(_np(L), orc.gauss_lse(x, y, w, sigma), f"tc lse {M}x{N} D{D} S{split}")


def test_tensor_core_lse_empty_weights_and_guard(orc):
    """All weights -inf gives -inf; large norms stand the tensor kernel down."""
    r = _rng(78)
    x = (r.standard_normal((300, 40)) / 6).astype(np.float32)
    y = (r.standard_normal((900, 40)) / 6).astype(np.float32)
    w = np.full((900, 1), -np.inf, np.float32)
    L = _np(kr.kernel_reduce(*_dev(x, y, w), 1.0, "lse", path=kr.KR_PATH_TENSOR_CORES))
    assert np.isneginf(L).all()
    x = (3.0 * r.standard_normal((200, 50))).astype(np.float32)
    y = (x[r.integers(0, 200, 700)] + 0.3 * r.standard_normal((700, 50))).astype(np.float32)
    w = r.standard_normal((700, 1)).astype(np.float32)
    L = kr.kernel_reduce(*_dev(x, y, w), 2.0, "lse", path=kr.KR_PATH_TENSOR_CORES)
    check_lse(_np(L), orc.gauss_lse(x, y, w, 2.0), "lse norm guard")


@pytest.mark.parametrize("op,split", [("sum", 0), ("sum", 2), ("lse", 0), ("lse", 3), ("grad", 0), ("grad", 2)])
def test_tensor_core_wait_bound_reports_status(orc, op, split):
    """Failure detection without a fault: with the B tiles withheld (a test hook that only
    the debug build honours) every bounded mbarrier wait of the tensor kernel runs out
    after 50 ms; the rows come out NaN (through the split-j combine too), the sticky device
    status says so, and the context stays usable."""
    r = _rng(79)
    x = (r.standard_normal((300, 50)) / np.sqrt(50)).astype(np.float32)
    y = (r.standard_normal((1000, 50)) / np.sqrt(50)).astype(np.float32)
    b = r.standard_normal((1000, 1)).astype(np.float32)
    g = r.standard_normal((300, 1)).astype(np.float32)
    xt, yt, bt, gt = _dev(x, y, b, g)

    def call():
        if op == "grad":
            return kr.kernel_reduce_grad_x(xt, yt, bt, gt, 1.0, split=split)
        return kr.kernel_reduce(xt, yt, bt, 1.0, op, split=split, path=kr.KR_PATH_TENSOR_CORES)

    release = kr.load_library()
    assert release.kr_set_tc_test_hooks(50, 1) == kr.KR_ERR_UNSUPPORTED
    debug = kr.load_debug_library()
    saved = kr._lib
    kr._lib = debug
    try:
        kr.device_status(clear=True)
        assert debug.kr_set_tc_test_hooks(50, 1) == kr.KR_OK
        try:
            a = _np(call())
        finally:
            assert debug.kr_set_tc_test_hooks(0, 0) == kr.KR_OK
        assert np.isnan(a).all()
        assert kr.device_status(clear=True) & 1
        assert kr.device_status() == 0
        a = _np(call())
        assert kr.device_status() == 0
    finally:
        kr._lib = saved
    if op == "sum":
        a_ref, S_ref = orc.gauss_sum(x, y, b, 1.0)
        check_sum(a, a_ref, S_ref, "after a run-out wait")
    elif op == "lse":
        check_lse(a, orc.gauss_lse(x, y, b, 1.0), "after a run-out wait")
    else:
        gx_ref, G_ref = orc.gauss_grad_x(x, y, b, g, 1.0)
        check_grad(a, gx_ref, G_ref, "after a run-out wait")


@pytest.mark.parametrize("M,N,D,sigma,split", TC_CASES + [
    (200, 3000, 61, 1.2, 2), (129, 257, 33, 0.7, 0),
    # one split of 5, 8 and 9 tiles of 128 points: the D2 groups of 4 tiles folded inside the
    # loop and after it in every combination
    (100, 513, 50, 1.0, 1), (100, 1024, 50, 1.0, 1), (100, 1025, 40, 1.0, 1)])
def test_tensor_core_grad(orc, M, N, D, sigma, split):
    """The x-gradient with both contractions on the tensor cores (S = A.B^T, then
    P.[y' | 1] with P = 2^S b split into fp16 hi + lo), against the oracle's gradient and
    its scale G; ragged row blocks and tiles, forced splits, D from 32 to 62."""
    r = _rng(M + 5 * N + D)
    x = (r.standard_normal((M, D)) / np.sqrt(D)).astype(np.float32)
    y = (r.standard_normal((N, D)) / np.sqrt(D)).astype(np.float32)
    b = r.standard_normal((N, 1)).astype(np.float32)
    g = r.standard_normal((M, 1)).astype(np.float32)
    assert kr.plan_device(kr.OP_GRAD, M, N, D, 1).path == kr.KR_PATH_TENSOR_CORES
    gx = kr.kernel_reduce_grad_x(*_dev(x, y, b, g), sigma, split=split)
    gx_ref, G_ref = orc.gauss_grad_x(x, y, b, g, sigma)
    check_grad(_np(gx), gx_ref, G_ref, f"tc grad {M}x{N} D{D} S{split}")


def test_tensor_core_grad_guard_and_agreement(orc):
    """Large norms (|x'|^2 + |y'|^2 > 16) stand the tensor kernel down and the CUDA-core
    gradient answers; on normal clouds the two paths agree within the tolerance and reruns
    give the same bits.  (The clouds here are independent, so no coordinate of x_i nearly
    equals that of all its neighbours: there fp32 coordinates, prescaled or expanded, lose
    the relative precision of the difference; that limit is described with the
    gradient's tolerance.)"""
    r = _rng(83)
    x = (3.0 * r.standard_normal((200, 50))).astype(np.float32)
    y = (3.0 * r.standard_normal((700, 50))).astype(np.float32)
    b = r.standard_normal((700, 1)).astype(np.float32)
    g = r.standard_normal((200, 1)).astype(np.float32)
    gx = kr.kernel_reduce_grad_x(*_dev(x, y, b, g), 8.0)
    gx_ref, G_ref = orc.gauss_grad_x(x, y, b, g, 8.0)
    check_grad(_np(gx), gx_ref, G_ref, "tc grad norm guard")
    inp = W.generate("falkon_d50", M=2000, N=50_000)
    gg = _rng(84).standard_normal((2000, 1)).astype(np.float32)
    xt, yt, bt, gt = _dev(inp["x"], inp["y"], inp["b"], gg)
    g_tc = _np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, 1.0))
    g_cc = _np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, 1.0, path=kr.KR_PATH_CUDA_CORES))
    rows = W.row_subset(2000, 200, 85)
    gx_ref, G_ref = orc.gauss_grad_x(inp["x"][rows], inp["y"], inp["b"], gg[rows], 1.0)
    check_grad(g_tc[rows], gx_ref, G_ref, "falkon-shaped tc grad")
    check_grad(g_cc[rows], gx_ref, G_ref, "falkon-shaped cuda-core grad")
    assert np.array_equal(g_tc, _np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, 1.0)))


@pytest.mark.parametrize("bscale,split", [(1.0, 0), (1e6, 3), (1e-8, 0), (3e4, 5)])
def test_tensor_core_grad_far_rows_and_signal_scale(orc, bscale, split):
    """The tensor-core gradient's P tile is fp16: the signal is scaled by a power of two into
    [-1, 1] (signals of 1e6 would overflow it, 1e-8 would vanish), and rows whose largest |P|
    in a split is below 2^-8 (here rows 2.2-3.0 units from a tight cloud, within the norm
    guard) are redone for that split by the CUDA-core kernel.  Every row must meet the
    oracle's tolerance."""
    r = _rng(91 + split)
    M, N, D = 300, 3000, 40
    y = (0.5 * r.standard_normal((N, D)) / np.sqrt(D)).astype(np.float32)
    x = (0.5 * r.standard_normal((M, D)) / np.sqrt(D)).astype(np.float32)
    u = r.standard_normal((M, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    far = np.arange(M) % 3 == 0
    x[far] = (u[far] * np.linspace(2.2, 3.0, far.sum())[:, None]).astype(np.float32)
    b = (bscale * r.standard_normal((N, 1))).astype(np.float32)
    g = r.standard_normal((M, 1)).astype(np.float32)
    assert kr.plan_device(kr.OP_GRAD, M, N, D, 1).path == kr.KR_PATH_TENSOR_CORES
    gx = kr.kernel_reduce_grad_x(*_dev(x, y, b, g), 1.0, split=split)
    gx_ref, G_ref = orc.gauss_grad_x(x, y, b, g, 1.0)
    check_grad(_np(gx), gx_ref, G_ref, f"tc grad far rows, b x {bscale}, S{split}")


def test_tensor_core_norm_guard_falls_back(orc):
    """Points far from the origin in units of sigma: the expansion would lose the
    tolerance, so the tensor kernel stands down and the CUDA-core kernel answers."""
    r = _rng(77)
    x = (3.0 * r.standard_normal((200, 50))).astype(np.float32)
    y = (x[r.integers(0, 200, 700)] + 0.3 * r.standard_normal((700, 50))).astype(np.float32)
    b = r.standard_normal((700, 1)).astype(np.float32)
    a = kr.kernel_reduce(*_dev(x, y, b), 2.0, "sum", path=kr.KR_PATH_TENSOR_CORES)
    a_ref, S_ref = orc.gauss_sum(x, y, b, 2.0)
    check_sum(_np(a), a_ref, S_ref, "norm guard")


def test_tensor_and_cuda_core_paths_agree():
    inp = W.generate("falkon_d50", M=2000, N=50_000)
    xt, yt, bt = _dev(inp["x"], inp["y"], inp["b"])
    a_tc = _np(kr.kernel_reduce(xt, yt, bt, 1.0, "sum", path=kr.KR_PATH_TENSOR_CORES))
    a_cc = _np(kr.kernel_reduce(xt, yt, bt, 1.0, "sum", path=kr.KR_PATH_CUDA_CORES))
    S = _np(kr.kernel_reduce(xt, yt, bt.abs(), 1.0, "sum", path=kr.KR_PATH_CUDA_CORES))
    assert (np.abs(a_tc - a_cc) <= 1e-4 * S).all()
    assert np.array_equal(a_tc, _np(kr.kernel_reduce(xt, yt, bt, 1.0, "sum", path=kr.KR_PATH_TENSOR_CORES)))
    L_tc = _np(kr.kernel_reduce(xt, yt, bt, 1.0, "lse", path=kr.KR_PATH_TENSOR_CORES))
    L_cc = _np(kr.kernel_reduce(xt, yt, bt, 1.0, "lse", path=kr.KR_PATH_CUDA_CORES))
    assert (np.abs(L_tc - L_cc) <= 2e-4).all()
    assert np.array_equal(L_tc, _np(kr.kernel_reduce(xt, yt, bt, 1.0, "lse", path=kr.KR_PATH_TENSOR_CORES)))


TC_KNN_CASES = [
    (1, 1, 32, 1, 0), (127, 300, 50, 10, 0), (300, 3000, 50, 10, 3), (513, 2000, 62, 32, 0),
    (256, 4096, 32, 4, 5), (1000, 257, 40, 16, 0),
    (130, 20001, 50, 10, 1),   # one split: 79 tiles a block
]


@pytest.mark.parametrize("M,N,D,K,split", TC_KNN_CASES)
def test_tensor_core_knn(orc, M, N, D, K, split):
    """K-min at 32 <= D <= 62 on the tensor cores: the product screens the points, passing
    ones get the direct fp32 distance; against the oracle (indices exact where separated),
    ragged row blocks and tiles, forced splits, K from 1 to 32."""
    r = _rng(M + 7 * N + D + K)
    x = (r.standard_normal((M, D)) / np.sqrt(D)).astype(np.float32)
    y = (r.standard_normal((N, D)) / np.sqrt(D)).astype(np.float32)
    assert kr.plan_device(kr.OP_KNN, M, N, D, K).path == kr.KR_PATH_TENSOR_CORES
    idx, dist = kr.kernel_knn(*_dev(x, y), K, split=split)
    i_ref, d_ref, n_ref = orc.knn(x, y, K)
    check_knn(_np(idx), _np(dist), x, y, i_ref, d_ref, n_ref, f"tc knn {M}x{N} D{D} K{K} S{split}")


def test_tensor_core_knn_ties_guard_and_agreement(orc):
    """Duplicated points (equal distances: the lowest index wins), clouds whose norms exceed
    the screen's limit (the CUDA-core kernel answers), and agreement with the CUDA-core K-min:
    the same indices wherever the distances are separated, distances within their rounding."""
    r = _rng(2024)
    x = (r.standard_normal((400, 50)) / 7).astype(np.float32)
    base = (r.standard_normal((60, 50)) / 7).astype(np.float32)
    y = base[r.integers(0, 60, size=3000)]
    for split in (0, 1, 4):
        idx, dist = kr.kernel_knn(*_dev(x, y), 10, split=split)
        i_ref, d_ref, n_ref = orc.knn(x, y, 10)
        check_knn(_np(idx), _np(dist), x, y, i_ref, d_ref, n_ref, f"tc knn ties S{split}")
    # norms far above the limit: |x|^2 + |y|^2 ~ 2 x 50 x 100^2
    xb, yb = (100.0 + r.standard_normal((300, 50))).astype(np.float32), (100.0 + r.standard_normal((2000, 50))).astype(np.float32)
    idx, dist = kr.kernel_knn(*_dev(xb, yb), 8)
    i_ref, d_ref, n_ref = orc.knn(xb, yb, 8)
    check_knn(_np(idx), _np(dist), xb, yb, i_ref, d_ref, n_ref, "tc knn guard")
    # tensor vs CUDA cores on the same clouds
    xc = (r.standard_normal((700, 62)) / 8).astype(np.float32)
    yc = (r.standard_normal((5000, 62)) / 8).astype(np.float32)
    it, dt = (_np(v) for v in kr.kernel_knn(*_dev(xc, yc), 16))
    ic, dc = (_np(v) for v in kr.kernel_knn(*_dev(xc, yc), 16, path=kr.KR_PATH_CUDA_CORES))
    i_ref, d_ref, n_ref = orc.knn(xc, yc, 16)
    check_knn(it, dt, xc, yc, i_ref, d_ref, n_ref, "tc knn vs oracle")
    check_knn(ic, dc, xc, yc, i_ref, d_ref, n_ref, "cuda knn vs oracle")
    assert np.allclose(dt, dc, rtol=1e-5, atol=0)


@pytest.mark.parametrize("scale", [1e-5, 1e-3, 5.5, 0.0])
def test_tensor_core_knn_scales(orc, scale):
    """The screen's margin at the ends of its range: clouds so small that their fp16 operands
    are subnormal (the margin's absolute part), clouds whose norms come near the limit of 4096
    (max |x|^2 + max |y|^2 about 3700), and (scale 0) coordinates of random sign spread
    log-uniformly over 1e-7 .. 1, every magnitude in between at once."""
    r = _rng(int(1e6 * scale) + 11)
    M, N, D, K = 300, 3000, 50, 8
    if scale > 0:
        x = (scale * r.standard_normal((M, D)) / 1.2).astype(np.float32)
        y = (scale * r.standard_normal((N, D)) / 1.2).astype(np.float32)
    else:
        def wide(n):
            return (np.sign(r.standard_normal((n, D))) * 10.0 ** r.uniform(-7, 0, (n, D))).astype(np.float32)
        x, y = wide(M), wide(N)
    assert kr.plan_device(kr.OP_KNN, M, N, D, K).path == kr.KR_PATH_TENSOR_CORES
    for split in (0, 3):
        idx, dist = kr.kernel_knn(*_dev(x, y), K, split=split)
        i_ref, d_ref, n_ref = orc.knn(x, y, K)
        check_knn(_np(idx), _np(dist), x, y, i_ref, d_ref, n_ref, f"tc knn scale {scale} S{split}")


@pytest.mark.parametrize("K,split", [(32, 8), (10, 0), (1, 5)])
def test_tensor_core_knn_shared_lists_ties(orc, K, split):
    """Every point duplicated hundreds of times across many splits: the splits' lists start
    from the row's shared list (stand-ins of other splits' distances), so exact ties between
    a stand-in and a point of the split decide which index is reported; the lowest must win."""
    r = _rng(77 + K + split)
    base = (r.standard_normal((50, 62)) / 8).astype(np.float32)
    y = base[r.integers(0, 50, size=40_000)]
    x = (base[r.integers(0, 50, size=600)] + 0.01 * r.standard_normal((600, 62))).astype(np.float32)
    idx, dist = kr.kernel_knn(*_dev(x, y), K, split=split)
    i_ref, d_ref, n_ref = orc.knn(x, y, K)
    check_knn(_np(idx), _np(dist), x, y, i_ref, d_ref, n_ref, f"tc knn shared-list ties K{K} S{split}")
    # the lowest index among the duplicates of the nearest centre, exactly
    near = np.argmin(((x[:, None, :].astype(np.float64) - base[None].astype(np.float64)) ** 2).sum(-1), axis=1)
    first = {c: int(np.flatnonzero((y == base[c]).all(1))[0]) for c in set(near.tolist())}
    assert all(int(_np(idx)[i, 0]) == first[near[i]] for i in range(600))
