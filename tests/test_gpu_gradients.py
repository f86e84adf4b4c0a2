"""y- and b-gradients of the Sum (the transposed product) vs the fp64 oracle,
through the C ABI, and the autograd wrapper that uses all three gradients.

Tolerances are those of the x-gradient and the Sum: |gy_gpu - gy| <= 1e-4 G with
G_jd = (2/sigma^2) sum_i k_ij |g_i . b_j| |x_id - y_jd|, and |gb_gpu - gb| <= 1e-4 S
with S_je = sum_i |k_ij g_ie|.
"""
import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr
from symbolic_matrix_reductions_gb300 import workloads as W

from parity import check_grad, check_sum

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
    g = r.standard_normal((M, E)).astype(np.float32)
    return x, y, b, g


# (M, N, D, E, sigma, split): the output has N rows here, so the ragged tails are
# on N (the rows of gy and gb) and the reduction runs over M.
CASES = [
    (1, 1, 3, 1, 1.0, 0), (7, 33, 3, 1, 0.7, 0), (1537, 513, 3, 1, 0.5, 0), (2049, 1100, 3, 1, 0.9, 5),
    (3000, 700, 1, 1, 0.3, 0), (1000, 257, 2, 2, 1.5, 3), (777, 300, 4, 3, 1.0, 0), (600, 129, 16, 1, 2.0, 2),
    (300, 150, 20, 5, 2.5, 0), (257, 100, 50, 1, 3.0, 0), (300, 100, 50, 1, 3.0, 4), (65, 40, 128, 16, 6.0, 2),
]


@pytest.mark.parametrize("M,N,D,E,sigma,split", CASES)
def test_grad_y_small(orc, M, N, D, E, sigma, split):
    x, y, b, g = _case(M + 13 * N + D, M, N, D, E)
    gy = kr.kernel_reduce_grad_y(*_dev(x, y, b, g), sigma, split=split)
    gy_ref, G_ref = orc.gauss_grad_y(x, y, b, g, sigma)
    check_grad(_np(gy), gy_ref, G_ref, f"grad-y {M}x{N} D{D} E{E} S{split}")


@pytest.mark.parametrize("M,N,D,E,sigma,split", CASES)
def test_grad_b_small(orc, M, N, D, E, sigma, split):
    x, y, _, g = _case(M + 17 * N + D, M, N, D, E)
    gb = kr.kernel_reduce_grad_b(*_dev(x, y, g), sigma, split=split)
    gb_ref, S_ref = orc.gauss_grad_b(x, y, g, sigma)
    check_sum(_np(gb), gb_ref, S_ref, f"grad-b {M}x{N} D{D} E{E} S{split}")


def test_grad_b_tensor_cores(orc):
    """D = 50, E = 1: the transposed product takes the tcgen05 path like the Sum."""
    x, y, _, g = _case(99, 3000, 700, 50, 1)
    x *= np.float32(1 / np.sqrt(50))
    y *= np.float32(1 / np.sqrt(50))
    p = kr.plan_device(kr.OP_SUM, 700, 3000, 50, 1)
    assert p.path == kr.KR_PATH_TENSOR_CORES
    gb = kr.kernel_reduce_grad_b(*_dev(x, y, g), 1.0)
    gb_ref, S_ref = orc.gauss_grad_b(x, y, g, 1.0)
    check_sum(_np(gb), gb_ref, S_ref, "grad-b tensor cores")


def test_grad_y_host_buffers(orc):
    """Host (CPU) tensors are staged by the library and give the same result."""
    x, y, b, g = _case(5, 500, 300, 3, 2)
    xt, yt, bt, gt = (torch.from_numpy(a) for a in (x, y, b, g))
    gy_h = kr.kernel_reduce_grad_y(xt, yt, bt, gt, 0.8).numpy()
    gy_d = _np(kr.kernel_reduce_grad_y(*_dev(x, y, b, g), 0.8))
    assert np.array_equal(gy_h, gy_d)


def test_autograd_all_inputs(orc):
    """GaussianSum differentiates L = sum(a^2) wrt x, y and b (the README example,
    extended to every input)."""
    inp = W.generate("gauss_small")
    s = inp["sigma"]
    x, y, b = (torch.from_numpy(inp[k]).to(DEV).requires_grad_(True) for k in ("x", "y", "b"))
    a = kr.GaussianSum.apply(x, y, b, s)
    gx, gy, gb = torch.autograd.grad((a ** 2).sum(), [x, y, b])
    g = 2 * _np(a.detach())
    gx_ref, G_ref = orc.gauss_grad_x(inp["x"], inp["y"], inp["b"], g, s)
    check_grad(_np(gx), gx_ref, G_ref, "autograd x")
    gy_ref, Gy_ref = orc.gauss_grad_y(inp["x"], inp["y"], inp["b"], g, s)
    check_grad(_np(gy), gy_ref, Gy_ref, "autograd y")
    gb_ref, Sb_ref = orc.gauss_grad_b(inp["x"], inp["y"], g, s)
    check_sum(_np(gb), gb_ref, Sb_ref, "autograd b")
    assert gb.shape == b.shape


def test_workload_gauss_d3_gradients(orc):
    """The gauss_d3 batch (M = N = 1e5) at full size on the GPU; a seeded subset of
    the output rows j against the oracle with the full reduction over i."""
    inp = W.generate("gauss_d3")
    s = inp["sigma"]
    xt, yt, bt, gt = _dev(inp["x"], inp["y"], inp["b"], inp["g"])
    gy = _np(kr.kernel_reduce_grad_y(xt, yt, bt, gt, s))
    gb = _np(kr.kernel_reduce_grad_b(xt, yt, gt, s))
    rows = W.row_subset(inp["y"].shape[0], 1024, 11)
    gy_ref, G_ref = orc.gauss_grad_y(inp["x"], inp["y"][rows], inp["b"][rows], inp["g"], s)
    check_grad(gy[rows], gy_ref, G_ref, "gauss_d3 grad-y")
    gb_ref, S_ref = orc.gauss_grad_b(inp["x"], inp["y"][rows], inp["g"], s)
    check_sum(gb[rows], gb_ref, S_ref, "gauss_d3 grad-b")
