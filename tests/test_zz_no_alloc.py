"""kernel_reduce_noalloc: the reduction for callers that cannot allocate device memory
when they call (their own arena already holds the GPU's memory, or they must not
wait on the driver's allocator).  The entry point keeps its split partials in the
library's 16 MiB static device array.  These tests call it through the C ABI and
through the Python wrapper, twice in a row, and compare it with kernel_reduce (which
takes its workspace from the allocator) and with the fp64 oracle on seeded row
subsets.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr

from parity import LSE_ATOL, LSE_RTOL, SUM_RTOL, check_lse, check_sum

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from symbolic_matrix_reductions_gb300 import build
    build.build()
    return kr.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, y, b, out, sigma, red):
    M, D = x.shape
    N, E = b.shape
    st = lib.kernel_reduce_noalloc(_p(x), _p(y), _p(b), _p(out), M, N, D, E, sigma, red,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st


def _agree(got, want, scale, red):
    got, want = got.cpu().double().numpy(), want.cpu().double().numpy()
    if red == kr.KR_SUM:
        assert (np.abs(got - want) <= SUM_RTOL * scale.cpu().double().numpy() + 1e-30).all()
    else:
        both = np.isneginf(got) & np.isneginf(want)
        with np.errstate(invalid="ignore"):
            err = np.where(both, 0.0, np.abs(got - want))
        assert (err <= LSE_ATOL + LSE_RTOL * np.where(np.isfinite(want), np.abs(want), 0.0)).all()


def test_noalloc_matches_kernel_reduce_on_two_calls_in_a_row(lib, orc):
    r = np.random.Generator(np.random.PCG64(21))
    M, N, D = 3000, 200_000, 3
    x = torch.from_numpy(r.standard_normal((M, D), dtype=np.float32)).cuda()
    y = torch.from_numpy(r.standard_normal((N, D), dtype=np.float32)).cuda()
    # the call is split over j, so the static partials are really used
    assert kr.plan_device(kr.OP_SUM, M, N, D, 1).split > 1
    cases = [(kr.KR_SUM, 1, 0.7), (kr.KR_SUM, 2, 1.3), (kr.KR_LSE, 1, 0.7), (kr.KR_LSE, 3, 0.4)]
    for red, E, sigma in cases:   # consecutive calls reuse (and overwrite) the shared array
        b = torch.from_numpy(r.standard_normal((N, E), dtype=np.float32)).cuda()
        out = torch.full((M, E), float("nan"), device="cuda")
        assert _noalloc(lib, x, y, b, out, sigma, red) == kr.KR_OK
        name = "sum" if red == kr.KR_SUM else "lse"
        ref = kr.kernel_reduce(x, y, b, sigma, name)
        got, want = out.cpu().double().numpy(), ref.cpu().double().numpy()
        if red == kr.KR_SUM:
            scale = kr.kernel_reduce(x, y, b.abs(), sigma, "sum").cpu().double().numpy()   # sum_j |k b|
            assert (np.abs(got - want) <= SUM_RTOL * scale + 1e-30).all()
        else:
            assert (np.abs(got - want) <= LSE_ATOL + LSE_RTOL * np.abs(want)).all()
        # and against the fp64 oracle on a seeded row subset with the full N
        rows = np.sort(r.choice(M, size=128, replace=False))
        xs, yn, bn = x.cpu().numpy()[rows], y.cpu().numpy(), b.cpu().numpy()
        if red == kr.KR_SUM:
            a_ref, S_ref = orc.gauss_sum(xs, yn, bn, sigma)
            check_sum(got[rows], a_ref, S_ref, f"noalloc sum E{E}")
        else:
            check_lse(got[rows], orc.gauss_lse(xs, yn, bn, sigma), f"noalloc lse E{E}")


@pytest.mark.parametrize("M,N,D,E,red", [
    (1_048_576, 3000, 3, 1, kr.KR_SUM),    # M * E at the limit: the scratch holds exactly two splits
    (524_288, 2000, 3, 2, kr.KR_LSE),      # the same limit with two columns
    (700, 0, 3, 2, kr.KR_SUM),             # N = 0: Sum 0
    (700, 0, 3, 2, kr.KR_LSE),             # N = 0: LogSumExp -inf
    (700, 1, 3, 1, kr.KR_SUM),             # N = 1: one split, no partials
    (700, 1, 3, 1, kr.KR_LSE),
    (300, 20_000, 50, 1, kr.KR_SUM),       # D = 50 (the CUDA-core kernel: this entry point has no tensor path)
    (300, 20_000, 50, 1, kr.KR_LSE),
])
def test_noalloc_edges_through_the_python_wrapper(lib, orc, M, N, D, E, red):
    r = np.random.Generator(np.random.PCG64(M + N + D + E))
    scale = 1.0 / np.sqrt(D)
    x = torch.from_numpy((r.standard_normal((M, D)) * scale).astype(np.float32)).cuda()
    y = torch.from_numpy((r.standard_normal((N, D)) * scale).astype(np.float32)).cuda()
    b = torch.from_numpy(r.standard_normal((N, E)).astype(np.float32)).cuda()
    name = "sum" if red == kr.KR_SUM else "lse"
    for _ in range(2):   # two calls in a row on the shared array
        out = torch.full((M, E), float("nan"), device="cuda")
        assert kr.kernel_reduce_noalloc(x, y, b, 0.8, name, out=out) is out
        torch.cuda.synchronize()
        want = kr.kernel_reduce(x, y, b, 0.8, name)
        _agree(out, want, kr.kernel_reduce(x, y, b.abs(), 0.8, "sum"), red)
    if N == 0:
        o = out.cpu().numpy()
        assert (o == 0).all() if red == kr.KR_SUM else np.isneginf(o).all()
        return
    rows = np.sort(r.choice(M, size=min(M, 96), replace=False))
    xs, yn, bn, got = x.cpu().numpy()[rows], y.cpu().numpy(), b.cpu().numpy(), out.cpu().numpy()[rows]
    if red == kr.KR_SUM:
        a_ref, S_ref = orc.gauss_sum(xs, yn, bn, 0.8)
        check_sum(got, a_ref, S_ref, f"noalloc {M}x{N} D{D}")
    else:
        check_lse(got, orc.gauss_lse(xs, yn, bn, 0.8), f"noalloc lse {M}x{N} D{D}")


def test_noalloc_rejects_what_it_cannot_serve(lib):
    y = torch.zeros((100, 3), device="cuda")
    b = torch.zeros((100, 1), device="cuda")
    # beyond the scratch: M * E > 1048576
    xb = torch.zeros((1_048_577, 3), device="cuda")
    ob = torch.zeros((1_048_577, 1), device="cuda")
    assert _noalloc(lib, xb, y, b, ob, 1.0, kr.KR_SUM) == kr.KR_ERR_UNSUPPORTED
    # host arrays would need staging memory
    xh = torch.zeros((10, 3))
    oh = torch.zeros((10, 1))
    assert _noalloc(lib, xh, y, b, oh, 1.0, kr.KR_SUM) == kr.KR_ERR_INVALID
