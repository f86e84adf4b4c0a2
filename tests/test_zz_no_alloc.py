"""kernel_reduce_noalloc: the reduction for callers that cannot allocate device memory
when they call (their own arena already holds the GPU's memory, or they must not
wait on the driver's allocator).  The entry point keeps its split partials in the
library's 16 MiB static device array; these tests call it through the C ABI, twice
in a row on different inputs, and compare it with kernel_reduce, which takes its
workspace from the allocator.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr

from parity import LSE_ATOL, LSE_RTOL, SUM_RTOL

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


def test_noalloc_matches_kernel_reduce_on_two_calls_in_a_row(lib):
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
