"""The debug build (-DKR_DEBUG) on odd shapes: every global element index of the
CUDA-core kernels is checked against its array's extent (a violation is skipped and
reported through kr_device_status), so these runs show that no kernel indexes outside
its arrays on ragged, padded, split, batched and block-sparse problems, and that the
checked build computes exactly what the release build computes."""
import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from symbolic_matrix_reductions_gb300 import build
    build.build()
    release = kr.load_library()
    debug = kr.load_debug_library()
    assert debug.kr_debug_build() == 1 and release.kr_debug_build() == 0
    return release, debug


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _with(lib, fn):
    """Runs fn with the package's calls going to `lib`."""
    saved = kr._lib
    kr._lib = lib
    try:
        return [_np(t) for t in fn() if t is not None]
    finally:
        kr._lib = saved


CASES = [(1, 1, 3, 1), (33, 7, 3, 1), (513, 1537, 3, 1), (300, 1001, 5, 3), (129, 600, 16, 1), (150, 300, 20, 5),
         (100, 300, 50, 1), (40, 100, 70, 4), (40, 65, 128, 16), (700, 3000, 1, 1)]


@pytest.mark.parametrize("M,N,D,E", CASES)
def test_debug_build_finds_no_bad_index(libs, M, N, D, E):
    release, debug = libs
    r = np.random.Generator(np.random.PCG64(M + N + D))
    x, y, b, g = (torch.from_numpy(r.standard_normal(s).astype(np.float32)).to(DEV)
                  for s in ((M, D), (N, D), (N, E), (M, E)))
    K = min(10, max(1, N // 3))
    ri, si, rj = np.array([[0, M // 2], [M // 2 + (M > 2), M]]), np.array([2, 3]), np.array([[0, N // 2], [N // 3, N], [0, N]])
    calls = {
        "sum": lambda: [kr.kernel_reduce(x, y, b, 0.9, "sum")],
        "sum split": lambda: [kr.kernel_reduce(x, y, b, 0.9, "sum", split=3)],
        "lse": lambda: [kr.kernel_reduce(x, y, b, 0.9, "lse", split=2)],
        "grad-x": lambda: [kr.kernel_reduce_grad_x(x, y, b, g, 0.9, split=2)],
        "grad-y": lambda: [kr.kernel_reduce_grad_y(x, y, b, g, 0.9)],
        "grad-b": lambda: [kr.kernel_reduce_grad_b(x, y, g, 0.9, path=kr.KR_PATH_CUDA_CORES)],
        "knn": lambda: list(kr.kernel_knn(x, y, K)),
        "knn split": lambda: list(kr.kernel_knn(x, y, K, split=3)),
        "cauchy max": lambda: list(kr.kernel_reduce_arg(x, y, b, 0.9, "max", split=2, kernel="cauchy")),
        "laplace sum": lambda: [kr.kernel_reduce(x, y, b, 0.9, "sum", kernel="laplace")],
        "ranges sum": lambda: [kr.kernel_reduce_ranges(x, y, b, 0.9, "sum", ri, si, rj)],
        "ranges min": lambda: list(kr.kernel_reduce_ranges(x, y, b, 0.9, "min", ri, si, rj, want_index=True)),
        "batched": lambda: [kr.kernel_reduce(torch.stack([x, x.flip(0)]), torch.stack([y, y]), torch.stack([b, b]),
                                             0.9, "sum", path=kr.KR_PATH_CUDA_CORES)],
        "noalloc sum": lambda: [kr.kernel_reduce_noalloc(x, y, b, 0.9, "sum", out=torch.empty((M, E), device=DEV))],
        "noalloc lse": lambda: [kr.kernel_reduce_noalloc(x, y, b, 0.9, "lse", out=torch.empty((M, E), device=DEV))],
    }
    kr.device_status(clear=True)
    for name, fn in calls.items():
        want = _with(release, fn)
        got = _with(debug, fn)
        st = ctypes_status(debug)
        assert st == 0, f"{name}: index check bits {st >> 8:#x}"
        for w_, g_ in zip(want, got):
            assert np.array_equal(w_, g_, equal_nan=True), name


def ctypes_status(lib):
    import ctypes
    v = ctypes.c_uint(0)
    assert lib.kr_device_status(ctypes.byref(v), 1) == kr.KR_OK
    return v.value
