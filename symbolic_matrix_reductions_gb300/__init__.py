"""kreduce for one GB300: reductions over symbolic Gaussian / squared-distance matrices.

The compute lives in ``libkreduce.so`` (CUDA for sm_103a, built from ``csrc/`` by
``build.py``); this package only marshals arguments to its C ABI through
``ctypes`` (which releases the interpreter lock around each call, so several
Python threads can run reductions at once).  There is no CPU fallback: if the
library is missing, every call raises.

Functions, named after the C entry points (see ``include/kreduce.h``):

* ``kernel_reduce(x, y, b, sigma, reduction="sum"|"lse"|"max"|"min", out=None, split=0,
  kernel="gaussian"|"laplace"|"cauchy"|"imq")``
* ``kernel_reduce_arg(x, y, b, sigma, reduction="max"|"min", idx=None, out=None, split=0, kernel=...)``
* ``kernel_reduce_ranges(x, y, b, sigma, "sum"|"max"|"min", ranges_i, slices_i, redranges_j, ...)``
* ``kernel_reduce_grad_x(x, y, b, g, sigma, out=None, split=0)``
* ``kernel_reduce_grad_y(x, y, b, g, sigma, out=None, split=0)``
* ``kernel_reduce_grad_b(x, y, g, sigma, out=None, split=0)``
* ``kernel_knn(x, y, K, idx=None, dist=None, split=0)``

Arguments are float32 torch tensors, contiguous, row-major: x (M, D), y (N, D),
b (N, E) or (N,), g (M, E) or (M,).  CUDA tensors run asynchronously on the
current stream; CPU tensors are staged through device memory by the library and
the call blocks until the result is back.  ``GaussianSum`` wraps the Sum with its
x-, y- and b-gradients as a ``torch.autograd.Function``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import workloads  # noqa: F401  (seeded inputs; no compute)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkreduce.so")

KR_SUM, KR_LSE, KR_MAX, KR_MIN = 0, 1, 2, 3
KERNELS = {"gaussian": 0, "laplace": 1, "cauchy": 2, "imq": 3}  # kr_options.kernel
KR_OK, KR_ERR_INVALID, KR_ERR_UNSUPPORTED, KR_ERR_ALLOC, KR_ERR_CUDA = 0, 1, 2, 3, 4
OP_SUM, OP_LSE, OP_GRAD, OP_KNN, OP_MAX = 0, 1, 2, 3, 4

# Names exported by libkreduce.so, in the order include/kreduce.h declares them.
EXPORTS = ("kernel_reduce", "kernel_reduce_ex", "kernel_reduce_arg", "kernel_reduce_arg_ex",
           "kernel_reduce_ranges", "kernel_reduce_noalloc", "kernel_reduce_grad_x",
           "kernel_reduce_grad_x_ex", "kernel_reduce_grad_y", "kernel_reduce_grad_y_ex",
           "kernel_reduce_grad_b", "kernel_reduce_grad_b_ex",
           "kernel_knn", "kernel_knn_ex", "kr_status_string", "kr_last_cuda_error", "kr_device_status",
           "kr_set_tc_test_hooks", "kr_debug_build", "kr_plan", "kr_plan_device")


class KrError(RuntimeError):
    """A kreduce call returned a status other than KR_OK."""

    def __init__(self, status: int, what: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{what}: {_status_text(status)} (status {status})"
        if status == KR_ERR_CUDA:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


class KrOptions(ctypes.Structure):
    _fields_ = [("split", ctypes.c_int), ("path", ctypes.c_int), ("kernel", ctypes.c_int),
                ("batch", ctypes.c_int), ("reserved", ctypes.c_int * 4)]


KR_PATH_AUTO, KR_PATH_CUDA_CORES, KR_PATH_TENSOR_CORES = 0, 1, 2


class KrPlan(ctypes.Structure):
    _fields_ = [("d_pad", ctypes.c_int), ("ek_pad", ctypes.c_int), ("rows_per_thread", ctypes.c_int),
                ("threads", ctypes.c_int), ("tile_points", ctypes.c_int), ("row_blocks", ctypes.c_int64),
                ("split", ctypes.c_int), ("chunk", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("path", ctypes.c_int)]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libkreduce.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libkreduce.so not found at {path}; build it with "
                "`python -m symbolic_matrix_reductions_gb300.build` (there is no CPU fallback)")
        _lib = _configure(ctypes.CDLL(path))
        return _lib


def load_debug_library() -> ctypes.CDLL:
    """Builds (if needed) and loads libkreduce_debug.so, the variant whose kernels check
    every global element index (test infrastructure; see kr_debug_build in the header).
    It is a separate handle: the module's functions keep using the release library."""
    from . import build
    return _configure(ctypes.CDLL(build.build_debug()))


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declares the C signatures on a loaded library."""
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    opt = ctypes.POINTER(KrOptions)
    lib.kernel_reduce.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp]
    lib.kernel_reduce_ex.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp, opt]
    lib.kernel_reduce_arg.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp]
    lib.kernel_reduce_arg_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp, opt]
    lib.kernel_reduce_ranges.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, i64, vp, vp, i64, vp,
                                         vp, opt]
    lib.kernel_reduce_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp]
    lib.kernel_reduce_grad_x.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, vp]
    lib.kernel_reduce_grad_x_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, vp, opt]
    lib.kernel_reduce_grad_y.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, vp]
    lib.kernel_reduce_grad_y_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, vp, opt]
    lib.kernel_reduce_grad_b.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, f32, vp]
    lib.kernel_reduce_grad_b_ex.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, f32, vp, opt]
    lib.kernel_knn.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, vp]
    lib.kernel_knn_ex.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, vp, opt]
    lib.kr_status_string.argtypes = [i32]
    lib.kr_status_string.restype = ctypes.c_char_p
    lib.kr_last_cuda_error.argtypes = []
    lib.kr_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
    lib.kr_set_tc_test_hooks.argtypes = [i32, i32]
    lib.kr_debug_build.argtypes = []
    lib.kr_plan.argtypes = [i32, i64, i64, i32, i32, i32, i32, opt, ctypes.POINTER(KrPlan)]
    lib.kr_plan_device.argtypes = [i32, i64, i64, i32, i32, opt, ctypes.POINTER(KrPlan)]
    for name in EXPORTS:
        if name != "kr_status_string":
            getattr(lib, name).restype = ctypes.c_int
    return lib


def _status_text(status: int) -> str:
    try:
        return load_library().kr_status_string(int(status)).decode()
    except Exception:  # library missing: keep the error readable
        return "status"


def _check(status: int, what: str) -> None:
    if status != KR_OK:
        cuda_err = load_library().kr_last_cuda_error() if status == KR_ERR_CUDA else 0
        raise KrError(status, what, cuda_err)


def device_status(clear: bool = False) -> int:
    """The sticky device status of the current device (bit 0: a tensor-core wait gave
    up and its rows came out NaN); waits for the device's work."""
    v = ctypes.c_uint(0)
    _check(load_library().kr_device_status(ctypes.byref(v), 1 if clear else 0), "kr_device_status")
    return int(v.value)


def _kernel_code(kernel) -> int:
    if isinstance(kernel, str):
        if kernel not in KERNELS:
            raise ValueError(f"kernel must be one of {sorted(KERNELS)}, got {kernel!r}")
        return KERNELS[kernel]
    return int(kernel)


def _options(split: int, path: int = 0, kernel=0, batch: int = 0):
    kernel = _kernel_code(kernel)
    if not split and not path and not kernel and batch <= 1:
        return None
    o = KrOptions()
    o.split = int(split)
    o.path = int(path)
    o.kernel = kernel
    o.batch = int(batch) if batch > 1 else 0
    return ctypes.byref(o)


def plan(op: int, M: int, N: int, D: int, EK: int, num_sms: int = 152, blocks_per_sm: int = 0,
         split: int = 0, path: int = 0, kernel=0) -> KrPlan:
    """The launch plan the library would use (host logic only, no GPU needed)."""
    p = KrPlan()
    _check(load_library().kr_plan(op, M, N, D, EK, num_sms, blocks_per_sm, _options(split, path, kernel),
                                  ctypes.byref(p)), "kr_plan")
    return p


def plan_device(op: int, M: int, N: int, D: int, EK: int, split: int = 0, path: int = 0, kernel=0) -> KrPlan:
    """The launch plan a call makes on the current CUDA device (queries the device)."""
    p = KrPlan()
    _check(load_library().kr_plan_device(op, M, N, D, EK, _options(split, path, kernel), ctypes.byref(p)),
           "kr_plan_device")
    return p


# ---------------------------------------------------------------------------
# tensor marshalling
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _mat(t, rows, name, cols=None, B=0):
    """t as a contiguous float32 (rows, cols) matrix, or (B, rows, cols) when B > 0; a
    missing last dimension (a vector per problem) is taken as one column."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    lead = (B,) if B else ()
    if t.dim() == len(lead) + 1:
        t = t.view(*t.shape, 1)
    if (t.dim() != len(lead) + 2 or tuple(t.shape[:len(lead)]) != lead
            or (rows is not None and t.shape[-2] != rows) or (cols is not None and t.shape[-1] != cols)):
        raise ValueError(f"{name}: bad shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _batch_of(x):
    """B for a batched call (x of shape (B, M, D)), 0 for a single problem (x (M, D))."""
    torch = _torch()
    if not isinstance(x, torch.Tensor):
        raise TypeError("x must be a torch.Tensor")
    if x.dim() == 3:
        if x.shape[0] < 1:
            raise ValueError("x: empty batch dimension")
        return int(x.shape[0])
    return 0


def _empty(B, rows, cols, dtype, dev):
    torch = _torch()
    return torch.empty(((B,) if B else ()) + (rows, cols), dtype=dtype, device=dev)


def _same_device(*ts):
    devs = {t.device for t in ts if t is not None}
    if len(devs) > 1:
        raise ValueError(f"tensors on different devices: {devs}")
    return devs.pop()


def _stream(device):
    torch = _torch()
    if device.type == "cuda":
        return torch.cuda.current_stream(device).cuda_stream
    return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else None


def _clouds(x, y):
    """(B, x, y, M, N, D) for a single problem (B = 0) or a batch of B problems."""
    B = _batch_of(x)
    x = _mat(x, None, "x", B=B)
    M, D = x.shape[-2:]
    y = _mat(y, None, "y", D, B=B)
    return B, x, y, M, y.shape[-2], D


def kernel_reduce(x, y, b, sigma: float, reduction: str = "sum", out=None, split: int = 0, path: int = 0,
                  kernel="gaussian"):
    """Sum (``"sum"``), LogSumExp (``"lse"``; b holds log-weights), Max or Min over j.

    Returns ``out`` (M, E): a_ie = sum_j k_ij b_je, L_ie = log sum_j exp(-|x_i-y_j|^2/sigma^2
    + b_je), or max_j / min_j k_ij b_je.  ``kernel``: "gaussian" (default), "laplace",
    "cauchy" or "imq" (Sum, Max and Min).  With x (B, M, D), y (B, N, D), b (B, N, E) the
    call reduces B independent problems and returns (B, M, E)."""
    red = {"sum": KR_SUM, "lse": KR_LSE, "max": KR_MAX, "min": KR_MIN}.get(reduction)
    if red is None:
        raise ValueError(f"reduction must be 'sum', 'lse', 'max' or 'min', got {reduction!r}")
    B, x, y, M, N, D = _clouds(x, y)
    b = _mat(b, N, "b", B=B)
    E = b.shape[-1]
    dev = _same_device(x, y, b)
    if out is None:
        out = _empty(B, M, E, x.dtype, dev)
    out2 = _mat(out, M, "out", E, B=B)
    _same_device(x, out2)
    st = load_library().kernel_reduce_ex(_ptr(x), _ptr(y), _ptr(b), _ptr(out2), M, N, D, E, float(sigma), red,
                                         _stream(dev), _options(split, path, kernel, B))
    _check(st, "kernel_reduce")
    return out


def kernel_reduce_arg(x, y, b, sigma: float, reduction: str = "max", idx=None, out=None, want_values: bool = True,
                      split: int = 0, kernel="gaussian"):
    """ArgMax / ArgMin of k_ij b_je over j (lowest index on ties) with the extreme value.

    Returns (idx int32 (M, E), values float32 (M, E) or None); (B, M, E) for a batch."""
    torch = _torch()
    red = {"max": KR_MAX, "min": KR_MIN}.get(reduction)
    if red is None:
        raise ValueError(f"reduction must be 'max' or 'min', got {reduction!r}")
    B, x, y, M, N, D = _clouds(x, y)
    b = _mat(b, N, "b", B=B)
    E = b.shape[-1]
    dev = _same_device(x, y, b)
    if idx is None:
        idx = _empty(B, M, E, torch.int32, dev)
    if out is None and want_values:
        out = _empty(B, M, E, torch.float32, dev)
    want = ((B,) if B else ()) + (M, E)
    if idx.dtype != torch.int32 or tuple(idx.shape) != want or not idx.is_contiguous():
        raise ValueError(f"idx must be a contiguous int32 tensor of shape {want}")
    if out is not None:
        out = _mat(out, M, "out", E, B=B)
    _same_device(x, idx, out)
    st = load_library().kernel_reduce_arg_ex(_ptr(x), _ptr(y), _ptr(b), _ptr(out), _ptr(idx), M, N, D, E,
                                             float(sigma), red, _stream(dev), _options(split, 0, kernel, B))
    _check(st, "kernel_reduce_arg")
    return idx, out


def kernel_reduce_ranges(x, y, b, sigma: float, reduction: str, ranges_i, slices_i, redranges_j, out=None,
                         idx=None, want_index: bool = False, kernel="gaussian"):
    """Block-sparse Sum / Max / Min: the rows of cluster c (ranges_i[c] = [start, end))
    reduce only over the column ranges redranges_j[slices_i[c-1]:slices_i[c]].

    ranges_i (nc, 2), slices_i (nc,), redranges_j (nr, 2): integer arrays on the host
    (NumPy or CPU tensors).  Returns ``out`` for "sum"; (idx, out) for "max" / "min" when
    ``want_index`` (else ``out``)."""
    import numpy as np
    torch = _torch()
    red = {"sum": KR_SUM, "max": KR_MAX, "min": KR_MIN}.get(reduction)
    if red is None:
        raise ValueError(f"reduction must be 'sum', 'max' or 'min', got {reduction!r}")
    B, x, y, M, N, D = _clouds(x, y)
    if B:
        raise ValueError("the block-sparse mode takes one problem (2-D x and y)")
    b = _mat(b, N, "b")
    E = b.shape[-1]
    dev = _same_device(x, y, b)
    tabs = []
    for name, arr, cols in (("ranges_i", ranges_i, 2), ("slices_i", slices_i, 1), ("redranges_j", redranges_j, 2)):
        if isinstance(arr, torch.Tensor):
            arr = arr.detach().cpu().numpy()
        a = np.ascontiguousarray(np.asarray(arr, dtype=np.int64))
        if (cols == 2 and a.size and (a.ndim != 2 or a.shape[1] != 2)) or (cols == 1 and a.ndim > 1):
            raise ValueError(f"{name}: bad shape {a.shape}")
        tabs.append(a.reshape(-1, cols) if cols == 2 else a.reshape(-1))
    ri, si, rj = tabs
    if out is None:
        out = _empty(0, M, E, torch.float32, dev)
    out = _mat(out, M, "out", E)
    if red != KR_SUM and want_index and idx is None:
        idx = _empty(0, M, E, torch.int32, dev)
    if idx is not None and (idx.dtype != torch.int32 or tuple(idx.shape) != (M, E) or not idx.is_contiguous()):
        raise ValueError("idx must be a contiguous int32 tensor of shape (M, E)")
    _same_device(x, out, idx)
    p64 = lambda a: ctypes.c_void_p(a.ctypes.data) if a.size else None
    st = load_library().kernel_reduce_ranges(_ptr(x), _ptr(y), _ptr(b), _ptr(out), _ptr(idx), M, N, D, E,
                                             float(sigma), red, ri.shape[0], p64(ri), p64(si), rj.shape[0], p64(rj),
                                             _stream(dev), _options(0, 0, kernel))
    _check(st, "kernel_reduce_ranges")
    return (idx, out) if (red != KR_SUM and want_index) else out


def kernel_reduce_noalloc(x, y, b, sigma: float, reduction: str, out):
    """kernel_reduce for callers that cannot allocate device memory at call time.

    The library allocates nothing: the split partials live in its 16 MiB static
    device array.  x, y, b and the caller's ``out`` (M, E) must be CUDA tensors;
    M * E may not exceed 1048576.  Calls that overlap on the GPU race on the shared
    array.  Returns ``out``."""
    red = {"sum": KR_SUM, "lse": KR_LSE}.get(reduction)
    if red is None:
        raise ValueError(f"reduction must be 'sum' or 'lse', got {reduction!r}")
    x = _mat(x, None, "x")
    M, D = x.shape
    y = _mat(y, None, "y", D)
    N = y.shape[0]
    b = _mat(b, N, "b")
    E = b.shape[1]
    out2 = _mat(out, M, "out", E)
    dev = _same_device(x, y, b, out2)
    st = load_library().kernel_reduce_noalloc(_ptr(x), _ptr(y), _ptr(b), _ptr(out2), M, N, D, E, float(sigma),
                                              red, _stream(dev))
    _check(st, "kernel_reduce_noalloc")
    return out


def kernel_reduce_grad_x(x, y, b, g, sigma: float, out=None, split: int = 0, path: int = 0):
    """Gradient wrt x of sum_ie g_ie a_ie (a the Sum reduction); returns (M, D) or (B, M, D).
    path: KR_PATH_AUTO (tensor cores for 32 <= D <= 62, E = 1) or KR_PATH_CUDA_CORES."""
    B, x, y, M, N, D = _clouds(x, y)
    b = _mat(b, N, "b", B=B)
    E = b.shape[-1]
    g = _mat(g, M, "g", E, B=B)
    dev = _same_device(x, y, b, g)
    if out is None:
        out = _empty(B, M, D, x.dtype, dev)
    out = _mat(out, M, "out", D, B=B)
    _same_device(x, out)
    st = load_library().kernel_reduce_grad_x_ex(_ptr(x), _ptr(y), _ptr(b), _ptr(g), _ptr(out), M, N, D, E,
                                                float(sigma), _stream(dev), _options(split, path, batch=B))
    _check(st, "kernel_reduce_grad_x")
    return out


def kernel_reduce_grad_y(x, y, b, g, sigma: float, out=None, split: int = 0):
    """Gradient wrt y of sum_ie g_ie a_ie (a the Sum reduction); returns (N, D) or (B, N, D)."""
    B, x, y, M, N, D = _clouds(x, y)
    b = _mat(b, N, "b", B=B)
    E = b.shape[-1]
    g = _mat(g, M, "g", E, B=B)
    dev = _same_device(x, y, b, g)
    if out is None:
        out = _empty(B, N, D, x.dtype, dev)
    out = _mat(out, N, "out", D, B=B)
    _same_device(x, out)
    st = load_library().kernel_reduce_grad_y_ex(_ptr(x), _ptr(y), _ptr(b), _ptr(g), _ptr(out), M, N, D, E,
                                                float(sigma), _stream(dev), _options(split, batch=B))
    _check(st, "kernel_reduce_grad_y")
    return out


def kernel_reduce_grad_b(x, y, g, sigma: float, out=None, split: int = 0, path: int = 0, kernel="gaussian"):
    """Gradient wrt b of sum_ie g_ie a_ie: gb_je = sum_i k_ij g_ie; returns (N, E) or (B, N, E)."""
    B, x, y, M, N, D = _clouds(x, y)
    g = _mat(g, M, "g", B=B)
    E = g.shape[-1]
    dev = _same_device(x, y, g)
    if out is None:
        out = _empty(B, N, E, x.dtype, dev)
    out2 = _mat(out, N, "out", E, B=B)
    _same_device(x, out2)
    st = load_library().kernel_reduce_grad_b_ex(_ptr(x), _ptr(y), _ptr(g), _ptr(out2), M, N, D, E, float(sigma),
                                                _stream(dev), _options(split, path, kernel, B))
    _check(st, "kernel_reduce_grad_b")
    return out


def kernel_knn(x, y, K: int, idx=None, dist=None, want_dist: bool = True, split: int = 0, path: int = 0):
    """K smallest (|x_i-y_j|^2, j) per row, ascending, lowest index on ties.  ``path``:
    KR_PATH_AUTO (default; the tensor-core screen at 32 <= D <= 62, K <= 32) or
    KR_PATH_CUDA_CORES.

    Returns (idx int32 (M, K), dist float32 (M, K) or None); (B, M, K) for a batch."""
    torch = _torch()
    B, x, y, M, N, D = _clouds(x, y)
    dev = _same_device(x, y)
    K = int(K)
    if idx is None:
        idx = _empty(B, M, K, torch.int32, dev)
    if dist is None and want_dist:
        dist = _empty(B, M, K, torch.float32, dev)
    want = ((B,) if B else ()) + (M, K)
    if idx.dtype != torch.int32 or tuple(idx.shape) != want or not idx.is_contiguous():
        raise ValueError(f"idx must be a contiguous int32 tensor of shape {want}")
    if dist is not None:
        dist = _mat(dist, M, "dist", K, B=B)
    _same_device(x, idx, dist)
    st = load_library().kernel_knn_ex(_ptr(x), _ptr(y), _ptr(idx), _ptr(dist), M, N, D, K, _stream(dev),
                                      _options(split, path, batch=B))
    _check(st, "kernel_knn")
    return idx, dist


def _make_gaussian_sum():
    torch = _torch()

    class GaussianSum(torch.autograd.Function):
        """a = sum_j exp(-|x_i-y_j|^2/sigma^2) b_j, differentiable wrt x, y and b.

        The backward pass runs the library's x-gradient, y-gradient and transposed
        product (b-gradient) kernels for the inputs that need a gradient.  Batched
        inputs (x (B, M, D), ...) are differentiated problem by problem."""

        @staticmethod
        def forward(ctx, x, y, b, sigma):
            ctx.save_for_backward(x, y, b)
            ctx.sigma = float(sigma)
            ctx.b_shape = b.shape
            return kernel_reduce(x.detach(), y.detach(), b.detach(), sigma, "sum")

        @staticmethod
        def backward(ctx, grad_out):
            x, y, b = ctx.saved_tensors
            xd, yd, bd = x.detach(), y.detach(), b.detach().contiguous()
            g = grad_out.contiguous()
            gx = gy = gb = None
            if ctx.needs_input_grad[0]:
                gx = kernel_reduce_grad_x(xd, yd, bd, g, ctx.sigma)
            if ctx.needs_input_grad[1]:
                gy = kernel_reduce_grad_y(xd, yd, bd, g, ctx.sigma)
            if ctx.needs_input_grad[2]:
                gb = kernel_reduce_grad_b(xd, yd, g, ctx.sigma).view(ctx.b_shape)
            return gx, gy, gb, None

    return GaussianSum


def __getattr__(name):
    if name == "GaussianSum":
        cls = _make_gaussian_sum()
        globals()["GaussianSum"] = cls
        return cls
    raise AttributeError(name)
