"""The C ABI without a GPU: the library loads, exports every function the header
declares, rejects bad arguments before any CUDA call, and plans launches with
pure host logic."""
import ctypes
import os
import re

import pytest

import symbolic_matrix_reductions_gb300 as kr
from symbolic_matrix_reductions_gb300 import build as kbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kreduce.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kr.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("kernel_reduce", "kernel_reduce_grad_x", "kernel_knn", "kr_status_string"):
        assert n in names
    assert tuple(names) == kr.EXPORTS


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_alone(tmp_path, lang, std):
    """The public header is self-contained C99 and C++17: it compiles with no other include
    and no warning under -Wall -Wextra -pedantic."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text('#include "kreduce.h"\nint main(void) { return (int)sizeof(kr_options) == 0; }\n')
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", os.path.dirname(HEADER), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_device_status_without_a_device(lib):
    v = ctypes.c_uint(7)
    assert lib.kr_device_status(None, 0) == kr.KR_ERR_INVALID
    if not lib.kernel_reduce:  # pragma: no cover
        return
    import torch
    if not torch.cuda.is_available():
        # no driver entry point here: no tensor-core kernel can have run
        assert lib.kr_device_status(ctypes.byref(v), 1) == kr.KR_OK and v.value == 0


def test_tc_test_hooks_release_has_no_fault_path(lib):
    """The release library refuses the starvation hook (only the debug build carries it);
    the wait bound itself may be set and reset.  No CUDA call is made."""
    assert lib.kr_debug_build() == 0
    assert lib.kr_set_tc_test_hooks(50, 1) == kr.KR_ERR_UNSUPPORTED
    assert lib.kr_set_tc_test_hooks(-1, 0) == kr.KR_ERR_INVALID
    assert lib.kr_set_tc_test_hooks(50, 2) == kr.KR_ERR_INVALID
    assert lib.kr_set_tc_test_hooks(50, 0) == kr.KR_OK
    assert lib.kr_set_tc_test_hooks(0, 0) == kr.KR_OK


def test_status_strings(lib):
    texts = {lib.kr_status_string(s).decode() for s in range(5)}
    assert len(texts) == 5
    assert lib.kr_status_string(99).decode() == "unknown status"


P = ctypes.c_void_p
FAKE = [P(0x10000 * (k + 1)) for k in range(8)]  # never dereferenced: validation fails first


def _reduce(lib, x=FAKE[0], y=FAKE[1], b=FAKE[2], out=FAKE[3], M=10, N=10, D=3, E=1, sigma=1.0, red=0,
            opt=None):
    return lib.kernel_reduce_ex(x, y, b, out, M, N, D, E, sigma, red, None, opt)


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), kr.KR_ERR_INVALID),
    (dict(N=-5), kr.KR_ERR_INVALID),
    (dict(D=0), kr.KR_ERR_INVALID),
    (dict(E=0), kr.KR_ERR_INVALID),
    (dict(sigma=0.0), kr.KR_ERR_INVALID),
    (dict(sigma=-1.0), kr.KR_ERR_INVALID),
    (dict(sigma=float("nan")), kr.KR_ERR_INVALID),
    (dict(sigma=float("inf")), kr.KR_ERR_INVALID),
    (dict(red=4), kr.KR_ERR_INVALID),
    (dict(red=-1), kr.KR_ERR_INVALID),
    (dict(x=None), kr.KR_ERR_INVALID),
    (dict(y=None), kr.KR_ERR_INVALID),
    (dict(b=None), kr.KR_ERR_INVALID),
    (dict(out=None), kr.KR_ERR_INVALID),
    (dict(D=129), kr.KR_ERR_UNSUPPORTED),
    (dict(E=17), kr.KR_ERR_UNSUPPORTED),
    (dict(M=1 << 59, D=3), kr.KR_ERR_UNSUPPORTED),      # M*D > 2^60 elements
    (dict(N=1 << 31, D=3), kr.KR_ERR_UNSUPPORTED),      # indices are int32
    (dict(out=P(0x10000 + 8)), kr.KR_ERR_INVALID),      # output overlaps x
    (dict(M=0, out=None, x=None), kr.KR_OK),            # M = 0 is a no-op, no device needed
])
def test_reduce_validation(lib, kw, status):
    assert _reduce(lib, **kw) == status


def test_options_validation(lib):
    o = kr.KrOptions()
    o.split = -1
    assert _reduce(lib, opt=ctypes.byref(o)) == kr.KR_ERR_INVALID
    o.split = 0
    o.path = 3
    assert _reduce(lib, opt=ctypes.byref(o)) == kr.KR_ERR_INVALID
    o.path = 0
    o.split = 0
    o.reserved[3] = 1
    assert _reduce(lib, opt=ctypes.byref(o)) == kr.KR_ERR_INVALID


def test_grad_and_knn_validation(lib):
    g = lib.kernel_reduce_grad_x_ex
    assert g(FAKE[0], FAKE[1], FAKE[2], None, FAKE[4], 10, 10, 3, 1, 1.0, None, None) == kr.KR_ERR_INVALID
    assert g(FAKE[0], FAKE[1], FAKE[2], FAKE[3], FAKE[4], 10, 10, 3, 1, 0.0, None, None) == kr.KR_ERR_INVALID
    assert g(FAKE[0], FAKE[1], FAKE[2], FAKE[3], FAKE[4], 10, 10, 200, 1, 1.0, None, None) == kr.KR_ERR_UNSUPPORTED
    k = lib.kernel_knn_ex
    assert k(FAKE[0], FAKE[1], FAKE[2], None, 10, 10, 3, 0, None, None) == kr.KR_ERR_INVALID
    assert k(FAKE[0], FAKE[1], FAKE[2], None, 10, 10, 3, 33, None, None) == kr.KR_ERR_UNSUPPORTED
    assert k(FAKE[0], FAKE[1], None, None, 10, 10, 3, 4, None, None) == kr.KR_ERR_INVALID
    # idx and dist may not overlap
    assert k(FAKE[0], FAKE[1], FAKE[2], P(0x30000 + 4), 10, 10, 3, 4, None, None) == kr.KR_ERR_INVALID
    assert k(None, None, None, None, 0, 0, 3, 4, None, None) == kr.KR_OK


def test_kernel_option_validation(lib):
    o = kr.KrOptions()
    for kern in range(4):
        o.kernel = kern
        # valid kinds pass validation for the Sum and Max/Min (then fail on the fake pointers
        # only when a device is used: here the request is rejected earlier for a bad width)
        assert _reduce(lib, sigma=0.0, opt=ctypes.byref(o)) == kr.KR_ERR_INVALID
        assert _reduce(lib, red=kr.KR_MAX, D=200, opt=ctypes.byref(o)) == kr.KR_ERR_UNSUPPORTED
    for bad in (-1, 4):
        o.kernel = bad
        assert _reduce(lib, opt=ctypes.byref(o)) == kr.KR_ERR_INVALID
    o.kernel = kr.KERNELS["laplace"]
    # the LogSumExp, gradients and K-min are Gaussian / distance only
    assert _reduce(lib, red=kr.KR_LSE, opt=ctypes.byref(o)) == kr.KR_ERR_UNSUPPORTED
    g = lib.kernel_reduce_grad_x_ex
    assert g(*FAKE[:5], 10, 10, 3, 1, 1.0, None, ctypes.byref(o)) == kr.KR_ERR_UNSUPPORTED
    assert lib.kernel_reduce_grad_y_ex(*FAKE[:5], 10, 10, 3, 1, 1.0, None, ctypes.byref(o)) == kr.KR_ERR_UNSUPPORTED
    assert lib.kernel_knn_ex(*FAKE[:4], 10, 10, 3, 4, None, ctypes.byref(o)) == kr.KR_ERR_UNSUPPORTED
    o.kernel = 0
    o.reserved[3] = 7
    assert _reduce(lib, opt=ctypes.byref(o)) == kr.KR_ERR_INVALID


def test_batch_option(lib):
    o = kr.KrOptions()
    o.batch = -1
    assert _reduce(lib, opt=ctypes.byref(o)) == kr.KR_ERR_INVALID
    o.batch = 65536
    assert _reduce(lib, opt=ctypes.byref(o)) == kr.KR_ERR_UNSUPPORTED
    # a batch of problems needs fewer splits to fill the GPU, and its workspace is B times larger
    one = kr.plan(kr.OP_SUM, 2000, 100_000, 3, 1, num_sms=152, blocks_per_sm=8)
    o.batch = 64
    many = kr.KrPlan()
    assert lib.kr_plan(kr.OP_SUM, 2000, 100_000, 3, 1, 152, 8, ctypes.byref(o), ctypes.byref(many)) == kr.KR_OK
    assert many.split < one.split
    parts = 64 * (2 * many.split * 2000 * 4 if many.split > 1 else 0)
    assert many.workspace_bytes == parts   # batched calls stage their own tiles: no records
    assert many.chunk % many.tile_points == 0   # but split on whole tiles like a single call
    # batched tensor-core-sized Sums plan on the CUDA cores
    tc = kr.KrPlan()
    assert lib.kr_plan(kr.OP_SUM, 2000, 100_000, 50, 1, 152, 1, ctypes.byref(o), ctypes.byref(tc)) == kr.KR_OK
    assert tc.path == kr.KR_PATH_CUDA_CORES


def test_ranges_validation(lib):
    I64 = ctypes.c_int64 * 64
    f = lib.kernel_reduce_ranges

    def call(red=kr.KR_SUM, out=FAKE[3], idx=None, M=10, N=20, ri=(0, 5, 5, 10), si=(1, 2), rj=(0, 10, 10, 20),
             opt=None, nc=None, nr=None):
        a_ri, a_si, a_rj = I64(*ri), I64(*si), I64(*rj)
        return f(FAKE[0], FAKE[1], FAKE[2], out, idx, M, N, 3, 1, 1.0, red,
                 len(si) if nc is None else nc, a_ri, a_si, len(rj) // 2 if nr is None else nr, a_rj, None, opt)

    assert call(red=kr.KR_LSE) == kr.KR_ERR_INVALID
    assert call(ri=(0, 6, 5, 10)) == kr.KR_ERR_INVALID          # overlapping clusters
    assert call(ri=(5, 10, 0, 6)) == kr.KR_ERR_INVALID          # ... in any order
    assert call(ri=(0, 5, 5, 11)) == kr.KR_ERR_INVALID          # past M
    assert call(ri=(3, 2, 5, 10)) == kr.KR_ERR_INVALID          # end before start
    assert call(si=(2, 1)) == kr.KR_ERR_INVALID                 # decreasing slices
    assert call(si=(1, 3)) == kr.KR_ERR_INVALID                 # past the last range
    assert call(rj=(0, 10, 10, 21)) == kr.KR_ERR_INVALID        # past N
    assert call(rj=(-1, 10, 10, 20)) == kr.KR_ERR_INVALID
    assert call(idx=FAKE[4]) == kr.KR_ERR_INVALID               # the Sum has no index
    assert call(red=kr.KR_MAX, out=None, idx=None) == kr.KR_ERR_INVALID
    assert f(FAKE[0], FAKE[1], FAKE[2], FAKE[3], None, 10, 20, 3, 1, 1.0, kr.KR_SUM, 2, None, None, 0, None,
             None, None) == kr.KR_ERR_INVALID                   # missing tables
    o = kr.KrOptions()
    o.split = 2
    assert call(opt=ctypes.byref(o)) == kr.KR_ERR_UNSUPPORTED
    o.split, o.batch = 0, 2
    assert call(opt=ctypes.byref(o)) == kr.KR_ERR_UNSUPPORTED
    assert call(M=0, ri=(0, 0), si=(0,), rj=(), out=None) == kr.KR_OK


def test_arg_validation(lib):
    f = lib.kernel_reduce_arg_ex
    # x, y, b, out (nullable), idx
    assert f(*FAKE[:3], None, None, 10, 10, 3, 1, 1.0, kr.KR_MAX, None, None) == kr.KR_ERR_INVALID   # idx missing
    assert f(*FAKE[:5], 10, 10, 3, 1, 1.0, kr.KR_SUM, None, None) == kr.KR_ERR_INVALID             # not Max/Min
    assert f(*FAKE[:5], 10, 10, 3, 1, 1.0, kr.KR_LSE, None, None) == kr.KR_ERR_INVALID
    assert f(*FAKE[:5], 10, 10, 3, 1, -1.0, kr.KR_MIN, None, None) == kr.KR_ERR_INVALID
    assert f(*FAKE[:5], 10, 10, 3, 17, 1.0, kr.KR_MIN, None, None) == kr.KR_ERR_UNSUPPORTED
    # idx (10 x 1 int32) overlapping out
    assert f(*FAKE[:4], P(0x40000 + 8), 10, 10, 3, 1, 1.0, kr.KR_MAX, None, None) == kr.KR_ERR_INVALID
    assert f(None, FAKE[1], FAKE[2], None, None, 0, 10, 3, 1, 1.0, kr.KR_MAX, None, None) == kr.KR_OK
    # kernel_reduce with Max needs out
    assert _reduce(lib, out=None, red=kr.KR_MAX) == kr.KR_ERR_INVALID


def test_maxmin_plan(lib):
    """Max/Min plans like the Sum (same rows and tiles), never on the tensor cores, and
    keeps (value, index) partials per split."""
    for D in (3, 50):
        ps = kr.plan(kr.OP_SUM, 100_000, 10_000_000, D, 1, num_sms=152, blocks_per_sm=4, path=kr.KR_PATH_CUDA_CORES)
        pm = kr.plan(kr.OP_MAX, 100_000, 10_000_000, D, 1, num_sms=152, blocks_per_sm=4)
        assert pm.path == kr.KR_PATH_CUDA_CORES
        assert (pm.rows_per_thread, pm.tile_points, pm.d_pad) == (ps.rows_per_thread, ps.tile_points, ps.d_pad)
        assert pm.split > 1 and pm.workspace_bytes == pm.split * 100_000 * 8
    # other kernels never take the tensor-core path
    assert kr.plan(kr.OP_SUM, 1000, 1000, 50, 1, kernel="laplace").path == kr.KR_PATH_CUDA_CORES
    assert kr.plan(kr.OP_SUM, 1000, 1000, 50, 1, kernel="gaussian").path == kr.KR_PATH_TENSOR_CORES


def test_grad_y_and_grad_b_validation(lib):
    gy = lib.kernel_reduce_grad_y_ex
    # argument order: x, y, b, g, gy -- each pointer checked
    for k in range(5):
        ptrs = list(FAKE[:5])
        ptrs[k] = None
        assert gy(*ptrs, 10, 20, 3, 1, 1.0, None, None) == kr.KR_ERR_INVALID, k
    assert gy(*FAKE[:5], 10, 20, 3, 1, -2.0, None, None) == kr.KR_ERR_INVALID
    assert gy(*FAKE[:5], 10, 20, 3, 17, 1.0, None, None) == kr.KR_ERR_UNSUPPORTED
    # gy (N x D) overlapping y
    assert gy(FAKE[0], FAKE[1], FAKE[2], FAKE[3], P(0x20000 + 4), 10, 20, 3, 1, 1.0, None, None) == kr.KR_ERR_INVALID
    assert gy(None, None, None, None, None, 5, 0, 3, 1, 1.0, None, None) == kr.KR_ERR_INVALID  # x missing, M > 0
    assert gy(None, None, None, None, None, 0, 0, 3, 1, 1.0, None, None) == kr.KR_OK
    gb = lib.kernel_reduce_grad_b_ex
    for k in range(4):
        ptrs = list(FAKE[:4])
        ptrs[k] = None
        assert gb(*ptrs, 10, 20, 3, 2, 1.0, None, None) == kr.KR_ERR_INVALID, k
    assert gb(*FAKE[:4], 10, 20, 3, 2, float("nan"), None, None) == kr.KR_ERR_INVALID
    assert gb(*FAKE[:4], 10, 20, 129, 2, 1.0, None, None) == kr.KR_ERR_UNSUPPORTED
    # N = 0: nothing to write (the transposed product has no rows)
    assert gb(FAKE[0], None, FAKE[2], None, 10, 0, 3, 2, 1.0, None, None) == kr.KR_OK


# ---------------------------------------------------------------------------
# planner (pure host logic)
# ---------------------------------------------------------------------------
def test_instance_choice(lib):
    p = kr.plan(kr.OP_SUM, 1000, 1000, 3, 1)
    assert (p.d_pad, p.ek_pad, p.threads) == (3, 1, 128)
    assert kr.plan(kr.OP_SUM, 10, 10, 5, 2).d_pad == 8 and kr.plan(kr.OP_SUM, 10, 10, 5, 2).ek_pad == 4
    assert kr.plan(kr.OP_SUM, 10, 10, 50, 1, path=kr.KR_PATH_CUDA_CORES).d_pad == 50
    assert kr.plan(kr.OP_LSE, 10, 10, 50, 1, path=kr.KR_PATH_CUDA_CORES).d_pad == 50
    assert kr.plan(kr.OP_SUM, 10, 10, 51, 16).d_pad == 64
    assert kr.plan(kr.OP_KNN, 10, 10, 16, 10).ek_pad == 10
    assert kr.plan(kr.OP_KNN, 10, 10, 16, 11).ek_pad == 16
    assert kr.plan(kr.OP_KNN, 10, 10, 16, 1).ek_pad == 1


@pytest.mark.parametrize("D,K,rows,tile", [
    (3, 10, 4, 1024), (3, 1, 4, 1024), (4, 10, 4, 512), (3, 16, 2, 1024), (3, 32, 2, 1024),
    (8, 10, 4, 512), (8, 16, 2, 512), (16, 10, 4, 256), (16, 32, 2, 256), (50, 10, 1, 128), (128, 10, 1, 64),
])
def test_knn_instances(lib, D, K, rows, tile):
    """K-min instances: the screened kernel (D <= 16) keeps both record arrays of a tile within
    36 KB (1024 points at D <= 3, 512 at D = 4, 8, 256 at D = 16) and four rows a thread for K <= 10
    (two for longer lists); the direct kernels above D = 16 one row."""
    p = kr.plan(kr.OP_KNN, 100_000, 100_000, D, K, path=kr.KR_PATH_CUDA_CORES)
    assert (p.rows_per_thread, p.tile_points) == (rows, tile)
    assert p.row_blocks == (100_000 + 128 * rows - 1) // (128 * rows)


def test_knn_tensor_core_plan(lib):
    """K-min at 32 <= D <= 62 with K <= 32 plans the tensor-core screen: 256 rows a block,
    128-point tiles, the list padded as on the CUDA cores, split lists of KP (distance, index)
    and the rows' shared lists in the workspace; other D, longer lists and batches stay
    on the CUDA cores."""
    p = kr.plan(kr.OP_KNN, 100_000, 1_000_000, 50, 10, num_sms=152, blocks_per_sm=1)
    assert p.path == kr.KR_PATH_TENSOR_CORES and (p.tile_points, p.threads, p.ek_pad) == (128, 320, 10)
    assert p.row_blocks == (100_000 + 255) // 256 and p.chunk % 128 == 0
    # operands as for the Sum (x padded to whole blocks of 256 rows), S x M lists of 10
    # (distance, index), one shared list of 10 distances a row
    n_pad = (1_000_000 + 255) // 256 * 256
    ops = ((100_000 + 255) // 256 * 256 + n_pad) * 256 + n_pad * 4 + (n_pad // 256 * 4 + 255) // 256 * 256
    lists = 2 * p.split * 100_000 * 10 * 4 if p.split > 1 else 0
    assert p.workspace_bytes == 256 + ops + lists + (4 * 100_000 * 10 + 255) // 256 * 256
    # any shape, automatic or forced splits: whole 128-point tiles, every split nonempty, the
    # same workspace formula (the list width padded as on the CUDA cores: K 32 -> 32)
    for M, N, D, K, forced in ((1, 1, 50, 1, 0), (300, 3000, 50, 10, 0), (300, 3000, 50, 10, 7),
                               (513, 2000, 62, 32, 0), (100_000, 10_000_000, 50, 10, 0)):
        q = kr.plan(kr.OP_KNN, M, N, D, K, num_sms=152, blocks_per_sm=1, split=forced)
        assert q.path == kr.KR_PATH_TENSOR_CORES and q.chunk % 128 == 0
        assert (q.split - 1) * q.chunk < N <= q.split * q.chunk
        assert q.row_blocks == (M + 255) // 256
        n_pad = (N + 255) // 256 * 256
        ops = ((M + 255) // 256 * 256 + n_pad) * 256 + n_pad * 4 + (n_pad // 256 * 4 + 255) // 256 * 256
        lists = 2 * q.split * M * q.ek_pad * 4 if q.split > 1 else 0
        assert q.workspace_bytes == 256 + ops + lists + (4 * M * q.ek_pad + 255) // 256 * 256, (M, N, K)
    for D in (32, 62):
        assert kr.plan(kr.OP_KNN, 1000, 5000, D, 4).path == kr.KR_PATH_TENSOR_CORES
    assert kr.plan(kr.OP_KNN, 1000, 5000, 50, 32).ek_pad == 32
    for D, K in ((16, 10), (31, 10), (63, 10)):
        assert kr.plan(kr.OP_KNN, 1000, 5000, D, K).path == kr.KR_PATH_CUDA_CORES, (D, K)
    assert kr.plan(kr.OP_KNN, 1000, 5000, 50, 10, path=kr.KR_PATH_CUDA_CORES).path == kr.KR_PATH_CUDA_CORES


@pytest.mark.parametrize("op,M,N,D,EK", [
    (kr.OP_SUM, 100_000, 100_000, 3, 1),
    (kr.OP_LSE, 1_000_000, 1_000_000, 3, 1),
    (kr.OP_SUM, 100_000, 10_000_000, 50, 1),
    (kr.OP_KNN, 1_000_000, 1_000_000, 16, 10),
    (kr.OP_GRAD, 1000, 1000, 3, 1),
    (kr.OP_SUM, 7, 3, 3, 1),
    (kr.OP_SUM, 5, 0, 3, 1),
])
def test_split_covers_all_columns(lib, op, M, N, D, EK):
    p = kr.plan(op, M, N, D, EK, num_sms=152, blocks_per_sm=8)
    assert 1 <= p.split <= 64
    assert p.split * p.chunk >= N
    assert N == 0 or (p.split - 1) * p.chunk < N      # no empty split
    # tensor-core blocks: 256 threads over 128 rows (two column halves per row)
    bm = 128 if p.path == kr.KR_PATH_TENSOR_CORES else p.threads * p.rows_per_thread
    assert p.row_blocks == (M + bm - 1) // bm
    if p.split == 1:
        streamed = p.path == kr.KR_PATH_CUDA_CORES and op != kr.OP_KNN and D <= 16
        assert p.workspace_bytes == (_record_bytes(op, D, EK, N) if streamed else 0)


def test_split_fills_the_gpu_for_tall_products(lib):
    # M = 1e5 rows at D = 50 are only a few hundred blocks: the j axis must be split.
    p = kr.plan(kr.OP_SUM, 100_000, 10_000_000, 50, 1, num_sms=152, blocks_per_sm=4, path=kr.KR_PATH_CUDA_CORES)
    assert p.path == kr.KR_PATH_CUDA_CORES
    assert p.split > 1
    waves = (p.row_blocks * p.split) / (152 * 4)
    assert waves >= 2
    assert p.workspace_bytes == 2 * p.split * 100_000 * 4
    # never split below 64 points per split
    assert kr.plan(kr.OP_SUM, 10, 100, 3, 1).split == 1
    assert kr.plan(kr.OP_SUM, 1000, 1000, 3, 1, blocks_per_sm=8).chunk >= 64


def test_tensor_core_plan(lib):
    """Sum with E = 1 and 32 <= D <= 62 plans the tcgen05 path: 128 rows per block, tiles
    and splits of 256 points, split fp16 operands (256 B per point) and a padded copy of
    the signal in the workspace."""
    M, N = 100_000, 10_000_000
    p = kr.plan(kr.OP_SUM, M, N, 50, 1, num_sms=152, blocks_per_sm=1)
    assert p.path == kr.KR_PATH_TENSOR_CORES
    assert (p.threads, p.rows_per_thread, p.tile_points, p.d_pad) == (320, 1, 256, 64)
    assert p.row_blocks == (M + 127) // 128
    assert p.chunk % 256 == 0 and p.split * p.chunk >= N and (p.split - 1) * p.chunk < N
    # whole waves of 152 blocks: 782 row blocks x split fill them to within 1 %
    assert (p.row_blocks * p.split) / (-(-p.row_blocks * p.split // 152) * 152) > 0.99
    # a split's B operands (256 B per point) stay within 48 MB, so the blocks sharing it read L2
    assert p.chunk * 256 <= 48 << 20
    assert kr.plan(kr.OP_SUM, M, 1_000_000, 50, 1, num_sms=152, blocks_per_sm=1).chunk * 256 <= 48 << 20
    n_pad = (N + 255) // 256 * 256
    frames = (n_pad // 256 * 4 + 255) // 256 * 256          # LSE tile frames
    ops = ((M + 127) // 128 * 128 + n_pad) * 256 + 4 * n_pad + frames
    assert p.workspace_bytes == 256 + ops + (2 * p.split * M * 4 if p.split > 1 else 0)
    # the LogSumExp takes the tensor cores under the same conditions, with the same plan
    q = kr.plan(kr.OP_LSE, M, N, 50, 1, num_sms=152, blocks_per_sm=1)
    assert q.path == kr.KR_PATH_TENSOR_CORES and (q.split, q.chunk, q.workspace_bytes) == (p.split, p.chunk,
                                                                                            p.workspace_bytes)
    for shape in [(kr.OP_SUM, 10, 10, 31, 1), (kr.OP_SUM, 10, 10, 63, 1), (kr.OP_SUM, 10, 10, 50, 2),
                  (kr.OP_LSE, 10, 10, 50, 2), (kr.OP_GRAD, 10, 10, 50, 2), (kr.OP_GRAD, 10, 10, 63, 1),
                  (kr.OP_MAX, 10, 10, 50, 1),
                  (kr.OP_LSE, 10, 10, 62, 1)]:     # the LogSumExp's weight slot leaves D <= 61
        assert kr.plan(*shape).path == kr.KR_PATH_CUDA_CORES, shape
    assert kr.plan(kr.OP_SUM, 10, 10, 62, 1).path == kr.KR_PATH_TENSOR_CORES
    assert kr.plan(kr.OP_LSE, 10, 10, 61, 1).path == kr.KR_PATH_TENSOR_CORES
    # the x-gradient: 128-point tiles, D x M partials per split
    g = kr.plan(kr.OP_GRAD, 100_000, 1_000_000, 50, 1, num_sms=152, blocks_per_sm=1)
    assert g.path == kr.KR_PATH_TENSOR_CORES and g.tile_points == 128 and g.chunk % 128 == 0
    assert g.split * g.chunk >= 1_000_000 and (g.split - 1) * g.chunk < 1_000_000
    n_pad = (1_000_000 + 255) // 256 * 256
    ops_g = ((100_000 + 127) // 128 * 128 + n_pad) * 256 + n_pad * 4 + (n_pad // 256 * 4 + 255) // 256 * 256
    flags = (g.split * 100_000 + 255) // 256 * 256
    assert g.workspace_bytes == 256 + ops_g + (2 * g.split * 100_000 * 50 * 4 if g.split > 1 else 0) + flags
    assert kr.plan(kr.OP_GRAD, 10, 10, 32, 1).path == kr.KR_PATH_TENSOR_CORES
    assert kr.plan(kr.OP_GRAD, 10, 10, 50, 1, path=kr.KR_PATH_CUDA_CORES).path == kr.KR_PATH_CUDA_CORES
    assert kr.plan(kr.OP_SUM, 10, 10, 50, 1, path=kr.KR_PATH_CUDA_CORES).path == kr.KR_PATH_CUDA_CORES
    assert kr.plan(kr.OP_SUM, 10, 2560, 50, 1, split=5).split == 5
    assert kr.plan(kr.OP_SUM, 10, 2000, 50, 1, split=5).split == 4   # 512-point chunks
    assert kr.plan(kr.OP_SUM, 10, 600, 50, 1, split=9).split == 3   # at most one split per 256-point tile


def test_forced_split(lib):
    p = kr.plan(kr.OP_KNN, 1000, 5000, 16, 10, split=7)
    assert p.split == 7 and p.chunk == 715
    assert p.workspace_bytes == 7 * 1000 * 10 * 8
    assert kr.plan(kr.OP_KNN, 10, 3, 3, 1, split=9).split == 3   # never more splits than columns
    # streamed instances split on whole tiles: 3 columns are one 512-point tile
    assert kr.plan(kr.OP_SUM, 10, 3, 3, 1, split=9).split == 1
    assert kr.plan(kr.OP_SUM, 10, 3, 3, 1, split=9, kernel="laplace").split == 3


def _r256(v):
    return (v + 255) // 256 * 256


def _record_bytes(op, D, E, N):
    """Workspace of the streamed records of a Sum / LSE / gradient call at D <= 16: whole
    tiles of pair records (points 2m, 2m+1 interleaved field by field, padded to 16 bytes),
    and for the LogSumExp one frame per tile and column."""
    dp = D if D <= 4 else 8 if D <= 8 else 16
    ep = 1 if E <= 1 else 4 if E <= 4 else 16
    ps2 = (2 * (dp + ep) + 3) // 4 * 4
    bn = next(t for t in (512, 256, 128, 64, 32) if 16384 // ps2 >= t)
    tiles = (N + bn - 1) // bn
    return _r256(tiles * (bn // 2) * ps2 * 4) + (_r256(tiles * ep * 4) if op == kr.OP_LSE else 0)


@pytest.mark.parametrize("op,D,E,N,split", [
    (kr.OP_SUM, 3, 1, 100_000, 0), (kr.OP_LSE, 3, 1, 1_000_000, 0), (kr.OP_GRAD, 3, 1, 100_000, 7),
    (kr.OP_SUM, 16, 4, 30_000, 5), (kr.OP_LSE, 8, 16, 9_999, 3), (kr.OP_GRAD, 16, 1, 70_001, 0),
    (kr.OP_SUM, 1, 1, 513, 9),
])
def test_streamed_plan(lib, op, D, E, N, split):
    """Gaussian Sum / LSE / gradient up to D = 16 stream prepass records: every split is whole
    tiles (so each block's tiles are the prepass's), every split nonempty, and the workspace is
    the split partials followed by the records (and the LogSumExp's tile frames)."""
    M = 5000
    p = kr.plan(op, M, N, D, E, num_sms=152, blocks_per_sm=4, split=split)
    assert p.chunk % p.tile_points == 0
    assert p.split * p.chunk >= N and (p.split - 1) * p.chunk < N
    w = D if op == kr.OP_GRAD else E
    parts = 2 * p.split * M * w * 4 if p.split > 1 else 0
    assert p.workspace_bytes == _r256(parts) + _record_bytes(op, D, E, N)
    # the other kernels, the K-min and D > 16 stream nothing
    c = kr.plan(kr.OP_SUM, M, N, D, E, kernel="cauchy")
    assert c.workspace_bytes == (2 * c.split * M * E * 4 if c.split > 1 else 0)
    q = kr.plan(kr.OP_SUM, M, N, 32, E, path=kr.KR_PATH_CUDA_CORES, split=split)
    assert q.workspace_bytes == (2 * q.split * M * E * 4 if q.split > 1 else 0)


def test_python_marshalling_errors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 3)
    with pytest.raises(TypeError):
        kr.kernel_reduce(x.double(), x, torch.zeros(4), 1.0)
    with pytest.raises(ValueError):
        kr.kernel_reduce(x, torch.zeros(4, 2), torch.zeros(4), 1.0)
    with pytest.raises(ValueError):
        kr.kernel_reduce(x, x, torch.zeros(4), 1.0, reduction="median")
    with pytest.raises(ValueError):
        kr.kernel_reduce(x, x, torch.zeros(4), 1.0, kernel="matern")
    with pytest.raises(ValueError):
        kr.kernel_reduce_arg(x, x, torch.zeros(4), 1.0, reduction="sum")
    with pytest.raises(ValueError):
        kr.kernel_reduce(x.t(), x, torch.zeros(3), 1.0)
