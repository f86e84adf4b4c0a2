"""Row sharding through the C ABI on one GPU: the slices a rank of R would compute (rows
[M r / R, M (r + 1) / R) of x and g, all of y and b, written into its slice of the
caller's output) are computed one after another here and put together.  With the same
split-j choice they give the bits of one call over all rows for the Sum, the gradient
and the K-min (rows are independent and every row's arithmetic depends only on the
j-ranges) and the LogSumExp up to the rounding of its frame; when each slice plans its
own split, the oracle's results within the usual tolerances."""
import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr
from symbolic_matrix_reductions_gb300.sharding import all_shards

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


def _ops(x, y, b, g, split, outs):
    a, L, gx, idx, dist = outs
    kr.kernel_reduce(x, y, b, 0.6, "sum", out=a, split=split)
    kr.kernel_reduce(x, y, b, 0.6, "lse", out=L, split=split)
    kr.kernel_reduce_grad_x(x, y, b, g, 0.6, out=gx, split=split)
    kr.kernel_knn(x, y, 8, idx=idx, dist=dist, split=split)


def _outs(M, D, E):
    return [torch.empty((M, E), device=DEV), torch.empty((M, E), device=DEV), torch.empty((M, D), device=DEV),
            torch.empty((M, 8), dtype=torch.int32, device=DEV), torch.empty((M, 8), device=DEV)]


@pytest.mark.parametrize("M,R,split", [(5001, 2, 4), (5001, 3, 1), (3, 4, 2), (20000, 8, 7)])
def test_slices_put_together_give_the_single_call(orc, M, R, split):
    r = np.random.Generator(np.random.PCG64(M + R))
    N, D, E = 30000, 3, 1
    x, y, b, g = (torch.from_numpy(r.standard_normal(s).astype(np.float32)).to(DEV)
                  for s in ((M, D), (N, D), (N, E), (M, E)))
    whole = _outs(M, D, E)
    _ops(x, y, b, g, split, whole)
    parts = _outs(M, D, E)
    for sh in all_shards(M, R):
        if sh.rows == 0:
            continue   # a rank with no rows calls nothing
        _ops(sh.take(x), y, b, sh.take(g), split, [sh.take(o) for o in parts])
    torch.cuda.synchronize()
    for k in (0, 2, 3, 4):   # Sum, gradient, K-min indices and distances: the same bits
        assert torch.equal(whole[k], parts[k]), k
    # The LogSumExp recomputes a tile in its row's own frame when one of a thread's rows needs
    # it, and which rows share a thread depends on where the slice starts: the same value up
    # to the rounding of the frame.
    Lw, Lp = whole[1].cpu().double(), parts[1].cpu().double()
    assert ((Lw - Lp).abs() <= 2e-6 * (1 + Lw.abs())).all()
    # and each rank planning its own split: still the oracle's results
    auto = _outs(M, D, E)
    for sh in all_shards(M, R):
        if sh.rows:
            _ops(sh.take(x), y, b, sh.take(g), 0, [sh.take(o) for o in auto])
    torch.cuda.synchronize()
    rows = np.sort(r.choice(M, size=min(M, 200), replace=False))
    xn, yn, bn, gn = (t.cpu().numpy() for t in (x, y, b, g))
    a_ref, S_ref = orc.gauss_sum(xn[rows], yn, bn, 0.6)
    check_sum(auto[0].cpu().numpy()[rows], a_ref, S_ref, "sharded sum")
    check_lse(auto[1].cpu().numpy()[rows], orc.gauss_lse(xn[rows], yn, bn, 0.6), "sharded lse")
    gx_ref, G_ref = orc.gauss_grad_x(xn[rows], yn, bn, gn[rows], 0.6)
    check_grad(auto[2].cpu().numpy()[rows], gx_ref, G_ref, "sharded grad")
    i_ref, d_ref, n_ref = orc.knn(xn[rows], yn, 8)
    check_knn(auto[3].cpu().numpy()[rows], auto[4].cpu().numpy()[rows], xn[rows], yn, i_ref, d_ref, n_ref,
              "sharded knn")
