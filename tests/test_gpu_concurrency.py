"""Calls from several host threads on several streams at once (the library keeps no mutable
global state besides per-device attributes and its memory pool): the results are the bits of
the same calls made one after another, for device and for host buffers."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from symbolic_matrix_reductions_gb300 import build
    build.build()
    kr.load_library()


def _inputs(device):
    r = np.random.Generator(np.random.PCG64(77))
    x = r.standard_normal((3000, 3)).astype(np.float32)
    y = r.standard_normal((20000, 3)).astype(np.float32)
    b = r.standard_normal((20000, 1)).astype(np.float32)
    g = r.standard_normal((3000, 1)).astype(np.float32)
    ts = [torch.from_numpy(a) for a in (x, y, b, g)]
    return [t.to(device) if device != "cpu" else t.pin_memory() for t in ts]


def _calls(x, y, b, g):
    return [lambda: kr.kernel_reduce(x, y, b, 0.5, "sum", split=4),
            lambda: kr.kernel_reduce(x, y, b, 0.5, "lse", split=4),
            lambda: kr.kernel_reduce_grad_x(x, y, b, g, 0.5, split=4),
            lambda: kr.kernel_knn(x, y, 10, split=3)[0],
            lambda: kr.kernel_reduce_arg(x, y, b, 0.5, "max")[0]]


def _host(t):
    return t.cpu().numpy() if t.is_cuda else t.numpy()


@pytest.mark.parametrize("device", ["cuda:0", "cpu"])
def test_threads_and_streams_give_the_sequential_bits(device):
    calls = _calls(*_inputs(device))
    seq = [_host(c()) for c in calls]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in calls]

    def run(k):
        with torch.cuda.stream(streams[k]):
            out = calls[k]()
            streams[k].synchronize()
            return _host(out)

    with ThreadPoolExecutor(max_workers=len(calls)) as pool:
        for _ in range(3):
            got = list(pool.map(run, range(len(calls))))
            for k, (u, v) in enumerate(zip(seq, got)):
                assert np.array_equal(u, v), f"call {k} differs when run concurrently"
