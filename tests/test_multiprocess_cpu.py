"""The multi-process (N > 1) paths on CPU, world size 2 and 3, gloo.

One problem is split by rows: rank r owns rows [M r / R, M (r + 1) / R) of x (and of the
upstream gradient), reduces them against all of y, and writes its slice; the job's
time is the slowest rank's (all-reduce MAX) and its value counts the whole problem's
pairs once.  Here each rank computes its slice with the fp64 oracle (rows are
independent, so the slices gathered in rank order must equal one run over all rows,
bit for bit), on ragged M, on M smaller than the world (empty slices) and on M = 0.
The reference arm runs on rank 0 alone; the other ranks exit 0 without work."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank(10.0 + 5.0 * rank, world)   # rank 1 is the slow one
        value = bench.job_value(4e10, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_timing_takes_the_slowest_rank(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert res[0]["ms"] == res[1]["ms"] == 15.0
    # one problem of 4e10 pairs, split over the ranks, done when the slowest rank is: 15 ms
    assert res[0]["value"] == pytest.approx(4e10 / 15e-3)


def _case(M, N=300, D=3, seed=0):
    r = np.random.Generator(np.random.PCG64(seed + M))
    x = r.standard_normal((M, D)).astype(np.float32)
    y = r.standard_normal((N, D)).astype(np.float32)
    b = r.standard_normal((N, 2)).astype(np.float32)
    g = r.standard_normal((M, 2)).astype(np.float32)
    return x, y, b, g


def _shard_main(rank, world, port, out_dir, Ms):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import oracle
    from symbolic_matrix_reductions_gb300.sharding import gather_rows, row_shard
    orc = oracle.load()
    orc.set_num_threads(1)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = {}
        for M in Ms:
            x, y, b, g = _case(M)
            sh = row_shard(M, world, rank)
            xs, gs = sh.take(x), sh.take(g)
            a, _ = orc.gauss_sum(xs, y, b, 0.7)
            gx, _ = orc.gauss_grad_x(xs, y, b, gs, 0.7)
            idx, d, _ = orc.knn(xs, y, 4)
            full = [gather_rows(torch.from_numpy(np.ascontiguousarray(v)), sh).numpy()
                    for v in (a, gx, idx.astype(np.int64), d)]
            res[M] = {"rows": sh.rows, "start": sh.start, "out": [v.tolist() for v in full]}
        with open(os.path.join(out_dir, f"shard{rank}.json"), "w") as f:
            json.dump({str(k): v for k, v in res.items()}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_row_sharding_gathers_the_single_rank_result(tmp_path, world, orc):
    Ms = [1001, 7, 2, 1, 0]   # ragged, small, fewer rows than ranks (empty slices), none
    port = _free_port()
    mp.start_processes(_shard_main, args=(world, port, str(tmp_path), Ms), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"shard{r}.json")) for r in range(world)]
    for M in Ms:
        x, y, b, g = _case(M)
        a, _ = orc.gauss_sum(x, y, b, 0.7)
        gx, _ = orc.gauss_grad_x(x, y, b, g, 0.7)
        idx, d, _ = orc.knn(x, y, 4)
        want = [a, gx, idx.astype(np.int64), d]
        starts = [res[r][str(M)]["start"] for r in range(world)]
        rows = [res[r][str(M)]["rows"] for r in range(world)]
        assert sum(rows) == M and starts == sorted(starts) and max(rows) - min(rows) <= 1
        for r in range(world):   # every rank holds the whole gathered output
            for got, w in zip(res[r][str(M)]["out"], want):
                got = np.asarray(got, dtype=w.dtype).reshape(w.shape)
                assert np.array_equal(got, w), (M, r)


def test_row_shard_cover():
    from symbolic_matrix_reductions_gb300.sharding import all_shards, row_shard
    for M in (0, 1, 5, 100, 10**6 + 3):
        for R in (1, 2, 3, 8):
            sh = all_shards(M, R)
            assert sh[0].start == 0 and sh[-1].stop == M
            assert all(p.stop == q.start for p, q in zip(sh, sh[1:]))
            assert max(s.rows for s in sh) - min(s.rows for s in sh) <= 1
    with pytest.raises(ValueError):
        row_shard(10, 2, 2)
    with pytest.raises(ValueError):
        row_shard(-1, 2, 0)


def test_reference_arm_under_torchrun():
    """bench.py --impl reference with two ranks: one JSON line from rank 0, exit 0, the same
    config as our arm's (rows sharded over the ranks)."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--size", "300,2000", "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    sys.path.insert(0, ROOT)
    import bench
    assert line["config"] == bench.step_config(bench.PRIMARY + " resized", 300, 2000, 3, 1, 0.1, 2)
