"""Benchmark of the symbolic kernel reductions on one GB300 (or one problem row-sharded
over N GPUs).

A step is one pass of the whole hot path over one batch of synthetic input.  The
headline batch is the largest D = 3 configuration, gauss_d3_unit: M = N = 10^6
points in the unit cube, sigma = 0.1, b ~ U(0.1, 1).  A step runs the Gaussian Sum,
the LogSumExp (w = log b as log-weights), the x-gradient (upstream g ~ N(0,1)) and
the K-min (K = 10), each through the C ABI; split-j runs whenever the planner picks
it.  The metric is pair-evaluations per second, M*N per reduction, over the step.
The D = 50 line (key "d50") is the tall kernel-vector product falkon_d50 (M = 10^5,
N = 10^7, split-j, tensor cores), measured with the same protocol, with the LogSumExp,
the x-gradient and the K-min of the same clouds beside it.

Prints ONE JSON line (rank 0).  Timing: W warm-up steps, then K steps, each bracketed
by CUDA events on the launching stream; L2 is flushed (a 256 MB write) before every
timed step, outside the events.  Also reported:
  * roofline of the dominant kernel against the FP32 / MUFU pipe peak derived from the
    SM count, the FP32 lanes per SM, the ex2 lanes per SM (measured by the pipe probe in
    this run) and the maximum SM clock; per-op times from a pass one op at a time;
  * e2e: the same step with HOST buffers through the same C ABI calls (the library
    stages inputs and results), timed on the host clock;
  * cpu_baseline and parity: the fp64 oracle on this host's cores on a seeded row
    subset with the full N, and the step's GPU outputs on those rows against it;
  * secondary lines (3 warm-up + 10 timed runs, median, each with its roofline): the
    step at M = N = 10^5 (gauss_d3), the other kernels and Max/Min, a batch of 256 small
    problems, a block-sparse Sum, the y- and b-gradients, the D = 50 LogSumExp and the
    D = 16 K-min.
``--impl reference`` times the oracle as the reference arm instead, on the same config.
Under torchrun (N > 1) the problem is split by rows: rank r owns rows
[M r / N, M (r + 1) / N) of x (and g) for every op, with all of y and b, and writes its
slice of every output (no data exchange; gloo carries only the barrier and the max over
ranks).  The job value is the whole problem's pairs over the slowest rank's time
(strong scaling: the total work is fixed).
"""
from __future__ import annotations

import argparse
from concurrent.futures import ThreadPoolExecutor
import ctypes
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Gaussian kernel pair-evals/s (M·N/t) at D=3 and D=50; % of FP32/MUFU roofline"
UNIT = "pair-evals/s"
PRIMARY = "gauss_d3_unit"
D50 = "falkon_d50"
K_NN = 10
WARM_SECONDARY, RUNS_SECONDARY = 3, 10

# Per-pair pipe operations of each kernel (the counts the hot loop must issue, with
# x and y prescaled once per point):  FP32 = FADD/FMUL/FFMA lanes, XU = MUFU ex2,
# CMP = compares / min-max on the ALU pipe.  Sum: D sub + D mul/fma + 1 fma;  LSE: the
# same (the per-tile offset W - w'_j starts the distance's fma chain, so no per-pair max
# is needed);  grad: D sub + D fma (distance) + 1 mul (k*b) + D fma;  K-min: D sub +
# D fma + 1 compare.  Other kernels (Sum, Max/Min): Laplace adds a square root on the XU
# pipe before the ex2; Cauchy and the inverse multiquadric start the distance sum at 1
# and take one rcp / rsqrt instead of the ex2.  Each XU operation has its own rate
# (measured by the pipe probe), so XU counts are kept per operation.  Max/Min: k*b is
# one multiply per column and the running comparison one compare per pair.  With one column
# the kernel scans a key instead (Gaussian q - log2|b|, the log2 starting the distance's fma
# chain: D sub + D fma + 1 compare; Laplace sqrt(q) - log2|b|: one more add and the sqrt;
# Cauchy (1 + q) / |b| and inverse multiquadric (1 + q) / b^2: one more multiply, no XU);
# its line reports that bound too ("own_bound"), beside the method's count.
XU_PER_KERNEL = {"gaussian": {"ex2": 1}, "laplace": {"sqrt": 1, "ex2": 1}, "cauchy": {"rcp": 1},
                 "imq": {"rsqrt": 1}}


def ops_per_pair(op: str, D: int, E: int = 1, kernel: str = "gaussian"):
    if op == "sum":
        return {"fp32": 2 * D + E, "xu": dict(XU_PER_KERNEL[kernel]), "cmp": 0}
    if op in ("max", "min"):
        return {"fp32": 2 * D + E, "xu": dict(XU_PER_KERNEL[kernel]), "cmp": E}
    if op == "lse":
        return {"fp32": 2 * D + E, "xu": {"ex2": E}, "cmp": 0}
    if op == "grad":
        return {"fp32": 3 * D + 1 + (E if E > 1 else 0), "xu": {"ex2": 1}, "cmp": 0}
    if op == "knn":
        return {"fp32": 2 * D, "xu": {}, "cmp": 1}
    raise ValueError(op)


FP32_LANES_PER_SM = 128   # Blackwell SM: 4 partitions x 32 FP32 lanes
ALU_LANES_PER_SM = 64     # integer/compare pipe: 4 partitions x 16 lanes

# DRAM traffic per launch from ncu captures (profiles/), keyed by kernel and the
# hash of the kernel sources it was taken on; stale entries report null.
TRAFFIC = {
    # profiles/grad2_kernel_d3_gauss_d3_unit.md: dram__bytes_read.sum + dram__bytes_write.sum of one
    # full-size launch of the step's x-gradient (1e6 x 1e6, 7 splits; a one-pass capture), with the hash
    # of the kernel sources it ran
    "grad_kernel[D=3,E=1]": {"bytes_per_launch": 42504960 + 117179648, "source_hash": "90173c85c31abf92"},
}


def _kernel_source_hash():
    h = hashlib.sha256()
    for f in ("kr_kernels.cuh", "kr_kernels_packed.cuh", "kr_config.h"):
        with open(os.path.join(ROOT, "symbolic_matrix_reductions_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in getattr(self, "lines", []):
            p = [s.strip() for s in l.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append((float(p[1]), float(p[2]), p[5], p[6], p[7], p[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = np.array([r[0] for r in rows])
        smax = max(r[1] for r in rows)
        load = sm[sm >= 0.5 * smax] if (sm >= 0.5 * smax).any() else sm
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[k] for r in rows for k in range(4) if r[2 + k].lower().startswith("active")})
        return {"sm_mhz": float(np.median(load)), "sm_max_mhz": float(smax), "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# pipe probe (ex2 lanes per clock per SM), measured in this run
# ---------------------------------------------------------------------------
def probe_pipes(torch, nsm):
    """ex2 lanes per clock per SM, from the ex2 : FFMA throughput ratio of the pipe
    probe (both timed with CUDA events back to back, so the SM clock cancels) times
    the 128 FP32 lanes of an SM; reported raw and rounded to the power of two the
    hardware has."""
    lib = ctypes.CDLL(os.path.join(ROOT, "symbolic_matrix_reductions_gb300", "libkrprobe.so"))
    lib.kr_probe_pipe.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 3
    bps, iters = 4, 8192
    blocks = nsm * bps
    sink = torch.zeros(1, device="cuda")
    cyc = torch.zeros(blocks, dtype=torch.int64, device="cuda")
    ms = {}
    for kind in (0, 2, 3, 4, 5, 0, 2, 3, 4, 5):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        rc = lib.kr_probe_pipe(kind, blocks, iters, ctypes.c_void_p(sink.data_ptr()),
                               ctypes.c_void_p(cyc.data_ptr()), None)
        e1.record()
        if rc != 0:
            raise RuntimeError(f"probe launch failed: {rc}")
        torch.cuda.synchronize()
        ms[kind] = e0.elapsed_time(e1)          # the second run of each kind is kept
    lanes = {}
    for name, kind in (("ex2", 2), ("rcp", 3), ("rsqrt", 4), ("sqrt", 5)):
        measured = FP32_LANES_PER_SM * ms[0] / ms[kind]   # same lane count in both probes
        lanes[name] = float(2 ** round(np.log2(measured)))
        lanes[name + "_measured"] = measured
    return {"xu": lanes["ex2"], "xu_lanes": {k: v for k, v in lanes.items() if not k.endswith("_measured")},
            "xu_measured": {k[:-9]: v for k, v in lanes.items() if k.endswith("_measured")},
            "ex2_to_ffma": ms[0] / ms[2], "ffma_lanes_per_s": nsm * bps * 256 * iters * 8 / (ms[0] / 1e3)}


# Tensor-core Sum and LSE (E = 1, 32 <= D <= 62): per pair, three fp16 products (hi.hi, hi.lo,
# lo.hi) of the K = 64 augmented vectors, 2 FLOP per multiply-add.  The x-gradient adds a second
# product P.[y' | 1] of the same width (three split products, N = 64): twice the FLOP.
TC_FLOP_PER_PAIR = 3 * 2 * 64
TC_GRAD_FLOP_PER_PAIR = 2 * TC_FLOP_PER_PAIR
TC_KNN_FLOP_PER_PAIR = 2 * 64  # the K-min's screen: one fp16 product of the high halves


def tensor_peak_tflops():
    """Dense fp16 tensor peak: the measured bf16 cuBLAS burst peak (fp16 and bf16 have
    the same nominal dense rate on this part), else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        v = json.load(open(path)).get("bf16_tflops")
        if v:
            return float(v), "measured bf16 burst (fp16 nominal ratio 1)"
    return 1900.0, "fallback 1.9 PFLOP/s bf16 (fp16 nominal ratio 1)"


def roofline_tensor(seconds_per_launch, pairs, kernel, fp32_line, flop_per_pair=TC_FLOP_PER_PAIR):
    peak, basis = tensor_peak_tflops()
    achieved = pairs * flop_per_pair / seconds_per_launch / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": None, "kernel": kernel, "flop_per_pair": flop_per_pair, "peak_basis": basis,
            "pairs_per_s": pairs / seconds_per_launch,
            "vs_fp32_direct_roofline": {"peak_pairs_per_s": fp32_line["peak"], "frac": fp32_line["frac"]}}


def roofline(op, D, E, seconds_per_launch, pairs, nsm, clk_mhz, xu_lanes, kernel, live_mhz=None,
             kind="gaussian"):
    """xu_lanes: {XU operation: lanes per clock per SM} from the pipe probe.  "bound" is
    "alu" (arithmetic units: the kernel is bound by plain FP32 / XU / compare arithmetic,
    not by memory or tensor cores); "limiting_pipe" names which of those pipes sets the
    peak."""
    n = ops_per_pair(op, D, E, kind)
    xu_clk = sum(cnt / xu_lanes[name] for name, cnt in n["xu"].items())   # XU clocks per pair per SM lane set

    def peak_at(mhz):
        f = mhz * 1e6
        t = max(n["fp32"] / (nsm * FP32_LANES_PER_SM * f), xu_clk / (nsm * f),
                n["cmp"] / (nsm * ALU_LANES_PER_SM * f) if n["cmp"] else 0.0)
        return 1.0 / t

    peak = peak_at(clk_mhz)
    achieved = pairs / seconds_per_launch
    pipe = "xu" if xu_clk > n["fp32"] / FP32_LANES_PER_SM else "fp32"
    tr = TRAFFIC.get(kernel)
    traffic = tr["bytes_per_launch"] if tr and tr.get("source_hash") == _kernel_source_hash() else None
    out = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
           "traffic": traffic, "kernel": kernel, "limiting_pipe": pipe, "ops_per_pair": n,
           "peak_basis": f"{nsm} SMs x (128 FP32, 64 ALU; XU per op " +
                         ", ".join(f"{k} {v:.0f}" for k, v in xu_lanes.items()) +
                         f") lanes/clk x {clk_mhz:.0f} MHz max SM clock"}
    if live_mhz:
        out["frac_at_live_clock"] = achieved / peak_at(live_mhz)
    if op in ("max", "min") and E == 1:
        # the key scan: the distance, one more add / multiply except for the Gaussian, the
        # Laplace's sqrt, and one compare a pair
        f = clk_mhz * 1e6
        own = {"fp32": 2 * D + (0 if kind == "gaussian" else 1),
               "xu": {"sqrt": 1} if kind == "laplace" else {}, "cmp": 1}
        own_xu = sum(cnt / xu_lanes[name] for name, cnt in own["xu"].items())
        own_peak = 1.0 / max(own["fp32"] / (nsm * FP32_LANES_PER_SM * f), own_xu / (nsm * f),
                             1.0 / (nsm * ALU_LANES_PER_SM * f))
        out["own_bound"] = {"ops_per_pair": own, "peak": own_peak, "frac": achieved / own_peak}
    if op == "knn" and D <= 16:
        # The K-min kernel at D <= 16 screens pairs with |y~|^2 - 2 x~.y~ (D FMAs) and computes the
        # direct distance only for passing groups; frac above is against the method's direct count.
        f = clk_mhz * 1e6
        screen_peak = 1.0 / max(D / (nsm * FP32_LANES_PER_SM * f), 1.0 / (nsm * ALU_LANES_PER_SM * f))
        out["screen"] = {"ops_per_pair": {"fp32": D, "xu": {}, "cmp": 1}, "peak": screen_peak,
                         "frac": achieved / screen_peak}
    return out


# ---------------------------------------------------------------------------
# several GPUs: one problem split by rows; the job is as slow as its slowest rank
# ---------------------------------------------------------------------------
def slowest_rank(ms: float, world: int) -> float:
    """The largest of the ranks' times (all-reduce MAX over the process group)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(pairs_per_step: float, ms_per_step: float) -> float:
    """Whole-job pair-evaluations per second: the whole problem's pairs (all ranks' slices
    together) over the slowest rank's step time."""
    return pairs_per_step / (ms_per_step / 1e3)


def step_config(wname, M, N, D, E, sigma, world):
    """The workload description both arms print (identical, so that the two lines are
    comparable)."""
    from symbolic_matrix_reductions_gb300 import workloads as W
    return {"workload": f"{wname}: {W.WORKLOADS[wname].note if wname in W.WORKLOADS else wname}; step = Sum + "
                        f"LogSumExp (w = log b) + grad-x (g ~ N(0,1)) + K-min (K={K_NN})",
            "M": M, "N": N, "D": D, "E": E, "K": K_NN, "sigma": sigma, "pairs_per_step": 4 * M * N,
            "l2": "flushed before every timed step (256 MB write)",
            "parallelism": f"rows sharded over {world} GPUs" if world > 1 else "single GPU"}


def _median_ms(torch, fn, warm=WARM_SECONDARY, runs=RUNS_SECONDARY):
    """Median of `runs` CUDA-event timings after `warm` untimed calls (current stream)."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(runs):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return float(np.median(ts)), {"warmup": warm, "runs": runs, "stat": "median",
                                  "min_ms": float(np.min(ts)), "max_ms": float(np.max(ts))}


def _steady_ms(torch, fn, warm=WARM_SECONDARY, calls=RUNS_SECONDARY, reps=3):
    """Time per call of `calls` back-to-back calls between one pair of CUDA events (the host
    queues the next call while the GPU runs the last, as a caller looping over batches
    does); the median of `reps` such runs after `warm` untimed calls."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(calls):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / calls)
    return float(np.median(ts)), {"warmup": warm, "calls_per_run": calls, "runs": reps,
                                  "stat": "median of per-call means (back-to-back calls)"}


def launches_of(kr, p, op="sum", batch=1) -> int:
    """Kernels of this library one call with plan p launches."""
    if p.path == kr.KR_PATH_TENSOR_CORES:
        # two operand prepasses (and for the gradient the signal bound), the tensor kernel, its
        # CUDA-core stand-in [, combine]
        return 4 + (op == "grad") + (p.split > 1)
    streamed = op in ("sum", "lse", "grad") and p.d_pad <= 16 and batch <= 1
    return 1 + streamed + (p.split > 1)   # [record prepass,] the kernel [, combine]


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch

    import symbolic_matrix_reductions_gb300 as kr
    from symbolic_matrix_reductions_gb300 import build, workloads as W
    from symbolic_matrix_reductions_gb300.sharding import row_shard

    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    kr.load_library()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    max_mhz = float(json.load(open(peaks_path)).get("sm_max_mhz", 2070.0)) if os.path.exists(peaks_path) else 2070.0

    if args.lines:  # only the named secondary lines (a short command to profile one kernel)
        probe = probe_pipes(torch, nsm)
        names = [n.strip() for n in args.lines.split(",") if n.strip()]
        return {"lines": names, "secondary": secondary(torch, kr, W, nsm, max_mhz, probe["xu_lanes"], dev, names)}

    inp = W.generate(args.workload, M=args.size[0], N=args.size[1]) if args.size else W.generate(args.workload)
    M, D = inp["x"].shape
    N, E = inp["y"].shape[0], inp["b"].shape[1]
    s = inp["sigma"]
    wkey = "w_log" if "w_log" in inp else "b"
    sh = row_shard(M, world, rank)
    m = sh.rows
    x = torch.from_numpy(np.ascontiguousarray(sh.take(inp["x"]))).to(dev)
    g = torch.from_numpy(np.ascontiguousarray(sh.take(inp["g"]))).to(dev)
    y, b, w = (torch.from_numpy(inp[k]).to(dev) for k in ("y", "b", wkey))
    a = torch.empty((m, E), device=dev)
    L = torch.empty((m, E), device=dev)
    gx = torch.empty((m, D), device=dev)
    idx = torch.empty((m, K_NN), dtype=torch.int32, device=dev)
    dist_ = torch.empty((m, K_NN), device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    ops = [("sum", lambda: kr.kernel_reduce(x, y, b, s, "sum", out=a)),
           ("lse", lambda: kr.kernel_reduce(x, y, w, s, "lse", out=L)),
           ("grad", lambda: kr.kernel_reduce_grad_x(x, y, b, g, s, out=gx)),
           ("knn", lambda: kr.kernel_knn(x, y, K_NN, idx=idx, dist=dist_))]
    op_code = {"sum": kr.OP_SUM, "lse": kr.OP_LSE, "grad": kr.OP_GRAD, "knn": kr.OP_KNN}
    plans = {name: kr.plan_device(op_code[name], max(m, 1), N, D, K_NN if name == "knn" else E) for name, _ in ops}
    launches_per_step = sum(launches_of(kr, plans[n], n) for n, _ in ops) if m > 0 else 0
    pairs_per_step = 4 * M * N   # the whole problem (every rank's slice)

    # The four reductions are independent calls on the same inputs: a step issues each on its
    # own stream (K-min and the gradient first, the longest), all waiting on the step's start
    # event and joined back into the launching stream at its end.
    op_streams = [torch.cuda.Stream(dev) for _ in ops]
    order = [3, 2, 0, 1]

    def step_concurrent(start, end):
        start.record(stream)
        for o in order:
            op_streams[o].wait_event(start)
            with torch.cuda.stream(op_streams[o]):
                ops[o][1]()
        for st in op_streams:
            stream.wait_stream(st)
        end.record(stream)

    for _ in range(args.warmup):
        step_concurrent(torch.cuda.Event(), torch.cuda.Event())
    torch.cuda.synchronize(dev)
    probe = probe_pipes(torch, nsm) if rank == 0 else {"xu_lanes": {"ex2": 32.0, "rcp": 16.0, "rsqrt": 16.0,
                                                                    "sqrt": 16.0}}
    xu_lanes = probe["xu_lanes"]

    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    n_seq = min(args.steps, 5)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(n_seq)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            flush.zero_()
            step_concurrent(evc[k][0], evc[k][1])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
    # the same steps once more, one op at a time on the launching stream: the per-op times the
    # rooflines use (outside the timed region)
    for k in range(n_seq):
        flush.zero_()
        ev[k][0].record(stream)
        for o, (_, fn) in enumerate(ops):
            fn()
            ev[k][o + 1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    step_ms = [evc[k][0].elapsed_time(evc[k][1]) for k in range(args.steps)]
    seq_step_ms = float(np.median([ev[k][0].elapsed_time(ev[k][-1]) for k in range(n_seq)]))
    op_ms = {name: float(np.median([ev[k][o].elapsed_time(ev[k][o + 1]) for k in range(n_seq)]))
             for o, (name, _) in enumerate(ops)}
    total_ms = slowest_rank(float(np.sum(step_ms)), world)
    ms_per_step = total_ms / args.steps
    value = job_value(pairs_per_step, ms_per_step)
    clocks = clk.summary()

    e2e_line = e2e_step(torch, kr, inp, wkey, s, sh, args, world)
    if rank != 0:
        return None

    dominant = max(op_ms, key=op_ms.get)
    kname = {"sum": "fwd_kernel<Sum>", "lse": "fwd_kernel<LSE>", "grad": "grad_kernel",
             "knn": "knn_kernel"}[dominant]
    kname += f"[D={D},K={K_NN}]" if dominant == "knn" else f"[D={D},E={E}]"
    cfg = step_config(args.workload + (" resized" if args.size else ""), M, N, D, E, s, world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
        "ms_per_step_median": float(np.median(step_ms)),
        "plans": {n: {"split": plans[n].split, "path": "tensor cores" if plans[n].path == kr.KR_PATH_TENSOR_CORES
                      else "cuda cores", "rows_on_rank0": m} for n, _ in ops},
        "streams": "one stream per op, joined every step (the timed region); per_op_ms (median of "
                   f"{n_seq} steps) and the rooflines from a pass of the same steps one op at a time",
        "step_sequential_ms": seq_step_ms,
        "per_op_ms": op_ms,
        "roofline": roofline(dominant, D, E, op_ms[dominant] / 1e3, m * N, nsm, max_mhz, xu_lanes, kname,
                             clocks.get("sm_mhz")),
        "per_op_frac": {n: roofline(n, D, E, op_ms[n] / 1e3, m * N, nsm, max_mhz, xu_lanes, n)["frac"]
                        for n, _ in ops},
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "pipe_probe": probe,
        "wall_s_timed": t_wall,
    }
    line["e2e"] = e2e_line
    if world == 1 and not args.no_secondary:
        line["cpu_baseline"], ref, rows = cpu_baseline(inp, wkey, s, target_s=args.cpu_seconds)
        # the step's outputs (last pass) on the oracle's rows
        line["parity"] = parity_stats(ref, *(t.cpu().numpy()[rows] for t in (a, L, gx, idx, dist_)))
        del x, y, b, w, g, a, L, gx, idx, dist_
        torch.cuda.empty_cache()
        line["d50"] = measure_d50(torch, kr, W, nsm, max_mhz, xu_lanes, dev, args)
        line["secondary"] = secondary(torch, kr, W, nsm, max_mhz, xu_lanes, dev)
    return line


def _host_calls(torch, kr, xc, yc, bc, wc, gc, s):
    """The step's four calls on pinned host buffers, and their outputs."""
    m, D = xc.shape
    E = bc.shape[1]
    outs = {"a": torch.empty((m, E)).pin_memory(), "L": torch.empty((m, E)).pin_memory(),
            "gx": torch.empty((m, D)).pin_memory(), "idx": torch.empty((m, K_NN), dtype=torch.int32).pin_memory(),
            "dist": torch.empty((m, K_NN)).pin_memory()}
    calls = [lambda: kr.kernel_knn(xc, yc, K_NN, idx=outs["idx"], dist=outs["dist"]),
             lambda: kr.kernel_reduce_grad_x(xc, yc, bc, gc, s, out=outs["gx"]),
             lambda: kr.kernel_reduce(xc, yc, bc, s, "sum", out=outs["a"]),
             lambda: kr.kernel_reduce(xc, yc, wc, s, "lse", out=outs["L"])]
    return calls, outs


def e2e_step(torch, kr, inp, wkey, s, sh, args, world):
    """The same step through the C ABI with pinned host buffers (every rank, its row slice)."""
    xc, gc = (torch.from_numpy(np.ascontiguousarray(sh.take(inp[k]))).pin_memory() for k in ("x", "g"))
    yc, bc, wc = (torch.from_numpy(inp[k]).pin_memory() for k in ("y", "b", wkey))
    M, N = inp["x"].shape[0], yc.shape[0]
    calls, outs = _host_calls(torch, kr, xc, yc, bc, wc, gc, s)
    # As in the device-timed step, the four independent calls run at once: one host thread and
    # one stream each (the calls release the GIL and return when their outputs are in host memory).
    dev = torch.cuda.current_device()
    streams = [torch.cuda.Stream(dev) for _ in calls]

    def on_stream(k):
        with torch.cuda.stream(streams[k]):
            calls[k]()

    pool = ThreadPoolExecutor(max_workers=len(calls))

    def step():
        if sh.rows == 0:
            return
        for f in [pool.submit(on_stream, k) for k in range(len(calls))]:
            f.result()

    nb = lambda t: t.numel() * t.element_size()
    h2d = 4 * (nb(xc) + nb(yc)) + 2 * nb(bc) + nb(wc) + nb(gc)
    d2h = sum(nb(t) for t in outs.values())
    for _ in range(2):
        step()
    steps = max(3, min(args.steps, 10))
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    t = slowest_rank((time.perf_counter() - t0) / steps, world)
    pool.shutdown()
    return {"value": 4 * M * N / t, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": t * 1e3, "steps": steps, "warmup": 2,
            "timer": "host perf_counter; the four calls on four host threads and streams, each blocking on "
                     "its host outputs"}


# ---------------------------------------------------------------------------
# D = 50: the tall kernel-vector product on the tensor cores
# ---------------------------------------------------------------------------
def measure_d50(torch, kr, W, nsm, max_mhz, xu_lanes, dev, args):
    """falkon_d50 (M = 1e5, N = 1e7, D = 50, split-j): the Sum (the product itself) as a
    first-class line with its own roofline, e2e through host buffers, oracle parity on a
    seeded row subset and CPU baseline; the LogSumExp of the same clouds beside it."""
    inp = W.generate(D50)
    M, D = inp["x"].shape
    N = inp["y"].shape[0]
    s = inp["sigma"]
    x, y, b, g = (torch.from_numpy(inp[k]).to(dev) for k in ("x", "y", "b", "g"))
    a = torch.empty((M, 1), device=dev)
    L = torch.empty((M, 1), device=dev)
    gx = torch.empty((M, D), device=dev)
    idx = torch.empty((M, K_NN), dtype=torch.int32, device=dev)
    dist = torch.empty((M, K_NN), device=dev)
    out = {"workload": f"{D50}: {W.WORKLOADS[D50].note}", "M": M, "N": N, "D": D, "E": 1, "sigma": s,
           "metric": METRIC, "unit": UNIT,
           "note": "value = the tall kernel-vector product (the Sum); the LogSumExp (b as log-weights), the "
                   f"x-gradient (g ~ N(0,1)) and the K-min (K = {K_NN}) of the same clouds beside it"}
    calls = {"sum": (kr.OP_SUM, lambda: kr.kernel_reduce(x, y, b, s, "sum", out=a)),
             "lse": (kr.OP_LSE, lambda: kr.kernel_reduce(x, y, b, s, "lse", out=L)),
             "grad": (kr.OP_GRAD, lambda: kr.kernel_reduce_grad_x(x, y, b, g, s, out=gx)),
             "knn": (kr.OP_KNN, lambda: kr.kernel_knn(x, y, K_NN, idx=idx, dist=dist))}
    flop = {"sum": TC_FLOP_PER_PAIR, "lse": TC_FLOP_PER_PAIR, "grad": TC_GRAD_FLOP_PER_PAIR,
            "knn": TC_KNN_FLOP_PER_PAIR}
    for op, (code, fn) in calls.items():
        p = kr.plan_device(code, M, N, D, K_NN if op == "knn" else 1)
        ms, how = _median_ms(torch, fn, warm=3, runs=10 if op not in ("grad", "knn") else 5)
        rl = roofline(op, D, 1, ms / 1e3, M * N, nsm, max_mhz, xu_lanes, f"{op}[D={D},E=1] (CUDA-core count)")
        if p.path == kr.KR_PATH_TENSOR_CORES:
            rl = roofline_tensor(ms / 1e3, M * N, f"tc_{op}_kernel (tcgen05)", rl, flop[op])
        out[op] = {"value": M * N / (ms / 1e3), "ms": ms, "timing": how, "split": p.split,
                   "path": "tensor cores" if p.path == kr.KR_PATH_TENSOR_CORES else "cuda cores",
                   "gpu_launches_per_call": launches_of(kr, p, op), "roofline": rl}
    out["value"] = out["sum"]["value"]
    out["roofline"] = out["sum"]["roofline"]
    a_dev, L_dev, gx_dev = a.cpu().numpy(), L.cpu().numpy(), gx.cpu().numpy()
    idx_dev, dist_dev = idx.cpu().numpy(), dist.cpu().numpy()
    del x, y, g, gx, idx, dist
    torch.cuda.empty_cache()
    # e2e: the product through the C ABI with pinned host buffers (inputs up, result down)
    xc, yc, bc = (torch.from_numpy(inp[k]).pin_memory() for k in ("x", "y", "b"))
    ac = torch.empty((M, 1)).pin_memory()
    for _ in range(2):
        kr.kernel_reduce(xc, yc, bc, s, "sum", out=ac)
    reps = 5
    t0 = time.perf_counter()
    for _ in range(reps):
        kr.kernel_reduce(xc, yc, bc, s, "sum", out=ac)
    t = (time.perf_counter() - t0) / reps
    nb = lambda t_: t_.numel() * t_.element_size()
    out["e2e"] = {"value": M * N / t, "unit": UNIT, "ms_per_step": t * 1e3, "steps": reps, "warmup": 2,
                  "h2d_bytes_per_step": nb(xc) + nb(yc) + nb(bc), "d2h_bytes_per_step": nb(ac),
                  "timer": "host perf_counter around the blocking host-buffer call"}
    del xc, yc, bc, ac
    # the oracle on a seeded row subset with the full N (CPU baseline and parity)
    import oracle
    orc = oracle.load()
    probe_rows = W.row_subset(M, 8, 41)
    t0 = time.perf_counter()
    orc.gauss_sum(inp["x"][probe_rows], inp["y"], inp["b"], s)
    per_row = (time.perf_counter() - t0) / probe_rows.size
    r = int(max(8, min(1000, args.cpu_seconds / max(per_row, 1e-9))))
    rows = W.row_subset(M, r, 9)
    t0 = time.perf_counter()
    a_ref, S_ref = orc.gauss_sum(inp["x"][rows], inp["y"], inp["b"], s)
    t = time.perf_counter() - t0
    out["cpu_baseline"] = {"value": r * N / t, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                           "sample": f"seeded subset of {r} rows of {D50}, full N={N}: the Sum in fp64, {t:.1f} s"}
    L_ref = orc.gauss_lse(inp["x"][rows[:64]], inp["y"], inp["b"], s)
    g_ref, G_ref = orc.gauss_grad_x(inp["x"][rows[:32]], inp["y"], inp["b"], inp["g"][rows[:32]], s)
    i_ref, d_ref, n_ref = orc.knn(inp["x"][rows[:32]], inp["y"], K_NN)
    sum_err = float(np.max(np.abs(a_dev[rows] - a_ref) / np.maximum(S_ref, 1e-300)))
    lse_err = np.abs(L_dev[rows[:64]] - L_ref)
    grad_err = float(np.max(np.abs(gx_dev[rows[:32]] - g_ref) / np.maximum(G_ref, 1e-300)))
    ext = np.concatenate([np.full((32, 1), -np.inf), d_ref, n_ref[:, None]], axis=1)
    cur = ext[:, 1:-1]
    with np.errstate(invalid="ignore"):
        sep = ((cur - ext[:, :-2]) > 1e-5 * np.abs(cur)) & ((ext[:, 2:] - cur) > 1e-5 * np.abs(cur))
    mism = int(np.sum(sep & (idx_dev[rows[:32]].astype(np.int64) != i_ref)))
    knn_dist_err = float(np.max(np.abs(dist_dev[rows[:32]] - d_ref) / np.maximum(np.abs(d_ref), 1e-30)))
    out["parity"] = {"rows": r, "sum_err_over_S": sum_err, "lse_rows": 64, "lse_abs_err": float(np.max(lse_err)),
                     "grad_rows": 32, "grad_err_over_G": grad_err,
                     "knn_rows": 32, "knn_separated_mismatches": mism, "knn_near_ties": int(np.sum(~sep)),
                     "knn_dist_rel_err": knn_dist_err,
                     "ok": bool(sum_err <= 1e-4 and np.all(lse_err <= 1e-4 + 2.0 ** -20 * np.abs(L_ref))
                                and grad_err <= 1e-4 and mism == 0),
                     "tolerances": "Sum 1e-4 S; LSE 1e-4 + 2^-20 |L|; grad 1e-4 G; "
                                   "K-min indices exact where separated"}
    return out


def secondary(torch, kr, W, nsm, max_mhz, xu_lanes, dev, only=None):
    """Other workloads and reductions, 3 warm-up + 10 timed runs each (median), with rooflines.
    only: names of the lines to run (an op name as the lines print it, e.g. "max (gaussian)",
    "sum (batched)"); None: all."""
    out = []

    def want(name):
        return only is None or name in only
    inp = W.generate("gauss_d3")
    x, y, bb, gg = (torch.from_numpy(inp[k]).to(dev) for k in ("x", "y", "b", "g"))
    M, D = x.shape
    N, E = y.shape[0], bb.shape[1]
    s = inp["sigma"]
    wl = f"gauss_d3: {W.WORKLOADS['gauss_d3'].note}"
    # the step's four ops at M = N = 1e5
    step_ops = (("sum", lambda: kr.kernel_reduce(x, y, bb, s, "sum"), kr.OP_SUM, E),
                ("lse", lambda: kr.kernel_reduce(x, y, bb, s, "lse"), kr.OP_LSE, E),
                ("grad", lambda: kr.kernel_reduce_grad_x(x, y, bb, gg, s), kr.OP_GRAD, E),
                ("knn", lambda: kr.kernel_knn(x, y, K_NN), kr.OP_KNN, K_NN))
    for op, fn, code, ek in step_ops:
        if not want(op):
            continue
        p = kr.plan_device(code, M, N, D, ek)
        ms, how = _median_ms(torch, fn)
        out.append({"workload": wl, "op": op, "ms": ms, "value": M * N / (ms / 1e3), "unit": UNIT,
                    "split": p.split, "path": "cuda cores", "timing": how,
                    "roofline": roofline(op, D, E, ms / 1e3, M * N, nsm, max_mhz, xu_lanes, f"{op}[D={D}]")})
    for op, kind in (("sum", "laplace"), ("sum", "cauchy"), ("sum", "imq"), ("max", "gaussian"),
                     ("min", "gaussian"), ("max", "cauchy")):
        if not want(f"{op} ({kind})"):
            continue
        fn = (lambda op=op, kind=kind: kr.kernel_reduce(x, y, bb, s, op, kernel=kind))
        p = kr.plan_device(kr.OP_SUM if op == "sum" else kr.OP_MAX, M, N, D, E, kernel=kind)
        ms, how = _median_ms(torch, fn)
        kname = f"radial_kernel<{kind},{'Sum' if op == 'sum' else 'Max'}>[D={D},E={E}]"
        rl = roofline(op, D, E, ms / 1e3, M * N, nsm, max_mhz, xu_lanes, kname, kind=kind)
        out.append({"workload": wl, "op": f"{op} ({kind})", "ms": ms, "value": M * N / (ms / 1e3), "unit": UNIT,
                    "split": p.split, "path": "cuda cores", "timing": how, "roofline": rl})
    # the transposed problem: N output rows, reduction over the M points of x
    for op in ("grad_y", "grad_b"):
        if not want(op):
            continue
        if op == "grad_y":
            fn = (lambda: kr.kernel_reduce_grad_y(x, y, bb, gg, s))
            p = kr.plan_device(kr.OP_GRAD, N, M, D, E)
            kname = f"grad_kernel[D={D},E={E}] on (y, x)"
        else:
            fn = (lambda: kr.kernel_reduce_grad_b(x, y, gg, s))
            p = kr.plan_device(kr.OP_SUM, N, M, D, E)
            kname = f"fwd_kernel<Sum>[D={D},E={E}] on (y, x)"
        ms, how = _median_ms(torch, fn)
        rl = roofline("grad" if op == "grad_y" else "sum", D, E, ms / 1e3, M * N, nsm, max_mhz, xu_lanes, kname)
        out.append({"workload": wl, "op": op, "ms": ms, "value": M * N / (ms / 1e3), "unit": UNIT,
                    "split": p.split, "path": "cuda cores", "timing": how, "roofline": rl})
    del x, y, bb, gg

    if want('sum (batched)'):
        # batch dimension: 256 independent gauss_d3-distributed problems of 2000 x 2000 points
        r = np.random.Generator(np.random.PCG64(2024))
        Bb, Mb = 256, 2000
        xb = torch.from_numpy(r.standard_normal((Bb, Mb, 3)).astype(np.float32)).to(dev)
        yb = torch.from_numpy(r.standard_normal((Bb, Mb, 3)).astype(np.float32)).to(dev)
        bb3 = torch.from_numpy(r.standard_normal((Bb, Mb, 1)).astype(np.float32)).to(dev)
        batch_fn = (lambda: kr.kernel_reduce(xb, yb, bb3, 0.5, "sum"))
        ms, how = _steady_ms(torch, batch_fn)
        ms1, how1 = _median_ms(torch, batch_fn)
        pairs = Bb * Mb * Mb
        how["single_call"] = dict(how1, ms=ms1, value=pairs / (ms1 / 1e3))
        out.append({"workload": f"batch of {Bb} problems, M=N={Mb}, D=3, x,y,b ~ N(0,1), sigma=0.5", "op": "sum (batched)",
                    "ms": ms, "value": pairs / (ms / 1e3), "unit": UNIT, "split": None, "path": "cuda cores",
                    "timing": how, "roofline": roofline("sum", 3, 1, ms / 1e3, pairs, nsm, max_mhz, xu_lanes,
                                                        f"fwd_kernel<Sum>[D=3,E=1] x {Bb} (grid z)")})
        del xb, yb, bb3

    if want('sum (block-sparse)'):
        # block-sparse: the gauss_d3_unit clouds (1e6 points each) sorted into 250 slabs along the
        # first coordinate; cluster c of x reduces over slabs c-1..c+1 of y (a truncated kernel
        # product; the value counts the pairs evaluated)
        inp = W.generate("gauss_d3_unit")
        xs = inp["x"][np.argsort(inp["x"][:, 0], kind="stable")]
        order = np.argsort(inp["y"][:, 0], kind="stable")
        ys, bs = inp["y"][order], inp["b"][order]
        M, N, C = xs.shape[0], ys.shape[0], 250
        ex, ey = np.linspace(0, M, C + 1).astype(np.int64), np.linspace(0, N, C + 1).astype(np.int64)
        ri = np.stack([ex[:-1], ex[1:]], 1)
        rj = np.array([[ey[max(c - 1, 0)], ey[min(c + 2, C)]] for c in range(C)])
        si = np.arange(1, C + 1)
        pairs = int(sum((ri[c, 1] - ri[c, 0]) * (rj[c, 1] - rj[c, 0]) for c in range(C)))
        xt, yt, bt = (torch.from_numpy(a_).to(dev) for a_ in (xs, ys, bs))
        ms, how = _median_ms(torch, lambda: kr.kernel_reduce_ranges(xt, yt, bt, inp["sigma"], "sum", ri, si, rj))
        out.append({"workload": f"gauss_d3_unit clouds (1e6 points) sorted into {C} slabs along x_0; each cluster reduces "
                                f"over its 3 neighbouring slabs ({pairs} of {M * N} pairs evaluated)",
                    "op": "sum (block-sparse)", "ms": ms, "value": pairs / (ms / 1e3), "unit": UNIT, "split": None,
                    "path": "cuda cores", "timing": how,
                    "roofline": roofline("sum", 3, 1, ms / 1e3, pairs, nsm, max_mhz, xu_lanes,
                                         "radial_kernel<gaussian,Sum>[D=3,E=1] (ranges)")})
        del xt, yt, bt

    if want('knn'):
        # the D = 16 K-min
        inp = W.generate("knn_d16")
        x, y = (torch.from_numpy(inp[k]).to(dev) for k in ("x", "y"))
        M, D = x.shape
        N = y.shape[0]
        K = inp["K"]
        p = kr.plan_device(kr.OP_KNN, M, N, D, K)
        ms, how = _median_ms(torch, lambda: kr.kernel_knn(x, y, K), warm=3, runs=5)
        out.append({"workload": f"knn_d16: {W.WORKLOADS['knn_d16'].note}", "op": "knn", "ms": ms,
                    "value": M * N / (ms / 1e3), "unit": UNIT, "split": p.split, "path": "cuda cores", "timing": how,
                    "roofline": roofline("knn", D, 1, ms / 1e3, M * N, nsm, max_mhz, xu_lanes,
                                         f"knn_kernel[D={D},K={K}]")})
        del x, y
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU baseline / reference arm: the fp64 oracle, as it stands
# ---------------------------------------------------------------------------
def _oracle_step(orc, inp, s, rows, wkey="b"):
    x = inp["x"][rows]
    return {"sum": orc.gauss_sum(x, inp["y"], inp["b"], s),
            "lse": orc.gauss_lse(x, inp["y"], inp[wkey], s),
            "grad": orc.gauss_grad_x(x, inp["y"], inp["b"], inp["g"][rows], s),
            "knn": orc.knn(x, inp["y"], K_NN)}


def parity_stats(ref, a, L, gx, idx, dist):
    """The step's GPU outputs on the oracle's sample rows (given in the same row order)
    against the oracle, with the library's tolerances: Sum |err| <= 1e-4 S (S = sum_j
    |k b|), LSE |err| <= 1e-4 + 2^-20 |L|, grad-x |err| <= 1e-4 G (G = its sum of
    magnitudes), K-min indices equal wherever the oracle's distance at that position is
    separated (1e-5 relative) from its neighbours; the other positions are near-ties,
    counted."""
    a_ref, S_ref = ref["sum"]
    L_ref = ref["lse"]
    g_ref, G_ref = ref["grad"]
    i_ref, d_ref, n_ref = ref["knn"]
    r = a_ref.shape[0]
    sum_err = float(np.max(np.abs(a[:r] - a_ref) / np.maximum(S_ref, 1e-300)))
    lse_err = np.abs(L[:r] - L_ref)
    lse_ok = bool(np.all(lse_err <= 1e-4 + 2.0 ** -20 * np.abs(L_ref)))
    grad_err = float(np.max(np.abs(gx[:r] - g_ref) / np.maximum(G_ref, 1e-300)))
    ext = np.concatenate([np.full((r, 1), -np.inf), d_ref, n_ref[:, None]], axis=1)
    cur = ext[:, 1:-1]
    with np.errstate(invalid="ignore"):
        sep = ((cur - ext[:, :-2]) > 1e-5 * np.abs(cur)) & ((ext[:, 2:] - cur) > 1e-5 * np.abs(cur))
    mism = int(np.sum(sep & (idx[:r].astype(np.int64) != i_ref)))
    dist_err = float(np.max(np.abs(dist[:r] - d_ref) / np.maximum(np.abs(d_ref), 1e-30)))
    ok = sum_err <= 1e-4 and lse_ok and grad_err <= 1e-4 and mism == 0
    return {"rows": r, "ok": ok, "sum_err_over_S": sum_err, "lse_abs_err": float(np.max(lse_err)),
            "grad_err_over_G": grad_err, "knn_separated_mismatches": mism,
            "knn_near_ties": int(np.sum(~sep)), "knn_dist_rel_err": dist_err,
            "tolerances": "Sum 1e-4 S; LSE 1e-4 + 2^-20 |L|; grad 1e-4 G; K-min indices exact where separated"}


def _oracle_rows_for(orc, inp, s, target_s, wkey):
    M = inp["x"].shape[0]
    r0 = 8
    t0 = time.perf_counter()
    _oracle_step(orc, inp, s, np.arange(r0), wkey)
    dt = time.perf_counter() - t0
    return int(min(M, 4096, max(r0, r0 * target_s / max(dt, 1e-6))))


def cpu_baseline(inp, wkey, s, target_s=15.0):
    """The oracle's step on a seeded row subset (full N), sized to about target_s seconds
    (at most 4096 rows); returns the baseline, the oracle's outputs and the rows."""
    import oracle
    from symbolic_matrix_reductions_gb300 import workloads as W
    orc = oracle.load()
    r = _oracle_rows_for(orc, inp, s, target_s, wkey)
    rows = W.row_subset(inp["x"].shape[0], r, 12)
    t0 = time.perf_counter()
    ref = _oracle_step(orc, inp, s, rows, wkey)
    t = time.perf_counter() - t0
    N = inp["y"].shape[0]
    return {"value": 4 * r * N / t, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"seeded subset of {r} rows of the step's batch, full N={N}: Sum + LSE + grad-x + K-min "
                      f"(K={K_NN}) in fp64, {t:.1f} s"}, ref, rows


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    from symbolic_matrix_reductions_gb300 import workloads as W
    orc = oracle.load()
    inp = W.generate(args.workload, M=args.size[0], N=args.size[1]) if args.size else W.generate(args.workload)
    s = inp["sigma"]
    wkey = "w_log" if "w_log" in inp else "b"
    M, D = inp["x"].shape
    N, E = inp["y"].shape[0], inp["b"].shape[1]
    # each step samples about a fifth of --cpu-seconds (3 s by default), fewer when many steps
    per_step = max(0.05, min(args.cpu_seconds / 5.0, 150.0 / max(1, args.steps + args.warmup)))
    r = _oracle_rows_for(orc, inp, s, per_step, wkey)
    rows = W.row_subset(M, r, 12)
    for _ in range(args.warmup):
        _oracle_step(orc, inp, s, rows, wkey)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(orc, inp, s, rows, wkey)
    t = (time.perf_counter() - t0) / max(1, args.steps)
    value = 4 * r * N / t
    sample = (f"seeded subset of {r} rows of the {args.workload} batch per step, full N={N}: Sum + LSE + grad-x + "
              f"K-min in fp64")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": step_config(args.workload + (" resized" if args.size else ""), M, N, D, E, s, world),
            "rows_per_step": r,
            "timing": "ms_per_step is one sampled step (rows_per_step rows, full N); value = 4 rows N / that time",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=PRIMARY, help=f"workload of the step (default: {PRIMARY})")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target length of the CPU baseline sample")
    ap.add_argument("--size", type=lambda v: tuple(int(t) for t in v.split(",")), default=None,
                    help="M,N: the workload's distributions at another size (e.g. a smaller case to profile)")
    ap.add_argument("--lines", default=None,
                    help="run only these secondary lines (comma-separated op names as printed, e.g. "
                         "'max (gaussian)'), nothing else: a short command to profile one kernel")
    ap.add_argument("--no-secondary", action="store_true",
                    help="only the step (no D = 50 line, no secondary lines, no CPU baseline): a short command "
                         "to profile")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3   # at least three warm-up steps

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)

    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
