"""Benchmark of the GEMM hot path: C = A * B through the C ABI on one GB300.

One step = one call of the library entry point on one seeded synthetic
problem, with inputs resident in HBM. The default workload is 4096^3 fp32
(uniform[-1, 1), seeds 2001/2002) through gemm_f32_3xtf32 -- the split
pre-pass, TMA ring, tcgen05 main loop and epilogue -- and the same problem
through the strict-fp32 SIMT path is reported beside it. Other workloads:
--workload c1 (256^3), c3 (3000 x 2050 x 1000), c4 (8192^3 3xTF32),
c5 (8192^3 bf16); s1 / s2 (512 x 512 x 8192, 3xTF32 / bf16: few tiles and a
long K, the single-CTA kernel's cluster split).

Prints ONE JSON line (rank 0). Metric: 2MNK / t in TFLOPS. L2 is flushed
(a 256 MiB write) between timed steps, outside the per-step CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2]
    python bench.py --impl reference ...   # the CPU oracle, timed as it stands

Under torchrun (N > 1) every rank runs its own independent problem on its own
GPU (weak scaling, no collective on the data path); the reported time is the
max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS (2MNK/t) at N=4096/8192 on 1 GB300; % of pipe roofline"

WORKLOADS = {
    "c1": dict(M=256, N=256, K=256, dist="uniform", seeds=(1001, 1002), path="3xtf32",
               also="f32", desc="fp32 square 256^3, uniform[-1,1)"),
    "c2": dict(M=4096, N=4096, K=4096, dist="uniform", seeds=(2001, 2002), path="3xtf32",
               also="f32", desc="fp32 square 4096^3, uniform[-1,1) (the pages' worked size)"),
    "c3": dict(M=3000, N=2050, K=1000, dist="normal", seeds=(3001, 3002), path="3xtf32",
               also="f32", desc="fp32 rectangular 3000x2050x1000, normal(0,1), ragged edges"),
    "c4": dict(M=8192, N=8192, K=8192, dist="uniform", seeds=(4001, 4002), path="3xtf32",
               also=None, desc="fp32-accurate 8192^3 via 3xTF32, uniform[-1,1)"),
    "c5": dict(M=8192, N=8192, K=8192, dist="normal", seeds=(5001, 5002), path="bf16",
               also=None, desc="bf16 inputs (normal(0,1) rounded), fp32 accumulate, 8192^3"),
    # extra measurements (not parity configurations): few tiles, long K
    "s1": dict(M=512, N=512, K=8192, dist="uniform", seeds=(6001, 6002), path="3xtf32",
               also="f32", desc="fp32 skinny-deep 512x512x8192 (few tiles, long K)"),
    "s2": dict(M=512, N=512, K=8192, dist="normal", seeds=(6101, 6102), path="bf16",
               also=None, desc="bf16 skinny-deep 512x512x8192 (few tiles, long K)"),
}
ENTRY = {"f32": "gemm_f32", "3xtf32": "gemm_f32_3xtf32", "bf16": "gemm_bf16_f32acc"}
DTYPE = {"f32": "f32", "3xtf32": "tf32x3", "bf16": "bf16"}
TF32_OVER_BF16 = 1.1 / 2.25   # nominal dense tensor rates (PFLOP/s) of GB300
# Dense tensor-core rate of one Blackwell SM per clock: 2.25 PFLOP/s bf16 over
# 152 SMs is 8192 FLOP/clk at ~1.8 GHz; tf32 runs at half the bf16 rate.
TENSOR_FLOP_PER_CLK_SM = {"bf16": 8192, "tf32": 4096}
FP32_LANES_PER_SM = 128
L2_FLUSH_BYTES = 256 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                sm_max_mhz=2070.0, source="fallback")


KERNEL_SOURCES = {  # the files whose text determines each kernel
    "tc_gemm_pair_kernel": ["tc_gemm_pair.cu", "tc_common.cuh", "mhr_device.cuh", "tf32_split.cuh"],
    "tc_gemm_kernel": ["tc_gemm_1cta.cu", "tc_common.cuh", "mhr_device.cuh"],
    "simt_f32_kernel": ["simt_f32.cu"],
    "split_vec_kernel": ["tc_prepass.cu", "tf32_split.cuh"],
}


def _code_only(text: str) -> str:
    """C++/CUDA source with comments removed and whitespace collapsed."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_digest(kernel: str | None = None) -> str:
    """Hash of the code (comments and layout ignored) of a kernel's source
    files (all sources if kernel is None), to tell whether stored ncu counters
    still apply."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "memory_hierarchy_reuse_gb300", "csrc")
    base = kernel.split("<")[0] if kernel else None
    files = KERNEL_SOURCES.get(base) if base else None
    for f in sorted(files or os.listdir(csrc)):
        h.update(f.encode())
        h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d[kernel][workload]
        if e.get("source_digest") != source_digest(kernel):
            return None
        return e["dram_bytes_per_launch"]
    except (KeyError, ValueError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 100 ms in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        import torch

        ident = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            ident = []
        cmd = ["nvidia-smi", *ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.time(), parts))

    def window(self, t0, t1):
        return [r for (t, r) in self.rows if t0 <= t <= t1]

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Ranks:
    """The bench's multi-process plumbing: one process per GPU, no collective
    on the data path -- only a barrier around the timed region and a max of
    each rank's time (NCCL on GPUs; gloo in the CPU tests)."""

    def __init__(self, world: int, device=None, backend: str = "nccl"):
        import torch

        self.world = world
        self.device = device if device is not None else torch.device("cpu")
        self.dist = None
        if world > 1:
            import torch.distributed as dist

            if not dist.is_initialized():
                if backend == "nccl":
                    dist.init_process_group("nccl", device_id=self.device)
                else:
                    dist.init_process_group(backend)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float) -> float:
        """Max of x over ranks (every rank gets it)."""
        if self.dist is None:
            return x
        import torch

        t = torch.tensor([x], device=self.device, dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


def aggregate_tflops(world: int, flop_per_rank: float, max_ms: float) -> float:
    """Whole-job throughput: every rank did flop_per_rank in at most max_ms."""
    return world * flop_per_rank / (max_ms * 1e-3) / 1e12


def oracle_rows(A, B, rows, nthreads=0):
    """CPU oracle on the first `rows` rows of C (the bounded CPU sample)."""
    import oracle

    t0 = time.perf_counter()
    C = oracle.gemm(A[:rows], B, nthreads=nthreads)
    return C, time.perf_counter() - t0


def calibrate_rows(A, B, budget_s, max_rows):
    """Rows of C the oracle computes in about budget_s seconds on this host."""
    r = 2
    _, t = oracle_rows(A, B, r)
    while t < 0.5 and r < max_rows:
        r = min(max_rows, r * 4)
        _, t = oracle_rows(A, B, r)
    return max(1, min(max_rows, int(r * budget_s / max(t, 1e-6)))), t / r


def host_operands(w):
    import seeded_inputs as si

    A = si.matrix(w["M"], w["K"], w["seeds"][0], w["dist"])
    B = si.matrix(w["K"], w["N"], w["seeds"][1], w["dist"])
    if w["path"] == "bf16":
        Ab, A = si.bf16_rne(A)
        Bb, B = si.bf16_rne(B)
        return A.reshape(w["M"], w["K"]), B.reshape(w["K"], w["N"]), Ab, Bb
    return A, B, None, None


def cublas_reference(path, M, N, K, dev, stream, achieved, steps, flush, dist):
    """cuBLAS (through torch) on the same shape in the same run, for context:
    tf32 for the 3xTF32 path (one tf32 pass); for the bf16 path bf16 inputs
    with fp32 output, the same operation as ours (torch.mm with
    out_dtype=float32), or bf16 output where that is not available.  Timed
    like our main kernel: `steps` calls, the L2 flushed before each, the mean
    of per-call CUDA events, on inputs drawn like the workload's (the tensor
    cores' power, and so the clock under the power cap, depends on the
    values).  Not a roofline denominator: the recipe's peak is."""
    import torch

    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        dt = torch.bfloat16 if path == "bf16" else torch.float32
        if dist == "uniform":
            a = (torch.rand(M, K, device=dev) * 2 - 1).to(dt)
            b = (torch.rand(K, N, device=dev) * 2 - 1).to(dt)
        else:
            a = torch.randn(M, K, device=dev).to(dt)
            b = torch.randn(K, N, device=dev).to(dt)
        kind = "tf32"
        fn = lambda: torch.matmul(a, b)  # noqa: E731
        if path == "bf16":
            kind = "bf16, bf16 output"
            try:
                torch.mm(a[:8, :8], b[:8, :8], out_dtype=torch.float32)
                fn = lambda: torch.mm(a, b, out_dtype=torch.float32)  # noqa: E731
                kind = "bf16, fp32 output"
            except (TypeError, RuntimeError):
                pass
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize(dev)
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
        tflops = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        return {"kind": kind, "tflops": tflops, "frac": achieved / tflops,
                "timing": f"mean of {steps} calls, L2 flushed before each, {dist} inputs"}
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old


def run_ladder(args):
    """The pages' ladder on this GPU at 4096^3 fp32 (uniform[-1, 1), seeds
    2001/2002): naive, 16x16 and 32x32 shared-memory tiles, the register-tiled
    SIMT kernel and the 3xTF32 tensor-core path, each timed with per-call
    CUDA events after warm-up (L2 flushed before each call), with the pages'
    global-load model 2MNK/T beside it. One JSON line."""
    import torch

    from memory_hierarchy_reuse_gb300 import build as mbuild

    mbuild.build()
    import memory_hierarchy_reuse_gb300 as mhr
    from memory_hierarchy_reuse_gb300 import model

    lib = mhr.load()
    w = WORKLOADS["c2"]
    M, N, K = w["M"], w["N"], w["K"]
    A_h, B_h, _, _ = host_operands(w)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    a, b = torch.from_numpy(A_h).to(dev), torch.from_numpy(B_h).to(dev)
    c = torch.empty((M, N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sh = stream.cuda_stream
    rungs = [("naive", lambda: lib.gemm_f32_ladder(0, a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                                   M, N, K, K, N, N, sh), 1),
             ("tiled16", lambda: lib.gemm_f32_ladder(1, a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                                     M, N, K, K, N, N, sh), 16),
             ("tiled32", lambda: lib.gemm_f32_ladder(2, a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                                     M, N, K, K, N, N, sh), 32),
             ("simt_f32", lambda: lib.gemm_f32(a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                               M, N, K, K, N, N, sh), 128),
             ("tc_3xtf32", lambda: lib.gemm_f32_3xtf32(a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                                       M, N, K, K, N, N, sh), 256)]
    out = {}
    flop = model.flops(M, N, K)
    for name, fn, T in rungs:
        for _ in range(args.warmup):
            assert fn() == 0
        torch.cuda.synchronize(dev)
        times = []
        steps = max(3, min(args.steps, 10 if name == "naive" else 30))
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            assert fn() == 0
            e1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1))
        assert lib.gemm_check(sh) == 0
        ms = sum(times) / len(times)
        out[name] = {"tflops": flop / (ms * 1e-3) / 1e12, "ms": ms, "tile": T,
                     "model_global_load_bytes": 4 * (model.naive_loads(M, N, K) if T == 1
                                                     else model.tiled_loads(M, N, K, T))}
    base = out["naive"]["tflops"]
    for v in out.values():
        v["speedup_vs_naive"] = v["tflops"] / base
    print(json.dumps({"metric": METRIC, "mode": "ladder", "unit": "TFLOPS", "n_gpus": 1,
                      "config": {"workload": w["desc"], "M": M, "N": N, "K": K,
                                 "l2": "flushed before every call"},
                      "ladder": out}), flush=True)


def run_reference(args, w, world, rank):
    """The oracle as it stands, timed on this host's cores: each step computes a
    bounded sample of rows of C; TFLOPS = 2 * rows * N * K / t."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    A, B, _, _ = host_operands(w)
    steps = args.steps
    per_step_budget = max(0.5, 100.0 / (steps + args.warmup))
    rows, _ = calibrate_rows(A, B, per_step_budget, w["M"])
    for _ in range(args.warmup):
        oracle_rows(A, B, rows)
    times = [oracle_rows(A, B, rows)[1] for _ in range(steps)]
    t = sum(times) / len(times)
    value = 2.0 * rows * w["N"] * w["K"] / t / 1e12
    cores = oracle.max_threads()
    sample = f"rows 0..{rows - 1} of C ({rows} x {w['N']} outputs, K={w['K']}) per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["desc"], "M": w["M"], "N": w["N"], "K": w["K"],
                   "entry": "CPU oracle (fp64 accumulate)", "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="c2", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="mhr", choices=["mhr", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ladder", action="store_true",
                    help="time the pages' naive/tiled kernels beside the build's paths at 4096^3")
    ap.add_argument("--split", default="auto", choices=["auto", "onchip"],
                    help="3xTF32 workloads: where the operands are split into tf32 parts "
                         "(auto: the library's choice, a pre-pass; onchip: inside the CTA-pair "
                         "kernel)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = WORKLOADS[args.workload]
    world, rank, local = dist_setup()
    if args.ladder:
        run_ladder(args)
        return

    if args.impl == "reference":
        run_reference(args, w, world, rank)
        return

    import numpy as np
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks(world, dev, "nccl")
    from memory_hierarchy_reuse_gb300 import build as mbuild

    mbuild.build()
    import memory_hierarchy_reuse_gb300 as mhr
    from memory_hierarchy_reuse_gb300 import model

    lib = mhr.load()
    if args.split == "onchip":
        lib.gemm_testing_set_split_mode(2)
    M, N, K = w["M"], w["N"], w["K"]
    A_h, B_h, Ab_h, Bb_h = host_operands(w)
    path = w["path"]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def device_operands(p):
        if p == "bf16":
            a = torch.from_numpy(Ab_h.view(np.int16).reshape(M, K)).pin_memory()
            b = torch.from_numpy(Bb_h.view(np.int16).reshape(K, N)).pin_memory()
        else:
            a = torch.from_numpy(A_h).pin_memory()
            b = torch.from_numpy(B_h).pin_memory()
        return a, b, a.to(dev), b.to(dev)

    a_pin, b_pin, a_d, b_d = device_operands(path)
    c_d = torch.empty((M, N), dtype=torch.float32, device=dev)
    c_pin = torch.empty((M, N), dtype=torch.float32).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    entry = getattr(lib, ENTRY[path])

    def call(p=path, a=None, b=None):
        a = a_d if a is None else a
        b = b_d if b is None else b
        rc = getattr(lib, ENTRY[p])(a.data_ptr(), b.data_ptr(), c_d.data_ptr(), M, N, K, K, N, N, sh)
        if rc != mhr.MHR_OK:
            raise mhr.GemmError(rc, ENTRY[p])

    def timed_steps(p, steps, kernel_events, a=None, b=None):
        """Per-step CUDA events around each call (L2 flushed before each, outside
        the events).  With kernel_events, events around the main kernel of each
        call instead: recorded between a pre-pass and the main kernel, they
        stop the main kernel from starting programmatically behind the
        pre-pass, so the step times of such a loop are not used."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e in ev:  # create the underlying events
            for x in e:
                x.record(stream)
        torch.cuda.synchronize(dev)
        for e0, e1 in ev:
            flush.zero_()
            if kernel_events:
                lib.gemm_testing_set_main_kernel_events(e0.cuda_event, e1.cuda_event)
            else:
                e0.record(stream)
            call(p, a, b)
            if not kernel_events:
                e1.record(stream)
        lib.gemm_testing_set_main_kernel_events(None, None)
        torch.cuda.synchronize(dev)
        return [e0.elapsed_time(e1) for e0, e1 in ev]

    barrier = ranks.barrier
    max_over_ranks = ranks.max

    sampler = ClockSampler(local) if rank == 0 else None
    # ---------------------------------------------------------------- warm-up
    for _ in range(args.warmup):
        call()
    rc = lib.gemm_check(sh)
    if rc != mhr.MHR_OK:
        raise mhr.GemmError(rc, "warm-up")
    main_kernel = lib.gemm_testing_last_main_kernel().decode()
    # our kernels per call, as counted by the library (pre-passes, zero fills
    # of split tiles, the main kernel)
    launches_per_call = lib.gemm_testing_last_launches()

    # ---------------------------------------------------------------- timed
    time.sleep(0.5)  # let the clock sampler start
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    step_ms = timed_steps(path, args.steps, kernel_events=False)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    # the main kernel alone, over as many steps again, right after (inside the
    # clock-sampling window); see timed_steps
    kern_ms = timed_steps(path, args.steps, kernel_events=True)
    rc = lib.gemm_check(sh)
    if rc != mhr.MHR_OK:
        raise mhr.GemmError(rc, "timed region")
    ms_step = max_over_ranks(sum(step_ms) / len(step_ms))
    ms_kern = max_over_ranks(sum(kern_ms) / len(kern_ms))
    flop = model.flops(M, N, K)
    value = aggregate_tflops(world, flop, ms_step)

    # ------------------------------------------------- end to end (host buffers)
    # Every step copies its inputs from pinned host memory, calls the C ABI and
    # reads C back to pinned host memory.  Serial: one stream, nothing overlaps.
    # Pipelined (the reported e2e): two device buffer sets and three streams,
    # so step i+1's host-to-device copy and step i-1's read-back run while step
    # i computes.
    e2e_steps = max(4, min(args.steps, 100))  # enough for the pipeline fill and drain to amortise
    h2d = a_pin.numel() * a_pin.element_size() + b_pin.numel() * b_pin.element_size()
    d2h = c_pin.numel() * 4
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        a_d.copy_(a_pin, non_blocking=True)
        b_d.copy_(b_pin, non_blocking=True)
        call()
        c_pin.copy_(c_d, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps)

    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = [(a_d, b_d, c_d, c_pin)]
    sets.append((torch.empty_like(a_d), torch.empty_like(b_d), torch.empty_like(c_d),
                 torch.empty_like(c_pin).pin_memory()))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for k in range(2):  # all buffers start free
        comp_done[k].record(stream)
        out_done[k].record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    t_e2e0 = torch.cuda.Event(enable_timing=True)
    t_e2e1 = torch.cuda.Event(enable_timing=True)
    t_e2e0.record(stream)
    s_in.wait_event(t_e2e0)
    s_out.wait_event(t_e2e0)
    for i in range(e2e_steps):
        k = i % 2
        ak, bk, ck, cpk = sets[k]
        s_in.wait_event(comp_done[k])          # inputs k no longer read
        with torch.cuda.stream(s_in):
            ak.copy_(a_pin, non_blocking=True)
            bk.copy_(b_pin, non_blocking=True)
        in_done[k].record(s_in)
        stream.wait_event(in_done[k])
        stream.wait_event(out_done[k])         # C k read back
        rc = getattr(lib, ENTRY[path])(ak.data_ptr(), bk.data_ptr(), ck.data_ptr(), M, N, K, K, N,
                                       N, sh)
        if rc != mhr.MHR_OK:
            raise mhr.GemmError(rc, "e2e")
        comp_done[k].record(stream)
        s_out.wait_event(comp_done[k])
        with torch.cuda.stream(s_out):
            cpk.copy_(ck, non_blocking=True)
        out_done[k].record(s_out)
    stream.wait_event(out_done[0])
    stream.wait_event(out_done[1])
    t_e2e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(t_e2e0.elapsed_time(t_e2e1) / e2e_steps)

    # ------------------------------------- the strict-fp32 SIMT path, same problem
    extra = {}
    if w["also"]:
        also = w["also"]
        call(also)
        simt_label = lib.gemm_testing_last_main_kernel().decode()
        n_also = max(3, min(args.steps, 50))
        s_ms = timed_steps(also, n_also, kernel_events=False)
        s_k = timed_steps(also, n_also, kernel_events=True)
        simt_ms = max_over_ranks(sum(s_ms) / len(s_ms))
        simt_k = max_over_ranks(sum(s_k) / len(s_k))
        clock_mhz = peaks()["sm_max_mhz"]
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        fp32_peak = sms * FP32_LANES_PER_SM * 2 * clock_mhz * 1e6 / 1e12
        extra[ENTRY[also]] = {
            "value": aggregate_tflops(world, flop, simt_ms), "unit": "TFLOPS", "ms_per_step": simt_ms,
            "roofline": {"bound": "alu", "achieved": flop / (simt_k * 1e-3) / 1e12,
                         "traffic": stored_traffic(simt_label.split(" ")[0], args.workload),
                         "kernel": simt_label,
                         "peak": fp32_peak, "unit": "TFLOP/s",
                         "frac": flop / (simt_k * 1e-3) / 1e12 / fp32_peak,
                         "peak_note": f"{sms} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2 x "
                                      f"{clock_mhz:.0f} MHz (max SM clock)"},
        }

    clocks = None
    if sampler:
        sampler.stop()
        clocks = ClockSampler.summary(sampler.window(t_wall0, t_wall1))

    # ---------------------------------------------------------------- roofline
    pk = peaks()
    if path == "bf16":
        tensor_flop, peak_tf, peak_note = flop, pk["bf16_tflops"], "bf16 dense, burst"
    elif path == "3xtf32":
        tensor_flop = 3 * flop
        peak_tf = pk["bf16_tflops"] * TF32_OVER_BF16
        peak_note = "tf32 = bf16 burst x 1.1/2.25 (nominal tf32/bf16 ratio); 3 MMAs per product"
    else:
        tensor_flop, peak_tf, peak_note = flop, None, ""
    kernel_name = main_kernel.split(" ")[0]
    achieved = tensor_flop / (ms_kern * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf if peak_tf else None,
                "traffic": stored_traffic(kernel_name, args.workload),
                "kernel": main_kernel, "kernel_ms": ms_kern,
                "kernel_timing": "CUDA events around the main kernel on its stream, over a second "
                                 "loop of the same steps right after the timed loop (events between "
                                 "a pre-pass and the main kernel would serialise them)",
                "peak_source": f"{pk['source']} ({peak_note})"}
    if path in ("3xtf32", "bf16"):
        roofline["cublas_same_run"] = cublas_reference(path, M, N, K, dev, stream, achieved,
                                                       args.steps, flush, w["dist"])
        # The nominal tf32 rate corresponds to a lower clock than this kernel
        # sustains, so also give the dense rate per SM per clock at the SM
        # clock sampled during the timed region.
        per_clk = TENSOR_FLOP_PER_CLK_SM["bf16" if path == "bf16" else "tf32"]
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = (clocks or {}).get("sm_mhz") or pk["sm_max_mhz"]
        pclk = per_clk * sms * mhz * 1e6 / 1e12
        roofline["peak_at_sm_clock"] = {
            "peak": pclk, "frac": achieved / pclk, "unit": "TFLOP/s",
            "note": f"{per_clk} dense FLOP/clk/SM x {sms} SMs x {mhz:.0f} MHz (median SM clock "
                    "in the timed region)"}

    # ---------------------------------------------------------------- CPU baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        rows, _ = calibrate_rows(A_h, B_h, args.cpu_budget, M)
        C_ref, t_cpu = oracle_rows(A_h, B_h, rows)
        # the same rows from the GPU (last timed call's output)
        call()
        torch.cuda.synchronize(dev)
        c_rows = c_d[:rows].cpu().numpy()
        S = np.abs(A_h[:rows].astype(np.float64)) @ np.abs(B_h.astype(np.float64))
        nerr = float(np.max(np.abs(c_rows.astype(np.float64) - C_ref) / np.maximum(S, 1e-300)))
        cpu = {"value": 2.0 * rows * N * K / t_cpu / 1e12, "unit": "TFLOPS",
               "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"rows 0..{rows - 1} of C ({rows} x {N} outputs, K={K}), "
                         f"{t_cpu:.1f} s of CPU work",
               "gpu_vs_sample_normalised_error": nerr}
        if args.workload in ("c1", "c2"):
            # the same oracle on one core, on a smaller sample (about 3 s)
            rows1 = max(1, min(M, int(rows * 3.0 / max(t_cpu * oracle.max_threads(), 1e-6))))
            _, t1 = oracle_rows(A_h, B_h, rows1, nthreads=1)
            cpu["single_core"] = {"value": 2.0 * rows1 * N * K / t1 / 1e12, "unit": "TFLOPS",
                                  "cores": 1,
                                  "sample": f"rows 0..{rows1 - 1} of C, {t1:.1f} s on one core"}

    # the pages' tiling on the host caches: a realistic CPU comparator (full problem)
    cpu_tiled_line = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import cpu_tiled

        cpu_tiled.build()
        cpu_tiled.gemm(A_h[:64], B_h)  # warm the threads and caches
        t0 = time.perf_counter()
        cpu_tiled.gemm(A_h, B_h)
        t_ct = time.perf_counter() - t0
        cpu_tiled_line = {"value": flop / t_ct / 1e12, "unit": "TFLOPS",
                          "cores": cpu_tiled.max_threads(), "kind": "cache-blocked fp32 CPU GEMM",
                          "sample": f"the whole {M}x{N}x{K} product, {t_ct:.2f} s"}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE[path], "data": "synthetic",
            "config": {"workload": w["desc"], "M": M, "N": N, "K": K, "entry": ENTRY[path],
                       "dist": w["dist"], "seeds": list(w["seeds"]),
                       "l2": "flushed before every timed step (256 MiB write, outside the step events)",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       **({"split": "on chip (CTA-pair kernel)" if args.split == "onchip"
                           else "pre-pass"} if path == "3xtf32" else {})},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "cpu_tiled": cpu_tiled_line,
            "e2e": {"value": aggregate_tflops(world, flop, e2e_ms), "unit": "TFLOPS",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "serial_value": aggregate_tflops(world, flop, e2e_serial_ms),
                    "note": "per step: pinned host A, B -> device, C API call, C -> pinned host; "
                            "value pipelines consecutive steps over three streams, serial_value "
                            "runs them one after another on one stream"},
            "gpu_launches": launches_per_call * args.steps,
            "clocks": clocks,
            "paths": extra,
            "source_digest": source_digest(),
        }
        print(json.dumps(out), flush=True)
    ranks.close()


if __name__ == "__main__":
    main()
