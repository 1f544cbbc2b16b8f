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
SPLIT_MODES = {"auto": 0, "prepass": 1, "onchip": 2}  # gemm_testing_set_split_mode
PAIR_MODES = {"auto": 0, "single": 1, "pair": 2}  # gemm_testing_set_cta_pair_mode
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
    "tc_gemm_pair_kernel": ["tc_gemm_pair.cu", "tc_common.cuh", "mhr_device.cuh", "tf32_split.cuh",
                            "tc_split.cuh"],
    "tc_gemm_kernel": ["tc_gemm_1cta.cu", "tc_common.cuh", "mhr_device.cuh", "tf32_split.cuh",
                       "tc_split.cuh"],
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
    """SM clock, power and clock-event (throttle) reasons of this process's GPU,
    sampled in the background: through NVML every 2 ms where libnvidia-ml can
    be loaded (read-only queries), else by nvidia-smi's own loop.  Each row is
    (sm MHz, max sm MHz, power W, hw_slowdown, hw_thermal_slowdown,
    sw_thermal_slowdown, sw_power_cap), the reasons as "Active"/"Not Active"."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits, in the order of the row's last four fields
    REASON_BITS = (0x8, 0x40, 0x20, 0x4)
    PERIOD_S = 0.002

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.source = None
        self._stop = threading.Event()
        import torch

        uuid = None
        try:
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            uuid = None
        if self._start_nvml(uuid):
            return
        cmd = ["nvidia-smi", *(["-i", uuid] if uuid else []), f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits", "-lms", "25"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi -lms 25"
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _start_nvml(self, uuid) -> bool:
        import ctypes

        if not uuid:
            return False
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                return False
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:  # 1 = SM clock
                return False
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            return False
        self._nv, self._h, self._max, self._reasons_fn = nv, h, mx.value, reasons_fn
        self.source = f"NVML every {self.PERIOD_S * 1e3:.0f} ms"
        self.t = threading.Thread(target=self._poll, daemon=True)
        self.t.start()
        return True

    def _poll(self):
        import ctypes

        nv, h = self._nv, self._h
        clk, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if (nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and
                    self._reasons_fn(h, ctypes.byref(rs)) == 0):
                pw = mw.value / 1e3 if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else 0.0
                flags = ["Active" if rs.value & b else "Not Active" for b in self.REASON_BITS]
                self.rows.append((time.time(), [str(clk.value), str(self._max), f"{pw:.1f}",
                                                *flags]))
            time.sleep(self.PERIOD_S)

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.time(), parts))

    def window(self, t0, t1):
        return [r for (t, r) in self.rows if t0 <= t <= t1]

    def stop(self):
        self._stop.set()
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
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "sm_mhz_min": min(sm) if sm else None}


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


def sampled_error(A, B, c_dev, M, N, K, seed, n_random=4096):
    """Normalised error max |C - C_ref| / sum_k |A_ik||B_kj| of the GPU result
    on sampled entries (random ones plus the first and last row and column),
    each computed by the CPU oracle."""
    import numpy as np
    import torch

    import oracle

    rng = np.random.default_rng(seed)
    r = np.concatenate([rng.integers(0, M, n_random), np.zeros(N, np.int64),
                        np.full(N, M - 1), np.arange(M), np.arange(M)]).astype(np.int64)
    c = np.concatenate([rng.integers(0, N, n_random), np.arange(N), np.arange(N),
                        np.zeros(M, np.int64), np.full(M, N - 1)]).astype(np.int64)
    ref, S = oracle.gemm_entries(A, B, r, c, M, N, K)
    got = c_dev[torch.from_numpy(r).to(c_dev.device), torch.from_numpy(c).to(c_dev.device)]
    got = got.cpu().numpy().astype(np.float64)
    ok = S > 0
    return {"value": float(np.max(np.abs(got - ref)[ok] / S[ok])) if ok.any() else 0.0,
            "entries": int(r.size), "all_finite": bool(np.all(np.isfinite(got)))}


def cublas_tf32_peak(dev, stream, flush, sampler, reps=10, n=8192):
    """The tf32 tensor-pipe ceiling measured on this GPU: cuBLAS single-pass
    tf32 (torch.matmul with TF32 allowed) on n^3 fp32 operands, uniform[-1, 1),
    best of `reps` calls, each timed with CUDA events after an L2 flush."""
    import torch

    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.rand(n, n, device=dev) * 2 - 1
        b = torch.rand(n, n, device=dev) * 2 - 1
        for _ in range(3):
            torch.matmul(a, b)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        torch.cuda.synchronize(dev)
        t0 = time.time()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            torch.matmul(a, b)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        ms = [e0.elapsed_time(e1) for e0, e1 in ev]
        flop = 2.0 * n ** 3
        out = {"tflops": flop / (min(ms) * 1e-3) / 1e12,
               "mean_tflops": flop / (sum(ms) / len(ms) * 1e-3) / 1e12,
               "how": f"cuBLAS single-pass tf32 (torch.matmul, TF32 allowed) at {n}^3 fp32, "
                      f"best of {reps} calls, L2 flushed before each, in this run"}
        if sampler:
            out["clocks"] = ClockSampler.summary(sampler.window(t0 - 0.05, t1 + 0.05))
        del a, b
        return out
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old


class Bench:
    """One GPU's measurement context: the library, the launching stream, the
    L2-flush buffer, the ranks and the clock sampler."""

    def __init__(self, lib, mhr, dev, stream, flush, ranks, sampler):
        self.lib, self.mhr, self.dev, self.stream = lib, mhr, dev, stream
        self.sh = stream.cuda_stream
        self.flush, self.ranks, self.sampler = flush, ranks, sampler

    def call(self, path, a, b, c, M, N, K):
        rc = getattr(self.lib, ENTRY[path])(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, K,
                                            N, N, self.sh)
        if rc != self.mhr.MHR_OK:
            raise self.mhr.GemmError(rc, ENTRY[path])

    def timed_steps(self, path, steps, kernel_events, a, b, c, M, N, K):
        """Per-step CUDA events around each call (L2 flushed before each,
        outside the events).  With kernel_events, events around the main
        kernel of each call instead: recorded between a pre-pass and the main
        kernel, they stop the main kernel from starting programmatically
        behind the pre-pass, so the step times of such a loop are not used."""
        import torch

        stream, lib = self.stream, self.lib
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e in ev:  # create the underlying events
            for x in e:
                x.record(stream)
        torch.cuda.synchronize(self.dev)
        for e0, e1 in ev:
            self.flush.zero_()
            if kernel_events:
                lib.gemm_testing_set_main_kernel_events(e0.cuda_event, e1.cuda_event)
            else:
                e0.record(stream)
            self.call(path, a, b, c, M, N, K)
            if not kernel_events:
                e1.record(stream)
        lib.gemm_testing_set_main_kernel_events(None, None)
        torch.cuda.synchronize(self.dev)
        return [e0.elapsed_time(e1) for e0, e1 in ev]

    def measure(self, path, a, b, c, M, N, K, steps, warmup):
        """Warm-up, then `steps` timed calls (the step time), then as many
        again with events around the main kernel alone; max over ranks."""
        import torch

        # a few clock samples before the timed region; taken before the
        # warm-up, so that the GPU is not left idle just before the first
        # timed step (with the idle gap there, 3-step runs of the 256^3
        # workload averaged 27-33 us per step against 13 us)
        time.sleep(0.2)
        for _ in range(warmup):
            self.call(path, a, b, c, M, N, K)
        rc = self.lib.gemm_check(self.sh)
        if rc != self.mhr.MHR_OK:
            raise self.mhr.GemmError(rc, "warm-up")
        main_kernel = self.lib.gemm_testing_last_main_kernel().decode()
        # our kernels per call, as counted by the library (pre-passes, zero
        # fills of split tiles, the main kernel)
        launches = self.lib.gemm_testing_last_launches()
        self.ranks.barrier()
        torch.cuda.synchronize(self.dev)
        t0 = time.time()
        step_ms = self.timed_steps(path, steps, False, a, b, c, M, N, K)
        torch.cuda.synchronize(self.dev)
        self.ranks.barrier()
        t1 = time.time()
        kern_ms = self.timed_steps(path, steps, True, a, b, c, M, N, K)
        rc = self.lib.gemm_check(self.sh)
        if rc != self.mhr.MHR_OK:
            raise self.mhr.GemmError(rc, "timed region")
        clocks = None
        if self.sampler:
            clocks = ClockSampler.summary(self.sampler.window(t0, t1))
        return {"ms_step": self.ranks.max(sum(step_ms) / len(step_ms)),
                "ms_kern": self.ranks.max(sum(kern_ms) / len(kern_ms)),
                "main_kernel": main_kernel, "launches_per_call": launches, "clocks": clocks,
                "t0": t0, "t1": t1}


def tensor_roofline(path, flop, meas, workload, tf32, sms):
    """Roofline of the dominant (main) kernel of a tensor-core path."""
    pk = peaks()
    if path == "bf16":
        tensor_flop, peak, src = flop, pk["bf16_tflops"], (
            f"{pk['source']} (MEASURED_PEAKS bf16 dense burst; the kernel is timed alone)")
    else:
        tensor_flop = 3 * flop  # three tf32 MMAs per product
        peak = tf32["tflops"] if tf32 else pk["bf16_tflops"] * TF32_OVER_BF16
        src = ("measured in this run: " + tf32["how"]) if tf32 else (
            f"{pk['source']} bf16 burst x 1.1/2.25 (nominal tf32/bf16 ratio)")
    achieved = tensor_flop / (meas["ms_kern"] * 1e-3) / 1e12
    kernel_name = meas["main_kernel"].split(" ")[0]
    out = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
           "frac": achieved / peak, "traffic": stored_traffic(kernel_name, workload),
           "kernel": meas["main_kernel"], "kernel_ms": meas["ms_kern"],
           "kernel_timing": "CUDA events around the main kernel on its stream, over a second "
                            "loop of the same steps right after the timed loop (events between "
                            "a pre-pass and the main kernel would serialise them)",
           "work": "3 x 2MNK tf32 MMA FLOPs (3xTF32)" if path != "bf16" else "2MNK bf16 FLOPs",
           "peak_source": src}
    if path != "bf16":
        nominal = pk["bf16_tflops"] * TF32_OVER_BF16
        out["peak_nominal_ratio"] = {"peak": nominal, "frac": achieved / nominal,
                                     "note": "bf16 burst x 1.1/2.25 (nominal dense tf32/bf16)"}
    per_clk = TENSOR_FLOP_PER_CLK_SM["bf16" if path == "bf16" else "tf32"]
    mhz = ((meas.get("clocks") or {}).get("sm_mhz")) or pk["sm_max_mhz"]
    pclk = per_clk * sms * mhz * 1e6 / 1e12
    out["peak_at_sm_clock"] = {
        "peak": pclk, "frac": achieved / pclk, "unit": "TFLOP/s",
        "note": f"{per_clk} dense FLOP/clk/SM x {sms} SMs x {mhz:.0f} MHz (median SM clock "
                "in the timed region)"}
    return out


def device_operands(w, dev):
    """Host operands of workload w, pinned host copies and device copies."""
    import numpy as np
    import torch

    M, N, K = w["M"], w["N"], w["K"]
    A_h, B_h, Ab_h, Bb_h = host_operands(w)
    if w["path"] == "bf16":
        a_pin = torch.from_numpy(Ab_h.view(np.int16).reshape(M, K)).pin_memory()
        b_pin = torch.from_numpy(Bb_h.view(np.int16).reshape(K, N)).pin_memory()
    else:
        a_pin = torch.from_numpy(A_h).pin_memory()
        b_pin = torch.from_numpy(B_h).pin_memory()
    return A_h, B_h, a_pin, b_pin, a_pin.to(dev), b_pin.to(dev)


def extra_workload(bench, name, args, tf32, sms, want_error):
    """A further workload of the default run: its own timed steps, main-kernel
    time, roofline and clocks, and the sampled GPU-vs-oracle error."""
    import torch

    w = WORKLOADS[name]
    M, N, K, path = w["M"], w["N"], w["K"], w["path"]
    A_h, B_h, _, _, a_d, b_d = device_operands(w, bench.dev)
    c_d = torch.empty((M, N), dtype=torch.float32, device=bench.dev)
    meas = bench.measure(path, a_d, b_d, c_d, M, N, K, args.steps, args.warmup)
    flop = 2.0 * M * N * K
    roof = tensor_roofline(path, flop, meas, name, tf32, sms)
    roof["cublas_same_run"] = cublas_reference(path, M, N, K, bench.dev, bench.stream,
                                               roof["achieved"], args.steps, bench.flush,
                                               w["dist"])
    out = {"workload": w["desc"], "M": M, "N": N, "K": K, "entry": ENTRY[path],
           "dtype": DTYPE[path], "dist": w["dist"], "seeds": list(w["seeds"]),
           "value": aggregate_tflops(bench.ranks.world, flop, meas["ms_step"]), "unit": "TFLOPS",
           "ms_per_step": meas["ms_step"], "main_kernel_ms": meas["ms_kern"],
           "roofline": roof, "clocks": meas["clocks"],
           "gpu_launches": meas["launches_per_call"] * args.steps}
    if want_error:
        bench.call(path, a_d, b_d, c_d, M, N, K)
        torch.cuda.synchronize(bench.dev)
        out["gpu_vs_oracle_sampled_error"] = sampled_error(A_h, B_h, c_d, M, N, K,
                                                           w["seeds"][0])
        out["gpu_vs_oracle_sampled_error"]["tolerance"] = 1e-2 if path == "bf16" else 1e-5
    del a_d, b_d, c_d
    torch.cuda.empty_cache()
    return out


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
    ap.add_argument("--no-extra", action="store_true",
                    help="with the default workload, skip the 8192^3 3xTF32 and bf16 entries")
    ap.add_argument("--ladder", action="store_true",
                    help="time the pages' naive/tiled kernels beside the build's paths at 4096^3")
    ap.add_argument("--split", default="auto", choices=sorted(SPLIT_MODES),
                    help="3xTF32 workloads: where the operands are split into tf32 parts "
                         "(auto: the library's choice; prepass: a split pre-pass; onchip: "
                         "converter warps of the CTA-pair kernel)")
    ap.add_argument("--cta-pair", default="auto", choices=sorted(PAIR_MODES),
                    help="tensor-core kernel (auto: the library's choice; single: the single-CTA "
                         "kernel; pair: the CTA-pair kernel)")
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
    lib.gemm_testing_set_split_mode(SPLIT_MODES[args.split])
    lib.gemm_testing_set_cta_pair_mode(PAIR_MODES[args.cta_pair])
    M, N, K = w["M"], w["N"], w["K"]
    path = w["path"]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    A_h, B_h, a_pin, b_pin, a_d, b_d = device_operands(w, dev)
    c_d = torch.empty((M, N), dtype=torch.float32, device=dev)
    c_pin = torch.empty((M, N), dtype=torch.float32).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sampler = ClockSampler(local) if rank == 0 else None
    bench = Bench(lib, mhr, dev, stream, flush, ranks, sampler)
    barrier = ranks.barrier
    max_over_ranks = ranks.max

    # ---------------------------------------------------------------- timed
    time.sleep(0.3)  # let the clock sampler start
    head = bench.measure(path, a_d, b_d, c_d, M, N, K, args.steps, args.warmup)
    ms_step, ms_kern = head["ms_step"], head["ms_kern"]
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
        bench.call(path, a_d, b_d, c_d, M, N, K)
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
    del sets[1]

    # ------------------------------------- the strict-fp32 SIMT path, same problem
    extra = {}
    if w["also"]:
        also = w["also"]
        bench.call(also, a_d, b_d, c_d, M, N, K)
        simt_label = lib.gemm_testing_last_main_kernel().decode()
        n_also = max(3, min(args.steps, 50))
        s_ms = bench.timed_steps(also, n_also, False, a_d, b_d, c_d, M, N, K)
        s_k = bench.timed_steps(also, n_also, True, a_d, b_d, c_d, M, N, K)
        simt_ms = max_over_ranks(sum(s_ms) / len(s_ms))
        simt_k = max_over_ranks(sum(s_k) / len(s_k))
        clock_mhz = peaks()["sm_max_mhz"]
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

    # ------------------------------------------- the tf32 tensor-pipe ceiling
    extras_wanted = args.workload == "c2" and not args.no_extra
    tf32 = None
    if path == "3xtf32" or extras_wanted:
        tf32 = cublas_tf32_peak(dev, stream, flush, sampler)

    # ---------------------------------------------------------------- roofline
    roofline = None
    if path in ("3xtf32", "bf16"):
        roofline = tensor_roofline(path, flop, head, args.workload, tf32, sms)
        roofline["cublas_same_run"] = cublas_reference(path, M, N, K, dev, stream,
                                                       roofline["achieved"], args.steps, flush,
                                                       w["dist"])

    # ------------------- the two 8192^3 tensor-core configurations of the target
    if extras_wanted:
        for name in ("c4", "c5"):
            extra[name] = extra_workload(bench, name, args, tf32, sms,
                                         want_error=rank == 0 and not args.no_cpu_baseline)

    # ---------------------------------------------------------------- CPU baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        rows, _ = calibrate_rows(A_h, B_h, args.cpu_budget, M)
        C_ref, t_cpu = oracle_rows(A_h, B_h, rows)
        # the same rows from the GPU
        bench.call(path, a_d, b_d, c_d, M, N, K)
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

    if sampler:
        sampler.stop()

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
                       **({"split": args.split} if path == "3xtf32" else {}),
                       **({"cta_pair": args.cta_pair} if args.cta_pair != "auto" else {})},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "cpu_tiled": cpu_tiled_line,
            "e2e": {"value": aggregate_tflops(world, flop, e2e_ms), "unit": "TFLOPS",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "serial_value": aggregate_tflops(world, flop, e2e_serial_ms),
                    "note": "per step: pinned host A, B -> device, C API call, C -> pinned host; "
                            "value pipelines consecutive steps over three streams, serial_value "
                            "runs them one after another on one stream"},
            "gpu_launches": head["launches_per_call"] * args.steps,
            "clocks": dict(head["clocks"] or {}, source=sampler.source if sampler else None),
            "tf32_peak": tf32,
            "paths": extra,
            "source_digest": source_digest(),
        }
        print(json.dumps(out), flush=True)
    ranks.close()


if __name__ == "__main__":
    main()
