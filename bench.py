"""Benchmark of the deterministic, batch-invariant BF16 GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  The headline workload is the decode-shaped
product: M in {1, 4, 16, 64} rows against N = K = 4096 weights drawn N(0, 0.02),
split_k = 8 chosen from K alone.  One step decodes through four layers at each
batch size: for each M, four products through bigemm_run, each against a
different weight matrix of a pool of 16 (512 MiB, four times the 129 MB L2),
so a step streams every weight once from HBM, as decoding does.  The step is
replayed from a CUDA graph.  The metric is the whole job's TFLOP/s (2 M N K
per product).  After the timed region the results are checked: the device
error word, every product of the last step against an eager call (bits), and
sampled rows against the binary64 oracle ("checked").

Also reported (N = 1, rank 0):
  roofline        the few-row kernel (the whole product at M <= 32, the
                  dominant kernel): algorithmic bytes 2MK + 2KN + 4MN per
                  product over its measured duration, against the measured HBM
                  copy bandwidth; per-M whole-product times and fractions.
  e2e             one product per M through the public API with host buffers:
                  A and B copied from pinned host memory, C read back, every step.
  cpu_baseline    the CPU oracle (binary64 triple loop) on one product per M.
  workloads       the other shapes in brief: squares (tensor-core bound), long
                  K, the small product, linear layers, the Ozaki products;
                  the full record goes to a side file, bench_detail.json.
  roofline_tensor the 16384^3 product against the dense BF16 peak, with the
                  SM clock sampled during its own timed region.
  clocks          SM clock and throttle reasons sampled during the timed region.

--impl reference times the CPU oracle (the reference for this build) on the
same products and prints its line with "impl": "reference".

For N > 1 (torchrun) every rank runs the same step on its own GPU (replicas:
the product shards by rows or columns with no exchange); ranks meet at a
barrier on both sides of the timed region and the slowest rank's time sets
the job's throughput.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "TFLOP/s and % of dense BF16 peak (HBM % at small M), bit-exact batch-invariant"
UNIT = "TFLOP/s"
DECODE = workloads.WORKLOADS["decode"]
MS = tuple(DECODE["Ms"])
N_DEC = DECODE["N"]
K_DEC = DECODE["K"]
POOL = 16
PER_M = POOL // len(MS)          # products (layers) per batch size in one step
L2_BYTES = 129 * 1000 * 1000

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------- helpers --

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def flops_of(ms) -> float:
    """2 M N K summed over products of the decode shape with the given M."""
    return float(sum(2.0 * M * N_DEC * K_DEC for M in ms))


def decode_flops_per_step() -> float:
    """The timed step: PER_M products at each M."""
    return PER_M * flops_of(MS)


def decode_alg_bytes(M: int) -> float:
    """Algorithmic bytes of one decode product: read A and B once (bf16), write
    C once (fp32).  The split-K workspace round trip is overhead, not counted."""
    return 2.0 * M * K_DEC + 2.0 * K_DEC * N_DEC + 4.0 * M * N_DEC


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's time."""
    return flops_per_rank * world / max_seconds / 1e12


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of one GPU
    while the timed region runs: NVML through ctypes every 2 ms, else
    nvidia-smi every 200 ms.  Read-only: it changes no setting."""

    REASONS = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
        0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
        0x100: "display_clock_setting",
    }
    REJECT = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")

    def __init__(self, index: int):
        self.index = index
        self.samples = []          # (mhz, mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        self._proc = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) == 0:
                    self._nvml, self._handle = lib, h
                    mx = ctypes.c_uint()
                    if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = float(mx.value)
        except OSError:
            self._nvml = None

    def _poll_nvml(self):
        lib, h = self._nvml, self._handle
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mhz = ctypes.c_uint()
        mask = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and \
                    reasons_fn(h, ctypes.byref(mask)) == 0:
                self.samples.append((float(mhz.value), int(mask.value)))
            time.sleep(0.002)

    def start(self):
        self.samples = []
        self._stop.clear()
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self._thread.start()
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._proc = None

    def stop(self) -> dict:
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    mhz, mx, mask = float(parts[0]), float(parts[1]), int(parts[2], 16)
                except (ValueError, IndexError):
                    continue
                self.max_mhz = mx
                self.samples.append((mhz, mask))
        reasons = set()
        for _, mask in self.samples:
            for bit, name in self.REASONS.items():
                if mask & bit:
                    reasons.add(name)
        busy = [m for m, mask in self.samples if not mask & 0x1] or [m for m, _ in self.samples]
        return {
            "sm_mhz": statistics.median(busy) if busy else None,
            "sm_max_mhz": self.max_mhz,
            "reasons": sorted(reasons),
            "samples": len(self.samples),
            "source": "nvml" if self._nvml is not None else "nvidia-smi",
        }

    @classmethod
    def rejected(cls, clocks: dict) -> bool:
        if any(r in cls.REJECT for r in clocks.get("reasons", [])):
            return True
        mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
        return bool(mhz and mx and mhz < 0.5 * mx and not clocks.get("reasons"))


def nvml_index(local: int) -> int:
    """NVML index of CUDA device `local` (CUDA_VISIBLE_DEVICES may remap it)."""
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    if local < len(vis) and vis[local].isdigit():
        return int(vis[local])
    return local


def code_only(text: str) -> str:
    """C/C++ source with each comment and each run of whitespace replaced by
    one space: what the compiler sees of it, up to layout.  String literals (the
    inline PTX) are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(" " if c.isspace() else c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the kernels and of the host code that sizes and configures their
    launches, comments and whitespace excluded: an edit to a comment changes no
    kernel, so it does not make an ncu capture stale."""
    import hashlib
    h = hashlib.sha256()
    for f in ("kernels.cuh", "ptx.cuh", "ozaki.cuh", "skinny.cuh", "pair.cuh", "bigemm.cu"):
        with open(os.path.join(ROOT, "deterministic_invariant_gemm_gb300", "csrc", f),
                  encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode("utf-8"))
    return h.hexdigest()[:16]


TRAFFIC_PROFILE = "profiles/bigemm_skinny_decode_N4096_K4096.md"


def profiled_traffic():
    """DRAM bytes per launch of the few-row decode kernel from the committed
    ncu summary, or None when that capture was taken on other kernel sources."""
    path = os.path.join(ROOT, TRAFFIC_PROFILE)
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None
    for line in text.splitlines():
        if line.startswith("traffic_bytes_per_launch:"):
            fields = dict(f.split("=", 1) for f in line.split(":", 1)[1].split())
            if fields.pop("source_sha", None) != kernel_source_hash():
                return None
            return {int(k[1:]): int(v) for k, v in fields.items()}
    return None


def external_events_supported() -> bool:
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


# --------------------------------------------------------- decode workload --

class DecodeBench:
    """Inputs, outputs and the captured step graph of the headline workload.
    One step: for each batch size M in (1, 4, 16, 64), PER_M products through
    bigemm_run against PER_M different weight matrices -- decoding through
    PER_M layers at that batch size -- so a step streams every weight of the
    pool once (512 MiB, four times L2).  linear=True: the same step as linear
    layers, weights stored [N, K] with a bias, through bigemm_linear."""

    def __init__(self, dev: torch.device, linear: bool = False):
        import deterministic_invariant_gemm_gb300 as dig
        self.dig = dig
        self.dev = dev
        self.linear = linear
        seed = workloads.BASE_SEED + DECODE["index"]
        self.split = dig.bigemm_default_split_k(K_DEC)
        self.A = {M: workloads.normal_bf16((M, K_DEC), seed + M, DECODE["a_std"]).to(dev) for M in MS}
        shape = (N_DEC, K_DEC) if linear else (K_DEC, N_DEC)
        self.B = [workloads.normal_bf16(shape, seed + 1000 + j, DECODE["b_std"]).to(dev)
                  for j in range(POOL)]
        self.bias = [workloads.normal_bf16((N_DEC,), seed + 2000 + j, 0.02).to(dev)
                     for j in range(POOL)] if linear else None
        # one output per product of a step, so that every product can be checked
        self.C = {(M, r): torch.empty((M, N_DEC), dtype=torch.float32, device=dev)
                  for M in MS for r in range(PER_M)}
        self.ws_bytes = {M: dig.bigemm_workspace_bytes(M, N_DEC, K_DEC, self.split) for M in MS}
        self.ws = {M: torch.empty(max(self.ws_bytes[M], 16), dtype=torch.uint8, device=dev) for M in MS}
        self.path = {M: dig.bigemm_split_path(M, N_DEC, K_DEC, self.split) for M in MS}
        self.graph = None
        self.launches_per_step = 0

    @staticmethod
    def weight(idx: int, r: int) -> int:
        return idx * PER_M + r

    def product(self, M: int, j: int, C: torch.Tensor):
        dig = self.dig
        if self.linear:
            dig.bigemm_linear(self.A[M], self.B[j], self.bias[j], C, M, N_DEC, K_DEC, K_DEC, K_DEC,
                              N_DEC, self.split, 0, self.ws[M], self.ws_bytes[M])
        else:
            dig.bigemm_run(self.A[M], self.B[j], C, M, N_DEC, K_DEC, K_DEC, N_DEC, N_DEC,
                           self.split, self.ws[M], self.ws_bytes[M])

    def step(self, count_launches: bool = False):
        n = 0
        for idx, M in enumerate(MS):
            for r in range(PER_M):
                self.product(M, self.weight(idx, r), self.C[(M, r)])
                n += self.dig.bigemm_last_launch_count()
        if count_launches:
            self.launches_per_step = n

    def _capture(self, fn):
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return g

    def capture(self):
        """The timed graph holds kernels only, so consecutive launches keep
        their programmatic (early-launch) dependencies."""
        self.graph = self._capture(self.step)

    def run_steps(self, count: int):
        for _ in range(count):
            self.graph.replay()

    def chain_us(self, reps: int = 40):
        """Per M: the average time of one whole product (every kernel it
        launches) in a graph of POOL back-to-back products of that M against
        every weight of the pool, CUDA events around `reps` replays."""
        out = {}
        for M in MS:
            C = torch.empty((M, N_DEC), dtype=torch.float32, device=self.dev)

            def chain(M=M, C=C):
                for j in range(POOL):
                    self.product(M, j, C)
            g = self._capture(chain)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            out[M] = e0.elapsed_time(e1) * 1e3 / (reps * POOL)
        return out

    def verify(self) -> dict:
        """After the timed region: the device error word is clear, every
        product of the last replayed step equals the same product computed
        again by an eager call, bit for bit, and rows 0 and M - 1 of the last
        product of each M are within 1e-5 * sum_k |a_ik b_kj| of the binary64
        oracle (plus |bias_j| for linear layers)."""
        import numpy as np
        import oracle
        dig = self.dig
        torch.cuda.synchronize()
        status = int(dig.bigemm_device_status(reset=True))
        bits_ok = True
        for idx, M in enumerate(MS):
            for r in range(PER_M):
                again = torch.empty_like(self.C[(M, r)])
                self.product(M, self.weight(idx, r), again)
                torch.cuda.synchronize()
                bits_ok &= bool(torch.equal(again.view(torch.int32), self.C[(M, r)].view(torch.int32)))
        worst = 0.0
        for idx, M in enumerate(MS):
            j = self.weight(idx, PER_M - 1)
            rows = sorted({0, M - 1})
            A = self.A[M].cpu()
            B = self.B[j].cpu()
            if self.linear:
                Cref, D = oracle.linear_rows(A, B, self.bias[j].cpu(), M, N_DEC, K_DEC, rows=rows)
            else:
                Cref, D = oracle.gemm_rows(A, B, M, N_DEC, K_DEC, rows=rows)
            got = self.C[(M, PER_M - 1)][rows].double().cpu().numpy()
            with np.errstate(divide="ignore", invalid="ignore"):
                rel = np.where(D > 0, np.abs(got - Cref) / D, np.abs(got - Cref))
            worst = max(worst, float(rel.max()))
        return {"device_status": status, "bits_equal_eager": bits_ok,
                "oracle_max_err_over_D": worst, "oracle_ok": worst <= 1e-5,
                "checked": status == 0 and bits_ok and worst <= 1e-5}


def time_region(fn, steps: int, world: int) -> float:
    """Seconds for `steps` calls of fn(i), device-timed with CUDA events, with
    a barrier and a device synchronise on both sides; max over ranks."""
    import torch.distributed as dist
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    return max_over_ranks(e0.elapsed_time(e1) / 1e3, world)


def time_region_steps(bench: DecodeBench, steps: int, world: int) -> float:
    """time_region for the decode step graph."""
    import torch.distributed as dist
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    bench.run_steps(steps)
    e1.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    return max_over_ranks(e0.elapsed_time(e1) / 1e3, world)


def run_e2e(bench: DecodeBench, steps: int, warmup: int) -> dict:
    """The decode products through the public API with host buffers: every
    step copies one A and one B matrix per M from pinned host memory, runs the
    four products, and reads the four results back.  The copies go on their own
    stream and each product waits only for its own inputs, so a step's
    products and result reads overlap the copies still in flight (the
    host-to-device link, about 200 GB/s here, is the bound)."""
    dig = bench.dig
    hostA = {M: bench.A[M].cpu().pin_memory() for M in MS}
    hostB = [bench.B[j].cpu().pin_memory() for j in range(len(MS))]
    devA = {M: torch.empty_like(bench.A[M]) for M in MS}
    devB = [torch.empty_like(bench.B[0]) for _ in MS]
    hostC = {M: torch.empty((M, N_DEC), dtype=torch.float32).pin_memory() for M in MS}
    h2d = sum(t.numel() * t.element_size() for t in hostA.values()) + \
        sum(t.numel() * t.element_size() for t in hostB)
    d2h = sum(t.numel() * t.element_size() for t in hostC.values())
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    loaded = [torch.cuda.Event() for _ in MS]     # inputs of product idx are on the device
    consumed = [torch.cuda.Event() for _ in MS]   # product idx no longer reads them
    for ev in consumed:
        ev.record(compute)

    def one(_i):
        # nothing of this step starts before the compute stream reaches it (so
        # the timed region's first event precedes every copy it times)
        copy.wait_stream(compute)
        for idx, M in enumerate(MS):
            copy.wait_event(consumed[idx])
            with torch.cuda.stream(copy):
                devA[M].copy_(hostA[M], non_blocking=True)
                devB[idx].copy_(hostB[idx], non_blocking=True)
            loaded[idx].record(copy)
        for idx, M in enumerate(MS):
            compute.wait_event(loaded[idx])
            dig.bigemm_run(devA[M], devB[idx], bench.C[(M, 0)], M, N_DEC, K_DEC, K_DEC, N_DEC, N_DEC,
                           bench.split, bench.ws[M], bench.ws_bytes[M], stream=compute)
            consumed[idx].record(compute)
            hostC[M].copy_(bench.C[(M, 0)], non_blocking=True)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    secs = time_region(one, steps, 1)
    return {"value": flops_of(MS) * steps / secs / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": secs * 1e3 / steps,
            "step": "one product per M, its A and weight copied in from pinned host memory"}


def run_split_paths(dev) -> dict:
    """A split product that clusters on this device, timed through bigemm_run
    (one kernel: the cluster adds the segment partials in shared memory) and
    through the explicit two-kernel path (partial kernel + reduction kernel);
    both give the same bits.  Graphs of launches over a rotating weight pool
    larger than L2, CUDA events around 50 replays."""
    import deterministic_invariant_gemm_gb300 as dig
    out = {}
    for M, N, K, S in ((64, 3840, 4096, 8), (16, 2048, 4096, 8), (16, 4096, 4096, 4)):
        pool = (2 * L2_BYTES) // (2 * K * N) + 1
        A = workloads.normal_bf16((M, K), 1).to(dev)
        Bs = [workloads.normal_bf16((K, N), 10 + j, 0.02).to(dev) for j in range(pool)]
        C = torch.empty((M, N), device=dev)
        need = dig.bigemm_partial_workspace_bytes(M, N, K, S)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        s_eff = dig.bigemm_effective_split_k(K, S)

        def one_call():
            for B in Bs:
                dig.bigemm_run(A, B, C, M, N, K, K, N, N, S, ws, need)

        def two_kernels():
            for B in Bs:
                dig.bigemm_run_partial(A, B, M, N, K, K, N, S, ws, need)
                dig.bigemm_splitk_reduce(ws, s_eff, M, N, C, N, 0)

        res = {"path": {0: "unsplit", 1: "workspace", 2: "folded", 3: "cluster", 4: "skinny"}.get(
            dig.bigemm_split_path(M, N, K, S), "?"), "tile_n": dig.bigemm_tile_n(M, N, K, S),
            "weights": pool}
        for name, fn in (("bigemm_run_us", one_call), ("two_kernel_us", two_kernels)):
            s = torch.cuda.Stream(device=dev)
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                fn()
            torch.cuda.current_stream().wait_stream(s)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(50):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            res[name] = round(e0.elapsed_time(e1) * 1e3 / (50 * pool), 3)
        out["M%d_N%d_K%d_S%d" % (M, N, K, S)] = res
        del Bs
        torch.cuda.empty_cache()
    return out


def run_ozaki(dev, peaks) -> dict:
    """The Ozaki scheme's binary64 product (bigemm_ozaki_dgemm) on N(0, 1)
    float64 squares: time per call, the split's share, FP64-equivalent
    TFLOP/s (2 M N K per call), the tensor-core rate of the slice-pair
    products against the measured BF16 peak, and the error against cuBLAS's
    own binary64 product.  At 8192 also a Fast Mode sweep of d; at both
    sizes Fast Mode's automatic d (d = -1, chosen per element)."""
    import deterministic_invariant_gemm_gb300 as dig
    out = {}
    bf16_peak = peaks["bf16_tflops"]
    for n, iters in ((4096, 5), (8192, 3)):
        g = workloads.generator(1000 + n)
        A = torch.randn(n, n, generator=g, dtype=torch.float64).to(dev)
        B = torch.randn(n, n, generator=g, dtype=torch.float64).to(dev)
        C = torch.empty(n, n, dtype=torch.float64, device=dev)
        s = dig.bigemm_ozaki_default_slices(n)
        rho = dig.bigemm_ozaki_rho(n)
        need = dig.bigemm_ozaki_workspace_bytes(n, n, n, 0)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        ref = A @ B                                  # cuBLAS binary64
        scale = A.abs() @ B.abs()
        cases = ([s] if n != 8192 else [s, s - 1, s - 2, s - 3]) + [-1]
        res = {"slices": s, "rho": rho}
        for d in cases:
            def call(i, d=d):
                dig.bigemm_ozaki_dgemm(A, B, C, n, n, n, n, n, n, s, d, ws, need)
            for i in range(2):
                call(i)
            secs = time_region(call, iters, 1)
            per = secs / iters
            pairs = dig.bigemm_ozaki_pairs(s, d) if d > 0 else None
            err = float(((C - ref).abs() / scale).max())
            res["d%d" % d if d > 0 else "d_auto"] = {"pairs": pairs, "ms": round(per * 1e3, 3),
                              "fp64_equiv_tflops": round(2.0 * n ** 3 / per / 1e12, 2),
                              "max_err_vs_cublas_fp64_over_absAabsB": err}
        # the split alone (rows of A, columns of B), to separate it from the products
        rows_out = ws[: s * n * n * 2].view(torch.bfloat16)
        exps = torch.empty(2 * n, dtype=torch.int32, device=dev)

        def split(i):
            dig.bigemm_ozaki_split(A, n, n, n, 0, rho, s, rows_out, n, n, exps)
            dig.bigemm_ozaki_split(B, n, n, n, 1, rho, s, rows_out, n, n, exps[n:])
        for i in range(2):
            split(i)
        t_split = time_region(split, iters, 1) / iters
        full = res["d%d" % s]
        t_gemm = full["ms"] / 1e3 - t_split
        tensor = full["pairs"] * 2.0 * n ** 3 / t_gemm / 1e12
        res["split_ms"] = round(t_split * 1e3, 3)
        res["products_tensor_tflops"] = round(tensor, 1)
        res["products_frac_of_bf16_peak"] = round(tensor / bf16_peak, 4)
        # cuBLAS binary64 for context (this GPU's FP64 rate is low)
        def dgemm(i):
            torch.matmul(A, B, out=ref)
        dgemm(0)
        t64 = time_region(dgemm, 1, 1)
        res["cublas_fp64_ms"] = round(t64 * 1e3, 2)
        res["cublas_fp64_tflops"] = round(2.0 * n ** 3 / t64 / 1e12, 2)
        out["ozaki_%d" % n] = res
        del A, B, C, ws, ref, scale
        torch.cuda.empty_cache()
    return out


def run_decode_linear(dev, args) -> dict:
    """The headline step as linear layers (bigemm_linear, weights [N, K] plus a
    bias), timed the same way."""
    lb = DecodeBench(dev, linear=True)
    for i in range(3):
        lb.step()
    torch.cuda.synchronize()
    lb.capture()
    lb.run_steps(5)
    torch.cuda.synchronize()
    steps = max(50, args.steps // 4)
    secs = time_region_steps(lb, steps, 1)
    check = lb.verify()
    out = {"tflops": round(decode_flops_per_step() * steps / secs / 1e12, 2),
           "us_per_step": round(secs * 1e6 / steps, 2), "split_k": lb.split,
           "weights": "[N, K] + bias (bigemm_linear)", "checked": check["checked"]}
    del lb
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------ single workloads --

# name -> (M, N, K, split_k, bf16 out, value distribution, roofline bound)
SINGLE = {
    "small": (64, 256, 512, 1, False, "normal", "latency"),
    "square2048": (2048, 2048, 2048, 1, False, "uniform", "tensor"),
    "square4096": (4096, 4096, 4096, 1, False, "uniform", "tensor"),
    "square8192": (8192, 8192, 8192, 1, False, "uniform", "tensor"),
    "large16384": (16384, 16384, 16384, 1, True, "normal", "tensor"),
    # one decode product (the few-row kernel), for profiling one launch
    "decode_m1": (1, 4096, 4096, 8, False, "normal", "hbm"),
    "decode_m16": (16, 4096, 4096, 8, False, "normal", "hbm"),
    "decode_m64": (64, 4096, 4096, 8, False, "normal", "hbm"),
    "longk": (256, 256, 65536, 16, False, "normal", "hbm"),
    "longk8": (256, 256, 65536, 8, False, "normal", "hbm"),
    "longk32": (256, 256, 65536, 32, False, "normal", "hbm"),
    # linear layers, weights [N, K], bf16 out: bf16 and 8-bit float (E4M3) operands
    "linear8192": (8192, 8192, 8192, 1, True, "linear", "tensor"),
    "linearfp8_8192": (8192, 8192, 8192, 1, True, "linear_fp8", "tensor_fp8"),
    # split-K at a size whose tiles fill the GPU: segments summed in the CTA
    "fold8192": (8192, 8192, 8192, 16, False, "uniform", "tensor"),
    # binary64 product by the Ozaki scheme (bf16 slices on the tensor cores)
    "ozaki8192": (8192, 8192, 8192, 1, False, "ozaki", "tensor"),
    "ozaki4096": (4096, 4096, 4096, 1, False, "ozaki", "tensor"),
}


def run_single(name, args, world, rank, dev, peaks, peak_src):
    """One product per step through bigemm_run / bigemm_run_bf16out, inputs in
    rotating copies that together exceed L2."""
    import deterministic_invariant_gemm_gb300 as dig
    M, N, K, S, bf16, dist_name, bound = SINGLE[name]
    esize = {"linear_fp8": 1, "ozaki": 8}.get(dist_name, 2)
    in_bytes = esize * (M * K + K * N)
    copies = max(1, min(8, math.ceil(2 * L2_BYTES / in_bytes)))
    C = torch.empty((M, N), dtype=torch.bfloat16 if bf16 else torch.float32, device=dev)
    if dist_name == "ozaki":
        g = workloads.generator(98)
        AB = [(torch.randn(M, K, generator=g, dtype=torch.float64).to(dev),
               torch.randn(K, N, generator=g, dtype=torch.float64).to(dev))]
        copies = 1
        C = torch.empty((M, N), dtype=torch.float64, device=dev)
        need = dig.bigemm_ozaki_workspace_bytes(M, N, K, 0)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        launches = 4

        def call(i):
            a, b = AB[0]
            dig.bigemm_ozaki_dgemm(a, b, C, M, N, K, K, N, N, 0, 0, ws, need)
    elif dist_name in ("linear", "linear_fp8"):
        g = workloads.generator(99)
        AB = [(torch.randn(M, K, generator=g), torch.randn(N, K, generator=g)) for _ in range(copies)]
        td = torch.float8_e4m3fn if dist_name == "linear_fp8" else torch.bfloat16
        AB = [(a.to(td).to(dev), w.to(td).to(dev)) for a, w in AB]
        launches = 1

        def call(i):
            a, w = AB[i % copies]
            if dist_name == "linear_fp8":
                dig.linear_fp8(a, w, 1.0, out_dtype=C.dtype, out=C)
            else:
                dig.linear(a, w, out_dtype=C.dtype, out=C)
    else:
        AB = [workloads.pair(M, N, K, 4321 + c, dist=dist_name) for c in range(copies)]
        AB = [(a.to(dev), b.to(dev)) for a, b in AB]
        wsb = dig.bigemm_workspace_bytes(M, N, K, S)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        fn = dig.bigemm_run_bf16out if bf16 else dig.bigemm_run

        def call(i):
            a, b = AB[i % copies]
            fn(a, b, C, M, N, K, K, N, N, S, ws, wsb)

        call(0)
        launches = dig.bigemm_last_launch_count()

    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(nvml_index(dev.index or 0))
    sampler.start()
    secs = time_region(call, args.steps, world)
    clocks = sampler.stop()
    flops = 2.0 * M * N * K
    value = job_throughput(flops * args.steps, world, secs)
    per = secs / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"linear_fp8": "e4m3", "ozaki": "f64"}.get(dist_name, "bf16"), "data": "synthetic",
        "config": {"workload": "%s: M=%d N=%d K=%d split_k=%d, %s out, %s inputs" %
                   (name, M, N, K, S, "bf16" if bf16 else "fp32", dist_name),
                   "l2": "%d rotating input copies (%d MiB)" % (copies, copies * in_bytes >> 20),
                   "parallelism": "replicas"},
        "gpu_launches": launches * args.steps, "clocks": clocks,
    }
    if dist_name == "ozaki":
        # value: binary64-equivalent 2 M N K per call; the tensor cores run one
        # bf16 product per kept slice pair (split kernels included in the time)
        s_ = dig.bigemm_ozaki_default_slices(K)
        tens = dig.bigemm_ozaki_pairs(s_, s_) * flops
        peak = peaks["bf16_tflops"]
        line["config"]["slices"] = s_
        line["roofline"] = {"kernel": "ozaki split kernels + slice-pair kernel (%s)" % (
                                "bigemm_pair_kernel<kOutOzaki>" if (M >= 256 and K <= 4096)
                                else "bigemm_tc_kernel<kOutOzaki>"),
                            "bound": "tensor", "achieved": round(tens / per / 1e12, 1), "peak": peak,
                            "peak_source": peak_src, "unit": "TFLOP/s",
                            "frac": round(tens / per / 1e12 / peak, 4), "traffic": None}
    elif bound in ("tensor", "tensor_fp8"):
        # an 8-bit product takes the measured bf16 peak times the nominal ratio 2
        peak = peaks["bf16_tflops"] * (2.0 if bound == "tensor_fp8" else 1.0)
        line["roofline"] = {"kernel": "bigemm_pair_kernel" if dig.bigemm_uses_pair(M, N, K, S, bound == "tensor_fp8")
                            else "bigemm_tc_kernel", "bound": "tensor",
                            "achieved": round(flops / per / 1e12, 1), "peak": peak,
                            "peak_source": peak_src, "unit": "TFLOP/s",
                            "frac": round(flops / per / 1e12 / peak, 4), "traffic": None}
    elif bound == "hbm":
        alg = 2.0 * (M * K + K * N) + 4.0 * M * N
        kern = {0: "bigemm_tc_kernel", 1: "bigemm_tc_kernel + splitk_reduce_kernel",
                3: "bigemm_tc_kernel (cluster)", 4: "bigemm_skinny_kernel"}.get(
                    dig.bigemm_split_path(M, N, K, S), "bigemm_tc_kernel")
        line["roofline"] = {"kernel": kern, "bound": "hbm",
                            "achieved": round(alg / per / 1e9, 1), "peak": peaks["hbm_gbs"],
                            "peak_source": peak_src, "unit": "GB/s",
                            "frac": round(alg / per / 1e9 / peaks["hbm_gbs"], 4), "traffic": None}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ long K --

def run_longk(dev, peaks) -> dict:
    """M = N = 256, K = 65536 with split_k = 8, 16, 32 through bigemm_run (the
    path and tile width the library picks -- at this shape narrow tiles and
    the workspace + reduction kernel; the bits are the same every way), and the atomic-add
    contrast at the same splits: its time, and how many distinct results ten
    runs on the same inputs give (the workspace path gives one).  Four input
    copies rotate (256 MiB > L2)."""
    import deterministic_invariant_gemm_gb300 as dig
    M = N = 256
    K = 65536
    copies = 4
    AB = [workloads.pair(M, N, K, 4321 + c, dist="normal") for c in range(copies)]
    AB = [(a.to(dev), b.to(dev)) for a, b in AB]
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    alg = 2.0 * (M * K + K * N) + 4.0 * M * N
    out = {"shape": [M, N, K], "input_copies": copies,
           "alg_bytes": alg, "peak_gbs": peaks["hbm_gbs"]}
    # The accumulate chain, measured: one CTA computing a 128 x 64 tile of a
    # one-row product over all of K (M = 1, N = 64, split_k = 1) runs 4 * K/64
    # dependent K = 16 MMAs into one accumulator while its loads (12 KB per
    # K block for one SM) take a fraction of that; its time over the MMA count
    # is the latency of one dependent MMA.  A K segment of L blocks cannot take
    # less than 4 L of them, whatever the tile width or the memory system.
    kb = -(-K // 64)
    a1 = AB[0][0][:1].contiguous()
    b1 = AB[0][1][:, :64].contiguous()
    c1 = torch.empty((1, 64), dtype=torch.float32, device=dev)

    def chain_call(i):
        dig.bigemm_run(a1, b1, c1, 1, 64, K, K, 64, 64, 1, None, 0)

    for i in range(2):
        chain_call(i)
    t_mma = time_region(chain_call, 10, 1) / 10 / (4 * kb)
    out["mma_chain_ns"] = round(t_mma * 1e9, 1)
    out["mma_chain_probe"] = "1 x 64 x %d, split_k 1, tile width %d: %d dependent MMAs" % (
        K, dig.bigemm_tile_n(1, 64, K, 1), 4 * kb)
    iters = 40
    for S in (8, 16, 32):
        wsb = dig.bigemm_workspace_bytes(M, N, K, S)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)

        def call(i):
            a, b = AB[i % copies]
            dig.bigemm_run(a, b, C, M, N, K, K, N, N, S, ws, wsb)

        def atomic(i):
            a, b = AB[i % copies]
            dig.bigemm_run_atomic_splitk(a, b, C, M, N, K, K, N, N, S)

        floor_s = -(-kb // S) * 4 * t_mma
        res = {"path": {0: "unsplit", 1: "workspace", 2: "folded", 3: "cluster", 4: "skinny"}.get(
            dig.bigemm_split_path(M, N, K, S), "?"), "tile_n": dig.bigemm_tile_n(M, N, K, S),
            "chain_floor_us": round(floor_s * 1e6, 2)}
        for key, fn in (("bigemm_run", call), ("atomic", atomic)):
            for i in range(3):
                fn(i)
            secs = time_region(fn, iters, 1) / iters
            res[key] = {"us": round(secs * 1e6, 2),
                        "hbm_frac": round(alg / secs / 1e9 / peaks["hbm_gbs"], 4),
                        "tflops": round(2.0 * M * N * K / secs / 1e12, 2),
                        "frac_of_chain_floor": round(floor_s / secs, 4)}
            distinct = set()
            for _ in range(10):
                fn(0)
                torch.cuda.synchronize()
                distinct.add(hash(C.cpu().numpy().tobytes()))
            res[key]["distinct_results_in_10_runs"] = len(distinct)
        out["s%d" % S] = res
        del ws
    del AB, C
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------- other shapes --

def run_other_workloads(dev, peaks) -> dict:
    """Large squares (tensor-core bound) and long K, each a few timed calls on
    inputs larger than L2 (rotating copies where one copy fits)."""
    import deterministic_invariant_gemm_gb300 as dig
    out = {}
    bf16_peak = peaks["bf16_tflops"]
    # (calls per timed region: a few milliseconds of back-to-back products, so
    # that the region's first launch latency is not a visible share)
    cases = [("square_2048", 2048, 2048, 2048, 1, False, "uniform", 300),
             ("square_4096", 4096, 4096, 4096, 1, False, "uniform", 60),
             ("square_8192", 8192, 8192, 8192, 1, False, "uniform", 10),
             ("large_16384_bf16out", 16384, 16384, 16384, 1, True, "normal", 5),
             # split products large enough to fold their segments in the CTA
             ("square_4096_split8_folded", 4096, 4096, 4096, 8, False, "uniform", 60),
             ("square_8192_split16_folded", 8192, 8192, 8192, 16, False, "uniform", 10),
             ("prefill_1024x4096x4096_split8_folded", 1024, 4096, 4096, 8, False, "normal", 200)]
    for name, M, N, K, S, bf16, dist_name, iters in cases:
        in_bytes = 2 * (M * K + K * N)
        copies = max(1, min(8, math.ceil(2 * L2_BYTES / in_bytes)))
        AB = [workloads.pair(M, N, K, 4321 + c, dist=dist_name) for c in range(copies)]
        AB = [(a.to(dev), b.to(dev)) for a, b in AB]
        C = torch.empty((M, N), dtype=torch.bfloat16 if bf16 else torch.float32, device=dev)
        wsb = dig.bigemm_workspace_bytes(M, N, K, S)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        fn = dig.bigemm_run_bf16out if bf16 else dig.bigemm_run

        def call(i):
            a, b = AB[i % copies]
            fn(a, b, C, M, N, K, K, N, N, S, ws, wsb)

        for i in range(3):
            call(i)
        sampler = ClockSampler(nvml_index(dev.index or 0))
        sampler.start()
        secs = time_region(call, iters, 1)
        clocks = sampler.stop()
        tflops = 2.0 * M * N * K * iters / secs / 1e12
        out[name] = {"tflops": round(tflops, 2), "frac_of_bf16_peak": round(tflops / bf16_peak, 4),
                     "ms": round(secs * 1e3 / iters, 4), "split_k": S,
                     "out": "bf16" if bf16 else "fp32", "input_copies": copies,
                     "launches": dig.bigemm_last_launch_count(), "clocks": clocks,
                     "cta_pairs": bool(dig.bigemm_uses_pair(M, N, K, S))}
        del AB, C, ws
        torch.cuda.empty_cache()
    # The small product (64 x 256 x 512, split_k 1, FP32 out): a latency case
    # with no roofline target.  Per-call device time from a CUDA graph of 50
    # back-to-back calls (programmatic launches overlap their prologues), and
    # the time of one call alone between two events on its stream.
    M, N, K = 64, 256, 512
    a, b = workloads.pair(M, N, K, workloads.BASE_SEED)
    a, b = a.to(dev), b.to(dev)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(device=dev)
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(50):
            dig.bigemm_run(a, b, C, M, N, K, K, N, N, 1, None, 0, stream=st)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(20):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    chained_us = e0.elapsed_time(e1) * 1e3 / (20 * 50)
    alone = []
    with torch.cuda.stream(st):
        for _ in range(30):
            e0.record(st)
            dig.bigemm_run(a, b, C, M, N, K, K, N, N, 1, None, 0, stream=st)
            e1.record(st)
            st.synchronize()
            alone.append(e0.elapsed_time(e1) * 1e3)
    alone.sort()
    out["small_64x256x512"] = {"us_per_call_chained": round(chained_us, 2),
                               "us_one_call_median": round(alone[len(alone) // 2], 2),
                               "tflops_chained": round(2.0 * M * N * K / (chained_us * 1e-6) / 1e12, 3),
                               "split_k": 1, "out": "fp32", "launches": 1}
    del g, a, b, C
    # linear layers, weights [N, K]: BF16 and 8-bit floats (E4M3).  The FP8
    # peak is the measured BF16 peak times the nominal FP8 / BF16 ratio (2).
    fp8_peak = 2.0 * bf16_peak
    for name, n, fp8 in (("linear_bf16_8192", 8192, False), ("linear_fp8_e4m3_8192", 8192, True),
                         ("linear_fp8_e4m3_16384", 16384, True)):
        g = workloads.generator(99)
        x = torch.randn(n, n, generator=g)
        w = torch.randn(n, n, generator=g)
        if fp8:
            x, w = x.to(torch.float8_e4m3fn).to(dev), w.to(torch.float8_e4m3fn).to(dev)
        else:
            x, w = x.to(torch.bfloat16).to(dev), w.to(torch.bfloat16).to(dev)
        C = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
        call = (lambda i: dig.linear_fp8(x, w, 1.0, out_dtype=torch.bfloat16, out=C)) if fp8 else \
            (lambda i: dig.linear(x, w, out_dtype=torch.bfloat16, out=C))
        for i in range(3):
            call(i)
        iters = 10 if n <= 8192 else 4
        secs = time_region(call, iters, 1)
        tflops = 2.0 * n ** 3 * iters / secs / 1e12
        peak = fp8_peak if fp8 else bf16_peak
        out[name] = {"tflops": round(tflops, 2), "frac_of_peak": round(tflops / peak, 4),
                     "peak": peak, "peak_note": "measured bf16 x 2 (nominal fp8/bf16 ratio)"
                     if fp8 else "measured bf16", "ms": round(secs * 1e3 / iters, 4),
                     "out": "bf16", "inputs": "fp8 e4m3" if fp8 else "bf16",
                     "cta_pairs": bool(dig.bigemm_uses_pair(n, n, n, 1, fp8))}
        del x, w, C
        torch.cuda.empty_cache()
    return out


# -------------------------------------------------------------- CPU oracle --

_ORACLE_INPUTS = {}


def oracle_decode_step():
    """The decode step computed by the CPU oracle: the four products against
    four weight matrices (the same seeded inputs as the GPU step).  Returns
    (seconds, threads); input generation is outside the timing."""
    import oracle
    if not _ORACLE_INPUTS:
        seed = workloads.BASE_SEED + DECODE["index"]
        _ORACLE_INPUTS["A"] = {M: workloads.normal_bf16((M, K_DEC), seed + M, DECODE["a_std"]) for M in MS}
        _ORACLE_INPUTS["B"] = [workloads.normal_bf16((K_DEC, N_DEC), seed + 1000 + j, DECODE["b_std"])
                               for j in range(len(MS))]
        oracle.build()
    As, Bs = _ORACLE_INPUTS["A"], _ORACLE_INPUTS["B"]
    t0 = time.perf_counter()
    for idx, M in enumerate(MS):
        oracle.gemm_rows(As[M], Bs[idx], M, N_DEC, K_DEC)
    return time.perf_counter() - t0, oracle.num_threads()


def cpu_baseline(budget_s: float = 10.0) -> dict:
    """The oracle, as it stands, timed on this host's cores on whole decode
    steps, repeated until about `budget_s` seconds of CPU work."""
    total, reps, threads = 0.0, 0, 1
    while total < budget_s or reps == 0:
        dt, threads = oracle_decode_step()
        total += dt
        reps += 1
        if reps >= 200:
            break
    value = flops_of(MS) * reps / total / 1e12
    return {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d whole decode steps (M=1,4,16,64 x N=K=4096, binary64 triple loop, "
                      "OpenMP over rows), %.1f s" % (reps, total)}


def cpu_baseline_configs() -> dict:
    """The oracle on the other workloads, as per-config context:
    the small product and long K in full, the squares on a 256-row sample of
    A (every column of C; the full-size time extrapolated by rows).  The
    oracle also forms D = sum |a b| for the tolerance, so it does twice the
    arithmetic counted here."""
    import oracle
    oracle.build()
    out = {}
    cases = [("small_64x256x512", "small", 64, 256, 512, None),
             ("square_2048", "square", 2048, 2048, 2048, 256),
             ("square_4096", "square", 4096, 4096, 4096, 256),
             ("square_8192", "square", 8192, 8192, 8192, 256),
             ("large_16384", "large", 16384, 16384, 16384, 256),
             ("longk_256x256x65536", "longk", 256, 256, 65536, None)]
    threads = 1
    for name, wname, M, N, K, sample in cases:
        w = workloads.WORKLOADS[wname]
        dist = {"small": "normal", "square": "uniform", "large": "normal", "longk": "normal"}[wname]
        rows_m = M if sample is None else sample
        # only the sampled rows of A are drawn (their values do not change the time)
        A, B = workloads.pair(rows_m, N, K, workloads.BASE_SEED + w["index"], dist=dist)
        t0 = time.perf_counter()
        oracle.gemm_rows(A, B, rows_m, N, K)
        dt = time.perf_counter() - t0
        threads = oracle.num_threads()
        flops = 2.0 * rows_m * N * K
        out[name] = {"tflops": flops / dt / 1e12, "seconds": round(dt, 3), "rows_timed": rows_m,
                     "full_size_seconds": round(dt * M / rows_m, 2),
                     "extrapolated": sample is not None, "cores": threads}
    return out


def run_reference(args, world: int, rank: int):
    """--impl reference: the CPU oracle on the decode step, K timed steps."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_decode_step()
    total, threads = 0.0, 1
    for _ in range(args.steps):
        dt, threads = oracle_decode_step()
        total += dt
    value = flops_of(MS) * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(8),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "%d whole decode steps on the host cores" % args.steps},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def decode_config(split: int) -> dict:
    return {"workload": "decode-shaped BF16 GEMM: M in {1,4,16,64}, N=K=4096, A~N(0,1), "
                        "B~N(0,0.02) bf16, FP32 out, split_k=%d from K only; a step is %d products "
                        "(layers) at each M" % (split, PER_M),
            "M": list(MS), "N": N_DEC, "K": K_DEC, "split_k": split, "products_per_M": PER_M,
            "l2": "every product of a step multiplies a different weight of a pool of %d "
                  "(%d MiB > L2): inputs larger than L2" % (POOL, POOL * N_DEC * K_DEC * 2 >> 20),
            "parallelism": "replicas"}


# ------------------------------------------------------------ the record --

def write_detail(detail: dict) -> str:
    """The full per-workload record (Ozaki d-sweeps, split-path A/Bs, per-config
    CPU times, ...) goes to a side file; the JSON line keeps a summary."""
    out_dir = os.path.join(ROOT, "gpurun_out")
    try:
        os.makedirs(out_dir, exist_ok=True)
        path = os.path.join(out_dir, "bench_detail.json")
        with open(path, "w") as f:
            json.dump(detail, f, indent=1)
        return os.path.relpath(path, ROOT)
    except OSError:
        return None


def compact_workloads(detail: dict, peaks: dict, peak_src: str):
    """Per shape only what the metric needs: TFLOP/s and the fraction of the
    dense BF16 peak for the tensor-bound shapes, time and HBM fraction for the
    long-K ones; and a roofline object for the largest square."""
    out = {}
    for k in ("square_2048", "square_4096", "square_8192", "large_16384_bf16out",
              "square_8192_split16_folded", "prefill_1024x4096x4096_split8_folded"):
        d = detail.get(k)
        if d:
            out[k] = {"tflops": d["tflops"], "frac": d["frac_of_bf16_peak"], "ms": d["ms"],
                      "pairs": d.get("cta_pairs", False)}
    for k in ("linear_bf16_8192", "linear_fp8_e4m3_16384"):
        d = detail.get(k)
        if d:
            out[k] = {"tflops": d["tflops"], "frac": d["frac_of_peak"], "ms": d["ms"],
                      "pairs": d.get("cta_pairs", False)}
    lk = detail.get("longk_256x256x65536")
    if lk:
        out["longk_256x256x65536"] = {
            "s%d" % S: {"us": lk["s%d" % S]["bigemm_run"]["us"],
                        "hbm_frac": lk["s%d" % S]["bigemm_run"]["hbm_frac"],
                        "frac_of_chain_floor": lk["s%d" % S]["bigemm_run"]["frac_of_chain_floor"],
                        "distinct_in_10": lk["s%d" % S]["bigemm_run"]["distinct_results_in_10_runs"],
                        "atomic_distinct_in_10": lk["s%d" % S]["atomic"]["distinct_results_in_10_runs"]}
            for S in (8, 16, 32)}
    sm = detail.get("small_64x256x512")
    if sm:
        out["small_64x256x512"] = {"us_chained": sm["us_per_call_chained"], "us_alone": sm["us_one_call_median"]}
    dl = detail.get("decode_linear")
    if dl:
        out["decode_linear"] = {"tflops": dl["tflops"], "us_per_step": dl["us_per_step"], "checked": dl["checked"]}
    for n in (4096, 8192):
        oz = detail.get("ozaki_%d" % n)
        if oz:
            full = oz["d%d" % oz["slices"]]
            out["ozaki_%d" % n] = {"ms": full["ms"], "fp64_equiv_tflops": full["fp64_equiv_tflops"],
                                   "products_frac_of_bf16_peak": oz["products_frac_of_bf16_peak"]}
            auto = oz.get("d_auto")
            if auto:
                out["ozaki_%d" % n]["fast_auto_d"] = {"ms": auto["ms"], "fp64_equiv_tflops": auto["fp64_equiv_tflops"],
                                                      "max_err": auto["max_err_vs_cublas_fp64_over_absAabsB"]}
    big = detail.get("large_16384_bf16out")
    roof = None
    if big:
        kname = ("bigemm_pair_kernel<kOutBF16> (16384^3 on CTA pairs, bf16 out)" if big.get("cta_pairs")
                 else "bigemm_tc_kernel<kOutBF16> (16384^3, bf16 out)")
        roof = {"kernel": kname, "bound": "tensor",
                "achieved": big["tflops"], "peak": peaks["bf16_tflops"], "peak_source": peak_src,
                "peak_kind": "burst (the product is timed alone)", "unit": "TFLOP/s",
                "frac": round(big["tflops"] / peaks["bf16_tflops"], 4), "traffic": None,
                "clocks": big.get("clocks")}
    return out, roof


# ------------------------------------------------------------------- main --

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other shapes, e2e and the CPU baseline")
    ap.add_argument("--workload", default="decode", choices=("decode",) + tuple(SINGLE),
                    help="decode (the headline step) or one of the other workload shapes")
    ap.add_argument("--pair-mode", default="auto", choices=("never", "auto", "always"),
                    help="when products run on CTA pairs (the 2-SM kernel): the library's rule "
                         "(auto, the default), never, or whenever they can -- for comparisons and "
                         "profiles; the arithmetic is the same either way")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    if args.pair_mode != "auto":
        import deterministic_invariant_gemm_gb300 as dig
        dig.bigemm_set_pair_mode({"never": dig.PAIR_NEVER, "always": dig.PAIR_ALWAYS}[args.pair_mode])
    if args.workload != "decode":
        run_single(args.workload, args, world, rank, dev, peaks, peak_src)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    bench = DecodeBench(dev)
    bench.step(count_launches=True)       # eager warm-up (loads the module)
    for i in range(args.warmup - 1):
        bench.step()
    torch.cuda.synchronize()
    bench.capture()
    bench.run_steps(args.warmup)
    torch.cuda.synchronize()

    sampler = ClockSampler(nvml_index(local))
    remeasured = False
    for attempt in range(2):
        sampler.start()
        secs = time_region_steps(bench, args.steps, world)
        clocks = sampler.stop()
        if not ClockSampler.rejected(clocks):
            break
        remeasured = True
    check = bench.verify()
    chain = bench.chain_us()

    flops_step = decode_flops_per_step()
    value = job_throughput(flops_step * args.steps, world, secs)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": decode_config(bench.split),
        "gpu_launches": bench.launches_per_step * args.steps,
        "clocks": clocks, "checked": check,
    }
    if remeasured:
        line["clocks"]["remeasured"] = True
    # The dominant kernel: the few-row kernel, which is the whole product at
    # M = 1, 4, 16 (one launch each; 12 of the step's 16 products).
    few = [M for M in MS if bench.path[M] == 4]   # PATH_SKINNY
    alg = sum(decode_alg_bytes(M) for M in few)
    dur_s = sum(chain[M] for M in few) / 1e6
    achieved = alg / dur_s / 1e9
    step_bytes = PER_M * sum(decode_alg_bytes(M) for M in MS)
    line["roofline"] = {
        "kernel": "bigemm_skinny_kernel (split_k=%d summed in 8-CTA clusters), M=%s"
                  % (bench.split, ",".join(str(M) for M in few)),
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
        "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
        "traffic": None,
        "bytes_per_launch": {str(M): decode_alg_bytes(M) for M in few},
        "timing": "CUDA events around graph replays of %d back-to-back products per M (every "
                  "weight of the pool); achieved = sum of bytes / sum of times" % POOL,
        "whole_product_us": {str(M): round(chain[M], 3) for M in MS},
        "whole_product_hbm_frac": {str(M): round(decode_alg_bytes(M) / (chain[M] / 1e6) / 1e9 /
                                                 peaks["hbm_gbs"], 4) for M in MS},
        "paths": {str(M): {0: "unsplit", 1: "workspace", 2: "folded", 3: "cluster", 4: "skinny"}.get(
            bench.path[M], "?") for M in MS},
        "step_hbm_frac": round(step_bytes / (secs / args.steps) / 1e9 / peaks["hbm_gbs"], 4),
    }
    traffic = profiled_traffic()
    if traffic:
        tm = {M: v for M, v in traffic.items() if M in few}
        if tm:
            line["roofline"]["traffic"] = sum(tm.values()) / len(tm)
            line["roofline"]["traffic_source"] = (
                "dram__bytes_read.sum + dram__bytes_write.sum per launch, ncu capture of the current "
                "kernel sources (%s), mean of M=%s" % (TRAFFIC_PROFILE, ",".join(str(m) for m in sorted(tm))))
    if rank == 0 and world == 1 and not args.no_extras:
        line["e2e"] = run_e2e(bench, max(20, args.steps // 20), 5)
        del bench
        torch.cuda.empty_cache()
        detail = run_other_workloads(dev, peaks)
        detail["longk_256x256x65536"] = run_longk(dev, peaks)
        detail["decode_linear"] = run_decode_linear(dev, args)
        detail["split_paths"] = run_split_paths(dev)
        detail.update(run_ozaki(dev, peaks))
        line["cpu_baseline"] = cpu_baseline()
        detail["cpu_baseline_per_config"] = cpu_baseline_configs()
        line["workloads"], line["roofline_tensor"] = compact_workloads(detail, peaks, peak_src)
        line["workloads"]["detail_file"] = write_detail(detail)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
