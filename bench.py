"""Benchmark of the fused attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one fa_fwd call over the whole workload (every (batch, head) and
every query row): the complete hot path.  Backward workloads (bwd_*): one
step = one fa_bwd call (dQ, dK, dV for a seeded dO, three kernels) on the
forward outputs computed once before timing; 10*B*H*N^2*d flops per step.
The K timed steps are captured once into a CUDA graph and replayed (the
same kernels, without the host's per-call work between them; --no-graph
times plain launches).  Default workload: B=2, H=32, N=8192, d=128, bf16 inputs drawn N(0,1)*0.5 from a seed (the compute-bound
headline shape).  The metric is attention-forward TFLOP/s counting
4*B*H*N^2*d flops per step.

`value` is device-timed (CUDA events on the launching stream around exactly K
steps, inputs resident in HBM; 539 MB of inputs+outputs per step exceed the
129 MB L2).  `e2e` is the same metric through fa_fwd_host, the C-ABI call on
HOST tensors (pinned): each step copies Q, K, V to the GPU and O, lse back,
overlapped with the computation chunk by chunk inside the call (backward
workloads: fa_bwd_host the same way).  `roofline` compares the kernel with the measured dense bf16
tensor peak.  `cpu_baseline` times the fp64 CPU oracle on a bounded sample of
the same workload on the host cores (rank 0 only).

Multi-GPU (torchrun, one process per GPU): each rank runs its own independent
copy of the workload (attention heads are independent; no collective on the
data path): weak scaling, value = all ranks' flops / max-over-ranks time.

`--impl reference` times the CPU oracle (the only reference implementation
there is) on bounded samples of the workload and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (4·B·H·N²·d) on 1 GB300 and % of dense tensor peak"
METRIC_BWD = "attention bwd TFLOP/s (10·B·H·N²·d) on 1 GB300 and % of dense tensor peak"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
NOMINAL_TF32_OVER_BF16 = 0.5  # dense TF32 rate relative to dense bf16 (1.1 vs 2.25 PFLOP/s nominal)


# ------------------------------------------------------------------ helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_max(value: float, dist, device=None) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_workload(w, rank: int):
    """The workload a rank runs: the same shape with its own seed (weak
    scaling, independent replicas: rank r draws its inputs from seed
    w.seed + 17 r, so no two ranks compute the same problem)."""
    return dataclasses.replace(w, seed=w.seed + 17 * rank)


def aggregate(ms_local: float, flops_rank: float, dist, device=None):
    """Whole-job figures from one rank's timed region: the slowest rank's
    time (max over ranks) and every rank's work (sum), so value = all ranks'
    flops / max-over-ranks time.  Returns (ms_total, flops_all, TFLOP/s)."""
    ms_total = reduce_max(ms_local, dist, device)
    flops_all = reduce_sum(flops_rank, dist, device)
    return ms_total, flops_all, flops_all / (ms_total * 1e-3) / 1e12


def result_line(w, world: int, steps: int, warmup: int, ms_total: float, value: float, *,
                splits: int, launch: str, frac_of_peak, roofline: dict, e2e: dict,
                gpu_launches: int, clocks: dict, entry: str) -> dict:
    """The JSON line rank 0 prints for our arm (every rank's figures already
    aggregated by `aggregate`)."""
    return {
        "metric": METRIC_BWD if w.backward else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms_total / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(config_of(w, world, splits), launch=launch, entry_point=entry),
        "frac_of_peak": frac_of_peak,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


SHARED_SOURCES = ("fa_ptx.cuh", "fa_internal.h", "fa_host.h")


def kernel_source_hash(backward: bool = False) -> str:
    """Hash of the CUDA sources a pass's kernels and launches are built from:
    ties a stored ncu traffic figure to the kernel it was measured on.
    Forward: fa_fwd*, fa_dec*, fa_decode*, fa_merge*, fa_api.cu; backward:
    fa_bwd*; both: the headers they share."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_04_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        mine = (name.startswith("fa_bwd") if backward
                else name.startswith(("fa_fwd", "fa_dec", "fa_merge")) or name == "fa_api.cu")
        if mine or name in SHARED_SOURCES:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str, backward: bool = False):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            lines = [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]
    except OSError:
        return None
    want = kernel_source_hash(backward)
    for ln in lines:
        kv = dict(x.split("=", 1) for x in ln.split() if "=" in x)
        if kv.get("workload") == workload and kv.get("kernel_hash") == want:
            try:
                return float(kv["dram_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # start timing only once the sampler produces rows
        t0 = time.time()
        while self.proc is not None and self.count() == 0 and time.time() - t0 < 3.0:
            time.sleep(0.01)
        self.start_rows = self.count()
        return self

    def count(self) -> int:
        """Rows written so far."""
        try:
            with open(self.file.name) as f:
                return sum(1 for r in f if r.strip())
        except OSError:
            return 0

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        return False

    def summary(self, busy_threshold_frac: float = 0.0):
        try:
            with open(self.file.name) as f:
                rows = [r.strip() for r in f if r.strip()]
        finally:
            try:
                os.unlink(self.file.name)
            except OSError:
                pass
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names[1:], parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        # rows written before the timed region started are left out
        skip = min(getattr(self, "start_rows", 0), max(0, len(sm) - 1))
        sm, smax = sm[skip:], smax[skip:]
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi every 100 ms"}


class NvmlClockSampler(ClockSampler):
    """The same record from NVML in-process (the driver's libnvidia-ml, read
    only): SM clock, its maximum and the clock event reasons every 2 ms, so
    that a timed region of a few tens of milliseconds (a short graph) still
    holds tens of samples where nvidia-smi's 100 ms cadence gives one.
    `open` returns None where NVML is unavailable; nvidia-smi is then used."""
    REASON_BITS = ((0x8, "hw_slowdown"), (0x40, "hw_thermal_slowdown"), (0x20, "sw_thermal_slowdown"),
                   (0x4, "sw_power_cap"))
    INTERVAL_S = 0.002

    @classmethod
    def open(cls, gpu_index: int):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
        except (OSError, AttributeError):
            return None
        handle = ctypes.c_void_p()
        found = False
        try:  # the CUDA device's NVML handle, through its PCI address
            import torch
            pr = torch.cuda.get_device_properties(gpu_index)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            found = lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(handle)) == 0
        except Exception:  # noqa: BLE001 - fall back to the index
            found = False
        if not found and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(handle)) != 0:
            return None
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        if reasons is None:
            return None
        smp = cls(gpu_index)
        smp.lib, smp.handle, smp.reasons_fn = lib, handle, reasons
        return smp

    def _sample(self):
        import ctypes
        clk, mx, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        if (self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) != 0 or
                self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) != 0 or
                self.reasons_fn(self.handle, ctypes.byref(rs)) != 0):
            return None
        return (clk.value, mx.value, rs.value)

    def _run(self):
        while not self._stop.is_set():
            r = self._sample()
            if r is not None:
                self.rows.append(r)
            self._stop.wait(self.INTERVAL_S)

    def __enter__(self):
        import threading
        self.rows = []
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 1.0:
            time.sleep(0.001)
        self.start_rows = len(self.rows)
        return self

    def count(self) -> int:
        return len(self.rows)

    def __exit__(self, *exc):
        self._stop.set()
        self._thread.join(timeout=2.0)
        return False

    def summary(self, busy_threshold_frac: float = 0.0):
        rows = self.rows[min(self.start_rows, max(0, len(self.rows) - 1)):]
        try:
            self.lib.nvmlShutdown()
        except Exception:  # noqa: BLE001
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({name for _, _, bits in rows for bit, name in self.REASON_BITS if bits & bit})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "source": "NVML every 2 ms"}


def clock_sampler(gpu_index: int):
    """NVML in-process where it loads, else nvidia-smi."""
    return NvmlClockSampler.open(gpu_index) or ClockSampler(gpu_index)


# --------------------------------------------------------------- CPU oracle
def cpu_oracle_rate(w, q, k, v, dout, target_s: float, max_rows: int | None = None):
    """Time the fp64 oracle on seeded rows of the workload, sized to run
    about `target_s` seconds on every host core.  Returns (TFLOP/s, cores,
    rows, seconds)."""
    import oracle
    from exact_tiled_attention_04_gb300 import inputs as I
    cores = oracle.default_threads()
    rows = I.sample_rows(w, 64, seed_offset=1000)
    t0 = time.perf_counter()
    oracle_rows(w, q, k, v, dout, rows)
    dt = max(time.perf_counter() - t0, 1e-6)
    n = int(64 * target_s / dt)
    n = max(cores, min(n, max_rows or n, w.B * w.H * w.N))
    rows = I.sample_rows(w, n, seed_offset=1001)
    t0 = time.perf_counter()
    oracle_rows(w, q, k, v, dout, rows)
    dt = time.perf_counter() - t0
    return row_flops(w, rows) / dt / 1e12, cores, n, dt


def row_flops(w, rows) -> float:
    """Flops the oracle spends on the given (b, h, i) query rows: forward,
    4 d per visible key (scores, weighted sum of V); backward (dQ of the
    row), 6 d per visible key (scores, dP, dS K)."""
    import numpy as np
    i = np.asarray(rows)[:, 2].astype(np.float64)
    visible = np.full_like(i, float(w.Nkv))
    if w.causal:
        visible = np.clip(i + (w.Nkv - w.N) + 1, 0, w.Nkv)
    return float((6.0 if w.backward else 4.0) * w.d * visible.sum())


def oracle_rows(w, q, k, v, dout, rows):
    """The oracle on sampled query rows: the forward (O, lse) or, for a
    backward workload, the rows' dQ."""
    import oracle
    if w.backward:
        return oracle.attention_bwd_dq_rows_f64(q, k, v, dout, float(w.scale), rows, causal=w.causal)
    return oracle.attention_f64_ex(q, k, v, float(w.scale), rows=rows, causal=w.causal)


def sample_text(w, n, cores, secs=None):
    what = ("dQ of" if w.backward else "") + f" {n} seeded query rows of the workload (of {w.B * w.H * w.N})"
    how = "fp64, recomputed softmax" if w.backward else "fp64 three-pass"
    return what.strip() + f", {how}, {cores} threads" + (f", {secs:.1f} s" if secs is not None else "")


# ------------------------------------------------------------------- arms
def run_reference(args, w):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the workload's query rows."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from exact_tiled_attention_04_gb300 import inputs as I
    q, k, v = I.make(w)
    dout = I.make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed) if w.backward else None
    cores = oracle.default_threads()
    budget_s = 150.0 / max(1, args.steps + args.warmup)
    rows = I.sample_rows(w, 16, seed_offset=2000)
    t0 = time.perf_counter()
    oracle_rows(w, q, k, v, dout, rows)
    per_row = max((time.perf_counter() - t0) / 16, 1e-7)
    n = int(max(1, min(4096, w.B * w.H * w.N, budget_s / per_row)))
    for i in range(args.warmup):
        oracle_rows(w, q, k, v, dout, I.sample_rows(w, n, seed_offset=3000 + i))
    total = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        rows = I.sample_rows(w, n, seed_offset=4000 + i)
        oracle_rows(w, q, k, v, dout, rows)
        total += row_flops(w, rows)
    dt = time.perf_counter() - t0
    value = total / dt / 1e12
    sample = sample_text(w, n, cores) + " per step"
    line = {
        "impl": "reference", "metric": METRIC_BWD if w.backward else METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129e6          # GB300 L2
FLUSH_BYTES = 512 << 20   # written between timed steps when the inputs fit in L2


def input_bytes(w) -> float:
    """Bytes a step reads as inputs: q, k, v (forward); q, k, v, o, dO, lse
    (backward)."""
    elem = 4 if w.dtype == "f32" else 2
    q = w.B * w.H * w.N * w.d * elem
    kv = 2 * w.B * w.H_kv * w.Nkv * w.d * elem
    return float(q + kv if not w.backward else 3 * q + kv + 4 * w.B * w.H * w.N)


def needs_flush(w) -> bool:
    return input_bytes(w) <= L2_BYTES


def uses_fa_fwd(w) -> bool:
    """Whether the benchmark's forward step calls fa_fwd (the workload fits
    its signature and takes the automatic plan) rather than fa_fwd_ex."""
    return w.H_kv == w.H and w.N == w.Nkv and w.splits == 0


def config_of(w, n_gpus: int, splits: int = 1):
    what = "q,k,v,o,dO,lse" if w.backward else "q,k,v"
    nin = input_bytes(w)
    l2 = (f"inputs larger than L2: {what} = {nin / 1e6:.0f} MB read per step (L2 129 MB), no flush"
          if not needs_flush(w) else
          f"inputs fit in L2 ({what} = {nin / 1e6:.1f} MB): a {FLUSH_BYTES >> 20} MB buffer is written "
          f"before every timed step, outside its CUDA events")
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype,
           "inputs": f"seeded N(0,1) x {w.factor}", "scale": float(w.scale), "l2": l2,
           "parallelism": f"independent replica per GPU x{n_gpus}"}
    if w.general:
        cfg.update({"H_kv": w.H_kv, "N_kv": w.Nkv})
    if w.causal:
        cfg["causal"] = True
    if splits == 0 and not w.backward:
        cfg["splits"] = ("automatic: the library's plan for this GPU (key partitions of underfilled "
                         "launches and of a partly filled last wave merged inside thread-block clusters)")
    elif splits > 1:
        cfg["splits"] = splits
    if w.backward:
        cfg["pass"] = "backward: dQ, dK, dV for a seeded dO (forward outputs o, lse computed once)"
    return cfg


def run_ours(args, w):
    import numpy as np
    import torch
    from exact_tiled_attention_04_gb300 import binding as fab
    from exact_tiled_attention_04_gb300 import inputs as I

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, "nccl")
    fab.load()

    # per-rank inputs (weak scaling: every rank its own seeded copy)
    wr = rank_workload(w, rank)
    q, k, v = I.make(wr)

    def host_tensor(x):
        if w.dtype == "bf16":
            return torch.from_numpy(I.bf16_bits(x).view(np.int16)).view(torch.bfloat16)
        if w.dtype == "f16":
            return torch.from_numpy(np.ascontiguousarray(x, np.float32).astype(np.float16))
        return torch.from_numpy(np.ascontiguousarray(x, np.float32))

    hq, hk, hv = (host_tensor(x).pin_memory() for x in (q, k, v))
    dq, dk, dv = (t.to(dev) for t in (hq, hk, hv))
    do = torch.empty_like(dq)
    dlse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    dt_code = {"bf16": fab.FA_DTYPE_BF16, "f16": fab.FA_DTYPE_F16, "f32": fab.FA_DTYPE_F32}[w.dtype]
    if w.causal:
        dt_code |= fab.FA_FLAG_CAUSAL
    scale = float(w.scale)
    splits = w.splits  # 0: the library's automatic plan for this GPU
    wbytes = fab.fa_fwd_ex_workspace_size(w.B, w.H, w.N, w.Nkv, w.d, splits)
    work = torch.empty(max(wbytes, 16), dtype=torch.uint8, device=dev)  # caller-owned scratch
    launches = 0

    # The forward step is fa_fwd, the library's primary entry point, wherever
    # the workload fits its signature (one key/value head per query head,
    # as many keys as queries, the automatic plan); grouped-head and decode
    # workloads go through fa_fwd_ex with the automatic plan.
    use_fa_fwd = uses_fa_fwd(w)

    def forward():
        if use_fa_fwd:
            st = fab.fa_fwd(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), do.data_ptr(), dlse.data_ptr(),
                            w.B, w.H, w.N, w.d, scale, dt_code, sp)
            if st != fab.FA_OK:
                raise fab.FAError(st, "fa_fwd")
            return
        st = fab.fa_fwd_ex(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), do.data_ptr(), dlse.data_ptr(),
                           w.B, w.H, w.H_kv, w.N, w.Nkv, w.d, scale, dt_code, splits,
                           work.data_ptr() if wbytes else None, wbytes, sp)
        if st != fab.FA_OK:
            raise fab.FAError(st, "fa_fwd_ex")

    entry_name = ("fa_bwd" if w.backward else "fa_fwd" if use_fa_fwd
                  else "fa_fwd_ex (num_splits = 0, caller workspace)")
    if not w.backward:
        # the step's kernels: the forward kernel, plus a split last wave or a merge kernel
        kernels_per_step = (fab.fa_fwd_launches(w.B, w.H, w.N, w.d, dt_code) if use_fa_fwd else
                            fab.fa_fwd_ex_launches(w.B, w.H, w.H_kv, w.N, w.Nkv, w.d, dt_code, splits))
        step_fn = forward
        # end to end: fa_fwd_host on pinned host tensors (q, k, v up; o and
        # lse back, overlapped with the computation inside the call)
        ho = torch.empty_like(hq).pin_memory()
        hl = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
        host_bytes = fab.fa_fwd_host_workspace_size(w.B, w.H, w.H_kv, w.N, w.Nkv, w.d, dt_code)
        host_work = torch.empty(host_bytes + 256, dtype=torch.uint8, device=dev)
        host_ws = (host_work.data_ptr() + 255) // 256 * 256

        def e2e_step():
            st = fab.fa_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(), hl.data_ptr(),
                                 w.B, w.H, w.H_kv, w.N, w.Nkv, w.d, scale, dt_code, host_ws, host_bytes, sp)
            if st != fab.FA_OK:
                raise fab.FAError(st, "fa_fwd_host")

        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    else:
        # the forward outputs o, lse the backward consumes, computed once
        with torch.cuda.stream(stream):
            forward()
        torch.cuda.synchronize(dev)
        hdout = host_tensor(I.make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=wr.seed)).pin_memory()
        ddout = hdout.to(dev)
        ho, hl = do.cpu().pin_memory(), dlse.cpu().pin_memory()
        gq, gk, gv = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
        bwd_bytes = fab.fa_bwd_workspace_size(w.B, w.H, w.N, w.d)
        bwork = torch.empty(bwd_bytes, dtype=torch.uint8, device=dev)
        kernels_per_step = 3  # prep, main, dQ conversion

        def step_fn():
            st = fab.fa_bwd(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), do.data_ptr(), ddout.data_ptr(),
                            dlse.data_ptr(), gq.data_ptr(), gk.data_ptr(), gv.data_ptr(), w.B, w.H, w.H_kv,
                            w.N, w.Nkv, w.d, scale, dt_code, bwork.data_ptr(), bwd_bytes, sp)
            if st != fab.FA_OK:
                raise fab.FAError(st, "fa_bwd")

        # end to end: fa_bwd_host on pinned host tensors (q, k, v, o, dO, lse
        # up; dq, dk, dv back, overlapped with the computation inside the call)
        hgq, hgk, hgv = (torch.empty_like(t).pin_memory() for t in (hq, hk, hv))
        host_bytes = fab.fa_bwd_host_workspace_size(w.B, w.H, w.H_kv, w.N, w.Nkv, w.d)
        host_work = torch.empty(host_bytes + 256, dtype=torch.uint8, device=dev)
        host_ws = (host_work.data_ptr() + 255) // 256 * 256
        host_in = (hq, hk, hv, ho, hdout, hl)

        def e2e_step():
            st = fab.fa_bwd_host(*(t.data_ptr() for t in host_in), hgq.data_ptr(), hgk.data_ptr(),
                                 hgv.data_ptr(), w.B, w.H, w.H_kv, w.N, w.Nkv, w.d, scale, dt_code, host_ws,
                                 host_bytes, sp)
            if st != fab.FA_OK:
                raise fab.FAError(st, "fa_bwd_host")

        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in (hgq, hgk, hgv))

    def step():
        nonlocal launches
        step_fn()
        launches += kernels_per_step

    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    st = fab.fa_device_status(sp)
    if st != fab.FA_OK:
        raise fab.FAError(st, "warm-up")

    # ---- device-timed region: exactly K steps, launched as one CUDA graph
    # (the same kernels on the same data without the host's per-call work
    # between them; plain launches if capture is unavailable).  Inputs that
    # fit in L2 would stay there from one step to the next: then every step
    # is a plain launch preceded by a write of a buffer larger than L2, and
    # CUDA events bracket each step alone.
    flush = needs_flush(w)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    graph = None
    step_graph = None  # flushed mode: one step as a graph, replayed between the flushes
    if flush and not args.no_graph:
        try:
            step_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(step_graph, stream=stream, capture_error_mode="relaxed"):
                step_fn()
            with torch.cuda.stream(stream):
                step_graph.replay()  # one untimed replay
            torch.cuda.synchronize(dev)
        except Exception as exc:  # noqa: BLE001 - report and time without the graph
            print(f"bench: graph capture unavailable ({exc}); timing plain launches", file=sys.stderr)
            step_graph = None
            torch.cuda.synchronize(dev)
    if not args.no_graph and not flush:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
                for _ in range(args.steps):
                    step_fn()
            with torch.cuda.stream(stream):
                graph.replay()  # one untimed replay
            torch.cuda.synchronize(dev)
        except Exception as exc:  # noqa: BLE001 - report and time without the graph
            print(f"bench: graph capture unavailable ({exc}); timing plain launches", file=sys.stderr)
            graph = None
            torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches = 0
    step_events = []
    with clock_sampler(local) as clocks:
        with torch.cuda.stream(stream):
            if flush:
                for _ in range(args.steps):
                    flush_buf.zero_()
                    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e_a.record(stream)
                    if step_graph is not None:
                        step_graph.replay()
                        launches += kernels_per_step
                    else:
                        step()
                    e_b.record(stream)
                    step_events.append((e_a, e_b))
            else:
                ev0.record(stream)
                if graph is not None:
                    graph.replay()
                    launches = args.steps * kernels_per_step
                else:
                    for _ in range(args.steps):
                        step()
                ev1.record(stream)
        torch.cuda.synchronize(dev)
        # a region shorter than the sampling interval: keep the same load
        # (untimed replays) until one more clock sample has landed
        clock_window = "during the timed region"
        if (graph is not None or flush) and clocks.count() <= clocks.start_rows:
            clock_window = ("around the timed region (same " + ("graph replayed" if graph is not None else
                            "flushes and steps repeated") + "; region shorter than a sample)")
            t_end = time.time() + 2.0
            with torch.cuda.stream(stream):
                while clocks.count() <= clocks.start_rows and time.time() < t_end:
                    if graph is not None:
                        graph.replay()
                    else:
                        for _ in range(20):
                            flush_buf.zero_()
                            if step_graph is not None:
                                step_graph.replay()
                            else:
                                step_fn()
                    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    timed_launches = launches
    st = fab.fa_device_status(sp)
    if st != fab.FA_OK:
        raise fab.FAError(st, "timed region")
    ms_local = (sum(e_a.elapsed_time(e_b) for e_a, e_b in step_events) if flush
                else ev0.elapsed_time(ev1))
    ms_total, _, value = aggregate(ms_local, w.flops() * args.steps, dist, dev)
    kernel_ms = ms_local / args.steps  # the step's kernels, all on this stream
    clk = clocks.summary()

    # ---- end to end: host copies inside the timed region
    e2e_steps = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        e2e_step()  # first call creates the copy streams
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_events = []
    with torch.cuda.stream(stream):
        if flush:
            for _ in range(e2e_steps):
                flush_buf.zero_()
                e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e_a.record(stream)
                e2e_step()
                e_b.record(stream)
                e2e_events.append((e_a, e_b))
        else:
            e0.record(stream)
            for _ in range(e2e_steps):
                e2e_step()
            e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_local = (sum(e_a.elapsed_time(e_b) for e_a, e_b in e2e_events) if flush
                 else e0.elapsed_time(e1))
    e2e_ms, _, e2e_value = aggregate(e2e_local, w.flops() * e2e_steps, dist, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks = measured_peaks()
    bf16_peak = (peaks or {}).get("bf16_tflops")
    hbm_peak = (peaks or {}).get("hbm_gbs")
    peak_note = "measured bf16 burst (MEASURED_PEAKS.json)"
    if not bf16_peak:
        bf16_peak, peak_note = FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s bf16"
    if not hbm_peak:
        hbm_peak = FALLBACK_HBM_GBS
    tensor_peak = bf16_peak if w.dtype != "f32" else bf16_peak * NOMINAL_TF32_OVER_BF16
    if w.dtype == "f32":
        peak_note += " x nominal tf32/bf16 ratio 0.5"
    elif w.dtype == "f16":
        peak_note += " (fp16 and bf16 share the dense rate)"
    step_s = kernel_ms * 1e-3
    intensity = w.flops() / w.bytes()
    ridge = tensor_peak * 1e12 / (hbm_peak * 1e9)
    if w.backward:
        kernel_name = (f"fa_bwd_kernel<{w.dtype},{w.d}{',causal' if w.causal else ''}> + fa_bwd_prep_kernel"
                       " + fa_bwd_dq_kernel (timed as the whole step)")
    else:
        # the decode kernel takes 16-bit inputs with at most 32 query rows per
        # key/value head (N x H / H_kv), like the library's own dispatch
        decode = w.dtype != "f32" and w.N * (w.H // w.H_kv) <= 32
        base = (f"{'fa_decode_kernel' if decode else 'fa_fwd_kernel'}"
                f"<{w.dtype},{w.d}{',causal' if w.causal else ''}>")
        if use_fa_fwd:
            kernel_name = base if kernels_per_step == 1 else (
                f"{base} (full waves) + {base} (last wave, keys split across the CTAs of a cluster)")
        else:
            # decode steps and packed grouped heads merge their partitions
            # through the workspace; unpacked launches split only their last
            # wave, in clusters
            packed = w.H_kv < w.H and w.N * (w.H // w.H_kv) <= 128
            if kernels_per_step == 1:
                kernel_name = base
            elif decode or packed:
                kernel_name = f"{base} + fa_merge_kernel"
            else:
                kernel_name = f"{base} (full waves) + {base} (last wave, keys split across the CTAs of a cluster)"
    if intensity >= ridge:
        achieved = w.flops() / step_s / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tensor_peak, "unit": UNIT,
                    "frac": achieved / tensor_peak, "peak_source": peak_note}
    else:
        achieved = w.bytes() / step_s / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak,
                    "peak_source": "measured copy bandwidth (MEASURED_PEAKS.json)" if peaks else "fallback"}
    roofline.update({"traffic": stored_traffic(w.name, w.backward), "kernel": kernel_name,
                     "algorithmic_flops_per_launch": w.flops(),
                     "algorithmic_bytes_per_launch": w.bytes(),
                     "arithmetic_intensity": intensity})
    frac_tensor = value / world / tensor_peak

    launch_text = (("K replays of a one-step CUDA graph" if step_graph is not None else "K plain launches")
                   + ", each step bracketed by its own CUDA events" if flush
                   else "one CUDA graph of the K steps" if graph is not None else "K plain launches")
    line = result_line(
        w, world, args.steps, args.warmup, ms_total, value, splits=splits, launch=launch_text,
        frac_of_peak=frac_tensor, roofline=roofline,
        e2e={"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
             "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps},
        gpu_launches=timed_launches,
        clocks=dict({k2: clk[k2] for k2 in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "source") if k2 in clk},
                    window=clock_window),
        entry=entry_name)
    if world == 1 and not args.no_cpu_baseline:
        dout_np = I.make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=wr.seed) if w.backward else None
        rate, cores, n, secs = cpu_oracle_rate(wr, q, k, v, dout_np, target_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample_text(w, n, cores, secs)}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="workload name (default: the headline shape)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time plain launches instead of a CUDA graph")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from exact_tiled_attention_04_gb300 import inputs as I
    w = I.WORKLOADS[args.workload or I.HEADLINE]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
