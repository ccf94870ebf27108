"""Benchmark: fused-epilogue GEMM TFLOP/s on one GB300 (or N replicas).

A step is one launch of the whole path (the fused GEMM) over the workload's
inputs, already resident in HBM.  Default workload: bf16 8192^3 with
D = ReLU(0.5*A*B + 1.0*C + bias[n]) (inputs 384 MiB + 128 MiB output, far
larger than the 129 MB L2, so no flush is needed between steps).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle as
the reference arm on a bounded row sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "fused_bf16_8192"
METRIC = "GEMM TFLOP/s (2MNK/s) bf16 8192^3 and % of GB300 dense tensor peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
KERNEL_SOURCES = ["dense_gemm_epilogue_sm_gb300/csrc/gemm_kernel.cuh", "dense_gemm_epilogue_sm_gb300/csrc/ptx.cuh",
                  "dense_gemm_epilogue_sm_gb300/csrc/gemm_internal.h"]


def _code_only(text):
    """C++ source without comments, trailing blanks and empty lines: what the
    compiler sees, so editing a comment does not change the hash."""
    out, i, n, quote = [], 0, len(text), None
    while i < n:
        c = text[i]
        if quote:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(text[i + 1])
                i += 2
                continue
            if c == quote:
                quote = None
            i += 1
        elif c in "\"'":
            quote = c
            out.append(c)
            i += 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).split("\n") if line.strip())


def kernel_hash():
    """Hash of the kernel's sources as compiled (comments excluded)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def workloads_module():
    """The workload generator, loaded by path: it holds no GEMM code and
    imports only torch, so the reference arm never runs the package's
    __init__ (which loads the CUDA library)."""
    import importlib.util

    name = "dense_gemm_epilogue_sm_gb300_workloads"
    if name in sys.modules:
        return sys.modules[name]
    spec = importlib.util.spec_from_file_location(
        name, os.path.join(ROOT, "dense_gemm_epilogue_sm_gb300", "workloads.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod
    spec.loader.exec_module(mod)
    return mod


# Dense tensor-core rate per SM and clock, by operand width: one cta_group::2
# 256x256x16 bf16 MMA per CTA pair every 128 cycles (8192 FLOP/clk/SM), twice
# that for 8-bit and four times for 4-bit operands.  ncu on this kernel gives
# 7988 FLOP per tensor-active cycle per SM for bf16 (cuBLAS: 7819), and about
# 32k for NVFP4 (profiles/).
SPEC_FLOP_PER_CLK_SM = {"bf16": 8192, "f16": 8192, "e4m3": 16384, "e2m1": 32768}
SPEC_SM_MHZ = 2070.0                 # the part's maximum SM clock


def spec_peak_tflops(dtype_in, sms, mhz=SPEC_SM_MHZ):
    """sms x dense FLOP/clk/SM x clock, in TFLOP/s."""
    return sms * SPEC_FLOP_PER_CLK_SM[dtype_in] * mhz * 1e6 / 1e12


def roofline_bound(flops, nbytes, tensor_tflops, hbm_gbs):
    """'tensor' or 'hbm': whichever of FLOPs / tensor peak and bytes / HBM
    peak takes longer."""
    return "hbm" if nbytes / (hbm_gbs * 1e9) > flops / (tensor_tflops * 1e12) else "tensor"


def workload_config(spec, flushed):
    """The workload part of the JSON line's config: the same in both arms."""
    cfg = {"workload": spec.name, "M": spec.M, "N": spec.N, "K": spec.K, "batch": spec.batch}
    if getattr(spec, "groups", 0):
        cfg["groups"] = spec.groups
    cfg.update({"alpha": spec.alpha, "beta": spec.beta, "act": spec.act, "bias": spec.bias,
                "in": spec.dtype_in, "out": spec.dtype_d,
                "l2": "L2 flushed between steps" if flushed else "inputs larger than L2"})
    return cfg


L2_BYTES = 129e6


def needs_flush(spec):
    """Inputs smaller than twice the L2 are flushed from it before every launch."""
    return spec.algorithmic_bytes() < 2 * L2_BYTES


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entries = json.load(f)
    kh = kernel_hash()
    for e in entries:
        if e.get("kernel_hash") == kh and e.get("workload") == workload:
            return e.get("dram_bytes_per_launch")
    return None


class NvmlSampler:
    """SM clock, power and clock-event reasons read through NVML (ctypes on
    libnvidia-ml) every `period` seconds on a thread: dense enough that a
    timed region of a few ms holds samples.  Reads only; changes nothing."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid, period=0.001):
        import ctypes

        self.samples = []
        self.period = period
        self._stop = False
        self.thread = None
        self.ok = False
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
                return
            self.nv = nv
            self.ct = ctypes
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))      # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _read(self):
        ct, nv, h = self.ct, self.nv, self.handle
        mhz, mw, reasons = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        while not self._stop:
            t = time.time()
            nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz))
            nv.nvmlDeviceGetPowerUsage(h, ct.byref(mw))
            nv.nvmlDeviceGetCurrentClocksEventReasons(h, ct.byref(reasons))
            self.samples.append((t, float(mhz.value), mw.value / 1000.0, int(reasons.value)))
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()

    def stop(self):
        self._stop = True
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        if not inside:
            return None
        bits = 0
        for x in inside:
            bits |= x[3]
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(name for b, name in self.REASONS.items() if bits & b),
                "samples": len(inside), "window": "timed region (NVML, 1 ms)",
                "power_w_max": max(x[2] for x in inside)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms (used
    where NVML cannot be loaded)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside:
            inside = [p for _, p in self.samples]
            window = "whole run (no sample fell inside the timed region)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def job_step_ms(total_ms, kernel_ms, steps, flushed, world, device="cpu"):
    """Per-step time of the whole job: this rank's step time (the timed
    region over the steps, or the mean launch time when an L2 flush runs
    between launches), then the maximum over ranks."""
    import torch
    import torch.distributed as dist

    local = statistics.mean(kernel_ms) if flushed else total_ms / steps
    if world > 1:
        t = torch.tensor([local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        local = float(t.item())
    return local


def job_value(flops_per_rank, world, step_ms):
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's step."""
    return flops_per_rank * world / (step_ms * 1e-3) / 1e12


def oracle_view(spec, inputs):
    """The problem the oracle samples rows of: the workload itself, or for a
    grouped workload its first group (the whole A with B and bias of group
    0; rows of that group only).  A block-scaled D (e4m3 or e2m1 with
    factors) is the oracle's fp32 t followed by its output quantiser.
    Returns (spec, inputs, rows to draw from, rows -> result function)."""
    import dataclasses

    from oracle import gemm_ref

    wl = workloads_module()
    total = spec.batch * spec.M
    if getattr(spec, "groups", 0):
        sub = dataclasses.replace(spec, groups=0, group_sizes=())
        per = spec.matrix_elems("b")
        bias = None if inputs.bias is None else inputs.bias[: spec.N].contiguous()
        total = int(inputs.extras["group_rows"][1])
        inputs = wl.Inputs(sub, inputs.A, inputs.B[:per].contiguous(), inputs.C, bias, inputs.scale_a,
                           inputs.scale_b)
        spec = sub
    quant = None
    if spec.dtype_d == "e4m3":
        quant = gemm_ref.mx_quantise_rows
    elif spec.dtype_d == "e2m1":
        quant = lambda t, g=spec.scale_d: gemm_ref.nv_quantise_rows(t, g)
    if quant is not None:
        spec = dataclasses.replace(spec, dtype_d="f32")

    def run(rows, nthreads=0):
        bits, t = gemm_ref.run_spec_rows(spec, inputs, rows=rows, want_t=quant is not None, nthreads=nthreads)
        return quant(t) if quant is not None else bits
    return spec, inputs, total, run


def host_cpu():
    """The host's CPU model and logical core count, as the OS reports them."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"model": model or "unknown", "logical_cores": os.cpu_count()}


def single_core_tflops(spec, run, total_rows, seconds=3.0, seed=2):
    """The oracle on one thread over a small random row sample, sized for
    about `seconds`; returns (TFLOP/s, rows)."""
    import numpy as np

    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(total_rows, size=1, replace=False))
    t0 = time.perf_counter()
    run(rows, nthreads=1)
    per_row = max(time.perf_counter() - t0, 1e-6)
    n = int(min(total_rows, max(1, seconds / per_row)))
    rows = np.sort(rng.choice(total_rows, size=n, replace=False))
    t0 = time.perf_counter()
    run(rows, nthreads=1)
    dt = time.perf_counter() - t0
    return 2.0 * n * spec.N * spec.K / dt / 1e12, n


def oracle_sample(spec, inputs, rows_target_s=12.0):
    """Times the oracle on a bounded random row sample sized for about
    `rows_target_s` seconds; returns (tflops, number of rows, secs, threads,
    the rows, the oracle's result for them)."""
    import numpy as np

    from oracle import gemm_ref

    threads = gemm_ref.max_threads()
    rng = np.random.default_rng(0)
    spec, inputs, total_rows, run = oracle_view(spec, inputs)
    run(np.array([0]))                                             # decodes B once (kept by the oracle)
    probe = np.sort(rng.choice(total_rows, size=min(total_rows, 2 * threads), replace=False))
    t0 = time.perf_counter()
    run(probe)
    rows_per_s = len(probe) / (time.perf_counter() - t0)
    n = int(min(total_rows, max(len(probe), rows_target_s * rows_per_s)))
    rows = np.sort(rng.choice(total_rows, size=n, replace=False))
    t0 = time.perf_counter()
    result = run(rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * len(rows) * spec.N * spec.K
    one, one_rows = single_core_tflops(spec, run, total_rows)
    return flops / dt / 1e12, len(rows), dt, threads, rows, result, one, one_rows


def parity_on_rows(spec, inputs, D, rows, ref_bits):
    """The timed launches' own output checked on the oracle's sampled rows
    (l*M + m) with the method's tolerance: per element
    tau * sqrt(K) * max|A| * max|B| + one output ulp, tau 1e-3 for 16-bit and
    2e-2 for 8-bit operands.  IEEE output types only; returns a summary."""
    import numpy as np
    import torch

    if spec.dtype_d not in ("f32", "f16", "bf16") or spec.block_scale != "none" or getattr(spec, "groups", 0):
        return None
    per, ld = spec.matrix_elems("d"), spec.ld("d")
    l, m = rows // spec.M, rows % spec.M
    n = np.arange(spec.N)
    idx = (l * per)[:, None] + ((m * ld)[:, None] + n[None, :] if spec.order_d == "row" else
                                m[:, None] + (n * ld)[None, :])
    flat = D.reshape(-1).cpu()
    got = flat[torch.from_numpy(idx.reshape(-1))].to(torch.float64).numpy().reshape(len(rows), spec.N)
    bits = torch.from_numpy(np.ascontiguousarray(ref_bits).view(np.int32 if spec.dtype_d == "f32" else np.int16))
    ref = bits.view({"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[spec.dtype_d])
    ref = ref.to(torch.float64).numpy()
    a = inputs.A.to(torch.float32).abs().max().item() * inputs.scale_a
    b = inputs.B.to(torch.float32).abs().max().item() * inputs.scale_b
    tau = 2e-2 if spec.dtype_in == "e4m3" else 1e-3
    mbits = {"f32": 23, "f16": 10, "bf16": 7}[spec.dtype_d]
    emin = {"f32": -126, "f16": -14, "bf16": -126}[spec.dtype_d]
    ulp = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** emin))), emin) - mbits)
    slope = 1.13 if spec.act == "gelu" else 1.0
    tol = slope * tau * np.sqrt(spec.K) * a * b + ulp
    worst = float(np.max(np.abs(got - ref) / tol)) if got.size else 0.0
    return {"rows": int(len(rows)), "elements": int(got.size), "max_err_over_tol": worst,
            "pass": bool(np.isfinite(got).all() and worst <= 1.0)}


def run_reference(args):
    """Reference arm: the CPU oracle, as it stands, on bounded row samples."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    from oracle import gemm_ref
    import numpy as np

    wl = workloads_module()
    spec = wl.get(args.workload)
    inputs = wl.make_inputs(spec)
    config = workload_config(spec, needs_flush(spec))
    threads = gemm_ref.max_threads()
    rng = np.random.default_rng(1)
    grouped = getattr(spec, "groups", 0) > 0
    spec, inputs, total_rows, run = oracle_view(spec, inputs)
    # size each step so the whole --steps/--warmup run stays within about
    # args.ref_seconds; a step is at least one full row, and consecutive steps
    # share an oracle call (about one row per host core) so the cores work in
    # parallel
    probe = np.sort(rng.choice(total_rows, size=min(total_rows, threads), replace=False))
    run(probe[:1])                                           # decodes B once (kept by the oracle)
    t0 = time.perf_counter()
    run(probe)
    per_row = (time.perf_counter() - t0) / len(probe)
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    nrows = int(min(total_rows, max(1, budget / max(per_row, 1e-9))))
    per_call = max(1, threads // nrows)                      # steps per oracle call

    def run_steps(count):
        for c0 in range(0, count, per_call):
            k = min(per_call, count - c0)
            run(np.sort(rng.choice(total_rows, size=min(total_rows, k * nrows), replace=False)))

    run_steps(args.warmup)
    t0 = time.perf_counter()
    run_steps(args.steps)
    dt = time.perf_counter() - t0
    flops = 2.0 * nrows * spec.N * spec.K * args.steps
    value = flops / dt / 1e12
    one, one_rows = single_core_tflops(spec, run, total_rows)
    sample = f"{nrows} random full rows of the {spec.M}x{spec.N}x{spec.K} workload per step" + \
        (" (rows of group 0)" if grouped else "") + f", {per_call} steps per oracle call"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded torch CPU generator; N(0,1) operands, bias N(0,0.1))", "config": config,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
                         "single_core": {"value": one, "rows": one_rows}, "host": host_cpu()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(launch, spec, inputs, dev, steps, flops):
    """The same GEMM end to end through the public API with host buffers:
    every step uploads its inputs from pinned host memory, runs the GEMM and
    reads D back.  Steps are pipelined on three streams (upload, compute,
    download) over two device buffer sets, so step i+1's upload and step
    i-1's download overlap step i's GEMM."""
    import torch

    ex = inputs.extras or {}
    host = [inputs.A.pin_memory(), inputs.B.pin_memory(),
            inputs.C.pin_memory() if inputs.C is not None else None,
            inputs.bias.pin_memory() if inputs.bias is not None else None,
            ex["sfa"].pin_memory() if "sfa" in ex else None,
            ex["sfb"].pin_memory() if "sfb" in ex else None,
            ex["group_rows"].pin_memory() if "group_rows" in ex else None]
    nbuf = 2
    dev_in = [[None if t is None else torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host]
              for _ in range(nbuf)]
    nd = spec.batch * spec.matrix_elems("d")
    dev_out = [torch.empty(nd, dtype=torch.float32 if spec.dtype_d == "f32" else
                           (torch.float16 if spec.dtype_d == "f16" else torch.bfloat16), device=dev)
               for _ in range(nbuf)]
    host_out = [torch.empty(nd, dtype=dev_out[0].dtype).pin_memory() for _ in range(nbuf)]
    h2d = sum(t.numel() * t.element_size() for t in host if t is not None)
    d2h = host_out[0].numel() * host_out[0].element_size()
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in range(nbuf)]
    comp_done = [torch.cuda.Event() for _ in range(nbuf)]
    out_done = [torch.cuda.Event() for _ in range(nbuf)]

    def step(i):
        b = i % nbuf
        A, B, C, bias, sfa, sfb, gr = dev_in[b]
        with torch.cuda.stream(s_in):
            if i >= nbuf:
                s_in.wait_event(comp_done[b])       # the GEMM of step i-2 has read these inputs
            for d_t, h_t in zip(dev_in[b], host):
                if h_t is not None:
                    d_t.copy_(h_t, non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done[b])
            if i >= nbuf:
                s_comp.wait_event(out_done[b])      # step i-2's D has been read back
            launch(A, B, C, dev_out[b], bias, s_comp, sfa, sfb, gr)
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            host_out[b].copy_(dev_out[b], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(2):                              # warm-up
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": dt * 1e3, "steps": steps,
            "how": "pinned host buffers; upload, GEMM and download on three streams over two device buffer sets"}


def run_plain(wl, g, GemmOp, desc_from_spec, A, B, dev, stream, launches=300):
    """Plain bf16 8192^3 (no C, no bias, no activation) on the fused workload's A and B."""
    import torch
    pspec = wl.get("plain_bf16_8192")
    op = GemmOp(desc_from_spec(pspec))
    D = torch.empty(pspec.matrix_elems("d"), dtype=wl.DT[pspec.dtype_d], device=dev)
    for _ in range(5):
        op(A, B, None, D, None, stream)
    op.check()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(launches):
        op(A, B, None, D, None, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    op.check()
    ms = e0.elapsed_time(e1) / launches
    op.close()
    return {"workload": pspec.name, "value": pspec.flops() / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_launch": ms, "launches": launches,
            "note": "same A and B, beta = 0, no bias, no activation; back-to-back launches after the headline run"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import dense_gemm_epilogue_sm_gb300 as g
    from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec

    wl = workloads_module()

    world, rank, local = dist_setup()
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    spec = wl.get(args.workload)
    inputs = wl.make_inputs(spec)

    # oracle sample first (on the host cores, before the GPU is busy)
    cpu = None
    cpu_rows = cpu_ref = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tflops, nrows, secs, threads, cpu_rows, cpu_ref, one, one_rows = oracle_sample(
            spec, inputs, rows_target_s=args.cpu_seconds)
        cpu = {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{nrows} random full rows of {spec.M}x{spec.N}x{spec.K} ({secs:.1f} s, fp64 C loop)",
               "single_core": {"value": one, "rows": one_rows}, "host": host_cpu()}

    A = inputs.A.to(dev)
    B = inputs.B.to(dev)
    C = inputs.C.to(dev) if inputs.C is not None else None
    bias = inputs.bias.to(dev) if inputs.bias is not None else None
    ex = inputs.extras or {}
    sfa_d = ex["sfa"].to(dev) if "sfa" in ex else None
    sfb_d = ex["sfb"].to(dev) if "sfb" in ex else None
    sfd_d = None
    if spec.dtype_d in ("e4m3", "e2m1"):        # MX / NVFP4 output: the factor tensor beside D
        sfk = (spec.N + (31 if spec.dtype_d == "e4m3" else 15)) // (32 if spec.dtype_d == "e4m3" else 16)
        sfd_d = torch.empty(spec.batch * ((spec.M + 127) // 128) * ((sfk + 3) // 4) * 512, dtype=torch.uint8,
                            device=dev)
    d_elems = spec.batch * spec.matrix_elems("d")
    D = torch.empty(d_elems // 2 if spec.dtype_d == "e2m1" else d_elems, dtype=wl.DT[spec.dtype_d], device=dev)
    desc = desc_from_spec(spec, inputs.scale_a, inputs.scale_b)
    info = g.gemm_plan(desc)
    groups = getattr(spec, "groups", 0)
    op = GemmOp(desc, groups=groups)
    gr_d = ex["group_rows"].to(dev) if "group_rows" in ex else None

    def launch(A, B, C, D, bias, stream, sfa=None, sfb=None, gr=None):
        # block-scaled descriptors carry their scale factors through gemm_run_args
        if groups:
            op.run_grouped(A, B, C, D, gr if gr is not None else gr_d, bias, stream=stream)
        elif spec.block_scale != "none" or sfd_d is not None:
            op.run_args(A, B, C, D, bias, sfa=sfa if sfa is not None else sfa_d,
                        sfb=sfb if sfb is not None else sfb_d, sfd=sfd_d, stream=stream)
        else:
            op(A, B, C, D, bias, stream)

    stream = torch.cuda.current_stream(dev)
    flops = spec.flops()
    in_bytes = spec.algorithmic_bytes()
    flush = None
    if needs_flush(spec):
        flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        launch(A, B, C, D, bias, stream)
    op.check()
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    uuid = uuid if uuid.startswith("GPU-") else (f"GPU-{uuid}" if uuid else "")
    sampler = ClockSampler(uuid or str(local))
    sampler.start()
    nvml = NvmlSampler(uuid) if uuid else None
    if nvml is not None:
        nvml.start()
    time.sleep(0.3)

    launches0 = op.launches
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    total0 = torch.cuda.Event(enable_timing=True)
    total1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    total0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        launch(A, B, C, D, bias, stream)
        ends[i].record(stream)
    total1.record(stream)
    torch.cuda.synchronize()
    barrier()
    wall1 = time.time()
    op.check()
    launches = op.launches - launches0
    # the timed launches' own D against the oracle rows sampled above
    parity = parity_on_rows(spec, inputs, D, cpu_rows, cpu_ref) if cpu_rows is not None else None
    total_ms = total0.elapsed_time(total1)
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    step_ms = job_step_ms(total_ms, kernel_ms, args.steps, flush is not None, world, dev)
    time.sleep(0.2)
    sampler.stop()
    clocks = None
    if nvml is not None:
        nvml.stop()
        clocks = nvml.summary(wall0, wall1)
    if clocks is None:
        clocks = sampler.summary(wall0, wall1)

    # (the timed region includes the flush writes when a flush is needed;
    # the per-launch kernel time excludes them)
    value = job_value(flops, world, step_ms)
    avg_kernel_ms = statistics.mean(kernel_ms)

    # end to end through the public API with host buffers: H2D of the inputs,
    # the GEMM, D2H of the result, every step
    e2e = None
    if not args.no_e2e and spec.dtype_d not in ("e4m3", "e2m1"):     # (block-scaled output: not measured end to end)
        e2e = run_e2e(launch, spec, inputs, dev, max(1, min(args.steps, args.e2e_steps)), flops)
        op.check()

    # The bare GEMM of the same size (beta = 0, no bias, no activation) on the
    # same operands, timed separately and reported beside the headline.
    plain = None
    if spec.name == "fused_bf16_8192" and world == 1 and not args.no_plain:
        plain = run_plain(wl, g, GemmOp, desc_from_spec, A, B, dev, stream)

    peaks, peak_src = load_peaks()
    long_region = total_ms > 1000.0
    pkey = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    peak = float(peaks.get(pkey, FALLBACK_PEAKS[pkey]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # nominal dense ratios to bf16: fp8 4.5 : 2.25, fp4 13.5 : 2.25
    ratio = {"e4m3": 2.0, "e2m1": 6.0}.get(spec.dtype_in, 1.0)
    peak *= ratio
    achieved = flops / (avg_kernel_ms * 1e-3) / 1e12
    gbs = in_bytes / (avg_kernel_ms * 1e-3) / 1e9
    traffic = load_traffic(spec.name)
    bound = roofline_bound(flops, in_bytes, peak, hbm)
    sms = props.multi_processor_count
    spec_peak = spec_peak_tflops(spec.dtype_in, sms)
    at_clock = spec_peak_tflops(spec.dtype_in, sms, clocks["sm_mhz"]) if clocks.get("sm_mhz") else None
    if bound == "hbm":
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes": in_bytes,
                    "tflops": achieved, "tensor_frac": achieved / peak}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "peak_source": f"{peak_src} {pkey}" + (f" x{ratio:g} ({spec.dtype_in} nominal ratio)"
                                                           if ratio != 1.0 else ""),
                    "algorithmic_bytes": in_bytes, "hbm_frac": gbs / hbm}
    # the tensor peak of the part itself: SMs x dense FLOP/clk/SM x 2070 MHz,
    # and the same at the SM clock sampled during the timed region
    roofline["spec_peak"] = spec_peak
    roofline["spec_frac"] = achieved / spec_peak
    roofline["spec_frac_at_clock"] = achieved / at_clock if at_clock else None
    roofline["spec_source"] = (f"{sms} SMs x {SPEC_FLOP_PER_CLK_SM[spec.dtype_in]} FLOP/clk/SM "
                               f"({spec.dtype_in} dense) x {SPEC_SM_MHZ:g} MHz")

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": spec.dtype_in,
        "data": "synthetic (seeded torch CPU generator; N(0,1) operands, bias N(0,0.1))",
        "config": workload_config(spec, flush is not None),
        "plan": {"tile": f"{info.tile_m}x{info.tile_n}x{info.tile_k}", "stages": info.stages,
                 "cta_group": info.cta_group, "tiles": info.tiles, "kernel_hash": kernel_hash()},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if plain is not None:
        plain["frac_of_burst_peak"] = plain["value"] / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        line["plain_gemm"] = plain
    if rank == 0:
        print(json.dumps(line), flush=True)
    op.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-plain", action="store_true", help="skip the plain-GEMM line beside the fused headline")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--ref-seconds", type=float, default=100.0,
                    help="reference arm: about how long the whole --steps/--warmup run takes")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
