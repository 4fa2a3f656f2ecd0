"""Benchmark: the full NVFP4 linear-layer step of the 3B model's FFN at 16384
tokens on one GB300 (Fprop / Dgrad / Wgrad of the up 3072->9216 and down
9216->3072 projections, each operand quantized before its first use; H and
dY_up are the outputs of Fprop-up and Dgrad-down, whose epilogues take their
tensor amaxes).

Prints one JSON line.  `value` is the step's GEMM work (6 GEMMs x 2*M*N*K)
divided by the device time of the whole step (all quantize and GEMM kernels),
inputs resident in HBM.  `e2e` is the same metric with the bf16 inputs (X,
W_up, W_down, dY_down) copied from pinned host memory and the step's results
(Y, dX, dW_down, dW_up) copied back, every step, inside the timed region
(copies on their own streams, two device buffer sets, so a step's copies
overlap its neighbours' compute; H and dY_up never leave the device).  `roofline` reports the kernel that takes most of the step's time
against its measured peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (torchrun) each rank runs an independent replica of the step: the
path has no exchange step, so there is no collective on the data path.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMM TFLOPS & quantize GB/s at 3B shapes, % of FP4/HBM roofline (1 GB300)"
HIDDEN, FFN = 3072, 9216
TOKENS = 16384          # the full layer step; --tokens scales it down for profiling
# FP4 dense peak = measured bf16 peak x nominal fp4/bf16 ratio (13.5 / 2.25)
FP4_OVER_BF16 = 13.5 / 2.25
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ setup --
# DRAM bytes per step of each kernel class on the 16384-token step, summed
# over the class's launches in one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum, one pass per launch); the figure holds while the
# kernel sources hash to the recorded value, and is reported as null otherwise.
TRAFFIC = {
    "quantize": ("b7237ac0b154193c", ("quantize.cu", "device_common.cuh"), 1537645568),
    "gemm": ("4e0a4b19100d7376", ("gemm.cu", "device_common.cuh"), 1240032256),
}


def measured_traffic(kind):
    import hashlib
    digest, files, nbytes = TRAFFIC[kind]
    if TOKENS != 16384:
        return None
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "fp4_gemm_nvfp4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return nbytes if h.hexdigest()[:16] == digest else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    """The slowest rank's time: the job's time (every rank gets it)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.item()


def whole_job_tflops(flops_per_rank, world, ms):
    """Weak scaling: every rank runs the full step on its own data."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


# The step: (name, input, kwargs for ops.quantize) and the six GEMMs.
QUANTS = [
    # X, H and the two output gradients give a row-wise operand (Fprop /
    # Dgrad) and a col-wise RHT operand (Wgrad) from one call; weights 16x16.
    ("X.pair", "X", dict(pair=True, rht_mask="mask")),
    ("W_up.2d", "W_up", dict(rowwise=True, colwise=True, two_d=True)),
    ("H.pair", "H", dict(pair=True, rht_mask="mask")),
    ("W_down.2d", "W_down", dict(rowwise=True, colwise=True, two_d=True)),
    ("dY_down.pair", "dY_down", dict(pair=True, rht_mask="mask", sr=True, stream_row=1, stream_col=2)),
    ("dY_up.pair", "dY_up", dict(pair=True, rht_mask="mask", sr=True, stream_row=3, stream_col=4)),
]
GEMMS = [
    # name, A (quant name, orientation), B (quant name, orientation)
    ("fprop_up", ("X.pair", "row"), ("W_up.2d", "row")),
    ("fprop_down", ("H.pair", "row"), ("W_down.2d", "row")),
    ("dgrad_down", ("dY_down.pair", "row"), ("W_down.2d", "col")),
    ("dgrad_up", ("dY_up.pair", "row"), ("W_up.2d", "col")),
    ("wgrad_down", ("dY_down.pair", "col"), ("H.pair", "col")),
    ("wgrad_up", ("dY_up.pair", "col"), ("X.pair", "col")),
]
# The layer's dataflow: H is the Fprop-up output and dY_up the Dgrad-down
# output (the activation between is not part of this step), so those two
# GEMMs write them and take their two tensor amaxes in the epilogue, and the
# pair quantization of H and dY_up runs without its amax pass.  Off with
# --no-fuse-amax (then H and dY_up are inputs like X and dY_down).
FUSE_AMAX = True
PRODUCED = {"H": "fprop_up", "dY_up": "dgrad_down"}
ORDER = [("q", "X.pair"), ("q", "W_up.2d"), ("q", "W_down.2d"), ("g", "fprop_up"), ("q", "H.pair"),
         ("g", "fprop_down"), ("q", "dY_down.pair"), ("g", "dgrad_down"), ("q", "dY_up.pair"),
         ("g", "wgrad_down"), ("g", "dgrad_up"), ("g", "wgrad_up")]
SHAPES = {}


def produced(src):
    return FUSE_AMAX and src in PRODUCED


def set_tokens(tokens):
    global TOKENS
    TOKENS = tokens
    SHAPES.update({"X": (tokens, HIDDEN), "W_up": (FFN, HIDDEN), "H": (tokens, FFN),
                   "W_down": (HIDDEN, FFN), "dY_down": (tokens, HIDDEN), "dY_up": (tokens, FFN)})


set_tokens(TOKENS)


def workload_name():
    return f"c4_ffn_layer_step_{TOKENS}tok"


def host_inputs(seed_base=4):
    from fp4_gemm_nvfp4_gb300 import inputs
    wl = inputs.c4_ffn_layer_step(TOKENS)
    return {name: wl.make(name) for name in SHAPES}, inputs.rht_sign_mask(seed_base)


def quant_launches(kw):
    """Kernels one quantize call launches: an amax pass (one per emitted
    orientation when the RHT is on, each orientation's transform having its
    own amax) and one encode pass emitting every requested orientation; a
    row-wise plus col-wise RHT pair of one input shares one amax pass, and
    with the amax taken by the producing GEMM only the encode pass runs."""
    if kw.get("pair"):
        return 1 if kw.get("amax_given") else 2
    outs = int(kw.get("rowwise", True)) + int(kw.get("colwise", False))
    amax_passes = outs if (kw.get("rht_mask") is not None and not kw.get("two_d")) else 1
    return amax_passes + 1


def quant_bytes(rows, cols, kw):
    """Algorithmic HBM bytes of one quantize call: each amax pass reads the
    input once; the encode pass reads it once more and writes 0.5 B of codes
    and 1/16 B of scales per element per emitted orientation."""
    n = rows * cols
    if kw.get("pair"):                      # one amax pass, one encode pass emitting both orientations
        return n * 2 * (1 if kw.get("amax_given") else 2) + n * 2 * (0.5 + 1 / 16)
    outs = int(kw.get("rowwise", True)) + int(kw.get("colwise", False))
    amax_passes = outs if (kw.get("rht_mask") is not None and not kw.get("two_d")) else 1
    return n * 2 * (amax_passes + 1) + n * outs * (0.5 + 1 / 16)


class Step:
    """Device buffers and the launch sequence of one layer step."""

    def __init__(self, dev_inputs, mask, seed):
        import torch
        from fp4_gemm_nvfp4_gb300 import ops
        self.torch, self.ops = torch, ops
        self.x = dev_inputs
        self.mask = mask
        self.seed = seed
        self.q = {}
        self.kw = {}
        for name, src, kw in QUANTS:
            kw = dict(kw)
            if kw.get("rht_mask") == "mask":
                kw["rht_mask"] = mask
            if produced(src):
                kw["amax_given"] = True
            rows, cols = SHAPES[src]
            pair = kw.get("pair", False)
            row = ops.alloc_operand(rows, cols) if pair or kw.get("rowwise", True) else None
            col = ops.alloc_operand(cols, rows) if pair or kw.get("colwise", False) else None
            self.q[name] = (row, col)
            self.kw[name] = kw
        self.out = {}
        self.amax = {}
        for gname, (an, ao), (bn, bo) in GEMMS:
            a = self.operand(an, ao)
            b = self.operand(bn, bo)
            src = [k for k, g in PRODUCED.items() if g == gname]
            if FUSE_AMAX and src:
                self.out[gname] = self.x[src[0]]      # the GEMM writes the tensor the step quantizes next
                self.amax[gname] = torch.zeros(2, dtype=torch.float32, device="cuda")
            else:
                self.out[gname] = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device="cuda")
        self.ws = ops.Workspace()

    def operand(self, name, orient):
        row, col = self.q[name]
        return row if orient == "row" else col

    def flops(self):
        total = 0
        for gname, (an, ao), (bn, bo) in GEMMS:
            a, b = self.operand(an, ao), self.operand(bn, bo)
            total += 2 * a.rows * b.rows * a.cols
        return total

    def launches(self):
        return sum(quant_launches(self.kw[n]) for n, _, _ in QUANTS) + len(GEMMS)

    def run_quantize(self, only=None):
        for name, src, _ in QUANTS:
            if only is not None and name != only:
                continue
            row, col = self.q[name]
            kw = self.kw[name]
            if kw.get("amax_given"):
                self.ops.quantize_row_col_rht_amax(self.x[src], kw["rht_mask"], self.amax[PRODUCED[src]],
                                                   sr=kw.get("sr", False), seed=self.seed,
                                                   stream_row=kw.get("stream_row", 0),
                                                   stream_col=kw.get("stream_col", 0), out_row=row, out_col=col)
            elif kw.get("pair"):
                self.ops.quantize_row_col_rht(self.x[src], kw["rht_mask"], sr=kw.get("sr", False), seed=self.seed,
                                              stream_row=kw.get("stream_row", 0),
                                              stream_col=kw.get("stream_col", 0), out_row=row, out_col=col,
                                              workspace=self.ws)
            else:
                self.ops.quantize(self.x[src], out_row=row, out_col=col, seed=self.seed, workspace=self.ws, **kw)

    def run_gemms(self, only=None):
        for gname, (an, ao), (bn, bo) in GEMMS:
            if only is not None and gname != only:
                continue
            if gname in self.amax:
                self.ops.gemm_amax(self.operand(an, ao), self.operand(bn, bo), self.mask, out=self.out[gname],
                                   amax=self.amax[gname])
            else:
                self.ops.gemm(self.operand(an, ao), self.operand(bn, bo), out=self.out[gname])

    def run(self):
        """Enqueue one step: in the layer's dataflow order when the producing
        GEMMs take the amax, else every quantize call, then the six GEMMs."""
        if FUSE_AMAX:
            for kind, name in ORDER:
                (self.run_quantize if kind == "q" else self.run_gemms)(name)
        else:
            self.run_quantize()
            self.run_gemms()


# ----------------------------------------------------------------- clocks --
def smi_gpu_id(local):
    """nvidia-smi's name for the GPU torch uses as device `local`: its UUID
    (CUDA_VISIBLE_DEVICES may renumber devices, so the ordinal can name
    another GPU), else the ordinal."""
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except (AttributeError, RuntimeError):
        pass
    return str(local)


def gpu_local_cpus(local):
    """The CPUs the OS lists as local to the GPU torch uses as device `local`
    (sysfs of its PCI function), or None."""
    import torch
    try:
        p = torch.cuda.get_device_properties(local)
        bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            spec = f.read().strip()
    except (AttributeError, OSError, RuntimeError):
        return None
    cpus = set()
    for part in spec.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus or None


class LocalPinning:
    """Within the block the calling thread runs on the GPU-local CPUs, so the
    pinned host buffers it allocates land on the memory next to the GPU (a
    copy from the far socket's memory crosses one more link)."""

    def __init__(self, local):
        self.cpus = gpu_local_cpus(local)
        self.saved = None

    def __enter__(self):
        if self.cpus:
            try:
                self.saved = os.sched_getaffinity(0)
                os.sched_setaffinity(0, self.cpus & self.saved or self.cpus)
            except OSError:
                self.saved = None
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)


def host_cpu():
    """The host CPU model and the cores the OS reports."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_model": model or "unknown", "nproc": os.cpu_count()}


class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"nvfp4_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.5)     # let the sampler start before the timed region
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, windows):
        """Median SM clock and throttle reasons over the samples taken inside
        the timed windows [(t0, t1) host wall-clock seconds]."""
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    clk, mxv = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                if not any(t0 <= ts <= t1 for t0, t1 in windows):
                    continue
                sm.append(clk)
                mx = mxv
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------ CPU oracle --
def _oracle_kw(kw, mask, seed, orient):
    if kw.get("pair"):   # row-wise without RHT, col-wise with RHT, each on its own stream
        rht = orient == "col"
        return dict(scaling=0, rounding=1 if kw.get("sr") else 0, use_rht=rht, sign_mask=mask if rht else 0,
                    seed=seed, stream_id=kw.get("stream_col" if rht else "stream_row", 0))
    return dict(scaling=1 if kw.get("two_d") else 0, rounding=1 if kw.get("sr") else 0,
                use_rht=kw.get("rht_mask") is not None,
                sign_mask=mask if kw.get("rht_mask") is not None else 0,
                seed=seed, stream_id=kw.get("stream_id", 0))


def cpu_baseline(host, mask, seed, rows_a=8, rows_b=1024):
    """The oracle, as it stands, on a bounded sample of the step.  Each GEMM
    computes a rows_a x rows_b block of its output; the quantize calls encode
    exactly the operand rows that block needs, after the oracle's own
    full-tensor amax pass.  Returns a dict: the sample's GEMM FLOP rate over
    its whole time (TFLOP/s), its seconds, a description, the threads used,
    and the full step's time extrapolated from the sample (the amax passes as
    timed, the encode scaled by elements, the GEMM by FLOPs)."""
    import oracle
    src_of = {n: s for n, s, _ in QUANTS}
    kw_of = {n: k for n, _, k in QUANTS}
    t_amax = t_enc = t_gemm = 0.0
    enc_elems = full_elems = flops = full_flops = 0
    for gname, (an, ao), (bn, bo) in GEMMS:
        ops_, full_rows = [], []
        for qn, orient, nrows in ((an, ao, rows_a), (bn, bo, rows_b)):
            o = oracle.ROWWISE if orient == "row" else oracle.COLWISE
            bits = host[src_of[qn]]
            lrows, lcols = (bits.shape if o == oracle.ROWWISE else bits.shape[::-1])
            kw = _oracle_kw(kw_of[qn], mask, seed, orient)
            n = min(nrows, lrows)
            t0 = time.perf_counter()
            amax = oracle.amax(bits, o, kw["use_rht"], kw["sign_mask"])
            t1 = time.perf_counter()
            ops_.append(oracle.quantize(bits, o, rows_subset=(0, n), amax_value=amax, **kw))
            t2 = time.perf_counter()
            t_amax += t1 - t0
            t_enc += t2 - t1
            enc_elems += n * lcols
            full_elems += lrows * lcols
            full_rows.append(lrows)
        a, b = ops_
        t0 = time.perf_counter()
        oracle.gemm_f64(a, b, with_abs=False)
        t_gemm += time.perf_counter() - t0
        K = a["codes"].shape[1] * 2
        flops += 2 * a["codes"].shape[0] * b["codes"].shape[0] * K
        full_flops += 2 * full_rows[0] * full_rows[1] * K
    dt = t_amax + t_enc + t_gemm
    desc = (f"oracle on the host cores: each of the 6 GEMMs on a {rows_a} x {rows_b} block of its "
            f"output, its operand rows quantized by the oracle (full-tensor amax pass included)")
    extrapolated = t_amax + t_enc * full_elems / max(enc_elems, 1) + t_gemm * full_flops / max(flops, 1)
    return {"value": flops / dt / 1e12, "seconds": dt, "sample": desc, "threads": oracle.num_threads(),
            "extrapolated_full_step_s": extrapolated,
            "sample_split_s": {"amax_passes": round(t_amax, 3), "encode": round(t_enc, 3), "gemm": round(t_gemm, 3)}}


# --------------------------------------------------------------- measure --
def capture(torch, fn, stream):
    """One CUDA graph of fn() on `stream` (launch gaps vanish on replay)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_replays(torch, graph, n, stream):
    """Device milliseconds of n back-to-back replays, events on `stream`."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        graph.replay()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def measure(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    from fp4_gemm_nvfp4_gb300 import capi, ops

    host, mask = host_inputs()
    seed = 4 + 1000 * rank
    dev = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in host.items()}
    step = Step(dev, mask, seed)
    stream = torch.cuda.Stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
            torch.cuda.synchronize()

    # eager warm-up: first calls set kernel attributes and cache device queries
    with torch.cuda.stream(stream):
        step.run()
    barrier()
    status = ops.device_error()
    if status != capi.NVFP4_OK:
        raise RuntimeError(f"device status after the first step: {capi.status_string(status)}")
    g_step = capture(torch, step.run, stream)
    g_quant = {n: capture(torch, lambda n=n: step.run_quantize(n), stream) for n, _, _ in QUANTS}
    g_gemm = {n: capture(torch, lambda n=n: step.run_gemms(n), stream) for n, _, _ in GEMMS}
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_step.replay()
    barrier()

    # ---- the timed region: exactly K steps, inputs resident in HBM
    windows = []
    with ClockSampler(smi_gpu_id(local)) as clocks:
        barrier()
        t0 = time.time()
        with torch.cuda.stream(stream):
            total_ms = time_replays(torch, g_step, args.steps, stream)
        barrier()
        windows.append((t0, time.time()))
        # per kernel class: the same launches replayed alone, K times each
        launch_ms = {}
        t0 = time.time()
        with torch.cuda.stream(stream):
            for n, g in g_quant.items():
                launch_ms["q:" + n] = time_replays(torch, g, args.steps, stream) / args.steps
            for n, g in g_gemm.items():
                launch_ms["g:" + n] = time_replays(torch, g, args.steps, stream) / args.steps
        barrier()
        windows.append((t0, time.time()))
    total_ms = max_over_ranks(total_ms, world, "cuda")
    ms_per_step = total_ms / args.steps
    flops = step.flops()
    value = whole_job_tflops(flops, world, ms_per_step)

    # ---- end to end: pinned host inputs in and the step's four results out, every step.
    # Copies run on their own streams (one per direction) and two device
    # buffer sets alternate, so step i's copy-in and copy-out overlap the
    # compute of steps i + 1 and i - 1; the time runs from the first copy-in
    # to the last copy-out.
    with LocalPinning(local):
        pinned_in = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
                     for k, v in host.items() if not produced(k)}
        # the step's results: Y (fprop_down), dX (dgrad_up), dW_down and dW_up; H and
        # dY_up are the layer's internal tensors and stay on the device
        pinned_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in step.out.items()
                      if k not in PRODUCED.values()}
    h2d = sum(t.numel() * 2 for t in pinned_in.values())
    d2h = sum(t.numel() * 2 for t in pinned_out.values())
    e2e_steps = max(2, args.steps)
    dev_b = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in host.items()}
    step_b = Step(dev_b, mask, seed)
    with torch.cuda.stream(stream):
        step_b.run()
    barrier()
    g_step_b = capture(torch, step_b.run, stream)
    sets = [(dev, step, g_step), (dev_b, step_b, g_step_b)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        b = i & 1
        d, st, g = sets[b]
        if i >= 2:
            s_in.wait_event(comp_done[b])       # step i - 2 has read this set's inputs
        with torch.cuda.stream(s_in):
            for k, t in pinned_in.items():
                d[k].copy_(t, non_blocking=True)
        in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if i >= 2:
            stream.wait_event(out_done[b])      # step i - 2's outputs are out
        with torch.cuda.stream(stream):
            g.replay()
        comp_done[b].record(stream)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            for k, t in pinned_out.items():
                t.copy_(st.out[k], non_blocking=True)
        out_done[b].record(s_out)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, "cuda")
    status = ops.device_error()
    if status != capi.NVFP4_OK:
        raise RuntimeError(f"device status after timing: {capi.status_string(status)}")

    # ---- roofline of the dominant kernel class
    peaks, peak_src = load_peaks()
    gemm_ms = sum(v for k, v in launch_ms.items() if k.startswith("g:"))
    quant_ms = sum(v for k, v in launch_ms.items() if k.startswith("q:"))
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    qbytes = sum(quant_bytes(*SHAPES[src], step.kw[name]) for name, src, _ in QUANTS)
    quant_gbs = qbytes / (quant_ms * 1e-3) / 1e9
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    if gemm_ms >= quant_ms:
        roof = {"kernel": "gemm_nvf4_kernel (the step's 6 GEMMs)", "bound": "tensor",
                "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                "frac": round(gemm_tflops / fp4_peak, 4), "traffic": measured_traffic("gemm"),
                "traffic_basis": "DRAM bytes per step over the class's launches (ncu)",
                "peak_source": f"{peak_src} bf16 burst x {FP4_OVER_BF16:g} (nominal fp4/bf16)"}
        if FUSE_AMAX:
            roof["note"] = ("fprop_up and dgrad_down also take their BF16 output's two tensor amaxes in the "
                            "epilogue (the work of the quantizer's amax pass, moved there); achieved counts "
                            "only the FP4 GEMM FLOPs")
    else:
        roof = {"kernel": "quantize (amax + encode passes of the step)", "bound": "hbm",
                "achieved": round(quant_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(quant_gbs / peaks["hbm_gbs"], 4), "traffic": measured_traffic("quantize"),
                "traffic_basis": "DRAM bytes per step over the class's launches (ncu)",
                "algorithmic_bytes_per_step": round(qbytes),
                "peak_source": f"{peak_src} hbm_gbs"}

    quant_roof = {"kernel": "quantize (amax + encode passes of the step)", "bound": "hbm",
                  "achieved": round(quant_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                  "frac": round(quant_gbs / peaks["hbm_gbs"], 4), "traffic": measured_traffic("quantize"),
                  "traffic_basis": "DRAM bytes per step over the class's launches (ncu)",
                  "algorithmic_bytes_per_step": round(qbytes), "peak_source": f"{peak_src} hbm_gbs"}
    gemm_roof = {"kernel": "gemm_nvf4_kernel (the step's 6 GEMMs)", "bound": "tensor",
                 "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                 "frac": round(gemm_tflops / fp4_peak, 4), "traffic": measured_traffic("gemm"),
                 "traffic_basis": "DRAM bytes per step over the class's launches (ncu)",
                 "peak_source": f"{peak_src} bf16 burst x {FP4_OVER_BF16:g} (nominal fp4/bf16)"}
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic",
        "config": {"workload": workload_name(), "tokens": TOKENS, "hidden": HIDDEN, "ffn": FFN,
                   "gemm_gflop_per_step": round(flops / 1e9, 1), "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (one step touches about 2.5 GB)",
                   "dataflow": ("H and dY_up written by fprop_up and dgrad_down, their tensor amax taken in "
                                "those GEMMs' epilogue" if FUSE_AMAX else "all six bf16 tensors are inputs"),
                   "launch": "each step is one CUDA graph replay"},
        "roofline": roof,
        "roofline_by_class": {"gemm": gemm_roof, "quantize": quant_roof},
        "gemm_tflops": round(gemm_tflops, 1),
        "gemm_frac_of_fp4_peak": round(gemm_tflops / fp4_peak, 4),
        "quantize_gbs": round(quant_gbs, 1),
        "quantize_frac_of_hbm": round(quant_gbs / peaks["hbm_gbs"], 4),
        "per_launch_ms": {k: round(v, 4) for k, v in sorted(launch_ms.items())},
        "e2e": {"value": round(whole_job_tflops(flops, world, e2e_ms), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "host_buffers": ("pinned, allocated on the GPU-local CPUs" if gpu_local_cpus(local)
                                 else "pinned (no GPU-local CPU list found)")},
        "gpu_launches": step.launches() * args.steps,
        "clocks": clocks.summary(windows),
    }
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline(host, mask, seed, rows_a=512, rows_b=4096)
        result["cpu_baseline"] = {"value": cb["value"], "unit": "TFLOP/s", "cores": cb["threads"], "kind": "oracle",
                                  "sample": cb["sample"], "seconds": round(cb["seconds"], 2),
                                  **host_cpu(),
                                  "extrapolated_full_step_s": round(cb["extrapolated_full_step_s"], 1),
                                  "extrapolated_note": ("extrapolated, not measured: the sample's amax passes as "
                                                        "timed, its encode time scaled by the step's elements and "
                                                        "its GEMM time by the step's FLOPs"),
                                  "sample_split_s": cb["sample_split_s"]}
    if world > 1:
        torch.distributed.destroy_process_group()
    return result, rank


def reference_arm(args):
    """The oracle as the reference implementation, on the host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    host, mask = host_inputs()
    seed = 4
    kw = dict(rows_a=2, rows_b=256)
    vals = []
    for _ in range(args.warmup):
        cpu_baseline(host, mask, seed, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cb = cpu_baseline(host, mask, seed, **kw)
        vals.append(cb["value"])
        desc, cores = cb["sample"], cb["threads"]
    total = time.perf_counter() - t0
    value = statistics.mean(vals)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_name(), "tokens": TOKENS, "hidden": HIDDEN,
                                            "ffn": FFN},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": desc, **host_cpu()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def sweep_c5(args):
    """Quantizer bandwidth sweep: 2^20..2^29 elements at row lengths 3072,
    9216 and 8192, Student-t(3) values, six modes (two with 4/6 adaptive
    block scales; the last re-quantizes the row-wise operand of x into the
    col-wise RHT operand).  One JSON line per case;
    L2 is flushed before every timed call (a write of twice its size)."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    from fp4_gemm_nvfp4_gb300 import inputs, ops
    peaks, peak_src = load_peaks()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    ws = ops.Workspace()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    mask = inputs.rht_sign_mask(5)
    modes = [("1x16_rne", dict(rowwise=True)),
             ("16x16_rne", dict(rowwise=True, colwise=True, two_d=True)),
             ("rht_1x16_sr", dict(rowwise=True, sr=True, rht_mask=mask, seed=5)),
             ("1x16_46_rne", dict(rowwise=True, scale46=True)),
             ("rht_1x16_46_sr", dict(rowwise=True, sr=True, rht_mask=mask, seed=5, scale46=True)),
             ("requant_col_rht_sr", dict(requant=True, rht_mask=mask, seed=5))]
    stream = torch.cuda.current_stream()
    for rows, L in inputs.c5_sweep_sizes():
        x = torch.empty((rows, L), dtype=torch.bfloat16, device="cuda")
        for r0 in range(0, rows, 4096):   # t(3) = Z / sqrt(chi2_3 / 3), drawn in chunks
            r1 = min(rows, r0 + 4096)
            z = torch.randn((r1 - r0, L), generator=gen, device="cuda")
            chi = torch.randn((3, r1 - r0, L), generator=gen, device="cuda").square_().mean(0).sqrt_()
            x[r0:r1] = (z / chi * 1e-3).to(torch.bfloat16)
        del z, chi
        n = rows * L
        for name, kw in modes:
            row = ops.alloc_operand(rows, L)
            if kw.get("requant"):
                # Wgrad's operand re-quantized from the row-wise operand of x
                # (input: 0.5625 B per element, read by both passes)
                ops.quantize(x, out_row=row, workspace=ws)
                col = ops.alloc_operand(L, rows)
                run = lambda: ops.requantize_col_rht(row, kw["rht_mask"], sr=True, seed=kw["seed"], out_col=col,
                                                     workspace=ws)
            else:
                col = ops.alloc_operand(L, rows) if kw.get("colwise") else None
                run = lambda: ops.quantize(x, out_row=row, out_col=col, workspace=ws, **kw)
            for _ in range(max(args.warmup, 5)):
                run()
            times = []
            for _ in range(max(args.steps, 20)):
                flush.fill_(1.0)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run()
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.median(times)
            if kw.get("requant"):
                unique = n * 2 * (0.5 + 1 / 16)
                alg = n * 3 * (0.5 + 1 / 16)
            else:
                outs = 1 + int(bool(kw.get("colwise")))
                unique = n * (2 + outs * (0.5 + 1 / 16))
                alg = quant_bytes(rows, L, kw)
            print(json.dumps({"sweep": "c5", "mode": name, "rows": rows, "row_len": L, "elements": n,
                              "ms": round(ms, 4), "unique_gbs": round(unique / (ms * 1e-3) / 1e9, 1),
                              "algorithmic_gbs": round(alg / (ms * 1e-3) / 1e9, 1),
                              "frac_of_hbm": round(alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                              "peak_source": f"{peak_src} hbm_gbs", "l2_flush": True,
                              "status": ops.device_error()}), flush=True)
            del row, col
        del x
        torch.cuda.empty_cache()


def sweep_ns(args):
    """The NVFP4 Newton-Schulz step ("Full-Stack FP4", Sec. 3.4) on the 3B
    model's weight shapes (X is [m][n] with m the smaller dimension: FFN 3072 x
    9216, QKV 3072 x 6144, O 3072 x 3072), Muon coefficients, inputs G / ||G||_F.
    One JSON line per shape: the step through nvfp4_newton_schulz_step, and its
    three quantize calls and three GEMMs timed one by one (CUDA events on the
    launching stream, L2 flushed before every timed call)."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    from fp4_gemm_nvfp4_gb300 import capi, inputs, ops
    peaks, peak_src = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    a, b, c = 3.4445, -4.7750, 2.0315
    mask = inputs.rht_sign_mask(6)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(6)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        times = []
        for _ in range(max(args.steps, 10)):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    for name, m, n in [("ffn", 3072, 9216), ("qkv", 3072, 6144), ("o", 3072, 3072)]:
        g = torch.randn((m, n), generator=gen, device="cuda")
        x = (g / g.norm()).to(torch.bfloat16)
        del g
        ws = torch.empty(capi.nvfp4_newton_schulz_workspace_size(m, n), dtype=torch.uint8, device="cuda")
        out = torch.empty_like(x)
        step_ms = timed(lambda: ops.newton_schulz_step(x, a, b, c, mask, out=out, workspace=ws))
        # the same work call by call
        qws = ops.Workspace()
        qx, qxc = ops.alloc_operand(m, n), ops.alloc_operand(n, m)
        qa, qac, qb = ops.alloc_operand(m, m), ops.alloc_operand(m, m), ops.alloc_operand(m, m)
        A = torch.empty((m, m), dtype=torch.bfloat16, device="cuda")
        B = torch.empty_like(A)
        parts = [
            ("q_x_pair", lambda: ops.quantize(x, rht_mask=mask, rowwise=True, colwise=True, scale46=True,
                                              out_row=qx, out_col=qxc, workspace=qws), None),
            ("gemm_xxt", lambda: ops.gemm(qx, qx, out=A), 2 * m * m * n),
            ("q_a_pair", lambda: ops.quantize(A, rht_mask=mask, rowwise=True, colwise=True, scale46=True,
                                              out_row=qa, out_col=qac, workspace=qws), None),
            ("gemm_aa", lambda: ops.gemm_axpby(qa, qac, c, A, b, out=B), 2 * m * m * m),
            ("q_b_row", lambda: ops.quantize(B, rht_mask=mask, rowwise=True, scale46=True, out_row=qb,
                                             workspace=qws), None),
            ("gemm_bx", lambda: ops.gemm_axpby(qb, qxc, 1.0, x, a, out=out), 2 * m * n * m),
        ]
        for _, fn, _ in parts:   # intermediates for the later parts
            fn()
        res = {}
        gemm_ms = gemm_flop = 0.0
        for pname, fn, flop in parts:
            ms = timed(fn)
            res[pname] = {"ms": round(ms, 4)}
            if flop:
                res[pname]["tflops"] = round(flop / (ms * 1e-3) / 1e12, 1)
                gemm_ms += ms
                gemm_flop += flop
        flop = 4 * m * m * n + 2 * m ** 3
        print(json.dumps({"sweep": "newton_schulz", "weight": name, "m": m, "n": n, "coefficients": [a, b, c],
                          "step_ms": round(step_ms, 4), "step_tflops": round(flop / (step_ms * 1e-3) / 1e12, 1),
                          "gemm_tflops": round(gemm_flop / (gemm_ms * 1e-3) / 1e12, 1),
                          "gemm_frac_of_fp4_peak": round(gemm_flop / (gemm_ms * 1e-3) / 1e12 / fp4_peak, 4),
                          "peak_source": f"{peak_src} bf16 burst x 6", "parts": res, "l2_flush": True,
                          "status": ops.device_error()}), flush=True)
        del x, ws, out, qx, qxc, qa, qac, qb, A, B
        torch.cuda.empty_cache()


def sweep_lora(args):
    """The GEMM with the BF16 low-rank (LoRA-SVD) branch, D = A B^T + beta U V^T
    ("Full-Stack FP4", the LoRA-SVD correction of a linear layer), against the
    plain GEMM on the C4 layer's Fprop shapes at ranks 64 and 128.  Random
    FP4 operands (codes and in-range E4M3 scales), U and V N(0, 0.02^2) BF16;
    one JSON line per case; L2 flushed before every timed call."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    from fp4_gemm_nvfp4_gb300 import capi, ops
    peaks, peak_src = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(8)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        times = []
        for _ in range(max(args.steps, 10)):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    for name, M, N, K in [("fprop_up", 16384, 9216, 3072), ("fprop_down", 16384, 3072, 9216)]:
        a, b = ops.alloc_operand(M, K), ops.alloc_operand(N, K)
        for op in (a, b):
            op.codes.copy_(torch.randint(0, 256, op.codes.shape, generator=gen, device="cuda",
                                         dtype=torch.int32).to(torch.uint8))
            op.scales.copy_(torch.randint(0x20, 0x48, op.scales.shape, generator=gen, device="cuda",
                                          dtype=torch.int32).to(torch.uint8))
            op.global_scale.fill_(1.0)
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        plain_ms = timed(lambda: ops.gemm(a, b, out=out))
        for r in (64, 128):
            u = (torch.randn((M, r), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
            v = (torch.randn((N, r), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
            scratch = torch.empty(capi.nvfp4_gemm_lora_workspace_size(M, r), dtype=torch.uint8,
                                  device="cuda")
            lora_ms = timed(lambda: ops.gemm_lora(a, b, u, v, 0.5, out=out, scratch=scratch))
            fp4_flop = 2 * M * N * K
            print(json.dumps({"sweep": "lora", "gemm": name, "m": M, "n": N, "k": K, "rank": r,
                              "plain_us": round(plain_ms * 1e3, 1), "lora_us": round(lora_ms * 1e3, 1),
                              "overhead_pct": round(100 * (lora_ms / plain_ms - 1), 1),
                              "low_rank_flop_pct": round(100 * 2 * M * N * r / fp4_flop, 2),
                              "fp4_tflops": round(fp4_flop / (lora_ms * 1e-3) / 1e12, 1),
                              "fp4_frac_of_peak": round(fp4_flop / (lora_ms * 1e-3) / 1e12 / fp4_peak, 4),
                              "peak_source": f"{peak_src} bf16 burst x 6", "l2_flush": True,
                              "status": ops.device_error()}), flush=True)
            del u, v, scratch
        del a, b, out
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fuse-amax", action="store_true",
                    help="quantize H and dY_up as inputs with their own amax pass (no fused GEMM amax)")
    ap.add_argument("--sweep", choices=["c5", "ns", "lora"], default=None,
                    help="instead of the layer step, run the quantizer bandwidth sweep (c5), the NVFP4 "
                         "Newton-Schulz step on the 3B weight shapes (ns) or the GEMM with the low-rank "
                         "branch against the plain GEMM (lora); one JSON line per case")
    ap.add_argument("--tokens", type=int, default=TOKENS,
                    help="tokens of the layer step (16384 is the benchmarked workload)")
    args = ap.parse_args()
    set_tokens(args.tokens)
    global FUSE_AMAX
    FUSE_AMAX = not args.no_fuse_amax
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    if args.sweep == "c5":
        sweep_c5(args)
        return
    if args.sweep == "ns":
        sweep_ns(args)
        return
    if args.sweep == "lora":
        sweep_lora(args)
        return
    if args.impl == "reference":
        r = reference_arm(args)
        if r is not None:
            print(json.dumps(r))
        return
    result, rank = measure(args)
    if rank == 0:
        print(json.dumps(result))


if __name__ == "__main__":
    main()
