#!/usr/bin/env python3
"""Decode-GEMV benchmark: one JSON line per run.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl wobs|reference]

A step is one pass of the decode path over one batch of synthetic input.
The default workload is the Q4_0 x Q8_1 M = 1 decode of an 8B model's four
projection shapes (4096x4096, 1024x4096, 14336x4096, 4096x14336): per
shape, one wobs_gemv_q4_0_f32 launch quantises the fp32 activation vector
to Q8_1 (writing the blocks) and runs the GEMV on it.  The weights are rotated over enough seeded copies that the working set exceeds
1.07 GB (the batch1-cdna README rotates 32 copies of a 4096^2 fp16 matrix
for the same reason), so every step reads its weights from HBM, not L2.

Other workloads (``--workload``): q4_m1_2call (the same decode as two
launches per shape, quantize_q8_1 then gemv_q4_0_q8_1), q8_m1 (Q8_0
weights, same shapes, quantisation fused; q8_m1_2call: two launches), argcmp (standalone argmax / argmin rows),
fp16_4096 (dense fp16 4096x4096), nf4
(NF4 28672x8192), q4_m_sweep (Q4_0 x Q8_1 for M in {1,..,32} on 4096x4096
and 14336x4096), lm_head (bf16 128000x4096 with fused argmax, M = 1 and 32).

Timing: W untimed warm-up steps, then exactly K steps between CUDA events
on the launching stream, bracketed by a barrier and a device synchronise;
the steps are replayed from CUDA graphs (one graph per rotation cycle of
the weight copies, single-step graphs for a remainder).  The
``value`` is bytes counted from the method (each weight, scale,
activation and output byte once) divided by the measured time.

``--impl reference`` times the CPU oracle instead (host cores, a row
sample of the same workload per step).  With N > 1 every rank runs an
independent replica (the path has no exchange step), ``value`` is the sum
over ranks divided by the slowest rank's time.
"""
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "M=1 GEMV µs/call and HBM GB/s as % of measured GB300 read ceiling (MBU)"
ROTATE_BYTES = 1.07e9
PROBE_BYTES = 8 << 30          # streaming-read ceiling buffer (>> L2)

# ----------------------------------------------------------------- dist


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(backend):
    import torch.distributed as dist
    if dist.is_available() and not dist.is_initialized() and int(os.environ.get("WORLD_SIZE", "1")) > 1:
        dist.init_process_group(backend=backend)


def _dist_on():
    import torch.distributed as dist
    return dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1


def barrier(device=None):
    import torch.distributed as dist
    if _dist_on():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_over_ranks(value, op, device=None):
    """MAX or SUM of a float over ranks (identity without a process group)."""
    import torch.distributed as dist
    if not _dist_on():
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(per_rank_bytes, per_rank_ms, device=None):
    """Whole-job throughput: bytes of all ranks / the slowest rank's time."""
    total = reduce_over_ranks(per_rank_bytes, "sum", device)
    ms = reduce_over_ranks(per_rank_ms, "max", device)
    return total / (ms * 1e-3) / 1e9, ms


# --------------------------------------------------------------- clocks

_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
            0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x100: "display_clock_setting"}


class ClockSampler:
    """SM clock and clock-event reasons sampled during the timed region.

    NVML through ctypes (every ~2 ms); ``nvidia-smi -lms 100`` if NVML is not
    loadable.  Reading clocks changes nothing on the GPU.
    """

    def __init__(self, device):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thr = None
        self._proc = None
        self._nvml = None
        self._handle = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                ok = False
                props = torch.cuda.get_device_properties(device)
                if hasattr(props, "pci_bus_id"):
                    bus = f"{getattr(props, 'pci_domain_id', 0):08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
                    ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
                if not ok:
                    ok = lib.nvmlDeviceGetHandleByIndex_v2(self._nvml_index(device), ctypes.byref(h)) == 0
                if ok:
                    self._nvml, self._handle = lib, h
                    m = ctypes.c_uint()
                    if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                        self.max_mhz = int(m.value)
        except OSError:
            self._nvml = None
        self._index = self._nvml_index(device)

    @staticmethod
    def _nvml_index(device):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        parts = [p for p in vis.split(",") if p.strip()]
        if parts and all(p.strip().isdigit() for p in parts):
            return int(parts[device.index].strip())
        return device.index

    def _poll(self):
        lib, h = self._nvml, self._handle
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        get_r = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0 and get_r(h, ctypes.byref(r)) == 0:
                self.samples.append((int(c.value), int(r.value)))
            time.sleep(0.002)

    def start(self):
        if self._nvml is not None:
            self._thr = threading.Thread(target=self._poll, daemon=True)
            self._thr.start()
        else:
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active")
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self._index), f"--query-gpu={q}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._proc = None

    def stop(self):
        if self._thr is not None:
            self._stop.set()
            self._thr.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            for line in out.splitlines():
                p = [s.strip() for s in line.split(",")]
                try:
                    self.samples.append((int(float(p[0])), int(p[2], 16)))
                    self.max_mhz = int(float(p[1]))
                except (ValueError, IndexError):
                    pass

    def report(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        seen = 0
        for _, r in self.samples:
            seen |= r
        names = [n for b, n in _REASONS.items() if seen & b and b != 0x1]
        return {"sm_mhz": statistics.median(s for s, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


# ------------------------------------------------------------- timing


class StepRunner:
    """Replays exactly ``n`` steps from CUDA graphs: whole rotation cycles of
    the weight copies from one graph, the remainder from one more graph
    (captured once per remainder length), so any step count costs at most
    q + 1 graph launches."""

    def __init__(self, wl, stream):
        self.wl, self.stream = wl, stream
        self.cycle = capture(lambda: [wl.step(c) for c in range(wl.copies)], stream)
        self.rest = {}

    def _rest(self, r):
        if r not in self.rest:
            self.rest[r] = capture(lambda: [self.wl.step(c) for c in range(r)], self.stream)
        return self.rest[r]

    def replay(self, n):
        q, r = divmod(n, self.wl.copies)
        for _ in range(q):
            self.cycle.replay()
        if r:
            self._rest(r).replay()

    def prepare(self, n):
        """Capture the remainder graph for ``n`` steps outside any timed region."""
        r = n % self.wl.copies
        if r:
            self._rest(r)


def time_steps(runner, steps, stream):
    """Exactly ``steps`` steps between CUDA events on ``stream``: milliseconds."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        runner.replay(steps)
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


class _GraphRunner:
    """A single captured graph replayed ``n`` times (one call site over all copies)."""

    def __init__(self, graph):
        self.g = graph

    def replay(self, n):
        for _ in range(n):
            self.g.replay()


def time_call_site(wl, fn, stream, reps):
    """One call site timed three ways: back to back over the rotated copies
    (one graph per rotation, five samples: median and interquartile range, us
    per call), and as an isolated launch (a one-call graph on copy 0, replayed
    right after a full rotation has evicted that copy from L2; events around
    it; median of seven)."""
    gk = _GraphRunner(capture(lambda: [fn(c) for c in range(wl.copies)], stream))
    time_steps(gk, 2, stream)
    samples = sorted(time_steps(gk, reps, stream) * 1e3 / (reps * wl.copies) for _ in range(5))
    g1 = capture(lambda: fn(0), stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    iso = []
    with torch.cuda.stream(stream):
        for _ in range(7):
            gk.replay(1)
            e0.record(stream)
            g1.replay()
            e1.record(stream)
            e1.synchronize()
            iso.append(e0.elapsed_time(e1) * 1e3)
    return samples[2], samples[3] - samples[1], statistics.median(iso)


def packed(shapes, dtype, device):
    """One flat device buffer and views of it with the given shapes (16-byte
    aligned offsets), so a step's inputs or outputs move in one copy."""
    esize = torch.empty(0, dtype=dtype).element_size()
    align = max(1, 16 // esize)
    offs, total = [], 0
    for shp in shapes:
        offs.append(total)
        total += (math.prod(shp) + align - 1) // align * align
    flat = torch.empty(total, dtype=dtype, device=device)
    return flat, [flat[o:o + math.prod(shp)].view(shp) for o, shp in zip(offs, shapes)]


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def read_ceiling(device, stream, nbytes=PROBE_BYTES):
    """Best streaming-read GB/s over load variants and grid sizes (bw_probe)."""
    import weight_only_bit_split_gb300 as wobs
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    buf.fill_(0x5A)
    out = torch.zeros(1, dtype=torch.int32, device=device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    best = (0.0, None)
    table = []
    with torch.cuda.stream(stream):
        for variant in (1, 2, 3):
            for per_sm in (1, 2, 4, 8):
                grid = sms * per_sm
                wobs.wobs_bw_probe(buf, grid=grid, variant=variant, xor_out=out)
                ts = []
                for _ in range(5):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    wobs.wobs_bw_probe(buf, grid=grid, variant=variant, xor_out=out)
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1))
                gbs = nbytes / (statistics.median(ts) * 1e-3) / 1e9
                table.append({"variant": variant, "grid": grid, "gbs": round(gbs, 1)})
                if gbs > best[0]:
                    best = (gbs, {"variant": variant, "grid": grid})
    if wobs.wobs_error_word(device) != 0:
        raise RuntimeError("bw_probe reported a device error")
    del buf
    torch.cuda.empty_cache()
    return best[0], best[1], table


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_record(kernel):
    """ncu DRAM bytes per launch for ``kernel`` if recorded for the current source."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    recs = {}
    for line in open(p):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        if len(parts) >= 4:
            recs[parts[0]] = (parts[1], parts[2], parts[3])
    if kernel not in recs:
        return None
    src, digest, per_launch = recs[kernel]
    path = os.path.join(ROOT, "weight_only_bit_split_gb300", "csrc", src)
    if not os.path.exists(path):
        return None
    if hashlib.sha256(open(path, "rb").read()).hexdigest()[:16] != digest:
        return None
    return float(per_launch)


# ------------------------------------------------------------ workloads


class Q4M1:
    """Q4_0 x Q8_1, M = 1, the four 8B projection shapes: quantise then GEMV
    as two launches per shape."""
    name = "q4_0_q8_1_m1_8b_shapes_two_launch"
    shapes = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]
    dtype = "int8"
    kernel = "q4_0_q8_1_m1_cp"
    kernel_src = "q4_0.cu"
    workload_id = 2

    def __init__(self, device):
        import weight_only_bit_split_gb300 as wobs
        from weight_only_bit_split_gb300 import synth
        self.wobs = wobs
        wbytes = sum(0.5625 * n * k for n, k in self.shapes)
        self.copies = max(1, math.ceil(ROTATE_BYTES / wbytes))
        self.planes = []
        for c in range(self.copies):
            row = []
            for n, k in self.shapes:
                w = synth.weights(self.workload_id, (n, k), copy=c, device=device)
                row.append(wobs.wobs_quantize_q4_0(w))
                del w
            self.planes.append(row)
        self.x_all, self.x = packed([(1, k) for _, k in self.shapes], torch.float32, device)
        for xv, (_, k) in zip(self.x, self.shapes):
            xv.copy_(synth.activations(self.workload_id, (1, k), device=device))
        self.xq = [torch.empty(1, k // 32 * 36, dtype=torch.uint8, device=device) for _, k in self.shapes]
        self.y_all, self.y = packed([(1, n) for n, _ in self.shapes], torch.float32, device)
        torch.cuda.synchronize(device)

    @staticmethod
    def gemv_bytes(n, k):
        return int(0.5625 * n * k) + 36 * k // 32 + 4 * n

    @staticmethod
    def quant_bytes(k):
        return 4 * k + 36 * k // 32

    def bytes_per_step(self):
        return sum(self.gemv_bytes(n, k) + self.quant_bytes(k) for n, k in self.shapes)

    launches_per_step = 8

    def step(self, c):
        w = self.wobs
        for s in range(len(self.shapes)):
            w.wobs_quantize_q8_1(self.x[s], self.xq[s])
            qs, d = self.planes[c][s]
            w.wobs_gemv_q4_0_q8_1(qs, d, self.xq[s], y=self.y[s])

    def kernel_calls(self):
        """(label, bytes, fn(copy)) for each launch of the dominant kernel."""
        out = []
        for s, (n, k) in enumerate(self.shapes):
            def fn(c, s=s):
                qs, d = self.planes[c][s]
                self.wobs.wobs_gemv_q4_0_q8_1(qs, d, self.xq[s], y=self.y[s])
            out.append((f"{n}x{k}", self.gemv_bytes(n, k), fn))
        return out

    def e2e_setup(self):
        # the step's activations and outputs each live in one packed buffer
        self.xh = self.x_all.cpu().pin_memory()
        self.yh = torch.empty(self.y_all.shape, dtype=self.y_all.dtype).pin_memory()
        return self.xh.numel() * 4, self.yh.numel() * 4

    def e2e_step(self, c):
        self.x_all.copy_(self.xh, non_blocking=True)
        self.step(c)
        self.yh.copy_(self.y_all, non_blocking=True)

    def config(self):
        return {"workload": self.name, "shapes_NxK": [f"{n}x{k}" for n, k in self.shapes], "M": 1,
                "step": "per shape: quantize_q8_1(x) then gemv_q4_0_q8_1",
                "weight_copies": self.copies,
                "working_set_gb": round(self.copies * sum(0.5625 * n * k for n, k in self.shapes) / 1e9, 3),
                "l2": "inputs larger than L2: rotated weight copies, working set above 1 GB"}

    # ---- oracle (CPU) ----
    @classmethod
    def oracle_prepare(cls, frac):
        import oracle
        from weight_only_bit_split_gb300 import synth
        prep = []
        for n, k in cls.shapes:
            rows = max(1, int(round(n * frac)))
            w = synth.weights(cls.workload_id, (rows, k)).numpy()
            q4, d4 = oracle.quantize_q4_0(w)
            x = synth.activations(cls.workload_id, (1, k)).numpy()
            prep.append((oracle.pack_q4_0(q4), d4, x, rows, k))
        return prep

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        nbytes = 0
        for qs, d4, x, rows, k in prep:
            q8, d8, _ = oracle.quantize_q8_1(x)
            oracle.gemv_q4_0_q8_1(qs, d4, q8, d8)
            nbytes += cls.gemv_bytes(rows, k) + cls.quant_bytes(k)
        return nbytes


class Q4M1Fused(Q4M1):
    """The same decode with the Q8_1 quantisation fused into the GEMV
    (wobs_gemv_q4_0_f32): one launch per shape reads the fp32 activations,
    writes their Q8_1 blocks (sum field included) and the outputs."""
    name = "q4_0_q8_1_m1_8b_shapes"
    kernel = "q4_0_f32_m1_cp"
    launches_per_step = 4

    @staticmethod
    def fused_bytes(n, k):
        return int(0.5625 * n * k) + 4 * k + 36 * k // 32 + 4 * n

    def bytes_per_step(self):
        return sum(self.fused_bytes(n, k) for n, k in self.shapes)

    def step(self, c):
        w = self.wobs
        for s in range(len(self.shapes)):
            qs, d = self.planes[c][s]
            w.wobs_gemv_q4_0_f32(qs, d, self.x[s], y=self.y[s], xq_out=self.xq[s])

    def kernel_calls(self):
        out = []
        for s, (n, k) in enumerate(self.shapes):
            def fn(c, s=s):
                qs, d = self.planes[c][s]
                self.wobs.wobs_gemv_q4_0_f32(qs, d, self.x[s], y=self.y[s], xq_out=self.xq[s])
            out.append((f"{n}x{k}", self.fused_bytes(n, k), fn))
        return out

    def config(self):
        cfg = super().config()
        cfg["step"] = ("per shape: gemv_q4_0_f32(x) -- quantize_q8_1 fused into the GEMV kernel "
                       "(Q8_1 blocks written, bit-identical to the two-launch path)")
        return cfg

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        nbytes = 0
        for qs, d4, x, rows, k in prep:
            q8, d8, s8 = oracle.quantize_q8_1(x)
            oracle.pack_q8_1(q8, d8, s8)
            oracle.gemv_q4_0_q8_1(qs, d4, q8, d8)
            nbytes += cls.fused_bytes(rows, k)
        return nbytes


class Q4Sweep(Q4M1):
    """Q4_0 x Q8_1 for M in {1, 2, 4, 8, 12, 16, 24, 32} on two shapes."""
    name = "q4_0_q8_1_m_sweep"
    shapes = [(4096, 4096), (14336, 4096)]
    Ms = (1, 2, 4, 8, 12, 16, 24, 32)
    # the roofline figure is the dominant kernel's: the mma.sync kernel
    # (M = 5..16) takes the largest share of the step
    kernel = "q4_0_q8_1_mma"
    kernel_src = "q4_mma.cu"
    workload_id = 4

    @classmethod
    def roofline_call(cls, label):
        return int(label[1:].split("_")[0]) in (8, 12, 16)

    def __init__(self, device):
        super().__init__(device)
        from weight_only_bit_split_gb300 import synth
        k = self.shapes[0][1]
        self.X_all, xs = packed([(m, k) for m in self.Ms], torch.float32, device)
        self.X = dict(zip(self.Ms, xs))
        for m in self.Ms:
            self.X[m].copy_(synth.activations(self.workload_id, (m, k), copy=m, device=device))
        self.XQ = {m: torch.empty(m, k // 32 * 36, dtype=torch.uint8, device=device) for m in self.Ms}
        keys = [(m, s) for m in self.Ms for s in range(len(self.shapes))]
        self.Y_all, ys = packed([(m, self.shapes[s][0]) for m, s in keys], torch.float32, device)
        self.Y = dict(zip(keys, ys))
        self.ws = {(m, s): self.wobs.workspace(self.wobs.OP_GEMV_Q4_0_Q8_1, m, n, k, device)
                   for m in self.Ms for s, (n, _) in enumerate(self.shapes)}
        self.ws = {key: (torch.zeros_like(v) if v is not None else None) for key, v in self.ws.items()}

    @staticmethod
    def gemv_bytes_m(n, k, m):
        return int(0.5625 * n * k) + m * 36 * k // 32 + 4 * m * n

    def bytes_per_step(self):
        k = self.shapes[0][1]
        return sum(self.gemv_bytes_m(n, k, m) for m in self.Ms for n, _ in self.shapes) + \
            sum(m * self.quant_bytes(k) for m in self.Ms)

    launches_per_step = len(Ms) * 3

    def _gemv(self, c, s, m):
        qs, d = self.planes[c][s]
        ws = self.ws[(m, s)]
        self.wobs.wobs_gemv_q4_0_q8_1(qs, d, self.XQ[m], y=self.Y[(m, s)], ws=ws)

    def step(self, c):
        for m in self.Ms:
            self.wobs.wobs_quantize_q8_1(self.X[m], self.XQ[m])
            for s in range(len(self.shapes)):
                self._gemv(c, s, m)

    def kernel_calls(self):
        out = []
        for m in self.Ms:
            for s, (n, k) in enumerate(self.shapes):
                out.append((f"M{m}_{n}x{k}", self.gemv_bytes_m(n, k, m),
                            lambda c, s=s, m=m: self._gemv(c, s, m)))
        return out

    def e2e_setup(self):
        self.xh = self.X_all.cpu().pin_memory()
        self.yh = torch.empty(self.Y_all.shape, dtype=self.Y_all.dtype).pin_memory()
        return self.xh.numel() * 4, self.yh.numel() * 4

    def e2e_step(self, c):
        self.X_all.copy_(self.xh, non_blocking=True)
        self.step(c)
        self.yh.copy_(self.Y_all, non_blocking=True)

    def config(self):
        c = super().config()
        c.update({"workload": self.name, "M": list(self.Ms),
                  "step": "per M: quantize_q8_1(X) then gemv_q4_0_q8_1 on both shapes"})
        return c

    @classmethod
    def oracle_prepare(cls, frac):
        import oracle
        from weight_only_bit_split_gb300 import synth
        prep = []
        for n, k in cls.shapes:
            rows = max(1, int(round(n * frac)))
            w = synth.weights(cls.workload_id, (rows, k)).numpy()
            q4, d4 = oracle.quantize_q4_0(w)
            prep.append((oracle.pack_q4_0(q4), d4, rows, k))
        xs = {m: synth.activations(cls.workload_id, (m, cls.shapes[0][1]), copy=m).numpy() for m in cls.Ms}
        return prep, xs

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        mats, xs = prep
        nbytes = 0
        for m in cls.Ms:
            q8, d8, _ = oracle.quantize_q8_1(xs[m])
            for qs, d4, rows, k in mats:
                oracle.gemv_q4_0_q8_1(qs, d4, q8, d8)
                nbytes += cls.gemv_bytes_m(rows, k, m)
            nbytes += m * cls.quant_bytes(mats[0][3])
        return nbytes


class DenseF16:
    name = "fp16_gemv_4096x4096"
    n, k = 4096, 4096
    dtype = "f32"
    kernel = "dense_m1_cp"
    kernel_src = "dense.cu"
    workload_id = 1
    launches_per_step = 1

    def __init__(self, device):
        import weight_only_bit_split_gb300 as wobs
        from weight_only_bit_split_gb300 import synth
        self.wobs = wobs
        self.copies = max(1, math.ceil(ROTATE_BYTES / (2 * self.n * self.k)))
        self.W = [synth.weights(self.workload_id, (self.n, self.k), copy=c, device=device, dtype=torch.float16)
                  for c in range(self.copies)]
        self.x = synth.activations(self.workload_id, (1, self.k), device=device, dtype=torch.float16)
        self.y = torch.empty(1, self.n, dtype=torch.float16, device=device)

    @classmethod
    def gemv_bytes(cls):
        return 2 * cls.n * cls.k + 2 * cls.k + 2 * cls.n

    def bytes_per_step(self):
        return self.gemv_bytes()

    def step(self, c):
        self.wobs.wobs_gemv_f16(self.W[c], self.x, self.y)

    def kernel_calls(self):
        return [(f"{self.n}x{self.k}", self.gemv_bytes(), self.step)]

    def e2e_setup(self):
        self.xh = self.x.cpu().pin_memory()
        self.yh = torch.empty(self.y.shape, dtype=self.y.dtype).pin_memory()
        return self.xh.numel() * 2, self.yh.numel() * 2

    def e2e_step(self, c):
        self.x.copy_(self.xh, non_blocking=True)
        self.step(c)
        self.yh.copy_(self.y, non_blocking=True)

    def config(self):
        return {"workload": self.name, "shapes_NxK": [f"{self.n}x{self.k}"], "M": 1,
                "weight_copies": self.copies,
                "working_set_gb": round(self.copies * 2 * self.n * self.k / 1e9, 3),
                "l2": "inputs larger than L2: rotated weight copies, working set above 1 GB"}

    @classmethod
    def oracle_prepare(cls, frac):
        from weight_only_bit_split_gb300 import synth
        rows = max(1, int(round(cls.n * frac)))
        w = synth.weights(cls.workload_id, (rows, cls.k), dtype=torch.float16).numpy()
        x = synth.activations(cls.workload_id, (1, cls.k), dtype=torch.float16).numpy()
        return w, x, rows

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        w, x, rows = prep
        oracle.gemv_dense(w, x)
        return 2 * rows * cls.k + 2 * cls.k + 2 * rows


class NF4:
    name = "nf4_gemv_28672x8192"
    n, k = 28672, 8192
    dtype = "f32"
    kernel = "nf4_mma"
    kernel_src = "nf4_mma.cu"
    workload_id = 3
    launches_per_step = 1

    def __init__(self, device):
        import weight_only_bit_split_gb300 as wobs
        from weight_only_bit_split_gb300 import synth
        from weight_only_bit_split_gb300.nf4_levels import normal_float_levels
        self.wobs = wobs
        self.cb = normal_float_levels().numpy()
        self.copies = max(1, math.ceil(ROTATE_BYTES / self.gemv_bytes()))
        self.planes = []
        for c in range(self.copies):
            w = synth.weights(self.workload_id, (self.n, self.k), copy=c, device=device, dtype=torch.bfloat16)
            self.planes.append(wobs.wobs_quantize_nf4(w, self.cb))
            del w
        self.x = synth.activations(self.workload_id, (self.k,), device=device, dtype=torch.bfloat16)
        self.y = torch.empty(self.n, dtype=torch.bfloat16, device=device)

    @classmethod
    def gemv_bytes(cls):
        return cls.n * cls.k // 2 + 4 * cls.n * cls.k // 64 + 2 * cls.k + 2 * cls.n

    def bytes_per_step(self):
        return self.gemv_bytes()

    def step(self, c):
        qs, am = self.planes[c]
        self.wobs.wobs_gemv_nf4(qs, am, self.cb, self.x, y=self.y)

    def kernel_calls(self):
        return [(f"{self.n}x{self.k}", self.gemv_bytes(), self.step)]

    def e2e_setup(self):
        self.xh = self.x.cpu().pin_memory()
        self.yh = torch.empty(self.y.shape, dtype=self.y.dtype).pin_memory()
        return self.xh.numel() * 2, self.yh.numel() * 2

    def e2e_step(self, c):
        self.x.copy_(self.xh, non_blocking=True)
        self.step(c)
        self.yh.copy_(self.y, non_blocking=True)

    def config(self):
        return {"workload": self.name, "shapes_NxK": [f"{self.n}x{self.k}"], "M": 1,
                "weight_copies": self.copies,
                "working_set_gb": round(self.copies * self.gemv_bytes() / 1e9, 3),
                "l2": "inputs larger than L2: rotated weight copies, working set above 1 GB"}

    @classmethod
    def oracle_prepare(cls, frac):
        import oracle
        from weight_only_bit_split_gb300 import synth
        from weight_only_bit_split_gb300.nf4_levels import normal_float_levels
        cb = normal_float_levels().numpy()
        rows = max(1, int(round(cls.n * frac)))
        w = synth.weights(cls.workload_id, (rows, cls.k), dtype=torch.bfloat16).float().numpy()
        codes, absmax = oracle.quantize_nf4(w, cb)
        x = synth.activations(cls.workload_id, (cls.k,), dtype=torch.bfloat16).float().numpy()
        return oracle.pack_nf4(codes), absmax, cb, x, rows

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        qs, absmax, cb, x, rows = prep
        oracle.gemv_nf4(qs, absmax, cb, x)
        return rows * cls.k // 2 + 4 * rows * cls.k // 64 + 2 * cls.k + 2 * rows


class NF4Sweep:
    """NF4 28672x8192 with M in {1, 2, 4, 8, 16, 32} activation columns (the
    bitsandbytes thread's 70B MLP matrix; M = 1 is the one-token decode, M > 1
    a small decode batch), one wobs_gemv_nf4 per M per step.  The dequantise-
    then-GEMM alternative (wobs_dequantize_nf4 into a bf16 matrix, then the
    dense bf16 GEMV over 32 columns) is timed beside it as an extra call."""
    name = "nf4_gemv_28672x8192_m_sweep"
    n, k = 28672, 8192
    Ms = (1, 2, 4, 8, 16, 32)
    dtype = "f32"
    kernel = "nf4_tc"
    kernel_src = "nf4_tc.cu"
    workload_id = 3
    launches_per_step = len(Ms)

    @classmethod
    def roofline_call(cls, label):
        return int(label[1:]) > 4                # M = 1..4 run nf4_mma

    def __init__(self, device):
        import weight_only_bit_split_gb300 as wobs
        from weight_only_bit_split_gb300 import synth
        from weight_only_bit_split_gb300.nf4_levels import normal_float_levels
        self.wobs = wobs
        self.cb = normal_float_levels().numpy()
        self.copies = max(1, math.ceil(ROTATE_BYTES / self.gemv_bytes(1)))
        self.planes = []
        for c in range(self.copies):
            w = synth.weights(self.workload_id, (self.n, self.k), copy=c, device=device, dtype=torch.bfloat16)
            self.planes.append(wobs.wobs_quantize_nf4(w, self.cb))
            del w
        self.X_all, xs = packed([(m, self.k) for m in self.Ms], torch.bfloat16, device)
        self.X = dict(zip(self.Ms, xs))
        for m in self.Ms:
            self.X[m].copy_(synth.activations(self.workload_id, (m, self.k), copy=m, device=device,
                                              dtype=torch.bfloat16))
        self.Y_all, ys = packed([(m, self.n) for m in self.Ms], torch.bfloat16, device)
        self.Y = dict(zip(self.Ms, ys))
        self.ws = {m: wobs.workspace(wobs.OP_GEMV_NF4, m, self.n, self.k, device) for m in self.Ms}
        self.Wd = torch.empty(self.n, self.k, dtype=torch.bfloat16, device=device)
        self.Ld = torch.empty(32, self.n, dtype=torch.float32, device=device)
        torch.cuda.synchronize(device)

    @classmethod
    def gemv_bytes(cls, m):
        return cls.n * cls.k // 2 + 4 * cls.n * cls.k // 64 + 2 * m * cls.k + 2 * m * cls.n

    def bytes_per_step(self):
        return sum(self.gemv_bytes(m) for m in self.Ms)

    def _call(self, c, m):
        qs, am = self.planes[c]
        self.wobs.wobs_gemv_nf4(qs, am, self.cb, self.X[m], y=self.Y[m], ws=self.ws[m])

    def step(self, c):
        for m in self.Ms:
            self._call(c, m)

    def kernel_calls(self):
        return [(f"M{m}", self.gemv_bytes(m), lambda c, m=m: self._call(c, m)) for m in self.Ms]

    def extra_calls(self):
        def dq(c):
            qs, am = self.planes[c]
            self.wobs.wobs_dequantize_nf4(qs, am, self.cb, W=self.Wd)
            self.wobs.wobs_gemv_bf16(self.Wd, self.X[32], logits=self.Ld)
        return [("dequant+gemm_M32", self.gemv_bytes(32), dq)]

    def e2e_setup(self):
        self.xh = self.X_all.cpu().pin_memory()
        self.yh = torch.empty(self.Y_all.shape, dtype=self.Y_all.dtype).pin_memory()
        return self.xh.numel() * 2, self.yh.numel() * 2

    def e2e_step(self, c):
        self.X_all.copy_(self.xh, non_blocking=True)
        self.step(c)
        self.yh.copy_(self.Y_all, non_blocking=True)

    def config(self):
        return {"workload": self.name, "shapes_NxK": [f"{self.n}x{self.k}"], "M": list(self.Ms),
                "weight_copies": self.copies,
                "working_set_gb": round(self.copies * self.gemv_bytes(1) / 1e9, 3),
                "l2": "inputs larger than L2: rotated weight copies, working set above 1 GB"}

    @classmethod
    def oracle_prepare(cls, frac):
        import oracle
        from weight_only_bit_split_gb300 import synth
        from weight_only_bit_split_gb300.nf4_levels import normal_float_levels
        cb = normal_float_levels().numpy()
        rows = max(1, int(round(cls.n * frac)))
        w = synth.weights(cls.workload_id, (rows, cls.k), dtype=torch.bfloat16).float().numpy()
        codes, absmax = oracle.quantize_nf4(w, cb)
        xs = {m: synth.activations(cls.workload_id, (m, cls.k), copy=m, dtype=torch.bfloat16).float().numpy()
              for m in cls.Ms}
        return oracle.pack_nf4(codes), absmax, cb, xs, rows

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        qs, absmax, cb, xs, rows = prep
        nbytes = 0
        for m in cls.Ms:
            oracle.gemv_nf4(qs, absmax, cb, xs[m])
            nbytes += rows * cls.k // 2 + 4 * rows * cls.k // 64 + 2 * m * cls.k + 2 * m * rows
        return nbytes


class LmHead:
    name = "bf16_lm_head_argmax_128000x4096"
    n, k = 128000, 4096
    Ms = (1, 32)
    dtype = "f32"
    kernel = "dense_tc"
    kernel_src = "dense_tc.cu"
    workload_id = 5
    launches_per_step = 2

    def __init__(self, device):
        import weight_only_bit_split_gb300 as wobs
        from weight_only_bit_split_gb300 import synth
        self.wobs = wobs
        self.copies = max(2, math.ceil(ROTATE_BYTES / (2 * self.n * self.k)))
        self.W = [synth.weights(self.workload_id, (self.n, self.k), copy=c, device=device, dtype=torch.bfloat16)
                  for c in range(self.copies)]
        self.X = {m: synth.activations(self.workload_id, (m, self.k), copy=m, device=device, dtype=torch.bfloat16)
                  for m in self.Ms}
        self.L = {m: torch.empty(m, self.n, dtype=torch.float32, device=device) for m in self.Ms}
        self.A = {m: torch.empty(m, dtype=torch.int64, device=device) for m in self.Ms}
        self.ws = {m: torch.zeros(wobs.wobs_workspace_size(wobs.OP_GEMV_BF16, m, self.n, self.k),
                                  dtype=torch.uint8, device=device) for m in self.Ms}

    @classmethod
    def gemv_bytes(cls, m):
        return 2 * cls.n * cls.k + 2 * m * cls.k + 4 * m * cls.n + 8 * m

    def bytes_per_step(self):
        return sum(self.gemv_bytes(m) for m in self.Ms)

    def _call(self, c, m):
        self.wobs.wobs_gemv_bf16(self.W[c], self.X[m], logits=self.L[m], argmax=self.A[m], ws=self.ws[m])

    def step(self, c):
        for m in self.Ms:
            self._call(c, m)

    def kernel_calls(self):
        return [(f"M{m}", self.gemv_bytes(m), lambda c, m=m: self._call(c, m)) for m in self.Ms]

    def e2e_setup(self):
        self.xh = {m: x.cpu().pin_memory() for m, x in self.X.items()}
        self.ah = {m: torch.empty(m, dtype=torch.int64).pin_memory() for m in self.Ms}
        return sum(x.numel() * 2 for x in self.xh.values()), sum(8 * m for m in self.Ms)

    def e2e_step(self, c):
        for m in self.Ms:
            self.X[m].copy_(self.xh[m], non_blocking=True)
            self._call(c, m)
            self.ah[m].copy_(self.A[m], non_blocking=True)

    def config(self):
        return {"workload": self.name, "shapes_NxK": [f"{self.n}x{self.k}"], "M": list(self.Ms),
                "weight_copies": self.copies, "working_set_gb": round(self.copies * 2 * self.n * self.k / 1e9, 3),
                "l2": "inputs larger than L2: each weight copy is 1.05 GB"}

    @classmethod
    def oracle_prepare(cls, frac):
        from weight_only_bit_split_gb300 import synth
        rows = max(1, int(round(cls.n * frac)))
        w = synth.weights(cls.workload_id, (rows, cls.k), dtype=torch.bfloat16).float().numpy()
        xs = {m: synth.activations(cls.workload_id, (m, cls.k), copy=m, dtype=torch.bfloat16).float().numpy()
              for m in cls.Ms}
        return w, xs, rows

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        w, xs, rows = prep
        nbytes = 0
        for m in cls.Ms:
            oracle.argmax_rows(oracle.gemv_dense(w, xs[m]).astype(np.float32))
            nbytes += 2 * rows * cls.k + 2 * m * cls.k + 4 * m * rows + 8 * m
        return nbytes


class Q8M1(Q4M1):
    """Q8_0 x Q8_1, M = 1, the four 8B projection shapes (the case study's
    other tested weight format): quantise then GEMV, two launches per shape."""
    name = "q8_0_q8_1_m1_8b_shapes_two_launch"
    kernel = "q8_0_q8_1_mc_cp"
    kernel_src = "q8_0.cu"
    wbpw = 1.0625                                   # bytes per weight

    def __init__(self, device):
        import weight_only_bit_split_gb300 as wobs
        from weight_only_bit_split_gb300 import synth
        self.wobs = wobs
        wbytes = sum(self.wbpw * n * k for n, k in self.shapes)
        self.copies = max(1, math.ceil(ROTATE_BYTES / wbytes))
        self.planes = []
        for c in range(self.copies):
            row = []
            for n, k in self.shapes:
                w = synth.weights(self.workload_id, (n, k), copy=c, device=device)
                row.append(wobs.wobs_quantize_q8_0(w))
                del w
            self.planes.append(row)
        self.x_all, self.x = packed([(1, k) for _, k in self.shapes], torch.float32, device)
        for xv, (_, k) in zip(self.x, self.shapes):
            xv.copy_(synth.activations(self.workload_id, (1, k), device=device))
        self.xq = [torch.empty(1, k // 32 * 36, dtype=torch.uint8, device=device) for _, k in self.shapes]
        self.y_all, self.y = packed([(1, n) for n, _ in self.shapes], torch.float32, device)
        torch.cuda.synchronize(device)

    @staticmethod
    def gemv_bytes(n, k):
        return n * k + 2 * (n * k // 32) + 36 * k // 32 + 4 * n

    def step(self, c):
        w = self.wobs
        for s in range(len(self.shapes)):
            w.wobs_quantize_q8_1(self.x[s], self.xq[s])
            qs, d = self.planes[c][s]
            w.wobs_gemv_q8_0_q8_1(qs, d, self.xq[s], y=self.y[s])

    def kernel_calls(self):
        out = []
        for s, (n, k) in enumerate(self.shapes):
            def fn(c, s=s):
                qs, d = self.planes[c][s]
                self.wobs.wobs_gemv_q8_0_q8_1(qs, d, self.xq[s], y=self.y[s])
            out.append((f"{n}x{k}", self.gemv_bytes(n, k), fn))
        return out

    def config(self):
        cfg = super().config()
        cfg["step"] = "per shape: quantize_q8_1(x) then gemv_q8_0_q8_1"
        cfg["working_set_gb"] = round(self.copies * sum(self.wbpw * n * k for n, k in self.shapes) / 1e9, 3)
        return cfg

    @classmethod
    def oracle_prepare(cls, frac):
        import oracle
        from weight_only_bit_split_gb300 import synth
        prep = []
        for n, k in cls.shapes:
            rows = max(1, int(round(n * frac)))
            w = synth.weights(cls.workload_id, (rows, k)).numpy()
            qw, dw = oracle.quantize_q8_0(w)
            x = synth.activations(cls.workload_id, (1, k)).numpy()
            prep.append((qw, dw, x, rows, k))
        return prep

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        nbytes = 0
        for qw, dw, x, rows, k in prep:
            q8, d8, _ = oracle.quantize_q8_1(x)
            oracle.gemv_q8_0_q8_1(qw, dw, q8, d8)
            nbytes += cls.gemv_bytes(rows, k) + cls.quant_bytes(k)
        return nbytes


class Q8M1Fused(Q8M1):
    """Q8_0, M = 1, the four 8B shapes with the Q8_1 quantisation fused into
    the GEMV (wobs_gemv_q8_0_f32): one launch per shape."""
    name = "q8_0_q8_1_m1_8b_shapes"
    kernel = "q8_0_f32_m1_cp"
    launches_per_step = 4

    @classmethod
    def fused_bytes(cls, n, k):
        return n * k + 2 * (n * k // 32) + 4 * k + 36 * k // 32 + 4 * n

    def bytes_per_step(self):
        return sum(self.fused_bytes(n, k) for n, k in self.shapes)

    def step(self, c):
        w = self.wobs
        for s in range(len(self.shapes)):
            qs, d = self.planes[c][s]
            w.wobs_gemv_q8_0_f32(qs, d, self.x[s], y=self.y[s], xq_out=self.xq[s])

    def kernel_calls(self):
        out = []
        for s, (n, k) in enumerate(self.shapes):
            def fn(c, s=s):
                qs, d = self.planes[c][s]
                self.wobs.wobs_gemv_q8_0_f32(qs, d, self.x[s], y=self.y[s], xq_out=self.xq[s])
            out.append((f"{n}x{k}", self.fused_bytes(n, k), fn))
        return out

    def config(self):
        cfg = super().config()
        cfg["step"] = ("per shape: gemv_q8_0_f32(x) -- quantize_q8_1 fused into the GEMV kernel "
                       "(Q8_1 blocks written, bit-identical to the two-launch path)")
        return cfg

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        nbytes = 0
        for qw, dw, x, rows, k in prep:
            q8, d8, s8 = oracle.quantize_q8_1(x)
            oracle.pack_q8_1(q8, d8, s8)
            oracle.gemv_q8_0_q8_1(qw, dw, q8, d8)
            nbytes += cls.fused_bytes(rows, k)
        return nbytes


class ArgCmp:
    """Standalone argmax / argmin over rows of the ArgCompare discussion's
    model table: LLaMA-3-8B vocabulary rows at batch 1 and 32 (bf16), a
    256000-entry Gemma row (bf16) and the Image Retrieval argmin over
    [32, 1M] f32."""
    name = "argcompare_rows"
    cases = (("llama3_b1", 1, 128000, torch.bfloat16, False),
             ("llama3_b32", 32, 128000, torch.bfloat16, False),
             ("gemma_b1", 1, 256000, torch.bfloat16, False),
             ("retrieval_argmin", 32, 1048576, torch.float32, True))
    dtype = "f32"
    kernel = "argcmp_cta"
    kernel_src = "argcmp.cu"
    workload_id = 6
    launches_per_step = 4

    def __init__(self, device):
        import weight_only_bit_split_gb300 as wobs
        from weight_only_bit_split_gb300 import synth
        self.wobs = wobs
        self.copies = max(1, math.ceil(ROTATE_BYTES / self.bytes_per_step()))
        self.X = [[synth.normal((m, n), 1.0, synth.seed_of(self.workload_id, 2, c), device=device,
                                dtype=dt) for _, m, n, dt, _ in self.cases] for c in range(self.copies)]
        self.out = [torch.empty(m, dtype=torch.int64, device=device) for _, m, _, _, _ in self.cases]
        self.ws = [torch.zeros(max(16, wobs.wobs_workspace_size(wobs.OP_ARGCMP, m, n,
                                                                torch.empty(0, dtype=dt).element_size())),
                               dtype=torch.uint8, device=device) for _, m, n, dt, _ in self.cases]

    @classmethod
    def call_bytes(cls, i):
        _, m, n, dt, _ = cls.cases[i]
        return m * n * torch.empty(0, dtype=dt).element_size() + 8 * m

    @classmethod
    def bytes_per_step(cls):
        return sum(cls.call_bytes(i) for i in range(len(cls.cases)))

    def _call(self, c, i):
        f = self.wobs.wobs_argmin if self.cases[i][4] else self.wobs.wobs_argmax
        f(self.X[c][i], out=self.out[i], ws=self.ws[i])

    def step(self, c):
        for i in range(len(self.cases)):
            self._call(c, i)

    def kernel_calls(self):
        return [(self.cases[i][0], self.call_bytes(i), lambda c, i=i: self._call(c, i))
                for i in range(len(self.cases))]

    def e2e_setup(self):
        # the rows come from the host (pinned) and the indices go back each step
        self.xh = [x.cpu().pin_memory() for x in self.X[0]]
        self.oh = [torch.empty(o.shape, dtype=torch.int64).pin_memory() for o in self.out]
        return (sum(x.numel() * x.element_size() for x in self.xh),
                sum(o.numel() * 8 for o in self.oh))

    def e2e_step(self, c):
        for i in range(len(self.cases)):
            self.X[c][i].copy_(self.xh[i], non_blocking=True)
            self._call(c, i)
            self.oh[i].copy_(self.out[i], non_blocking=True)

    def config(self):
        return {"workload": self.name,
                "rows": [f"{name} [{m}, {n}] {str(dt).replace('torch.', '')} "
                         f"{'argmin' if mn else 'argmax'}" for name, m, n, dt, mn in self.cases],
                "row_copies": self.copies,
                "working_set_gb": round(self.copies * self.bytes_per_step() / 1e9, 3),
                "l2": "inputs larger than L2: rotated copies of the rows, working set above 1 GB"}

    @classmethod
    def oracle_prepare(cls, frac):
        from weight_only_bit_split_gb300 import synth
        prep = []
        for _, m, n, dt, mn in cls.cases:
            rows = max(1, int(round(m * frac))) if m > 1 else 1
            cols = n if m > 1 else max(1, int(round(n * frac)))
            x = synth.normal((rows, cols), 1.0, synth.seed_of(cls.workload_id, 2, 0), dtype=dt)
            prep.append((x.float().numpy(), mn, dt))
        return prep

    @classmethod
    def oracle_step(cls, prep):
        import oracle
        nbytes = 0
        for x, mn, dt in prep:
            (oracle.argmin_rows if mn else oracle.argmax_rows)(x)
            nbytes += x.size * torch.empty(0, dtype=dt).element_size() + 8 * x.shape[0]
        return nbytes


WORKLOADS = {"q4_m1": Q4M1Fused, "q4_m1_2call": Q4M1, "q4_m_sweep": Q4Sweep, "fp16_4096": DenseF16, "nf4": NF4,
             "nf4_m_sweep": NF4Sweep,
             "lm_head": LmHead, "argcmp": ArgCmp, "q8_m1": Q8M1Fused, "q8_m1_2call": Q8M1}
# oracle row fraction per step (bounds the CPU time of one oracle step)
ORACLE_FRACTION = {"q4_m1": 0.125, "q4_m1_2call": 0.125, "q4_m_sweep": 1 / 64, "fp16_4096": 0.5, "nf4": 1 / 32,
                   "nf4_m_sweep": 1 / 512,
                   "lm_head": 1 / 256, "argcmp": 1 / 4, "q8_m1": 1 / 16, "q8_m1_2call": 1 / 16}


def host_cpu():
    """(usable host threads, CPU model name) of this machine."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    return n, model or "unknown"


def oracle_rate(cls, frac, min_seconds, max_steps=None, threads=1):
    """Run the oracle on a row sample until ``min_seconds`` pass; GB/s, steps, seconds.

    With ``threads`` > 1 every host thread runs oracle steps on the same
    (read-only) sample concurrently; numpy releases the interpreter lock
    inside its array operations, so the threads use separate cores.
    """
    from concurrent.futures import ThreadPoolExecutor
    prep = cls.oracle_prepare(frac)
    t0 = time.perf_counter()

    def worker(_):
        nbytes, steps = 0, 0
        while True:
            nbytes += cls.oracle_step(prep)
            steps += 1
            el = time.perf_counter() - t0
            if el >= min_seconds or (max_steps is not None and steps >= max_steps):
                return nbytes, steps

    if threads <= 1:
        nbytes, steps = worker(0)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            res = list(ex.map(worker, range(threads)))
        nbytes, steps = sum(r[0] for r in res), sum(r[1] for r in res)
    el = time.perf_counter() - t0
    return nbytes / el / 1e9, steps, el, nbytes


# ------------------------------------------------------------------ main


def run_reference(args, cls, key, budget_s=90.0):
    """The CPU oracle as the reference arm: rank 0 only, on all host threads.

    A step is one oracle step per host thread, all on the same row sample of
    the workload, run concurrently (numpy releases the interpreter lock in
    its array operations).  The sample shrinks below the workload's default
    fraction when needed so that warm-up plus timed steps take about
    ``budget_s`` seconds.
    """
    from concurrent.futures import ThreadPoolExecutor
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    nthreads, cpu_model = host_cpu()
    frac = ORACLE_FRACTION[key]
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        def par_step(prep):
            return sum(ex.map(lambda _: cls.oracle_step(prep), range(nthreads)))

        t0 = time.perf_counter()
        par_step(cls.oracle_prepare(frac))
        per_step = time.perf_counter() - t0
        allowed = budget_s / max(1, args.steps + args.warmup)
        if per_step > allowed:
            frac *= allowed / per_step
        prep = cls.oracle_prepare(frac)
        for _ in range(args.warmup):
            par_step(prep)
        t0 = time.perf_counter()
        nbytes = 0
        for _ in range(args.steps):
            nbytes += par_step(prep)
        el = time.perf_counter() - t0
    gbs = nbytes / el / 1e9
    sample = (f"each step: {nthreads} host threads, each one oracle step on {frac:.4g} of each weight "
              f"matrix's rows, full K, same seeds and distributions (numpy fp64)")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cls.name, "oracle_row_fraction": frac},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="q4_m1", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="wobs", choices=["wobs", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--probe-gib", type=int, default=PROBE_BYTES >> 30,
                    help="size of the streaming-read ceiling buffer")
    ap.add_argument("--profile", action="store_true",
                    help="profiling case for ncu: build the workload, run --warmup + --steps "
                         "steps eagerly on the default stream, no probe, no timing")
    args = ap.parse_args(argv)
    if args.warmup < 3 and not args.profile:
        ap.error("--warmup must be at least 3")
    cls = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, cls, args.workload)

    import weight_only_bit_split_gb300 as wobs
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.profile:
        wl = cls(device)
        for i in range(args.warmup + args.steps):
            wl.step(i % wl.copies)
        torch.cuda.synchronize(device)
        print(f"profile case done: {cls.name}, {args.warmup + args.steps} steps, "
              f"{wl.launches_per_step} launches per step", flush=True)
        return 0
    init_dist("nccl")
    stream = torch.cuda.Stream(device)

    ceiling, ceil_cfg, ceil_table = read_ceiling(device, stream, args.probe_gib << 30)
    wl = cls(device)
    # eager pass first (kernel attributes, occupancy queries), then capture
    with torch.cuda.stream(stream):
        for c in range(wl.copies):
            wl.step(c)
    stream.synchronize()
    runner = StepRunner(wl, stream)
    runner.prepare(args.warmup)
    runner.prepare(args.steps)
    time_steps(runner, args.warmup, stream)

    # the timed region: exactly K steps, bracketed by a barrier and a device
    # synchronise; repeated so that it spans enough wall time for the clock
    # sampler (about 0.1 s), and the median region is reported
    clocks = ClockSampler(device)
    clocks.start()
    regions = []
    while True:
        barrier(device)
        torch.cuda.synchronize(device)
        regions.append(time_steps(runner, args.steps, stream))
        torch.cuda.synchronize(device)
        barrier(device)
        # every rank stops after the same region (its decision taken from the slowest)
        done = len(regions) >= 200 or (len(regions) >= 5 and sum(regions) >= 100.0)
        if reduce_over_ranks(1.0 if done else 0.0, "max", device) > 0:
            break
    clocks.stop()
    ms = statistics.median(regions)
    bytes_rank = wl.bytes_per_step() * args.steps
    gbs, ms_max = aggregate(bytes_rank, ms, device)

    # per-launch time of the dominant kernel: its launches alone, back to
    # back over the rotated copies, one graph per call site
    per_call = {}
    tot_b, tot_ms, launches = 0, 0.0, 0
    reps = max(3, min(20, 2000 // max(1, wl.copies)))
    for label, nbytes, fn in wl.kernel_calls():
        us, iqr, iso = time_call_site(wl, fn, stream, reps)
        per_call[label] = {"us": round(us, 3), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                           "iqr_us": round(iqr, 3), "isolated_us": round(iso, 3)}
        if hasattr(wl, "roofline_call") and not wl.roofline_call(label):
            continue                               # another kernel than the dominant one
        tot_b += nbytes
        tot_ms += us * 1e-3
        launches += 1
    achieved = tot_b / (tot_ms * 1e-3) / 1e9
    # other ways of computing the same product, timed the same way, outside
    # the roofline figure
    for label, nbytes, fn in (wl.extra_calls() if hasattr(wl, "extra_calls") else []):
        us, iqr, iso = time_call_site(wl, fn, stream, reps)
        per_call[label] = {"us": round(us, 3), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                           "iqr_us": round(iqr, 3), "isolated_us": round(iso, 3), "extra": True}
    peak, peak_kind = measured_peaks()
    traffic = traffic_record(cls.kernel if isinstance(cls.kernel, str) else None)

    # end to end through the public API with pinned host buffers: each
    # step's calls (H2D of the inputs, quantise/GEMV launches, D2H of the
    # outputs) captured once per weight copy in a StepGraph and replayed
    h2d, d2h = wl.e2e_setup()
    e2e_steps = max(3, min(args.steps, 200))
    step_graphs = [wobs.StepGraph(lambda c=c: wl.e2e_step(c), stream) for c in range(wl.copies)]
    with torch.cuda.stream(stream):
        for i in range(3):
            step_graphs[i % wl.copies].replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            step_graphs[i % wl.copies].replay()
        e1.record(stream)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_gbs = wl.bytes_per_step() / (e2e_ms * 1e-3) / 1e9
    e2e_gbs = reduce_over_ranks(e2e_gbs, "sum", device) if world > 1 else e2e_gbs

    # the same graphs with the launches left out: what the step's two pinned
    # copies cost on their own (latency of a host<->device round trip, not
    # bandwidth: the step moves a few hundred KB)
    shadow = [n for n in ("step", "_call") if hasattr(wl, n)]
    for n in shadow:
        setattr(wl, n, lambda *a, **k: None)
    try:
        copy_graphs = [wobs.StepGraph(lambda c=c: wl.e2e_step(c), stream) for c in range(min(4, wl.copies))]
        with torch.cuda.stream(stream):
            for i in range(3):
                copy_graphs[i % len(copy_graphs)].replay()
            stream.synchronize()
            e0.record(stream)
            for i in range(e2e_steps):
                copy_graphs[i % len(copy_graphs)].replay()
            e1.record(stream)
        e1.synchronize()
        copies_ms = e0.elapsed_time(e1) / e2e_steps
    finally:
        for n in shadow:
            delattr(wl, n)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        frac = ORACLE_FRACTION[args.workload]
        nthreads, cpu_model = host_cpu()
        v1, steps1, el1, _ = oracle_rate(cls, frac, 6.0, max_steps=200)
        vn, stepsn, eln, _ = oracle_rate(cls, frac, 8.0, threads=nthreads)
        cpu = {"value": vn, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
               "sample": f"{stepsn} oracle steps over {nthreads} host threads, each on {frac:.4g} of "
                         f"each weight matrix's rows (full K, same seeds), {eln:.1f} s, numpy fp64",
               "one_core": {"value": v1, "unit": "GB/s", "cores": 1,
                            "sample": f"{steps1} oracle steps, one thread, {el1:.1f} s"},
               "nproc": nthreads, "cpu_model": cpu_model}

    if rank == 0:
        line = {
            "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cls.dtype, "data": "synthetic",
            "config": wl.config(),
            "mbu": gbs / world / ceiling,
            "read_ceiling_gbs": round(ceiling, 1),
            "read_ceiling_how": f"bw_probe best of variants 1-3 x grids 1-8 CTAs/SM on an "
                                f"{args.probe_gib} GiB buffer: {ceil_cfg}",
            "read_ceiling_table": ceil_table,
            "us_per_call": per_call,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": cls.kernel, "peak_source": f"{peak_kind} hbm_gbs",
                         "per_launch": "algorithmic bytes per launch / CUDA-event time of the "
                                       "kernel's launches replayed back to back"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "us_per_step": round(e2e_ms * 1e3, 3),
                    "copies_only_us_per_step": round(copies_ms * 1e3, 3),
                    "how": "public Python API calls of one step captured once per weight copy "
                           "in a wobs.StepGraph and replayed every step: pinned H2D of the "
                           "activations, the step's launches, D2H of the outputs; "
                           "copies_only: the same graphs without the launches"},
            "gpu_launches": wl.launches_per_step * args.steps,
            "timed_regions": {"count": len(regions), "ms_min": round(min(regions), 5),
                              "ms_median": round(ms, 5), "ms_max": round(max(regions), 5),
                              "how": "each region: exactly --steps steps between a barrier and "
                                     "a device synchronise; value and ms_per_step use the median "
                                     "region"},
            "clocks": clocks.report(),
        }
        print(json.dumps(line), flush=True)
    if _dist_on():
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
