"""Benchmark of the block-quantized wire codec on GB300.

One step is one pass of the whole codec path over the prefill-scale workload:

    4 x BF16 [65536, 7168]  --quant_i8-->  4 INT8 wires
    4 wires                 --dequant_accum_i8 (W=4, FP32, source order)-->  1 wire
    that wire               --dequant_i8-->  BF16 [65536, 7168]
    wire 0 + BF16 buffer 1  --ring_hop_i8-->  1 wire
    6 x BF16 [4096, 7168]   --quant_mx (staged slices)-->  MXFP8 [4096, 43008]
    MXFP8 [4096, 43008]     --dequant_mx-->  BF16 [4096, 43008]

(14 kernel launches). ``value`` is the step's algorithmic bytes (every input byte
read once, every output byte written once) divided by the device time of the step,
summed over ranks; it is timed over K steps with nothing between the launches. The
per-kernel figures (``kernels``, ``roofline``) come from a second timed region of K
steps with a CUDA event after every launch. The step's working set (about 12.5 GB) is far larger than the
129 MB L2, so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bq|reference]

Under torchrun every rank runs its own replica of the workload on its own GPU (the
path shards into independent blocks; there is no exchange step), with a barrier and
the maximum over ranks of the timed region. ``--impl reference`` times the CPU oracle
on a bounded sample of the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "codec HBM GB/s (and % of ~8 TB/s peak) per kernel at 1 GB300; bit-exact vs oracle"
UNIT = "GB/s"
HIDDEN = 7168
W_SRC = 4
N_SLICES = 6
BF16 = 2
RAW_SAMPLES = 200  # raw timing samples kept per series in the JSON line


def wire_per_value() -> float:
    return 132.0 / 128.0


def kernel_bytes(name: str, n: int) -> int:
    """Algorithmic bytes of one launch over n values (inputs read once, outputs written once)."""
    w = wire_per_value()
    per = {
        "quant_i8": BF16 + w,
        "dequant_i8": w + BF16,
        "dequant_accum_i8": W_SRC * w + w,
        "ring_hop_i8": w + BF16 + w,
        "quant_mx": BF16 + w,
        "dequant_mx": w + BF16,
        "dequant_accum_mx": W_SRC * w + w,
        "ring_hop_mx": w + BF16 + w,
        "reduce_quant_i8": W_SRC * BF16 + w,
        "reduce_quant_e4m3": W_SRC * BF16 + w,
        "quant_e4m3": BF16 + w,
        "dequant_e4m3": w + BF16,
        "quant_mx_f16": BF16 + w,
        "quant_mx_slices": BF16 + w,
        "quant_mx_tiled": BF16 + w,
        "quant_mx_tiled_f16": BF16 + w,
    }[name]
    return int(round(per * n))


# ---------------------------------------------------------------- distributed plumbing
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (timing aggregation only; not part of the data path)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- measurement helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary (profiles/ncu_traffic.txt):
    lines 'kernel source_sha256 workload_values dram_bytes_per_launch_at_full_size'."""
    out = {}
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return out
    for line in open(path):
        line = line.split("#", 1)[0].split()
        if len(line) >= 3:
            out[line[0]] = (line[1], float(line[2]))
    return out


def kernel_sources_sha() -> str:
    """Hash of the kernel sources' code: every file of csrc with comments removed and
    whitespace collapsed, so that a comment edit does not invalidate the recorded ncu
    counters while any code change does."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_wire_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = " ".join(text.split())
        h.update(f.encode() + b"\0" + text.encode())
    return h.hexdigest()[:16]


class NvmlClocks:
    """SM clock, its maximum, power and throttle reasons read in-process through NVML
    (ctypes on libnvidia-ml; read-only queries). A thread samples every `period_s`
    between mark_start() and mark_stop(), and both marks take a sample themselves, so
    even a 40 ms timed region has a dozen or more samples of its own."""

    # nvmlClocksEventReasons bits
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, device: torch.device, period_s: float = 0.002):
        import ctypes
        self.ok = False
        self.samples = []
        self.period = period_s
        self._run = False
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device)
            uuid = str(getattr(props, "uuid", ""))
            bus = "%04x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), getattr(props, "pci_bus_id", 0),
                                        getattr(props, "pci_device_id", 0))
            found = False
            if uuid:
                u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                found = nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
            for b in ([] if found else [bus, "0000" + bus]):
                found = found or nv.nvmlDeviceGetHandleByPciBusId_v2(b.encode(), ctypes.byref(h)) == 0
            if not found:
                return
            self.nv, self.h, self.ct = nv, h, ctypes
            try:
                self.reasons_fn = nv.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                self.reasons_fn = nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:  # NVML_CLOCK_SM
                return
            self.max_mhz = float(mx.value)
            self.ok = self._sample() is not None
        except (OSError, AttributeError, RuntimeError):
            self.ok = False

    def _sample(self):
        ct, nv, h = self.ct, self.nv, self.h
        sm, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(sm)) != 0:
            return None
        p = float(pw.value) / 1000.0 if nv.nvmlDeviceGetPowerUsage(h, ct.byref(pw)) == 0 else None
        r = int(rs.value) if self.reasons_fn(h, ct.byref(rs)) == 0 else 0
        s = (float(sm.value), p, r)
        self.samples.append(s)
        return s

    def _loop(self):
        while self._run:
            self._sample()
            time.sleep(self.period)

    def mark_start(self):
        if not self.ok:
            return
        self.samples = []
        self._sample()
        self._run = True
        self._t = threading.Thread(target=self._loop, daemon=True)
        self._t.start()

    def mark_stop(self):
        if not self.ok:
            return
        self._run = False
        self._t.join(timeout=2)
        self._sample()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        sms = [s[0] for s in self.samples]
        pw = [s[1] for s in self.samples if s[1] is not None]
        reasons = sorted({nm for s in self.samples for bit, nm in self.REASONS.items() if s[2] & bit})
        return {"sm_mhz": statistics.median(sms), "sm_mhz_min": min(sms), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sms), "power_w_max": max(pw) if pw else None,
                "source": f"NVML in-process every {self.period * 1e3:.0f} ms plus one read at each end of the region"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms; only samples taken
    between mark_start() and mark_stop() (the timed region) are summarized. The fallback
    when NVML cannot be read in-process."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.5)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark_start(self):
        import datetime
        self.t0 = datetime.datetime.now()

    def mark_stop(self):
        import datetime
        self.t1 = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        import datetime
        sms, maxs, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            if self.t0 is not None and not (self.t0 <= ts <= self.t1):
                continue
            sms.append(sm)
            maxs.append(mx)
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- the workload
class Pipeline:
    """Device buffers and launch list of one codec step (caller-owned memory)."""

    def __init__(self, rows: int, slice_rows: int, device, generate: bool = True):
        from block_quantized_wire_gb300 import codec, inputs
        self.codec = codec
        self.device = device
        self.rows, self.slice_rows = rows, slice_rows
        self.n = rows * HIDDEN
        self.n_slice = slice_rows * HIDDEN
        if generate:
            self.xs = [inputs.prefill_buffer(w, device=device, rows=rows) for w in range(W_SRC)]
            self.slices = inputs.mx_slices_4096(device=device, rows=slice_rows)
        else:  # buffers only; the inputs arrive by copy
            self.xs = [torch.empty((rows, HIDDEN), dtype=torch.bfloat16, device=device) for _ in range(W_SRC)]
            self.slices = [torch.empty((slice_rows, HIDDEN), dtype=torch.bfloat16, device=device)
                           for _ in range(N_SLICES)]
        self.wires = [codec.empty_wire_i8(self.n, device) for _ in range(W_SRC)]
        self.acc = codec.empty_wire_i8(self.n, device)
        self.hop = codec.empty_wire_i8(self.n, device)
        self.out = torch.empty((rows, HIDDEN), dtype=torch.bfloat16, device=device)
        C = HIDDEN * N_SLICES
        self.mx_q, self.mx_s = codec.empty_mx(slice_rows, C, device)
        self.mx_out = torch.empty((slice_rows, C), dtype=torch.bfloat16, device=device)
        self.launches = self._launch_list()

    def _launch_list(self):
        c = self.codec
        L = []
        for w in range(W_SRC):
            L.append(("quant_i8", (lambda w=w: c.quant_i8(self.xs[w].view(-1), self.wires[w][1], self.wires[w][2])),
                      kernel_bytes("quant_i8", self.n)))
        L.append(("dequant_accum_i8", lambda: c.dequant_accum_i8(
            [w[1] for w in self.wires], [w[2] for w in self.wires], self.acc[1], self.acc[2], None),
            kernel_bytes("dequant_accum_i8", self.n)))
        L.append(("dequant_i8", lambda: c.dequant_i8(self.acc[1], self.acc[2], self.out.view(-1)),
                  kernel_bytes("dequant_i8", self.n)))
        L.append(("ring_hop_i8", lambda: c.ring_hop_i8(self.wires[0][1], self.wires[0][2], self.xs[1].view(-1),
                                                       self.hop[1], self.hop[2], None),
                  kernel_bytes("ring_hop_i8", self.n)))
        for i in range(N_SLICES):
            c0 = i * HIDDEN
            L.append(("quant_mx", (lambda i=i, c0=c0: c.quant_mx(
                self.slices[i], self.mx_q[:, c0:c0 + HIDDEN], self.mx_s[:, c0 // 32:(c0 + HIDDEN) // 32])),
                kernel_bytes("quant_mx", self.n_slice)))
        L.append(("dequant_mx", lambda: c.dequant_mx(self.mx_q, self.mx_s, self.mx_out),
                  kernel_bytes("dequant_mx", self.n_slice * N_SLICES)))
        return L

    def step_bytes(self) -> int:
        return sum(b for _, _, b in self.launches)

    def run(self, events=None):
        for i, (_, fn, _) in enumerate(self.launches):
            fn()
            if events is not None:
                events[i].record()

    def results(self):
        return [self.acc[0], self.out, self.hop[0], self.mx_q, self.mx_s, self.mx_out]


class EndToEnd:
    """The step through the public API from host memory: every step copies its inputs
    from pinned host buffers to the device and its results back to pinned host buffers.
    Two device buffer sets alternate between consecutive steps. The copies of both
    directions run in order on one copy stream (step k+1's inputs, then step k's
    results) and the codec launches on a second stream, so a step's computation hides
    behind the copies of its neighbours. Running the two copy directions at once was
    slower on GB300's shared host link than running them back to back. Events order
    the reuse of each buffer set: its inputs are overwritten only after the step that
    read them has computed, and its results only after they have been copied out."""

    def __init__(self, pipe: Pipeline):
        self.sets = [pipe, Pipeline(pipe.rows, pipe.slice_rows, pipe.device, generate=False)]
        pin = dict(pin_memory=True)
        self.h_xs = [torch.empty_like(x, device="cpu", **pin).copy_(x) for x in pipe.xs]
        self.h_slices = [torch.empty_like(x, device="cpu", **pin).copy_(x) for x in pipe.slices]
        self.h_results = [torch.empty_like(t, device="cpu", **pin) for t in pipe.results()]
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_xs + self.h_slices)
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_results)
        self.s_copy, self.s_comp = torch.cuda.Stream(), torch.cuda.Stream()
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.comp_done = [torch.cuda.Event() for _ in range(2)]

    def _copy_in(self, k: int):
        i = k % 2
        p = self.sets[i]
        with torch.cuda.stream(self.s_copy):
            if k >= 2:
                self.s_copy.wait_event(self.comp_done[i])  # step k-2 has read this set's inputs
            for d, h in zip(p.xs, self.h_xs):
                d.copy_(h, non_blocking=True)
            for d, h in zip(p.slices, self.h_slices):
                d.copy_(h, non_blocking=True)
            self.in_ready[i].record(self.s_copy)

    def _compute(self, k: int):
        i = k % 2
        with torch.cuda.stream(self.s_comp):
            # inputs are in; step k-2's results were copied out earlier on the copy
            # stream, before this step's inputs, so in_ready covers both
            self.s_comp.wait_event(self.in_ready[i])
            self.sets[i].run()
            self.comp_done[i].record(self.s_comp)

    def _copy_out(self, k: int):
        i = k % 2
        with torch.cuda.stream(self.s_copy):
            self.s_copy.wait_event(self.comp_done[i])
            for h, d in zip(self.h_results, self.sets[i].results()):
                h.copy_(d, non_blocking=True)

    def run(self, nsteps: int):
        cur = torch.cuda.current_stream()
        for st in (self.s_copy, self.s_comp):
            st.wait_stream(cur)
        # copy stream order: in(0), in(1), out(0), in(2), out(1), ..., out(n-1)
        for k in range(nsteps):
            self._copy_in(k)
            self._compute(k)
            if k >= 1:
                self._copy_out(k - 1)
        self._copy_out(nsteps - 1)
        for st in (self.s_copy, self.s_comp):
            cur.wait_stream(st)


# ---------------------------------------------------------------- CPU oracle leg
def oracle_step(xb, sb):
    """One step's operations by the oracle: xb the W INT8-path buffers and sb the MX
    slices, as BF16 bit arrays [rows, HIDDEN]. Returns the step's algorithmic bytes."""
    import numpy as np

    import oracle
    n, ns = xb[0].size, sb[0].size if sb else 0
    nbytes = 0
    if n:
        flat = [b.reshape(-1) for b in xb]
        qs = [oracle.quant_i8(b) for b in flat]
        qa, sa, _ = oracle.dequant_accum_i8([q for q, _ in qs], [s for _, s in qs], materialize=False)
        oracle.dequant_i8(qa, sa)
        oracle.ring_hop_i8(qs[0][0], qs[0][1], flat[1])
        nbytes += (W_SRC * kernel_bytes("quant_i8", n) + kernel_bytes("dequant_accum_i8", n) +
                   kernel_bytes("dequant_i8", n) + kernel_bytes("ring_hop_i8", n))
    if ns:
        C = HIDDEN * N_SLICES
        r = sb[0].shape[0]
        qb = np.empty((r, C), np.uint8)
        sbuf = np.empty((r, C // 32), np.uint8)
        for i, s in enumerate(sb):
            oracle.quant_mx_into(s, qb, sbuf, i * HIDDEN)
        oracle.dequant_mx(qb, sbuf)
        nbytes += N_SLICES * kernel_bytes("quant_mx", ns) + kernel_bytes("dequant_mx", ns * N_SLICES)
    return nbytes


def oracle_sample(pipe_inputs, rows: int, slice_rows: int, threads: int = 1):
    """Run the oracle over the first `rows` rows of every prefill buffer and the first
    `slice_rows` rows of every MX slice, in the step's order. With threads > 1 the rows
    are cut into `threads` contiguous ranges and each host thread runs the whole step
    on its range (blocks are independent, so the outputs are those of one call).
    Returns (wall seconds, bytes)."""
    from block_quantized_wire_gb300.inputs import bf16_bits
    from oracle import shards
    xs, slices = pipe_inputs
    xb = [bf16_bits(x[:rows]).reshape(rows, HIDDEN) for x in xs]
    sb = [bf16_bits(s[:slice_rows]).reshape(slice_rows, HIDDEN) for s in slices]
    ir, mr = shards.row_ranges(rows, threads), shards.row_ranges(slice_rows, threads)

    def work(p):
        lo, hi = ir[p] if p < len(ir) else (0, 0)
        ml, mh = mr[p] if p < len(mr) else (0, 0)
        return oracle_step([b[lo:hi] for b in xb], [s[ml:mh] for s in sb] if mh > ml else [])

    t0 = time.perf_counter()
    nbytes = sum(shards.run_indexed(work, max(len(ir), len(mr))))
    return time.perf_counter() - t0, nbytes


def oracle_next_rows(pipe_inputs, rows: int) -> dict:
    """The oracle on each of the next rows' operations, single-threaded, on the first `rows`
    rows of the prefill buffers (W = 4 sources where the row has sources) and of the
    first MX slice: GB/s of the algorithmic bytes the GPU rows count. Inputs the
    operation consumes (wires, FP16 copies) are prepared outside its timed call."""
    import numpy as np

    import oracle
    from block_quantized_wire_gb300.inputs import bf16_bits
    xs, slices = pipe_inputs
    xb = [bf16_bits(x[:rows]).reshape(-1) for x in xs]
    n = xb[0].size
    sl_t = slices[0][:rows]
    sl = bf16_bits(sl_t).reshape(rows, HIDDEN)
    sl16 = sl_t.to(torch.float16).contiguous().view(torch.int16).numpy().view(np.uint16).reshape(rows, HIDDEN)
    mx = [oracle.quant_mx_flat(b) for b in xb]
    e4 = oracle.quant_e4m3(xb[0])
    out = {}

    def timed(name, fn, values):
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        out[name] = {"GB/s": round(kernel_bytes(name, values) / dt / 1e9, 4), "seconds": round(dt, 3)}

    timed("quant_mx_slices", lambda: oracle.quant_mx(sl), rows * HIDDEN)
    timed("quant_mx_tiled", lambda: oracle.mx_scales_to_tiled(oracle.quant_mx(sl)[1]), rows * HIDDEN)
    timed("quant_mx_f16", lambda: oracle.quant_mx(sl16, fmt="f16"), rows * HIDDEN)
    timed("dequant_accum_mx", lambda: oracle.dequant_accum_mx([q for q, _ in mx], [s for _, s in mx],
                                                               materialize=False), n)
    timed("ring_hop_mx", lambda: oracle.ring_hop_mx(mx[0][0], mx[0][1], xb[1]), n)
    timed("reduce_quant_i8", lambda: oracle.reduce_quant_i8(xb), n)
    timed("reduce_quant_e4m3", lambda: oracle.reduce_quant_e4m3(xb), n)
    timed("quant_e4m3", lambda: oracle.quant_e4m3(xb[0]), n)
    timed("dequant_e4m3", lambda: oracle.dequant_e4m3(*e4), n)
    return {"rows": rows, "cores": 1, "kind": "oracle", "ops": out}


def oracle_parity(pipe, rows: int, slice_rows: int) -> dict:
    """Part of the CPU-oracle leg: the step's GPU outputs on the first `rows` rows of every
    INT8 buffer and `slice_rows` rows of every MX slice, compared byte for byte with the
    oracle's outputs for the same input bits (blocks and groups are independent, so the
    first rows of an output depend only on the first rows of its inputs)."""
    import numpy as np

    import oracle
    from block_quantized_wire_gb300.inputs import bf16_bits

    def same(dev, want):
        got = dev.detach().contiguous().cpu()
        got = got.view(torch.int16) if got.dtype == torch.bfloat16 else got
        return bool(np.array_equal(got.numpy().reshape(-1).view(np.uint8), np.asarray(want).reshape(-1).view(np.uint8)))

    pipe.run()  # the later sections reuse the step's output buffers: one more step restores them
    torch.cuda.synchronize()
    n = rows * HIDDEN
    xb = [bf16_bits(x[:rows]).reshape(-1) for x in pipe.xs]
    qs = [oracle.quant_i8(b) for b in xb]
    qa, sa, _ = oracle.dequant_accum_i8([q for q, _ in qs], [s for _, s in qs], materialize=False)
    qh, sh, _ = oracle.ring_hop_i8(qs[0][0], qs[0][1], xb[1])
    ok = {"quant_i8": all(same(pipe.wires[w][1][:n], qs[w][0]) and same(pipe.wires[w][2][:n // 128], qs[w][1])
                          for w in range(W_SRC)),
          "dequant_accum_i8": same(pipe.acc[1][:n], qa) and same(pipe.acc[2][:n // 128], sa),
          "dequant_i8": same(pipe.out.view(-1)[:n], oracle.dequant_i8(qa, sa)),
          "ring_hop_i8": same(pipe.hop[1][:n], qh) and same(pipe.hop[2][:n // 128], sh)}
    C = HIDDEN * N_SLICES
    qb = np.empty((slice_rows, C), np.uint8)
    sbuf = np.empty((slice_rows, C // 32), np.uint8)
    for i, s in enumerate(pipe.slices):
        oracle.quant_mx_into(bf16_bits(s[:slice_rows]).reshape(slice_rows, HIDDEN), qb, sbuf, i * HIDDEN)
    ok["quant_mx"] = same(pipe.mx_q[:slice_rows], qb) and same(pipe.mx_s[:slice_rows], sbuf)
    ok["dequant_mx"] = same(pipe.mx_out[:slice_rows], oracle.dequant_mx(qb, sbuf))
    return {"rows": rows, "slice_rows": slice_rows, "bitexact": all(ok.values()), "per_kernel": ok}


def run_env(dev) -> dict:
    """Where the numbers were taken: device, its UUID and SM count, driver, CUDA
    runtime, torch, the hash of the kernel sources, and the GPU's compute and
    persistence modes (read-only NVML queries)."""
    props = torch.cuda.get_device_properties(dev)
    env = {"device": torch.cuda.get_device_name(dev), "uuid": str(getattr(props, "uuid", "")),
           "sm_count": props.multi_processor_count, "cuda_runtime": torch.version.cuda, "torch": torch.__version__,
           "kernel_sources_sha": kernel_sources_sha(), "driver": None}
    try:
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        buf = ctypes.create_string_buffer(96)
        if nv.nvmlInit_v2() == 0 and nv.nvmlSystemGetDriverVersion(buf, 96) == 0:
            env["driver"] = buf.value.decode()
        h, mode = ctypes.c_void_p(), ctypes.c_int()
        uuid = env["uuid"] if env["uuid"].startswith("GPU-") else "GPU-" + env["uuid"]
        if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0:
            names = {0: "default", 2: "exclusive_process", 3: "prohibited"}
            if nv.nvmlDeviceGetComputeMode(h, ctypes.byref(mode)) == 0:
                env["compute_mode"] = names.get(mode.value, str(mode.value))
            if nv.nvmlDeviceGetPersistenceMode(h, ctypes.byref(mode)) == 0:
                env["persistence_mode"] = bool(mode.value)
    except (OSError, AttributeError):
        pass
    return env


def cpu_inputs(rows: int, slice_rows: int):
    """Workload inputs for the CPU oracle leg: the first rows of the GPU-drawn buffers
    when a GPU exists (the very bits the GPU path consumes), else CPU draws."""
    from block_quantized_wire_gb300 import inputs
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    xs = [inputs.prefill_buffer(w, device=dev, rows=rows) for w in range(W_SRC)]
    sl = inputs.mx_slices_4096(device=dev, rows=slice_rows)
    return [x.cpu() for x in xs], [s.cpu() for s in sl]


# ---------------------------------------------------------------- widened rows
GRAPH_REPLAYS = 5


def graph_stats(fn, reps: int, replays: int = GRAPH_REPLAYS):
    """Device time of one call of fn: `reps` calls captured into one CUDA graph (after 3
    eager warm-ups), the graph replayed `replays` times with CUDA events around each
    replay, so the host's launch overhead is not in the number (short launches would
    otherwise wait for the host). Returns the median per-call time (ms) and the
    per-replay samples."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    samples = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        samples.append(e0.elapsed_time(e1) / reps)
    del g
    return statistics.median(samples), samples


def graph_ms(fn, reps: int) -> float:
    return graph_stats(fn, reps)[0]


def spread(samples) -> dict:
    """Median, min, max (us) and the raw per-replay samples of graph_stats."""
    return {"replays": len(samples), "median_us": round(statistics.median(samples) * 1e3, 2),
            "min_us": round(min(samples) * 1e3, 2), "max_us": round(max(samples) * 1e3, 2),
            "samples_us": [round(t * 1e3, 2) for t in samples]}


def time_next_rows(pipe, args, peak):
    """Per-launch duration of the kernels beyond the step, on the prefill buffers:
    dequant_accum_mx (W=4) and ring_hop_mx on flat MX wires quantized from them,
    reduce_quant_i8 / reduce_quant_e4m3 (W=4: the all-gather modes' fused reduce),
    quant_e4m3 / dequant_e4m3 (legacy codec), and quant_mx on FP16 slices of the staged
    workload (rotating over six slices). Each kernel: `next_reps` back-to-back launches
    replayed as one CUDA graph (graph_ms); every launch (or, for the slices, every six
    consecutive launches) moves more than the 129 MB L2 holds."""
    from block_quantized_wire_gb300 import inputs
    c = pipe.codec
    n = pipe.n
    dev = pipe.xs[0].device
    xs = [x.view(-1) for x in pipe.xs]
    wires = [c.empty_wire_mx(n, dev) for _ in range(W_SRC + 2)]
    for w in range(W_SRC):
        c.quant_mx_flat(xs[w], wires[w][1], wires[w][2])
    acc, hop = wires[W_SRC], wires[W_SRC + 1]
    ew = c.empty_wire_e4m3(n, dev)
    iw = c.empty_wire_i8(n, dev)
    c.quant_e4m3(xs[0], ew[1], ew[2])
    f16 = inputs.mx_slices_4096(device=dev, rows=pipe.slice_rows, dtype=torch.float16)
    ns = f16[0].numel()
    turn = [0]

    def quant_f16():
        i = turn[0] % len(f16)
        turn[0] += 1
        c0 = i * HIDDEN
        c.quant_mx(f16[i], pipe.mx_q[:, c0:c0 + HIDDEN], pipe.mx_s[:, c0 // 32:(c0 + HIDDEN) // 32])

    g_total = N_SLICES * HIDDEN // 32
    tiled = torch.zeros((c.mx_tiled_scale_bytes(pipe.slice_rows, g_total),), dtype=torch.uint8, device=dev)

    def quant_tiled(xs_, turn_):
        i = turn_[0] % len(xs_)
        turn_[0] += 1
        c0 = i * HIDDEN
        c.quant_mx_tiled(xs_[i], pipe.mx_q[:, c0:c0 + HIDDEN], tiled, g_total, c0 // 32)

    turn_t, turn_t16 = [0], [0]
    runs = {
        "quant_mx_slices": (lambda: c.quant_mx_slices(pipe.slices, pipe.mx_q, pipe.mx_s), ns * N_SLICES),
        "quant_mx_tiled": (lambda: quant_tiled(pipe.slices, turn_t), ns),
        "quant_mx_tiled_f16": (lambda: quant_tiled(f16, turn_t16), ns),
        "dequant_accum_mx": (lambda: c.dequant_accum_mx([wires[w][1] for w in range(W_SRC)],
                                                        [wires[w][2] for w in range(W_SRC)], acc[1], acc[2], None), n),
        "ring_hop_mx": (lambda: c.ring_hop_mx(wires[0][1], wires[0][2], xs[1], hop[1], hop[2], None), n),
        "reduce_quant_i8": (lambda: c.reduce_quant_i8(xs, iw[1], iw[2], None), n),
        "reduce_quant_e4m3": (lambda: c.reduce_quant_e4m3(xs, ew[1], ew[2], None), n),
        "quant_e4m3": (lambda: c.quant_e4m3(xs[2], ew[1], ew[2]), n),
        "dequant_e4m3": (lambda: c.dequant_e4m3(ew[1], ew[2], pipe.out.view(-1)), n),
        "quant_mx_f16": (quant_f16, ns),
    }
    out = {}
    for name, (fn, nv) in runs.items():
        avg_ms, samples = graph_stats(fn, args.next_reps)
        nbytes = kernel_bytes(name, nv)
        gbs = nbytes / (avg_ms * 1e-3) / 1e9
        out[name] = {"launches": args.next_reps, "avg_us": round(avg_ms * 1e3, 2), "bytes_per_launch": nbytes,
                     "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4), **spread(samples)}
    out["quant_mx_slices"]["what"] = ("the six staged slices of the step quantized by one bq_quant_mx_slices "
                                      "call (one launch) instead of six bq_quant_mx calls")
    del wires, ew, iw, f16, tiled
    return out


# ---------------------------------------------------------------- the smaller configs
def time_configs(args, peak):
    """Per-kernel launch duration on the four smaller workloads (512, 3072, 3072 x W=4
    and 16384 x W=4 rows of 7168), inputs drawn on the device with the workloads' seeds
    and structure, each kernel timed as `next_reps` launches replayed from one CUDA
    graph (graph_ms). A launch whose bytes fit in the 129 MB L2 is labelled L2-warm:
    repeated launches read it from L2."""
    from block_quantized_wire_gb300 import codec, inputs
    dev = torch.device("cuda", torch.cuda.current_device())
    L2 = 129 * 10 ** 6
    out = {}

    def timed(fn, name, n, cfg):
        ms, samples = graph_stats(fn, args.next_reps)
        nbytes = kernel_bytes(name, n) if name in ("quant_i8", "dequant_i8", "quant_mx", "dequant_mx",
                                                   "dequant_accum_i8", "ring_hop_i8") else None
        if name == "dequant_accum_i8+bf16":
            nbytes = kernel_bytes("dequant_accum_i8", n) + 2 * n
        gbs = nbytes / (ms * 1e-3) / 1e9
        out.setdefault(cfg, {})[name] = {"avg_us": round(ms * 1e3, 2), "bytes_per_launch": nbytes,
                                         "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                                         "l2": "warm" if nbytes < L2 else "cold", **spread(samples)}

    x1 = inputs.roundtrip_512(device=dev)
    _, q1, s1 = codec.empty_wire_i8(x1.numel(), dev)
    o1 = torch.empty_like(x1)
    timed(lambda: codec.quant_i8(x1.view(-1), q1, s1), "quant_i8", x1.numel(), "roundtrip_512")
    timed(lambda: codec.dequant_i8(q1, s1, o1.view(-1)), "dequant_i8", x1.numel(), "roundtrip_512")
    x2 = inputs.mixed_3072(device=dev)
    n2 = x2.numel()
    _, q2, s2 = codec.empty_wire_i8(n2, dev)
    o2 = torch.empty_like(x2)
    mq, ms_ = codec.empty_mx(*x2.shape, dev)
    timed(lambda: codec.quant_i8(x2.view(-1), q2, s2), "quant_i8", n2, "mixed_3072")
    timed(lambda: codec.dequant_i8(q2, s2, o2.view(-1)), "dequant_i8", n2, "mixed_3072")
    timed(lambda: codec.quant_mx(x2, mq, ms_), "quant_mx", n2, "mixed_3072")
    timed(lambda: codec.dequant_mx(mq, ms_, o2), "dequant_mx", n2, "mixed_3072")
    xs3 = inputs.a2a_3072(device=dev)
    w3 = [codec.empty_wire_i8(n2, dev) for _ in range(W_SRC + 1)]
    for w in range(W_SRC):
        codec.quant_i8(xs3[w].view(-1), w3[w][1], w3[w][2])
    src_q, src_s = [w3[w][1] for w in range(W_SRC)], [w3[w][2] for w in range(W_SRC)]
    timed(lambda: codec.dequant_accum_i8(src_q, src_s, w3[W_SRC][1], w3[W_SRC][2], None), "dequant_accum_i8", n2,
          "a2a_3072")
    timed(lambda: codec.dequant_accum_i8(src_q, src_s, w3[W_SRC][1], w3[W_SRC][2], o2.view(-1)),
          "dequant_accum_i8+bf16", n2, "a2a_3072")
    del xs3, w3
    xs4 = inputs.ring_16384(device=dev)
    n4 = xs4[0].numel()
    w4 = [codec.empty_wire_i8(n4, dev) for _ in range(2)]
    codec.quant_i8(xs4[0].view(-1), w4[0][1], w4[0][2])
    timed(lambda: codec.ring_hop_i8(w4[0][1], w4[0][2], xs4[1].view(-1), w4[1][1], w4[1][2], None), "ring_hop_i8",
          n4, "ring_16384 (one hop step over the 4 shards)")
    del xs4, w4
    return out


# ---------------------------------------------------------------- one kernel alone (profiling)
PROFILE_OPS = ("quant_i8", "dequant_i8", "dequant_accum_i8", "ring_hop_i8", "quant_mx", "dequant_mx",
               "quant_mx_slices", "quant_mx_f16", "quant_mx_tiled", "dequant_accum_mx", "ring_hop_mx",
               "reduce_quant_i8", "reduce_quant_e4m3", "quant_e4m3", "dequant_e4m3")


def run_profile_op(args):
    """Launch one kernel of the workload `--profile-launches` times after `--warmup`
    launches, holding only that kernel's buffers (the prefill buffers at --rows, or the
    staged slices at --slice-rows), so that a profiler can capture one launch of a full-size
    kernel with a few GB on the device. Prints one line with the launch count; the
    timings of a run under a profiler are not benchmark values."""
    from block_quantized_wire_gb300 import build as bq_build, codec, inputs
    bq_build.build_library()
    dev = torch.device("cuda", 0)
    op, rows = args.profile_op, args.rows
    n = rows * HIDDEN
    if op in ("quant_mx", "quant_mx_slices", "dequant_mx", "quant_mx_f16", "quant_mx_tiled"):
        dt = torch.float16 if op == "quant_mx_f16" else torch.bfloat16
        sl = inputs.mx_slices_4096(device=dev, rows=args.slice_rows, dtype=dt)
        q, s = codec.empty_mx(args.slice_rows, HIDDEN * N_SLICES, dev)
        g_total = HIDDEN * N_SLICES // 32
        tiled = torch.zeros((codec.mx_tiled_scale_bytes(args.slice_rows, g_total),), dtype=torch.uint8, device=dev)
        turn = [0]

        def one_slice():
            i = turn[0] % N_SLICES
            turn[0] += 1
            c0 = i * HIDDEN
            if op == "quant_mx_tiled":
                codec.quant_mx_tiled(sl[i], q[:, c0:c0 + HIDDEN], tiled, g_total, c0 // 32)
            else:
                codec.quant_mx(sl[i], q[:, c0:c0 + HIDDEN], s[:, c0 // 32:(c0 + HIDDEN) // 32])
        if op == "dequant_mx":
            codec.quant_mx_slices(sl, q, s)  # the materialization's input
            del sl
            out = torch.empty((args.slice_rows, HIDDEN * N_SLICES), dtype=torch.bfloat16, device=dev)
            fn = lambda: codec.dequant_mx(q, s, out)
        else:
            fn = (lambda: codec.quant_mx_slices(sl, q, s)) if op == "quant_mx_slices" else one_slice
    elif op in ("dequant_accum_mx", "ring_hop_mx"):
        nsrc = W_SRC if op == "dequant_accum_mx" else 1
        wires = [codec.empty_wire_mx(n, dev) for _ in range(nsrc)]
        for w in range(nsrc):
            x = inputs.prefill_buffer(w, device=dev, rows=rows)
            codec.quant_mx_flat(x.view(-1), wires[w][1], wires[w][2])
            del x
        o = codec.empty_wire_mx(n, dev)
        if op == "dequant_accum_mx":
            fn = lambda: codec.dequant_accum_mx([w[1] for w in wires], [w[2] for w in wires], o[1], o[2], None)
        else:
            xl = inputs.prefill_buffer(1, device=dev, rows=rows).view(-1)
            fn = lambda: codec.ring_hop_mx(wires[0][1], wires[0][2], xl, o[1], o[2], None)
    elif op in ("reduce_quant_i8", "reduce_quant_e4m3"):
        xs = [inputs.prefill_buffer(w, device=dev, rows=rows).view(-1) for w in range(W_SRC)]
        if op == "reduce_quant_i8":
            o = codec.empty_wire_i8(n, dev)
            fn = lambda: codec.reduce_quant_i8(xs, o[1], o[2], None)
        else:
            o = codec.empty_wire_e4m3(n, dev)
            fn = lambda: codec.reduce_quant_e4m3(xs, o[1], o[2], None)
    elif op in ("quant_e4m3", "dequant_e4m3"):
        x0 = inputs.prefill_buffer(0, device=dev, rows=rows).view(-1)
        o = codec.empty_wire_e4m3(n, dev)
        codec.quant_e4m3(x0, o[1], o[2])
        if op == "quant_e4m3":
            fn = lambda: codec.quant_e4m3(x0, o[1], o[2])
        else:
            del x0
            out = torch.empty(n, dtype=torch.bfloat16, device=dev)
            fn = lambda: codec.dequant_e4m3(o[1], o[2], out)
    else:
        nsrc = {"quant_i8": 0, "dequant_i8": 1, "dequant_accum_i8": W_SRC, "ring_hop_i8": 1}[op]
        wires = [codec.empty_wire_i8(n, dev) for _ in range(nsrc)]
        for w in range(nsrc):
            x = inputs.prefill_buffer(w, device=dev, rows=rows)
            codec.quant_i8(x.view(-1), wires[w][1], wires[w][2])
            del x
        o = codec.empty_wire_i8(n, dev)
        if op == "quant_i8":
            x0 = inputs.prefill_buffer(0, device=dev, rows=rows).view(-1)
            fn = lambda: codec.quant_i8(x0, o[1], o[2])
        elif op == "dequant_i8":
            out = torch.empty(n, dtype=torch.bfloat16, device=dev)
            fn = lambda: codec.dequant_i8(wires[0][1], wires[0][2], out)
        elif op == "dequant_accum_i8":
            fn = lambda: codec.dequant_accum_i8([w[1] for w in wires], [w[2] for w in wires], o[1], o[2], None)
        else:
            xl = inputs.prefill_buffer(1, device=dev, rows=rows).view(-1)
            fn = lambda: codec.ring_hop_i8(wires[0][1], wires[0][2], xl, o[1], o[2], None)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # hand the generators' temporaries back: only the op's buffers stay on the device
    for _ in range(args.warmup + args.profile_launches):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"profile_op": op, "rows": rows, "slice_rows": args.slice_rows, "warmup": args.warmup,
                      "launches": args.profile_launches,
                      "device_bytes_held": torch.cuda.memory_reserved(dev)}), flush=True)


# ---------------------------------------------------------------- arms
def workload_config(args, world: int) -> dict:
    """The `config` of both arms' JSON lines: the prefill step's workload."""
    return {"workload": f"prefill pipeline: 4 x BF16 {args.rows}x{HIDDEN} quant_i8 -> dequant_accum_i8 (W=4) "
                        f"-> dequant_i8, ring_hop_i8; 6 x BF16 {args.slice_rows}x{HIDDEN} quant_mx staged into "
                        f"{args.slice_rows}x{HIDDEN * N_SLICES}, dequant_mx",
            "step_bytes": step_bytes_of(args.rows, args.slice_rows), "launches_per_step": 4 + 3 + N_SLICES + 1,
            "l2": "no flush: step working set ~12.5 GB >> 129 MB L2",
            "parallelism": f"replicas x{world} (no collective)"}


def step_bytes_of(rows: int, slice_rows: int) -> int:
    n, ns = rows * HIDDEN, slice_rows * HIDDEN
    return (W_SRC * kernel_bytes("quant_i8", n) + kernel_bytes("dequant_accum_i8", n) + kernel_bytes("dequant_i8", n)
            + kernel_bytes("ring_hop_i8", n) + N_SLICES * kernel_bytes("quant_mx", ns)
            + kernel_bytes("dequant_mx", ns * N_SLICES))


def run_bq(args, rank, world, local):
    from block_quantized_wire_gb300 import build as bq_build
    bq_build.build_library()
    dev = torch.device("cuda", local)
    pipe = Pipeline(args.rows, args.slice_rows, dev)
    step_bytes = pipe.step_bytes()
    nl = len(pipe.launches)
    for _ in range(args.warmup):
        pipe.run()
    torch.cuda.synchronize()

    # Timed region 1 (the reported value): K steps back to back, nothing between the
    # launches of a step, so consecutive kernels overlap their launch with the previous
    # tail; one event at each step boundary gives the per-step samples.
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    nvml = NvmlClocks(dev)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark_start()
        nvml.mark_start()
        start.record()
        for k in range(args.steps):
            pipe.run()
            step_ev[k].record()
        stop.record()
        torch.cuda.synchronize()
        nvml.mark_stop()
        clk.mark_stop()
    barrier(world)
    ms_local = start.elapsed_time(stop)
    ms = max_over_ranks(ms_local, world)
    ms_per_step = ms / args.steps
    step_ms = [start.elapsed_time(step_ev[0])] + [step_ev[k - 1].elapsed_time(step_ev[k])
                                                   for k in range(1, args.steps)]

    # Timed region 2 (per-kernel durations for the roofline): the same K steps with a
    # CUDA event recorded after every launch on the launching stream.
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nl)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record()
    for k in range(args.steps):
        pipe.run(events[k])
    stop.record()
    torch.cuda.synchronize()
    barrier(world)
    ms_instr = start.elapsed_time(stop)

    # per-kernel average launch duration (events on the launching stream)
    per = {}
    for k in range(args.steps):
        prev = start if k == 0 else events[k - 1][nl - 1]
        for i, (name, _, nbytes) in enumerate(pipe.launches):
            t = prev.elapsed_time(events[k][i])
            prev = events[k][i]
            d = per.setdefault(name, {"ms": 0.0, "launches": 0, "bytes": nbytes, "samples": []})
            d["ms"] += t
            d["launches"] += 1
            d["samples"].append(t)
    peak, peak_kind = load_peaks()
    kernels = {}
    for name, d in per.items():
        avg_ms = d["ms"] / d["launches"]
        gbs = d["bytes"] / (avg_ms * 1e-3) / 1e9
        q = sorted(d["samples"])
        pct = {f"p{p}_us": round(q[min(len(q) - 1, int(p / 100 * len(q)))] * 1e3, 2) for p in (10, 50, 90)}
        kernels[name] = {"launches_per_step": d["launches"] // args.steps, "avg_us": round(avg_ms * 1e3, 2), **pct,
                         "median_us": round(statistics.median(q) * 1e3, 2),
                         "bytes_per_launch": d["bytes"], "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                         "share": round(d["ms"] / ms_instr, 4),
                         "samples_us": [round(t * 1e3, 2) for t in d["samples"][:RAW_SAMPLES]],
                         "samples_note": f"launch durations in launch order, the first {min(RAW_SAMPLES, len(q))} "
                                         f"of {len(q)}"}
    # the same kernels timed without the gaps that an event after every launch leaves:
    # each one's launches of a step, repeated, replayed from one CUDA graph
    if not args.no_next:
        by_name = {}
        for name, fn, nbytes in pipe.launches:
            by_name.setdefault(name, []).append((fn, nbytes))
        for name, fns in by_name.items():
            turn = [0]

            def rotate(fns=fns, turn=turn):
                fns[turn[0] % len(fns)][0]()
                turn[0] += 1
            gms, gsamples = graph_stats(rotate, max(args.next_reps, len(fns) * 4))
            gbs_g = fns[0][1] / (gms * 1e-3) / 1e9
            kernels[name].update({"graph_avg_us": round(gms * 1e3, 2), "graph_GB/s": round(gbs_g, 1),
                                  "graph_frac": round(gbs_g / peak, 4),
                                  "graph_spread": spread(gsamples)})
    dominant = max(per, key=lambda k: per[k]["ms"])
    dk = kernels[dominant]
    traffic = None
    tinfo = load_traffic().get(dominant)
    scale = pipe.n / (65536 * HIDDEN) if dominant not in ("quant_mx", "dequant_mx") else 1.0
    if tinfo and tinfo[0] == kernel_sources_sha() and args.rows == 65536:
        traffic = int(tinfo[1] * scale)
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": dk["GB/s"], "peak": peak,
                "timing": "CUDA events after every launch, second timed region of the same K steps",
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s", "unit": "GB/s", "frac": dk["frac"], "traffic": traffic,
                "algorithmic_bytes": dk["bytes_per_launch"]}

    # The MXFP8 wire reductions (mx_a2a accumulate, mx_ring hop) on the same prefill
    # buffers: rows that widen the hot path, timed apart from the step.
    next_rows = None if args.no_next else time_next_rows(pipe, args, peak)
    configs = None if args.no_next else time_configs(args, peak)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        ee = EndToEnd(pipe)
        ee.run(2)
        torch.cuda.synchronize()
        n_e2e = max(2, min(args.steps, args.e2e_steps))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record()
        ee.run(n_e2e)
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        e_ms = max_over_ranks(e0.elapsed_time(e1), world) / n_e2e
        e2e = {"value": round(world * step_bytes / (e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
               "h2d_bytes_per_step": ee.h2d, "d2h_bytes_per_step": ee.d2h, "ms_per_step": round(e_ms, 3),
               "steps": n_e2e,
               "overlap": "two device buffer sets; both copy directions in order on one stream, codec launches "
                          "on another, so each step's computation overlaps its neighbours' copies"}
        del ee

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import shards
        T = args.cpu_threads or shards.host_cores()
        r1, sr1 = min(args.cpu_rows, args.rows), min(args.cpu_slice_rows, args.slice_rows)
        r, sr = min(args.cpu_rows * T, args.rows), min(args.cpu_slice_rows * T, args.slice_rows)
        ci = ([x[:r].cpu() for x in pipe.xs], [s[:sr].cpu() for s in pipe.slices])
        dt1, nb1 = oracle_sample(ci, r1, sr1, 1)
        dt, nb = oracle_sample(ci, r, sr, T)
        parity = oracle_parity(pipe, min(64, args.rows), min(64, args.slice_rows))
        nr = oracle_next_rows(ci, min(256, r, sr))
        cpu = {"value": round(nb / dt / 1e9, 4), "unit": UNIT, "cores": T, "kind": "oracle",
               "parity_sample": parity, "next_rows": nr,
               "sample": f"one step of the same pipeline on the first {r} of {args.rows} rows of each INT8 buffer "
                         f"and the first {sr} of {args.slice_rows} rows of each MX slice, cut into {T} row ranges "
                         f"run by {T} host threads ({nb} algorithmic bytes, {dt:.2f} s wall)",
               "single_thread": {"value": round(nb1 / dt1 / 1e9, 4), "cores": 1,
                                 "sample": f"the first {r1} rows of each INT8 buffer and {sr1} of each MX slice "
                                           f"({nb1} algorithmic bytes, {dt1:.2f} s)"}}

    value = world * step_bytes * args.steps / (ms * 1e-3) / 1e9
    clocks = nvml.summary() or clk.summary()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(args, world),
        "step_median_ms": round(statistics.median(step_ms), 4),
        "step_samples_ms": [round(t, 4) for t in step_ms[:RAW_SAMPLES]],
        "roofline": roofline, "kernels": kernels, "next_rows": next_rows, "configs": configs, "clocks": clocks,
        "e2e": e2e, "gpu_launches": nl * args.steps, "cpu_baseline": cpu,
        "device": torch.cuda.get_device_name(dev), "env": run_env(dev),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, rank, world, local):
    if rank != 0:
        return
    from oracle import shards
    T = args.cpu_threads or shards.host_cores()
    # calibrate a sample so that warmup + steps finish in about args.ref_budget seconds;
    # each step cuts its rows into T ranges run by T host threads
    rmax, smax = min(256 * T, args.rows), min(64 * T, args.slice_rows)
    rows, srows = min(16 * T, rmax), min(4 * T, smax)
    ci = cpu_inputs(rmax, smax)
    dt, nb = oracle_sample(ci, rows, srows, T)
    per_step = max(0.05, min(3.0, args.ref_budget / max(1, args.steps + args.warmup)))
    factor = max(1.0, per_step / max(dt, 1e-3))
    rows = int(min(rmax, max(rows, rows * factor)))
    srows = int(min(smax, max(srows, srows * factor)))
    for _ in range(args.warmup):
        oracle_sample(ci, rows, srows, T)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_sample(ci, rows, srows, T)
        tot_t += dt
        tot_b += nb
    value = tot_b / tot_t / 1e9
    sample = (f"each step: the full step's operations on the first {rows} of {args.rows} rows of each INT8 buffer "
              f"and the first {srows} of {args.slice_rows} rows of each MX slice ({nb} algorithmic bytes), cut "
              f"into {T} row ranges run by {T} host threads")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": workload_config(args, world),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "kind": "oracle", "cores": T, "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["bq", "reference"], default="bq")
    ap.add_argument("--rows", type=int, default=65536, help="rows of each INT8 buffer (65536 = the benchmark)")
    ap.add_argument("--slice-rows", type=int, default=4096, help="rows of each MX slice (4096 = the benchmark)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next", action="store_true",
                    help="skip timing the kernels beyond the step and the smaller configs")
    ap.add_argument("--next-reps", type=int, default=24)
    ap.add_argument("--cpu-rows", type=int, default=1024)
    ap.add_argument("--cpu-slice-rows", type=int, default=256)
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds of CPU work for --impl reference")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads for the oracle legs (0 = every core this process may use)")
    ap.add_argument("--profile-op", choices=PROFILE_OPS, default=None,
                    help="launch only this kernel (--warmup + --profile-launches times) on its own buffers, "
                         "for profiler captures; prints no benchmark line")
    ap.add_argument("--profile-launches", type=int, default=1)
    args = ap.parse_args(argv)
    if args.profile_op:
        run_profile_op(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    if world > 1 and world != args.gpus:
        print(f"bench: WORLD_SIZE={world} differs from --gpus {args.gpus}; using {world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world, local)
        else:
            run_bq(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
