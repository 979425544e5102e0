"""Benchmark of the fused LM-head exact sampler on GB300.

Metric: fused LM-head sample microseconds per decode step and the fraction of
the HBM / tensor-core roofline, versus batch, on a Llama-3-8B-shaped LM head
(d = 4096, V = 128256; synthetic bf16 weights and hidden states -- no trained
weights or datasets).  One step is one call of the public sampling entry point
(one fused-kernel launch; the cross-tile reduction finishes inside it) over one batch of hidden states with
its own step counter.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Under torchrun (N > 1) every rank samples its
own batch of B rows against a replicated W (data-parallel replicas, no
collective on the data path); the timed region is bracketed by a barrier and
a device synchronize, and the slowest rank's time is reported.
"""

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused LM-head sample µs/step & % of HBM/TC roofline vs batch (d4096,V128256)"
UNIT = "us/step"
SWEEP = (1, 2, 4, 8, 16, 32, 64)
SWEEP_LARGE = (128, 256, 512, 1024)


# ---------------------------------------------------------------- roofline
def algorithmic_bytes(B, d, V, bias=False):
    """Bytes one fused launch must move at minimum: W and h read once, the
    temperatures read, and per row an int64 id + fp32 max written (plus the
    fp32 bias when present).  The per-tile candidates are implementation
    overhead and not counted."""
    return 2 * V * d + 2 * B * d + 4 * B + 12 * B + (4 * B * V if bias else 0)


def algorithmic_flops(B, d, V):
    return 2 * B * d * V


# Sources that determine each fused kernel's code (and the compiler flags, in
# build.py); the recorded ncu traffic of a kernel (profiles/traffic.json) is
# only reported while their hash matches.
_CSRC = os.path.join(ROOT, "lm_head_exact_gb300", "csrc")
_SHARED = ["fs_device.cuh", "fs_sm100.cuh", "fs_finish.cuh", "fs_internal.h", "fs_tmap.cu", "fs_tmap.h",
           os.path.join("..", "build.py")]
_TC = ["fs_epilogue.cuh"] + _SHARED
KERNEL_SOURCES = {
    "tc_vocab_kernel": ["fs_tc_vocab.cu"] + _TC,
    "tc_batch_kernel": ["fs_tc_batch.cu"] + _TC,
    "simt_fused_kernel": ["fs_simt.cu"] + _SHARED,
    "tc_pair_kernel": ["fs_tc_pair.cu"] + _TC,
}
PATH_KERNEL = {1: "simt_fused_kernel", 2: "tc_vocab_kernel", 3: "tc_batch_kernel", 4: "tc_pair_kernel"}


def kernel_source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(_CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu capture of `kernel` on
    `workload`, or None if there is none or the kernel's sources changed."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f).get(f"{kernel}@{workload}")
    except (OSError, ValueError):
        return None
    if not entry or entry.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return entry["dram_bytes_per_launch"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def roofline(B, d, V, kernel_us, peaks, bias=False):
    """Roofline entry of the dominant (fused) kernel: bound = the slower of the
    bytes at HBM peak and the FLOPs at bf16 tensor peak."""
    nbytes = algorithmic_bytes(B, d, V, bias)
    flops = algorithmic_flops(B, d, V)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        achieved = nbytes / (kernel_us * 1e-6) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "algorithmic_bytes": nbytes, "roofline_us": round(t_hbm * 1e6, 2),
                "peak_source": peaks["source"]}
    achieved = flops / (kernel_us * 1e-6) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
            "algorithmic_flops": flops, "roofline_us": round(t_tc * 1e6, 2),
            "peak_source": peaks["source"]}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and throttle reasons of one GPU during the timed
    region, through NVML (ctypes; read-only queries) or, failing that, an
    nvidia-smi subprocess."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle"}

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) == 0:
                    self._nvml, self._h = nv, h
                    mx = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = mx.value
        except OSError:
            self._nvml = None

    def _poll(self):
        nv, h = self._nvml, self._h
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit and name != "gpu_idle":
                        self.reasons.add(name)
            time.sleep(0.0005)       # ~15 samples over the 8 ms headline region

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                     "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._proc = None

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append(int(f[0]))
                    self.max_mhz = int(f[1])
                except (ValueError, IndexError):
                    continue
                for n, v in zip(names, f[2:]):
                    if v == "Active":
                        self.reasons.add(n)

    def summary(self):
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples)}


# ---------------------------------------------------------------- dist
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, dist, device=None):
    """Largest value of ``x`` over all ranks (identity without a process group)."""
    if dist is None or not dist.is_initialized():
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- ours
def _to_dev(a, torch):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def time_steps(fs, torch, hd, Wd, td, seed, first_step, n, stream, events=True, bias=None):
    """Run n steps on ``stream``; return (total ms by events around all steps,
    mean fused-kernel ms from per-step profile events)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)] if events else []
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(n)] if events else []
    for ev in starts + stops:          # torch creates the CUDA event on first record
        ev.record(stream)
    ids = torch.empty(hd.shape[0], dtype=torch.int64, device="cuda")
    mx = torch.empty(hd.shape[0], dtype=torch.float32, device="cuda")
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(n):
            if events:
                fs.profile_events(starts[i], stops[i])
            fs.sample(hd, Wd, td, seed, first_step + i, bias=bias, out=(ids, mx), stream=stream)
        t1.record(stream)
    fs.profile_events(None, None)
    torch.cuda.synchronize()
    total = t0.elapsed_time(t1)
    kern = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, stops)) if events else None
    return total, kern


def run_ours(args):
    import torch
    from lm_head_exact_gb300 import binding as fs, synthetic

    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    fs.library()
    fs.set_path({"auto": fs.FS_PATH_AUTO, "simt": fs.FS_PATH_SIMT, "vocab": fs.FS_PATH_TC_VOCAB,
                 "batch": fs.FS_PATH_TC_BATCH, "pair": fs.FS_PATH_TC_PAIR}[args.path])
    peaks = load_peaks()
    kind = "llama3_8b"
    shape = synthetic.SHAPES[kind]
    d, V = shape["d"], shape["V"]
    B = args.batch
    bmax = max(max(SWEEP), B, max(synthetic.SHAPES["chunked"]["batches"]))
    # every rank gets its own batch rows (weak scaling); W is replicated
    h_all = synthetic.normal_rows_bf16(synthetic.SEED_H, bmax * world, d, 1.0)
    h_rank = h_all[rank * bmax:(rank + 1) * bmax]
    W = synthetic.weights(kind)
    Wd = _to_dev(W, torch)
    hd_all = _to_dev(h_rank, torch)
    temp_all = torch.ones(bmax, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    seed = synthetic.SAMPLING_SEED
    fs.workspace_reserve(bmax, V, stream=stream)

    hd, td = hd_all[:B], temp_all[:B]

    def want(section):
        """Extra measurements after the headline: all unless --no-sweep, or
        only those named by --only."""
        if args.only:
            return section in args.only.split(",")
        return not args.no_sweep

    # warm-up (untimed)
    time_steps(fs, torch, hd, Wd, td, seed, 0, args.warmup, stream, events=False)
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier(dist)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    # the timed region: back-to-back steps, events only around the region (a
    # per-step event between two launches would stop their overlap)
    total_ms, _ = time_steps(fs, torch, hd, Wd, td, seed, args.warmup, args.steps, stream, events=False)
    torch.cuda.synchronize()
    barrier(dist)
    if clocks:
        clocks.stop()
    step_ms = max_over_ranks(total_ms / args.steps, dist, device="cuda")
    launches = args.steps              # one fused kernel per step (the cross-tile finish is in-kernel)
    # one launch per step, so the average launch duration over the timed
    # region is the step time; the duration of a launch timed alone (events
    # around each launch, untimed pass) is reported beside it
    kern_ms = step_ms
    _, iso_ms = time_steps(fs, torch, hd, Wd, td, seed, 0, 10, stream)

    # end to end through the host-buffer entry point: pinned h / temp in,
    # ids / max out, every step
    h_pin = torch.from_numpy(h_rank[:B].view(np.int16)).pin_memory()
    t_pin = torch.ones(B, dtype=torch.float32).pin_memory()
    ids_pin = torch.empty(B, dtype=torch.int64).pin_memory()
    mx_pin = torch.empty(B, dtype=torch.float32).pin_memory()
    for i in range(args.warmup):
        fs.sample_host(h_pin, Wd, t_pin, seed, i, out_ids=ids_pin, out_max=mx_pin, stream=stream)
    barrier(dist)
    t0 = time.perf_counter()
    for i in range(args.steps):
        fs.sample_host(h_pin, Wd, t_pin, seed, args.warmup + i, out_ids=ids_pin, out_max=mx_pin,
                       stream=stream)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    barrier(dist)
    e2e_ms = max_over_ranks(e2e_ms, dist, device="cuda")

    # batch sweeps of the metric (same kernels, fewer steps per point): the
    # Llama-3-8B head over the decode range and the large-batch tensor-core
    # range, and the Qwen3-8B head's large batches
    big = max(SWEEP_LARGE)
    big_inputs = {}

    def big_batch():
        """h rows and temperatures for the large-batch points (made once)."""
        if not big_inputs:
            big_inputs["h"] = _to_dev(synthetic.normal_rows_bf16(synthetic.SEED_H, big, d, 1.0), torch)
            big_inputs["t"] = torch.ones(big, dtype=torch.float32, device="cuda")
        return big_inputs["h"], big_inputs["t"]

    sweep = []
    if want("sweep"):
        def point(kind, b, hdev, Wdev, tdev, Vk, dk, bias=None):
            bb = None if bias is None else bias[:b]
            time_steps(fs, torch, hdev[:b], Wdev, tdev[:b], seed, 0, 3, stream, events=False, bias=bb)
            tot, _ = time_steps(fs, torch, hdev[:b], Wdev, tdev[:b], seed, 3, 20, stream, events=False, bias=bb)
            _, km = time_steps(fs, torch, hdev[:b], Wdev, tdev[:b], seed, 23, 5, stream, bias=bb)
            us = tot / 20 * 1e3
            rf = roofline(b, dk, Vk, us, peaks, bias=bias is not None)
            out = {"workload": kind, "B": b, "us_per_step": round(us, 2),
                   "fused_kernel_us_isolated": round(km * 1e3, 2), "roofline_us": rf["roofline_us"],
                   "frac": rf["frac"], "bound": rf["bound"], "path": fs.path_for_batch(b)}
            if b >= 128:
                out["library_gemm_us"] = library_gemm_us(hdev[:b], Wdev)
            return out

        def library_gemm_us(hdev, Wdev, n=20):
            """Context for the contraction regime: the vendor library's plain
            bf16 GEMM (torch.mm -> cuBLAS) on the same shape, logits only (bf16
            out, no bias, no sampling), back to back, µs per call."""
            logits = torch.empty((hdev.shape[0], Wdev.shape[0]), dtype=torch.bfloat16, device="cuda")
            with torch.cuda.stream(stream):
                for _ in range(3):
                    torch.mm(hdev, Wdev.t(), out=logits)
                g0 = torch.cuda.Event(enable_timing=True)
                g1 = torch.cuda.Event(enable_timing=True)
                g0.record(stream)
                for _ in range(n):
                    torch.mm(hdev, Wdev.t(), out=logits)
                g1.record(stream)
            torch.cuda.synchronize()
            del logits
            return round(g0.elapsed_time(g1) / n * 1e3, 2)

        h_big, t_big = big_batch()
        for b in SWEEP:
            sweep.append(point(kind, b, hd_all, Wd, temp_all, V, d))
        for b in SWEEP_LARGE:
            sweep.append(point(kind, b, h_big, Wd, t_big, V, d))
        qshape = synthetic.SHAPES["qwen3_8b"]
        Wq = _to_dev(synthetic.weights("qwen3_8b"), torch)
        tq = _to_dev(synthetic.temperatures("qwen3_8b", big), torch)
        for b in qshape["batches"]:
            sweep.append(point("qwen3_8b", b, h_big, Wq, tq, qshape["V"], qshape["d"]))
        del Wq
        # the Llama-3-70B-shaped head (d 8192) with its dense per-row spike bias
        lshape = synthetic.SHAPES["llama3_70b"]
        bmax70 = max(lshape["batches"])
        W70 = _to_dev(synthetic.weights("llama3_70b"), torch)
        h70 = _to_dev(synthetic.normal_rows_bf16(synthetic.SEED_H, bmax70, lshape["d"], 1.0), torch)
        t70 = torch.ones(bmax70, dtype=torch.float32, device="cuda")
        bias70 = _to_dev(synthetic.spike_bias(bmax70, lshape["V"]), torch)
        for b in lshape["batches"]:
            sweep.append(point("llama3_70b", b, h70, W70, t70, lshape["V"], lshape["d"], bias=bias70))
        del W70, h70, bias70

    # the grouped online (chunked) variant: 8 and 32 contiguous vocabulary
    # chunks per decode step, each chunk one launch; the step is captured in a
    # CUDA graph and replayed (launches amortized), timed with events
    def graph_us(step_fn, reps=20):
        """Capture one step into a CUDA graph, replay it, µs per replay."""
        with torch.cuda.stream(stream):
            step_fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step_fn()
        for _ in range(3):
            graph.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        del graph
        return e0.elapsed_time(e1) / reps * 1e3

    def direct_us(step_fn, reps=20):
        """Back-to-back steps launched directly on the stream (as the one-shot
        rows are timed): 3 untimed, then µs per step over `reps`."""
        with torch.cuda.stream(stream):
            for _ in range(3):
                step_fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                step_fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3

    chunked = []
    if want("chunked"):
        # B = 64 besides the chunked workload's batches: chunk calls there run
        # another tensor-core family than the one-shot call
        configs = [(b, n) for b in sorted(set(synthetic.SHAPES["chunked"]["batches"]) | {64}) for n in (8, 32)]
        if args.chunk_config:
            cb, cn = (int(x) for x in args.chunk_config.split(":"))
            configs = [(cb, cn)]
        for b, n in configs:
            bounds = synthetic.chunk_bounds(V, n)
            cm = torch.empty(b, device="cuda")
            ci = torch.empty(b, dtype=torch.int64, device="cuda")
            cids = torch.empty(b, dtype=torch.int64, device="cuda")
            cmx = torch.empty(b, dtype=torch.float32, device="cuda")
            fs.workspace_reserve(b, V, stream=stream)

            bounds_np = np.asarray(bounds, np.int64)

            def chunk_step():
                for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
                    fs.sample_chunked(hd_all[:b], Wd[lo:hi], lo, temp_all[:b],
                                      seed, 5, cm, ci, i == 0, i == n - 1, out=(cids, cmx), stream=stream)

            def chunk_step_one_call():
                fs.sample_chunked_step(hd_all[:b], Wd, bounds_np, temp_all[:b], seed, 5, cm, ci,
                                       out=(cids, cmx), stream=stream)

            # the step's chunk calls issued from C, steps back to back on the
            # stream (as the one-shot rows); beside it the per-chunk calls
            # replayed as a CUDA graph of one step (graph replays measure
            # slower on GB300 for any kernel, cuBLAS's GEMM included)
            us = direct_us(chunk_step_one_call)
            us_graph = graph_us(chunk_step)
            rf = roofline(b, d, V, us, peaks)
            chunked.append({"workload": "chunked", "B": b, "chunks": n, "us_per_step": round(us, 2),
                            "frac": rf["frac"], "bound": rf["bound"],
                            "path": fs.path_for_chunks(b, bounds[1] - bounds[0], n),
                            "launches_per_step": n, "launch": "fs_sample_chunked_step, back to back",
                            "graph_us_per_step": round(us_graph, 2)})

    # online early finalization (8 chunks): rows without a dominant winner
    # ("flat", every chunk runs) and rows with a +200 spike in the first
    # chunk ("spiked", the later chunks skip their work); the plain chunked
    # step on the same inputs beside it.  The step includes the h row norms.
    early = []
    if want("early"):
        n = 8
        bounds = synthetic.chunk_bounds(V, n)
        rest = fs.chunk_rest_norms(Wd, bounds, stream=stream)
        done = torch.zeros(1, dtype=torch.int32, device="cuda")
        for b in synthetic.SHAPES["chunked"]["batches"]:
            cm = torch.empty(b, device="cuda")
            ci = torch.empty(b, dtype=torch.int64, device="cuda")
            cids = torch.empty(b, dtype=torch.int64, device="cuda")
            cmx = torch.empty(b, dtype=torch.float32, device="cuda")
            hn = torch.empty(b, dtype=torch.float32, device="cuda")
            fs.workspace_reserve(b, V, stream=stream)
            for kind in ("flat", "spiked"):
                bias = None
                if kind == "spiked":
                    bias = _to_dev(synthetic.leading_spike_bias(b, V, bounds[1], 200.0), torch)
                chunks = [(lo, hi, None if bias is None else bias[:, lo:hi])
                          for lo, hi in zip(bounds[:-1], bounds[1:])]

                def early_step(serial=False):
                    fs.row_norms(hd_all[:b], out=hn, stream=stream)
                    for i, (lo, hi, bc) in enumerate(chunks):
                        fs.sample_chunked_early(hd_all[:b], Wd[lo:hi], lo, temp_all[:b], seed, 5, cm, ci,
                                                i == 0, i == n - 1, hn, rest[i], 0.0, done, bias_chunk=bc,
                                                out=(cids, cmx), stream=stream, serial=serial)

                def plain_step():
                    for i, (lo, hi, bc) in enumerate(chunks):
                        fs.sample_chunked(hd_all[:b], Wd[lo:hi], lo, temp_all[:b], seed, 5, cm, ci,
                                          i == 0, i == n - 1, bias_chunk=bc, out=(cids, cmx), stream=stream)

                us_e = graph_us(early_step)
                done_flag = int(done.item())
                us_s = graph_us(lambda: early_step(serial=True))
                us_p = graph_us(plain_step)
                early.append({"workload": "chunked", "inputs": kind, "B": b, "chunks": n,
                              "early_us_per_step": round(us_e, 2), "early_serial_us_per_step": round(us_s, 2),
                              "chunked_us_per_step": round(us_p, 2),
                              "done_after_step": done_flag, "path": fs.path_for_batch(b),
                              "launches_per_step": n + 1, "cuda_graph": True})
                del chunks, bias

    # Gumbel-top-k (k ids per row without replacement) on the same head: a
    # tensor-core kernel with a per-row list epilogue + a merge launch
    topk = []
    if want("topk"):
        for b, k in ((1, 8), (16, 8), (16, 16), (64, 8), (256, 8), (1024, 4)):
            hsrc, tsrc = (hd_all, temp_all) if b <= bmax else big_batch()
            ids_k = torch.empty((b, k), dtype=torch.int64, device="cuda")
            z_k = torch.empty((b, k), dtype=torch.float32, device="cuda")
            with torch.cuda.stream(stream):
                for i in range(3):
                    fs.sample_topk(hsrc[:b], Wd, tsrc[:b], seed, i, k, out=(ids_k, z_k), stream=stream)
                k0 = torch.cuda.Event(enable_timing=True)
                k1 = torch.cuda.Event(enable_timing=True)
                k0.record(stream)
                for i in range(20):
                    fs.sample_topk(hsrc[:b], Wd, tsrc[:b], seed, 3 + i, k, out=(ids_k, z_k), stream=stream)
                k1.record(stream)
            torch.cuda.synchronize()
            us = k0.elapsed_time(k1) / 20 * 1e3
            rf = roofline(b, d, V, us, peaks)
            topk.append({"workload": "llama3_8b", "B": b, "k": k, "us_per_step": round(us, 2), "frac": rf["frac"],
                         "bound": rf["bound"], "launches_per_step": 2})

    # the decode loop: a random-weight Llama-3-8B-shaped decoder body (32
    # layers of projections + SwiGLU MLP) then the LM head, fused vs unfused
    # sampling; the LM head's share of the decode step
    decode = []
    if want("decode"):
        from lm_head_exact_gb300 import decode_loop
        decode = decode_loop.measure(Wd, batches=(1, 16, 256), layers=32, steps=10, warmup=3)
        torch.cuda.empty_cache()

    # the unfused comparison pipeline on the same workload: GEMM -> fp32
    # logits in HBM -> softmax -> sample (the traffic fusion removes)
    unfused = None
    if want("unfused"):
        with torch.cuda.stream(stream):
            for i in range(3):
                fs.sample_unfused(hd, Wd, td, seed, i, stream=stream)
            u0 = torch.cuda.Event(enable_timing=True)
            u1 = torch.cuda.Event(enable_timing=True)
            u0.record(stream)
            for i in range(20):
                fs.sample_unfused(hd, Wd, td, seed, 3 + i, stream=stream)
            u1.record(stream)
        torch.cuda.synchronize()
        uus = u0.elapsed_time(u1) / 20 * 1e3
        unfused = {"us_per_step": round(uus, 2), "fused_us_per_step": round(step_ms * 1e3, 2),
                   "speedup_of_fusion": round(uus / (step_ms * 1e3), 3),
                   "extra_hbm_bytes_per_step": 20 * B * V,
                   "note": "logits write 4BV + softmax reads 8BV, writes 4BV + sample reads 4BV"}

    result = None
    if rank == 0:
        us = step_ms * 1e3
        rf = roofline(B, d, V, kern_ms * 1e3, peaks)
        rf["kernel"] = PATH_KERNEL.get(fs.path_for_batch(B))
        rf["traffic"] = recorded_traffic(rf["kernel"], f"llama3_8b_B{B}")
        rf["kernel_us"] = round(kern_ms * 1e3, 2)
        rf["kernel_us_isolated"] = round(iso_ms * 1e3, 2)
        result = {
            "metric": METRIC, "value": round(us, 2), "unit": UNIT, "higher_is_better": False,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_ms, 4), "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"llama3_8b LM head d={d} V={V} B={B} (Llama-3-8B-shaped, random init)",
                       "global_batch": B * world, "per_gpu_batch": B, "d": d, "V": V,
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "l2": "inputs larger than L2 (W is 1.05 GB); no flush",
                       "tokens_per_s": round(B * world / (us * 1e-6), 1),
                       "path": fs.path_for_batch(B)},
            "roofline": rf,
            "e2e": {"value": round(e2e_ms * 1e3, 2), "unit": UNIT,
                    "h2d_bytes_per_step": B * d * 2 + B * 4, "d2h_bytes_per_step": B * 12},
            "clocks": clocks.summary() if clocks else None,
            "gpu_launches": launches,
            "sweep": sweep,
            "unfused": unfused,
            "chunked": chunked,
            "early_finalization": early,
            "topk": topk,
            "decode_loop": decode,
        }
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(B, args.cpu_seconds)
        # compact table of every timed configuration, kept LAST so that a
        # reader of the line's tail sees it: [workload, B, us/step, fraction
        # of roofline, bound]; chunked entries name their chunk count
        short = {"llama3_8b": "8b", "qwen3_8b": "qwen3", "llama3_70b": "70b+bias"}
        summ = [["8b", B, round(us, 1), rf["frac"], rf["bound"][0]]]
        summ += [[short[p["workload"]], p["B"], round(p["us_per_step"], 1), p["frac"], p["bound"][0]]
                 for p in sweep]
        summ += [[f"chunk{c['chunks']}", c["B"], round(c["us_per_step"], 1), c["frac"], c["bound"][0]]
                 for c in chunked]
        summ += [[f"decode{r['B']}", r["B"], r["fused_step_us"], r["fused_head_share"], "share"]
                 for r in decode]
        result["sweep_summary"] = summ
    if dist is not None:
        dist.destroy_process_group()
    return result


# ---------------------------------------------------------------- oracle arm
def _oracle_step(wl_h, W, temp, seed, step, vocab_rows):
    """One oracle step on the first ``vocab_rows`` rows of W; returns seconds."""
    from oracle import sampler
    t0 = time.perf_counter()
    sampler.sample(wl_h, W[:vocab_rows], temp, seed, step)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline_single_thread(B, seconds):
    """The same oracle measurement in a child process whose BLAS and OpenMP
    pools have one thread (the pools are sized when numpy loads, hence the
    fresh process).  Returns its cpu_baseline dict, or None on failure."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_baseline(%d, %r, single=False)))" % (ROOT, B, seconds))
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                           timeout=30 * seconds + 120)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


def cpu_baseline(B, seconds=20.0, single=True):
    """The fp64 oracle, as it stands, timed on this host's cores on a bounded
    sample: all B rows against a slice of the vocabulary, scaled to the full
    vocabulary (the oracle's cost is linear in V).  With ``single`` the same
    measurement is repeated with one thread (a child process) and reported
    beside it, with the CPU model."""
    from lm_head_exact_gb300 import synthetic
    kind = "llama3_8b"
    V = synthetic.SHAPES[kind]["V"]
    W = synthetic.weights(kind)
    h = synthetic.normal_rows_bf16(synthetic.SEED_H, B, synthetic.SHAPES[kind]["d"], 1.0)
    temp = np.ones(B, np.float32)
    rows = 4096
    t = _oracle_step(h, W, temp, synthetic.SAMPLING_SEED, 0, rows)
    # grow the slice until one sample costs about `seconds / 4`
    while t < seconds / 4 and rows < V:
        rows = min(V, rows * 2)
        t = _oracle_step(h, W, temp, synthetic.SAMPLING_SEED, 0, rows)
    reps, total = 1, t
    while total < seconds * 0.75:
        total += _oracle_step(h, W, temp, synthetic.SAMPLING_SEED, reps, rows)
        reps += 1
    per_step_us = total / reps * (V / rows) * 1e6
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or str(cpu_cores())
    out = {"value": round(per_step_us, 1), "unit": UNIT, "cores": cpu_cores() if threads != "1" else 1,
           "kind": "oracle", "cpu_model": cpu_model(),
           "sample": f"{reps} oracle steps of B={B} rows x {rows} of {V} vocabulary rows, "
                     f"scaled x{V / rows:.2f} to the full vocabulary; numpy fp64 (BLAS threads = {threads})"}
    if single:
        one = cpu_baseline_single_thread(B, seconds / 2)
        if one is not None:
            out["single_thread"] = {"value": one["value"], "unit": UNIT, "cores": 1, "sample": one["sample"]}
    return out


def run_reference(args):
    """Reference arm: the fp64 CPU oracle timed on the host cores, on this
    benchmark's workload (each step a bounded vocabulary slice, scaled)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    from lm_head_exact_gb300 import synthetic
    kind = "llama3_8b"
    d, V = synthetic.SHAPES[kind]["d"], synthetic.SHAPES[kind]["V"]
    B = args.batch
    W = synthetic.weights(kind)
    h = synthetic.normal_rows_bf16(synthetic.SEED_H, B, d, 1.0)
    temp = np.ones(B, np.float32)
    budget = 150.0 / max(1, args.steps + args.warmup)     # seconds per step
    rows = 2048
    while rows < V and _oracle_step(h, W, temp, 1234, 0, min(V, rows * 2)) < budget:
        rows = min(V, rows * 2)
    for i in range(args.warmup):
        _oracle_step(h, W, temp, 1234, i, rows)
    t = sum(_oracle_step(h, W, temp, 1234, args.warmup + i, rows) for i in range(args.steps))
    us = t / args.steps * (V / rows) * 1e6
    sample = (f"B={B} rows x {rows} of {V} vocabulary rows per step, scaled x{V / rows:.2f}; "
              f"numpy fp64 oracle")
    return {"metric": METRIC, "value": round(us, 1), "unit": UNIT, "higher_is_better": False,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(us / 1e3, 3), "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": f"llama3_8b LM head d={d} V={V} B={B} (Llama-3-8B-shaped, random init)",
                       "global_batch": B, "d": d, "V": V, "parallelism": "single"},
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--batch", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--path", choices=["auto", "simt", "vocab", "batch", "pair"], default="auto",
                    help="force a kernel family (profiling)")
    ap.add_argument("--only", default="",
                    help="comma list of extra sections: sweep,chunked,early,topk,decode,unfused")
    ap.add_argument("--chunk-config", default="",
                    help="B:chunks -- the chunked section runs only this configuration (for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


def main(argv=None):
    args = parse_args(argv)
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
