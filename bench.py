"""Benchmark: attention forward + backward TFLOPS on GB300.

One step = the whole hot path on one batch: the fused forward (O, L) and the
backward (D preprocess, fused recomputing backward, dQ conversion), plus the
block-mask compaction when the workload has a mask.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     (the fp64 CPU oracle, timed)

With N > 1 (launched by torch.distributed.run, one rank per GPU) every rank
runs its own replica of the workload (weak scaling; attention over
independent heads needs no exchange), the ranks meet at a barrier around the
timed region and the slowest rank's time counts.
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
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "attention fwd+bwd TFLOPS (bf16, causal/non-causal) & % of GB300 dense BF16 peak"
SPEC_BF16_TFLOPS = 2250.0
L2_BYTES = 129 * 2 ** 20
# the headline: causal, d = 128, the longest sequence of the long-context
# sweep (the largest configuration that fits one GPU)
DEFAULT_WORKLOAD = "long-causal-16384"
# measured beside it, each with its own clocks and roofline
SECONDARY = ("bert-large", "gpt2-1k", "long-causal-4096")
# sequences up to this length sit below the ridge point of the roofline
# (about N / 2 FLOP per byte in the forward): their HBM GB/s is reported too
SHORT_N = 1024
# buffer sets of the e2e leg: step k uploads into set k mod E2E_SETS while
# step k-1 computes and step k-2 downloads, so the three overlap fully
E2E_SETS = 3
# the sources each kernel is built from: a traffic figure taken by ncu
# counts only while their hash is the one recorded beside it
CSRC = os.path.join(ROOT, "exact_attention_12_gb300", "csrc")
KERNEL_SOURCES = {
    "fwd_bf16_kernel": ("attn_fwd.cu", "attn_kernels.cuh", "sm103.cuh", "philox.cuh"),
    "bwd_bf16_kernel": ("attn_bwd.cu", "attn_kernels.cuh", "sm103.cuh", "philox.cuh"),
    "bwd_preprocess_kernel": ("attn_bwd.cu", "attn_kernels.cuh"),
    "dq_convert_kernel": ("attn_bwd.cu", "attn_kernels.cuh"),
}
STAGE_KERNELS = ("fwd_bf16_kernel", "bwd_preprocess_kernel", "bwd_bf16_kernel",
                 "dq_convert_kernel")
PROFILES = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------- FLOPs --

def fwd_flops(w, key_lens=None, block_mask=None):
    """Algorithmic forward FLOPs: 4 d per allowed (query, key) pair.

    Causal counts N^2/2 per head, key padding N*len_b, block-sparse the kept
    128x128 blocks (clipped to N).
    """
    N, d = w.N, w.d
    if block_mask is not None:
        nb = block_mask.shape[-1]
        sizes = torch.full((nb,), 128.0)
        sizes[-1] = N - 128 * (nb - 1)
        bm = block_mask.double()
        pairs = float((sizes[:, None] * sizes[None, :] * bm).sum()) * w.B * w.H
    elif key_lens is not None:
        pairs = float(N * key_lens.double().sum()) * w.H
    elif w.causal:
        pairs = N * N / 2.0 * w.B * w.H
    else:
        pairs = float(N) * N * w.B * w.H
    return 4.0 * d * pairs


def stage_bytes(w):
    """Algorithmic HBM bytes of the four kernels of a step, in the order
    fwd, bwd preprocess, bwd main, dQ conversion.

    fwd reads Q, K, V and writes O, L; the preprocess reads O, dO, L and
    writes D and L*log2(e) (rows padded to whole tiles) and the zeroed fp32
    dQ accumulator; the main kernel reads Q, K, V, dO and the two row
    statistics, writes dK, dV and adds into the accumulator (counted once,
    the adds themselves resolve in L2); the conversion reads the accumulator
    and writes dQ.  bf16 tensors, fp32 statistics and accumulator.
    """
    e = 2
    q = w.B * w.H * w.N * w.d
    kv = w.B * w.kv_heads * w.N * w.d
    rows = w.B * w.H * w.N
    pad = w.B * w.H * ((w.N + 127) // 128 * 128)
    fwd = e * (q + 2 * kv + q) + 4 * rows
    pre = e * 2 * q + 4 * rows + 4 * 2 * pad + 4 * q
    main = e * (q + 2 * kv + q) + 4 * 2 * pad + e * 2 * kv + 4 * q
    dq = 4 * q + e * q
    return fwd, pre, main, dq


def nvtx(name):
    """An NVTX range around a phase of the bench, named in nsys and ncu
    timelines (--nvtx); without a profiler attached it costs a host call."""
    import contextlib
    try:
        return torch.cuda.nvtx.range(f"bench: {name}")
    except (AttributeError, RuntimeError):
        return contextlib.nullcontext()


def kernel_source_hash(kernel):
    """First 16 hex digits of the SHA-256 of the kernel's source files."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` as an
    ncu capture recorded them under profiles/, in lines of the form

        traffic-per-launch | <kernel> | <workload> | <bytes> | src <hash>

    Returns (bytes, note); bytes is None when no capture is recorded or when
    the kernel's sources have changed since (their hash differs)."""
    want = kernel_source_hash(kernel)
    stale = None
    try:
        names = sorted(os.listdir(PROFILES))
    except OSError:
        return None, "no profiles directory"
    for name in names:
        if not name.endswith(".md"):
            continue
        with open(os.path.join(PROFILES, name)) as f:
            for line in f:
                parts = [x.strip() for x in line.strip().strip("`").split("|")]
                if len(parts) != 5 or parts[0] != "traffic-per-launch":
                    continue
                if parts[1] != kernel or parts[2] != workload:
                    continue
                src = parts[4].split()[-1]
                if src == want:
                    return float(parts[3]), f"ncu capture, profiles/{name}"
                stale = f"the capture in profiles/{name} predates the current sources"
    return None, stale or "no ncu capture recorded for this kernel and workload"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["bf16_tflops"], p["bf16_tflops_sustained"], p["hbm_gbs"], "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_ms=50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []      # (host monotonic time, csv line)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, window=None):
        """Median SM clock and the throttle reasons seen: over the samples
        taken inside `window` (host monotonic start, end) when there are
        any, else over every sample (all taken while the step ran)."""
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        lines = self.lines
        inside = [x for x in lines if window and window[0] <= x[0] <= window[1]]
        scope = "timed region" if inside else "step loop around the timed region"
        for _, line in (inside or lines):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "sampled": scope}


# --------------------------------------------------------------- GPU arm --

class Step:
    """One forward + backward through the C interface, stage by stage."""

    def __init__(self, ea, inp, dev):
        from exact_attention_12_gb300 import _abi
        self.abi = _abi
        self.lib = _abi.lib()
        self.dev = dev
        self.q, self.k, self.v, self.do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
        self.key_lens = None if inp["key_lens"] is None else inp["key_lens"].to(dev)
        self.block_mask = None if inp["block_mask"] is None else inp["block_mask"].to(dev)
        self.p = ea.make_params(self.q, k=self.k, scale=inp["scale"], causal=inp["causal"],
                                key_lens=self.key_lens, dropout_p=inp["dropout_p"],
                                seed=inp["seed"], offset=inp["offset"],
                                block_mask=self.block_mask)
        B, H, N, d = self.q.shape
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(self.q)
        self.dk, self.dv = torch.empty_like(self.k), torch.empty_like(self.k)
        nbytes = max(ea.workspace_size(self.p, True), ea.workspace_size(self.p, False))
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self.launches = 1 + 3 + (2 if self.block_mask is not None else 0)

    def run(self, stream, ev=None):
        """Enqueue the step; `ev` = 4 events around fwd / preprocess / main / dq."""
        lib, P, s = self.lib, ctypes.byref(self.p), ctypes.c_void_p(stream.cuda_stream)
        wsp, wsn = self.ws.data_ptr(), self.ws.numel()
        if ev:
            ev[0].record(stream)
        st = lib.attn_fwd(P, self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(),
                          self.o.data_ptr(), self.lse.data_ptr(), wsp, wsn, s)
        self.abi.check_status(st, "attn_fwd")
        if ev:
            ev[1].record(stream)
        st = lib.attn_bwd_preprocess(P, self.o.data_ptr(), self.lse.data_ptr(), self.do.data_ptr(),
                                     wsp, wsn, s)
        self.abi.check_status(st, "attn_bwd_preprocess")
        if ev:
            ev[2].record(stream)
        st = lib.attn_bwd_main(P, self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(),
                               self.do.data_ptr(), self.dk.data_ptr(), self.dv.data_ptr(),
                               wsp, wsn, s)
        self.abi.check_status(st, "attn_bwd_main")
        if ev:
            ev[3].record(stream)
        st = lib.attn_bwd_dq(P, self.dq.data_ptr(), wsp, wsn, s)
        self.abi.check_status(st, "attn_bwd_dq")
        if ev:
            ev[4].record(stream)

    def bytes_resident(self):
        t = [self.q, self.k, self.v, self.do, self.o, self.lse, self.dq, self.dk, self.dv, self.ws]
        return sum(x.numel() * x.element_size() for x in t)


class StepGraphs:
    """The step captured in CUDA graphs, for timing without host launch cost.

    `enqueue(k, stream)` enqueues one step on input set k.  `block` holds
    `per` consecutive steps (the sets in rotation; `per` is a multiple of
    `nsets`), `one[k]` a single step on set k, so that `replay(n)` enqueues
    exactly n steps in rotation order on the current stream.  Nothing is
    allocated inside the captures: every step writes into buffers that exist
    before them.
    """

    def __init__(self, enqueue, nsets, dev, per_target=16):
        self.nsets = nsets
        self.per = max(1, per_target // nsets) * nsets
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        self.block = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.block, stream=side):
            for i in range(self.per):
                enqueue(i % nsets, torch.cuda.current_stream(dev))
        self.one = []
        for k in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                enqueue(k, torch.cuda.current_stream(dev))
            self.one.append(g)
        torch.cuda.synchronize(dev)

    def replay(self, steps):
        for kind, k in replay_plan(steps, self.per, self.nsets):
            (self.block if kind == "block" else self.one[k]).replay()


def replay_plan(steps, per, nsets):
    """The graph launches that enqueue exactly `steps` steps with the input
    sets in rotation: ("block", None) for a graph of `per` steps (a multiple
    of `nsets`, starting at set 0), ("one", k) for a single step on set k."""
    if per % nsets:
        raise ValueError("a block must hold whole rotations of the input sets")
    blocks, rest = divmod(steps, per)
    return [("block", None)] * blocks + [("one", i % nsets) for i in range(rest)]


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, x, dev):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measure_device(ea, w, dev, steps, warmup, dist=None):
    """Device-resident timing of `steps` steps; returns a dict of results.

    Clocks are sampled from the start of the per-kernel event pass to the end
    of the timed region; the summary takes the samples inside the timed
    region (all of them when it is shorter than the sampling period)."""
    inp = workloads.make_inputs(w)
    first = Step(ea, inp, dev)
    # rotate input sets so consecutive steps do not find their data in L2
    nsets = max(1, min(8, math.ceil(2 * L2_BYTES / max(1, first.bytes_resident()))))
    sets = [first] + [Step(ea, inp, dev) for _ in range(nsets - 1)]
    stream = torch.cuda.current_stream(dev)
    with nvtx(f"{w.name} warm-up"):
        for i in range(warmup):
            sets[i % nsets].run(stream)
        torch.cuda.synchronize(dev)
    with nvtx(f"{w.name} graph capture"):
        graphs = StepGraphs(lambda k, s: sets[k].run(s), nsets, dev)
        graphs.replay(nsets)
        torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.__enter__()
    time.sleep(0.2)       # let the sampler start before the loaded window
    # kernel times: the same steps launched one by one, an event around each
    # launch (the events cost ~10 us per step, so the step itself is timed
    # below without them)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    with nvtx(f"{w.name} per-kernel event pass"):
        for i in range(steps):
            sets[i % nsets].run(stream, evs[i])
        torch.cuda.synchronize(dev)
    stage = [sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)) / steps
             for j in range(4)]
    # the step: replayed from CUDA graphs (the host launch cost of four ctypes
    # calls is not the kernels'), input sets in rotation as above
    _barrier(dist)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.monotonic()
    with nvtx(f"{w.name} timed steps"):
        start.record(stream)
        graphs.replay(steps)
        end.record(stream)
        torch.cuda.synchronize(dev)
    t1 = time.monotonic()
    _barrier(dist)
    time.sleep(0.06)
    sampler.__exit__()
    ea.check(first.ws, dev)
    total_ms = _max_over_ranks(dist, start.elapsed_time(end), dev)
    flops_f = fwd_flops(w, inp["key_lens"], inp["block_mask"])
    return dict(inp=inp, total_ms=total_ms, ms_per_step=total_ms / steps, stage_ms=stage,
                fwd_flops=flops_f, bwd_flops=2.5 * flops_f, nsets=nsets,
                resident_bytes=first.bytes_resident(), launches=first.launches * steps,
                clocks=sampler.summary((t0, t1)))


def roofline(w, r):
    """The roofline of the step's dominant kernel (the longest of the four
    stages in the event pass): its algorithmic FLOPs and bytes over its
    measured time, against the measured burst bf16 peak (the kernel is timed
    launch by launch) and the measured HBM bandwidth; `bound` is whichever
    of the two it is closer to."""
    burst, _, hbm, src = peaks()
    stage = r["stage_ms"]
    k = max(range(4), key=lambda i: stage[i])
    flops = (r["fwd_flops"], 0.0, r["bwd_flops"], 0.0)[k]
    nbytes = stage_bytes(w)[k]
    t = stage[k] * 1e-3
    tf, gbs = flops / t / 1e12, nbytes / t / 1e9
    tensor_frac, hbm_frac = tf / burst, gbs / hbm
    kernel = STAGE_KERNELS[k]
    traffic, note = profiled_traffic(kernel, w.name)
    if tensor_frac >= hbm_frac:
        bound, achieved, peak, unit = "tensor", tf, burst, "TFLOP/s"
        psrc = f"bf16_tflops, burst ({src})"
    else:
        bound, achieved, peak, unit = "hbm", gbs, hbm, "GB/s"
        psrc = f"hbm_gbs ({src})"
    return {"kernel": kernel, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": psrc, "kernel_ms": stage[k],
            "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
            "tensor_frac": tensor_frac, "hbm_frac": hbm_frac,
            "traffic": traffic, "traffic_unit": "DRAM bytes read + written per launch (ncu)",
            "traffic_source": note}


def hbm_rates(w, r):
    """Achieved HBM GB/s of the whole step and of each kernel, algorithmic
    bytes (stage_bytes) over measured time, against the measured copy
    bandwidth; reported for the short sequences that sit below the ridge."""
    _, _, hbm, src = peaks()
    nb = stage_bytes(w)
    per = {k: b / (ms * 1e-3) / 1e9 for k, b, ms in zip(STAGE_KERNELS, nb, r["stage_ms"])}
    step = sum(nb) / (r["ms_per_step"] * 1e-3) / 1e9
    return {"achieved_gbs": step, "peak_gbs": hbm, "frac": step / hbm,
            "peak_source": f"hbm_gbs ({src})", "bytes_per_step": sum(nb),
            "kernel_gbs": per}


def workload_result(w, r, world=1):
    """The figures of one measured workload (measure_device's result)."""
    burst, sustained, _, _ = peaks()
    ms = r["ms_per_step"]
    value = world * (r["fwd_flops"] + r["bwd_flops"]) / (ms * 1e-3) / 1e12
    fwd_ms, pre_ms, main_ms, dq_ms = r["stage_ms"]
    out = {"value": value, "ms_per_step": ms,
           "fwd_tflops": r["fwd_flops"] / (fwd_ms * 1e-3) / 1e12,
           "bwd_tflops": r["bwd_flops"] / ((pre_ms + main_ms + dq_ms) * 1e-3) / 1e12,
           "stage_ms": {"fwd": fwd_ms, "bwd_preprocess": pre_ms, "bwd_main": main_ms,
                        "bwd_dq": dq_ms},
           "pct_of_peak": {"of_spec_2250": 100 * value / world / SPEC_BF16_TFLOPS,
                           "of_measured_burst": 100 * value / world / burst,
                           "of_measured_sustained": 100 * value / world / sustained},
           "roofline": roofline(w, r),
           "clocks": r["clocks"]}
    if w.N <= SHORT_N:
        out["hbm"] = hbm_rates(w, r)
    return out


def headline_line(w, r, steps, warmup, world):
    """The JSON line of the training-step bench from a measure_device result
    (the cpu_baseline, e2e and secondary entries are added by the caller)."""
    res = workload_result(w, r, world)
    line = {
        "metric": METRIC, "value": res.pop("value"), "unit": "TFLOPS", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": res.pop("ms_per_step"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": describe(w), "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "dropout_p": w.dropout_p,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs rotate over {r['nsets']} resident sets of "
                         f"{r['resident_bytes'] / 2**20:.0f} MiB (> 2x the 129 MB L2)",
                   "timing": "steps captured in CUDA graphs and replayed, CUDA events around "
                             "the K steps; stage_ms and the roofline kernel time from a "
                             "separate pass of K steps launched one by one with an event "
                             "around each launch"},
        "gpu_launches": r["launches"],
    }
    line.update(res)
    return line


def measure_e2e(ea, w, dev, steps, warmup):
    """Same metric through the Python API with host (pinned) inputs and outputs.

    Every step copies its inputs host -> device, runs the forward and the
    backward, and copies dQ, dK, dV device -> host.  Steps are pipelined over
    three streams (uploads, compute, downloads) with E2E_SETS buffer sets, so the
    copies of one step overlap the compute of its neighbours; the time is
    taken from the first upload to the last download.
    """
    inp = workloads.make_inputs(w)
    names = ("q", "k", "v", "do")
    host = {n: inp[n].pin_memory() for n in names}
    kl = None if inp["key_lens"] is None else inp["key_lens"].to(dev)
    bm = None if inp["block_mask"] is None else inp["block_mask"].to(dev)
    kw = dict(scale=inp["scale"], causal=inp["causal"], key_lens=kl, dropout_p=inp["dropout_p"],
              seed=inp["seed"], offset=inp["offset"], block_mask=bm)
    shape, dtype = inp["q"].shape, inp["q"].dtype
    shapes = {n: inp[n].shape for n in names}
    out_shapes = (inp["q"].shape, inp["k"].shape, inp["v"].shape)   # dQ, dK, dV
    dev_in = [{n: torch.empty(shapes[n], dtype=dtype, device=dev) for n in names}
              for _ in range(E2E_SETS)]
    dev_out = [[torch.empty(sh, dtype=dtype, device=dev) for sh in out_shapes]
               for _ in range(E2E_SETS)]
    host_out = [[torch.empty(sh, dtype=dtype).pin_memory() for sh in out_shapes]
                for _ in range(E2E_SETS)]
    up, comp, down = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(E2E_SETS)]     # inputs of buffer set uploaded
    ev_used = [torch.cuda.Event() for _ in range(E2E_SETS)]   # compute done with buffer set
    ev_out = [torch.cuda.Event() for _ in range(E2E_SETS)]    # downloads of buffer set done
    def step(k):
        b = k % E2E_SETS
        with torch.cuda.stream(up):
            up.wait_event(ev_used[b])
            for n in names:
                dev_in[b][n].copy_(host[n], non_blocking=True)
            ev_in[b].record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(ev_in[b])
            comp.wait_event(ev_out[b])
            d = dev_in[b]
            o, lse = ea.attention_fwd(d["q"], d["k"], d["v"], **kw)
            ea.attention_bwd(d["do"], d["q"], d["k"], d["v"], o, lse, dq=dev_out[b][0],
                             dk=dev_out[b][1], dv=dev_out[b][2], **kw)
            ev_used[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev_used[b])
            for dst, src in zip(host_out[b], dev_out[b]):
                dst.copy_(src, non_blocking=True)
            ev_out[b].record(down)

    with nvtx(f"{w.name} e2e warm-up"):
        for k in range(warmup):
            step(k)
        torch.cuda.synchronize(dev)
    with nvtx(f"{w.name} e2e timed steps"):
        t0 = time.perf_counter()
        for k in range(steps):
            step(k)
        torch.cuda.synchronize(dev)
        dt = (time.perf_counter() - t0) / steps
    flops = 3.5 * fwd_flops(w, inp["key_lens"], inp["block_mask"])
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3,
            "pipelining": f"uploads, compute and downloads on three streams, {E2E_SETS} buffer sets"}


# ---------------------------------------------------------- oracle (CPU) --

def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else os.cpu_count()
    except ImportError:
        return os.cpu_count()


ORACLE_ROWS = 256     # query rows per oracle timing unit (the oracle's own chunk)


def oracle_units(w, seed=0):
    """The oracle's timing units of a workload, in a seeded random order:
    (b, h, rows) with rows a whole head when N <= SHORT_N, else one block of
    ORACLE_ROWS consecutive query rows."""
    import numpy as np
    if w.N <= SHORT_N:
        blocks = [np.arange(w.N)]
    else:
        blocks = [np.arange(s0, min(w.N, s0 + ORACLE_ROWS)) for s0 in range(0, w.N, ORACLE_ROWS)]
    units = [(b, h, r) for b in range(w.B) for h in range(w.H) for r in blocks]
    order = np.random.default_rng(seed).permutation(len(units))
    return [units[i] for i in order]


def rows_flops(w, inp, b, rows):
    """fwd+bwd FLOPs of query rows `rows` of batch b: 3.5 x 4 d per allowed
    (query, key) pair, with the workload's causal, padding and block masks."""
    import numpy as np
    rows = np.asarray(rows, dtype=np.int64)
    kl = inp["key_lens"]
    key_len = w.N if kl is None else min(w.N, max(0, int(kl[b])))
    lim = np.minimum(key_len, rows + 1 if w.causal else np.full(rows.shape, w.N))
    bm = inp["block_mask"]
    if bm is None:
        pairs = float(np.maximum(lim, 0).sum())
    else:
        m = bm.numpy().astype(bool)[rows // 128]                       # [R, nb]
        starts = 128 * np.arange(m.shape[1])
        overlap = np.clip(lim[:, None] - starts[None, :], 0, 128)
        pairs = float((m * overlap).sum())
    return 3.5 * 4.0 * w.d * pairs


def oracle_inputs(inp):
    """The workload's tensors as numpy fp32 (exact for bf16 values; the
    oracle takes each head to fp64 itself) and its oracle keyword arguments."""
    arr = {n: inp[n].float().numpy() for n in ("q", "k", "v", "do")}
    kl, bm = inp["key_lens"], inp["block_mask"]
    kw = dict(scale=inp["scale"], causal=inp["causal"],
              key_lens=None if kl is None else kl.numpy(),
              block_mask=None if bm is None else bm.numpy(),
              dropout_p=inp["dropout_p"], seed=inp["seed"], offset=inp["offset"])
    return arr, kw


def oracle_sample(w, inp, units, arrays, budget_s, start=0):
    """Time the oracle's fwd+bwd on `units` (from oracle_units) starting at
    index `start`, until `budget_s` has passed (at least one unit).  Each
    unit's rows go through oracle.backward_rows, which evaluates O, L, dQ and
    the rows' dK, dV contributions.  Returns (flops, seconds, units done)."""
    from oracle import attention as oracle
    arr, kw = arrays
    done, flops = 0, 0.0
    t0 = time.perf_counter()
    while True:
        b, h, rows = units[(start + done) % len(units)]
        oracle.backward_rows(arr["q"], arr["k"], arr["v"], arr["do"], b, h, rows, **kw)
        flops += rows_flops(w, inp, b, rows)
        done += 1
        if time.perf_counter() - t0 > budget_s or done >= len(units):
            break
    return flops, time.perf_counter() - t0, done


def oracle_unit_name(w):
    return "(b, h) heads" if w.N <= SHORT_N else f"blocks of {ORACLE_ROWS} query rows"


def run_reference(args, w):
    """The reference arm: the fp64 CPU oracle, as it stands, on host cores.
    Each step is a bounded sample of the workload: timing units (whole
    heads, or blocks of query rows at long N) for about half a second."""
    inp = workloads.make_inputs(w)
    units = oracle_units(w)
    arrays = oracle_inputs(inp)
    pos = 0
    for _ in range(args.warmup):
        _, _, n = oracle_sample(w, inp, units, arrays, 0.5, pos)
        pos += n
    total_f, total_t, total_n = 0.0, 0.0, 0
    for _ in range(args.steps):
        f, dt, n = oracle_sample(w, inp, units, arrays, 0.5, pos)
        pos += n
        total_f, total_t, total_n = total_f + f, total_t + dt, total_n + n
    value = total_f / total_t / 1e12
    cores = _blas_threads()
    sample = (f"{total_n} timing units ({oracle_unit_name(w)}, about 0.5 s per step) of "
              f"{w.name}, fp64 numpy fwd+bwd")
    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(w), "parallelism": "none (host cores)"},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def describe(w):
    heads = f"H={w.H}" if w.kv_heads == w.H else f"H={w.H} H_kv={w.kv_heads}"
    parts = [f"{w.name}: B={w.B} {heads} N={w.N} d={w.d} {w.dtype}"]
    parts.append("causal" if w.causal else "non-causal")
    if w.key_len_range:
        parts.append(f"key lengths U{{{w.key_len_range[0]}..{w.key_len_range[1]}}}")
    if w.dropout_p:
        parts.append(f"dropout p={w.dropout_p}")
    if w.block_density:
        parts.append(f"block-sparse 128x128, density ~{w.block_density}")
    return ", ".join(parts)


# ------------------------------------------------------------ decode step --

def decode_flops(w, key_lens):
    """Matmul FLOPs of one decode step: 4 d per (query row, allowed key)."""
    n_q = w.decode_n_q
    total = 0
    for n in key_lens.tolist():
        n = max(0, min(int(n), w.N))
        # query t at position n - n_q + t attends keys j <= its position (causal)
        allowed = sum(max(0, min(n, n - n_q + t + 1)) for t in range(n_q)) if w.causal \
            else n_q * n
        total += allowed
    return 4.0 * w.d * w.H * total


def decode_bytes(w, key_lens):
    """HBM bytes a decode step must move: the cached keys and values it reads
    (bf16), the query rows read and the output rows written."""
    cached = sum(max(0, min(int(n), w.N)) for n in key_lens.tolist())
    kv = 2 * cached * w.kv_heads * w.d * 2
    rows = w.B * w.H * w.decode_n_q
    return kv + 2 * rows * w.d * 2 + rows * 4


def measure_decode(ea, w, dev, steps, warmup):
    """Device-timed decode steps over one resident cache (larger than the L2),
    plus the e2e leg: each step uploads its query rows from pinned host memory
    and downloads O, the cache staying resident as it would between tokens."""
    inp = workloads.make_inputs(w)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    lens = inp["key_lens"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        ea.attention_decode(q, k, v, lens, scale=inp["scale"], causal=w.causal, out=o, lse=lse)
    torch.cuda.synchronize(dev)
    graphs = StepGraphs(lambda _k, _s: ea.attention_decode(q, k, v, lens, scale=inp["scale"],
                                                          causal=w.causal, out=o, lse=lse),
                        1, dev)
    graphs.replay(1)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.__enter__()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    graphs.replay(steps)
    end.record(stream)
    torch.cuda.synchronize(dev)
    sampler.__exit__()
    ea.check()
    ms = start.elapsed_time(end) / steps
    # e2e: query rows up, output rows down, every step
    hq = inp["q"].pin_memory()
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    for _ in range(3):
        q.copy_(hq, non_blocking=True)
        ea.attention_decode(q, k, v, lens, scale=inp["scale"], causal=w.causal, out=o, lse=lse)
        ho.copy_(o, non_blocking=True)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    n_e2e = max(3, min(steps, 200))
    for _ in range(n_e2e):
        q.copy_(hq, non_blocking=True)
        ea.attention_decode(q, k, v, lens, scale=inp["scale"], causal=w.causal, out=o, lse=lse)
        ho.copy_(o, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_ms = (time.perf_counter() - t0) / n_e2e * 1e3
    return dict(inp=inp, ms=ms, e2e_ms=e2e_ms, clocks=sampler.summary(),
                h2d=hq.numel() * hq.element_size(), d2h=ho.numel() * ho.element_size())


def run_decode(args, w):
    import numpy as np
    from oracle import attention as oracle
    inp_cpu = workloads.make_inputs(w)
    # oracle: sequences timed one by one until the budget is spent
    t0 = time.perf_counter()
    done, flops_cpu = 0, 0.0
    for b in range(w.B):
        oracle.decode_forward(inp_cpu["q"][b:b + 1].double().numpy(),
                              inp_cpu["k"][b:b + 1].double().numpy(),
                              inp_cpu["v"][b:b + 1].double().numpy(), scale=inp_cpu["scale"],
                              cache_lens=inp_cpu["key_lens"][b:b + 1].numpy(), causal=w.causal)
        flops_cpu += decode_flops(workloads.get(w.name, B=1), inp_cpu["key_lens"][b:b + 1])
        done += 1
        if time.perf_counter() - t0 > args.cpu_budget:
            break
    dt_cpu = time.perf_counter() - t0
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    r = measure_decode(ea, w, dev, args.steps, args.warmup)
    lens = r["inp"]["key_lens"]
    flops = decode_flops(w, lens)
    nbytes = decode_bytes(w, lens)
    _, _, hbm, src = peaks()
    gbs = nbytes / (r["ms"] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": flops / (r["ms"] * 1e-3) / 1e12, "unit": "TFLOPS",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": describe(w), "B": w.B, "H": w.H, "H_kv": w.kv_heads,
                   "n_q": w.decode_n_q, "cache_capacity": w.N, "d": w.d, "causal": w.causal,
                   "parallelism": "single GPU",
                   "l2": f"the resident cache ({nbytes / 2**20:.0f} MiB read per step) is larger "
                         f"than the 129 MB L2",
                   "timing": "decode calls captured in a CUDA graph, replayed; CUDA events"},
        "roofline": {"kernel": "decode_mma_kernel" if (w.H // w.kv_heads) * w.decode_n_q <= 16
                     else "decode_kernel", "bound": "hbm", "achieved": gbs, "peak": hbm,
                     "unit": "GB/s", "frac": gbs / hbm, "peak_source": f"hbm_gbs ({src})",
                     "traffic": None},
        "gpu_launches": 2 * args.steps,
        "clocks": r["clocks"],
        "cpu_baseline": {"value": flops_cpu / dt_cpu / 1e12, "unit": "TFLOPS",
                         "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"{done} of {w.B} sequences of {w.name}, fp64 numpy, "
                                   f"{dt_cpu:.1f} s"},
        "e2e": {"value": flops / (r["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": r["e2e_ms"],
                "note": "query rows up and output rows down per step; the cache stays resident"},
    }
    print(json.dumps(line))


# ------------------------------------------------------------- FP8 forward --

FP8_METRIC = "attention fwd TFLOPS (E4M3 Q, K, V; bf16 O) & % of GB300 dense FP8 peak"
FP8_NOMINAL_RATIO = 2.0   # dense FP8 / dense BF16 tensor throughput (4.5 / 2.25 PFLOP/s)


FP32_METRIC = "attention fwd TFLOPS (fp32 Q, K, V, O; tcgen05 kind::tf32) & % of GB300 TF32 peak"
TF32_NOMINAL_RATIO = 1.1 / 2.25   # dense TF32 / dense BF16 tensor throughput (PFLOP/s)


def _fp8_kw(inp):
    return dict(scale=inp["scale"], causal=inp["causal"], q_descale=inp["q_descale"],
                k_descale=inp["k_descale"], v_descale=inp["v_descale"])


def _fwd_kw(w, inp, dev):
    """attention_fwd keywords of a forward-only workload (FP8 or fp32)."""
    if w.dtype == "fp8":
        return _fp8_kw(inp)
    kl, bm = inp["key_lens"], inp["block_mask"]
    return dict(scale=inp["scale"], causal=inp["causal"], dropout_p=inp["dropout_p"],
                seed=inp["seed"], offset=inp["offset"],
                key_lens=None if kl is None else kl.to(dev),
                block_mask=None if bm is None else bm.to(dev))


def measure_fwd(ea, w, dev, steps, warmup):
    """Device-timed forward steps (one attn_fwd call: for FP8 the V transpose
    + fused forward, for fp32 the operand split + TF32 forward) over input
    sets that rotate so each step misses the L2, then the e2e leg: Q, K, V up
    from pinned host memory and O down, every step."""
    inp = workloads.make_inputs(w)
    kw = _fwd_kw(w, inp, dev)

    def make_set():
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        o, lse = ea.attention_fwd(q, k, v, **kw)
        return q, k, v, o, lse

    first = make_set()
    nbytes = sum(t.numel() * t.element_size() for t in first) + \
        w.B * w.kv_heads * w.d * ((w.N + 127) // 128 * 128)
    nsets = max(1, min(8, math.ceil(2 * L2_BYTES / nbytes)))
    sets = [first] + [make_set() for _ in range(nsets - 1)]
    ws = ea.workspace(dev, 0)
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        q, k, v, o, lse = sets[i % nsets]
        ea.attention_fwd(q, k, v, out=o, lse=lse, **kw)
    torch.cuda.synchronize(dev)
    def enqueue(i, s):
        q, k, v, o, lse = sets[i]
        ea.attention_fwd(q, k, v, out=o, lse=lse, **kw)

    graphs = StepGraphs(enqueue, nsets, dev)
    graphs.replay(nsets)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.__enter__()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    graphs.replay(steps)
    end.record(stream)
    torch.cuda.synchronize(dev)
    sampler.__exit__()
    ea.check(ws, dev)
    ms = start.elapsed_time(end) / steps
    # e2e
    host = [inp[n].pin_memory() for n in ("q", "k", "v")]
    q, k, v, o, lse = first
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()

    def e2e_step():
        for d, h in zip((q, k, v), host):
            d.copy_(h, non_blocking=True)
        ea.attention_fwd(q, k, v, out=o, lse=lse, **kw)
        ho.copy_(o, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    n_e2e = max(3, min(steps, 100))
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms = (time.perf_counter() - t0) / n_e2e * 1e3
    return dict(inp=inp, ms=ms, e2e_ms=e2e_ms, clocks=sampler.summary(), nsets=nsets,
                resident=nbytes, h2d=sum(h.numel() * h.element_size() for h in host),
                d2h=ho.numel() * ho.element_size())


def fwd_only_oracle_sample(w, budget_s):
    """Time the oracle's forward of a forward-only workload head by head (the
    FP8 oracle for E4M3 inputs, the fp64 forward otherwise) until `budget_s`
    has passed (at least one head).  Returns (flops, seconds, heads done)."""
    fp8 = w.dtype == "fp8"
    inp = workloads.make_inputs(w)
    grp = w.H // w.kv_heads
    per_head = fwd_flops(workloads.get(w.name, B=1, H=1, H_kv=1))
    if fp8:
        from oracle import fp8 as oracle_fp8
        ds = (inp["q_descale"], inp["k_descale"], inp["v_descale"])
    else:
        import numpy as np
        from oracle import attention as oracle
        arr = {n: inp[n].float().numpy() for n in ("q", "k", "v")}
        okw = dict(scale=inp["scale"], causal=inp["causal"], dropout_p=inp["dropout_p"],
                   seed=inp["seed"], offset=inp["offset"])
    t0 = time.perf_counter()
    done, flops = 0, 0.0
    for b, h in ((b, h) for b in range(w.B) for h in range(w.H)):
        if fp8:
            codes = [inp[n][b:b + 1, sl].view(torch.uint8).numpy() for n, sl in
                     (("q", slice(h, h + 1)), ("k", slice(h // grp, h // grp + 1)),
                      ("v", slice(h // grp, h // grp + 1)))]
            oracle_fp8.fp8_forward(*codes, *ds, inp["scale"], causal=w.causal)
        else:
            oracle.forward_rows(arr["q"], arr["k"], arr["v"], b, h, np.arange(w.N), **okw)
        flops += per_head
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return flops, time.perf_counter() - t0, done


def run_fwd_only(args, w):
    """A forward-only workload (FP8, or fp32 on the TF32 tensor path): fwd
    TFLOPS against that type's tensor peak (the measured BF16 peak times the
    nominal FP8/BF16 or TF32/BF16 ratio), the oracle timed beside it."""
    fp8 = w.dtype == "fp8"
    flops_cpu, dt_cpu, done = fwd_only_oracle_sample(w, args.cpu_budget)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    r = measure_fwd(ea, w, dev, args.steps, args.warmup)
    flops = fwd_flops(w)
    burst, _, _, src = peaks()
    ratio = FP8_NOMINAL_RATIO if fp8 else TF32_NOMINAL_RATIO
    peak = ratio * burst
    tflops = flops / (r["ms"] * 1e-3) / 1e12
    line = {
        "metric": FP8_METRIC if fp8 else FP32_METRIC, "value": tflops, "unit": "TFLOPS",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if fp8 else "f32", "data": "synthetic",
        "config": {"workload": describe(w), "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "parallelism": "single GPU",
                   "l2": f"inputs rotate over {r['nsets']} resident sets of "
                         f"{r['resident'] / 2**20:.0f} MiB (> 2x the 129 MB L2)",
                   "timing": "attn_fwd calls captured in CUDA graphs, replayed; CUDA events"},
        "roofline": {"kernel": "fwd_fp8_kernel" if fp8 else "fwd_tf32_kernel", "bound": "tensor",
                     "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "peak_source": f"bf16_tflops ({src}) x {ratio:.4g} "
                                    f"(nominal dense {'FP8' if fp8 else 'TF32'} / BF16)",
                     "timed": "the attn_fwd call: V transpose + fused forward" if fp8 else
                              "the attn_fwd call: operand split + TF32 forward (the scores "
                              "take three TF32 passes: the tensor work is 2x the counted FLOPs)",
                     "traffic": None},
        "gpu_launches": 2 * args.steps,
        "clocks": r["clocks"],
        "cpu_baseline": {"value": flops_cpu / dt_cpu / 1e12, "unit": "TFLOPS",
                         "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"{done} of {w.B * w.H} heads of {w.name}, fp64 numpy "
                                   f"forward, {dt_cpu:.1f} s"},
        "e2e": {"value": flops / (r["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": r["e2e_ms"]},
    }
    print(json.dumps(line))


# ------------------------------------------------------------- profiling --

def profile_steps(w, n):
    """`n` forward + backward steps of one resident input set, four kernel
    launches each (six with a block mask; two forward-only launches for FP8
    inputs or a decode step), then a status check."""
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if w.decode_n_q:   # decode steps: split-KV kernel + merge per step
        inp = workloads.make_inputs(w)
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        lens = inp["key_lens"].to(dev)
        for _ in range(n):
            ea.attention_decode(q, k, v, lens, scale=inp["scale"], causal=w.causal)
        torch.cuda.synchronize(dev)
        ea.check()
        print(f"profile-steps: {n} steps of {w.name} done")
        return
    if w.fwd_only:   # forward only: one attn_fwd call per step
        inp = workloads.make_inputs(w)
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        for _ in range(n):
            ea.attention_fwd(q, k, v, **_fwd_kw(w, inp, dev))
        torch.cuda.synchronize(dev)
        ea.check()
        print(f"profile-steps: {n} steps of {w.name} done")
        return
    step = Step(ea, workloads.make_inputs(w), dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(n):
        step.run(stream)
    torch.cuda.synchronize(dev)
    ea.check(step.ws, dev)
    print(f"profile-steps: {n} steps of {w.name} done")


# -------------------------------------------------------------------- main --

def parse_overrides(items):
    """FIELD=VALUE strings -> a dict of workload fields (ints where they parse)."""
    out = {}
    for item in items:
        key, sep, val = item.partition("=")
        if not sep or key not in workloads.Workload.__dataclass_fields__:
            raise SystemExit(f"--set wants FIELD=VALUE with a workload field, got {item!r}")
        try:
            out[key] = int(val)
        except ValueError:
            try:
                out[key] = float(val)
            except ValueError:
                out[key] = val
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle timing")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many untimed steps of one input set and exit (a short, "
                         "fixed launch sequence for ncu captures; no oracle, no JSON line)")
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                    help="replace a field of the workload, e.g. --set H=2 (repeatable)")
    args = ap.parse_args()
    w = workloads.get(args.workload, **parse_overrides(args.set))

    if args.profile_steps > 0:
        profile_steps(w, args.profile_steps)
        return
    if w.fwd_only and not w.decode_n_q:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference",
                              "unavailable": "the reference arm times the bf16 training step"}))
        elif int(os.environ.get("RANK", "0")) == 0:
            run_fwd_only(args, w)
        return
    if w.decode_n_q:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference",
                              "unavailable": "the reference arm times the training step"}))
        elif int(os.environ.get("RANK", "0")) == 0:
            run_decode(args, w)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return

    # the oracle is timed before any GPU work so that its BLAS threads start
    # in a process that has not touched CUDA yet
    cpu = None
    if rank == 0 and world == 1:
        inp_cpu = workloads.make_inputs(w)
        units = oracle_units(w)
        f, dt, n = oracle_sample(w, inp_cpu, units, oracle_inputs(inp_cpu), args.cpu_budget)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOPS", "cores": _blas_threads(),
               "kind": "oracle",
               "sample": f"{n} of {len(units)} {oracle_unit_name(w)} of {w.name} (seeded "
                         f"random order), fp64 numpy fwd+bwd, {dt:.1f} s"}
        del inp_cpu

    dist = None
    if world > 1:
        import torch.distributed as td
        td.init_process_group("nccl")
        dist = td
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if dist is not None:
        dist.barrier()

    r = measure_device(ea, w, dev, args.steps, args.warmup, dist)
    line = headline_line(w, r, args.steps, args.warmup, world)
    if cpu is not None:
        line["cpu_baseline"] = cpu
    line["e2e"] = measure_e2e(ea, w, dev, max(3, min(args.steps, 100)), 3)
    if not args.no_secondary and world == 1:
        sec = []
        for name in SECONDARY:
            if name == w.name:
                continue
            ws = workloads.get(name)
            rs = measure_device(ea, ws, dev, max(10, args.steps // 10), 5, None)
            entry = {"workload": describe(ws)}
            entry.update(workload_result(ws, rs))
            entry["fwd_bwd_tflops"] = entry.pop("value")
            sec.append(entry)
        line["secondary"] = sec
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
