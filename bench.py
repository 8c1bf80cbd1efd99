"""Benchmark of one paged-decode step on GB300.

A step is one pass of the whole hot path over one batch: the cache write of one
new token per sequence, the copy-on-write block copies of the workload (if it
has any) and paged decode attention over the grown contexts (split-K partition
kernel + merge kernel).  The default workload is the Llama-7B-shaped decode
layer (32 heads MHA, head_dim 128, bf16, batch 64, context lengths uniform in
[128, 2048], block tables drawn from a shuffled pool 1.1x the blocks in use).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line.  Under torchrun every rank runs its own copy of the
workload (weak scaling, no collective on the data path); rank 0 prints.
``--impl reference`` times the fp64 oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention tokens/s and KV GB/s (% of GB300 HBM peak), 1 GPU"
PREFILL_METRIC = ("chunked paged prefill attention query tokens/s and TFLOP/s "
                  "(% of GB300 bf16 tensor peak), 1 GPU")
NOMINAL_HBM_GBS = 7900.0     # GB300 HBM3e nominal
FALLBACK_HBM_GBS = 6800.0    # earlier GB300 measurement, used only without MEASURED_PEAKS.json
L2_BYTES = 129 * 10**6


# ---------------------------------------------------------------------------
# Byte accounting ("KV cache: la memoria de trabajo que sostiene la inferencia
# LLM", section "El precio: cuánto pesa la mochila": K and V of every token,
# 2 * layers * kv_heads * head_dim * bytes per element)
# ---------------------------------------------------------------------------
def kv_bytes_per_token(n_layers, n_kv_heads, head_dim, bytes_per_elem=2) -> int:
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_elem


def _window_range(L, window):
    """Positions [start, L) a decode attends to (all of them when window is 0)."""
    return (L - window if (window and L > window) else 0), L


def decode_algorithmic_bytes(wl: W.Workload, lens=None, kv_elem_bytes=None, window=0) -> dict:
    """Least bytes one decode call moves: K/V of every attended context token, Q, O,
    the table entries of the attended blocks, lengths."""
    lens = wl.step_context_lens if lens is None else np.asarray(lens)
    lens = lens.astype(np.int64)
    e = wl.elem_bytes
    rows = sum(L - _window_range(int(L), window)[0] for L in lens)
    blocks = sum(-(-int(L) // 16) - _window_range(int(L), window)[0] // 16 for L in lens)
    kv = int(rows) * kv_bytes_per_token(1, wl.num_kv_heads, wl.head_dim, kv_elem_bytes or e)
    q = wl.num_seqs * wl.num_q_heads * wl.head_dim * e
    tables = int(blocks) * 4 + 4 * wl.num_seqs
    return {"kv": kv, "q": q, "o": q, "tables": tables, "total": kv + 2 * q + tables}


def unique_kv_bytes(wl: W.Workload, lens=None, kv_elem_bytes=None, window=0) -> int:
    """K/V bytes of distinct (block, slot) pairs read: shared prefix blocks count once."""
    lens = wl.step_context_lens if lens is None else np.asarray(lens)
    slots = []
    for b in range(wl.num_seqs):
        start, L = _window_range(int(lens[b]), window)
        t = np.arange(start, L, dtype=np.int64)
        slots.append(wl.block_tables[b, t // 16].astype(np.int64) * 16 + t % 16)
    n = np.unique(np.concatenate(slots)).size if slots else 0
    return n * kv_bytes_per_token(1, wl.num_kv_heads, wl.head_dim,
                                          kv_elem_bytes or wl.elem_bytes)


def step_write_bytes(wl: W.Workload) -> int:
    row = wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    cow = int(wl.cow_pairs.shape[0]) * wl.num_kv_heads * 16 * wl.head_dim * wl.elem_bytes * 2
    return 2 * 2 * wl.num_seqs * row + 2 * cow


# ---------------------------------------------------------------------------
# Distributed plumbing (weak scaling: no collective on the data path)
# ---------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# Peaks, clocks, traffic
# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """SM clock and throttle-reason samples taken while the timed region runs.

    Reads NVML (the library nvidia-smi uses) every 20 ms from a background
    thread.  Read-only: no clock or other GPU setting is changed.
    """
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int, pci_bus_id: str | None = None, period_s: float = 0.02):
        import threading
        self.samples = []
        self.recording = False
        self._stop = threading.Event()
        self._nvml = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            ok = False
            if pci_bus_id:
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index),
                                                           ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self._nvml, self._h, self._ct = nv, h, ctypes
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self.max_mhz = float(mx.value)
        except Exception:
            self._nvml = None
        self._thread = threading.Thread(target=self._run, args=(period_s,), daemon=True)
        self._thread.start()

    def _read(self):
        ct, nv = self._ct, self._nvml
        clk = ct.c_uint()
        nv.nvmlDeviceGetClockInfo(self._h, 1, ct.byref(clk))
        reasons = ct.c_ulonglong()
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        fn(self._h, ct.byref(reasons))
        return float(clk.value), int(reasons.value)

    def _run(self, period_s):
        if self._nvml is None:
            return
        while not self._stop.is_set():
            if self.recording:
                try:
                    self.samples.append(self._read())
                except Exception:
                    pass
            self._stop.wait(period_s)

    def start(self):
        self.recording = True

    def stop(self):
        if self._nvml is not None and not self.samples:
            try:
                self.samples.append(self._read())       # at least one reading at the end
            except Exception:
                pass
        self.recording = False
        self._stop.set()
        self._thread.join(timeout=2)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "unavailable"}
        reasons = set()
        for _, bits in self.samples:
            for bit, name in self.REASONS.items():
                if bits & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "NVML, 20 ms period"}


def pci_bus_id(dev):
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        return "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        return None


def _code_only(src: str) -> str:
    """C/CUDA source without comments, blank lines and indentation, so that an
    edit of comments alone keeps the hash (the compiled kernel is the same)."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.strip() for line in src.splitlines() if line.strip())


DECODE_SOURCES = ("pa_decode.cu", "pa_device.cuh", "pa_internal.h")
# the shared-prefix cascade also runs the tensor-core kernel in prefix mode
CASCADE_SOURCES = DECODE_SOURCES + ("pa_prefill.cu", "pa_tc.cuh")


def kernel_source_hash(files=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_100_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_key(workload: str, kv_dtype: str = "bf16", window: int = 0, partition_size: int = 0,
                decode: str = "auto") -> str:
    """Key of a decode configuration in the traffic record: the workload name
    alone for its default line (bf16 pools, whole context, library-chosen
    partition), else every setting that changes the kernel or its bytes."""
    if kv_dtype == "bf16" and window == 0 and partition_size == 0 and decode == "auto":
        return workload
    return f"{workload}|{kv_dtype}|window={window}|partition={partition_size}|decode={decode}"


def measured_traffic(key: str):
    """DRAM bytes per decode call from the committed ncu summary for exactly
    this configuration, if it still describes the current kernel source (else
    None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        entry = rec[key]
        if entry.get("kernel_source_hash") != kernel_source_hash(tuple(entry.get("sources", DECODE_SOURCES))):
            return None
        return float(entry["dram_bytes_per_call"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class StepOps:
    """The library calls of one step for bf16 (or f32) pools or FP8 pools."""

    def __init__(self, pkv, wl, kc, vc, ks, vs, P, ws, n_prefix=0, window=0):
        self.pkv, self.wl, self.kc, self.vc, self.ks, self.vs = pkv, wl, kc, vc, ks, vs
        self.P, self.ws = P, ws
        self.fp8 = ks is not None
        self.n_prefix = n_prefix          # > 0: shared-prefix (cascade) decode
        self.window = window              # > 0: sliding-window decode

    def write(self, kn, vn, slots):
        if self.fp8:
            self.pkv.cache_write_fp8(self.kc, self.vc, kn, vn, slots, self.ks, self.vs)
        else:
            self.pkv.cache_write(self.kc, self.vc, kn, vn, slots)

    def decode(self, q, bt, lens, out):
        if self.window:
            self.pkv.decode_sliding_window(q, self.kc, self.vc, bt, lens, self.window,
                                           self.wl.scale, k_scales=self.ks, v_scales=self.vs,
                                           out=out, partition_size=self.P, workspace=self.ws)
        elif self.n_prefix and self.fp8:
            self.pkv.decode_shared_prefix_fp8(q, self.kc, self.vc, self.ks, self.vs, bt, lens,
                                              self.n_prefix, self.wl.scale, out=out,
                                              partition_size=self.P, workspace=self.ws)
        elif self.n_prefix:
            self.pkv.decode_shared_prefix(q, self.kc, self.vc, bt, lens, self.n_prefix,
                                          self.wl.scale, out=out, partition_size=self.P,
                                          workspace=self.ws)
        elif self.fp8:
            self.pkv.decode_fp8(q, self.kc, self.vc, self.ks, self.vs, bt, lens, self.wl.scale,
                                out=out, partition_size=self.P, workspace=self.ws)
        else:
            self.pkv.decode(q, self.kc, self.vc, bt, lens, self.wl.scale, out=out,
                            partition_size=self.P, workspace=self.ws)

def rotation_copies(unique_kv_bytes: int) -> int:
    """Pool copies used in turn, step after step, so that no step finds K/V of the
    step before it in L2: between two reads of one copy at least twice the L2
    size of other K/V streams through.  K/V of four times the L2 size or more
    (and parity-sized pools too small to measure) need no rotation."""
    if unique_kv_bytes >= 4 * L2_BYTES or unique_kv_bytes < 16 * 10**6:
        return 1
    return min(8, 1 + -(-2 * L2_BYTES // unique_kv_bytes))


def l2_note(unique_kv: int, copies: int) -> str:
    if copies > 1:
        return ("%.0f MB of distinct K/V per step vs 129 MB L2: %d pool copies used in turn, "
                "%.0f MB of other K/V between two reads of a copy"
                % (unique_kv / 1e6, copies, (copies - 1) * unique_kv / 1e6))
    if unique_kv >= 4 * L2_BYTES:
        return "inputs larger than L2: %.2f GB of distinct K/V per step vs 129 MB L2" % (unique_kv / 1e9)
    return ("%.2f MB of distinct K/V per step fits in the 129 MB L2 (a parity-sized "
            "configuration; its timing is not an HBM figure)" % (unique_kv / 1e6))


def cpu_model() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine() or "unknown"


def measure_decode(pkv, dev, stream, args, workload, kv_dtype="bf16", window=0, decode="auto",
                   partition_size=0, soak_s=0.5, rank=0, world=1, sample_clocks=True):
    """One decode configuration: W warm-up steps, K timed steps back to back, K
    steps with every decode call bracketed by events, a loop of the same step for
    at least ``soak_s`` seconds (NVML clock samples over it and the timed steps),
    and the end-to-end run through the public API with host inputs.  Returns the
    measurements and the workload description."""
    import torch
    wl = W.make_workload(workload, seed=args.seed)
    fp8 = kv_dtype == "fp8"
    if fp8:
        q, kc, vc, kn, vn, ks, vs = W.fp8_device_values(wl, dev, seed=args.seed + 17 + rank)
    else:
        q, kc, vc, kn, vn = W.device_values(wl, dev, seed=args.seed + 17 + rank)
        ks = vs = None
    kv_e = 1 if fp8 else None
    logical = decode_algorithmic_bytes(wl, kv_elem_bytes=kv_e, window=window)
    unique_kv = unique_kv_bytes(wl, kv_elem_bytes=kv_e, window=window)
    copies = rotation_copies(unique_kv)
    pools = [(kc, vc)] + [(kc.clone(), vc.clone()) for _ in range(copies - 1)]
    bt = torch.from_numpy(wl.block_tables).to(dev)
    lens = torch.from_numpy(wl.step_context_lens).to(dev)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    pairs = torch.from_numpy(wl.cow_pairs).to(dev)
    has_cow = wl.cow_pairs.shape[0] > 0
    kvd = "fp8" if fp8 else wl.dtype
    P = partition_size or wl.partition_size or pkv.decode_partition_size(
        wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.max_blocks, kvd)
    out = torch.empty_like(q)
    ws = torch.empty(max(pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads,
                                                    wl.head_dim, wl.max_blocks, P, kvd), 16),
                     dtype=torch.uint8, device=dev)
    n_prefix = 0
    if window:
        P = partition_size
        ws = torch.empty(max(pkv.lib().pa_decode_sliding_window_workspace_bytes(
            wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.max_blocks, 16, window,
            P, 2 if fp8 else (1 if wl.dtype == "bf16" else 0)), 16), dtype=torch.uint8, device=dev)
    elif decode != "plain":
        n_prefix = pkv.shared_prefix_blocks(wl.block_tables)
        if decode == "auto" and n_prefix < 4:
            n_prefix = 0
    if n_prefix:
        P = partition_size or wl.partition_size
        ws_bytes = (pkv.lib().pa_decode_shared_prefix_fp8_workspace_bytes if fp8 else
                    pkv.lib().pa_decode_shared_prefix_workspace_bytes)
        ws = torch.empty(max(ws_bytes(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                      wl.max_blocks, n_prefix, P), 16),
                         dtype=torch.uint8, device=dev)
    ops = [StepOps(pkv, wl, k_, v_, ks, vs, P, ws, n_prefix, window) for k_, v_ in pools]
    state = {"i": 0}

    def step_pre(o, kn_=kn, vn_=vn, slots_=slots, pairs_=pairs):
        o.write(kn_, vn_, slots_)
        if has_cow:
            pkv.block_copy(o.kc, o.vc, pairs_)

    def step(ev_pre=None, ev_post=None, q_=q, kn_=kn, vn_=vn, slots_=slots, pairs_=pairs, bt_=bt,
             lens_=lens, out_=out):
        o = ops[state["i"] % copies]
        state["i"] += 1
        step_pre(o, kn_, vn_, slots_, pairs_)
        if ev_pre is not None:
            ev_pre.record(stream)
        o.decode(q_, bt_, lens_, out_)
        if ev_post is not None:
            ev_post.record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # With --graphs the device-timed runs replay CUDA graphs of the step's
    # library calls, one set per pool copy: the whole step (write,
    # copy-on-write, decode), and its write/copy and its decode call apart (for
    # the per-call events).  The kernels, their order and their launch
    # attributes are the captured calls'; replaying them takes the host's
    # per-call work (argument checks, tensor-map encoding, one launch per
    # kernel) out of the GPU's way, as a serving loop that replays a captured
    # decode step does, but each replay starts only when the one before has
    # ended.  The end-to-end run below calls the public API directly.
    timed_step = step
    kernels_per_step = None
    if args.graphs:
        graphs = []
        for o in ops:
            gs, gp, gd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            n0 = pkv.launch_count()
            with torch.cuda.graph(gs, capture_error_mode="thread_local"):
                step_pre(o)
                o.decode(q, bt, lens, out)
            kernels_per_step = pkv.launch_count() - n0
            with torch.cuda.graph(gp, capture_error_mode="thread_local"):
                step_pre(o)
            with torch.cuda.graph(gd, capture_error_mode="thread_local"):
                o.decode(q, bt, lens, out)
            graphs.append((gs, gp, gd))

        def graph_step(ev_pre=None, ev_post=None):
            gs, gp, gd = graphs[state["i"] % copies]
            state["i"] += 1
            if ev_pre is None:
                gs.replay()
            else:
                gp.replay()
                ev_pre.record(stream)
                gd.replay()
                ev_post.record(stream)

        timed_step = graph_step
        for _ in range(max(3, args.warmup)):
            timed_step()
        torch.cuda.synchronize(dev)
    # a first estimate of the step time sizes the clock-sampling loop
    t0 = time.perf_counter()
    for _ in range(3):
        timed_step()
    torch.cuda.synchronize(dev)
    est = max((time.perf_counter() - t0) / 3, 1e-5)
    n_soak = int(max(1, soak_s / est)) if soak_s > 0 else 0

    K = args.steps
    sampler = ClockSampler(dev.index or 0, pci_bus_id(dev)) if (rank == 0 and sample_clocks) else None
    barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
    # a loop of the same step right before the timed region: the GPU is under
    # this load when the timed steps begin, and the clock samples cover both
    es0 = torch.cuda.Event(enable_timing=True)
    es1 = torch.cuda.Event(enable_timing=True)
    es0.record(stream)
    for _ in range(n_soak):
        timed_step()
    es1.record(stream)
    launches0 = pkv.launch_count()
    # timed region: K whole steps back to back
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        timed_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    barrier()
    # kernels of the library launched in the timed region: counted by the
    # library's own launch counter, or (graphs) as its launches per captured
    # step times the replays
    launches = (kernels_per_step * K if kernels_per_step is not None
                else pkv.launch_count() - launches0)
    # K steps again, each decode call bracketed by events on the launching
    # stream (the roofline's per-call duration)
    pre = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    post = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for i in range(K):
        timed_step(pre[i], post[i])
    e3.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), dev)
    decode_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(pre, post)) / K, dev)
    ms_step_with_events = max_over_ranks(e2.elapsed_time(e3), dev) / K
    soak_ms = es0.elapsed_time(es1) / n_soak if n_soak else None
    ms_per_step = ms_total / K

    e2e = run_e2e(args, pkv, wl, q, kn, vn, dev, stream, step, out)
    res = {
        "wl": wl, "fp8": fp8, "kv_dtype": kvd, "window": window, "n_prefix": n_prefix, "P": P,
        "ms_per_step": ms_per_step, "decode_ms": decode_ms,
        "ms_per_step_with_call_events": ms_step_with_events,
        "soak": {"steps": n_soak, "ms_per_step": soak_ms,
                 "s": None if soak_ms is None else n_soak * soak_ms / 1e3},
        "launches": int(launches), "clocks": clocks, "e2e": e2e,
        "launch_mode": ("CUDA graph replay of the step's captured library calls "
                        "(%d kernels per step)" % kernels_per_step) if kernels_per_step is not None
                       else "direct library calls",
        "logical": logical, "unique_kv": unique_kv, "copies": copies,
        "q": q, "kc": kc, "vc": vc, "ks": ks, "vs": vs,
    }
    return res


def decode_method(res) -> str:
    window, n_prefix, fp8 = res["window"], res["n_prefix"], res["fp8"]
    if window:
        return f"sliding window of the last {window} positions"
    if n_prefix:
        return (f"shared-prefix cascade ({n_prefix} shared blocks read once per KV head; " +
                ("widen, " if fp8 else "") + "prefix, suffix and merge kernels)")
    return "paged decode"


def decode_kernel_desc(res) -> str:
    if res["window"]:
        return ("pa_decode_sliding_window call (partition kernel, plus the merge kernel when a "
                "window spans several partitions)")
    if res["n_prefix"]:
        return ("pa_decode_shared_prefix_fp8 call (widen + prefix + suffix + merge kernels)"
                if res["fp8"] else "pa_decode_shared_prefix call (prefix + suffix + merge kernels)")
    return ("pa_decode call (partition kernel, plus the merge kernel when a sequence spans "
            "several partitions)")


def partition_label(res):
    """The split-K partition size the run used, or who chose it."""
    if res["P"]:
        return res["P"]
    if res["window"]:
        return "library choice per window"
    return "library choice (shared-prefix suffix)" if res["n_prefix"] else "library choice"


def decode_summary(res, args, workload, decode, partition_size, world) -> dict:
    """The figures of one decode configuration (the per-configuration record)."""
    wl = res["wl"]
    hbm_bytes = res["logical"]["total"] - res["logical"]["kv"] + res["unique_kv"]
    peak, peak_kind = load_peaks()
    decode_ms = res["decode_ms"]
    achieved = hbm_bytes / (decode_ms * 1e-3) / 1e9
    kvd_arg = "fp8" if res["fp8"] else "bf16"
    traffic = measured_traffic(traffic_key(workload, kvd_arg, res["window"], partition_size, decode))
    clocks = res["clocks"]
    mhz = clocks.get("sm_mhz") if clocks else None
    out = {
        "workload": workload_config(wl, world, kvd_arg, res["window"], res["unique_kv"])["workload"],
        "decode_method": decode_method(res),
        "partition_size": partition_label(res),
        "ms_per_step": res["ms_per_step"],
        "decode_ms": decode_ms,
        "tokens_per_s": wl.num_seqs * world / (res["ms_per_step"] * 1e-3),
        "context_tokens_per_s": float(wl.step_context_lens.sum()) * world / (res["ms_per_step"] * 1e-3),
        "kv_gbs": res["unique_kv"] / (decode_ms * 1e-3) / 1e9,
        "logical_kv_gbs": res["logical"]["kv"] / (decode_ms * 1e-3) / 1e9,
        "roofline": {
            "kernel": decode_kernel_desc(res), "bound": "hbm", "achieved": achieved, "peak": peak,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6800 GB/s",
            "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
            "algorithmic_bytes_per_call": hbm_bytes,
            "bytes_rule": "K/V of every distinct (block, slot) read + Q + O + table entries + "
                          "context lengths",
        },
        "hbm_frac_of_nominal_7900": achieved / NOMINAL_HBM_GBS,
        "sustained": res["soak"],
        "clocks": clocks,
        "decode_kcycles_at_median_clock": (decode_ms * mhz) if mhz else None,
        "gpu_launches_per_step": res["launches"] / max(args.steps, 1),
        "launch_mode": res["launch_mode"],
        "e2e": res["e2e"],
        "l2": l2_note(res["unique_kv"], res["copies"]),
    }
    if traffic is not None:
        out["roofline"]["traffic_over_algorithmic"] = traffic / hbm_bytes
    return out


# the configurations of the per-configuration record (one GPU run): every
# decode workload, the FP8 pools, the sliding windows, and the plain paged
# decode of the shared-prefix mix next to its cascade
PER_CONFIG = [
    dict(workload="tiny"),
    dict(workload="llama7b_mha"),
    dict(workload="llama70b_gqa"),
    dict(workload="long_splitk"),
    dict(workload="shared_prefix"),
    dict(workload="shared_prefix", decode="plain"),
    dict(workload="llama7b_mha", kv_dtype="fp8"),
    dict(workload="llama70b_gqa", kv_dtype="fp8"),
    dict(workload="long_splitk", kv_dtype="fp8"),
    dict(workload="shared_prefix", kv_dtype="fp8"),
    dict(workload="long_splitk", window=4096),
    dict(workload="llama70b_gqa", window=1024),
    dict(workload="llama70b_gqa", window=1024, kv_dtype="fp8"),
]
PER_CONFIG_PREFILL = ["prefill_llama70b_chunked", "prefill_llama7b"]


def per_config_key(c) -> str:
    k = c["workload"]
    if c.get("kv_dtype", "bf16") == "fp8":
        k += "+fp8_kv"
    if c.get("window"):
        k += f"+window{c['window']}"
    if c.get("decode", "auto") != "auto":
        k += f"+{c['decode']}"
    return k


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        init_dist("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    from paged_kv_cache_100_gb300.build import build
    if rank == 0 or world == 1:
        build()
    barrier()
    import paged_kv_cache_100_gb300 as pkv
    stream = torch.cuda.current_stream(dev)

    res = measure_decode(pkv, dev, stream, args, args.workload, args.kv_dtype, args.window,
                         args.decode, args.partition_size, soak_s=args.soak_seconds, rank=rank,
                         world=world)
    summ = decode_summary(res, args, args.workload, args.decode, args.partition_size, world)
    wl = res["wl"]
    line = None
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": summ["tokens_per_s"],
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": res["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "fp8_e4m3 K/V, bf16 Q/O" if res["fp8"] else wl.dtype,
            "data": "synthetic (seeded; N(0, %g) values, shuffled block pool)" % wl.value_std,
            "config": workload_config(wl, world, args.kv_dtype, args.window, res["unique_kv"]),
            "partition_size_used": partition_label(res),
            "decode_ms": res["decode_ms"],
            "ms_per_step_with_call_events": res["ms_per_step_with_call_events"],
            "kv_gbs": summ["kv_gbs"],
            "logical_kv_gbs": summ["logical_kv_gbs"],
            "context_tokens_per_s": summ["context_tokens_per_s"],
            "hbm_frac_of_measured": summ["roofline"]["frac"]
            if summ["roofline"]["peak_source"].startswith("measured") else None,
            "hbm_frac_of_nominal_7900": summ["hbm_frac_of_nominal_7900"],
            "decode_method": summ["decode_method"],
            "roofline": summ["roofline"],
            "gpu_launches": res["launches"],
            "launch_mode": res["launch_mode"],
            "clocks": res["clocks"],
            "clocks_window": "NVML every 20 ms over a loop of the same step (%d steps, %.2f s) "
                             "that ends where the timed region begins, and the timed region"
                             % (res["soak"]["steps"], res["soak"]["s"] or 0.0),
            "sustained": res["soak"],
            "decode_kcycles_at_median_clock": summ["decode_kcycles_at_median_clock"],
            "e2e": res["e2e"],
        }
        if res["unique_kv"] != res["logical"]["kv"]:
            line["logical_kv_bytes"] = res["logical"]["kv"]
            line["unique_kv_bytes"] = res["unique_kv"]
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(args, wl, res["q"], res["kc"], res["vc"],
                                                budget_s=args.cpu_seconds, ks=res["ks"],
                                                vs=res["vs"], window=args.window)
    del res
    torch.cuda.empty_cache()
    if world == 1 and not args.no_per_config:
        per = {}
        for c in PER_CONFIG:
            r = measure_decode(pkv, dev, stream, args, c["workload"], c.get("kv_dtype", "bf16"),
                               c.get("window", 0), c.get("decode", "auto"), 0,
                               soak_s=args.soak_seconds)
            per[per_config_key(c)] = decode_summary(r, args, c["workload"], c.get("decode", "auto"),
                                                    0, world)
            del r
            torch.cuda.empty_cache()
        for name in PER_CONFIG_PREFILL:
            pa = argparse.Namespace(**vars(args))
            pa.workload, pa.window = name, 0
            per[name] = prefill_summary(measure_prefill(pkv, dev, stream, pa, soak_s=args.soak_seconds),
                                        world)
            torch.cuda.empty_cache()
        line["per_config"] = per
    return line


def workload_config(wl, world, kv_dtype=None, window=0, unique_kv=None):
    """The workload as both arms describe it (nothing the library chooses)."""
    lens = wl.step_context_lens
    kv_e = 1 if kv_dtype == "fp8" else None
    if unique_kv is None:
        unique_kv = unique_kv_bytes(wl, kv_elem_bytes=kv_e, window=window)
    copies = rotation_copies(unique_kv)
    cfg = {
        "workload": wl.name + ("+fp8_kv" if kv_dtype == "fp8" else "") +
                    (f"+window{window}" if window else ""),
        "kv_dtype": kv_dtype or wl.dtype,
        "num_seqs_per_gpu": wl.num_seqs,
        "global_batch": wl.num_seqs * world,
        "num_q_heads": wl.num_q_heads,
        "num_kv_heads": wl.num_kv_heads,
        "head_dim": wl.head_dim,
        "block_size": wl.block_size,
        "context_lens_min_max_mean": [int(lens.min()), int(lens.max()), float(lens.mean())],
        "num_blocks": wl.num_blocks,
        "partition_size": wl.partition_size or "library choice",
        "cow_pairs_per_step": int(wl.cow_pairs.shape[0]),
        "parallelism": f"weak scaling, {world} independent replica(s)",
        "l2": l2_note(unique_kv, copies),
    }
    if window:
        cfg["window"] = window
    return cfg


class PackedInputs:
    """A step's host inputs packed into one pinned buffer (256-byte aligned
    pieces) with a device twin: one host-to-device copy per step instead of one
    per tensor.  `dev[name]` are views of the device buffer with each input's
    dtype and shape."""

    def __init__(self, tensors: dict, dev):
        import torch
        offs, off = {}, 0
        for k, t in tensors.items():
            offs[k] = off
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        self.nbytes = off
        self.host = torch.empty(max(off, 1), dtype=torch.uint8).pin_memory()
        self.device = torch.empty(max(off, 1), dtype=torch.uint8, device=dev)
        self.dev = {}
        for k, t in tensors.items():
            n = t.numel() * t.element_size()
            self.host[offs[k]:offs[k] + n].copy_(t.contiguous().view(-1).view(torch.uint8))
            self.dev[k] = self.device[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
        self.used = sum(t.numel() * t.element_size() for t in tensors.values())

    def upload(self):
        self.device.copy_(self.host, non_blocking=True)


def _cudart():
    """The CUDA runtime library torch has loaded (for stream-ordered copies
    without switching torch's current stream), or None."""
    import ctypes
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            lib = ctypes.CDLL(name)
        except OSError:
            continue
        fn = lib.cudaMemcpyAsync
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                       ctypes.c_void_p]
        return lib
    return None


class E2ELoop:
    """Steps through the public API with host inputs, every step copying its own
    inputs from pinned host memory (one packed copy) and its output back.

    The uploads and the read-backs run on two streams of their own, with two
    device input buffers and two output buffers used in turn: step i + 1's
    inputs go up and step i - 1's output comes back while step i's kernels run,
    as a serving loop overlaps its transfers with compute.  (On one copy stream
    the next upload would queue behind the read-back that waits for the current
    step.)  Events order each copy against the step that uses its buffer.  The
    timed region starts before the first upload and ends after the last output
    has reached host memory."""

    H2D, D2H = 1, 2   # cudaMemcpyKind

    def __init__(self, inputs: dict, out, dev, stream, run_step):
        import torch
        self.torch, self.stream, self.run_step = torch, stream, run_step
        self.up = torch.cuda.Stream(dev)
        self.down = torch.cuda.Stream(dev)
        self.bufs = [PackedInputs(inputs, dev) for _ in range(2)]
        self.outs = [out, torch.empty_like(out)]
        self.hosts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        self.uploaded = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.read_back = [torch.cuda.Event() for _ in range(2)]
        self.i = 0
        self.h2d = self.bufs[0].nbytes
        self.d2h = out.numel() * out.element_size()
        self.rt = _cudart()

    def _copy(self, dst, src, nbytes, kind, stream):
        if self.rt is not None:
            rc = self.rt.cudaMemcpyAsync(dst.data_ptr(), src.data_ptr(), nbytes, kind,
                                         stream.cuda_stream)
            if rc != 0:
                raise RuntimeError(f"cudaMemcpyAsync failed ({rc})")
        else:
            with self.torch.cuda.stream(stream):
                dst.copy_(src, non_blocking=True)

    def step(self):
        b = self.i & 1
        self.i += 1
        buf, up, down = self.bufs[b], self.up, self.down
        up.wait_event(self.computed[b])          # the step that last read buffer b has run
        self._copy(buf.device, buf.host, buf.nbytes, self.H2D, up)
        self.uploaded[b].record(up)
        self.stream.wait_event(self.uploaded[b])
        self.stream.wait_event(self.read_back[b])   # output b of two steps back is home
        self.run_step(buf.dev, self.outs[b])
        self.computed[b].record(self.stream)
        down.wait_event(self.computed[b])
        self._copy(self.hosts[b], self.outs[b], self.d2h, self.D2H, down)
        self.read_back[b].record(down)

    def time(self, K: int, dev) -> float:
        """Milliseconds per step over K steps (after three untimed ones)."""
        torch = self.torch
        for _ in range(3):
            self.step()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(self.stream)
        self.up.wait_event(e0)
        self.down.wait_event(e0)
        for _ in range(K):
            self.step()
        for ev in self.read_back:
            self.stream.wait_event(ev)
        e1.record(self.stream)
        torch.cuda.synchronize(dev)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1) / K, dev)


E2E_NOTE = ("public API with host inputs: every step's inputs copied from pinned host "
            "memory (one packed copy) and its output copied back, on an upload and a "
            "read-back stream with two input and two output buffers in turn, overlapping the "
            "neighbouring steps' kernels")


def run_e2e(args, pkv, wl, q, kn, vn, dev, stream, step, out):
    """Same step through the public API with host inputs (query, new K/V rows,
    slots, tables, lengths, copy pairs) uploaded and the output read back every
    step, inside the timed region."""
    import torch
    has_cow = wl.cow_pairs.shape[0] > 0
    inputs = {
        "q": q.cpu(), "kn": kn.cpu(), "vn": vn.cpu(),
        "slots": torch.from_numpy(wl.slot_mapping),
        "bt": torch.from_numpy(wl.block_tables),
        "lens": torch.from_numpy(wl.step_context_lens),
    }
    if has_cow:
        inputs["pairs"] = torch.from_numpy(wl.cow_pairs)

    def run_step(d, o):
        step(q_=d["q"], kn_=d["kn"], vn_=d["vn"], slots_=d["slots"], pairs_=d.get("pairs"),
             bt_=d["bt"], lens_=d["lens"], out_=o)

    loop = E2ELoop(inputs, out, dev, stream, run_step)
    K = max(1, min(args.steps, args.e2e_steps))
    ms = loop.time(K, dev)
    _, world, _ = dist_env()
    return {"value": wl.num_seqs * world / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "steps": K, "h2d_bytes_per_step": int(loop.h2d), "d2h_bytes_per_step": int(loop.d2h),
            "how": E2E_NOTE}


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on the host cores over a bounded sample
# ---------------------------------------------------------------------------
def _compact(wl, seqs, kc_host_fn):
    lens = wl.step_context_lens[seqs].astype(np.int64)
    need = -(-lens // 16)
    tabs = np.full((len(seqs), int(need.max())), -1, dtype=np.int32)
    for i, b in enumerate(seqs):
        tabs[i, :need[i]] = wl.block_tables[b, :need[i]]
    used = np.unique(tabs[tabs >= 0])
    remap = np.full(wl.num_blocks, -1, dtype=np.int64)
    remap[used] = np.arange(used.size)
    new = np.where(tabs >= 0, remap[np.maximum(tabs, 0)], -1).astype(np.int32)
    return used, new, lens.astype(np.int32)


def _bits(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def cpu_baseline(args, wl, q, kc, vc, budget_s=10.0, ks=None, vs=None, window=0):
    import torch
    import oracle
    threads = oracle.max_threads()
    rng = np.random.default_rng(3)
    n_seq = min(wl.num_seqs, 8)
    seqs = np.sort(rng.choice(wl.num_seqs, size=n_seq, replace=False))
    used, tabs, lens = _compact(wl, seqs, None)
    idx = torch.from_numpy(used.astype(np.int64)).to(kc.device)
    kch, vch = _bits(kc.index_select(0, idx)), _bits(vc.index_select(0, idx))
    qh = _bits(q[torch.from_numpy(seqs).to(q.device)])
    t0 = time.perf_counter()
    reps = 0
    scales = {} if ks is None else {"k_scales": ks.cpu().numpy(), "v_scales": vs.cpu().numpy()}
    while True:
        oracle.paged_decode(qh, kch, vch, tabs, lens, wl.scale, threads=threads, window=window,
                            **scales)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    # scale the sample's time to the whole batch by attended context tokens
    att = lambda ls: float(sum(min(int(L), window) if window else int(L) for L in ls))
    frac = att(lens) / att(wl.step_context_lens)
    t_batch = dt / reps / frac
    return {"value": wl.num_seqs / t_batch, "unit": "tokens/s", "cores": threads, "cpu": cpu_model(), "kind": "oracle",
            "sample": f"{n_seq} of {wl.num_seqs} sequences (all {wl.num_q_heads} heads, "
                      f"{int(lens.sum())} context tokens) x {reps} repetitions in {dt:.1f} s; "
                      "time scaled to the batch by context tokens"}


# ---------------------------------------------------------------------------
# Reference arm: the oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return None
    import oracle
    oracle.build()
    wl = W.make_workload(args.workload, seed=args.seed)
    threads = oracle.max_threads()
    # a bounded sample: a few sequences of the workload drawn on the host; each
    # step decodes one of them (all heads), cycling through the sample
    rng = np.random.default_rng(5)
    n_seq = min(wl.num_seqs, 8)
    seqs = np.sort(rng.choice(wl.num_seqs, size=n_seq, replace=False))
    used, tabs, lens = _compact(wl, seqs, None)
    vrng = np.random.Generator(np.random.PCG64(args.seed + 99))
    shape = (used.size, wl.num_kv_heads, 16, wl.head_dim)

    def draw(s):
        x = vrng.standard_normal(s, dtype=np.float32) * np.float32(wl.value_std)
        return W.to_bf16_bits(x) if wl.dtype == "bf16" else x

    kch, vch = draw(shape), draw(shape)
    qh = draw((n_seq, wl.num_q_heads, wl.head_dim))
    scales = {}
    if getattr(args, "kv_dtype", "bf16") == "fp8":
        s8 = W.fp8_scales(wl)
        kch = W.to_e4m3_codes(W.bf16_bits_to_f32(kch), s8)
        vch = W.to_e4m3_codes(W.bf16_bits_to_f32(vch), s8)
        scales = {"k_scales": s8, "v_scales": s8}
    for _ in range(args.warmup):
        oracle.paged_decode(qh[:1], kch, vch, tabs[:1], lens[:1], wl.scale, threads=threads,
                            window=args.window, **scales)
    steps = args.steps
    tokens = 0
    ctx = 0
    t0 = time.perf_counter()
    deadline = t0 + args.reference_seconds
    done = 0
    for i in range(steps):
        j = i % n_seq
        oracle.paged_decode(qh[j:j + 1], kch, vch, tabs[j:j + 1], lens[j:j + 1], wl.scale,
                            threads=threads, window=args.window, **scales)
        tokens += 1
        ctx += min(int(lens[j]), args.window) if args.window else int(lens[j])
        done += 1
        if time.perf_counter() > deadline:
            break
    dt = time.perf_counter() - t0
    # tokens/s of the whole batch at this rate of context tokens per second
    batch_ctx = float(sum(min(int(L), args.window) if args.window else int(L)
                          for L in wl.step_context_lens))
    value = wl.num_seqs / (batch_ctx / (ctx / dt))
    sample = (f"{done} steps, each one sequence of {n_seq} sampled ({int(lens.sum())} context "
              f"tokens in the sample), all {wl.num_q_heads} heads; rate scaled to the "
              f"{wl.num_seqs}-sequence batch by context tokens")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": done,
        "warmup": args.warmup,
        "ms_per_step": dt / max(done, 1) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": workload_config(wl, world, getattr(args, "kv_dtype", "bf16"), args.window),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "cpu": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# Chunked prefill ("PagedAttention por dentro", "Chunked prefill integrado con
# paged KV"): a step is the cache write of every chunk token's K/V followed by
# causal attention of the chunk rows over their paged contexts.
# ---------------------------------------------------------------------------
def prefill_pairs(pw, window=0) -> int:
    """(query row, attended position) pairs of one query head over the batch."""
    total = 0
    for b in range(pw.num_seqs):
        p = np.arange(int(pw.cached[b]), int(pw.cached[b] + pw.chunk[b]), dtype=np.int64)
        n = p + 1
        if window:
            n = np.minimum(n, window)
        total += int(n.sum())
    return total


def prefill_flops(pw, window=0) -> int:
    """QK^T and PV over the attended pairs: 2 * 2 * head_dim flops per pair and head."""
    return 4 * pw.head_dim * pw.num_q_heads * prefill_pairs(pw, window)


def load_tensor_peak():
    """Measured cuBLAS bf16 throughput, sustained (the prefill loop runs for seconds)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops_sustained"]), "measured sustained"
    except Exception:
        return 1700.0, "fallback sustained"


def prefill_config(pw, world, window):
    cfg = {
        "workload": pw.name + (f"+window{window}" if window else ""),
        "num_seqs_per_gpu": pw.num_seqs,
        "global_batch": pw.num_seqs * world,
        "query_tokens_per_gpu": pw.num_tokens,
        "num_q_heads": pw.num_q_heads,
        "num_kv_heads": pw.num_kv_heads,
        "head_dim": pw.head_dim,
        "block_size": pw.block_size,
        "cached_min_max_mean": [int(pw.cached.min()), int(pw.cached.max()), float(pw.cached.mean())],
        "chunk_min_max": [int(pw.chunk.min()), int(pw.chunk.max())],
        "num_blocks": pw.num_blocks,
        "parallelism": f"weak scaling, {world} independent replica(s)",
        "l2": "inputs larger than L2: %.2f GB of K/V pools vs 129 MB L2"
              % (2 * np.prod(pw.pool_shape()) * 2 / 1e9),
    }
    if window:
        cfg["window"] = window
    return cfg


def measure_prefill(pkv, dev, stream, args, soak_s=0.5, rank=0, world=1):
    """One chunked-prefill configuration, timed as measure_decode times decode."""
    import torch
    pw = W.make_prefill_workload(args.workload, seed=args.seed)
    q, kc, vc, kn, vn = W.prefill_device_values(pw, dev, seed=args.seed + 17 + rank)
    bt = torch.from_numpy(pw.block_tables).to(dev)
    lens = torch.from_numpy(pw.context_lens).to(dev)
    qs = torch.from_numpy(pw.query_start).to(dev)
    slots = torch.from_numpy(pw.slot_mapping).to(dev)
    maxq = int(pw.chunk.max())
    out = torch.empty_like(q)
    ws = torch.empty(int(pkv.lib().pa_prefill_workspace_bytes()), dtype=torch.uint8, device=dev)
    window = args.window

    def step(ev_pre=None, ev_post=None, q_=q, kn_=kn, vn_=vn, slots_=slots, bt_=bt, lens_=lens,
             qs_=qs, out_=out):
        pkv.cache_write(kc, vc, kn_, vn_, slots_)
        if ev_pre is not None:
            ev_pre.record(stream)
        pkv.prefill(q_, kc, vc, bt_, lens_, qs_, maxq, pw.scale, window=window, out=out_,
                    workspace=ws)
        if ev_post is not None:
            ev_post.record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    step()
    torch.cuda.synchronize(dev)
    est = max(time.perf_counter() - t0, 1e-5)
    n_soak = int(max(1, soak_s / est)) if soak_s > 0 else 0
    K = args.steps
    sampler = ClockSampler(dev.index or 0, pci_bus_id(dev)) if rank == 0 else None
    barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
    es0 = torch.cuda.Event(enable_timing=True)
    es1 = torch.cuda.Event(enable_timing=True)
    es0.record(stream)
    for _ in range(n_soak):
        step()
    es1.record(stream)
    launches0 = pkv.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    barrier()
    launches = pkv.launch_count() - launches0
    pre = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    post = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        step(pre[i], post[i])
    torch.cuda.synchronize(dev)
    barrier()
    ms_per_step = max_over_ranks(e0.elapsed_time(e1), dev) / K
    prefill_ms = max_over_ranks(sum(a_.elapsed_time(b_) for a_, b_ in zip(pre, post)) / K, dev)
    soak_ms = es0.elapsed_time(es1) / n_soak if n_soak else None

    # end to end: the chunk's inputs from pinned host memory and the output back,
    # every step
    inputs = {"q": q.cpu(), "kn": kn.cpu(), "vn": vn.cpu(),
              "slots": torch.from_numpy(pw.slot_mapping),
              "bt": torch.from_numpy(pw.block_tables),
              "lens": torch.from_numpy(pw.context_lens),
              "qs": torch.from_numpy(pw.query_start)}

    def run_step(d, o):
        step(q_=d["q"], kn_=d["kn"], vn_=d["vn"], slots_=d["slots"], bt_=d["bt"],
             lens_=d["lens"], qs_=d["qs"], out_=o)

    loop = E2ELoop(inputs, out, dev, stream, run_step)
    KE = max(1, min(K, args.e2e_steps))
    e2e_ms = loop.time(KE, dev)
    return {"pw": pw, "window": window, "steps": K, "ms_per_step": ms_per_step, "prefill_ms": prefill_ms,
            "soak": {"steps": n_soak, "ms_per_step": soak_ms,
                     "s": None if soak_ms is None else n_soak * soak_ms / 1e3},
            "launches": int(launches), "clocks": clocks,
            "e2e": {"value": pw.num_tokens * world / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "ms_per_step": e2e_ms, "steps": KE,
                    "h2d_bytes_per_step": int(loop.h2d), "d2h_bytes_per_step": int(loop.d2h),
                    "how": E2E_NOTE},
            "q": q, "kc": kc, "vc": vc}


def prefill_summary(res, world) -> dict:
    pw, window = res["pw"], res["window"]
    flops = prefill_flops(pw, window)
    peak, peak_kind = load_tensor_peak()
    achieved = flops / (res["prefill_ms"] * 1e-3) / 1e12
    clocks = res["clocks"]
    mhz = clocks.get("sm_mhz") if clocks else None
    return {
        "workload": prefill_config(pw, world, window)["workload"],
        "ms_per_step": res["ms_per_step"],
        "prefill_ms": res["prefill_ms"],
        "query_tokens_per_s": pw.num_tokens * world / (res["ms_per_step"] * 1e-3),
        "roofline": {
            "kernel": "pa_prefill_kernel (tcgen05 S = QK^T and O = PV, TMEM accumulators)",
            "bound": "tensor", "achieved": achieved, "peak": peak,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops_sustained)",
            "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
            "algorithmic_flops_per_call": flops,
            "flops_rule": "4 * head_dim flops per (query row, query head, attended position): "
                          "causal pairs only, masked tile halves not counted",
        },
        "sustained": res["soak"],
        "clocks": clocks,
        "prefill_kcycles_at_median_clock": (res["prefill_ms"] * mhz) if mhz else None,
        "gpu_launches_per_step": res["launches"] / max(1, res["steps"]),
        "e2e": res["e2e"],
    }


def run_prefill_gpu(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        init_dist("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    from paged_kv_cache_100_gb300.build import build
    if rank == 0 or world == 1:
        build()
    barrier()
    import paged_kv_cache_100_gb300 as pkv
    stream = torch.cuda.current_stream(dev)
    res = measure_prefill(pkv, dev, stream, args, soak_s=args.soak_seconds, rank=rank, world=world)
    if rank != 0:
        return None
    summ = prefill_summary(res, world)
    pw = res["pw"]
    line = {
        "metric": PREFILL_METRIC,
        "value": summ["query_tokens_per_s"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; N(0, %g) values, shuffled block pool)" % pw.value_std,
        "config": prefill_config(pw, world, args.window),
        "prefill_ms": res["prefill_ms"],
        "roofline": summ["roofline"],
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "sustained": res["soak"],
        "e2e": res["e2e"],
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = prefill_cpu_baseline(pw, res["q"], res["kc"], res["vc"],
                                                    args.cpu_seconds, args.window)
    return line


def _prefill_sample(pw, rows=16):
    """The last ``rows`` chunk rows of the sequence with the longest context."""
    b = int(np.argmax(pw.context_lens))
    L = int(pw.context_lens[b])
    rows = min(rows, int(pw.chunk[b]))
    r0 = int(pw.query_start[b] + pw.chunk[b]) - rows
    return b, L, rows, r0


def prefill_cpu_baseline(pw, q, kc, vc, budget_s, window):
    import torch
    import oracle
    threads = oracle.max_threads()
    b, L, rows, r0 = _prefill_sample(pw)
    need = -(-L // 16)
    used = pw.block_tables[b, :need]
    idx = torch.from_numpy(used.astype(np.int64)).to(kc.device)
    kch, vch = _bits(kc.index_select(0, idx)), _bits(vc.index_select(0, idx))
    qh = _bits(q[r0:r0 + rows])
    tab = np.arange(need, dtype=np.int32)[None]
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.paged_prefill(qh, kch, vch, tab, np.array([L], np.int32),
                             np.array([0, rows], np.int32), pw.scale, threads=threads,
                             window=window)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    pos = np.arange(L - rows, L, dtype=np.int64) + 1
    sample_pairs = int((np.minimum(pos, window) if window else pos).sum())
    t_batch = dt / reps * prefill_pairs(pw, window) / sample_pairs
    return {"value": pw.num_tokens / t_batch, "unit": "tokens/s", "cores": threads,
            "cpu": cpu_model(), "kind": "oracle",
            "sample": f"last {rows} chunk rows of the longest sequence (context {L}, all "
                      f"{pw.num_q_heads} heads) x {reps} repetitions in {dt:.1f} s; time scaled "
                      "to the batch by attended (row, position) pairs"}


def run_prefill_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return None
    import oracle
    oracle.build()
    pw = W.make_prefill_workload(args.workload, seed=args.seed)
    threads = oracle.max_threads()
    b, L, rows, r0 = _prefill_sample(pw)
    need = -(-L // 16)
    vrng = np.random.Generator(np.random.PCG64(args.seed + 99))

    def draw(shape):
        return W.to_bf16_bits(vrng.standard_normal(shape, dtype=np.float32) * np.float32(pw.value_std))

    kch = draw((need, pw.num_kv_heads, 16, pw.head_dim))
    vch = draw((need, pw.num_kv_heads, 16, pw.head_dim))
    qh = draw((rows, pw.num_q_heads, pw.head_dim))
    tab = np.arange(need, dtype=np.int32)[None]
    lens, qs = np.array([L], np.int32), np.array([0, rows], np.int32)
    for _ in range(args.warmup):
        oracle.paged_prefill(qh[:1], kch, vch, tab, np.array([L - rows + 1], np.int32),
                             np.array([0, 1], np.int32), pw.scale, threads=threads,
                             window=args.window)
    t0 = time.perf_counter()
    deadline = t0 + args.reference_seconds
    done = 0
    for _ in range(args.steps):
        oracle.paged_prefill(qh, kch, vch, tab, lens, qs, pw.scale, threads=threads,
                             window=args.window)
        done += 1
        if time.perf_counter() > deadline:
            break
    dt = time.perf_counter() - t0
    pos = np.arange(L - rows, L, dtype=np.int64) + 1
    sample_pairs = int((np.minimum(pos, args.window) if args.window else pos).sum())
    value = pw.num_tokens / (dt / done * prefill_pairs(pw, args.window) / sample_pairs)
    return {
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": done, "warmup": args.warmup,
        "ms_per_step": dt / max(done, 1) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": prefill_config(pw, world, args.window),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "cpu": cpu_model(), "kind": "oracle",
                         "sample": f"{done} steps, each the last {rows} chunk rows of the longest "
                                   f"sequence (context {L}); rate scaled to the batch by "
                                   "attended (row, position) pairs"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--op", default="decode", choices=["decode", "prefill"],
                    help="decode (default) or chunked prefill (--workload prefill_*)")
    ap.add_argument("--workload", default=None, choices=W.WORKLOADS + W.PREFILL_WORKLOADS)
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--window", type=int, default=0,
                    help="> 0: sliding-window decode over the last WINDOW positions")
    ap.add_argument("--decode", default="auto", choices=["auto", "plain", "shared-prefix"],
                    help="auto: the shared-prefix cascade when every table shares >= 4 leading "
                         "blocks, else paged decode")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="element type of the K/V pools (fp8 = E4M3 with per-head scales)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=1000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-seconds", type=float, default=0.5,
                    help="length of the loop of the same step that precedes each timed region "
                         "(the NVML clock samples cover it and the timed steps)")
    ap.add_argument("--graphs", action="store_true",
                    help="time CUDA graph replays of the step's library calls instead of the "
                         "calls themselves")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration record (every workload, FP8, windows, "
                         "prefill) that a one-GPU decode run adds to its line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.op == "prefill":
        args.workload = args.workload or "prefill_llama70b_chunked"
        if args.workload not in W.PREFILL_WORKLOADS:
            ap.error("--op prefill takes a prefill_* workload")
        line = run_prefill_reference(args) if args.impl == "reference" else run_prefill_gpu(args)
    else:
        args.workload = args.workload or "llama7b_mha"
        if args.workload not in W.WORKLOADS:
            ap.error("--op decode takes a decode workload")
        line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
