#!/usr/bin/env python
"""Benchmark of the MoE expert layer with tile-level overlapped return copy on GB300.

One step = one whole layer (route, plan, permute, SwiGLU grouped GEMM, down-projection GEMM with
per-tile flags + consumer copy, combine) over one batch of synthetic tokens already resident in
HBM. Default workload: the Mixtral-shaped layer (T=4096, d=4096, ffn=14336, E=8, top-2, R=4,
tile_M=128). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Multi-GPU: the layer does not shard in this build (R owners are logical partitions on one GPU),
so N GPUs run N independent replicas (weak scaling), timed between barriers, max over ranks.
`--impl reference` times the CPU oracle (float64, NumPy) on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from tile_level_copy_gb300 import inputs  # noqa: E402

METRIC = "MoE-layer tokens/s; grouped-GEMM % of BF16 peak; return-copy overlap %"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes per launch of the SwiGLU GEMM (dram__bytes_read.sum + dram__bytes_write.sum) from an
# ncu capture of one launch on the Mixtral-shaped layer, per (workload, CTA-pair kernel), with the
# SHA-256 of the kernel sources it was taken on: the bench reports it only while those sources are
# unchanged and the launch configuration is the captured one.
SWIGLU_TRAFFIC = {("mixtral", True): {"bytes": 1952729856 + 246886912,
                                      "sources_sha256": "cca0468f65513ffa387746cf9718df5a87d318385d6943fe19d3db1e5529f6e6"}}
KERNEL_SOURCES = ("tile_level_copy_gb300/csrc/gemm.cu", "tile_level_copy_gb300/csrc/moe_internal.cuh",
                  "tile_level_copy_gb300/csrc/copy_ring.cuh")


def captured_traffic(workload: str, pair_umma: bool):
    import hashlib
    entry = SWIGLU_TRAFFIC.get((workload, bool(pair_umma)))
    if entry is None:
        return None
    h = hashlib.sha256()
    root = os.path.dirname(os.path.abspath(__file__))
    for f in KERNEL_SOURCES:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    return entry["bytes"] if h.hexdigest() == entry["sources_sha256"] else None


# Copy configuration per workload (consumer CTAs, copy warps in the producer CTAs), the fastest
# measured on one GB300: the Mixtral-shaped layer with 4 dedicated CTAs and the skewed one with 8
# (both then run the down-projection on CTA pairs); the fine-grained layer, whose copy is five
# times longer, with the producers' copy warps and no dedicated partition.
DEFAULT_COPY = {"tiny": (4, False), "mixtral": (4, False), "skew": (8, False), "fine": (0, True)}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--consumers", type=int, default=None,
                    help="c_CTA: SMs of the consumer partition (default per workload, see DEFAULT_COPY)")
    ap.add_argument("--mgb", type=int, default=1)
    ap.add_argument("--no-tail-assist", action="store_true", help="keep finished producer CTAs out of the copy")
    ap.add_argument("--copy-warps", action=argparse.BooleanOptionalAction, default=None,
                    help="also run copy engines as extra warps in every producer CTA (consumers may then be 0; "
                         "default per workload, see DEFAULT_COPY)")
    ap.add_argument("--pair-umma", action=argparse.BooleanOptionalAction, default=True,
                    help="SwiGLU GEMM on CTA pairs (UMMA 256 x 256 over two SMs; the default, the fastest "
                         "measured on every workload)")
    ap.add_argument("--direct-tail", action=argparse.BooleanOptionalAction, default=True,
                    help="the down-projection's epilogue returns the last wave's bands itself (default); the "
                         "layer without it is timed beside in the same alternation")
    ap.add_argument("--fused-dispatch", action=argparse.BooleanOptionalAction, default=False,
                    help="copy the token rows inside the SwiGLU GEMM instead of a permute launch (the other "
                         "choice is timed beside in the same alternation)")
    ap.add_argument("--fused-gemms", action=argparse.BooleanOptionalAction, default=False,
                    help="both expert GEMMs in one launch (the other choice is timed beside in the same alternation)")
    ap.add_argument("--pdl", action=argparse.BooleanOptionalAction, default=None,
                    help="programmatic dependent launch between the layer's kernels (default: on unless the copy "
                         "warps run; the other choice is timed beside in the same alternation)")
    ap.add_argument("--alt-consumers", type=int, nargs="*", default=[],
                    help="also time these consumer partitions in the alternation")
    ap.add_argument("--tail-window", type=int, default=0,
                    help="tile hand-out positions of the direct tail (0: one wave)")
    ap.add_argument("--dma", action=argparse.BooleanOptionalAction, default=True,
                    help="also time the return copy on the copy engines (moe_forward_dma) in the eager alternation")
    ap.add_argument("--workloads", nargs="*", default=["skew", "fine"], choices=sorted(inputs.WORKLOADS),
                    help="other workloads given a compact line in the default run (none: --workloads)")
    ap.add_argument("--graph", action=argparse.BooleanOptionalAction, default=True,
                    help="time the steps as replays of a CUDA graph of one step (default); the eager "
                         "launches are timed too and reported beside")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu DRAM bytes per launch of the SwiGLU GEMM, for the roofline")
    return ap.parse_args()


def workload_desc(w) -> str:
    return (f"{w.name}: T={w.T} d={w.d} ffn={w.ffn} E={w.E} top-{w.topk} R={w.R} tile_M={w.tile_M}"
            + (" zipf-bias" if w.skew else ""))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------- dist
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        rank = dist.get_rank()
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
        return rank, world
    return 0, 1


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(local_seconds: float, local_units: float, world: int):
    """Whole-job throughput: units over all ranks / the slowest rank's time."""
    t = reduce_max(local_seconds, world)
    return local_units * world / t, t


# ------------------------------------------------------------------------------------ clocks
class Nvml:
    """Read-only NVML queries (libnvidia-ml through ctypes) of one GPU: SM clock, maximum SM clock,
    clock event (throttle) reason bits and power draw. Raises OSError where NVML is unavailable."""

    CLOCK_SM = 1

    def __init__(self, cuda_index: int):
        import ctypes
        self.ct = ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError as e:
            raise OSError(f"libnvidia-ml: {e}")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.lib = lib
        dev = ctypes.c_void_p()
        ok = False
        try:  # the CUDA device's UUID names the same GPU whatever CUDA_VISIBLE_DEVICES says
            uuid = "GPU-" + str(torch.cuda.get_device_properties(cuda_index).uuid)
            ok = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev)) == 0
        except Exception:
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(dev)) != 0:
            raise OSError("no NVML handle for the device")
        self.dev = dev
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(dev, self.CLOCK_SM, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        try:
            self._reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def read(self):
        """(SM MHz, max SM MHz, reason bits, power in W)."""
        ct = self.ct
        c, r, pw = ct.c_uint(0), ct.c_ulonglong(0), ct.c_uint(0)
        self.lib.nvmlDeviceGetClockInfo(self.dev, self.CLOCK_SM, ct.byref(c))
        self._reasons(self.dev, ct.byref(r))
        self.lib.nvmlDeviceGetPowerUsage(self.dev, ct.byref(pw))
        return float(c.value), self.max_mhz, int(r.value), pw.value / 1000.0

    def close(self):
        self.lib.nvmlShutdown()


# NVML clock event reason bits (nvml.h) reported by name (0x1, GPU idle, is not a limit)
REASON_BITS = {0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x10: "sync_boost",
               0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    """SM clock, power and clock event (throttle) reasons sampled during the timed region.

    A background thread reads NVML every 2 ms between __enter__ and __exit__, so even a timed region
    of a few tens of milliseconds holds many samples taken under load. `reader` (for tests) replaces
    NVML; where NVML cannot be opened, nvidia-smi is sampled every 200 ms instead (it needs a timed
    region of a second or more to see the load)."""

    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.002

    def __init__(self, gpu_index: int, reader=None):
        self.gpu = gpu_index
        self.reader = reader
        self.nvml = None
        self.proc = None
        self.thread = None
        self.samples = []  # (sm MHz, max MHz, reason names, power W)
        self.source = "unsampled"

    def _poll(self, stop):
        read = self.reader or self.nvml.read
        while True:
            try:
                mhz, mx, bits, pw = read()
                self.samples.append((mhz, mx, [n for b, n in REASON_BITS.items() if bits & b], pw))
            except Exception:
                return
            if stop.wait(self.PERIOD_S):
                return

    def __enter__(self):
        import threading
        if self.reader is None:
            try:
                self.nvml = Nvml(self.gpu)
            except OSError:
                self.nvml = None
        if self.reader is not None or self.nvml is not None:
            self.source = "nvml" if self.reader is None else "reader"
            self._stop = threading.Event()
            self.thread = threading.Thread(target=self._poll, args=(self._stop,), daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.SMI_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self._stop.set()
            self.thread.join(timeout=5)
            if self.nvml is not None:
                self.nvml.close()
            return
        out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz, mx = float(parts[1]), float(parts[2])
                pw = float(parts[3])
            except ValueError:
                continue
            self.samples.append((mhz, mx, [n for n, v in zip(names, parts[5:9]) if v.lower().startswith("active")],
                                 pw))

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "source": self.source}
        reasons = sorted({n for s in self.samples for n in s[2]})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples),
                "sm_mhz_min": min(s[0] for s in self.samples),
                "sm_mhz_distinct": len({s[0] for s in self.samples}),
                "power_w_max": round(max(s[3] for s in self.samples), 1),
                "reasons": reasons, "samples": len(self.samples), "source": self.source}


def zero_kernel_clocks(ws):
    """Zero the workspace's SM clock counters (the GEMM launches add to them)."""
    ws.view("trace")[8:12].zero_()


def kernel_clocks(ws) -> dict:
    """Mean SM clock (MHz) of the expert-GEMM launches since the counters were zeroed: CTA 0 of each
    launch adds its SM's cycle count and the global-timer nanoseconds of the same span."""
    v = ws.view("trace")[8:12].cpu().numpy().astype(np.int64)
    mhz = lambda c, n: round(1000.0 * float(c) / float(n), 1) if n > 0 else None  # noqa: E731
    return {"swiglu_gemm": mhz(v[0], v[1]), "down_projection": mhz(v[2], v[3]),
            "source": "SM cycle counter over the global timer, CTA 0 of each GEMM launch in the region"}


# ---------------------------------------------------------------------------------- our arm
def default_flags(copy_warps: bool, direct_tail: bool = True, tail_assist: bool = True, pair: bool = True,
                  fused_dispatch: bool = False, fused_gemms: bool = False, pdl=None) -> int:
    """The bench's launch configuration: both expert GEMMs on CTA pairs (the down-projection's consumer
    partition picked at run time from its tile count), finished producers joining the copy, the last
    wave's bands returned by the down-projection's epilogue, and (per workload) the producers' copy
    warps; programmatic dependent launch between the kernels unless the copy
    warps run (their down-projection is the cooperative single-CTA kernel, with which it measured
    slower)."""
    import tile_level_copy_gb300 as tlc
    if pdl is None:
        pdl = not copy_warps
    return ((tlc.MOE_TAIL_ASSIST if tail_assist else 0) | (tlc.MOE_COPY_WARPS if copy_warps else 0) |
            (tlc.MOE_PAIR_UMMA | tlc.MOE_ADAPTIVE_CONSUMERS if pair else 0) |
            (tlc.MOE_DIRECT_TAIL if direct_tail else 0) |
            (tlc.MOE_FUSED_DISPATCH if fused_dispatch else 0) | (tlc.MOE_FUSED_GEMMS if fused_gemms else 0) |
            (tlc.MOE_PDL if pdl else 0))


class LayerBench:
    """One workload's inputs, weights, workspace and output on the device, and the ways to run it."""

    def __init__(self, w, seed: int, dev):
        import tile_level_copy_gb300 as tlc
        self.tlc, self.w, self.dev = tlc, w, dev
        self.logits_np = inputs.make_logits(w, seed)
        self.x_cpu = inputs.make_x(w, seed)
        self.logits, self.x = torch.from_numpy(self.logits_np).to(dev), self.x_cpu.to(dev)
        self.W = {}
        for n in ("W1", "W3", "W2"):
            shape = (w.E, w.ffn, w.d) if n != "W2" else (w.E, w.d, w.ffn)
            self.W[n] = torch.empty(shape, dtype=torch.bfloat16, device=dev)
            inputs.make_weight_into(w, seed, n, self.W[n])
        self.ws = tlc.Workspace(tlc.Config.from_workload(w), dev)  # the layout depends on the shape only
        self.out = torch.empty(w.T, w.d, dtype=torch.float32, device=dev)

    def step(self, cfg, seq, events=None):
        """One layer step: overlapped (seq False), GEMM-then-copy (seq True) or with the return copy
        on the copy engines (seq "dma", eager only: the host issues the copies)."""
        if seq == "dma":
            if getattr(self, "host_rec", None) is None:
                n = self.tlc.dma_host_bytes(cfg)
                self.host_rec = torch.zeros((n + 15) // 16 * 4, dtype=torch.int32).pin_memory()
            self.tlc.forward_dma(cfg, self.logits, self.x, self.W["W1"], self.W["W3"], self.W["W2"], self.out,
                                 self.ws, self.host_rec, events=events)
            return
        self.tlc.forward(cfg, self.logits, self.x, self.W["W1"], self.W["W3"], self.W["W2"], self.out, self.ws,
                         sequential=seq, events=events)

    def check(self, cfg, where: str):
        rc, detail = self.tlc.status(cfg, self.ws)
        if rc != self.tlc.MOE_OK:
            raise RuntimeError(f"device status {rc} ({detail}) {where}: {self.tlc.lib().moe_last_error().decode()}")

    def graph(self, cfg, seq: bool):
        """One step captured as a CUDA graph (after two eager steps on a side stream)."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                self.step(cfg, seq)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(cfg, seq)
        return g

    def graph_steps(self, cfg, events):
        """len(events) overlapped steps captured as one CUDA graph, step i recording its stage events
        (event-record nodes of the graph) unless events[i] is None, after two eager steps on a side
        stream."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                self.step(cfg, False)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for ev in events:
                self.step(cfg, False, ev)
        return g

    def tails(self, cfg, reps: int):
        """Copy tail after the last flag (ms) and the tail's trace marks (us) of `reps` overlapped steps."""
        tails, marks = [], []
        tlc = self.tlc
        for _ in range(reps):
            self.step(cfg, False)
            torch.cuda.synchronize()
            tr = self.ws.view("trace").cpu().numpy().astype(np.int64)
            tails.append(max(0, int(tr[tlc.TRACE_COPY_END]) - int(tr[tlc.TRACE_GEMM2_END])) / 1e6)
            marks.append([(int(tr[i]) - int(tr[tlc.TRACE_GEMM2_END])) / 1e3 for i in
                          (tlc.TRACE_BAND_DONE, tlc.TRACE_LAST_ACQUIRE, tlc.TRACE_LAST_LOAD, tlc.TRACE_LAST_DRAIN,
                           tlc.TRACE_COPY_END)])
        self.check(cfg, "in the trace steps")
        return tails, marks


STAGES = ("route_plan_permute", "swiglu_gemm", "down_gemm", "copy", "combine")


def alternate_eager(lb: LayerBench, arms, K: int, Wm: int):
    """Eager steps of every arm, interleaved step by step (A B C A B C ...), each with stage events.
    Returns {arm: array [K, 5] of stage ms}."""
    tlc = lb.tlc
    for _ in range(Wm):
        for cfg, seq in arms.values():
            lb.step(cfg, seq)
    evs = {a: [tlc.stage_events() for _ in range(K)] for a in arms}
    zero_kernel_clocks(lb.ws)  # kernel_clocks(lb.ws) afterwards: the GEMMs' clock over these steps
    torch.cuda.synchronize()
    for i in range(K):
        for a, (cfg, seq) in arms.items():
            lb.step(cfg, seq, evs[a][i])
    torch.cuda.synchronize()
    for a, (cfg, _) in arms.items():
        lb.check(cfg, f"in the alternating eager steps ({a})")
    return {a: np.array([[e[j].elapsed_time(e[j + 1]) for j in range(tlc.EV_COUNT - 1)] for e in evs[a]])
            for a in arms}


def alternate_graphs(lb: LayerBench, arms, K: int, Wm: int, dev_index: int):
    """CUDA-graph replays of every arm interleaved replay by replay, each replay between two events on
    the replaying stream. Returns ({arm: [K] ms}, clock summary of the whole interleaved region)."""
    graphs = {a: lb.graph(cfg, seq) for a, (cfg, seq) in arms.items()}
    for _ in range(Wm):
        for g in graphs.values():
            g.replay()
    ev = {a: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
          for a in arms}
    zero_kernel_clocks(lb.ws)
    torch.cuda.synchronize()
    with ClockSampler(dev_index) as clk:
        for i in range(K):
            for a, g in graphs.items():
                ev[a][i][0].record()
                g.replay()
                ev[a][i][1].record()
        torch.cuda.synchronize()
    for a, (cfg, _) in arms.items():
        lb.check(cfg, f"in the alternating graph replays ({a})")
    summary = clk.summary()
    summary["kernel_sm_mhz"] = kernel_clocks(lb.ws)
    return {a: np.array([e0.elapsed_time(e1) for e0, e1 in ev[a]]) for a in arms}, summary


def spread_ms(x) -> float:
    """Step-to-step spread of a series of step times: 1.4826 x median absolute deviation (about one
    standard deviation for normal noise, robust to outliers)."""
    x = np.asarray(x, float)
    return float(1.4826 * np.median(np.abs(x - np.median(x))))


def run_ours(args, rank: int, world: int):
    import tile_level_copy_gb300 as tlc
    from tile_level_copy_gb300 import build as tlc_build

    tlc_build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = inputs.WORKLOADS[args.workload]
    dc, dw = DEFAULT_COPY.get(args.workload, (8, False))
    if args.consumers is None:
        args.consumers = dc
    if args.copy_warps is None:
        args.copy_warps = dw
    seed = args.seed + rank
    flags = default_flags(args.copy_warps, direct_tail=args.direct_tail, tail_assist=not args.no_tail_assist,
                          pair=args.pair_umma, fused_dispatch=args.fused_dispatch, fused_gemms=args.fused_gemms,
                          pdl=args.pdl)
    cfg = tlc.Config.from_workload(w, consumer_ctas=args.consumers, mgb=args.mgb, flags=flags,
                                   tail_window=args.tail_window)
    peaks, peaks_src = load_peaks()
    lb = LayerBench(w, seed, dev)
    K, Wm = args.steps, args.warmup

    # ---- headline: K contiguous steps of the overlapped layer: one replay of a CUDA graph holding the
    # K captured steps (or K eager steps). Every fifth step (the last one when K < 5) records its
    # stage events, so each kernel's duration is measured inside the timed region itself; an event
    # record costs about 0.5% of a step, so the other steps record none.
    sampled = [i for i in range(K) if i % 5 == 4] or [K - 1]
    hl_ev = [tlc.stage_events() if i in sampled else None for i in range(K)]
    if args.graph:
        g1 = lb.graph(cfg, False)
        gk = lb.graph_steps(cfg, hl_ev)
        for _ in range(Wm):
            g1.replay()
        lb.check(cfg, "in the graph warm-up")
        run_k = gk.replay
    else:
        for _ in range(Wm):
            lb.step(cfg, False)
        lb.check(cfg, "in the warm-up")
        run_k = lambda: [lb.step(cfg, False, hl_ev[i]) for i in range(K)]  # noqa: E731
    zero_kernel_clocks(lb.ws)
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        t0.record()
        run_k()
        t1.record()
        torch.cuda.synchronize()
    barrier(world)
    lb.check(cfg, "in the timed region")
    sec_ovl = t0.elapsed_time(t1) / 1e3
    clocks = clk.summary()
    # NVML averages over a longer window than this region: the kernels' own clock beside it
    clocks["kernel_sm_mhz"] = kernel_clocks(lb.ws)
    value, sec_max = aggregate(sec_ovl, w.T * K, world)
    hl_st = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(tlc.EV_COUNT - 1)] for e in hl_ev if e])
    hl_med = {n: float(np.median(hl_st[:, i])) for i, n in enumerate(STAGES)}
    # the CTA-pair down-projection's producer CTAs in the timed steps (MOE_ADAPTIVE_CONSUMERS picks
    # them from the tile count; 0 when no overlapped pair launch ran)
    producer_ctas = int(lb.ws.view("meta")[10].item())

    # eager launches of the same K steps, contiguous, beside the headline
    for _ in range(Wm):
        lb.step(cfg, False)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk_e:
        e0.record()
        for _ in range(K):
            lb.step(cfg, False)
        e1.record()
        torch.cuda.synchronize()
    lb.check(cfg, "in the eager steps")
    eager_value, eager_sec = aggregate(e0.elapsed_time(e1) / 1e3, w.T * K, world)

    # ---- the arms compared in alternation: overlapped, GEMM-then-copy, and (with the direct tail)
    # the overlapped layer without it, i.e. every band through the consumer
    arms = {"overlapped": (cfg, False), "sequential": (cfg, True)}
    direct = bool(cfg.flags & tlc.MOE_DIRECT_TAIL)
    if direct:
        arms["overlapped_all_bands_copied"] = (dataclasses.replace(cfg, flags=cfg.flags & ~tlc.MOE_DIRECT_TAIL), False)
    # the permute as its own launch against the row copies fused into the SwiGLU GEMM, whichever is
    # not the default
    fused = bool(cfg.flags & tlc.MOE_FUSED_DISPATCH)
    other_dispatch = "overlapped_separate_permute" if fused else "overlapped_fused_dispatch"
    arms[other_dispatch] = (dataclasses.replace(cfg, flags=cfg.flags ^ tlc.MOE_FUSED_DISPATCH), False)
    # both GEMMs in one launch against two launches, whichever is not the default (needs the
    # down-projection on CTA pairs)
    fused_gemms = bool(cfg.flags & tlc.MOE_FUSED_GEMMS)
    other_gemms = "overlapped_separate_gemms" if fused_gemms else "overlapped_fused_gemms"
    arms[other_gemms] = (dataclasses.replace(cfg, flags=cfg.flags ^ tlc.MOE_FUSED_GEMMS), False)
    # another (fixed) consumer partition, when asked for (same flags otherwise)
    for c_alt in args.alt_consumers:
        arms[f"overlapped_c{c_alt}"] = (dataclasses.replace(cfg, consumer_ctas=c_alt,
                                                            flags=cfg.flags & ~tlc.MOE_ADAPTIVE_CONSUMERS), False)
    # programmatic dependent launch between the kernels against serial launches
    pdl = bool(cfg.flags & tlc.MOE_PDL)
    other_pdl = "overlapped_serial_launches" if pdl else "overlapped_pdl"
    arms[other_pdl] = (dataclasses.replace(cfg, flags=cfg.flags ^ tlc.MOE_PDL), False)
    eager_arms = dict(arms)
    if args.dma:  # the copy-engine variant: eager only (its host thread issues the copies)
        eager_arms["copy_engines"] = (cfg, "dma")
    st = alternate_eager(lb, eager_arms, K, Wm)
    eager_kclk = kernel_clocks(lb.ws)
    rep, clocks_alt = alternate_graphs(lb, arms, K, Wm, dev.index) if args.graph else (
        {a: st[a].sum(1) for a in arms}, None)
    med = {a: float(np.median(rep[a])) for a in arms}
    eager_ms = {a: float(np.median(st[a].sum(1))) for a in eager_arms}
    stage_med = {a: {n: float(np.median(st[a][:, i])) for i, n in enumerate(STAGES)} for a in eager_arms}
    copy_alone_ms = stage_med["sequential"]["copy"]

    # overlap from %globaltimer stamps of a few more overlapped steps of each overlapped arm
    trace = {}
    for _ in range(2):  # alternating, 3 steps per arm per round
        for a in [x for x in arms if x != "sequential"]:
            t_, m_ = lb.tails(arms[a][0], 3)
            trace.setdefault(a, ([], []))
            trace[a][0].extend(t_)
            trace[a][1].extend(m_)

    def hidden_of(a):
        tails, marks = trace[a]
        return {"hidden_pct": round(100 * (1 - statistics.median(tails) / copy_alone_ms), 2),
                "tail_ms": round(statistics.median(tails), 4),
                "tail_marks_us": dict(zip(["band_done", "last_acquire", "last_load", "last_drain", "copy_end"],
                                          [round(float(v), 2) for v in np.median(np.array(marks), 0)]))}

    ms_ovl, ms_seq = med["overlapped"], med["sequential"]
    # the arms ran interleaved, so replay i of each arm saw the same clock: the step-to-step spread of
    # their paired differences is the noise a wall-time difference must exceed
    diff = rep["sequential"] - rep["overlapped"]
    diff_ms, spread = float(np.median(diff)), spread_ms(diff)
    wall = None
    wall_note = (f"median paired T_seq - T_ovl = {diff_ms * 1e3:.1f} us is within its step-to-step spread "
                 f"({spread * 1e3:.1f} us): no wall overlap is claimed")
    if abs(diff_ms) > spread:
        wall = round(100 * diff_ms / copy_alone_ms, 2)
        wall_note = (f"median paired T_seq - T_ovl = {diff_ms * 1e3:.1f} us, above its step-to-step spread "
                     f"({spread * 1e3:.1f} us)")
    swiglu_ratio = stage_med["sequential"]["swiglu_gemm"] / stage_med["overlapped"]["swiglu_gemm"]

    # the page's own copy design beside it: a dedicated consumer partition of 8 CTAs (no copy warps,
    # no direct tail), same GEMMs; its hidden fraction (trace stamps) and eager step time
    cfg_page = dataclasses.replace(cfg, consumer_ctas=8,
                                   flags=(cfg.flags & ~(tlc.MOE_COPY_WARPS | tlc.MOE_DIRECT_TAIL |
                                                        tlc.MOE_ADAPTIVE_CONSUMERS)) | tlc.MOE_TAIL_ASSIST)
    page_tails, _ = lb.tails(cfg_page, 5)
    page_ev = [tlc.stage_events() for _ in range(5)]
    for i in range(5):
        lb.step(cfg_page, False, page_ev[i])
    torch.cuda.synchronize()
    lb.check(cfg_page, "in the dedicated-partition steps")
    page_ms = float(np.median([e[tlc.EV_BEGIN].elapsed_time(e[tlc.EV_END]) for e in page_ev]))

    # GEMM numbers: real rows = T*k; executed rows = 128 per work item: both GEMMs take the same
    # items, 128 rows of one expert in the compact layout (with CTA pairs, an expert's odd item also
    # occupies the idle half of its pair); P = padded rows of the owner-aligned layout (the
    # down-projection's output rows), PC = rows of the compact layout
    ws = lb.ws
    meta = ws.view("meta").cpu()
    P, items, items_up, PC = (int(meta[i].item()) for i in (0, 7, 8, 9))
    TK = w.T * w.topk
    experts = ws.view("experts").cpu().numpy()
    if cfg.flags & tlc.MOE_PAIR_UMMA:
        iu = experts[:, 4]
        exec_rows_up = 128 * int(np.sum(2 * ((iu + 1) // 2)))
    else:
        exec_rows_up = 128 * items_up
    # the down-projection runs on CTA pairs under the same conditions as in the library
    pair_down = bool(cfg.flags & tlc.MOE_PAIR_UMMA) and not (cfg.flags & tlc.MOE_COPY_WARPS) and \
        w.d % 256 == 0 and args.consumers % 2 == 0
    if pair_down:  # an expert's items in pairs: an odd one also occupies the idle half of its pair
        first = np.sort(experts[:, 6])
        cnt = np.diff(np.append(first, items))
        exec_rows = 128 * int(np.sum(2 * ((cnt + 1) // 2)))
    else:
        exec_rows = 128 * items
    up_ms = hl_med["swiglu_gemm"]                   # inside the headline timed region
    down_ms = stage_med["sequential"]["down_gemm"]  # the down-projection alone (sequential arm, alternation)
    fl_up_alg, fl_down_alg = 4.0 * TK * w.d * w.ffn, 2.0 * TK * w.d * w.ffn
    fl_up_exe, fl_down_exe = 4.0 * exec_rows_up * w.d * w.ffn, 2.0 * exec_rows * w.d * w.ffn
    gemm_exec_tflops = (fl_up_exe + fl_down_exe) / ((up_ms + down_ms) * 1e-3) / 1e12
    gemm_alg_tflops = (fl_up_alg + fl_down_alg) / ((up_ms + down_ms) * 1e-3) / 1e12
    # The SwiGLU launch time comes from the headline timed region. The measured sustained rate is a
    # seconds-long GEMM loop under the power limit, the burst rate a best-of-10 run; a region shorter
    # than a second is held to the burst rate (the GEMMs' own clock counters show the limiter acting
    # inside it too, about as it does in a burst).
    region_s = sec_ovl
    if region_s >= 1.0:
        peak_tc, peak_kind = peaks["bf16_tflops_sustained"], "bf16_tflops_sustained"
    else:
        peak_tc, peak_kind = peaks["bf16_tflops"], "bf16_tflops (burst)"
    peak_note = f"{peaks_src} {peak_kind}: the kernel's launches were timed over a {region_s:.3f} s region"

    roof_achieved = fl_up_alg / (up_ms * 1e-3) / 1e12
    # algorithmic DRAM bytes of the SwiGLU GEMM: W1 and W3 once, the compact rows in, the hidden out
    alg_bytes_up = 2 * w.E * w.ffn * w.d * 2 + PC * w.d * 2 + PC * w.ffn * 2
    traffic = args.traffic if args.traffic is not None else captured_traffic(args.workload, args.pair_umma)
    roofline = {"kernel": ("gemm_pair_kernel<1> (SwiGLU up-projection, CTA pairs)" if args.pair_umma
                           else "gemm_kernel<1> (SwiGLU up-projection)"), "bound": "tensor",
                "achieved": round(roof_achieved, 1), "peak": peak_tc, "unit": "TFLOP/s",
                "frac": round(roof_achieved / peak_tc, 4),
                "traffic": traffic,
                "traffic_source": ("--traffic argument" if args.traffic is not None else
                                   "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch of this kernel, "
                                   "captured on another GB300 of the pool, not measured in this run (null when "
                                   "the kernel sources differ from the captured ones)"),
                "algorithmic_bytes_per_launch": alg_bytes_up,
                "peak_source": peak_note,
                "executed_tflops": round(fl_up_exe / (up_ms * 1e-3) / 1e12, 1),
                "algorithmic_flops_per_launch": fl_up_alg, "launch_ms": round(up_ms, 4),
                "launch_ms_source": f"median of {len(sampled)} of the {K} launches inside the timed region (steps "
                                    f"{', '.join(str(i) for i in sampled)} record stage events)"}
    # the same launches against the tensor pipe's own peak at the clock they ran at (8192 dense bf16
    # FLOP per SM per clock)
    up_mhz, dn_mhz = clocks["kernel_sm_mhz"]["swiglu_gemm"], clocks["kernel_sm_mhz"]["down_projection"]
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    if up_mhz:
        roofline["kernel_sm_mhz"] = up_mhz
        roofline["executed_frac_of_tensor_peak_at_kernel_clock"] = round(
            fl_up_exe / (up_ms * 1e-3) / (n_sm * 8192 * up_mhz * 1e6), 4)

    # HBM-bound stages against the measured copy bandwidth (algorithmic bytes / stage time)
    hbm = peaks["hbm_gbs"]
    E_, k_, d_ = w.E, w.topk, w.d
    pad_rows = PC - TK
    stage_bytes = {
        # route: logits in, idx/gate/rank out; permute: x in, k rows + padding rows of Xc out
        "route_plan_permute": w.T * E_ * 4 + TK * 12 + w.T * d_ * 2 + (TK + pad_rows) * d_ * 2,
        "copy": 2 * TK * d_ * 2,                                  # Yp rows in, Ret rows out
        "combine": TK * d_ * 2 + w.T * d_ * 4 + TK * 8,          # Ret rows + gates in, out written
    }
    stage_ms = {"route_plan_permute": hl_med["route_plan_permute"],  # inside the timed region
                "copy": copy_alone_ms, "combine": hl_med["combine"]}
    hbm_stages = {n: {"bytes": int(b), "ms": round(stage_ms[n], 4),
                      "achieved_gbs": round(b / (stage_ms[n] * 1e-3) / 1e9, 1),
                      "frac_of_measured_hbm": round(b / (stage_ms[n] * 1e-3) / 1e9 / hbm, 3)}
                  for n, b in stage_bytes.items()}

    # Layer roofline: each GEMM at the larger of its algorithmic FLOPs / the tensor peak and its
    # algorithmic DRAM bytes (weights once, activations in and out) / the copy bandwidth; routing,
    # plan, permute and combine at their algorithmic bytes / the copy bandwidth; the return copy
    # hidden under the down-projection, which is what the overlap aims at.
    w_bytes = w.E * w.d * w.ffn * 2
    roof_terms_ms = {
        "swiglu_gemm": 1e3 * max(fl_up_alg / (peak_tc * 1e12), (2 * w_bytes + TK * (w.d + w.ffn) * 2) / (hbm * 1e9)),
        "down_gemm": 1e3 * max(fl_down_alg / (peak_tc * 1e12), (w_bytes + TK * (w.ffn + w.d) * 2) / (hbm * 1e9)),
        "route_plan_permute": 1e3 * stage_bytes["route_plan_permute"] / (hbm * 1e9),
        "combine": 1e3 * stage_bytes["combine"] / (hbm * 1e9),
    }
    roof_ms = sum(roof_terms_ms.values())
    step_ms = sec_max * 1e3 / K
    layer_roofline = {"ms_per_step": round(roof_ms, 4), "tokens_per_s": round(w.T / (roof_ms * 1e-3), 1),
                      "frac": round(roof_ms / step_ms, 4),
                      "terms_ms": {n: round(v, 4) for n, v in roof_terms_ms.items()},
                      "peaks": {"tflops": peak_tc, "hbm_gbs": hbm},
                      "note": "roofline step time / measured step time; the return copy counted as hidden"}

    overlap = {**hidden_of("overlapped"), "copy_alone_ms": round(copy_alone_ms, 4),
               "definition": "hidden = 1 - max(0, copy end - last down-projection flag) / the sequential copy's "
                             "time (%globaltimer stamps of the same step)",
               "wall_pct": wall, "wall_note": wall_note,
               "sequential_ms_per_step": round(ms_seq, 4), "sequential_tokens_per_s": round(w.T / (ms_seq * 1e-3), 1),
               "speedup_vs_sequential": round(ms_seq / ms_ovl, 4),
               "alternating": {
                   "method": (f"{K} CUDA-graph replays per arm, interleaved replay by replay "
                              f"({' / '.join(arms)}), each between two events; medians per arm" if args.graph else
                              f"{K} eager steps per arm, interleaved step by step; medians per arm"),
                   "ms_per_step": {a: round(v, 4) for a, v in med.items()},
                   "paired_diff_seq_minus_ovl_ms": round(diff_ms, 4),
                   "paired_spread_ms": round(spread, 4),
                   "eager_ms_per_step": {a: round(v, 4) for a, v in eager_ms.items()},
                   "swiglu_stage_ratio_seq_over_ovl": round(swiglu_ratio, 4),
                   "swiglu_stage_check": "ok" if abs(swiglu_ratio - 1) <= 0.01 else
                   "the identical SwiGLU launch differs by more than 1% between the arms",
                   "clocks": clocks_alt},
               "dedicated_partition_c8": {
                   "hidden_pct": round(100 * (1 - statistics.median(page_tails) / copy_alone_ms), 2),
                   "tail_ms": round(statistics.median(page_tails), 4),
                   "eager_ms_per_step": round(page_ms, 4)}}
    overlap["dispatch"] = {
        "default": "fused into the SwiGLU GEMM" if fused else "separate permute launch",
        "other": other_dispatch, "ms_per_step": round(med[other_dispatch], 4),
        "paired_diff_other_minus_default_ms": round(float(np.median(rep[other_dispatch] - rep["overlapped"])), 4),
        "paired_spread_ms": round(spread_ms(rep[other_dispatch] - rep["overlapped"]), 4),
        "swiglu_and_permute_ms": {a: round(stage_med[a]["route_plan_permute"] + stage_med[a]["swiglu_gemm"], 4)
                                  for a in ("overlapped", other_dispatch)}}
    if args.alt_consumers:
        overlap["consumer_partitions"] = {
            f"c{c_alt}": {"ms_per_step": round(med[f"overlapped_c{c_alt}"], 4),
                          "paired_diff_minus_default_ms": round(float(np.median(rep[f"overlapped_c{c_alt}"] -
                                                                                 rep["overlapped"])), 4),
                          "paired_spread_ms": round(spread_ms(rep[f"overlapped_c{c_alt}"] - rep["overlapped"]), 4),
                          "hidden_pct": hidden_of(f"overlapped_c{c_alt}")["hidden_pct"]}
            for c_alt in args.alt_consumers}
    overlap["launch_dependencies"] = {
        "default": "programmatic dependent launch" if pdl else "serial launches",
        "other": other_pdl, "ms_per_step": round(med[other_pdl], 4),
        "paired_diff_other_minus_default_ms": round(float(np.median(rep[other_pdl] - rep["overlapped"])), 4),
        "paired_spread_ms": round(spread_ms(rep[other_pdl] - rep["overlapped"]), 4)}
    overlap["gemm_launches"] = {
        "default": "one launch for both GEMMs" if fused_gemms else "a launch per GEMM",
        "other": other_gemms, "ms_per_step": round(med[other_gemms], 4),
        "paired_diff_other_minus_default_ms": round(float(np.median(rep[other_gemms] - rep["overlapped"])), 4),
        "paired_spread_ms": round(spread_ms(rep[other_gemms] - rep["overlapped"]), 4)}
    if args.dma:
        # copy engines: the "copy" stage runs from the down-projection's end to the last band copy's end
        # (the copy stream's event), so its median is the exposed tail
        dma_tail = max(0.0, stage_med["copy_engines"]["copy"])
        overlap["copy_engines"] = {
            "call": "moe_forward_dma: no consumer SMs; one cudaMemcpyAsync per ready band (per run of ready bands "
                    "adjacent in Yp and Ret) issued by the calling thread as the records arrive in pinned host memory; "
                    "with the default flags the bands the last wave completes are written by the epilogue (direct tail)",
            "eager_ms_per_step": round(eager_ms["copy_engines"], 4),
            "eager_ms_per_step_sm_consumers": round(eager_ms["overlapped"], 4),
            "down_gemm_ms": round(stage_med["copy_engines"]["down_gemm"], 4),
            "tail_ms": round(dma_tail, 4),
            "hidden_pct": round(100 * (1 - dma_tail / copy_alone_ms), 2)}
    if direct:
        overlap["direct_tail"] = {
            "tail_window": cfg.tail_window or "one wave (one tile per producer CTA pair)",
            "bands_returned_by_epilogue": None,
            "all_bands_copied": {**hidden_of("overlapped_all_bands_copied"),
                                 "ms_per_step": round(med["overlapped_all_bands_copied"], 4),
                                 "note": "the same layer without MOE_DIRECT_TAIL (every band through the "
                                         "consumer), timed in the same alternation"}}
        # which bands the epilogue returned: their Yp rows are left unwritten; count them from a step
        # with Yp zeroed first
        ws.view("Yp").zero_()
        lb.step(cfg, False)
        torch.cuda.synchronize()
        tiles = ws.view("tiles").cpu().numpy()
        MT = int(meta[1].item())
        yp = ws.view("Yp")[:P].view(torch.int16).cpu().numpy()  # one copy, counted on the host
        n_direct = sum(1 for m in range(MT) if not yp[int(tiles[m, 2]):int(tiles[m, 2]) + int(tiles[m, 3])].any())
        overlap["direct_tail"]["bands_returned_by_epilogue"] = f"{n_direct} of {MT}"

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": round(sec_max * 1e3 / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w), "T": w.T, "d": w.d, "ffn": w.ffn, "E": w.E, "topk": w.topk,
                   "R": w.R, "tile_M": w.tile_M, "consumer_ctas": args.consumers,
                   "adaptive_consumers": bool(flags & tlc.MOE_ADAPTIVE_CONSUMERS),
                   "down_producer_ctas": producer_ctas or None, "copy_warps": bool(args.copy_warps),
                   "pair_umma": bool(args.pair_umma), "mgb": args.mgb, "direct_tail": direct,
                   "tail_window": args.tail_window, "fused_dispatch": bool(args.fused_dispatch),
                   "fused_gemms": bool(args.fused_gemms), "pdl": bool(flags & tlc.MOE_PDL),
                   "tail_assist": not args.no_tail_assist, "seed": args.seed,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": f"no flush: each step streams {3 * w.E * w.d * w.ffn * 2 / 1e9:.2f} GB of expert weights "
                      f"(> 129 MB L2)"},
        "gpu_launches": 6 * K,
        "timing": (f"one replay of a CUDA graph of {K} captured steps (each: route, plan, permute, SwiGLU GEMM, "
                   "down-projection + copy, combine)" if args.graph else "eager launches"),
        "eager": {"value": round(eager_value, 1), "ms_per_step": round(eager_sec * 1e3 / K, 4),
                  "clocks": clk_e.summary(), "note": f"{K} contiguous eager steps after the timed region"},
        "clocks": clocks,
        "roofline": roofline,
        "gemm": {"executed_tflops": round(gemm_exec_tflops, 1), "algorithmic_tflops": round(gemm_alg_tflops, 1),
                 "executed_frac_of_peak": round(gemm_exec_tflops / peak_tc, 4),
                 "algorithmic_frac_of_peak": round(gemm_alg_tflops / peak_tc, 4),
                 "executed_frac_of_sustained_peak": round(gemm_exec_tflops / peaks["bf16_tflops_sustained"], 4),
                 "peak_tflops": peak_tc, "peak_source": peak_note, "up_ms": round(up_ms, 4),
                 "down_ms": round(down_ms, 4),
                 "down_ms_source": "the sequential arm's down-projection launches in the eager alternation, whose "
                                   "GEMMs ran at the eager_kernel_sm_mhz clock",
                 "eager_kernel_sm_mhz": eager_kclk,
                 "down_kernel": "gemm_pair_kernel<2> (CTA pairs)" if pair_down
                 else "gemm_kernel<2>", "padded_rows": P, "compact_rows": PC,
                 "down_algorithmic_frac_of_peak": round(fl_down_alg / (down_ms * 1e-3) / 1e12 / peak_tc, 4),
                 "down_and_copy_ms_timed_region": round(hl_med["down_gemm"], 4),
                 "down_and_copy_algorithmic_frac_of_peak": round(
                     fl_down_alg / (hl_med["down_gemm"] * 1e-3) / 1e12 / peak_tc, 4),
                 "down_and_copy_executed_frac_of_tensor_peak_at_kernel_clock": (round(
                     fl_down_exe / (hl_med["down_gemm"] * 1e-3) / (n_sm * 8192 * dn_mhz * 1e6), 4) if dn_mhz else None),
                 "executed_rows_up": exec_rows_up, "executed_rows_down": exec_rows, "work_items_up": items_up,
                 "work_items_down": items, "real_rows": TK},
        "overlap": overlap,
        "stages_ms": {"timed_region": {n: round(v, 4) for n, v in hl_med.items()},
                      **{f"alternating_{a}": {n: round(v, 4) for n, v in stage_med[a].items()} for a in eager_arms}},
        "hbm_stages": hbm_stages,
        "layer_roofline": layer_roofline,
    }

    if not args.no_e2e:
        # End to end from pinned host memory: every step copies its logits and tokens in and its
        # output out. Headline: one moe_forward_host_pipelined call over the K steps (the transfers
        # of neighbouring steps overlap the layer); beside it, K separate moe_forward_host calls.
        W = lb.W
        logits_h = torch.from_numpy(lb.logits_np).pin_memory()
        x_h = lb.x_cpu.pin_memory()
        outs_h = [torch.empty(w.T, w.d, dtype=torch.float32).pin_memory() for _ in range(2)]
        h2d = logits_h.numel() * 4 + x_h.numel() * 2
        d2h = outs_h[0].numel() * 4

        def run_pipelined(n):
            tlc.forward_host_pipelined(cfg, [logits_h] * n, [x_h] * n, W["W1"], W["W3"], W["W2"],
                                       [outs_h[i % 2] for i in range(n)], ws)

        def timed_e2e(fn):
            torch.cuda.synchronize()
            barrier(world)
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            fn()
            t1.record()
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / 1e3

        run_pipelined(Wm)
        e2e_value, _ = aggregate(timed_e2e(lambda: run_pipelined(K)), w.T * K, world)
        for _ in range(Wm):
            tlc.forward_host(cfg, logits_h, x_h, W["W1"], W["W3"], W["W2"], outs_h[0], ws)

        def per_call():
            for _ in range(K):
                tlc.forward_host(cfg, logits_h, x_h, W["W1"], W["W3"], W["W2"], outs_h[0], ws)

        e2e_single, _ = aggregate(timed_e2e(per_call), w.T * K, world)
        lb.check(cfg, "in the end-to-end steps")
        res["e2e"] = {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "call": f"moe_forward_host_pipelined ({K} batches in one call)",
                      "per_call_value": round(e2e_single, 1), "per_call": "moe_forward_host, one call per batch"}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.seed, tokens=256, W=lb.W)
    if rank == 0 and world == 1 and args.workloads:
        del lb
        torch.cuda.empty_cache()
        res["workloads"] = {n: other_workload(n, args, peaks) for n in args.workloads if n != args.workload}
    return res


def other_workload(name: str, args, peaks) -> dict:
    """A compact line for another workload in its default launch configuration: tokens/s over one
    replay of a graph of K steps, hidden fraction of the return copy, SwiGLU GEMM roofline fraction
    (its launches inside that replay)."""
    import tile_level_copy_gb300 as tlc
    dev = torch.device("cuda", torch.cuda.current_device())
    w = inputs.WORKLOADS[name]
    c, warps = DEFAULT_COPY[name]
    cfg = tlc.Config.from_workload(w, consumer_ctas=c, flags=default_flags(warps))
    lb = LayerBench(w, args.seed, dev)
    K, Wm = max(5, args.steps // 2), max(3, args.warmup)
    ev = [tlc.stage_events() if i % 5 == 4 else None for i in range(K)]
    g1, gk = lb.graph(cfg, False), lb.graph_steps(cfg, ev)
    for _ in range(Wm):
        g1.replay()
    zero_kernel_clocks(lb.ws)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        t0.record()
        gk.replay()
        t1.record()
        torch.cuda.synchronize()
    lb.check(cfg, f"in the {name} replays")
    kclk = kernel_clocks(lb.ws)
    ms = t0.elapsed_time(t1) / K
    up_ms = float(np.median([e[tlc.EV_PLANNED].elapsed_time(e[tlc.EV_UP]) for e in ev if e]))
    arms = {"overlapped": (cfg, False), "sequential": (cfg, True),
            "overlapped_all_bands_copied": (dataclasses.replace(cfg, flags=cfg.flags & ~tlc.MOE_DIRECT_TAIL), False)}
    st = alternate_eager(lb, arms, 5, 2)
    copy_alone = float(np.median(st["sequential"][:, 3]))
    tails, _ = lb.tails(cfg, 5)
    tails_all, _ = lb.tails(arms["overlapped_all_bands_copied"][0], 5)
    fl_up = 4.0 * w.T * w.topk * w.d * w.ffn
    up_tflops = fl_up / (up_ms * 1e-3) / 1e12
    return {"workload": workload_desc(w), "consumer_ctas": c, "copy_warps": warps, "steps": K,
            "tokens_per_s": round(w.T / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
            "hidden_pct": round(100 * (1 - statistics.median(tails) / copy_alone), 2),
            "hidden_pct_all_bands_copied": round(100 * (1 - statistics.median(tails_all) / copy_alone), 2),
            "copy_alone_ms": round(copy_alone, 4),
            "swiglu_gemm": {"ms": round(up_ms, 4), "achieved_tflops": round(up_tflops, 1),
                            "frac_of_measured_burst_peak": round(up_tflops / peaks["bf16_tflops"], 4)},
            "eager_ms_per_step": {a: round(float(np.median(v.sum(1))), 4) for a, v in st.items()},
            "clocks": dict(clk.summary(), kernel_sm_mhz=kclk)}


# ------------------------------------------------------------------------ CPU oracle timing
def sample_workload(w, tokens: int):
    per = max(1, tokens // w.R)
    return w.replace(T=per * w.R)


def oracle_weights(w, seed, W=None):
    if W is not None:
        return {n: W[n].double().cpu().numpy() for n in ("W1", "W3", "W2")}
    return {n: inputs.make_weight(w, seed, n).double().numpy() for n in ("W1", "W3", "W2")}


def cpu_baseline(w, seed: int, tokens: int, W=None, Wf=None):
    """The oracle (fp64 NumPy) on the first `tokens` tokens of the same workload."""
    from oracle import moe_ref

    ws_ = sample_workload(w, tokens)
    logits = inputs.make_logits(w, seed)[:ws_.T]
    x = inputs.bf16_to_f64(inputs.make_x(w, seed)[:ws_.T])
    Wf = Wf or oracle_weights(w, seed, W)
    t = time.perf_counter()
    moe_ref.moe_layer(logits, x, Wf["W1"], Wf["W3"], Wf["W2"], R=w.R, tbM=w.tile_M, k=w.topk)
    dt = time.perf_counter() - t
    return {"value": round(ws_.T / dt, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {ws_.T} tokens of the {w.name} workload (same d, ffn, E, top-k, R, tile_M, weights), "
                      f"one oracle pass of {dt:.1f} s, float64 NumPy with its default BLAS threads"}


def run_reference(args, rank: int, world: int):
    w = inputs.WORKLOADS[args.workload]
    if rank != 0:
        return None
    tokens = 256
    Wf = oracle_weights(w, args.seed)
    for _ in range(args.warmup):
        cpu_baseline(w, args.seed, tokens, Wf=Wf)
    times = []
    for _ in range(args.steps):
        r = cpu_baseline(w, args.seed, tokens, Wf=Wf)
        times.append(sample_workload(w, tokens).T / r["value"])
    T_s = sample_workload(w, tokens).T
    value = T_s * len(times) / sum(times)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w), "T": w.T, "d": w.d, "ffn": w.ffn, "E": w.E, "topk": w.topk,
                   "R": w.R, "tile_M": w.tile_M, "sample_tokens": T_s},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"each step: the first {T_s} tokens of the {w.name} workload through the "
                                   f"fp64 oracle"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py --impl ours needs a CUDA device")
        res = run_ours(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
