"""Consumer-partition study of the Mixtral-shaped layer on one GB300.

The tile-level signaling page sweeps the consumer SM budget c_CTA from 2 to 24 and reports layer
latency against a GEMM-then-transfer baseline (its Figure 9), the overlap ratio as experts per rank
vary (Figure 4b), and the consumer's copy bandwidth and segment size (mgb). This module measures
the same on one GB300, in three parts (one JSON object per point on stdout, "part" names it):

  layer  for every (T, R, c): the overlapped layer, the GEMM-then-copy layer (the two interleaved
         step by step, so both see the same clocks; times also given in SM clock cycles), the copy
         alone, the exposed copy tail, the hidden fraction, and the GEMM slowdown of taking c SMs
         from the down-projection (its producer span over the span of the same GEMM on all SMs)
  mgb    at T=4096, R=4: hidden fraction and tail against the segment size mgb and c
  copy   the return copy alone on c SMs (moe_copy_only): copy bandwidth against c

  python -m tile_level_copy_gb300.sweep [--parts layer mgb copy] [--tokens 1024 4096 ...]
      [--consumers 4 8 ...] [--owners 2 4 8] [--mgbs 1 2 4] [--copy-ctas 1 2 4 ...]
      [--copy-warps] [--no-pair] [--no-tail-assist]

Both expert GEMMs run on CTA pairs unless --no-pair (the down-projection on pairs needs an even
consumer_ctas and no copy warps, else it runs on single CTAs); tail assist is on unless
--no-tail-assist.
"""
from __future__ import annotations

import argparse
import json
import statistics

import numpy as np
import torch

import tile_level_copy_gb300 as tlc
from tile_level_copy_gb300 import build, inputs


class ClockWatch:
    """Median SM clock (nvidia-smi, every 100 ms) while the block runs."""

    def __enter__(self):
        import subprocess
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(torch.cuda.current_device()), "--query-gpu=clocks.sm",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        return self

    def __exit__(self, *exc):
        self.vals = []
        if self.p is not None:
            self.p.terminate()
            out, _ = self.p.communicate()
            self.vals = [float(v) for v in out.split() if v.replace(".", "", 1).isdigit()]

    def median(self):
        return statistics.median(self.vals) if self.vals else None


def time_arms(arms, args_, ws, steps: int, warmup: int):
    """Eager steps of every arm (name -> (cfg, sequential)) interleaved step by step, each step
    between stage events; returns {name: (median step ms, median stage ms [5])}. Interleaving gives
    every arm the same clock and power conditions."""
    for _ in range(warmup):
        for cfg, seq in arms.values():
            tlc.forward(cfg, *args_, ws, sequential=seq)
    evs = {a: [tlc.stage_events() for _ in range(steps)] for a in arms}
    torch.cuda.synchronize()
    for i in range(steps):
        for a, (cfg, seq) in arms.items():
            tlc.forward(cfg, *args_, ws, sequential=seq, events=evs[a][i])
    torch.cuda.synchronize()
    out = {}
    for a, (cfg, _) in arms.items():
        rc, detail = tlc.status(cfg, ws)
        if rc != tlc.MOE_OK:
            raise RuntimeError(f"device status {rc} ({detail})")
        st = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(tlc.EV_COUNT - 1)] for e in evs[a]])
        out[a] = (float(np.median(st.sum(1))), np.median(st, 0))
    return out


def trace_of(cfg, args_, ws, seq: bool, reps: int = 5):
    """Median over reps of (copy tail after the last flag, down-projection span) in ms."""
    tails, spans = [], []
    for _ in range(reps):
        tlc.forward(cfg, *args_, ws, sequential=seq)
        torch.cuda.synchronize()
        tr = ws.view("trace").cpu().numpy().astype(np.int64)
        tails.append(max(0, int(tr[tlc.TRACE_COPY_END]) - int(tr[tlc.TRACE_GEMM2_END])) / 1e6)
        spans.append((int(tr[tlc.TRACE_GEMM2_END]) - int(tr[tlc.TRACE_GEMM2_START])) / 1e6)
    return statistics.median(tails), statistics.median(spans)


class Setup:
    """Mixtral-shaped weights on the device, inputs per (T, R)."""

    def __init__(self):
        build.build()
        self.dev = torch.device("cuda")
        self.base = inputs.WORKLOADS["mixtral"]
        self.W = {}
        for n in ("W1", "W3", "W2"):
            b = self.base
            shape = (b.E, b.ffn, b.d) if n != "W2" else (b.E, b.d, b.ffn)
            self.W[n] = torch.empty(shape, dtype=torch.bfloat16, device=self.dev)
            inputs.make_weight_into(b, 0, n, self.W[n])

    def layer(self, T, R):
        w = self.base.replace(T=T, R=R)
        logits = torch.from_numpy(inputs.make_logits(w, 0)).to(self.dev)
        x = inputs.make_x(w, 0).to(self.dev)
        out = torch.empty(T, w.d, dtype=torch.float32, device=self.dev)
        return w, (logits, x, self.W["W1"], self.W["W3"], self.W["W2"], out)


def part_layer(S: Setup, a, flags):
    for T in a.tokens:
        for R in a.owners:
            w, args_ = S.layer(T, R)
            ws = tlc.Workspace(tlc.Config.from_workload(w, consumer_ctas=8, flags=flags), S.dev)
            for c in a.consumers:
                cfg = tlc.Config.from_workload(w, consumer_ctas=c, flags=flags)
                with ClockWatch() as clk:  # sequential and overlapped interleaved step by step
                    r = time_arms({"seq": (cfg, True), "ovl": (cfg, False)}, args_, ws, a.steps, a.warmup)
                (seq_ms, seq_st), (ovl_ms, _) = r["seq"], r["ovl"]
                copy_ms = float(seq_st[tlc.EV_DOWN])
                tail, span_ovl = trace_of(cfg, args_, ws, False)
                _, span_seq = trace_of(cfg, args_, ws, True)
                mhz = clk.median()
                print(json.dumps({"part": "layer", "T": T, "R": R, "consumer_ctas": c,
                                  "copy_warps": bool(flags & tlc.MOE_COPY_WARPS),
                                  "pair_umma": bool(flags & tlc.MOE_PAIR_UMMA),
                                  "direct_tail": bool(flags & tlc.MOE_DIRECT_TAIL),
                                  "overlapped_ms": round(ovl_ms, 4), "sequential_ms": round(seq_ms, 4),
                                  "copy_alone_ms": round(copy_ms, 4), "tail_ms": round(tail, 4),
                                  "hidden_pct": round(100 * (1 - tail / copy_ms), 2),
                                  "speedup": round(seq_ms / ovl_ms, 4),
                                  "gemm_span_overlapped_ms": round(span_ovl, 4),
                                  "gemm_span_all_sms_ms": round(span_seq, 4),
                                  "gemm_slowdown": round(span_ovl / span_seq, 4),
                                  "tokens_per_s": round(T / ovl_ms * 1e3, 1), "sm_mhz": mhz,
                                  "overlapped_mcycles": round(ovl_ms * mhz / 1e3, 3) if mhz else None,
                                  "sequential_mcycles": round(seq_ms * mhz / 1e3, 3) if mhz else None}),
                      flush=True)
            del ws


def part_mgb(S: Setup, a, flags):
    w, args_ = S.layer(4096, 4)
    ws = tlc.Workspace(tlc.Config.from_workload(w, consumer_ctas=8, flags=flags, mgb=max(a.mgbs)), S.dev)
    for mgb in a.mgbs:
        for c in a.consumers:
            cfg = tlc.Config.from_workload(w, consumer_ctas=c, flags=flags, mgb=mgb)
            r = time_arms({"seq": (cfg, True), "ovl": (cfg, False)}, args_, ws, a.steps, a.warmup)
            (_, seq_st), (ovl_ms, _) = r["seq"], r["ovl"]
            tail, _ = trace_of(cfg, args_, ws, False)
            copy_ms = float(seq_st[tlc.EV_DOWN])
            print(json.dumps({"part": "mgb", "T": 4096, "R": 4, "mgb": mgb, "consumer_ctas": c,
                              "overlapped_ms": round(ovl_ms, 4), "copy_alone_ms": round(copy_ms, 4),
                              "tail_ms": round(tail, 4), "hidden_pct": round(100 * (1 - tail / copy_ms), 2)}),
                  flush=True)


def part_copy(S: Setup, a):
    w, args_ = S.layer(4096, 4)
    cfg = tlc.Config.from_workload(w, consumer_ctas=8)
    ws = tlc.Workspace(cfg, S.dev)
    tlc.forward(cfg, *args_, ws, sequential=True)  # plan and Yp in the workspace
    nbytes = 2 * w.T * w.topk * w.d * 2              # every real row read from Yp and written to Ret
    sms, _ = tlc.device_info()
    for c in a.copy_ctas:
        if c > sms:
            continue
        for _ in range(a.warmup):
            tlc.copy_only(cfg, ws, c)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(a.steps):
            t0.record()
            tlc.copy_only(cfg, ws, c)
            t1.record()
            torch.cuda.synchronize()
            times.append(t0.elapsed_time(t1))
        rc, detail = tlc.status(cfg, ws)
        if rc != tlc.MOE_OK:
            raise RuntimeError(f"device status {rc} ({detail})")
        ms = statistics.median(times)
        print(json.dumps({"part": "copy", "T": 4096, "R": 4, "ctas": c, "copy_ms": round(ms, 4),
                          "bytes": nbytes, "gb_per_s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                          "gb_per_s_per_sm": round(nbytes / (ms * 1e-3) / 1e9 / c, 2)}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--parts", nargs="+", default=["layer", "mgb", "copy"], choices=["layer", "mgb", "copy"])
    ap.add_argument("--tokens", type=int, nargs="+", default=[1024, 4096, 16384, 32768])
    ap.add_argument("--consumers", type=int, nargs="+", default=[4, 8, 16, 24, 32])
    ap.add_argument("--owners", type=int, nargs="+", default=[2, 4, 8])
    ap.add_argument("--mgbs", type=int, nargs="+", default=[1, 2, 4])
    ap.add_argument("--copy-ctas", type=int, nargs="+", default=[1, 2, 4, 8, 16, 24, 32, 64, 152])
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--no-tail-assist", action="store_true")
    ap.add_argument("--copy-warps", action="store_true", help="also run copy warps in the producer CTAs")
    ap.add_argument("--no-pair", action="store_true", help="single-CTA GEMMs instead of CTA pairs")
    ap.add_argument("--direct-tail", action="store_true",
                    help="the down-projection's epilogue returns the last wave's bands itself")
    a = ap.parse_args()

    flags = (0 if a.no_tail_assist else tlc.MOE_TAIL_ASSIST) | (tlc.MOE_COPY_WARPS if a.copy_warps else 0) | \
        (0 if a.no_pair else tlc.MOE_PAIR_UMMA) | (tlc.MOE_DIRECT_TAIL if a.direct_tail else 0)
    S = Setup()
    if "copy" in a.parts:
        part_copy(S, a)
    if "mgb" in a.parts:
        part_mgb(S, a, flags)
    if "layer" in a.parts:
        part_layer(S, a, flags)


if __name__ == "__main__":
    main()
