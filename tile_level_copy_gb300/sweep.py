"""Consumer-partition sweep of the Mixtral-shaped layer (tokens x consumer CTAs x owners).

The tile-level signaling page sweeps the consumer SM budget c_CTA from 2 to 24 and reports layer
latency against a GEMM-then-transfer baseline (its Figure 9) and the overlap ratio as experts per
rank vary (Figure 4b). This module measures the same on one GB300: for every (T, c, R) the
overlapped layer, the sequential layer, the copy alone, the exposed copy tail and the hidden
fraction. One JSON object per point on stdout.

  python -m tile_level_copy_gb300.sweep [--tokens 1024 4096 ...] [--consumers 4 8 ...] [--owners 2 4 8]
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


def time_steps(cfg, args_, ws, seq: bool, steps: int, warmup: int):
    for _ in range(warmup):
        tlc.forward(cfg, *args_, ws, sequential=seq)
    evs = [tlc.stage_events() for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        tlc.forward(cfg, *args_, ws, sequential=seq, events=evs[i])
    torch.cuda.synchronize()
    rc, detail = tlc.status(cfg, ws)
    if rc != tlc.MOE_OK:
        raise RuntimeError(f"device status {rc} ({detail})")
    st = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(tlc.EV_COUNT - 1)] for e in evs])
    return float(np.median(st.sum(1))), np.median(st, 0)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--tokens", type=int, nargs="+", default=[1024, 4096, 16384, 32768])
    ap.add_argument("--consumers", type=int, nargs="+", default=[4, 8, 16, 24, 32])
    ap.add_argument("--owners", type=int, nargs="+", default=[2, 4, 8])
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--no-tail-assist", action="store_true")
    a = ap.parse_args()

    build.build()
    dev = torch.device("cuda")
    base = inputs.WORKLOADS["mixtral"]
    W = {}
    for n in ("W1", "W3", "W2"):
        shape = (base.E, base.ffn, base.d) if n != "W2" else (base.E, base.d, base.ffn)
        W[n] = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        inputs.make_weight_into(base, 0, n, W[n])
    flags = 0 if a.no_tail_assist else tlc.MOE_TAIL_ASSIST
    for T in a.tokens:
        out = torch.empty(T, base.d, dtype=torch.float32, device=dev)
        for R in a.owners:
            w = base.replace(T=T, R=R)
            logits = torch.from_numpy(inputs.make_logits(w, 0)).to(dev)
            x = inputs.make_x(w, 0).to(dev)
            cfg0 = tlc.Config.from_workload(w, consumer_ctas=8, flags=flags)
            ws = tlc.Workspace(cfg0, dev)
            args_ = (logits, x, W["W1"], W["W3"], W["W2"], out)
            for c in a.consumers:
                cfg = tlc.Config.from_workload(w, consumer_ctas=c, flags=flags)
                # sequential and overlapped measured in alternation, so both see the same clocks
                seqs, ovls, copies = [], [], []
                with ClockWatch() as clk:
                    for _ in range(2):
                        seq_ms, seq_st = time_steps(cfg, args_, ws, True, a.steps, a.warmup)
                        ovl_ms, _ = time_steps(cfg, args_, ws, False, a.steps, a.warmup)
                        seqs.append(seq_ms)
                        ovls.append(ovl_ms)
                        copies.append(float(seq_st[tlc.EV_DOWN]))
                seq_ms, ovl_ms, copy_ms = min(seqs), min(ovls), statistics.median(copies)
                tails = []
                for _ in range(5):
                    tlc.forward(cfg, *args_, ws)
                    torch.cuda.synchronize()
                    tr = ws.view("trace").cpu().numpy().astype(np.int64)
                    tails.append(max(0, int(tr[tlc.TRACE_COPY_END]) - int(tr[tlc.TRACE_GEMM2_END])) / 1e6)
                tail = statistics.median(tails)
                print(json.dumps({"T": T, "R": R, "consumer_ctas": c, "tail_assist": not a.no_tail_assist,
                                  "overlapped_ms": round(ovl_ms, 4), "sequential_ms": round(seq_ms, 4),
                                  "copy_alone_ms": round(copy_ms, 4), "tail_ms": round(tail, 4),
                                  "hidden_pct": round(100 * (1 - tail / copy_ms), 2),
                                  "speedup": round(seq_ms / ovl_ms, 4),
                                  "tokens_per_s": round(T / ovl_ms * 1e3, 1), "sm_mhz": clk.median()}), flush=True)
            del ws


if __name__ == "__main__":
    main()
