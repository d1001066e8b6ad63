"""Shared helpers of the GPU parity tests: seeded inputs on the device and oracle results."""
import functools

import numpy as np
import torch

import tile_level_copy_gb300 as tlc
from oracle import moe_ref
from tile_level_copy_gb300 import inputs

# Float parity bar of the layer output against the fp64 oracle.
MAX_ABS = 2e-2
REL_L2 = 5e-3


def small(name: str, **kw) -> inputs.Workload:
    """Reduced shapes of the four workloads that the fp64 oracle finishes in about a second."""
    base = {
        "tiny": dict(),
        "mixtral": dict(T=1024, d=1024, ffn=2048),
        "skew": dict(T=2048, d=512, ffn=1024),
        "fine": dict(T=2048, d=256, ffn=384),
    }[name]
    w = inputs.WORKLOADS[name].replace(**base)
    return w.replace(name=name + "-small", **kw)


class Layer:
    """Inputs of one workload on the GPU plus a workspace."""

    def __init__(self, w: inputs.Workload, seed: int, cfg_kw=None, host_weights=True):
        self.w, self.seed = w, seed
        self.cfg = tlc.Config.from_workload(w, **(cfg_kw or {}))
        dev = torch.device("cuda")
        self.logits_np = inputs.make_logits(w, seed)
        self.x_cpu = inputs.make_x(w, seed)
        self.logits = torch.from_numpy(self.logits_np).to(dev)
        self.x = self.x_cpu.to(dev)
        self.W = {}
        for n in ("W1", "W3", "W2"):
            shape = (w.E, w.ffn, w.d) if n != "W2" else (w.E, w.d, w.ffn)
            t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
            inputs.make_weight_into(w, seed, n, t)
            self.W[n] = t
        self.ws = tlc.Workspace(self.cfg, dev)
        self.out = torch.empty(w.T, w.d, dtype=torch.float32, device=dev)

    def run(self, sequential=False, cfg=None):
        cfg = cfg or self.cfg
        tlc.forward(cfg, self.logits, self.x, self.W["W1"], self.W["W3"], self.W["W2"], self.out, self.ws,
                    sequential=sequential)
        rc, detail = tlc.status(cfg, self.ws)
        assert rc == tlc.MOE_OK, (rc, detail, tlc.lib().moe_last_error())
        return self.out.clone()

    def weights_f64(self, e):
        return tuple(self.W[n][e].double().cpu().numpy() for n in ("W1", "W3", "W2"))

    def oracle_layer(self):
        w = self.w
        return moe_ref.moe_layer(self.logits_np, inputs.bf16_to_f64(self.x_cpu),
                                 self.W["W1"].double().cpu().numpy(), self.W["W3"].double().cpu().numpy(),
                                 self.W["W2"].double().cpu().numpy(), R=w.R, tbM=w.tile_M, mgb=self.cfg.mgb,
                                 k=w.topk)


def compact_layout(plan: moe_ref.Plan, idx: np.ndarray):
    """Expected expert-compact layout of the GEMM inputs for an oracle plan.

    Each expert's rows contiguous, its run padded to a multiple of the 128-row UMMA tile; inside the
    run the expert's bands follow one another in hand-out order (plan.order), each band's valid rows
    in row order. Returns (cbase [E], tile_crow [MT], cslot [T, k], yrow [PC], PC): the run starts,
    the compact row of each band's first row, the compact row of every pair and the padded (Yp) row
    of every compact row (-1 for the rows that pad a run)."""
    E, tbM = plan.E, plan.tbM
    runs = -(-plan.n.sum(1).astype(np.int64) // 128) * 128
    cbase = np.concatenate([[0], np.cumsum(runs)])[:E]
    tile_crow = np.zeros(plan.num_tiles, np.int64)
    fill = cbase.copy()
    for m in plan.order.tolist():
        e, valid = int(plan.tiles[m, 0]), int(plan.tiles[m, 3])
        tile_crow[m] = fill[e]
        fill[e] += valid
    slot = plan.slot.astype(np.int64)
    cslot = tile_crow[slot // tbM] + slot % tbM  # band m holds padded rows m*tbM .. m*tbM + valid - 1
    PC = int(runs.sum())
    yrow = np.full(PC, -1, np.int64)
    yrow[cslot.reshape(-1)] = slot.reshape(-1)
    return cbase, tile_crow, cslot, yrow, PC


def parity(got: np.ndarray, want: np.ndarray):
    err = np.abs(got - want)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    return float(err.max()), float(rel)


def per_token_rel_distance(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Per-token relative distance ||got_t - want_t|| / ||want_t|| (the page's correctness metric)."""
    return np.linalg.norm(got - want, axis=1) / np.maximum(np.linalg.norm(want, axis=1), 1e-30)


@functools.lru_cache(maxsize=8)
def plan_oracle(name: str, seed: int, mgb: int):
    w = inputs.WORKLOADS[name]
    logits = inputs.make_logits(w, seed)
    idx, gate = moe_ref.route_topk(logits, w.topk)
    return idx, gate, moe_ref.build_plan(idx, w.E, w.R, w.tile_M, mgb)


def check_flag_counts(L: "Layer", plan: moe_ref.Plan):
    """After an overlapped run: every tile flag holds its band's valid rows (each stored row counted
    once per N tile) and every band counter valid rows x N tiles."""
    MT, n2 = plan.num_tiles, L.ws.layout["n_tiles_n2"]
    valid = torch.from_numpy(plan.tiles[:, 3].astype(np.int32)).to(L.ws.view("flags").device)
    flags = L.ws.view("flags").reshape(-1)[:MT * n2].reshape(MT, n2)
    assert torch.all(flags == valid[:, None]), "tile flags"
    assert torch.all(L.ws.view("bands")[:MT] == valid * n2), "band counters"

