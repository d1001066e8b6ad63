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

    Each expert's rows contiguous (its groups in owner order, each group's rows in plan order), each
    expert's run padded to a multiple of the 128-row UMMA tile. Returns (cbase [E], ccoff [E*R],
    cslot [T, k], PC)."""
    E, R, T = plan.E, plan.R, plan.T
    n = plan.n.astype(np.int64)
    runs = -(-n.sum(1) // 128) * 128
    cbase = np.concatenate([[0], np.cumsum(runs)])[:E]
    before = np.concatenate([np.zeros((E, 1), np.int64), np.cumsum(n, 1)[:, :-1]], 1)
    ccoff = (cbase[:, None] + before).reshape(-1)
    g = np.asarray(idx, np.int64) * R + moe_ref.owners(T, R)[:, None]
    cslot = ccoff[g] + (plan.slot - plan.off[g])
    return cbase, ccoff, cslot, int(runs.sum())


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
