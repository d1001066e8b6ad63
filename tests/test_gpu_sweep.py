"""The Mixtral-shaped sweep: tokens x consumer partition x owners.

T in {1024, 4096, 16384, 32768}, consumer CTAs in {4, 8, 16, 24, 32}, R in {2, 4, 8}, on the
Mixtral-shaped layer (d=4096, ffn=14336, E=8, top-2, tile_M=128) with the same seeded
distributions. For every point the overlapped path must equal the GEMM-then-copy path bitwise and
the device status must be clean; at each T, 16 sampled tokens are checked against the oracle's
per-token definition.
"""
import numpy as np
import pytest
import torch

import tile_level_copy_gb300 as tlc
from oracle import moe_ref
from tile_level_copy_gb300 import inputs
from tests.gpu_util import MAX_ABS, REL_L2, parity

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BASE = inputs.WORKLOADS["mixtral"]
TOKENS = (1024, 4096, 16384, 32768)
CONSUMERS = (4, 8, 16, 24, 32)
OWNERS = (2, 4, 8)


@pytest.fixture(scope="module")
def weights():
    dev = torch.device("cuda")
    W = {}
    for n in ("W1", "W3", "W2"):
        shape = (BASE.E, BASE.ffn, BASE.d) if n != "W2" else (BASE.E, BASE.d, BASE.ffn)
        W[n] = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        inputs.make_weight_into(BASE, 0, n, W[n])
    return W


def expert_f64(W):
    return lambda e: tuple(W[n][e].double().cpu().numpy() for n in ("W1", "W3", "W2"))


@pytest.mark.parametrize("T", TOKENS)
def test_sweep_overlapped_equals_sequential(weights, T):
    dev = torch.device("cuda")
    out = torch.empty(T, BASE.d, dtype=torch.float32, device=dev)
    checked = False
    for R in OWNERS:
        w = BASE.replace(T=T, R=R)
        logits_np = inputs.make_logits(w, 0)
        logits = torch.from_numpy(logits_np).to(dev)
        x_cpu = inputs.make_x(w, 0)
        x = x_cpu.to(dev)
        base_cfg = tlc.Config.from_workload(w, consumer_ctas=8)
        ws = tlc.Workspace(base_cfg, dev)
        tlc.forward(base_cfg, logits, x, weights["W1"], weights["W3"], weights["W2"], out, ws, sequential=True)
        assert tlc.status(base_cfg, ws)[0] == tlc.MOE_OK
        want = out.clone()
        for c in CONSUMERS:
            for flags in (0, tlc.MOE_TAIL_ASSIST, tlc.MOE_TAIL_ASSIST | tlc.MOE_COPY_WARPS,
                          tlc.MOE_PAIR_UMMA | tlc.MOE_TAIL_ASSIST | tlc.MOE_DIRECT_TAIL):
                cfg = tlc.Config.from_workload(w, consumer_ctas=c, flags=flags)
                out.zero_()
                tlc.forward(cfg, logits, x, weights["W1"], weights["W3"], weights["W2"], out, ws)
                rc, detail = tlc.status(cfg, ws)
                assert rc == tlc.MOE_OK, (T, R, c, flags, rc, detail)
                assert torch.equal(out, want), (T, R, c, flags)
        cfg = tlc.Config.from_workload(w, consumer_ctas=0, flags=tlc.MOE_TAIL_ASSIST | tlc.MOE_COPY_WARPS)
        out.zero_()
        tlc.forward(cfg, logits, x, weights["W1"], weights["W3"], weights["W2"], out, ws)
        assert tlc.status(cfg, ws)[0] == tlc.MOE_OK and torch.equal(out, want), (T, R, 0)
        if not checked:  # sampled tokens against the oracle once per T
            rng = np.random.default_rng(T)
            tokens = np.sort(rng.choice(T, size=16, replace=False))
            x_rows = inputs.bf16_to_f64(x_cpu[tokens])
            _, _, ref = moe_ref.moe_tokens(tokens, logits_np, x_rows, expert_f64(weights), w.topk)
            err, rel = parity(want.double().cpu().numpy()[tokens], ref)
            assert err <= MAX_ABS and rel <= REL_L2, (T, err, rel)
            checked = True
