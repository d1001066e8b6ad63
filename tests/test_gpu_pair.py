"""The SwiGLU GEMM on CTA pairs (MOE_PAIR_UMMA: tcgen05 cta_group::2, UMMA 256 x 256 over two SMs).

Bar: the SwiGLU hidden rows Hc and the layer output within the fp64 oracle's tolerance (max-abs
2e-2, relative L2 5e-3); the pair path's Hc equal, bit for bit, to the single-CTA path's on the same
inputs (both accumulate each output element over K in the same 16-wide steps); clean device status.
Shapes include experts with an odd number of work items (the pair's odd CTA then has no rows).
"""
import numpy as np
import pytest
import torch

import tile_level_copy_gb300 as tlc
from oracle import moe_ref
from tile_level_copy_gb300 import inputs
from tests.gpu_util import MAX_ABS, REL_L2, Layer, parity, small

pytestmark = pytest.mark.gpu

PAIR = tlc.MOE_PAIR_UMMA


def odd_item_experts(L: Layer) -> int:
    """Experts whose number of GEMM work items is odd (counted from the device plan)."""
    experts = L.ws.view("experts").cpu().numpy().reshape(-1, 8)
    return int(np.sum(experts[:L.w.E, 4] % 2 == 1))


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
def test_pair_matches_oracle_and_single_cta(name):
    w = small(name)
    L = Layer(w, seed=3, cfg_kw=dict(consumer_ctas=8, timeout_us=200000))
    single = L.run(sequential=True)
    hc_single = L.ws.view("Hc")[:].clone()
    cfg = tlc.Config.from_workload(w, consumer_ctas=8, flags=PAIR, timeout_us=200000)
    L.ws.view("Hc").zero_()
    got = L.run(sequential=True, cfg=cfg)
    ref = L.oracle_layer()
    rows = ref.plan.slot.reshape(-1)
    crows = torch.from_numpy(L.ws.view("cslot").cpu().numpy().reshape(-1)).long().cuda()
    _, hrel = parity(L.ws.view("Hc")[crows].double().cpu().numpy(), ref.Hp[rows])
    assert hrel <= 5e-3, hrel
    err, rel = parity(got.double().cpu().numpy(), ref.out)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
    PC = int(L.ws.view("meta")[9].item())  # every compact row, padding included, is computed by both paths
    assert torch.equal(L.ws.view("Hc")[:PC], hc_single[:PC])
    assert torch.equal(got, single)


def test_pair_covers_odd_item_counts():
    """Seeds until an expert with an odd number of work items appears, then checks it bitwise."""
    w = small("skew")
    for seed in range(20):
        L = Layer(w, seed=seed, cfg_kw=dict(consumer_ctas=8, timeout_us=200000))
        single = L.run(sequential=True)
        if odd_item_experts(L) == 0:
            continue
        cfg = tlc.Config.from_workload(w, consumer_ctas=8, flags=PAIR, timeout_us=200000)
        assert torch.equal(L.run(sequential=True, cfg=cfg), single)
        return
    pytest.fail("no seed gave an expert with an odd number of work items")


@pytest.mark.parametrize("flags", [PAIR, PAIR | tlc.MOE_TAIL_ASSIST, PAIR | tlc.MOE_COPY_WARPS])
def test_pair_with_overlapped_down_projection(flags):
    w = small("mixtral")
    L = Layer(w, seed=4)
    want = L.run(sequential=True)
    cfg = tlc.Config.from_workload(w, consumer_ctas=0 if flags & tlc.MOE_COPY_WARPS else 4, flags=flags)
    assert torch.equal(L.run(sequential=False, cfg=cfg), want)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral", "skew", "fine"])
def test_pair_full_size_sampled_tokens(name):
    w = inputs.WORKLOADS[name]
    L = Layer(w, seed=0, cfg_kw=dict(consumer_ctas=8, flags=tlc.MOE_TAIL_ASSIST))
    single = L.run(sequential=False)
    cfg = tlc.Config.from_workload(w, consumer_ctas=8, flags=tlc.MOE_TAIL_ASSIST | PAIR)
    got = L.run(sequential=False, cfg=cfg)
    assert torch.equal(got, single)
    rng = np.random.default_rng(11)
    tokens = np.sort(rng.choice(w.T, size=32, replace=False))
    x_rows = inputs.bf16_to_f64(L.x_cpu[tokens])
    _, _, want = moe_ref.moe_tokens(tokens, L.logits_np, x_rows, L.weights_f64, w.topk)
    err, rel = parity(got.double().cpu().numpy()[tokens], want)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
