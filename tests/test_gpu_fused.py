"""Both expert GEMMs in one launch (MOE_FUSED_GEMMS) on CTA pairs.

The SwiGLU tiles are handed out first; an expert's down-projection tiles start once every SwiGLU
tile quarter of the expert has published (stores complete, async proxy fenced, release count), and
the consumer clusters take SwiGLU tiles before they copy. Bar: Hc, Yp, Ret and the layer output
bitwise equal to the separate launches on the same inputs (the same tile code computes every
element), every expert's published count complete, the tile flags and band counters complete;
a stopped pipeline is reported and the context stays usable.
"""
import numpy as np
import pytest
import torch

import tile_level_copy_gb300 as tlc
from oracle import moe_ref
from tile_level_copy_gb300 import inputs
from tests.gpu_util import MAX_ABS, REL_L2, Layer, check_flag_counts, parity, small

pytestmark = pytest.mark.gpu

PAIR, TA, DT, FG = tlc.MOE_PAIR_UMMA, tlc.MOE_TAIL_ASSIST, tlc.MOE_DIRECT_TAIL, tlc.MOE_FUSED_GEMMS


def compare(L: Layer, flags, consumers):
    cfg = tlc.Config.from_workload(L.w, consumer_ctas=consumers, flags=flags, timeout_us=500000)
    want = L.run(sequential=False, cfg=cfg)
    PC = int(L.ws.view("meta")[9].item())
    P = int(L.ws.view("meta")[0].item())
    hc, ret = L.ws.view("Hc")[:PC].clone(), L.ws.view("Ret").clone()
    for n in ("Hc", "Ret"):
        L.ws.view(n).zero_()
    got = L.run(sequential=False, cfg=tlc.Config.from_workload(L.w, consumer_ctas=consumers, flags=flags | FG,
                                                                timeout_us=500000))
    assert torch.equal(got, want)
    assert torch.equal(L.ws.view("Hc")[:PC], hc)
    assert torch.equal(L.ws.view("Ret"), ret)
    if L.w.d % 256 == 0:  # the fused launch ran: every expert's SwiGLU quarters published
        experts = L.ws.view("experts").cpu().numpy()
        want_x = (experts[:, 4] + 1) // 2 * (L.w.ffn // 128) * 8
        np.testing.assert_array_equal(L.ws.view("xready").cpu().numpy(), want_x)
        idx, _ = moe_ref.route_topk(L.logits_np, L.w.topk)
        check_flag_counts(L, moe_ref.build_plan(idx, L.w.E, L.w.R, L.w.tile_M, L.cfg.mgb))
    return P


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
@pytest.mark.parametrize("flags,consumers", [(PAIR | TA, 4), (PAIR, 2), (PAIR | TA | DT, 8)],
                         ids=["assist-c4", "c2", "assist-direct-c8"])
def test_fused_gemms_equal_separate_launches(name, flags, consumers):
    compare(Layer(small(name), seed=5), flags, consumers)


@pytest.mark.parametrize("name", ["mixtral", "skew"])
def test_fused_gemms_full_size_in_the_bench_configuration(name):
    import bench
    c, warps = bench.DEFAULT_COPY[name]
    compare(Layer(inputs.WORKLOADS[name], seed=1), bench.default_flags(warps), c)


@pytest.mark.parametrize("seed", range(8))
def test_fused_gemms_checksum_falsifier(seed):
    """Every returned row equals the row the fused launch's producers computed, over seeds, small
    consumer partitions, segments of 1-2 bands, with and without the direct tail."""
    w = inputs.WORKLOADS["skew"].replace(T=2048, d=256, ffn=384)
    L = Layer(w, seed=seed, cfg_kw=dict(consumer_ctas=2 + 2 * (seed % 3), mgb=1 + seed % 2,
                                        flags=PAIR | FG | (TA if seed % 2 else 0) | (DT if seed % 3 == 0 else 0)))
    got = L.run(sequential=False)
    seq = L.run(sequential=True)
    assert torch.equal(got, seq)


def test_fused_gemms_layer_matches_oracle():
    w = small("mixtral")
    L = Layer(w, seed=8, cfg_kw=dict(consumer_ctas=4, flags=PAIR | TA | DT | FG))
    ref = L.oracle_layer()
    err, rel = parity(L.run(sequential=False).double().cpu().numpy(), ref.out)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)


@pytest.mark.parametrize("hook", [tlc.MOE_TEST_STALL_PIPE0, tlc.MOE_TEST_STALL_PIPE1], ids=["rank0", "rank1"])
def test_fused_gemms_abort_settles_and_context_survives(hook):
    w = small("mixtral")
    L = Layer(w, seed=0)
    want = L.run(sequential=True)
    cfg = tlc.Config.from_workload(w, consumer_ctas=4, flags=PAIR | FG | hook, timeout_us=20000)
    tlc.forward(cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws)
    assert tlc.status(cfg, L.ws)[0] == tlc.MOE_ERR_TIMEOUT
    ok = tlc.Config.from_workload(w, consumer_ctas=4, flags=PAIR | FG | TA)
    assert torch.equal(L.run(sequential=False, cfg=ok), want)
