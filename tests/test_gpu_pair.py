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
from tests.gpu_util import MAX_ABS, REL_L2, Layer, check_flag_counts, parity, small

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


@pytest.mark.parametrize("name,consumers", [("mixtral", 4), ("mixtral", 24), ("skew", 8), ("mixtral", 2)])
@pytest.mark.parametrize("direct", [False, True])
def test_adaptive_consumer_partition(name, consumers, direct):
    """MOE_ADAPTIVE_CONSUMERS: the pair down-projection sets its producer pairs from its tile count
    (the fewest that finish in the fewest waves a partition with a consumer pair allows), whatever
    consumer_ctas says; the result stays bitwise equal to the GEMM-then-copy path and every band
    completes."""
    w = small(name)
    L = Layer(w, seed=3)
    want = L.run(sequential=True)
    ret_seq = L.ws.view("Ret").clone()
    flags = PAIR | tlc.MOE_TAIL_ASSIST | tlc.MOE_ADAPTIVE_CONSUMERS | (tlc.MOE_DIRECT_TAIL if direct else 0)
    cfg = tlc.Config.from_workload(w, consumer_ctas=consumers, flags=flags)
    L.ws.view("Ret").zero_()
    assert torch.equal(L.run(sequential=False, cfg=cfg), want)
    assert torch.equal(L.ws.view("Ret"), ret_seq)
    idx, _ = moe_ref.route_topk(L.logits_np, w.topk)
    check_flag_counts(L, moe_ref.build_plan(idx, w.E, w.R, w.tile_M, cfg.mgb))
    # the producer count the kernel chose, against the rule on the plan's item counts (the pair
    # grid is one cluster of two per two SMs)
    items = L.ws.view("experts").cpu().numpy()[:, 4]
    tiles = int(np.sum((items + 1) // 2)) * L.ws.layout["n_tiles_n2"]
    pairs = tlc.device_info()[0] // 2
    w_min = -(-tiles // (pairs - 1))
    assert int(L.ws.view("meta")[10].item()) == 2 * (-(-tiles // w_min))


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


# ---- the down-projection on CTA pairs (d % 256 == 0, even consumer_ctas, no copy warps) ----------

def check_ret_is_copy_of_yp(L: Layer, plan):
    Yp = L.ws.view("Yp").view(torch.int16)
    Ret = L.ws.view("Ret").view(torch.int16)
    slot = torch.from_numpy(plan.slot.reshape(-1)).long().cuda()
    rslot = torch.from_numpy(plan.ret_slot.reshape(-1)).long().cuda()
    assert torch.equal(Ret[rslot], Yp[slot])


def down_items_per_expert(L: Layer) -> np.ndarray:
    """Down-projection work items of each expert (schedule order), from the device plan."""
    experts = L.ws.view("experts").cpu().numpy().reshape(-1, 8)[:L.w.E]
    items = int(L.ws.view("meta")[7].item())
    first = np.sort(experts[:, 6])
    return np.diff(np.append(first, items))


@pytest.mark.parametrize("name,tile_M", [("mixtral", 128), ("skew", 128), ("skew", 64), ("fine", 128)])
@pytest.mark.parametrize("consumers", [2, 8])
def test_pair_down_projection_matches_single_cta(name, tile_M, consumers):
    """The pair down-projection's owner-aligned output rows Yp, return buffer and layer output equal the
    single-CTA kernel's bit for bit (same 16-wide K steps per element), overlapped and sequential;
    every tile flag and band counter is complete. tile_M = 64 makes every band a half band, so the
    pairs' items are two 64-row boxes each."""
    w = small(name, tile_M=tile_M)
    assert w.d % 256 == 0
    L = Layer(w, seed=5, cfg_kw=dict(consumer_ctas=consumers, flags=tlc.MOE_TAIL_ASSIST, timeout_us=200000))
    single = L.run(sequential=True)
    yp_single = L.ws.view("Yp").clone()
    P = int(L.ws.view("meta")[0].item())
    ref = L.oracle_layer()
    rows = torch.from_numpy(ref.plan.slot.reshape(-1)).long().cuda()
    for seq in (False, True):
        cfg = tlc.Config.from_workload(w, consumer_ctas=consumers, flags=PAIR | tlc.MOE_TAIL_ASSIST,
                                       timeout_us=200000)
        L.ws.view("Yp").zero_()
        got = L.run(sequential=seq, cfg=cfg)
        assert torch.equal(got, single)
        assert torch.equal(L.ws.view("Yp")[rows], yp_single[rows])
        check_ret_is_copy_of_yp(L, ref.plan)
        if not seq:
            check_flag_counts(L, ref.plan)
    assert P == ref.plan.P
    err, rel = parity(got.double().cpu().numpy(), ref.out)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)


def test_pair_down_covers_odd_item_counts():
    """Seeds until an expert has an odd number of down-projection items (its last pair has an idle
    half), then checks the pair kernel bitwise against the single-CTA one."""
    w = small("skew")
    for seed in range(20):
        L = Layer(w, seed=seed, cfg_kw=dict(consumer_ctas=4, flags=tlc.MOE_TAIL_ASSIST))
        single = L.run(sequential=False)
        if not np.any(down_items_per_expert(L) % 2 == 1):
            continue
        cfg = tlc.Config.from_workload(w, consumer_ctas=4, flags=PAIR | tlc.MOE_TAIL_ASSIST)
        assert torch.equal(L.run(sequential=False, cfg=cfg), single)
        return
    pytest.fail("no seed gave an expert with an odd number of down-projection items")


@pytest.mark.parametrize("seed", range(24))
def test_pair_down_tile_checksum_falsifier(seed):
    """The page's falsifier (every copied row equals the stored row) for the pair kernel's flags:
    small consumer partitions (2-6 CTAs), tail assist on half the seeds, segments of 1-2 bands."""
    w = inputs.WORKLOADS["skew"].replace(T=1024, d=256, ffn=256)
    L = Layer(w, seed=seed, cfg_kw=dict(consumer_ctas=2 + 2 * (seed % 3), mgb=1 + seed % 2,
                                        flags=PAIR | (tlc.MOE_TAIL_ASSIST if seed % 2 else 0)))
    L.run(sequential=False)
    idx, _ = moe_ref.route_topk(L.logits_np, w.topk)
    plan = moe_ref.build_plan(idx, w.E, w.R, w.tile_M, L.cfg.mgb)
    check_ret_is_copy_of_yp(L, plan)


def test_pair_down_stalled_consumer_times_out_and_context_survives():
    """Consumers of the pair kernel wait for a flag value that no producer writes: the bounded wait
    runs out, the status says so, and the next call is correct."""
    w = small("skew")
    L = Layer(w, seed=0)
    want = L.run(sequential=True)
    cfg = tlc.Config.from_workload(w, consumer_ctas=4, flags=PAIR | tlc.MOE_TEST_STALL_CONSUMER, timeout_us=20000)
    tlc.forward(cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws)
    rc, _ = tlc.status(cfg, L.ws)
    assert rc == tlc.MOE_ERR_TIMEOUT
    cfg_ok = tlc.Config.from_workload(w, consumer_ctas=4, flags=PAIR)
    assert torch.equal(L.run(sequential=False, cfg=cfg_ok), want)


@pytest.mark.parametrize("hook", [tlc.MOE_TEST_STALL_PIPE0, tlc.MOE_TEST_STALL_PIPE1], ids=["rank0", "rank1"])
@pytest.mark.parametrize("sequential", [False, True])
def test_pair_pipeline_abort_settles_loads_and_context_survives(hook, sequential):
    """One CTA of every pair stops issuing its TMA loads halfway through its first tile (rank 0: its
    peer runs up to a ring of stages ahead; rank 1: rank 0 arms stages whose peer bytes never come).
    The pair's bounded waits run out, the status says so, the abort path settles every load still in
    flight before either CTA leaves, and the next call on the same context is correct."""
    w = small("mixtral")  # d % 256 == 0: both GEMMs run on CTA pairs
    L = Layer(w, seed=0)
    want = L.run(sequential=True)
    cfg = tlc.Config.from_workload(w, consumer_ctas=4, flags=PAIR | hook, timeout_us=20000)
    tlc.forward(cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws, sequential=sequential)
    rc, _ = tlc.status(cfg, L.ws)
    assert rc == tlc.MOE_ERR_TIMEOUT
    assert "timed out" in tlc.lib().moe_last_error().decode()
    cfg_ok = tlc.Config.from_workload(w, consumer_ctas=4, flags=PAIR | tlc.MOE_TAIL_ASSIST)
    assert torch.equal(L.run(sequential=sequential, cfg=cfg_ok), want)
