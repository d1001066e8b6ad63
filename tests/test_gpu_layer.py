"""The whole MoE layer on the GPU against the fp64 oracle, and overlapped against sequential.

Bar: layer output within max-abs 2e-2 and relative L2 5e-3 of the fp64 oracle; routing indices
bit-exact; the overlapped path bitwise equal to the GEMM-then-copy path (both run the same tile
code); every copied row of Ret byte-equal to its row of Yp.
"""
import numpy as np
import pytest
import torch

import tile_level_copy_gb300 as tlc
from oracle import moe_ref
from tile_level_copy_gb300 import inputs
from tests.gpu_util import MAX_ABS, REL_L2, Layer, check_flag_counts, parity, per_token_rel_distance, small

pytestmark = pytest.mark.gpu


def check_ret_is_copy_of_yp(L: Layer, plan):
    Yp = L.ws.view("Yp").view(torch.int16)
    Ret = L.ws.view("Ret").view(torch.int16)
    slot = torch.from_numpy(plan.slot.reshape(-1)).long().cuda()
    rslot = torch.from_numpy(plan.ret_slot.reshape(-1)).long().cuda()
    assert torch.equal(Ret[rslot], Yp[slot])


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
def test_layer_matches_oracle_small_shapes(name):
    w = small(name)
    L = Layer(w, seed=0, cfg_kw=dict(consumer_ctas=8))
    ref = L.oracle_layer()
    out_ovl = L.run(sequential=False).double().cpu().numpy()
    np.testing.assert_array_equal(L.ws.view("idx").cpu().numpy(), ref.idx)
    err, rel = parity(out_ovl, ref.out)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
    # intermediates: SwiGLU hidden and expert outputs on the real rows
    rows = ref.plan.slot.reshape(-1)
    crows = torch.from_numpy(L.ws.view("cslot").cpu().numpy().reshape(-1)).long().cuda()
    Hc = L.ws.view("Hc")[crows].double().cpu().numpy()  # the compact rows of the same pairs
    _, hrel = parity(Hc, ref.Hp[rows])
    assert hrel <= 5e-3, hrel
    Yp = L.ws.view("Yp")[:ref.plan.P].double().cpu().numpy()
    _, yrel = parity(Yp[rows], ref.Yp[rows])
    assert yrel <= 5e-3, yrel
    check_ret_is_copy_of_yp(L, ref.plan)
    # every tile flag counted each of its rows once; every band counter all its rows of all its tiles
    check_flag_counts(L, ref.plan)
    # the page's per-token relative distance, reported beside the gate
    assert per_token_rel_distance(out_ovl, ref.out).max() < 5e-2
    # sequential baseline: bitwise equal
    ret_ovl = L.ws.view("Ret").clone()
    out_seq = L.run(sequential=True).double().cpu().numpy()
    np.testing.assert_array_equal(out_seq, out_ovl)
    assert torch.equal(L.ws.view("Ret"), ret_ovl)


CW = tlc.MOE_COPY_WARPS


EDGE_SHAPES = [
    dict(T=8, d=128, ffn=128, E=1, topk=1, R=1, tile_M=64),      # one group, one ragged tile, N tiles of 128
    dict(T=6, d=128, ffn=128, E=3, topk=2, R=3, tile_M=128),     # T/R = 2: chunks of 2 tokens
    dict(T=300, d=256, ffn=128, E=5, topk=3, R=5, tile_M=64),    # 64-row bands, uneven groups
    dict(T=1000, d=128, ffn=256, E=256, topk=8, R=4, tile_M=128),  # max E, max k, mostly 1-row groups
    dict(T=64, d=128, ffn=128, E=16, topk=1, R=64, tile_M=128),  # one token per owner
    dict(T=512, d=384, ffn=384, E=6, topk=2, R=2, tile_M=128),   # d, ffn not multiples of 256
    # d = 256: the down-projection runs on CTA pairs too (even consumer_ctas, no copy warps)
    dict(T=8, d=256, ffn=128, E=1, topk=1, R=1, tile_M=64),      # one expert, one pair item, idle half
    dict(T=1000, d=256, ffn=256, E=256, topk=8, R=4, tile_M=128),  # max E: many experts with 0 or 1 item
    dict(T=64, d=256, ffn=128, E=16, topk=1, R=64, tile_M=128),  # one token per owner
]


@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda sh: "-".join(f"{k}{v}" for k, v in sh.items()))
def test_layer_edge_shapes(shape):
    """Degenerate and extreme shapes through the whole layer: oracle parity, and the overlapped path
    (dedicated consumers; copy warps only; CTA-pair SwiGLU GEMM) bitwise equal to the sequential one."""
    w = inputs.Workload("edge", **shape)
    L = Layer(w, seed=4, cfg_kw=dict(consumer_ctas=4, timeout_us=500000))
    ref = L.oracle_layer()
    seq = L.run(sequential=True)
    np.testing.assert_array_equal(L.ws.view("idx").cpu().numpy(), ref.idx)
    err, rel = parity(seq.double().cpu().numpy(), ref.out)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
    for c, flags in ((4, tlc.MOE_TAIL_ASSIST), (0, tlc.MOE_COPY_WARPS), (2, tlc.MOE_PAIR_UMMA)):
        cfg = tlc.Config.from_workload(w, consumer_ctas=c, flags=flags, timeout_us=500000)
        assert torch.equal(L.run(sequential=False, cfg=cfg), seq), (c, flags)
    check_ret_is_copy_of_yp(L, ref.plan)


def test_all_tokens_to_one_expert_layer():
    """Every token routed to the same two experts: all other experts have no rows (no work items)."""
    w = inputs.WORKLOADS["skew"].replace(T=2048, d=256, ffn=256)
    L = Layer(w, seed=1, cfg_kw=dict(consumer_ctas=4))
    lg = np.full((w.T, w.E), -5.0, np.float32)
    lg[:, 7], lg[:, 2] = 1.0, 0.5
    L.logits_np, L.logits = lg, torch.from_numpy(lg).cuda()
    ref = L.oracle_layer()
    seq = L.run(sequential=True)
    err, rel = parity(seq.double().cpu().numpy(), ref.out)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
    for flags in (tlc.MOE_TAIL_ASSIST, tlc.MOE_PAIR_UMMA, tlc.MOE_PAIR_UMMA | tlc.MOE_TAIL_ASSIST):
        cfg = tlc.Config.from_workload(w, consumer_ctas=4, flags=flags)
        assert torch.equal(L.run(sequential=False, cfg=cfg), seq)


@pytest.mark.parametrize("consumers,mgb,flags", [
    (1, 1, 0), (2, 2, 0), (4, 1, tlc.MOE_TAIL_ASSIST), (16, 2, tlc.MOE_TAIL_ASSIST), (32, 4, 0),
    (0, 1, CW), (0, 2, CW | tlc.MOE_TAIL_ASSIST), (4, 1, CW | tlc.MOE_TAIL_ASSIST), (8, 4, CW),
])
def test_partition_and_segment_knobs_do_not_change_results(consumers, mgb, flags):
    w = small("skew")
    L = Layer(w, seed=1)
    base = L.run(sequential=True)
    cfg = tlc.Config.from_workload(w, consumer_ctas=consumers, mgb=mgb, flags=flags)
    got = L.run(sequential=False, cfg=cfg)
    assert torch.equal(got, base)


@pytest.mark.parametrize("seed", range(100))
def test_tile_checksum_falsifier(seed):
    """Every tile the consumer copied must equal, byte for byte, the tile the producer stored.

    This is the page's proposed falsifier of the flag protocol ("What would settle it": checksummed
    tiles under stress) run over 100 seeds of the skewed workload with a tiny consumer partition.
    """
    w = inputs.WORKLOADS["skew"].replace(T=1024, d=256, ffn=256)
    copy_warps = seed % 4 == 1  # a quarter of the seeds copy with the producers' extra warps only
    L = Layer(w, seed=seed, cfg_kw=dict(consumer_ctas=0 if copy_warps else 2 + seed % 7, mgb=1 + seed % 2,
                                        flags=(tlc.MOE_TAIL_ASSIST if seed % 3 == 0 else 0) |
                                        (CW if copy_warps else 0)))
    L.run(sequential=False)
    idx, _ = moe_ref.route_topk(L.logits_np, w.topk)
    plan = moe_ref.build_plan(idx, w.E, w.R, w.tile_M, L.cfg.mgb)
    check_ret_is_copy_of_yp(L, plan)


@pytest.mark.parametrize("consumers,flags", [(4, 0), (0, CW)])
def test_stalled_consumer_times_out_and_context_survives(consumers, flags):
    w = small("tiny")
    L = Layer(w, seed=0)
    want = L.run(sequential=True)
    cfg = tlc.Config.from_workload(w, consumer_ctas=consumers, flags=flags | tlc.MOE_TEST_STALL_CONSUMER,
                                   timeout_us=20000)
    tlc.forward(cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws)
    rc, detail = tlc.status(cfg, L.ws)
    assert rc == tlc.MOE_ERR_TIMEOUT
    assert "timed out" in tlc.lib().moe_last_error().decode()
    # the context is still usable and the next call is correct
    assert torch.equal(L.run(sequential=False), want)


@pytest.mark.parametrize("pdl", [False, True], ids=["serial", "pdl"])
def test_stalled_layout_wait_times_out_and_context_survives(pdl):
    """MOE_TEST_STALL_LAYOUT: the plan never publishes the row layout, so the permute's bounded wait
    for it runs out; the call reports MOE_ERR_TIMEOUT, and the next call is correct."""
    w = small("tiny")
    L = Layer(w, seed=0)
    want = L.run(sequential=True)
    flags = tlc.MOE_TEST_STALL_LAYOUT | (tlc.MOE_PDL if pdl else 0)
    cfg = tlc.Config.from_workload(w, consumer_ctas=4, flags=flags, timeout_us=20000)
    tlc.forward(cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws)
    rc, detail = tlc.status(cfg, L.ws)
    assert rc == tlc.MOE_ERR_TIMEOUT
    assert "row layout" in tlc.lib().moe_last_error().decode()
    assert torch.equal(L.run(sequential=False), want)


def test_forward_host_equals_device_forward():
    w = small("mixtral")
    L = Layer(w, seed=2, cfg_kw=dict(consumer_ctas=8))
    want = L.run(sequential=False).cpu()
    logits_h = torch.from_numpy(L.logits_np).pin_memory()
    x_h = L.x_cpu.pin_memory()
    out_h = torch.empty(w.T, w.d, dtype=torch.float32).pin_memory()
    tlc.forward_host(L.cfg, logits_h, x_h, L.W["W1"], L.W["W3"], L.W["W2"], out_h, L.ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h, want)


@pytest.mark.parametrize("sequential", [False, True])
def test_forward_host_pipelined_equals_device_forward(sequential):
    """Four batches with different tokens and routing through the pipelined host call (both staging
    slots used twice): each output equals the device forward of its batch."""
    w = small("mixtral")
    L = Layer(w, seed=2, cfg_kw=dict(consumer_ctas=8))
    seeds = (2, 5, 7, 11)
    logits_h, x_h, want = [], [], []
    for sd in seeds:
        lg, x = inputs.make_logits(w, sd), inputs.make_x(w, sd)
        tlc.forward(L.cfg, torch.from_numpy(lg).cuda(), x.cuda(), L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws,
                    sequential=sequential)
        want.append(L.out.cpu().clone())
        logits_h.append(torch.from_numpy(lg).pin_memory())
        x_h.append(x.pin_memory())
    out_h = [torch.full((w.T, w.d), float("nan")).pin_memory() for _ in seeds]
    tlc.forward_host_pipelined(L.cfg, logits_h, x_h, L.W["W1"], L.W["W3"], L.W["W2"], out_h, L.ws,
                               sequential=sequential)
    torch.cuda.synchronize()
    assert tlc.status(L.cfg, L.ws)[0] == tlc.MOE_OK
    for got, ref in zip(out_h, want):
        assert torch.equal(got, ref)


def test_copy_only_reproduces_the_return_copy():
    """moe_copy_only on a few SMs rewrites Ret exactly as the forward's copy did."""
    w = small("skew")
    L = Layer(w, seed=3)
    L.run(sequential=True)
    want = L.ws.view("Ret").clone()
    for ctas in (1, 3, 16):
        L.ws.view("Ret").zero_()
        tlc.copy_only(L.cfg, L.ws, ctas)
        assert tlc.status(L.cfg, L.ws)[0] == tlc.MOE_OK
        assert torch.equal(L.ws.view("Ret"), want)
    with pytest.raises(tlc.MoEError) as ei:
        tlc.copy_only(L.cfg, L.ws, 0)
    assert ei.value.code == tlc.MOE_ERR_ARG


def test_corrupt_plan_entry_is_reported_not_used():
    """A hand-out order entry pointing past the last band makes the copy report MOE_ERR_PLAN (its
    bounds check runs before the entry is used); the next forward re-plans and is correct again."""
    w = small("skew")
    L = Layer(w, seed=3)
    want = L.run(sequential=True)
    MT = int(L.ws.view("meta")[1].item())
    L.ws.view("order")[0] = MT + 7
    tlc.copy_only(L.cfg, L.ws, 4)
    rc, detail = tlc.status(L.cfg, L.ws)
    assert rc == tlc.MOE_ERR_PLAN and detail == 0
    assert torch.equal(L.run(sequential=False), want)


def test_argument_errors_on_gpu():
    w = small("tiny")
    L = Layer(w, seed=0)
    small_ws = tlc.Workspace(L.cfg)
    small_ws.nbytes = small_ws.nbytes - 1024
    with pytest.raises(tlc.MoEError) as ei:
        tlc.forward(L.cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, small_ws)
    assert ei.value.code == tlc.MOE_ERR_WORKSPACE
    sms, ok = tlc.device_info()
    assert ok and sms >= 100
    for bad in (tlc.Config.from_workload(w, consumer_ctas=sms), tlc.Config.from_workload(w, consumer_ctas=0)):
        with pytest.raises(tlc.MoEError) as ei:
            tlc.forward(bad, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws)
        assert ei.value.code == tlc.MOE_ERR_ARG


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral", "skew", "fine"])
def test_full_size_sampled_tokens(name):
    """Full workload sizes in the bench's launch configuration (its per-workload copy configuration,
    CTA-pair GEMMs, tail assist, direct tail); 48 sampled tokens against the oracle's per-token definition,
    plus bitwise overlapped == sequential over all tokens, also for the page's dedicated partition
    (8 consumer CTAs, single-CTA GEMMs) and for copy warps alone."""
    import bench
    w = inputs.WORKLOADS[name]
    c, warps = bench.DEFAULT_COPY[name]
    flags = bench.default_flags(warps)
    L = Layer(w, seed=0, cfg_kw=dict(consumer_ctas=c, flags=flags))
    got = L.run(sequential=False)
    seq = L.run(sequential=True)
    assert torch.equal(got, seq)
    for c2, f2 in ((8, tlc.MOE_TAIL_ASSIST), (0, CW | tlc.MOE_TAIL_ASSIST)):
        assert torch.equal(L.run(sequential=False, cfg=tlc.Config.from_workload(w, consumer_ctas=c2, flags=f2)), seq)
    rng = np.random.default_rng(7)
    tokens = np.sort(rng.choice(w.T, size=48, replace=False))
    tokens[0], tokens[-1] = 0, w.T - 1  # include both ends
    x_rows = inputs.bf16_to_f64(L.x_cpu[tokens])
    _, _, want = moe_ref.moe_tokens(tokens, L.logits_np, x_rows, L.weights_f64, w.topk)
    err, rel = parity(got.double().cpu().numpy()[tokens], want)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)


@pytest.mark.slow
@pytest.mark.parametrize("name,seed", [("mixtral", 0), ("skew", 3)])
def test_full_size_every_token_against_the_oracle(name, seed):
    """Every token of the full-size layer, in the bench's launch configuration (its copy configuration,
    CTA-pair GEMMs, tail assist, direct tail), against the oracle's per-token definition in fp64,
    element by element: covers every band of the down-projection's hand-out order, the N-tile-outer
    order of the Mixtral shape and the bands the epilogue returns itself."""
    import bench
    w = inputs.WORKLOADS[name]
    c, warps = bench.DEFAULT_COPY[name]
    L = Layer(w, seed=seed, cfg_kw=dict(consumer_ctas=c, flags=bench.default_flags(warps)))
    got = L.run(sequential=False).double().cpu().numpy()
    idx, _, want = moe_ref.moe_tokens(np.arange(w.T), L.logits_np, inputs.bf16_to_f64(L.x_cpu), L.weights_f64,
                                      w.topk)
    np.testing.assert_array_equal(L.ws.view("idx").cpu().numpy(), idx)
    err, rel = parity(got, want)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
    assert per_token_rel_distance(got, want).max() < 5e-2
