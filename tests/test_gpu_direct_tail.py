"""Direct return of the last wave's bands (MOE_DIRECT_TAIL).

With the flag, the down-projection's epilogue writes the bands completed by work items with a tile
among the launch's last `tail_window` tile hand-out positions straight into their owner's slice of
Ret (0 = one wave), and the consumer skips them: after the last tile there is nothing left to copy.

Bar: the layer output and Ret bitwise equal to the GEMM-then-copy path on the same inputs; every tile
flag and band counter complete; the bands whose Yp rows were left unwritten are exactly the bands of a
suffix of the down-projection's work items (the hand-out order), and every other band's Ret rows are
byte copies of its Yp rows. Ret is zeroed before each overlapped run, so a row written by neither the
epilogue nor the consumer would show.
"""
import numpy as np
import pytest
import torch

import tile_level_copy_gb300 as tlc
from oracle import moe_ref
from tile_level_copy_gb300 import inputs
from tests.gpu_util import MAX_ABS, REL_L2, Layer, check_flag_counts, parity, small

pytestmark = pytest.mark.gpu

PAIR, TA, CW, DT = tlc.MOE_PAIR_UMMA, tlc.MOE_TAIL_ASSIST, tlc.MOE_COPY_WARPS, tlc.MOE_DIRECT_TAIL


def run_direct(L: Layer, cfg):
    """Sequential reference, then the overlapped run with Yp and Ret zeroed first. Returns the set of
    bands whose real Yp rows stayed zero (returned by the epilogue) and the plan."""
    want = L.run(sequential=True)
    ret_seq = L.ws.view("Ret").clone()
    idx, _ = moe_ref.route_topk(L.logits_np, L.w.topk)
    plan = moe_ref.build_plan(idx, L.w.E, L.w.R, L.w.tile_M, cfg.mgb)
    L.ws.view("Yp").zero_()
    L.ws.view("Ret").zero_()
    got = L.run(sequential=False, cfg=cfg)
    assert torch.equal(got, want)
    assert torch.equal(L.ws.view("Ret"), ret_seq)
    MT = plan.num_tiles
    check_flag_counts(L, plan)
    Yp = L.ws.view("Yp").view(torch.int16).cpu().numpy()
    Ret = L.ws.view("Ret").view(torch.int16).cpu().numpy()
    band_item = L.ws.view("band_item").cpu().numpy()[:MT]
    direct = set()
    for m in range(MT):
        _, _, row0, valid = plan.tiles[m]
        dst = plan.ret_row0[m]
        if not np.any(Yp[row0:row0 + valid]):
            direct.add(m)
        else:
            np.testing.assert_array_equal(Ret[dst:dst + valid], Yp[row0:row0 + valid])
    if direct:  # a suffix of the work items: every band of an item from the first direct one on
        first = min(band_item[m] for m in direct)
        assert direct == {m for m in range(MT) if band_item[m] >= first}
        # and the last positions of the hand-out order
        pos = sorted(plan.order.tolist().index(m) for m in direct)
        assert pos == list(range(MT - len(direct), MT))
    return direct, plan


@pytest.mark.parametrize("flags,consumers", [(PAIR | TA, 4), (PAIR, 2), (TA, 8), (CW | TA, 0), (CW, 4)],
                         ids=["pair-assist", "pair", "single-assist", "copywarps-assist", "copywarps"])
@pytest.mark.parametrize("window", [0, 6, 20, 1 << 20])
def test_direct_tail_equals_sequential(flags, consumers, window):
    w = small("skew")
    L = Layer(w, seed=2, cfg_kw=dict(consumer_ctas=8, timeout_us=500000))
    cfg = tlc.Config.from_workload(w, consumer_ctas=consumers, flags=flags | DT, tail_window=window,
                                   timeout_us=500000)
    direct, plan = run_direct(L, cfg)
    if window == 1 << 20 or window == 0:  # the small layer has fewer tiles than one wave
        assert len(direct) == plan.num_tiles
    elif window == 20:
        assert 0 < len(direct) < plan.num_tiles


@pytest.mark.parametrize("name", ["mixtral", "skew", "fine"])
def test_direct_tail_at_full_size_in_the_bench_configuration(name):
    """Full workload sizes, the bench's copy configuration with the direct tail: bitwise equal to the
    sequential path; some but not all bands returned by the epilogue (the last wave)."""
    import bench
    w = inputs.WORKLOADS[name]
    c, warps = bench.DEFAULT_COPY[name]
    cfg_kw = dict(consumer_ctas=c, flags=bench.default_flags(warps))
    assert cfg_kw["flags"] & DT
    L = Layer(w, seed=1, cfg_kw=cfg_kw)
    direct, plan = run_direct(L, L.cfg)
    assert 0 < len(direct) < plan.num_tiles


@pytest.mark.parametrize("seed", range(16))
def test_direct_tail_checksum_falsifier(seed):
    """The page's falsifier (every returned row equals the row the producer computed) with the direct
    tail: small consumer partitions, windows from a few tiles to a few waves, segments of 1-2 bands."""
    w = inputs.WORKLOADS["skew"].replace(T=4096, d=256, ffn=256)
    flags = (PAIR if seed % 4 != 3 else CW) | (TA if seed % 2 else 0) | DT
    consumers = 0 if flags & CW else 2 + 2 * (seed % 3)
    L = Layer(w, seed=seed, cfg_kw=dict(consumer_ctas=4))
    cfg = tlc.Config.from_workload(w, consumer_ctas=consumers, mgb=1 + seed % 2, flags=flags,
                                   tail_window=[4, 16, 64, 0][seed % 4])
    run_direct(L, cfg)


def test_direct_tail_layer_matches_oracle():
    w = small("mixtral")
    L = Layer(w, seed=6, cfg_kw=dict(consumer_ctas=4, flags=PAIR | TA | DT, tail_window=8))
    ref = L.oracle_layer()
    got = L.run(sequential=False).double().cpu().numpy()
    err, rel = parity(got, ref.out)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)

