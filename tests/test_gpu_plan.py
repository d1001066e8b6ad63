"""Routing, plan and permute on the GPU, bit-exact against the oracle.

Indices, counts, offsets, tile-owner map, schedule, hand-out order, segments, slots, return slots and
the permuted rows (with zero padding) have exactly one correct value each, so they are compared for
equality.
The permuted rows are checked in the expert-compact layout of the GEMM inputs, whose rows follow
from the oracle's plan (tests.gpu_util.compact_layout).
"""
import numpy as np
import pytest
import torch

import tile_level_copy_gb300 as tlc
from oracle import moe_ref
from tile_level_copy_gb300 import inputs
from tests.gpu_util import compact_layout

pytestmark = pytest.mark.gpu


def run_plan(w: inputs.Workload, logits_np: np.ndarray, x_cpu, mgb=1, skip_permute=False):
    cfg = tlc.Config.from_workload(w, mgb=mgb, flags=tlc.MOE_PLAN_SKIP_PERMUTE if skip_permute else 0)
    ws = tlc.Workspace(cfg)
    logits = torch.from_numpy(logits_np).cuda()
    x = None if x_cpu is None else x_cpu.cuda()
    idx = torch.empty(w.T, w.topk, dtype=torch.int32, device="cuda")
    gate = torch.empty(w.T, w.topk, dtype=torch.float32, device="cuda")
    tlc.plan(cfg, logits, x, ws, idx, gate)
    rc, detail = tlc.status(cfg, ws)
    assert rc == tlc.MOE_OK, (rc, detail)
    return cfg, ws, idx.cpu().numpy(), gate.cpu().numpy()


def check_plan(w, logits_np, x_cpu, mgb=1):
    cfg, ws, idx, gate = run_plan(w, logits_np, x_cpu, mgb, skip_permute=x_cpu is None)
    ridx, rgate = moe_ref.route_topk(logits_np, w.topk)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(gate, rgate, rtol=2e-6, atol=1e-7)
    plan = moe_ref.build_plan(ridx, w.E, w.R, w.tile_M, mgb)
    v = lambda n: ws.view(n).cpu().numpy()
    meta = v("meta")
    assert meta[0] == plan.P and meta[1] == plan.num_tiles
    MT = plan.num_tiles
    np.testing.assert_array_equal(v("counts"), plan.n)
    np.testing.assert_array_equal(v("offsets"), plan.off)
    np.testing.assert_array_equal(v("ret_off"), plan.ret_off)
    np.testing.assert_array_equal(v("tiles")[:MT], plan.tiles)
    np.testing.assert_array_equal(v("tile_ret")[:MT], plan.ret_row0)
    np.testing.assert_array_equal(v("sched")[:MT], plan.sched)
    np.testing.assert_array_equal(v("order")[:MT], plan.order)
    np.testing.assert_array_equal(v("seg")[:MT], plan.seg)
    np.testing.assert_array_equal(v("slot"), plan.slot)
    np.testing.assert_array_equal(v("ret_slot"), plan.ret_slot)
    # expert-compact layout of the GEMM inputs
    cbase, tile_crow, cslot, yrow, PC = compact_layout(plan, ridx)
    assert meta[9] == PC and meta[8] == PC // 128
    np.testing.assert_array_equal(v("tile_crow")[:MT], tile_crow)
    np.testing.assert_array_equal(v("cslot"), cslot)
    np.testing.assert_array_equal(v("yrow")[:PC], yrow)
    runs = -(-plan.n.sum(1) // 128)
    experts = v("experts").reshape(-1, 8)
    np.testing.assert_array_equal(experts[:, 4], runs)
    np.testing.assert_array_equal(experts[:, 5], cbase // 128)
    np.testing.assert_array_equal(experts[:, 7], cbase)
    want_items = [(cbase[e] + 128 * i, e) for e in range(w.E) for i in range(runs[e])]
    np.testing.assert_array_equal(v("items_up")[:PC // 128], np.array(want_items).reshape(-1, 2))
    # the down-projection takes the same items, experts in hand-out rank order (most rows first,
    # ties to the lower id), and the item holding each band's last row
    rank_order = sorted(range(w.E), key=lambda e: (-int(plan.n[e].sum()), e))
    down = [(cbase[e] + 128 * i, e) for e in rank_order for i in range(runs[e])]
    np.testing.assert_array_equal(v("items_down")[:PC // 128], np.array(down).reshape(-1, 2))
    first_down = {e: sum(runs[f] for f in rank_order[:rank_order.index(e)]) for e in range(w.E)}
    np.testing.assert_array_equal(experts[:, 6], [first_down[e] for e in range(w.E)])
    want_bi = [first_down[int(plan.tiles[m, 0])] + (tile_crow[m] + plan.tiles[m, 3] - 1 - cbase[plan.tiles[m, 0]]) // 128
               for m in range(MT)]
    np.testing.assert_array_equal(v("band_item")[:MT], want_bi)
    # the token of every compact row (-1 for the zero rows that pad each expert's run)
    tok = np.full(PC, -1, np.int64)
    tok[cslot.reshape(-1)] = np.repeat(np.arange(w.T), w.topk)
    np.testing.assert_array_equal(v("tok_of")[:PC], tok)
    if x_cpu is not None:
        xb = x_cpu.view(torch.int16).numpy()
        want = np.zeros((PC, w.d), np.int16)  # padding rows are zero
        want[cslot.reshape(-1)] = np.repeat(xb, w.topk, axis=0)
        got = ws.view("Xc")[:PC].view(torch.int16).cpu().numpy()
        np.testing.assert_array_equal(got, want)
        # the same rows as the page's padded layout, row for row
        np.testing.assert_array_equal(got[cslot.reshape(-1)], moe_ref.permute(xb, plan)[plan.slot.reshape(-1)])
    return plan


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
@pytest.mark.parametrize("mgb", [1, 2])
def test_plan_bitexact_full_size(name, mgb):
    w = inputs.WORKLOADS[name]
    check_plan(w, inputs.make_logits(w, 0), inputs.make_x(w, 0) if mgb == 1 else None, mgb)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_plan_bitexact_seeds_skew(seed):
    w = inputs.WORKLOADS["skew"]
    plan = check_plan(w, inputs.make_logits(w, seed), inputs.make_x(w, seed))
    assert (plan.n == 0).any()  # the Zipf bias leaves some groups empty


def test_forced_ties_go_to_lowest_expert():
    w = inputs.WORKLOADS["fine"].replace(T=1024)
    rng = np.random.default_rng(5)
    logits = rng.integers(-1, 2, size=(w.T, w.E)).astype(np.float32)  # massive ties
    logits[::7] = 0.0                                                  # whole rows tied
    logits[3, :] = -0.0
    check_plan(w, logits, inputs.make_x(w, 0))


@pytest.mark.parametrize("shape", [
    dict(T=8, d=128, ffn=128, E=1, topk=1, R=1, tile_M=64),     # one group, ragged tile
    dict(T=6, d=128, ffn=128, E=3, topk=2, R=3, tile_M=128),    # T/R = 2: chunks of 2 tokens
    dict(T=300, d=256, ffn=128, E=5, topk=3, R=5, tile_M=64),   # T/R = 60: chunks of 4 tokens
    dict(T=1000, d=128, ffn=256, E=256, topk=8, R=4, tile_M=128),  # max E, max k, mostly 1-row groups
    dict(T=64, d=128, ffn=128, E=16, topk=1, R=64, tile_M=128),  # one token per owner
])
def test_plan_edge_shapes(shape):
    w = inputs.Workload("edge", **shape)
    check_plan(w, inputs.make_logits(w, 3), inputs.make_x(w, 3))


def test_all_tokens_to_one_expert():
    w = inputs.WORKLOADS["skew"].replace(T=2048)
    logits = np.full((w.T, w.E), -5.0, np.float32)
    logits[:, 7] = 1.0
    logits[:, 2] = 0.5
    plan = check_plan(w, logits, inputs.make_x(w, 1))
    assert set(plan.tiles[:, 0].tolist()) == {2, 7}


def test_plan_skip_permute_leaves_xp_untouched():
    w = inputs.WORKLOADS["tiny"]
    cfg, ws, _, _ = run_plan(w, inputs.make_logits(w, 0), None, skip_permute=True)
    ref_idx, _ = moe_ref.route_topk(inputs.make_logits(w, 0), w.topk)
    plan = moe_ref.build_plan(ref_idx, w.E, w.R, w.tile_M)
    np.testing.assert_array_equal(ws.view("slot").cpu().numpy(), plan.slot)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
def test_work_items_cover_every_row_once(name):
    """Work items of both GEMMs: 128 compact rows of one expert each, disjoint, covering every real
    row once; the down-projection's list holds the same items with the experts in hand-out order, so
    each band's rows lie in the item band_item names and, when they start before it, in the item
    before it of the same expert; a full band of tile height 128 fills exactly one item."""
    w = inputs.WORKLOADS[name]
    cfg, ws, _, _ = run_plan(w, inputs.make_logits(w, 0), None, skip_permute=True)  # slots, no row copy
    meta = ws.view("meta").cpu().numpy()
    MT, NI, NU, PC = int(meta[1]), int(meta[7]), int(meta[8]), int(meta[9])
    tiles = ws.view("tiles").cpu().numpy()[:MT]
    tile_crow = ws.view("tile_crow").cpu().numpy()[:MT]
    band_item = ws.view("band_item").cpu().numpy()[:MT]
    items = ws.view("items_down").cpu().numpy()[:NI]
    up = ws.view("items_up").cpu().numpy()[:NU]
    assert NI == NU and NU * 128 == PC and NI <= MT
    assert sorted(map(tuple, items.tolist())) == sorted(map(tuple, up.tolist()))
    for m in range(MT):
        e, valid, c0 = int(tiles[m, 0]), int(tiles[m, 3]), int(tile_crow[m])
        i = int(band_item[m])
        r0, ie = items[i]
        assert ie == e and r0 <= c0 + valid - 1 < r0 + 128
        if c0 < r0:  # the band starts in the item before, of the same expert
            assert i > 0 and items[i - 1][1] == e and items[i - 1][0] == r0 - 128 <= c0
        if valid == 128 and w.tile_M == 128:
            assert c0 == r0
    # along the hand-out order the completing item never decreases (the copy engines stop at the
    # first band the epilogue returns, so those bands must be the last positions)
    order = ws.view("order").cpu().numpy()[:MT]
    assert np.all(np.diff(band_item[order]) >= 0)
    cslot = ws.view("cslot").cpu().numpy().reshape(-1)
    idx = ws.view("idx").cpu().numpy().reshape(-1)
    yrow = ws.view("yrow").cpu().numpy()[:PC]
    slot = ws.view("slot").cpu().numpy().reshape(-1)
    rows_of = {(r0 + i): e for r0, e in up.tolist() for i in range(128)}
    assert len(rows_of) == PC  # disjoint 128-row items
    assert all(rows_of[c] == e for c, e in zip(cslot.tolist(), idx.tolist()))
    np.testing.assert_array_equal(yrow[cslot], slot)  # each pair's compact row names its Yp row
    assert (yrow >= 0).sum() == len(slot)              # and every other compact row is padding
