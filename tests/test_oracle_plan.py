"""Pins of the oracle's layout (histogram, offsets, tiles, slots, return plan, schedule).

Brute force: pure-Python lists and loops on tiny inputs. Invariants: the layout
properties the tile-level signaling method rests on (every real row appears once,
each (expert, owner) group carries fewer than tbM padding rows, every tile has one
owner, padding is bounded by E*R*(tbM-1)).
"""
import numpy as np
import pytest

from oracle import moe_ref as ref
from tile_level_copy_gb300 import inputs


def brute_plan(idx, E, R, tbM):
    T, k = len(idx), len(idx[0])
    per = T // R
    G = [[[] for _ in range(R)] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            G[idx[t][j]][t // per].append((t, j))
    off, cur = {}, 0
    for e in range(E):
        for r in range(R):
            off[(e, r)] = cur
            cur += ((len(G[e][r]) + tbM - 1) // tbM) * tbM
    P = cur
    slot = [[None] * k for _ in range(T)]
    tiles = []
    for e in range(E):
        for r in range(R):
            for i, (t, j) in enumerate(G[e][r]):
                slot[t][j] = off[(e, r)] + i
            nt = (len(G[e][r]) + tbM - 1) // tbM
            for q in range(nt):
                tiles.append((e, r, off[(e, r)] + q * tbM, min(tbM, len(G[e][r]) - q * tbM)))
    ret_slot = [[None] * k for _ in range(T)]
    for r in range(R):
        row = r * per * k
        for e in range(E):
            for (t, j) in G[e][r]:
                ret_slot[t][j] = row
                row += 1
    return P, slot, tiles, ret_slot, G


def random_idx(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


CASES = [  # T, E, k, R, tbM
    (8, 3, 2, 2, 4), (12, 1, 1, 3, 2), (16, 4, 4, 4, 1), (30, 5, 2, 3, 4),
    (64, 6, 3, 8, 8), (40, 8, 1, 5, 16), (9, 2, 2, 1, 3), (48, 4, 2, 2, 64),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("seed", range(4))
def test_plan_matches_bruteforce(case, seed):
    T, E, k, R, tbM = case
    rng = np.random.default_rng(seed)
    idx = random_idx(rng, T, E, k)
    plan = ref.build_plan(idx, E, R, tbM)
    P, slot, tiles, ret_slot, G = brute_plan(idx.tolist(), E, R, tbM)
    assert plan.P == P
    np.testing.assert_array_equal(plan.slot, np.array(slot))
    np.testing.assert_array_equal(plan.tiles, np.array(tiles).reshape(-1, 4))
    np.testing.assert_array_equal(plan.ret_slot, np.array(ret_slot))
    np.testing.assert_array_equal(plan.n, [[len(G[e][r]) for r in range(R)] for e in range(E)])
    # tile destination rows: first member of the tile in Ret
    for m, (e, r, row0, valid) in enumerate(plan.tiles):
        first = G[e][r][(row0 - plan.off[e * R + r])]
        assert plan.ret_row0[m] == ret_slot[first[0]][first[1]]


def check_invariants(plan, idx):
    T, k = idx.shape
    E, R, tbM = plan.E, plan.R, plan.tbM
    own = ref.owners(T, R)
    flat = plan.slot.reshape(-1)
    # every real row appears exactly once
    assert len(np.unique(flat)) == T * k
    assert flat.min() >= 0 and flat.max() < plan.P
    # padding per group < tbM, groups tile-aligned
    pad = (plan.off[1:] - plan.off[:-1]).reshape(E, R) - plan.n
    assert np.all(pad >= 0) and np.all(pad < tbM)
    assert np.all(plan.off % tbM == 0)
    assert plan.P <= T * k + E * R * (tbM - 1)
    # each tile lies in one group; all its rows are that group's owner
    row_owner = np.full(plan.P, -1)
    row_owner[flat] = own[np.repeat(np.arange(T), k)]
    row_expert = np.full(plan.P, -1)
    row_expert[flat] = idx.reshape(-1)
    covered = np.zeros(plan.P, bool)
    for (e, r, row0, valid) in plan.tiles:
        g = e * R + r
        assert plan.off[g] <= row0 and row0 + tbM <= plan.off[g + 1]
        assert 1 <= valid <= tbM
        rows = np.arange(row0, row0 + valid)
        assert np.all(row_owner[rows] == r) and np.all(row_expert[rows] == e)
        assert np.all(row_owner[row0 + valid:row0 + tbM] == -1)
        covered[row0:row0 + tbM] = True
    assert covered.all()
    assert plan.tiles[:, 3].sum() == T * k
    # return slots: a permutation; owner r's pairs land in slice r
    rs = plan.ret_slot.reshape(-1)
    assert np.array_equal(np.sort(rs), np.arange(T * k))
    slice_rows = (T // R) * k
    assert np.all(rs // slice_rows == own[np.repeat(np.arange(T), k)])
    # schedule and hand-out order: permutations of the tiles
    assert np.array_equal(np.sort(plan.sched), np.arange(plan.num_tiles))
    assert np.array_equal(np.sort(plan.order), np.arange(plan.num_tiles))


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
def test_plan_invariants_on_workloads(name):
    w = inputs.WORKLOADS[name]
    logits = inputs.make_logits(w, seed=0)
    idx, _ = ref.route_topk(logits, w.topk)
    for mgb in (1, 2):
        plan = ref.build_plan(idx, w.E, w.R, w.tile_M, mgb)
        check_invariants(plan, idx)


def test_skew_has_empty_groups_and_invariants_hold():
    w = inputs.WORKLOADS["skew"].replace(T=512)
    logits = inputs.make_logits(w, seed=1)
    idx, _ = ref.route_topk(logits, w.topk)
    plan = ref.build_plan(idx, w.E, w.R, w.tile_M)
    assert (plan.n == 0).any()
    check_invariants(plan, idx)


def brute_schedule(plan):
    """Largest transfer (valid rows) first, ties in layout order: a pure-Python sort on the key."""
    keys = [(-t[3], t[0], t[1], t[2]) for t in plan.tiles.tolist()]
    return sorted(range(len(keys)), key=lambda m: keys[m])


def brute_order(plan):
    """Hand-out order: experts by (load descending, id), each expert's bands in schedule order;
    written as nested loops over experts, not as a sort of the schedule."""
    load = [sum(row) for row in plan.n.tolist()]
    experts = sorted(range(plan.E), key=lambda e: (-load[e], e))
    sched = brute_schedule(plan)
    out = []
    for e in experts:
        out += [m for m in sched if plan.tiles[m][0] == e]
    return out


def brute_segments(plan, mgb):
    s = plan.order
    T = plan.tiles

    def adjacent(p, q):
        a, b = T[s[p]], T[s[q]]
        return a[0] == b[0] and a[1] == b[1] and b[2] == a[2] + plan.tbM

    out = []
    for p in range(len(s)):
        start = p
        while start > 0 and adjacent(start - 1, start):
            start -= 1
        end = p + 1
        while end < len(s) and adjacent(end - 1, end):
            end += 1
        first = start + ((p - start) // mgb) * mgb
        out.append((first, min(mgb, end - first)))
    return out


@pytest.mark.parametrize("mgb", [1, 2, 3])
@pytest.mark.parametrize("seed", range(3))
def test_schedule_and_segments_bruteforce(mgb, seed):
    rng = np.random.default_rng(seed + 10)
    T, E, k, R, tbM = 96, 5, 2, 3, 8
    # skewed routing so groups have several full bands and a partial one
    idx = np.stack([rng.choice(E, size=k, replace=False, p=[.5, .2, .15, .1, .05]) for _ in range(T)])
    plan = ref.build_plan(idx.astype(np.int32), E, R, tbM, mgb)
    assert plan.sched.tolist() == brute_schedule(plan)
    assert plan.order.tolist() == brute_order(plan)
    assert [tuple(v) for v in plan.seg.tolist()] == brute_segments(plan, mgb)
    # the schedule: transfer sizes never grow along it
    assert np.all(np.diff(plan.tiles[plan.sched, 3]) <= 0)
    # the hand-out order: experts one after another, most loaded first; inside an expert full
    # bands before partial ones; segments never span groups
    e = plan.tiles[plan.order, 0]
    assert all(len(set(e[i:].tolist()) & set(e[:i].tolist())) == 0 for i in range(1, len(e)) if e[i] != e[i - 1])
    load = plan.n.sum(1)[e]
    assert np.all(np.diff(load) <= 0)
    for x in np.unique(e):
        assert np.all(np.diff(plan.tiles[plan.order[e == x], 3]) <= 0)
    for p, (first, ln) in enumerate(plan.seg.tolist()):
        assert first <= p < first + ln <= len(plan.order) and 1 <= ln <= mgb
        grp = {tuple(plan.tiles[plan.order[q], :2]) for q in range(first, first + ln)}
        assert len(grp) == 1


def test_permute_places_rows_and_zero_pads():
    rng = np.random.default_rng(2)
    T, E, k, R, tbM, d = 20, 3, 2, 2, 4, 5
    idx = random_idx(rng, T, E, k)
    x = rng.standard_normal((T, d))
    plan = ref.build_plan(idx, E, R, tbM)
    Xp = ref.permute(x, plan)
    for t in range(T):
        for j in range(k):
            assert np.array_equal(Xp[plan.slot[t, j]], x[t])
    used = np.zeros(plan.P, bool)
    used[plan.slot.reshape(-1)] = True
    assert np.all(Xp[~used] == 0)


def test_empty_routing_degenerate_cases():
    # R = 1, E = 1, k = 1: one group, one owner
    idx = np.zeros((10, 1), np.int32)
    plan = ref.build_plan(idx, 1, 1, 4)
    assert plan.P == 12 and plan.num_tiles == 3
    assert plan.tiles.tolist() == [[0, 0, 0, 4], [0, 0, 4, 4], [0, 0, 8, 2]]
    # an expert nobody picks gets no tiles and no rows
    idx = np.zeros((6, 1), np.int32)
    plan = ref.build_plan(idx, 3, 2, 2)
    assert plan.n[1:].sum() == 0 and set(plan.tiles[:, 0].tolist()) == {0}
    assert plan.off.tolist() == [0, 4, 8, 8, 8, 8, 8]


@pytest.mark.parametrize("mutation", ["smallest_first", "ties_reversed", "least_loaded_first"])
def test_schedule_pins_catch_planted_mistakes(monkeypatch, mutation):
    """A planted schedule or hand-out order mistake must fail the brute-force pins."""
    rng = np.random.default_rng(31)
    T, E, k, R, tbM = 96, 5, 2, 3, 8
    idx = np.stack([rng.choice(E, size=k, replace=False, p=[.5, .2, .15, .1, .05]) for _ in range(T)])
    orig_order = ref.handout_order
    if mutation == "smallest_first":
        monkeypatch.setattr(ref, "remote_first_schedule",
                            lambda tiles: np.lexsort((np.arange(len(tiles)), tiles[:, 3])))
    elif mutation == "ties_reversed":
        monkeypatch.setattr(ref, "remote_first_schedule",
                            lambda tiles: np.lexsort((-np.arange(len(tiles)), -tiles[:, 3])))
    else:
        monkeypatch.setattr(ref, "handout_order",
                            lambda tiles, sched, n: orig_order(tiles, sched, -n))
    plan = ref.build_plan(idx.astype(np.int32), E, R, tbM, 1)
    assert not (plan.sched.tolist() == brute_schedule(plan) and plan.order.tolist() == brute_order(plan))
