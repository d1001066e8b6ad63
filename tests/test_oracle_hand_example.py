"""A small layout worked out by hand from the definitions, pinned against the oracle.

The pages print no worked example, so this one was derived on paper from the layout rules of the
tile-level signaling page ("What carries the argument": group rows by expert then owner, pad each
group to the tile height, schedule the largest transfers first) and the readings in the oracle's
header. T = 8 tokens, E = 3 experts, top-2, R = 2 owners (tokens 0-3 and 4-7), tile height 2.

Routing (descending logit, ties to the lower id):
  t0 [3,1,2] -> (0,2)   t1 [0,5,5] -> (1,2)   t2 [1,1,1] -> (0,1)   t3 [-1,0,2] -> (2,1)
  t4 [4,0,0] -> (0,1)   t5 [0,2,1] -> (1,2)   t6 [2,2,0] -> (0,1)   t7 [0,0,3] -> (2,0)
Groups (pairs (t, j), ascending t): e0r0 (0,0)(2,0); e0r1 (4,0)(6,0)(7,1); e1r0 (1,0)(2,1)(3,1);
  e1r1 (4,1)(5,0)(6,1); e2r0 (0,1)(1,1)(3,0); e2r1 (5,1)(7,0).
Padded sizes 2,4,4,4,4,2 -> offsets 0,2,6,10,14,18,20.
Schedule (largest transfers first): the six full bands m0 m1 m3 m5 m7 m9 (2 rows each, layout
order), then the four 1-row bands m2 m4 m6 m8.
Hand-out order: expert loads 5, 6, 5 -> experts e1, e0, e2, each expert's bands in schedule order.
"""
import math

import numpy as np

from oracle import moe_ref as ref

LOGITS = np.array([[3, 1, 2], [0, 5, 5], [1, 1, 1], [-1, 0, 2], [4, 0, 0], [0, 2, 1], [2, 2, 0], [0, 0, 3]],
                  np.float32)


def test_hand_example_routing():
    idx, w = ref.route_topk(LOGITS, 2)
    assert idx.tolist() == [[0, 2], [1, 2], [0, 1], [2, 1], [0, 1], [1, 2], [0, 1], [2, 0]]
    s = 1 / (1 + math.exp(-1))
    assert abs(w[0, 0] - s) < 1e-15 and abs(w[0, 1] - (1 - s)) < 1e-15
    assert w[1].tolist() == [0.5, 0.5] and w[2].tolist() == [0.5, 0.5]


def test_hand_example_layout():
    idx, _ = ref.route_topk(LOGITS, 2)
    p = ref.build_plan(idx, 3, 2, 2, mgb=2)
    assert p.n.tolist() == [[2, 3], [3, 3], [3, 2]]
    assert p.off.tolist() == [0, 2, 6, 10, 14, 18, 20]
    assert p.slot.tolist() == [[0, 14], [6, 15], [1, 7], [16, 8], [2, 10], [11, 18], [3, 12], [19, 4]]
    assert p.tiles.tolist() == [[0, 0, 0, 2], [0, 1, 2, 2], [0, 1, 4, 1], [1, 0, 6, 2], [1, 0, 8, 1],
                                [1, 1, 10, 2], [1, 1, 12, 1], [2, 0, 14, 2], [2, 0, 16, 1], [2, 1, 18, 2]]
    assert p.ret_off.tolist() == [[0, 2, 5, 8], [0, 3, 6, 8]]
    assert p.ret_slot.tolist() == [[0, 5], [2, 6], [1, 3], [7, 4], [8, 11], [12, 14], [9, 13], [15, 10]]
    assert p.ret_row0.tolist() == [0, 8, 10, 2, 4, 11, 13, 5, 7, 14]
    assert p.sched.tolist() == [0, 1, 3, 5, 7, 9, 2, 4, 6, 8]
    # e1: m3, m5 (full), m4, m6; e0: m0, m1, m2; e2: m7, m9, m8
    assert p.order.tolist() == [3, 5, 4, 6, 0, 1, 2, 7, 9, 8]
    # in hand-out order m1 (rows 2-3) and m2 (row 4) are adjacent bands of group e0r1 -> one
    # segment of 2 bands
    assert p.seg.tolist() == [[0, 1], [1, 1], [2, 1], [3, 1], [4, 1], [5, 2], [5, 2], [7, 1], [8, 1], [9, 1]]


def test_hand_example_segments():
    # T = 4, E = 2, top-1, R = 1, tile height 1: e0 gets t0, t2, t3 (rows 0-2), e1 gets t1 (row 3).
    logits = np.array([[1, 0], [0, 1], [2, 0], [3, 0]], np.float32)
    idx, _ = ref.route_topk(logits, 1)
    p = ref.build_plan(idx, 2, 1, 1, mgb=2)
    assert p.slot.tolist() == [[0], [3], [1], [2]]
    assert p.sched.tolist() == [0, 1, 2, 3] and p.order.tolist() == [0, 1, 2, 3]
    assert p.seg.tolist() == [[0, 2], [0, 2], [2, 1], [3, 1]]
