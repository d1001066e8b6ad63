"""The expected expert-compact layout that the GPU plan tests compare against (tests.gpu_util), worked
out by hand on the small layout of tests/test_oracle_hand_example.py.

Layout rules (the GEMM inputs' rows, one run per expert padded to 128 rows): inside an expert's run
its bands follow one another in hand-out order, each band's valid rows in row order; the output
(Yp) row of every compact row is recorded, -1 for the rows that pad a run.

Hand-out order of the example: m3 m5 m4 m6 (expert 1), m0 m1 m2 (expert 0), m7 m9 m8 (expert 2);
valid rows 2 2 1 1 | 2 2 1 | 2 2 1; runs of 128 rows from 0 (e0), 128 (e1), 256 (e2). So the first
compact rows of the bands are m0 0, m1 2, m2 4, m3 128, m5 130, m4 132, m6 133, m7 256, m9 258,
m8 260.
"""
import numpy as np

from oracle import moe_ref
from tests.gpu_util import compact_layout
from tests.test_oracle_hand_example import LOGITS


def test_compact_layout_by_hand():
    idx, _ = moe_ref.route_topk(LOGITS, 2)
    p = moe_ref.build_plan(idx, 3, 2, 2, mgb=2)
    cbase, tile_crow, cslot, yrow, PC = compact_layout(p, idx)
    assert cbase.tolist() == [0, 128, 256] and PC == 384
    assert tile_crow.tolist() == [0, 2, 4, 128, 132, 130, 133, 256, 260, 258]
    assert cslot.tolist() == [[0, 256], [128, 257], [1, 129], [260, 132], [2, 130], [131, 258], [3, 133],
                              [259, 4]]
    want = np.full(PC, -1)
    for c, y in [(0, 0), (1, 1), (2, 2), (3, 3), (4, 4), (128, 6), (129, 7), (130, 10), (131, 11), (132, 8),
                 (133, 12), (256, 14), (257, 15), (258, 18), (259, 19), (260, 16)]:
        want[c] = y
    assert yrow.tolist() == want.tolist()


def test_compact_layout_invariants_random():
    """On seeded random routings: every pair has one compact row, the rows of a band are consecutive
    from its first compact row, each expert's run holds exactly its rows from its start, and yrow
    inverts cslot."""
    rng = np.random.default_rng(7)
    for trial in range(20):
        T, E, R, k = 64, int(rng.integers(2, 9)), int(rng.choice([1, 2, 4])), 2
        tbM = int(rng.choice([2, 4, 8]))
        logits = rng.standard_normal((T, E)).astype(np.float32)
        idx, _ = moe_ref.route_topk(logits, k)
        p = moe_ref.build_plan(idx, E, R, tbM, mgb=1)
        cbase, tile_crow, cslot, yrow, PC = compact_layout(p, idx)
        flat = cslot.reshape(-1)
        assert len(set(flat.tolist())) == T * k
        assert np.array_equal(yrow[flat], p.slot.reshape(-1))
        for e in range(E):
            load = int(p.n[e].sum())
            rows = sorted(c for c, ee in zip(flat.tolist(), np.asarray(idx).reshape(-1).tolist()) if ee == e)
            assert rows == list(range(cbase[e], cbase[e] + load))
        for m in range(p.num_tiles):
            row0, valid = int(p.tiles[m, 2]), int(p.tiles[m, 3])
            assert np.array_equal(yrow[tile_crow[m]:tile_crow[m] + valid], np.arange(row0, row0 + valid))
