"""Plain CPU oracle of the MoE expert layer on the remote-owner-aligned layout.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline / reference legs may import this module. The product path never does, and
this module imports nothing from the product package.

It follows the method of the review page "Fine-grained Computation-Communication
Overlap via Tile-level Signaling and Scheduling for Mixture-of-Experts" (Cui,
Wingkvist, Ericsson; pith.science/paper/W2ZARMHG), cited below as [TLS] with the
section of that page:

  [TLS "What carries the argument"]  remote-owner-aligned row layout: each expert's
      rows grouped by destination (owner) rank and padded to a multiple of the tile
      height, so every output tile has exactly one owner; remote-first tile schedule
      emitting the largest owner-bound transfers earliest; row-band segments
      (contiguous strips of output rows over the full width) copied per owner.
  [TLS "Referee Report", major comment 1, §4.5 / Algorithm 1]  every (expert, rank)
      group is padded on its own, so padding is bounded by E*R*(tbM-1) rows.
  [TLS "Axiom & Free-Parameter Ledger"]  router output is known before the return
      path (the combine plan is precomputed); mgb = bands per interior segment.
  [TLS Figure 9 caption]  the sequential baseline (per-expert GEMM, then bulk
      return) on identical inputs is the correctness reference.

Arithmetic is float64 throughout, from the exact float64 values of the bfloat16
inputs; there is no intermediate rounding. Matrix products call numpy's matmul as a
library step, one expert region at a time; no other blocking or reordering.

Readings where the page is silent (each listed in the design notes):
  * gates: softmax over the k chosen logits (equal to a full softmax renormalised
    over the top-k), so identical experts reduce to one dense FFN;
  * top-k order: descending logit, ties to the lower expert id;
  * owner of token t: t // (T/R) (R equal contiguous partitions);
  * all R owner groups of each expert are padded (one GPU has no "self" rank);
  * expert FFN: SwiGLU, h = silu(x W1_e^T) * (x W3_e^T), y = h W2_e^T,
    silu(a) = a / (1 + exp(-a));
  * rows inside a group: ascending token id; padding rows of Xp are zero;
  * owner return buffer: packed rows, experts ascending, then group order;
  * schedule ("the largest remote-bound transfers earliest"): a band's transfer is its
    valid rows (the consumer writes one row-band segment at a time); bands sorted by
    valid rows, descending, ties kept in layout order (expert, owner, row);
  * hand-out order: the order in which the down-projection takes the bands, derived
    from the schedule by a stated rule (experts one after another, most loaded first,
    each expert's bands in schedule order); not a step of the page, pinned so that the
    order the kernels execute is checked;
  * segment: up to mgb consecutive hand-out positions holding adjacent bands of one
    group, counted from the start of each such run.

Parity pins live in tests/test_oracle_*.py: brute-force pure-Python versions on tiny
inputs, invariants of the layout, and special cases (identical experts give a dense
FFN, E = 1 and k = 1 give one FFN, W2 = I gives the gated hidden sum, gates sum to 1).
"""
from __future__ import annotations

import dataclasses

import numpy as np


# --------------------------------------------------------------------------- routing
def owners(T: int, R: int) -> np.ndarray:
    """Owner partition of every token: R equal contiguous blocks of T/R tokens.

    [TLS "Core claim"]: expert outputs return to the rank that sent each token; on
    one GPU the ranks are R logical partitions of the token batch.
    """
    if R <= 0 or T % R:
        raise ValueError("R must divide T")
    return np.arange(T, dtype=np.int64) // (T // R)


def route_topk(logits: np.ndarray, k: int):
    """Top-k routing and gates.

    For each token: the k experts with the largest logit, in descending order, ties
    going to the lower expert id; gate w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max)
    over the k chosen logits, in float64. [TLS "Axiom & Free-Parameter Ledger"]: the
    router output is available before the return path.

    Returns (idx int32 [T, k], w float64 [T, k]).
    """
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = l.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((ids, -l), axis=-1)  # primary key: -logit; secondary: expert id
    idx = order[:, :k]
    chosen = np.take_along_axis(l, idx, axis=1)
    z = np.exp(chosen - chosen.max(axis=1, keepdims=True))
    w = z / z.sum(axis=1, keepdims=True)
    return idx.astype(np.int32), w


# ---------------------------------------------------------------------------- layout
@dataclasses.dataclass
class Plan:
    """The remote-owner-aligned layout and its combine plan.

    n[e, r]       rows routed to expert e from owner r (|G_{e,r}|)
    off[g]        first padded row of group g = e*R + r; off[E*R] = P
    tiles[m]      (e, r, row0, valid) of M-tile m, in layout (memory) order
    slot[t, j]    row of pair (t, j) in Xp / Yp
    ret_off[r, e] first row of (e, r) inside owner r's return slice (exclusive prefix)
    ret_row0[m]   destination row in Ret of tile m's first row
    ret_slot[t,j] row of pair (t, j) in Ret
    sched[p]      M-tile at position p of the page's remote-first schedule
    order[p]      M-tile at position p of the hand-out order derived from the schedule
    seg[p]        (first position, number of bands) of the segment holding hand-out position p
    """

    T: int
    E: int
    R: int
    k: int
    tbM: int
    mgb: int
    n: np.ndarray
    off: np.ndarray
    tiles: np.ndarray
    slot: np.ndarray
    ret_off: np.ndarray
    ret_row0: np.ndarray
    ret_slot: np.ndarray
    sched: np.ndarray
    order: np.ndarray
    seg: np.ndarray

    @property
    def P(self) -> int:
        return int(self.off[-1])

    @property
    def num_tiles(self) -> int:
        return int(self.tiles.shape[0])


def build_plan(idx: np.ndarray, E: int, R: int, tbM: int, mgb: int = 1) -> Plan:
    """Histogram, padded offsets, tile-owner map, slots, return plan and schedule.

    [TLS "What carries the argument"]: rows of each expert are grouped by owner and
    each group is padded to a multiple of the tile height tbM, so that an M-tile
    lies in one (expert, owner) group and has one owner. [TLS "Referee Report",
    major comment 1]: the padding is per (expert, rank) group.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    if tbM <= 0 or mgb <= 0:
        raise ValueError("tbM and mgb must be positive")
    own = owners(T, R)

    # pairs (t, j) in ascending (t, j) order
    pe = idx.reshape(-1)
    pt = np.repeat(np.arange(T, dtype=np.int64), k)
    pr = own[pt]

    # histogram |G_{e,r}|
    n = np.zeros((E, R), dtype=np.int64)
    np.add.at(n, (pe, pr), 1)

    # padded group sizes and their exclusive prefix over (e-major, r-minor)
    padded = -(-n // tbM) * tbM
    off = np.zeros(E * R + 1, dtype=np.int64)
    off[1:] = np.cumsum(padded.reshape(-1))

    # rank of each pair inside its group: groups listed by (e, r), members by t
    order = np.lexsort((pt, pr, pe))
    g_sorted = pe[order] * R + pr[order]
    first = np.searchsorted(g_sorted, g_sorted, side="left")
    rank = np.empty(T * k, dtype=np.int64)
    rank[order] = np.arange(T * k) - first
    g = pe * R + pr
    slot = (off[g] + rank).reshape(T, k)

    # owner return buffers: slice r holds (T/R)*k packed rows, experts ascending
    ret_off = np.zeros((R, E + 1), dtype=np.int64)
    ret_off[:, 1:] = np.cumsum(n.T, axis=1)
    slice_rows = (T // R) * k
    ret_slot = (pr * slice_rows + ret_off[pr, pe] + rank).reshape(T, k)

    # tile-owner map: ceil(n/tbM) tiles per group, in layout order
    tiles, ret_row0 = [], []
    for e in range(E):
        for r in range(R):
            cnt = int(n[e, r])
            base = int(off[e * R + r])
            for i in range(-(-cnt // tbM)):
                tiles.append((e, r, base + i * tbM, min(tbM, cnt - i * tbM)))
                ret_row0.append(r * slice_rows + int(ret_off[r, e]) + i * tbM)
    tiles = np.array(tiles, dtype=np.int64).reshape(-1, 4)
    ret_row0 = np.array(ret_row0, dtype=np.int64)

    sched = remote_first_schedule(tiles)
    order = handout_order(tiles, sched, n)
    seg = segments(tiles, order, tbM, mgb)
    return Plan(T, E, R, k, tbM, mgb, n, off, tiles, slot, ret_off, ret_row0, ret_slot, sched, order, seg)


def remote_first_schedule(tiles: np.ndarray) -> np.ndarray:
    """Order of the M-tiles (row bands): the largest owner-bound transfers first.

    [TLS "What carries the argument"]: a remote-first tile schedule emits the largest
    remote-bound transfers earliest; [TLS "Core claim"]: the consumer issues one
    contiguous write per row-band segment, so the transfer a band makes is its valid
    rows over the full width. Reading: every band is owner-bound on one GPU (there is
    no local rank); bands are sorted by valid rows, descending, and bands of equal
    size keep their layout order (expert, owner, row).
    """
    if tiles.shape[0] == 0:
        return np.zeros(0, dtype=np.int64)
    valid = tiles[:, 3]
    return np.lexsort((np.arange(tiles.shape[0]), -valid)).astype(np.int64)


def handout_order(tiles: np.ndarray, sched: np.ndarray, n: np.ndarray) -> np.ndarray:
    """Order in which the down-projection takes the bands, derived from the schedule.

    Not a step of the page: the rule by which the producer turns the schedule into its
    hand-out order, kept here so that the order the kernels execute is pinned too. The
    schedule is re-sorted stably by expert, the experts taken one after another, the
    most loaded (most real rows) first, ties to the lower expert id; inside an expert
    the bands keep their schedule order.
    """
    if sched.shape[0] == 0:
        return np.zeros(0, dtype=np.int64)
    E = n.shape[0]
    load = n.sum(axis=1)
    rank = np.empty(E, dtype=np.int64)
    rank[np.lexsort((np.arange(E), -load))] = np.arange(E)
    e = tiles[sched, 0]
    return sched[np.lexsort((np.arange(sched.shape[0]), rank[e]))].astype(np.int64)


def segments(tiles: np.ndarray, order: np.ndarray, tbM: int, mgb: int) -> np.ndarray:
    """Row-band segments: up to mgb adjacent bands of one group, copied as one piece.

    [TLS "What carries the argument"]: a row band is a strip of output rows over the
    full width; [TLS "Axiom & Free-Parameter Ledger"]: mgb consecutive bands are
    merged into an interior segment. Runs are maximal stretches of hand-out positions
    (the order in which bands are produced and copied) whose bands are in the same
    group with rows directly following each other; each run is cut into pieces of mgb
    bands from its start.
    """
    m = len(order)
    seg = np.zeros((m, 2), dtype=np.int64)
    p = 0
    while p < m:
        q = p + 1
        while q < m:
            a, b = tiles[order[q - 1]], tiles[order[q]]
            if a[0] != b[0] or a[1] != b[1] or b[2] != a[2] + tbM:
                break
            q += 1
        for s in range(p, q, mgb):
            ln = min(mgb, q - s)
            seg[s:s + ln, 0] = s
            seg[s:s + ln, 1] = ln
        p = q
    return seg


def permute(x: np.ndarray, plan: Plan) -> np.ndarray:
    """Xp [P, d]: row slot[t, j] holds x[t]; padding rows are zero."""
    x = np.asarray(x)
    Xp = np.zeros((plan.P, x.shape[1]), dtype=x.dtype)
    for j in range(plan.k):
        Xp[plan.slot[:, j]] = x
    return Xp


# ------------------------------------------------------------------------ expert math
def silu(a: np.ndarray) -> np.ndarray:
    """silu(a) = a / (1 + exp(-a))."""
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def swiglu_ffn(xrows: np.ndarray, W1e: np.ndarray, W3e: np.ndarray, W2e: np.ndarray):
    """One expert: h = silu(x W1^T) * (x W3^T), y = h W2^T. Returns (h, y)."""
    h = silu(xrows @ W1e.T) * (xrows @ W3e.T)
    return h, h @ W2e.T


@dataclasses.dataclass
class LayerResult:
    idx: np.ndarray
    w: np.ndarray
    plan: Plan
    Xp: np.ndarray
    Hp: np.ndarray
    Yp: np.ndarray
    Ret: np.ndarray
    out: np.ndarray


def moe_layer(logits, x, W1, W3, W2, R: int, tbM: int, mgb: int = 1, k: int = 2) -> LayerResult:
    """The whole layer through the layout, in the method's order.

    route -> plan -> permute -> grouped SwiGLU GEMM over each expert's padded rows ->
    row-band copy of the valid rows of every tile into its owner's return slice ->
    weighted top-k combine out[t] = sum_j w[t, j] * Ret[ret_slot[t, j]] (j ascending).
    """
    x = np.asarray(x, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W3 = np.asarray(W3, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    T, d = x.shape
    E, F = W1.shape[0], W1.shape[1]
    idx, w = route_topk(logits, k)
    plan = build_plan(idx, E, R, tbM, mgb)

    Xp = permute(x, plan)
    Hp = np.zeros((plan.P, F))
    Yp = np.zeros((plan.P, d))
    for e in range(E):  # one library matmul per expert region of the layout
        a, b = int(plan.off[e * R]), int(plan.off[(e + 1) * R])
        if b > a:
            Hp[a:b], Yp[a:b] = swiglu_ffn(Xp[a:b], W1[e], W3[e], W2[e])

    Ret = np.zeros((T * k, d))
    for m in range(plan.num_tiles):
        _, _, row0, valid = plan.tiles[m]
        dst = plan.ret_row0[m]
        Ret[dst:dst + valid] = Yp[row0:row0 + valid]

    out = np.zeros((T, d))
    for j in range(k):
        out += w[:, j:j + 1] * Ret[plan.ret_slot[:, j]]
    return LayerResult(idx, w, plan, Xp, Hp, Yp, Ret, out)


def moe_tokens(tokens, logits, x_rows, expert_weights, k: int):
    """The layer's definition on selected tokens, without the layout.

    out[t] = sum_j w[t, j] * FFN_{idx[t, j]}(x[t]) for t in ``tokens``. ``x_rows`` holds
    the rows x[t] for those tokens (float64-exact); ``expert_weights(e)`` returns
    (W1_e, W3_e, W2_e). Used for sampled checks at full size.
    """
    tokens = np.asarray(tokens)
    idx, w = route_topk(np.asarray(logits)[tokens], k)
    xr = np.asarray(x_rows, dtype=np.float64)
    y = np.zeros((xr.shape[0], k, xr.shape[1]))
    for e in np.unique(idx):
        W1e, W3e, W2e = (np.asarray(a, dtype=np.float64) for a in expert_weights(int(e)))
        rows, cols = np.nonzero(idx == e)
        _, y[rows, cols] = swiglu_ffn(xr[rows], W1e, W3e, W2e)
    out = np.zeros_like(xr)
    for j in range(k):
        out += w[:, j:j + 1] * y[:, j]
    return idx, w, out
