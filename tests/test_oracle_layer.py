"""Pins of the oracle's expert math, copy and combine.

* brute force: the layer written element by element in pure Python on tiny inputs;
* special cases: identical experts give one dense SwiGLU FFN for any routing,
  E = 1 with k = 1 gives that FFN, W2 = I gives the gated hidden sum;
* closed forms of silu; byte-equality of the row-band copy; linearity in W2.
"""
import math

import numpy as np
import pytest

from oracle import moe_ref as ref
from tile_level_copy_gb300 import inputs


def brute_layer(logits, x, W1, W3, W2, k):
    T, d = len(x), len(x[0])
    E, F = len(W1), len(W1[0])
    out = [[0.0] * d for _ in range(T)]
    for t in range(T):
        row = [float(v) for v in logits[t]]
        chosen = sorted(range(E), key=lambda e: (-row[e], e))[:k]
        z = [math.exp(row[e] - row[chosen[0]]) for e in chosen]
        s = sum(z)
        for j, e in enumerate(chosen):
            h = []
            for f in range(F):
                g = sum(x[t][i] * W1[e][f][i] for i in range(d))
                u = sum(x[t][i] * W3[e][f][i] for i in range(d))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for c in range(d):
                y = sum(h[f] * W2[e][c][f] for f in range(F))
                out[t][c] += (z[j] / s) * y
    return np.array(out)


def rand_layer(rng, T, d, F, E):
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((E, F, d)) / math.sqrt(d)
    W3 = rng.standard_normal((E, F, d)) / math.sqrt(d)
    W2 = rng.standard_normal((E, d, F)) / math.sqrt(d)
    return logits, x, W1, W3, W2


@pytest.mark.parametrize("T,d,F,E,k,R,tbM", [
    (8, 4, 6, 3, 2, 2, 4), (12, 3, 5, 4, 3, 3, 2), (6, 5, 4, 1, 1, 2, 8), (10, 4, 4, 5, 1, 5, 1),
])
@pytest.mark.parametrize("seed", range(3))
def test_layer_matches_bruteforce(T, d, F, E, k, R, tbM, seed):
    rng = np.random.default_rng(seed)
    logits, x, W1, W3, W2 = rand_layer(rng, T, d, F, E)
    res = ref.moe_layer(logits, x, W1, W3, W2, R=R, tbM=tbM, k=k)
    want = brute_layer(logits.tolist(), x.tolist(), W1.tolist(), W3.tolist(), W2.tolist(), k)
    np.testing.assert_allclose(res.out, want, rtol=0, atol=1e-12)
    # the same numbers without the layout
    _, _, tok = ref.moe_tokens(np.arange(T), logits, x, lambda e: (W1[e], W3[e], W2[e]), k)
    np.testing.assert_allclose(tok, want, rtol=0, atol=1e-12)


def dense_swiglu(x, W1e, W3e, W2e):
    g = x @ W1e.T
    return (g * (1.0 / (1.0 + np.exp(-g))) * (x @ W3e.T)) @ W2e.T


@pytest.mark.parametrize("k,R,tbM", [(2, 2, 64), (3, 4, 16), (1, 1, 8)])
def test_identical_experts_reduce_to_dense_ffn(k, R, tbM):
    rng = np.random.default_rng(11)
    T, d, F, E = 64, 16, 24, 4
    logits, x, W1, W3, W2 = rand_layer(rng, T, d, F, E)
    W1[:] = W1[0]
    W3[:] = W3[0]
    W2[:] = W2[0]
    res = ref.moe_layer(logits, x, W1, W3, W2, R=R, tbM=tbM, k=k)
    np.testing.assert_allclose(res.out, dense_swiglu(x, W1[0], W3[0], W2[0]), rtol=1e-12, atol=1e-12)


def test_single_expert_top1_is_one_ffn():
    rng = np.random.default_rng(12)
    logits, x, W1, W3, W2 = rand_layer(rng, 32, 8, 12, 1)
    res = ref.moe_layer(logits, x, W1, W3, W2, R=4, tbM=4, k=1)
    np.testing.assert_allclose(res.out, dense_swiglu(x, W1[0], W3[0], W2[0]), rtol=1e-13, atol=1e-13)


def test_identity_down_projection_gives_gated_hidden_sum():
    rng = np.random.default_rng(13)
    T, d, E, k = 24, 6, 3, 2
    logits, x, W1, W3, _ = rand_layer(rng, T, d, d, E)
    W2 = np.broadcast_to(np.eye(d), (E, d, d)).copy()
    res = ref.moe_layer(logits, x, W1, W3, W2, R=2, tbM=4, k=k)
    idx, w = ref.route_topk(logits, k)
    want = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            g = W1[e] @ x[t]
            want[t] += w[t, j] * (g / (1 + np.exp(-g))) * (W3[e] @ x[t])
    np.testing.assert_allclose(res.out, want, rtol=1e-13, atol=1e-13)


def test_silu_closed_forms():
    a = np.array([0.0, 1.0, -1.0, 50.0, -800.0, 800.0])
    s = ref.silu(a)
    assert s[0] == 0.0
    assert abs(s[1] - 0.7310585786300049) < 1e-16
    assert abs(s[2] + 0.2689414213699951) < 1e-16
    assert abs(s[3] - 50.0) < 1e-12
    assert s[4] == 0.0 and not np.isnan(s[4])
    assert s[5] == 800.0
    # silu(a) - silu(-a) = a
    b = np.linspace(-6, 6, 101)
    np.testing.assert_allclose(ref.silu(b) - ref.silu(-b), b, atol=1e-14)


def test_copy_moves_valid_rows_exactly_and_linearity():
    rng = np.random.default_rng(14)
    T, d, F, E, k, R, tbM = 40, 8, 8, 3, 2, 4, 4
    logits, x, W1, W3, W2 = rand_layer(rng, T, d, F, E)
    res = ref.moe_layer(logits, x, W1, W3, W2, R=R, tbM=tbM, k=k)
    p = res.plan
    for m, (e, r, row0, valid) in enumerate(p.tiles):
        assert np.array_equal(res.Ret[p.ret_row0[m]:p.ret_row0[m] + valid], res.Yp[row0:row0 + valid])
    for t in range(T):
        for j in range(k):
            assert np.array_equal(res.Ret[p.ret_slot[t, j]], res.Yp[p.slot[t, j]])
    # padding rows stay zero through the expert math (silu(0) * 0 = 0)
    used = np.zeros(p.P, bool)
    used[p.slot.reshape(-1)] = True
    assert np.all(res.Hp[~used] == 0) and np.all(res.Yp[~used] == 0)
    res2 = ref.moe_layer(logits, x, W1, W3, 2 * W2, R=R, tbM=tbM, k=k)
    np.testing.assert_allclose(res2.out, 2 * res.out, rtol=1e-14, atol=1e-14)


def test_tiny_workload_runs_fast_and_is_finite():
    w = inputs.WORKLOADS["tiny"]
    a = inputs.make_all(w, seed=0)
    res = ref.moe_layer(a["logits"], inputs.bf16_to_f64(a["x"]), inputs.bf16_to_f64(a["W1"]),
                        inputs.bf16_to_f64(a["W3"]), inputs.bf16_to_f64(a["W2"]),
                        R=w.R, tbM=w.tile_M, k=w.topk)
    assert np.isfinite(res.out).all()
    assert res.out.shape == (w.T, w.d)
    assert 0.3 < res.out.std() < 3.0


@pytest.mark.parametrize("mutation", ["tie_high_id", "drop_gate", "transpose_w2"])
def test_pins_catch_planted_mistakes(monkeypatch, mutation):
    """Each planted oracle mistake must make the brute-force layer pin fail."""
    rng = np.random.default_rng(21)
    T, d, F, E, k, R, tbM = 8, 4, 4, 3, 2, 2, 4
    logits, x, W1, W3, W2 = rand_layer(rng, T, d, F, E)
    logits = np.round(logits).astype(np.float32)  # ties
    orig_route = ref.route_topk
    Wd = W2
    if mutation == "tie_high_id":
        def bad(lg, kk):
            l = np.asarray(lg, np.float32).astype(np.float64)
            ids = np.broadcast_to(-np.arange(l.shape[1]), l.shape)
            i = np.lexsort((ids, -l), axis=-1)[:, :kk]
            chosen = np.take_along_axis(l, i, 1)
            z = np.exp(chosen - chosen[:, :1])
            return i.astype(np.int32), z / z.sum(1, keepdims=True)
        monkeypatch.setattr(ref, "route_topk", bad)
    elif mutation == "drop_gate":
        monkeypatch.setattr(ref, "route_topk", lambda lg, kk: (orig_route(lg, kk)[0], np.ones((T, kk))))
    elif mutation == "transpose_w2":
        Wd = np.swapaxes(W2, 1, 2).copy()  # d == F here, so the shapes still fit
    res = ref.moe_layer(logits, x, W1, W3, Wd, R=R, tbM=tbM, k=k)
    want = brute_layer(logits.tolist(), x.tolist(), W1.tolist(), W3.tolist(), W2.tolist(), k)
    assert not np.allclose(res.out, want, atol=1e-9)


def test_plan_pin_catches_swapped_owners(monkeypatch):
    """A planted owner mistake (blocks in reverse order) must fail the plan pin."""
    from tests.test_oracle_plan import brute_plan
    rng = np.random.default_rng(22)
    T, E, k, R, tbM = 16, 3, 2, 2, 4
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    orig = ref.owners
    monkeypatch.setattr(ref, "owners", lambda T_, R_: (R_ - 1) - orig(T_, R_))
    plan = ref.build_plan(idx, E, R, tbM)
    _, slot, _, ret_slot, _ = brute_plan(idx.tolist(), E, R, tbM)
    assert not (np.array_equal(plan.slot, slot) and np.array_equal(plan.ret_slot, ret_slot))
