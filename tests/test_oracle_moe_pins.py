"""Pins of the oracle's mixture of experts with tensor-parallel experts,
without the GPU: a single expert with weight 1 is the MLP block, linearity
in the routing weights, tp invariance, relabelling experts, integer brute
force, and a planted mistake."""
import numpy as np
import pytest

from oracle import tp_oracle as O


def experts(seed, E, H, I, act="swiglu", ints=False):
    r = np.random.default_rng(seed)
    draw = (lambda sh: r.integers(-2, 3, size=sh).astype(np.int64)) if ints else (lambda sh: r.normal(size=sh))
    return [dict(W1=draw((H, I)), W_up=draw((H, I)) if act == "swiglu" else None, W2=draw((I, H))) for _ in range(E)]


def test_single_expert_weight_one_is_the_mlp_block():
    r = np.random.default_rng(1)
    X = r.normal(size=(7, 8))
    ex = experts(2, 3, 8, 12)
    ids = np.full((7, 1), 2)
    Y = O.moe_tp(X, ex, ids, np.ones((7, 1)), 4)
    _, want = O.mlp_block(X, ex[2]["W1"], ex[2]["W2"], 4, "swiglu", W_up=ex[2]["W_up"])
    np.testing.assert_allclose(Y, want, rtol=1e-13)


def test_weighted_sum_of_experts():
    r = np.random.default_rng(3)
    X = r.normal(size=(5, 6))
    ex = experts(4, 4, 6, 8)
    ids = np.array([[0, 1], [2, 3], [1, 1], [3, 0], [2, 2]])
    w = r.random(size=(5, 2))
    Y = O.moe_tp(X, ex, ids, w, 2)
    for t in range(5):
        want = sum(w[t, j] * O.mlp_block(X[t:t + 1], ex[ids[t, j]]["W1"], ex[ids[t, j]]["W2"], 2, "swiglu",
                                         W_up=ex[ids[t, j]]["W_up"])[1][0] for j in range(2))
        np.testing.assert_allclose(Y[t], want, rtol=1e-12)


@pytest.mark.parametrize("tp", [1, 2, 4])
def test_tp_invariant_and_relabelling(tp):
    r = np.random.default_rng(5)
    X = r.normal(size=(9, 8))
    ex = experts(6, 4, 8, 16)
    ids = r.integers(0, 4, size=(9, 2))
    w = r.random(size=(9, 2))
    ref = O.moe_tp(X, ex, ids, w, 1)
    np.testing.assert_allclose(O.moe_tp(X, ex, ids, w, tp), ref, rtol=1e-12, atol=1e-12)
    perm = np.array([2, 0, 3, 1])  # expert e becomes perm[e]
    ex2 = [None] * 4
    for e in range(4):
        ex2[perm[e]] = ex[e]
    np.testing.assert_allclose(O.moe_tp(X, ex2, perm[ids], w, tp), ref, rtol=1e-12, atol=1e-12)


def test_int_bruteforce_relu():
    r = np.random.default_rng(7)
    T, H, I, E, k, tp = 4, 3, 4, 3, 2, 2
    X = r.integers(-2, 3, size=(T, H)).astype(np.int64)
    ex = experts(8, E, H, I, act="relu", ints=True)
    ids = r.integers(0, E, size=(T, k))
    w = r.integers(1, 4, size=(T, k)).astype(np.int64)
    Y = O.moe_tp(X, ex, ids, w, tp, act="relu")
    for t in range(T):
        for h in range(H):
            tot = 0
            for j in range(k):
                W1, W2 = ex[ids[t][j]]["W1"], ex[ids[t][j]]["W2"]
                hid = [max(0, sum(X[t][a] * W1[a][i] for a in range(H))) for i in range(I)]
                tot += w[t][j] * sum(hid[i] * W2[i][h] for i in range(I))
            assert Y[t][h] == tot


def test_residual_and_unused_expert():
    r = np.random.default_rng(9)
    X = r.normal(size=(4, 6))
    ex = experts(10, 3, 6, 8)
    ids = np.array([[0], [0], [2], [2]])  # expert 1 unused
    R = r.normal(size=(4, 6))
    np.testing.assert_allclose(O.moe_tp(X, ex, ids, np.ones((4, 1)), 2, residual=R) - R,
                               O.moe_tp(X, ex, ids, np.ones((4, 1)), 2), rtol=1e-12, atol=1e-12)


def test_planted_wrong_expert_is_caught(monkeypatch):
    r = np.random.default_rng(11)
    X = r.normal(size=(5, 6))
    ex = experts(12, 3, 6, 8)
    ids = np.array([[0], [1], [2], [1], [0]])
    ref = O.moe_tp(X, ex, ids, np.ones((5, 1)), 2)
    real = O.mlp_block
    calls = []

    def wrong(Xr, W1, W2, tp, act="relu", W_up=None, **kw):  # the up projection of the wrong expert
        calls.append(1)
        return real(Xr, W1, W2, tp, act, W_up=ex[(len(calls)) % 3]["W_up"], **kw)
    monkeypatch.setattr(O, "mlp_block", wrong)
    assert not np.allclose(O.moe_tp(X, ex, ids, np.ones((5, 1)), 2), ref)
