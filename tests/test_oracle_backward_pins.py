"""Pins of the oracle's backward of the column/row pair, without the GPU.

What fixes the backward independently of the oracle's own formulas:
  * central finite differences of the forward (mlp_block) on tiny float64
    inputs: every entry of X, W1, W_up and W2;
  * tp invariance: sharded gradients equal the unsharded ones (tp = 1);
  * brute force on small integer inputs (explicit sums over indices) for
    the activations whose gradient is exact on integers (none, ReLU);
  * closed forms of the linear case (act = none);
  * planted mistakes (a dropped derivative term, a missing shard in the
    input-gradient sum, a transposed weight) that the checks must catch.
"""
import itertools

import numpy as np
import pytest

from oracle import tp_oracle as O

ACTS = ["none", "relu", "gelu", "silu", "swiglu"]


def _loss(X, W1, W2, Wu, dY, dR, tp, act):
    """L = <Y, dY> + <X, dR>: its gradient is the backward of dY (and dR)."""
    _, Y = O.mlp_block(X, W1, W2, tp, act, W_up=Wu)
    return float(np.sum(Y * dY) + np.sum(X * dR))


def _fd_errors(seed, act, tp=2, T=3, H=4, I=6, eps=1e-6):
    r = np.random.default_rng(seed)
    X, W1, W2 = r.normal(size=(T, H)), r.normal(size=(H, I)), r.normal(size=(I, H))
    Wu = r.normal(size=(H, I)) if act == "swiglu" else None
    dY, dR = r.normal(size=(T, H)), r.normal(size=(T, H))
    g = O.mlp_backward(X, W1, W2, tp, dY, act, W_up=Wu, dR=dR)
    got = {"X": g["dX"], "W1": np.concatenate(g["dW1"], 1), "W2": np.concatenate(g["dW2"], 0)}
    if Wu is not None:
        got["Wu"] = np.concatenate(g["dW_up"], 1)
    params = {"X": X, "W1": W1, "W2": W2, "Wu": Wu}
    err = {}
    for name in got:
        P = params[name]
        num = np.zeros_like(P)
        for idx in itertools.product(*map(range, P.shape)):
            old = P[idx]
            P[idx] = old + eps
            lp = _loss(params["X"], params["W1"], params["W2"], params["Wu"], dY, dR, tp, act)
            P[idx] = old - eps
            lm = _loss(params["X"], params["W1"], params["W2"], params["Wu"], dY, dR, tp, act)
            P[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        err[name] = float(np.max(np.abs(num - got[name])) / (np.max(np.abs(num)) + 1e-30))
    return err


@pytest.mark.parametrize("act", ACTS)
def test_mlp_backward_matches_finite_differences(act):
    err = _fd_errors(11, act)
    assert max(err.values()) < 1e-7, err


@pytest.mark.parametrize("act", ["relu", "swiglu"])
@pytest.mark.parametrize("tp", [1, 3, 6])
def test_mlp_backward_finite_differences_every_tp(act, tp):
    err = _fd_errors(12 + tp, act, tp=tp)
    assert max(err.values()) < 1e-7, err


@pytest.mark.parametrize("act", ACTS)
def test_mlp_backward_tp_invariant(act):
    """Shard gradients, put back together, equal the unsharded (tp = 1) ones."""
    r = np.random.default_rng(21)
    T, H, I = 5, 6, 12
    X, W1, W2, dY = r.normal(size=(T, H)), r.normal(size=(H, I)), r.normal(size=(I, H)), r.normal(size=(T, H))
    Wu = r.normal(size=(H, I)) if act == "swiglu" else None
    ref = O.mlp_backward(X, W1, W2, 1, dY, act, W_up=Wu)
    for tp in (2, 3, 4, 6, 12):
        g = O.mlp_backward(X, W1, W2, tp, dY, act, W_up=Wu)
        np.testing.assert_allclose(g["dX"], ref["dX"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(np.concatenate(g["dW1"], 1), ref["dW1"][0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(np.concatenate(g["dW2"], 0), ref["dW2"][0], rtol=1e-12, atol=1e-12)
        if Wu is not None:
            np.testing.assert_allclose(np.concatenate(g["dW_up"], 1), ref["dW_up"][0], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["none", "relu"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_mlp_backward_int_bruteforce(act, seed):
    """Integer inputs, gradients written as explicit index sums."""
    r = np.random.default_rng(100 + seed)
    T, H, I, tp = 3, 4, 6, 2
    X = r.integers(-3, 4, size=(T, H)).astype(np.int64)
    W1 = r.integers(-3, 4, size=(H, I)).astype(np.int64)
    W2 = r.integers(-3, 4, size=(I, H)).astype(np.int64)
    dY = r.integers(-3, 4, size=(T, H)).astype(np.int64)
    g = O.mlp_backward(X, W1, W2, tp, dY, act)
    G = [[sum(X[t][h] * W1[h][i] for h in range(H)) for i in range(I)] for t in range(T)]
    on = [[1 if (act == "none" or G[t][i] > 0) else 0 for i in range(I)] for t in range(T)]
    Hs = [[G[t][i] * on[t][i] for i in range(I)] for t in range(T)]
    dH = [[sum(dY[t][h] * W2[i][h] for h in range(H)) for i in range(I)] for t in range(T)]
    dG = [[dH[t][i] * on[t][i] for i in range(I)] for t in range(T)]
    dX = [[sum(dG[t][i] * W1[h][i] for i in range(I)) for h in range(H)] for t in range(T)]
    dW1 = [[sum(X[t][h] * dG[t][i] for t in range(T)) for i in range(I)] for h in range(H)]
    dW2 = [[sum(Hs[t][i] * dY[t][h] for t in range(T)) for h in range(H)] for i in range(I)]
    assert g["dX"].dtype == np.int64
    np.testing.assert_array_equal(g["dX"], np.array(dX))
    np.testing.assert_array_equal(np.concatenate(g["dW1"], 1), np.array(dW1))
    np.testing.assert_array_equal(np.concatenate(g["dW2"], 0), np.array(dW2))


def test_linear_case_closed_forms():
    """act = none: Y = X W1 W2, so dX = dY (W1 W2)^T, dW1 = X^T dY W2^T,
    dW2 = (X W1)^T dY."""
    r = np.random.default_rng(31)
    X, W1, W2, dY = r.normal(size=(4, 6)), r.normal(size=(6, 8)), r.normal(size=(8, 6)), r.normal(size=(4, 6))
    g = O.mlp_backward(X, W1, W2, 4, dY, "none")
    np.testing.assert_allclose(g["dX"], dY @ (W1 @ W2).T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(g["dW1"], 1), X.T @ dY @ W2.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(g["dW2"], 0), (X @ W1).T @ dY, rtol=1e-12, atol=1e-12)


def test_row_backward_hands_every_shard_the_same_dy():
    """The forward all-reduce is an identity in the backward: shard s's
    input gradient is dY @ W_s^T with the full dY."""
    r = np.random.default_rng(41)
    W, dY = r.normal(size=(6, 4)), r.normal(size=(3, 4))
    Xs = O.split_columns(r.normal(size=(3, 6)), 3)
    dXs, _ = O.row_linear_backward(Xs, W, 3, dY)
    for s in range(3):
        np.testing.assert_allclose(dXs[s], dY @ W[2 * s:2 * s + 2].T, rtol=1e-12)


def test_column_backward_input_gradient_is_the_shard_sum():
    r = np.random.default_rng(42)
    X, W = r.normal(size=(3, 4)), r.normal(size=(4, 6))
    dYs = [r.normal(size=(3, 2)) for _ in range(3)]
    dX, dW = O.column_linear_backward(X, W, 3, dYs)
    want = sum(dYs[s] @ W[:, 2 * s:2 * s + 2].T for s in range(3))
    np.testing.assert_allclose(dX, want, rtol=1e-12)
    for s in range(3):
        np.testing.assert_allclose(dW[s], X.T @ dYs[s], rtol=1e-12)


@pytest.mark.parametrize("act", ["relu", "swiglu"])
def test_backward_from_saved_values_int_bruteforce(act):
    """Saved values that need not come from this X (a training step hands
    over whatever the forward stored): the formulas as explicit index sums
    on small integers."""
    r = np.random.default_rng(51)
    T, H, I, tp = 3, 4, 6, 3
    X, W1, Wu, W2, dY = (r.integers(-3, 4, size=sh).astype(np.int64)
                         for sh in ((T, H), (H, I), (H, I), (I, H), (T, H)))
    G = r.integers(-3, 4, size=(T, I)).astype(np.int64)
    U = r.integers(-3, 4, size=(T, I)).astype(np.int64)
    Hs = r.integers(-3, 4, size=(T, I)).astype(np.int64)
    parts = lambda M: [M[:, s * 2:(s + 1) * 2] for s in range(tp)]
    g = O.mlp_backward_saved(X, W1, W2, tp, dY, parts(G), parts(Hs), act, W_up=Wu if act == "swiglu" else None,
                             U=parts(U) if act == "swiglu" else None)
    dH = [[sum(dY[t][h] * W2[i][h] for h in range(H)) for i in range(I)] for t in range(T)]
    if act == "relu":
        dG = [[dH[t][i] * (1 if G[t][i] > 0 else 0) for i in range(I)] for t in range(T)]
        dX = [[sum(dG[t][i] * W1[h][i] for i in range(I)) for h in range(H)] for t in range(T)]
        np.testing.assert_array_equal(g["dX"], np.array(dX))
    else:
        sg = 1.0 / (1.0 + np.exp(-G.astype(np.float64)))
        dG = np.array(dH) * U * sg * (1 + G * (1 - sg))
        dU = np.array(dH) * G * sg
        np.testing.assert_allclose(g["dX"], dG @ W1.T + dU @ Wu.T, rtol=1e-12)
        np.testing.assert_allclose(np.concatenate(g["dW_up"], 1), X.T @ dU, rtol=1e-12)
    dW2 = [[sum(Hs[t][i] * dY[t][h] for t in range(T)) for h in range(H)] for i in range(I)]
    np.testing.assert_array_equal(np.concatenate(g["dW2"], 0), np.array(dW2))


def test_activation_backward_special_values():
    g = np.array([-2.0, 0.0, 3.0])
    dh = np.ones(3)
    np.testing.assert_array_equal(O.activation_backward("relu", g, dh)[0], [0.0, 0.0, 1.0])
    assert O.activation_backward("gelu", np.array([0.0]), np.ones(1))[0][0] == pytest.approx(0.5)
    assert O.activation_backward("silu", np.array([0.0]), np.ones(1))[0][0] == pytest.approx(0.5)
    dG, dU = O.activation_backward("swiglu", np.array([0.0]), np.ones(1), np.array([2.0]))
    assert dG[0] == pytest.approx(1.0) and dU[0] == pytest.approx(0.0)


# --- planted mistakes (in the oracle, on the CPU) --------------------------

def test_planted_dropped_silu_term_is_caught(monkeypatch):
    real = O.activation_backward

    def wrong(act, G, dH, U=None):
        if act == "swiglu":
            sg = 1.0 / (1.0 + np.exp(-G))
            return dH * U * sg, dH * G * sg  # silu' without its g (1 - s) term
        return real(act, G, dH, U)

    monkeypatch.setattr(O, "activation_backward", wrong)
    assert max(_fd_errors(11, "swiglu").values()) > 1e-3


def test_planted_missing_shard_in_input_gradient_is_caught(monkeypatch):
    def wrong(X, W, tp, dYs, dR=None):
        Ws = O.column_shards(W, tp)
        dX = dYs[0] @ Ws[0].T  # the other shards' shares left out
        if dR is not None:
            dX = dX + dR
        return dX, [X.T @ dYs[s] for s in range(tp)]

    monkeypatch.setattr(O, "column_linear_backward", wrong)
    err = _fd_errors(11, "relu")
    assert err["X"] > 1e-3


def test_planted_transposed_row_weight_gradient_is_caught(monkeypatch):
    def wrong(Xs, W, tp, dY):
        Ws = O.row_shards(W, tp)
        return [dY @ Ws[s].T for s in range(tp)], [(dY.T @ Xs[s]).T[::-1] for s in range(tp)]

    monkeypatch.setattr(O, "row_linear_backward", wrong)
    assert _fd_errors(11, "gelu")["W2"] > 1e-3
