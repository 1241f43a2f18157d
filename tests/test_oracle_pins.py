"""Pins for the oracle, on the CPU.

Each test checks the oracle against something other than itself: the values
printed in the pages' worked example, brute force on tiny integer inputs,
closed forms, library routines (scipy's normal CDF and logistic function),
and invariants that the pages state (column shards concatenate to the
unsharded product; row-shard contributions sum to it). A plausible mistake in
the oracle (a dropped shard, a wrong block index, a transposed operand, a
swapped gate/up, a bias added per shard) fails at least one of them; the
``test_planted_*`` cases plant such mistakes in the oracle and check that.
"""
import itertools
import math

import numpy as np
import pytest
from scipy.special import expit
from scipy.stats import norm

from oracle import tp_oracle as O
import synth_inputs as S


# ---------------------------------------------------------------------------
# Helpers independent of the oracle
# ---------------------------------------------------------------------------

def brute_matmul(X, W):
    """Pure-Python triple loop: y[t][n] = sum_k x[t][k] * w[k][n]."""
    T, K = len(X), len(X[0])
    N = len(W[0])
    return [[sum(X[t][k] * W[k][n] for k in range(K)) for n in range(N)]
            for t in range(T)]


def brute_mlp(X, W1, W2, act):
    h = [[act(v) for v in row] for row in brute_matmul(X, W1)]
    return brute_matmul(h, W2)


def divisors(n):
    return [d for d in range(1, n + 1) if n % d == 0]


def rand_ints(rng, shape, lo=-2, hi=2):
    return rng.integers(lo, hi + 1, size=shape).astype(np.int64)


# ---------------------------------------------------------------------------
# 1. The worked example, values as printed on the page
# ---------------------------------------------------------------------------

def test_worked_example_unsharded(golden_worked_example):
    g = golden_worked_example
    X = np.array(g["X"], np.int64)
    W = np.array(g["W"], np.int64)
    assert O.linear(X, W).tolist() == g["XW"]


def test_worked_example_column_parallel(golden_worked_example):
    g = golden_worked_example
    X, W = np.array(g["X"], np.int64), np.array(g["W"], np.int64)
    W0, W1 = O.column_shards(W, 2)
    assert W0.tolist() == g["col_W0"] and W1.tolist() == g["col_W1"]
    Y0, Y1 = O.column_parallel(X, W, 2)
    assert Y0.tolist() == g["col_Y0"] and Y1.tolist() == g["col_Y1"]
    assert O.all_gather([Y0, Y1]).tolist() == g["all_gather"]


def test_worked_example_row_parallel(golden_worked_example):
    g = golden_worked_example
    X, W = np.array(g["X"], np.int64), np.array(g["W"], np.int64)
    X0, X1 = O.split_columns(X, 2)
    assert X0.tolist() == g["row_X0"] and X1.tolist() == g["row_X1"]
    W0, W1 = O.row_shards(W, 2)
    assert W0.tolist() == g["row_W0"] and W1.tolist() == g["row_W1"]
    P0, P1 = O.row_parallel_partials([X0, X1], W, 2)
    assert P0.tolist() == g["row_P0"] and P1.tolist() == g["row_P1"]
    assert O.all_reduce([P0, P1]).tolist() == g["all_reduce"]


def test_worked_example_from_input_generator(golden_worked_example):
    X, W = S.worked_example()
    assert X.astype(np.int64).tolist() == golden_worked_example["X"]
    assert W.astype(np.int64).tolist() == golden_worked_example["W"]


# ---------------------------------------------------------------------------
# 2. Brute force on tiny integer inputs, every tp that divides the dims
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_column_parallel_concat_equals_bruteforce(seed):
    rng = np.random.default_rng(seed)
    T, K, N = 2, 3, 12
    X, W = rand_ints(rng, (T, K)), rand_ints(rng, (K, N))
    ref = brute_matmul(X.tolist(), W.tolist())
    for tp in divisors(N):
        parts = O.column_parallel(X, W, tp)
        assert [p.shape for p in parts] == [(T, N // tp)] * tp
        assert O.all_gather(parts).tolist() == ref
        # shard s holds exactly output columns [s*N/tp, (s+1)*N/tp)
        for s, p in enumerate(parts):
            assert p.tolist() == [row[s * N // tp:(s + 1) * N // tp] for row in ref]


@pytest.mark.parametrize("seed", range(6))
def test_row_parallel_sum_equals_bruteforce(seed):
    rng = np.random.default_rng(100 + seed)
    T, K, N = 2, 12, 3
    X, W = rand_ints(rng, (T, K)), rand_ints(rng, (K, N))
    ref = brute_matmul(X.tolist(), W.tolist())
    for tp in divisors(K):
        Xs = O.split_columns(X, tp)
        P = O.row_parallel_partials(Xs, W, tp)
        assert O.all_reduce(P).tolist() == ref
        # each partial is the contribution of its own K block only
        k = K // tp
        for s in range(tp):
            sub = brute_matmul(X[:, s * k:(s + 1) * k].tolist(), W[s * k:(s + 1) * k].tolist())
            assert P[s].tolist() == sub


def test_enumerated_2x2_all_values():
    """Every X in {-1,0,1}^2 against a fixed W, column and row splits."""
    W = np.array([[1, -2], [3, 2]], np.int64)
    for xs in itertools.product([-1, 0, 1], repeat=2):
        X = np.array([xs], np.int64)
        ref = brute_matmul(X.tolist(), W.tolist())
        assert O.all_gather(O.column_parallel(X, W, 2)).tolist() == ref
        assert O.all_reduce(O.row_parallel_partials(O.split_columns(X, 2), W, 2)).tolist() == ref


def test_indivisible_dims_rejected():
    W = np.zeros((4, 6), np.int64)
    with pytest.raises(ValueError):
        O.column_shards(W, 4)
    with pytest.raises(ValueError):
        O.row_shards(W, 3)


# ---------------------------------------------------------------------------
# 3. The MLP block: column -> local act -> row -> sum == unsharded, all tp
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_mlp_relu_int_all_tp_bruteforce(seed):
    rng = np.random.default_rng(200 + seed)
    T, H, I = 3, 4, 12
    X, W1, W2 = rand_ints(rng, (T, H)), rand_ints(rng, (H, I)), rand_ints(rng, (I, H))
    ref = brute_mlp(X.tolist(), W1.tolist(), W2.tolist(), lambda v: max(v, 0))
    for tp in divisors(I):
        Hs, Y = O.mlp_block(X, W1, W2, tp, "relu")
        assert Y.tolist() == ref
        assert len(Hs) == tp


@pytest.mark.parametrize("act", ["gelu", "silu", "none"])
def test_mlp_float_acts_all_tp(act):
    rng = np.random.default_rng(7)
    T, H, I = 3, 4, 8
    X = rng.standard_normal((T, H))
    W1, W2 = rng.standard_normal((H, I)), rng.standard_normal((I, H))
    f = {"gelu": lambda v: v * norm.cdf(v), "silu": lambda v: v * expit(v),
         "none": lambda v: v}[act]
    ref = np.array(brute_mlp(X.tolist(), W1.tolist(), W2.tolist(), f))
    for tp in divisors(I):
        _, Y = O.mlp_block(X, W1, W2, tp, act)
        np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_mlp_swiglu_all_tp():
    rng = np.random.default_rng(8)
    T, H, I = 2, 4, 8
    X = rng.standard_normal((T, H))
    Wg, Wu, Wd = (rng.standard_normal(s) for s in [(H, I), (H, I), (I, H)])
    g = np.array(brute_matmul(X.tolist(), Wg.tolist()))
    u = np.array(brute_matmul(X.tolist(), Wu.tolist()))
    h = g * expit(g) * u
    ref = np.array(brute_matmul(h.tolist(), Wd.tolist()))
    for tp in divisors(I):
        _, Y = O.mlp_block(X, Wg, Wd, tp, "swiglu", W_up=Wu)
        np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_mlp_bias_once_and_residual():
    """Row bias enters once after the sum (not once per shard); the column
    bias is split with its columns; the residual adds once."""
    X = np.array([[1, 0]], np.int64)
    W1 = np.array([[1, 2, 3, 4], [0, 0, 0, 0]], np.int64)
    W2 = np.eye(4, 2, dtype=np.int64)  # picks h[0], h[1]
    b1 = np.array([10, 20, 30, 40], np.int64)
    b2 = np.array([100, 200], np.int64)
    R = np.array([[1000, 2000]], np.int64)
    for tp in (1, 2, 4):
        Hs, Y = O.mlp_block(X, W1, W2, tp, "none", b1=b1, b2=b2, residual=R)
        assert O.all_gather(Hs).tolist() == [[11, 22, 33, 44]]
        assert Y.tolist() == [[1111, 2222]]


# ---------------------------------------------------------------------------
# 4. Closed forms
# ---------------------------------------------------------------------------

def test_closed_forms():
    rng = np.random.default_rng(3)
    K, N = 6, 8
    W = rand_ints(rng, (K, N), -5, 5)
    for tp in (1, 2, 4, 8):
        for k in range(K):  # X = e_k picks row k of W
            e = np.zeros((1, K), np.int64)
            e[0, k] = 1
            assert O.all_gather(O.column_parallel(e, W, tp)).tolist() == [W[k].tolist()]
        ones = np.ones((1, K), np.int64)  # X = ones gives column sums
        assert O.all_gather(O.column_parallel(ones, W, tp)).tolist() == [
            [int(sum(W[k, n] for k in range(K))) for n in range(N)]]
    X = rand_ints(rng, (3, N))
    for tp in (1, 2, 4, 8):  # W = I returns X, in both splits
        Ieye = np.eye(N, dtype=np.int64)
        assert O.all_gather(O.column_parallel(X, Ieye, tp)).tolist() == X.tolist()
        assert O.all_reduce(O.row_parallel_partials(O.split_columns(X, tp), Ieye, tp)).tolist() == X.tolist()


def test_tp1_is_plain_product():
    rng = np.random.default_rng(4)
    X, W = rand_ints(rng, (3, 5)), rand_ints(rng, (5, 7))
    ref = brute_matmul(X.tolist(), W.tolist())
    assert O.column_parallel(X, W, 1)[0].tolist() == ref
    assert O.row_parallel_partials([X], W, 1)[0].tolist() == ref


# ---------------------------------------------------------------------------
# 5. Combine operators
# ---------------------------------------------------------------------------

def test_reduce_scatter_explicit():
    P0 = np.array([[1, 2], [3, 4], [5, 6], [7, 8]], np.int64)
    P1 = np.array([[10, 20], [30, 40], [50, 60], [70, 80]], np.int64)
    out = O.reduce_scatter([P0, P1], 2)
    assert [o.tolist() for o in out] == [[[11, 22], [33, 44]], [[55, 66], [77, 88]]]
    out4 = O.reduce_scatter([P0, P1], 4)
    assert [o.tolist() for o in out4] == [[[11, 22]], [[33, 44]], [[55, 66]], [[77, 88]]]
    with pytest.raises(ValueError):
        O.reduce_scatter([P0, P1], 3)


def test_all_reduce_worked_partials_in_order():
    # the page's two contributions; and a three-way sum checked by hand
    assert O.all_reduce([np.array([10, 20, 30, 40]), np.array([100, 120, 140, 160])]).tolist() == [110, 140, 170, 200]
    assert O.all_reduce([np.array([1]), np.array([2]), np.array([4])]).tolist() == [7]


# ---------------------------------------------------------------------------
# 6. Activations against library routines and special values
# ---------------------------------------------------------------------------

def test_activations_against_library():
    x = np.linspace(-6, 6, 97)
    np.testing.assert_allclose(O.gelu(x), x * norm.cdf(x), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(O.silu(x), x * expit(x), rtol=1e-14, atol=1e-15)
    assert O.relu(np.array([-3, 0, 2])).tolist() == [0, 0, 2]
    assert O.gelu(np.array([0.0]))[0] == 0.0 and O.silu(np.array([0.0]))[0] == 0.0
    # GELU(1) = Phi(1); SiLU(1) = 1/(1+e^-1)
    assert abs(O.gelu(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    assert abs(O.silu(np.array([1.0]))[0] - 0.7310585786300049) < 1e-15


def test_swiglu_gate_is_the_silu_operand():
    g, u = np.array([1.0]), np.array([2.0])
    assert abs(O.swiglu(g, u)[0] - 2 * 0.7310585786300049) < 1e-15
    assert abs(O.swiglu(u, g)[0] - 1.7615941559557646) < 1e-15  # silu(2)*1


# ---------------------------------------------------------------------------
# 7. Attention projections: heads, KV replication, the single-key context
# ---------------------------------------------------------------------------

def test_qkv_head_layout_explicit():
    # 32 q / 8 kv heads: tp=2 splits both; tp=16 replicates each kv head twice
    L2 = O.qkv_head_layout(32, 8, 2)
    assert L2[0] == (list(range(16)), [0, 1, 2, 3])
    assert L2[1] == (list(range(16, 32)), [4, 5, 6, 7])
    L8 = O.qkv_head_layout(32, 8, 8)
    assert [kv for _, kv in L8] == [[s] for s in range(8)]
    L16 = O.qkv_head_layout(32, 8, 16)
    assert [q for q, _ in L16] == [[2 * s, 2 * s + 1] for s in range(16)]
    assert [kv for _, kv in L16] == [[s // 2] for s in range(16)]
    # every q head's kv head (h // 4) sits on the q head's shard
    for tp in (1, 2, 4, 8, 16, 32):
        for q, kv in O.qkv_head_layout(32, 8, tp):
            assert all(h // 4 in kv for h in q)
    with pytest.raises(ValueError):
        O.qkv_head_layout(32, 8, 3)
    with pytest.raises(ValueError):
        O.qkv_head_layout(32, 6, 4)  # hq not a multiple of hkv


@pytest.mark.parametrize("tp", [1, 2, 4, 8, 16])
def test_qkv_shards_dedup_equals_unsharded(tp):
    rng = np.random.default_rng(tp)
    H, hq, hkv, hd, T = 4, 16, 8, 2, 3
    Wq = rand_ints(rng, (H, hq * hd))
    Wk, Wv = rand_ints(rng, (H, hkv * hd)), rand_ints(rng, (H, hkv * hd))
    X = rand_ints(rng, (T, H))
    ref = np.array(brute_matmul(X.tolist(), np.concatenate([Wq, Wk, Wv], 1).tolist()))
    layout = O.qkv_head_layout(hq, hkv, tp)
    shards = O.qkv_shards(Wq, Wk, Wv, hq, hkv, hd, tp)
    q_seen, kv_seen = {}, {}
    for s in range(tp):
        y = O.linear(X, shards[s])
        q, kv = layout[s]
        for j, h in enumerate(q):
            q_seen[h] = y[:, j * hd:(j + 1) * hd]
        base = len(q) * hd
        for j, h in enumerate(kv):
            k = y[:, base + j * hd: base + (j + 1) * hd]
            v = y[:, base + (len(kv) + j) * hd: base + (len(kv) + j + 1) * hd]
            if h in kv_seen:  # a replica must equal the first copy
                assert (kv_seen[h][0] == k).all() and (kv_seen[h][1] == v).all()
            kv_seen[h] = (k, v)
    assert sorted(q_seen) == list(range(hq)) and sorted(kv_seen) == list(range(hkv))
    Q = np.concatenate([q_seen[h] for h in range(hq)], 1)
    K = np.concatenate([kv_seen[h][0] for h in range(hkv)], 1)
    V = np.concatenate([kv_seen[h][1] for h in range(hkv)], 1)
    assert np.concatenate([Q, K, V], 1).tolist() == ref.tolist()


def brute_attention_self_only(Q, K, V, hq, hkv, hd):
    """Scaled dot-product attention per head with a mask that lets token t
    see only key t: the softmax runs over a single score."""
    T = Q.shape[0]
    group = hq // hkv
    out = np.zeros((T, hq * hd))
    for h in range(hq):
        g = h // group
        for t in range(T):
            scores = {}
            for j in range(T):
                if j == t:  # the only unmasked key
                    scores[j] = float(Q[t, h * hd:(h + 1) * hd] @ K[j, g * hd:(g + 1) * hd]) / np.sqrt(hd)
            m = max(scores.values())
            z = sum(np.exp(v - m) for v in scores.values())
            for j, v in scores.items():
                out[t, h * hd:(h + 1) * hd] += np.exp(v - m) / z * V[j, g * hd:(g + 1) * hd]
    return out


@pytest.mark.parametrize("tp", [1, 2, 4, 8, 16])
def test_context_standin_is_single_key_attention(tp):
    rng = np.random.default_rng(50 + tp)
    H, hq, hkv, hd, T = 6, 16, 8, 2, 3
    Wq, Wk, Wv = (rng.standard_normal(s) for s in [(H, hq * hd), (H, hkv * hd), (H, hkv * hd)])
    Wo = rng.standard_normal((hq * hd, H))
    X = rng.standard_normal((T, H))
    Q, K, V = X @ Wq, X @ Wk, X @ Wv
    ctx_ref = brute_attention_self_only(Q, K, V, hq, hkv, hd)
    qkv, ctx, Y = O.attn_proj(X, Wq, Wk, Wv, Wo, hq, hkv, hd, tp)
    np.testing.assert_allclose(O.all_gather(ctx), ctx_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Y, ctx_ref @ Wo, rtol=1e-11, atol=1e-11)


def test_attn_proj_int_residual_and_explicit_ctx():
    rng = np.random.default_rng(9)
    H, hq, hkv, hd, T, tp = 4, 4, 2, 2, 2, 4
    Wq, Wk, Wv = rand_ints(rng, (H, 8)), rand_ints(rng, (H, 4)), rand_ints(rng, (H, 4))
    Wo = rand_ints(rng, (8, H))
    X, R = rand_ints(rng, (T, H)), rand_ints(rng, (T, H))
    ctx = [rand_ints(rng, (T, 2)) for _ in range(tp)]
    _, _, Y = O.attn_proj(X, Wq, Wk, Wv, Wo, hq, hkv, hd, tp, ctx=ctx, residual=R)
    full_ctx = np.concatenate(ctx, 1)
    assert Y.tolist() == (np.array(brute_matmul(full_ctx.tolist(), Wo.tolist())) + R).tolist()


# ---------------------------------------------------------------------------
# 8. RMSNorm and the stack
# ---------------------------------------------------------------------------

def test_rmsnorm_values():
    x = np.array([[3.0, 4.0]])
    y = O.rmsnorm(x, None, eps=0.0)
    np.testing.assert_allclose(y, [[3 / np.sqrt(12.5), 4 / np.sqrt(12.5)]], rtol=1e-15)
    y = O.rmsnorm(x, np.array([2.0, -1.0]), eps=1e-5)
    d = np.sqrt(12.5 + 1e-5)
    np.testing.assert_allclose(y, [[6 / d, -4 / d]], rtol=1e-15)
    c = np.full((1, 8), -2.5)
    np.testing.assert_allclose(O.rmsnorm(c, None, eps=0.0), -np.ones((1, 8)), rtol=1e-15)


def _tiny_stack(rng, H=8, I=16, hq=4, hkv=2, hd=2, V=8, layers=2):
    f = lambda *s: rng.standard_normal(s) * 0.3
    Ls = [dict(Wq=f(H, hq * hd), Wk=f(H, hkv * hd), Wv=f(H, hkv * hd), Wo=f(hq * hd, H),
               Wg=f(H, I), Wu=f(H, I), Wd=f(I, H)) for _ in range(layers)]
    return Ls, f(H, V), f(3, H)


def test_stack_tp_invariant():
    rng = np.random.default_rng(11)
    Ls, Wlm, X = _tiny_stack(rng)
    ref = O.stack_forward(X, Ls, Wlm, 1, 4, 2, 2)
    for tp in (2, 4):
        np.testing.assert_allclose(O.stack_forward(X, Ls, Wlm, tp, 4, 2, 2), ref, rtol=1e-12, atol=1e-12)


def test_stack_block_wiring_against_explicit_steps():
    """One block written out step by step with library primitives only."""
    rng = np.random.default_rng(12)
    Ls, Wlm, X = _tiny_stack(rng, layers=1)
    L = Ls[0]
    eps = 1e-5
    nrm = lambda x: x / np.sqrt((x ** 2).mean(-1, keepdims=True) + eps)
    h = nrm(X)
    V = h @ L["Wv"]
    ctx = np.concatenate([V[:, (q // 2) * 2:(q // 2) * 2 + 2] for q in range(4)], 1)
    x = X + ctx @ L["Wo"]
    h = nrm(x)
    g, u = h @ L["Wg"], h @ L["Wu"]
    x = x + (g * expit(g) * u) @ L["Wd"]
    ref = nrm(x) @ Wlm
    np.testing.assert_allclose(O.stack_forward(X, Ls, Wlm, 2, 4, 2, 2), ref, rtol=1e-12, atol=1e-12)


def test_stack_zero_weights_is_norm_then_head():
    rng = np.random.default_rng(13)
    Ls, Wlm, X = _tiny_stack(rng)
    for L in Ls:
        for k in L:
            L[k] = np.zeros_like(L[k])
    out = O.stack_forward(X, Ls, Wlm, 2, 4, 2, 2)
    np.testing.assert_allclose(out, O.rmsnorm(X) @ Wlm, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# 9. Input generator properties (the values both sides start from)
# ---------------------------------------------------------------------------

def test_input_generator_deterministic_and_bf16():
    a = S.normal(3, (257, 129), 0.02)
    b = S.normal(3, (257, 129), 0.02)
    assert (a == b).all() and a.dtype == np.float32
    assert (a.view(np.uint32) & 0xFFFF == 0).all()  # bf16-representable
    assert abs(a.std() - 0.02) < 0.002
    i = S.uniform_ints(0, (16, 64))
    assert set(np.unique(i).tolist()) <= set(range(-3, 4)) and len(np.unique(i)) == 7


def test_int_config_fits_fp32_exactly():
    d = S.int_mlp()
    X, W1, W2 = (d[k].astype(np.int64) for k in ("X", "W1", "W2"))
    for tp in (1, 2):
        _, Y = O.mlp_block(X, W1, W2, tp, "relu")
        assert np.abs(Y).max() < 2 ** 24


# ---------------------------------------------------------------------------
# 10. Planted mistakes: the pins above must catch them
# ---------------------------------------------------------------------------

def test_planted_dropped_shard_is_caught(monkeypatch, golden_worked_example):
    monkeypatch.setattr(O, "all_reduce", lambda parts: sum(parts[:-1]))
    with pytest.raises(AssertionError):
        test_worked_example_row_parallel(golden_worked_example)


def test_planted_wrong_column_block_is_caught(monkeypatch):
    def bad(W, tp):
        n = W.shape[1] // tp
        return [W[:, ((s + 1) % tp) * n:((s + 1) % tp + 1) * n] for s in range(tp)]
    monkeypatch.setattr(O, "column_shards", bad)
    with pytest.raises(AssertionError):
        test_column_parallel_concat_equals_bruteforce(0)


def test_planted_swapped_swiglu_is_caught(monkeypatch):
    monkeypatch.setattr(O, "swiglu", lambda g, u: O.silu(u) * g)
    with pytest.raises(AssertionError):
        test_mlp_swiglu_all_tp()


def test_planted_bias_per_shard_is_caught(monkeypatch):
    orig = O.all_reduce
    monkeypatch.setattr(O, "all_reduce", lambda parts: orig(parts) + 0)
    real_mlp = O.mlp_block

    def bad_mlp(X, W1, W2, tp, act="relu", W_up=None, b1=None, b1_up=None, b2=None, residual=None):
        Hs, Y = real_mlp(X, W1, W2, tp, act, W_up, b1, b1_up, None, residual)
        return Hs, Y + (tp * b2.reshape(1, -1) if b2 is not None else 0)
    monkeypatch.setattr(O, "mlp_block", bad_mlp)
    with pytest.raises(AssertionError):
        test_mlp_bias_once_and_residual()


def test_planted_transposed_operand_is_caught(monkeypatch):
    monkeypatch.setattr(O, "linear", lambda X, W: (W.T @ X.T).T if X.shape[1] == W.shape[0] else None)
    # (W^T X^T)^T is the same product: a correct rewrite must still pass
    test_column_parallel_concat_equals_bruteforce(1)
    monkeypatch.setattr(O, "linear", lambda X, W: X @ W[::-1])
    with pytest.raises(AssertionError):
        test_column_parallel_concat_equals_bruteforce(1)


# ---------------------------------------------------------------------------
# 11. Property tests over random shapes (Hypothesis), checked by brute force
# ---------------------------------------------------------------------------
from hypothesis import given, settings, strategies as st  # noqa: E402


@st.composite
def _shapes(draw):
    T = draw(st.integers(1, 3))
    K = draw(st.integers(1, 6))
    N = draw(st.integers(1, 6))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return T, K, N, seed


@settings(max_examples=60, deadline=None)
@given(_shapes())
def test_property_column_and_row_splits(shape):
    T, K, N, seed = shape
    rng = np.random.default_rng(seed)
    X, W = rand_ints(rng, (T, K), -3, 3), rand_ints(rng, (K, N), -3, 3)
    ref = brute_matmul(X.tolist(), W.tolist())
    for tp in divisors(N):
        assert O.all_gather(O.column_parallel(X, W, tp)).tolist() == ref
    for tp in divisors(K):
        assert O.all_reduce(O.row_parallel_partials(O.split_columns(X, tp), W, tp)).tolist() == ref
        if T % tp == 0:
            parts = O.row_parallel_partials(O.split_columns(X, tp), W, tp)
            assert np.concatenate(O.reduce_scatter(parts, tp), 0).tolist() == ref


@settings(max_examples=40, deadline=None)
@given(st.integers(1, 3), st.integers(1, 4), st.integers(1, 4), st.integers(0, 2 ** 31 - 1))
def test_property_mlp_relu_every_tp(T, H, I2, seed):
    I = 2 * I2
    rng = np.random.default_rng(seed)
    X, W1, W2 = rand_ints(rng, (T, H)), rand_ints(rng, (H, I)), rand_ints(rng, (I, H))
    b2 = rand_ints(rng, (H,))
    ref = np.array(brute_mlp(X.tolist(), W1.tolist(), W2.tolist(), lambda v: max(v, 0))) + b2
    for tp in divisors(I):
        assert O.mlp_block(X, W1, W2, tp, "relu", b2=b2)[1].tolist() == ref.tolist()


@settings(max_examples=30, deadline=None)
@given(st.sampled_from([(4, 2, 1), (4, 4, 2), (8, 2, 4), (8, 4, 8), (8, 1, 2), (4, 2, 4)]),
       st.integers(0, 2 ** 31 - 1))
def test_property_qkv_dedup_every_layout(heads, seed):
    hq, hkv, tp = heads
    rng = np.random.default_rng(seed)
    H, hd, T = 3, 2, 2
    Wq, Wk, Wv = rand_ints(rng, (H, hq * hd)), rand_ints(rng, (H, hkv * hd)), rand_ints(rng, (H, hkv * hd))
    X = rand_ints(rng, (T, H))
    ref = brute_matmul(X.tolist(), np.concatenate([Wq, Wk, Wv], 1).tolist())
    layout = O.qkv_head_layout(hq, hkv, tp)
    cols = {}
    for s, Ws in enumerate(O.qkv_shards(Wq, Wk, Wv, hq, hkv, hd, tp)):
        y = O.linear(X, Ws)
        q, kv = layout[s]
        for j, h in enumerate(q):
            cols[("q", h)] = y[:, j * hd:(j + 1) * hd].tolist()
        for j, h in enumerate(kv):
            o = (len(q) + j) * hd
            cols[("k", h)] = y[:, o:o + hd].tolist()
            o = (len(q) + len(kv) + j) * hd
            cols[("v", h)] = y[:, o:o + hd].tolist()
    full = [sum((cols[("q", h)][t] for h in range(hq)), []) + sum((cols[("k", h)][t] for h in range(hkv)), [])
            + sum((cols[("v", h)][t] for h in range(hkv)), []) for t in range(T)]
    assert full == ref


# ---------------------------------------------------------------------------
# Attention core (scaled dot-product attention of each local head)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("q_offset", [0, 5])
def test_attention_against_library_softmax_per_row(causal, q_offset):
    """Each query row on its own: scipy's softmax over the scaled scores of
    exactly the keys it sees (a slice, not a mask), then the weighted sum of
    their values, in pure Python."""
    from scipy.special import softmax
    rng = np.random.default_rng(211)
    T, Tq, hd = 11, 6, 16
    k, v = rng.standard_normal((T, hd)), rng.standard_normal((T, hd))
    q = rng.standard_normal((Tq, hd)) * 2.0
    got = O.attention_head(q, k, v, causal, q_offset=q_offset)
    for i in range(Tq):
        seen = range(q_offset + i + 1) if causal else range(T)
        w = softmax([float(np.dot(q[i], k[j])) / hd ** 0.5 for j in seen])
        want = [sum(w[n] * v[j][c] for n, j in enumerate(seen)) for c in range(hd)]
        np.testing.assert_allclose(got[i], want, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("q_offset", [0, 5])
def test_attention_weights_against_library_softmax_per_row(causal, q_offset):
    """The weights alone: each row is scipy's softmax over the scaled scores
    of exactly the keys that query sees (a slice), and 0 at every other key."""
    from scipy.special import softmax
    rng = np.random.default_rng(212)
    T, Tq, hd = 11, 6, 16
    k = rng.standard_normal((T, hd))
    q = rng.standard_normal((Tq, hd)) * 2.0
    w = O.attention_weights(q, k, causal, q_offset=q_offset)
    assert w.shape == (Tq, T)
    for i in range(Tq):
        n = q_offset + i + 1 if causal else T
        want = softmax([float(np.dot(q[i], k[j])) / hd ** 0.5 for j in range(n)])
        np.testing.assert_allclose(w[i, :n], want, rtol=1e-12, atol=1e-15)
        assert np.all(w[i, n:] == 0.0)


@pytest.mark.parametrize("causal", [True, False])
def test_attention_single_key_is_v(causal):
    """One token: the softmax over one score is 1, so the context is V exactly."""
    rng = np.random.default_rng(201)
    q, k, v = (rng.standard_normal((1, 8)) for _ in range(3))
    np.testing.assert_array_equal(O.attention_head(q, k, v, causal), v)


def test_attention_causal_first_query_sees_only_key_0():
    rng = np.random.default_rng(202)
    q, k, v = (rng.standard_normal((6, 4)) for _ in range(3))
    np.testing.assert_array_equal(O.attention_head(q, k, v, True)[0], v[0])


@pytest.mark.parametrize("causal", [True, False])
def test_attention_equal_keys_average_values(causal):
    """Equal keys give equal scores: uniform weights over the visible keys,
    so the context is the mean of V over keys 0..t (causal) or all keys."""
    rng = np.random.default_rng(203)
    T, hd = 7, 4
    q = rng.standard_normal((T, hd))
    k = np.tile(rng.standard_normal((1, hd)), (T, 1))
    v = rng.standard_normal((T, hd))
    want = (np.cumsum(v, 0) / np.arange(1, T + 1)[:, None]) if causal else np.tile(v.mean(0), (T, 1))
    np.testing.assert_allclose(O.attention_head(q, k, v, causal), want, rtol=0, atol=1e-13)


def test_attention_two_keys_closed_form():
    """hd = 2, q = (1, 0): scores are k[:,0] / sqrt(2). With k0 = 0 and
    k1[0] = sqrt(2) ln 3 the weights are 1/4 and 3/4 (checks the 1/sqrt(hd)
    scale and the softmax)."""
    q = np.array([[1.0, 0.0], [1.0, 0.0]])
    k = np.array([[0.0, 5.0], [math.sqrt(2.0) * math.log(3.0), -2.0]])
    v = np.array([[4.0, 8.0], [-4.0, 12.0]])
    out = O.attention_head(q, k, v, causal=False)
    np.testing.assert_allclose(out, np.tile(0.25 * v[0] + 0.75 * v[1], (2, 1)), rtol=0, atol=1e-12)
    out_c = O.attention_head(q, k, v, causal=True)    # row 0 sees key 0 only; row 1 as above
    np.testing.assert_allclose(out_c, np.stack([v[0], 0.25 * v[0] + 0.75 * v[1]]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_attention_key_shift_invariance(causal):
    """Adding one vector c to every key adds q.c/sqrt(hd) to all scores of a
    query, which the softmax cancels."""
    rng = np.random.default_rng(204)
    q, k, v = (rng.standard_normal((9, 6)) for _ in range(3))
    c = rng.standard_normal((1, 6))
    np.testing.assert_allclose(O.attention_head(q, k + c, v, causal), O.attention_head(q, k, v, causal),
                               rtol=0, atol=1e-12)


def test_attention_causal_ignores_future_tokens():
    rng = np.random.default_rng(205)
    q, k, v = (rng.standard_normal((8, 4)) for _ in range(3))
    k2, v2 = k.copy(), v.copy()
    k2[5:] += 3.0
    v2[5:] -= 7.0
    a, b = O.attention_head(q, k, v, True), O.attention_head(q, k2, v2, True)
    np.testing.assert_array_equal(a[:5], b[:5])
    assert not np.allclose(a[5:], b[5:])


def test_attention_full_is_key_permutation_invariant():
    rng = np.random.default_rng(206)
    q, k, v = (rng.standard_normal((8, 4)) for _ in range(3))
    perm = rng.permutation(8)
    np.testing.assert_allclose(O.attention_head(q, k[perm], v[perm], False), O.attention_head(q, k, v, False),
                               rtol=0, atol=1e-12)


def test_attention_gqa_head_map():
    """hq = 4, hkv = 2 on one shard: q heads 0, 1 read kv head 0 and 2, 3 read
    kv head 1. Zeroing kv head 1's V zeroes exactly heads 2 and 3; equal q
    vectors within a group give equal contexts."""
    rng = np.random.default_rng(207)
    T, hd, hq, hkv = 5, 4, 4, 2
    qkv = rng.standard_normal((T, (hq + 2 * hkv) * hd))
    qkv[:, hd:2 * hd] = qkv[:, 0:hd]                       # q head 1 = q head 0
    v1 = (hq + hkv + 1) * hd
    qkv[:, v1:v1 + hd] = 0.0                               # V of kv head 1
    (q, kv), = O.qkv_head_layout(hq, hkv, 1)
    ctx = O.context_attention(qkv, q, kv, hq, hkv, hd, causal=True)
    assert np.all(ctx[:, 2 * hd:] == 0.0) and not np.any(np.all(ctx[:, :2 * hd] == 0.0, axis=0))
    np.testing.assert_array_equal(ctx[:, 0:hd], ctx[:, hd:2 * hd])


def test_attention_sharded_equals_unsharded():
    """Per-shard attention (kv heads replicated where hkv < tp) gives the same
    context columns as running every head on one device."""
    rng = np.random.default_rng(208)
    T, H, hq, hkv, hd = 6, 8, 8, 2, 4
    X = rng.standard_normal((T, H))
    Wq, Wk, Wv = (rng.standard_normal((H, n * hd)) for n in (hq, hkv, hkv))
    (q1, kv1), = O.qkv_head_layout(hq, hkv, 1)
    full = O.context_attention(X @ np.concatenate([Wq, Wk, Wv], 1), q1, kv1, hq, hkv, hd)
    for tp in (2, 4, 8):
        layout = O.qkv_head_layout(hq, hkv, tp)
        parts = [O.context_attention(X @ Ws, layout[s][0], layout[s][1], hq, hkv, hd)
                 for s, Ws in enumerate(O.qkv_shards(Wq, Wk, Wv, hq, hkv, hd, tp))]
        np.testing.assert_allclose(np.concatenate(parts, 1), full, rtol=0, atol=1e-12)


def test_planted_missing_scale_is_caught(monkeypatch):
    """A planted mistake (no 1/sqrt(hd)) fails the closed-form pin."""
    def bad(q, k, v, causal=True):
        s = q @ k.T
        if causal:
            s = np.where(np.tril(np.ones(s.shape, dtype=bool)), s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        return (p / p.sum(1, keepdims=True)) @ v
    monkeypatch.setattr(O, "attention_head", bad)
    with pytest.raises(AssertionError):
        test_attention_two_keys_closed_form()


@pytest.mark.parametrize("causal", [True, False])
def test_attention_query_offset_selects_rows(causal):
    """Queries given from position a onwards reproduce rows a.. of the full call."""
    rng = np.random.default_rng(209)
    q, k, v = (rng.standard_normal((10, 4)) for _ in range(3))
    np.testing.assert_array_equal(O.attention_head(q[6:], k, v, causal, q_offset=6),
                                  O.attention_head(q, k, v, causal)[6:])
