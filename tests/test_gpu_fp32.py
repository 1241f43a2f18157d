"""GPU parity on the fp32 path: the worked example and the exact-integer MLP
are compared bit for bit with the oracle; real-valued fp32 within 1e-4*RMS."""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_F32, assert_close, assert_exact, dev, f64, i64

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")

F = torch.float32


def test_worked_example_column_row_gather_reduce():
    X, W = S.worked_example()
    Xd, Wd = dev(X, F), dev(W, F)
    Wc = tpl.tp_shard_weights(Wd, 2, "col")
    Y = tpl.tp_column_linear(Xd, Wc)                    # [2][1][2]
    ys = O.column_parallel(i64(X), i64(W), 2)
    assert_exact(Y, np.stack(ys), "col shards")         # [110,140] and [170,200]
    assert_exact(tpl.tp_shard_gather(Y), O.all_gather(ys), "all-gather")
    assert_exact(tpl.tp_column_linear(Xd, Wc, concat=True), O.linear(i64(X), i64(W)), "concat in place")

    Wr = tpl.tp_shard_weights(Wd, 2, "row")
    Xs = torch.stack([Xd[:, 0:1], Xd[:, 1:2]]).contiguous()  # [2][1][1]: 10 | 20
    P = tpl.tp_row_linear_partials(Xs, Wr)
    ps = O.row_parallel_partials(O.split_columns(i64(X), 2), i64(W), 2)
    assert_exact(P, np.stack(ps), "row partials")       # [10..40] and [100..160]
    assert_exact(tpl.tp_shard_reduce(P), O.all_reduce(ps), "all-reduce")
    assert_exact(tpl.tp_row_linear(Xs, Wr), O.all_reduce(ps), "fused row sum")


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_int_mlp_bit_exact(tp):
    d = S.int_mlp()
    X, W1, W2 = (dev(d[k], F) for k in ("X", "W1", "W2"))
    S1 = tpl.tp_shard_weights(W1, tp, "col")
    S2 = tpl.tp_shard_weights(W2, tp, "row")
    Hs_ref, Y_ref = O.mlp_block(i64(d["X"]), i64(d["W1"]), i64(d["W2"]), tp, "relu")
    Y = tpl.tp_mlp_block(X, S1, S2, act="relu")
    assert_exact(Y, Y_ref, f"mlp tp={tp}")
    Hs = tpl.tp_column_linear(X, S1, act="relu")
    assert_exact(Hs, np.stack(Hs_ref), "relu shards")
    P = tpl.tp_row_linear_partials(Hs, S2)
    assert_exact(P, np.stack(O.row_parallel_partials(Hs_ref, i64(d["W2"]), tp)), "partials")
    assert_exact(tpl.tp_shard_reduce(P), Y_ref, "reduce")
    if 16 % tp == 0:
        rs = tpl.tp_shard_reduce(P, op="scatter")
        ref = O.reduce_scatter(O.row_parallel_partials(Hs_ref, i64(d["W2"]), tp), tp)
        assert_exact(rs, np.stack(ref), "reduce-scatter")


def test_int_bias_residual_swiglu_shapes_exact():
    rng = np.random.default_rng(5)
    T, H, I, tp = 37, 24, 96, 4
    X, W1, W2 = (rng.integers(-3, 4, s).astype(np.float32) for s in [(T, H), (H, I), (I, H)])
    b1 = rng.integers(-5, 6, I).astype(np.float32)
    b2 = rng.integers(-5, 6, H).astype(np.float32)
    R = rng.integers(-9, 10, (T, H)).astype(np.float32)
    S1 = tpl.tp_shard_weights(dev(W1, F), tp, "col")
    S2 = tpl.tp_shard_weights(dev(W2, F), tp, "row")
    _, ref = O.mlp_block(i64(X), i64(W1), i64(W2), tp, "relu", b1=i64(b1), b2=i64(b2), residual=i64(R))
    Y = tpl.tp_mlp_block(dev(X, F), S1, S2, b1=dev(b1, F), b2=dev(b2, F), residual=dev(R, F), act="relu")
    assert_exact(Y, ref, "bias once + residual")
    P = tpl.tp_row_linear_partials(tpl.tp_column_linear(dev(X, F), S1, bias=dev(b1, F), act="relu"), S2)
    assert_exact(tpl.tp_shard_reduce(P, bias=dev(b2, F), residual=dev(R, F)), ref, "reduce + bias + residual")


@pytest.mark.parametrize("act", ["none", "gelu", "silu", "swiglu"])
def test_fp32_real_valued(act):
    rng = np.random.default_rng(11)
    T, H, I, tp = 70, 48, 160, 4
    X = rng.standard_normal((T, H)).astype(np.float32)
    W1, Wu = (rng.standard_normal((H, I)).astype(np.float32) * 0.2 for _ in range(2))
    W2 = rng.standard_normal((I, H)).astype(np.float32) * 0.2
    S1 = tpl.tp_shard_weights(dev(W1, F), tp, "col")
    Su = tpl.tp_shard_weights(dev(Wu, F), tp, "col") if act == "swiglu" else None
    S2 = tpl.tp_shard_weights(dev(W2, F), tp, "row")
    _, ref = O.mlp_block(f64(X), f64(W1), f64(W2), tp, act, W_up=f64(Wu) if Su else None)
    Y = tpl.tp_mlp_block(dev(X, F), S1, S2, W_up=Su, act=act)
    assert_close(Y, ref, TOL_F32, f"fp32 mlp {act}")


def test_fp32_attention_projection_int_exact():
    rng = np.random.default_rng(12)
    T, H, hq, hkv, hd = 19, 32, 8, 2, 8
    for tp in (1, 2, 4, 8):
        Wq, Wk, Wv = (rng.integers(-2, 3, s).astype(np.float32) for s in [(H, hq * hd), (H, hkv * hd), (H, hkv * hd)])
        Wo = rng.integers(-2, 3, (hq * hd, H)).astype(np.float32)
        X, R = (rng.integers(-2, 3, (T, H)).astype(np.float32) for _ in range(2))
        Sqkv = tpl.tp_shard_qkv(dev(Wq, F), dev(Wk, F), dev(Wv, F), hq, hkv, hd, tp)
        Sout = tpl.tp_shard_weights(dev(Wo, F), tp, "row")
        qkv_ref, _, Y_ref = O.attn_proj(i64(X), i64(Wq), i64(Wk), i64(Wv), i64(Wo), hq, hkv, hd, tp, residual=i64(R))
        qkv = torch.empty((tp, T, qkv_ref[0].shape[1]), dtype=F, device="cuda")
        Y = tpl.tp_attn_proj(dev(X, F), Sqkv, Sout, residual=dev(R, F), qkv_out=qkv)
        assert_exact(qkv, np.stack(qkv_ref), f"qkv tp={tp}")
        assert_exact(Y, Y_ref, f"attn tp={tp}")


def test_empty_and_single_token():
    rng = np.random.default_rng(13)
    W = rng.integers(-3, 4, (16, 32)).astype(np.float32)
    Sc = tpl.tp_shard_weights(dev(W, F), 4, "col")
    X0 = torch.empty((0, 16), dtype=F, device="cuda")
    assert tpl.tp_column_linear(X0, Sc).shape == (4, 0, 8)
    X1 = rng.integers(-3, 4, (1, 16)).astype(np.float32)
    assert_exact(tpl.tp_column_linear(dev(X1, F), Sc, concat=True), O.linear(i64(X1), i64(W)), "T=1")
    # tp equal to N: one output column per shard
    St = tpl.tp_shard_weights(dev(W, F), 32, "col")
    assert_exact(tpl.tp_column_linear(dev(X1, F), St, concat=True), O.linear(i64(X1), i64(W)), "tp=N")
    assert tpl.tp_get_error() == 0
