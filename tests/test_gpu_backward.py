"""Backward of the column/row pair on the GPU against the oracle.

The GPU runs forward then backward on bf16 data: the saved forward values
(G, U, Hs) are the GPU forward's own bf16 outputs, while the oracle
recomputes everything in float64 from the same inputs (X, weights, dY). Every
GPU intermediate (dHs, dG, dU, the saved G, U, Hs) is rounded to bf16, so all
outputs are held to the bf16 bound, 2e-2 * RMS of the oracle's result.
Weight gradients come out in the shards' storage layout (the transpose of
each shard's [in, out] block). With a single token a weight gradient is an
outer product of two rows: each element is one product, exact in fp32, and
the values are heavy-tailed (a product of two normals), so there the bound
is the one for bf16-stored elementwise values (plus 2^-8 of each element).
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_BF16, TOL_F32, assert_close, assert_close_stored, assert_exact, dev, f64, host, i64


def close_wgrad(gpu, ref, T, what):
    (assert_close_stored if T == 1 else assert_close)(gpu, ref, TOL_BF16, what)

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")
B = torch.bfloat16


@pytest.mark.parametrize("tp,T,K,N", [(1, 128, 256, 256), (2, 200, 688, 520), (4, 300, 704, 1024),
                                      (8, 64, 512, 384), (2, 1, 256, 512)])
def test_row_linear_backward(tp, T, K, N):
    """Ragged tails everywhere: T % 128, K/tp % 64 (344, 176), N % 256."""
    W, X, dY = S.normal(401, (K, N), 0.05), S.normal(402, (T, K)), S.normal(403, (T, N))
    Sw = tpl.tp_shard_weights(dev(W), tp, "row")
    Xs = torch.stack([t.contiguous() for t in dev(X).split(K // tp, dim=1)])
    dXs, dW = tpl.tp_row_linear_backward(Xs, Sw, dev(dY))
    assert tpl.tp_get_error() == 0
    ref_dX, ref_dW = O.row_linear_backward(O.split_columns(f64(X), tp), f64(W), tp, f64(dY))
    assert_close(dXs, np.stack(ref_dX), TOL_BF16, "dXs")
    close_wgrad(dW, np.stack([w.T for w in ref_dW]), T, "dW (storage layout)")


@pytest.mark.parametrize("tp,T,K,N", [(1, 128, 256, 256), (2, 200, 520, 688), (4, 300, 1024, 704),
                                      (8, 64, 384, 512), (2, 1, 512, 256)])
@pytest.mark.parametrize("with_dr", [False, True])
def test_column_linear_backward(tp, T, K, N, with_dr):
    W, X = S.normal(411, (K, N), 0.05), S.normal(412, (T, K))
    dYs = S.normal(413, (tp, T, N // tp))
    dR = S.normal(414, (T, K)) if with_dr else None
    Sw = tpl.tp_shard_weights(dev(W), tp, "col")
    ws = torch.empty(tpl.tp_gemm_workspace_bytes(T, Sw), dtype=torch.uint8, device="cuda")
    dX, dW = tpl.tp_column_linear_backward(dev(X), Sw, dev(dYs), dR=None if dR is None else dev(dR),
                                           workspace=ws)
    assert tpl.tp_get_error() == 0
    ref_dX, ref_dW = O.column_linear_backward(f64(X), f64(W), tp, [f64(dYs[s]) for s in range(tp)],
                                              None if dR is None else f64(dR))
    assert_close(dX, ref_dX, TOL_BF16, "dX")
    close_wgrad(dW, np.stack([w.T for w in ref_dW]), T, "dW (storage layout)")


def gpu_forward(d, tp, act):
    """Shards and the forward's saved values (G, U, Hs) from the GPU path."""
    X = dev(d["X"])
    Sg = tpl.tp_shard_weights(dev(d["Wg"]), tp, "col")
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    Su = tpl.tp_shard_weights(dev(d["Wu"]), tp, "col") if act == "swiglu" else None
    G = tpl.tp_column_linear(X, Sg, act="none")
    U = tpl.tp_column_linear(X, Su, act="none") if act == "swiglu" else None
    Hs = tpl.tp_column_linear(X, Sg, W_up=Su, act=act)
    return X, Sg, Su, Sd, G, U, Hs


def saved_values(seed, tp, T, Is, act):
    """Seeded saved forward values [tp][T][I/tp] (bf16-representable)."""
    G = S.normal(seed, (tp, T, Is))
    U = S.normal(seed + 1, (tp, T, Is)) if act == "swiglu" else None
    Hs = S.normal(seed + 2, (tp, T, Is), 0.5)
    return G, U, Hs


@pytest.mark.parametrize("act", ["none", "relu", "gelu", "silu", "swiglu"])
@pytest.mark.parametrize("tp,T,H,I", [(4, 260, 384, 704), (2, 128, 256, 512)])
def test_mlp_backward(act, tp, T, H, I):
    """The backward given saved forward values: both sides take the same
    seeded G, U and Hs, so the bf16 bound holds for every output."""
    d = S.mlp_backward(T, H, I, seeds=(421, 422, 423, 424, 425), std=0.05)
    G, U, Hs = saved_values(441, tp, T, I // tp, act)
    dR = S.normal(426, (T, H))
    Sg = tpl.tp_shard_weights(dev(d["Wg"]), tp, "col")
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    Su = tpl.tp_shard_weights(dev(d["Wu"]), tp, "col") if act == "swiglu" else None
    g = tpl.tp_mlp_backward(dev(d["X"]), Sg, Sd, dev(G), dev(Hs), dev(d["dY"]), W_up=Su,
                            U=None if U is None else dev(U), dR=dev(dR), act=act)
    assert tpl.tp_get_error() == 0
    ref = O.mlp_backward_saved(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, f64(d["dY"]), list(f64(G)),
                               list(f64(Hs)), act, W_up=f64(d["Wu"]) if act == "swiglu" else None,
                               U=None if U is None else list(f64(U)), dR=f64(dR))
    # The gate / up weight gradients sum T products of two or three random
    # factors (X, dH and the activation's derivative): heavy-tailed, with the
    # largest elements 5-10x the RMS, where the bf16 storage of one element
    # alone (2^-9 of it) can reach 2e-2 * RMS. Their bound adds each
    # element's storage rounding; dX and dW2 keep the plain bound.
    assert_close(g["dX"], ref["dX"], TOL_BF16, "dX")
    assert_close_stored(g["dW1"], np.stack([w.T for w in ref["dW1"]]), TOL_BF16, "dW1")
    assert_close(g["dW2"], np.stack([w.T for w in ref["dW2"]]), TOL_BF16, "dW2")
    if act == "swiglu":
        assert_close_stored(g["dW_up"], np.stack([w.T for w in ref["dW_up"]]), TOL_BF16, "dW_up")


# Forward then backward on the GPU against the oracle's float64 chain. The
# GPU's saved values G, U (and Hs) are bf16, which the oracle never rounds:
# each carries a uniform relative error of up to 2^-9 (std 0.11%), and the
# SwiGLU / GELU derivatives pass G's error on amplified by |g f''(g) / f'(g)|
# (up to about 2), so with dG's own rounding an element of dG carries a
# relative error of std about 0.26%. A weight-gradient element sums hundreds
# of such terms with random signs, so its error relative to the RMS has about
# that std; the largest of ~3e5 elements sits near 4.6 std (1.2%), and the
# output's own bf16 rounding adds up to 2^-9 times the largest |value| (about
# 4.5 RMS): a max error near 2-3% of the RMS. The bound is 4e-2 * RMS.
TOL_CHAIN = 4e-2


@pytest.mark.parametrize("act", ["none", "relu", "gelu", "silu", "swiglu"])
def test_mlp_forward_then_backward(act):
    """For ReLU the derivative [G > 0] is a decision taken from floating
    point: X and the gate weights are small integers there, so that G is an
    exact integer on both sides and the decision is the same."""
    tp, T, H, I = 4, 260, 384, 704
    d = S.mlp_backward(T, H, I, seeds=(421, 422, 423, 424, 425), std=0.05)
    if act == "relu":
        d["X"] = S.uniform_ints(427, (T, H), -2, 2)
        d["Wg"] = S.uniform_ints(428, (H, I), -2, 2)
    X, Sg, Su, Sd, G, U, Hs = gpu_forward(d, tp, act)
    dR = S.normal(426, (T, H))
    g = tpl.tp_mlp_backward(X, Sg, Sd, G, Hs, dev(d["dY"]), W_up=Su, U=U, dR=dev(dR), act=act)
    assert tpl.tp_get_error() == 0
    ref = O.mlp_backward(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, f64(d["dY"]), act,
                         W_up=f64(d["Wu"]) if act == "swiglu" else None, dR=f64(dR))
    assert_close(g["dX"], ref["dX"], TOL_CHAIN, "dX")
    assert_close(g["dW1"], np.stack([w.T for w in ref["dW1"]]), TOL_CHAIN, "dW1")
    assert_close(g["dW2"], np.stack([w.T for w in ref["dW2"]]), TOL_CHAIN, "dW2")
    if act == "swiglu":
        assert_close(g["dW_up"], np.stack([w.T for w in ref["dW_up"]]), TOL_CHAIN, "dW_up")


def test_mlp_backward_partial_outputs_and_single_token():
    """Skipped outputs stay untouched; T = 1 (one token, K = T ragged to 64)."""
    T, H, I, tp = 1, 256, 512, 2
    d = S.mlp_backward(T, H, I, seeds=(431, 432, 433, 434, 435), std=0.05)
    X, Sg, Su, Sd, G, U, Hs = gpu_forward(d, tp, "swiglu")
    g = tpl.tp_mlp_backward(X, Sg, Sd, G, Hs, dev(d["dY"]), W_up=Su, U=U, act="swiglu", want=("dX", "dW2"))
    assert tpl.tp_get_error() == 0
    assert g["dW1"] is None and g["dW_up"] is None
    ref = O.mlp_backward(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, f64(d["dY"]), "swiglu", W_up=f64(d["Wu"]))
    assert_close(g["dX"], ref["dX"], TOL_CHAIN, "dX")
    assert_close_stored(g["dW2"], np.stack([w.T for w in ref["dW2"]]), TOL_CHAIN, "dW2")


def test_backward_validation():
    Sb = tpl.tp_shard_weights(torch.zeros((256, 512), dtype=B, device="cuda"), 2, "col")
    with pytest.raises(tpl.TpError):  # a column view where a row view is needed
        tpl.tp_row_linear_backward(torch.zeros((2, 8, 128), dtype=B, device="cuda"), Sb,
                                   torch.zeros((8, 512), dtype=B, device="cuda"))


# --- fp32 views: the FFMA GEMM. Integer-valued inputs are exact, so the
# dataflow of the backward (which shards are summed, which dY each shard
# receives, the orientation of every weight gradient) is checked bit for bit
# against the oracle's int64 arithmetic.
F = torch.float32


@pytest.mark.parametrize("tp,T,H,I", [(2, 16, 64, 256), (4, 37, 96, 160), (1, 5, 32, 48)])
def test_int_relu_mlp_backward_bit_exact(tp, T, H, I):
    """Saved values from the GPU's fp32 forward (exact on integers), then
    the backward; the oracle recomputes everything in int64. Largest partial
    sums: |dX| <= I * 3 * (H * 3 * 3) = 442368 < 2^24 at the integer MLP's
    sizes (T = 16, H = 64, I = 256), less elsewhere."""
    X = S.uniform_ints(451, (T, H))
    W1, W2 = S.uniform_ints(452, (H, I)), S.uniform_ints(453, (I, H))
    dY, dR = S.uniform_ints(454, (T, H)), S.uniform_ints(455, (T, H))
    Xd = dev(X, F)
    S1 = tpl.tp_shard_weights(dev(W1, F), tp, "col")
    S2 = tpl.tp_shard_weights(dev(W2, F), tp, "row")
    G = tpl.tp_column_linear(Xd, S1, act="none")
    Hs = tpl.tp_column_linear(Xd, S1, act="relu")
    g = tpl.tp_mlp_backward(Xd, S1, S2, G, Hs, dev(dY, F), dR=dev(dR, F), act="relu")
    assert tpl.tp_get_error() == 0
    ref = O.mlp_backward(i64(X), i64(W1), i64(W2), tp, i64(dY), "relu", dR=i64(dR))
    assert_exact(g["dX"], ref["dX"], "dX")
    assert_exact(g["dW1"], np.stack([w.T for w in ref["dW1"]]), "dW1 (storage layout)")
    assert_exact(g["dW2"], np.stack([w.T for w in ref["dW2"]]), "dW2 (storage layout)")


@pytest.mark.parametrize("tp,T,K,N", [(2, 16, 64, 256), (4, 37, 96, 160)])
def test_int_single_linears_backward_bit_exact(tp, T, K, N):
    """The two layers alone on integers: the row layer hands every shard the
    same dY; the column layer sums its shards' input gradients (plus dR)."""
    W, X, dY = S.uniform_ints(461, (K, N)), S.uniform_ints(462, (T, K)), S.uniform_ints(463, (T, N))
    dR = S.uniform_ints(464, (T, K))
    Sr = tpl.tp_shard_weights(dev(W, F), tp, "row")
    Xs = torch.stack([t.contiguous() for t in dev(X, F).split(K // tp, dim=1)])
    dXs, dW = tpl.tp_row_linear_backward(Xs, Sr, dev(dY, F))
    assert tpl.tp_get_error() == 0
    ref_dX, ref_dW = O.row_linear_backward(O.split_columns(i64(X), tp), i64(W), tp, i64(dY))
    assert_exact(dXs, np.stack(ref_dX), "row dXs")
    assert_exact(dW, np.stack([w.T for w in ref_dW]), "row dW")
    Sc = tpl.tp_shard_weights(dev(W, F), tp, "col")
    dYs = S.uniform_ints(465, (tp, T, N // tp))
    dX, dWc = tpl.tp_column_linear_backward(dev(X, F), Sc, dev(dYs, F), dR=dev(dR, F))
    assert tpl.tp_get_error() == 0
    ref_dX, ref_dW = O.column_linear_backward(i64(X), i64(W), tp, [i64(dYs[s]) for s in range(tp)], i64(dR))
    assert_exact(dX, ref_dX, "column dX")
    assert_exact(dWc, np.stack([w.T for w in ref_dW]), "column dW")


@pytest.mark.parametrize("act", ["none", "relu", "gelu", "silu", "swiglu"])
def test_fp32_mlp_backward(act):
    """Real values on the fp32 path, every activation, saved values given to
    both sides: held to the fp32 bound, 1e-4 * RMS."""
    tp, T, H, I = 4, 70, 96, 160
    d = S.mlp_backward(T, H, I, seeds=(471, 472, 473, 474, 475), std=0.05)
    G, U, Hs = saved_values(476, tp, T, I // tp, act)
    dR = S.normal(479, (T, H))
    Sg = tpl.tp_shard_weights(dev(d["Wg"], F), tp, "col")
    Sd = tpl.tp_shard_weights(dev(d["Wd"], F), tp, "row")
    Su = tpl.tp_shard_weights(dev(d["Wu"], F), tp, "col") if act == "swiglu" else None
    g = tpl.tp_mlp_backward(dev(d["X"], F), Sg, Sd, dev(G, F), dev(Hs, F), dev(d["dY"], F), W_up=Su,
                            U=None if U is None else dev(U, F), dR=dev(dR, F), act=act)
    assert tpl.tp_get_error() == 0
    ref = O.mlp_backward_saved(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, f64(d["dY"]), list(f64(G)),
                               list(f64(Hs)), act, W_up=f64(d["Wu"]) if act == "swiglu" else None,
                               U=None if U is None else list(f64(U)), dR=f64(dR))
    assert_close(g["dX"], ref["dX"], TOL_F32, "dX")
    assert_close(g["dW1"], np.stack([w.T for w in ref["dW1"]]), TOL_F32, "dW1")
    assert_close(g["dW2"], np.stack([w.T for w in ref["dW2"]]), TOL_F32, "dW2")
    if act == "swiglu":
        assert_close(g["dW_up"], np.stack([w.T for w in ref["dW_up"]]), TOL_F32, "dW_up")


def test_mlp_backward_full_size_sampled():
    """The 7B SwiGLU MLP at tp = 8, T = 2048 (the bench workload), forward
    then backward on the GPU, against the oracle's float64 chain (the chain
    bound) on a sample. Token rows are independent, so dX of sampled rows is
    the oracle's backward of those rows alone (all eight shards). Columns of
    the intermediate are independent too: the gradients of sampled gate / up
    weight rows (columns of W1 and Wu) and down weight columns (rows of W2)
    are the oracle's backward of the block restricted to those intermediate
    columns, over all tokens, unsharded."""
    T, H, I, tp = 2048, 4096, 11008, 8
    d = S.mlp_backward(T, H, I)
    X, Sg, Su, Sd, G, U, Hs = gpu_forward(d, tp, "swiglu")
    g = tpl.tp_mlp_backward(X, Sg, Sd, G, Hs, dev(d["dY"]), W_up=Su, U=U, act="swiglu")
    assert tpl.tp_get_error() == 0
    Xf, Wg, Wu, Wd, dY = (f64(d[k]) for k in ("X", "Wg", "Wu", "Wd", "dY"))
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(T, 24, replace=False))
    ref_rows = O.mlp_backward(Xf[rows], Wg, Wd, tp, dY[rows], "swiglu", W_up=Wu)
    assert_close(host(g["dX"])[rows], ref_rows["dX"], TOL_CHAIN, "dX rows")
    cols = np.sort(rng.choice(I, 12, replace=False))
    ref_cols = O.mlp_backward(Xf, Wg[:, cols], Wd[cols], 1, dY, "swiglu", W_up=Wu[:, cols])
    Is = I // tp
    dW1 = host(g["dW1"]).reshape(I, H)[cols]  # storage [tp][I/tp][H] = [I][H] rows
    dWu = host(g["dW_up"]).reshape(I, H)[cols]
    assert_close(dW1, ref_cols["dW1"][0].T, TOL_CHAIN, "dW1 rows")
    assert_close(dWu, ref_cols["dW_up"][0].T, TOL_CHAIN, "dW_up rows")
    dW2 = host(g["dW2"])  # [tp][H][I/tp]
    got = np.stack([dW2[c // Is, :, c % Is] for c in cols])  # [len(cols)][H]
    assert_close(got, ref_cols["dW2"][0], TOL_CHAIN, "dW2 columns")
