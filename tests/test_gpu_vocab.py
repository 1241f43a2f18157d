"""Vocabulary-parallel embedding and cross-entropy on the GPU against the
oracle.

The embedding copies table rows: bit-exact. The cross-entropy reads the
given logits (bf16 or fp32 values, exact reals to the oracle) and computes
in fp32, so the per-token and mean losses are held to the fp32 bound,
1e-4 * RMS. The gradient softmax(z) - onehot(label) (scaled by 1/T) has one
large entry per token and ~V tiny ones: stored in bf16 it is held to the
bound for bf16-stored values (2e-2 * RMS plus each element's rounding);
stored in fp32 to 1e-4 * RMS plus 1e-6 of each element. The end-to-end
chain (embedding -> column-parallel LM head -> loss) rounds the logits to
bf16 in the GEMM, which moves a loss by about 2^-9 of the logits' scale:
held to 2e-2 * RMS.
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_BF16, TOL_F32, assert_close, assert_close_stored, dev, f64, host

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")
TP_ERR_INDEX = 10


def ids_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to("cuda")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,H,tp,T", [(1024, 256, 4, 300), (1000, 100, 8, 37), (32000, 4096, 4, 64),
                                      (640, 264, 1, 5)])
def test_embedding_bit_exact(dtype, V, H, tp, T):
    E = S.normal(501, (V, H))
    v = V // tp
    ids = S.token_ids(502, T, V)
    ids[: min(T, 2 * tp)] = np.array([s * v + d for s in range(tp) for d in (0, v - 1)])[: min(T, 2 * tp)]
    Y = tpl.tp_vocab_embedding(ids_dev(ids), dev(E, dtype), tp)
    assert tpl.tp_get_error() == 0
    np.testing.assert_array_equal(host(Y), O.vocab_embedding(ids, f64(host(dev(E, dtype))), tp))


def test_embedding_id_out_of_range_reports_index_error():
    E = dev(S.normal(503, (64, 32)))
    Y = tpl.tp_vocab_embedding(ids_dev([3, 64, -1, 5]), E, 4)
    assert tpl.tp_get_error() == TP_ERR_INDEX
    y = host(Y)
    assert (y[1] == 0).all() and (y[2] == 0).all()
    np.testing.assert_array_equal(y[[0, 3]], host(E)[[3, 5]])
    assert tpl.tp_get_error() == 0  # the error word was cleared


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("tp,T,V", [(4, 300, 32000), (8, 37, 1000), (1, 1, 4096), (2, 129, 520), (2, 33, 4100)])
@pytest.mark.parametrize("in_place", [False, True])
def test_cross_entropy(dtype, tp, T, V, in_place):
    z = S.normal(511, (tp, T, V // tp), 2.0)
    y = S.token_ids(512, T, V)
    zd = dev(z, dtype)
    zf = f64(host(zd))  # the values the kernel reads
    d = zd if in_place else torch.empty_like(zd)
    loss, mean = tpl.tp_vocab_cross_entropy(zd, ids_dev(y), dlogits=d)
    assert tpl.tp_get_error() == 0
    ref = O.vocab_parallel_cross_entropy(list(zf), y)
    assert_close(loss, ref, TOL_F32, "loss")
    assert abs(float(host(mean)[0]) - ref.mean()) <= TOL_F32 * np.sqrt(np.mean(ref ** 2)), "mean loss"
    gref = O.cross_entropy_grad(O.all_gather(list(zf)), y, 1.0 / T)
    got = host(d).transpose(1, 0, 2).reshape(T, V)  # [tp][T][v] -> [T][V]
    if dtype == torch.bfloat16:
        assert_close_stored(got, gref, TOL_BF16, "dlogits")
    else:
        err = np.abs(got - gref) - (TOL_F32 * np.sqrt(np.mean(gref ** 2)) + 1e-6 * np.abs(gref))
        assert (err <= 0).all(), f"dlogits fp32: worst excess {err.max():.3g}"


def test_cross_entropy_bad_label_reports_index_error():
    z = dev(S.normal(513, (2, 4, 16)))
    loss, _ = tpl.tp_vocab_cross_entropy(z, ids_dev([1, 40, 3, -2]))
    assert tpl.tp_get_error() == TP_ERR_INDEX
    l = host(loss)
    assert np.isnan(l[1]) and np.isnan(l[3]) and np.isfinite(l[[0, 2]]).all()


def lm_chain(d, tp):
    E, W = dev(d["E"]), dev(d["W_lm"])
    Slm = tpl.tp_shard_weights(W, tp, "col")
    X0 = tpl.tp_vocab_embedding(ids_dev(d["ids"]), E, tp)
    logits = tpl.tp_column_linear(X0, Slm)  # [tp][T][V/tp]
    loss, mean = tpl.tp_vocab_cross_entropy(logits, ids_dev(d["labels"]), dlogits=logits)
    return loss, mean, logits


@pytest.mark.parametrize("tp,T,H,V", [(4, 260, 256, 4096), (2, 128, 512, 2048)])
def test_embedding_lm_head_cross_entropy_chain(tp, T, H, V):
    d = S.vocab_lm(T, H, V)
    loss, mean, _ = lm_chain(d, tp)
    assert tpl.tp_get_error() == 0
    X0 = O.vocab_embedding(d["ids"], f64(d["E"]), tp)
    ref = O.vocab_parallel_cross_entropy(O.column_parallel(X0, f64(d["W_lm"]), tp), d["labels"])
    assert_close(loss, ref, TOL_BF16, "loss")
    assert abs(float(host(mean)[0]) - ref.mean()) <= TOL_BF16 * np.sqrt(np.mean(ref ** 2))


@pytest.mark.parametrize("tp,T,H,V,dtype", [
    (4, 260, 256, 4096, torch.bfloat16),      # statistics from the GEMM epilogue, 4 tiles per shard
    (2, 300, 512, 2000, torch.bfloat16),      # 1000 columns a shard: the last tile holds 232
    (1, 129, 256, 520, torch.bfloat16),       # one shard, a last tile of 8 columns, a ragged token block
    (8, 37, 128, 4096, torch.bfloat16),       # 37 tokens: weight-streaming GEMM, then a pass over the logits
    (2, 100, 128, 1024, torch.float32),       # fp32 views: FFMA GEMM, then a pass over the logits
])
def test_lm_head_cross_entropy_fused(tp, T, H, V, dtype):
    """The LM head and the loss in one call against the oracle's chain. On
    the fused bf16 path the statistics come from the fp32 accumulator, so
    the losses are those of unrounded logits: held to the fp32 bound. Where
    a pass reads stored bf16 logits (37 tokens) the chain bound applies."""
    d = S.vocab_lm(T, H, V)
    E, W = dev(d["E"], dtype), dev(d["W_lm"], dtype)
    Slm = tpl.tp_shard_weights(W, tp, "col")
    X0 = tpl.tp_vocab_embedding(ids_dev(d["ids"]), E, tp)
    dz = torch.empty((tp, T, V // tp), dtype=dtype, device="cuda")
    logits, loss, mean = tpl.tp_lm_head_cross_entropy(X0, Slm, ids_dev(d["labels"]), dlogits=dz)
    assert tpl.tp_get_error() == 0
    Xr = O.vocab_embedding(d["ids"], f64(host(E)), tp)
    z = O.column_parallel(Xr, f64(host(W)), tp)
    ref = O.vocab_parallel_cross_entropy(z, d["labels"])
    fused = dtype == torch.bfloat16 and T > 64
    tol = TOL_F32 if (fused or dtype == torch.float32) else TOL_BF16
    assert_close(logits, np.stack(z), TOL_BF16 if dtype == torch.bfloat16 else TOL_F32, "logits")
    assert_close(loss, ref, tol, "losses")
    assert abs(float(host(mean)[0]) - ref.mean()) <= tol * np.sqrt(np.mean(ref ** 2)), "mean loss"
    gref = O.cross_entropy_grad(O.all_gather(z), d["labels"], 1.0 / T)
    got = host(dz).transpose(1, 0, 2).reshape(T, V)
    if dtype == torch.bfloat16:
        assert_close_stored(got, gref, TOL_BF16, "dlogits")
    else:
        err = np.abs(got - gref) - (TOL_F32 * np.sqrt(np.mean(gref ** 2)) + 1e-6 * np.abs(gref))
        assert (err <= 0).all(), f"dlogits fp32: worst excess {err.max():.3g}"


def test_lm_head_cross_entropy_fused_bad_label():
    T, H, V, tp = 130, 128, 1024, 2
    d = S.vocab_lm(T, H, V)
    d["labels"][[3, 77]] = [V, -5]
    Slm = tpl.tp_shard_weights(dev(d["W_lm"]), tp, "col")
    X0 = tpl.tp_vocab_embedding(ids_dev(d["ids"]), dev(d["E"]), tp)
    _, loss, _ = tpl.tp_lm_head_cross_entropy(X0, Slm, ids_dev(d["labels"]))
    assert tpl.tp_get_error() == TP_ERR_INDEX
    l = host(loss)
    assert np.isnan(l[[3, 77]]).all() and np.isfinite(np.delete(l, [3, 77])).all()


def test_lm_head_cross_entropy_full_size():
    """The bench workload (T = 4096, H = 4096, V = 32000, tp = 4): every
    token's loss and the mean loss against the oracle's chain (vocabulary
    embedding, column-parallel LM head, vocabulary-parallel cross-entropy),
    which runs over blocks of token rows (rows are independent). Both ways:
    the LM head then a loss over its stored bf16 logits (the chain bound),
    and the fused call, whose statistics come from the fp32 accumulator (the
    fp32 bound)."""
    T, H, V, tp = 4096, 4096, 32000, 4
    d = S.vocab_lm(T, H, V)
    loss, mean, _ = lm_chain(d, tp)
    assert tpl.tp_get_error() == 0
    Slm = tpl.tp_shard_weights(dev(d["W_lm"]), tp, "col")
    X0 = tpl.tp_vocab_embedding(ids_dev(d["ids"]), dev(d["E"]), tp)
    _, loss_f, mean_f = tpl.tp_lm_head_cross_entropy(X0, Slm, ids_dev(d["labels"]))
    assert tpl.tp_get_error() == 0
    X0r = O.vocab_embedding(d["ids"], f64(d["E"]), tp)
    W = f64(d["W_lm"])
    ref = np.concatenate([O.vocab_parallel_cross_entropy(O.column_parallel(X0r[r:r + 512], W, tp),
                                                         d["labels"][r:r + 512]) for r in range(0, T, 512)])
    rms = np.sqrt(np.mean(ref ** 2))
    assert_close(loss, ref, TOL_BF16, "losses")
    assert abs(float(host(mean)[0]) - ref.mean()) <= TOL_BF16 * rms, "mean loss"
    assert_close(loss_f, ref, TOL_F32, "losses (fused)")
    assert abs(float(host(mean_f)[0]) - ref.mean()) <= TOL_F32 * rms, "mean loss (fused)"
