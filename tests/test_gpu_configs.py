"""GPU parity at the full sizes of the benchmarked workloads, through the same
calls bench.py times. Every workload here is independent across token rows
(the attention core is the single-key stand-in), so the oracle computes a
seeded sample of rows and the GPU's rows are compared with it one by one.
Tolerance: max|gpu - oracle| <= 2e-2 * RMS(oracle) (bf16)."""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_BF16, assert_close, dev, f64, host, sample_rows

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")

B = torch.bfloat16


@pytest.fixture(scope="module")
def mlp7b():
    d = S.swiglu_mlp(2048, 4096, 11008)
    g = {k: dev(v) for k, v in d.items()}
    return d, g


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_llama7b_swiglu_mlp_full(mlp7b, tp):
    d, g = mlp7b
    T = 2048
    Sg, Su = tpl.tp_shard_weights(g["Wg"], tp, "col"), tpl.tp_shard_weights(g["Wu"], tp, "col")
    Sd = tpl.tp_shard_weights(g["Wd"], tp, "row")
    Y = tpl.tp_mlp_block(g["X"], Sg, Sd, W_up=Su, act="swiglu")
    # the same block as two separate calls (column then row linear)
    Hs = tpl.tp_column_linear(g["X"], Sg, W_up=Su, act="swiglu")
    Y2 = tpl.tp_row_linear(Hs, Sd)
    assert tpl.tp_get_error() == 0
    rows = sample_rows(T, 192)
    _, ref = O.mlp_block(f64(d["X"][rows]), f64(d["Wg"]), f64(d["Wd"]), tp, "swiglu", W_up=f64(d["Wu"]))
    assert_close(Y[rows], ref, TOL_BF16, f"7B MLP tp={tp} (fused launch)")
    assert_close(Y2[rows], ref, TOL_BF16, f"7B MLP tp={tp} (two launches)")


@pytest.fixture(scope="module")
def gqa():
    d = S.gqa_proj(4096, 4096, 32, 8, 128)
    return d, {k: dev(v) for k, v in d.items()}


@pytest.mark.parametrize("tp", [2, 4, 8, 16])
def test_gqa_attn_proj_full(gqa, tp):
    d, g = gqa
    T, hq, hkv, hd = 4096, 32, 8, 128
    Sqkv = tpl.tp_shard_qkv(g["Wq"], g["Wk"], g["Wv"], hq, hkv, hd, tp)
    So = tpl.tp_shard_weights(g["Wo"], tp, "row")
    qkv = torch.empty((tp, T, Sqkv.shard_width), dtype=B, device="cuda")
    Y = tpl.tp_attn_proj(g["X"], Sqkv, So, qkv_out=qkv)
    assert tpl.tp_get_error() == 0
    rows = sample_rows(T, 192)
    qkv_ref, _, ref = O.attn_proj(f64(d["X"][rows]), *(f64(d[k]) for k in ("Wq", "Wk", "Wv", "Wo")),
                                  hq, hkv, hd, tp)
    assert_close(qkv[:, rows], np.stack(qkv_ref), TOL_BF16, f"GQA qkv tp={tp}")
    assert_close(Y[rows], ref, TOL_BF16, f"GQA attn tp={tp}")


@pytest.fixture(scope="module")
def decode70b():
    d = S.decode_mlp(64)
    g = {k: dev(v) for k, v in d.items()}
    W = {k: f64(d[k]) for k in ("Wg", "Wu", "Wd")}
    Sg, Su = tpl.tp_shard_weights(g["Wg"], 8, "col"), tpl.tp_shard_weights(g["Wu"], 8, "col")
    Sd = tpl.tp_shard_weights(g["Wd"], 8, "row")
    del g["Wg"], g["Wu"], g["Wd"]
    return d, g, W, (Sg, Su, Sd)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_decode_70b_mlp_full(decode70b, T):
    d, g, W, (Sg, Su, Sd) = decode70b
    X = g["X"][:T].contiguous()   # the first T rows of one 64-row draw; the oracle gets the same rows
    Y = tpl.tp_mlp_block(X, Sg, Sd, W_up=Su, act="swiglu")
    assert tpl.tp_get_error() == 0
    _, ref = O.mlp_block(f64(d["X"][:T]), W["Wg"], W["Wd"], 8, "swiglu", W_up=W["Wu"])
    assert_close(Y, ref, TOL_BF16, f"70B decode T={T}")


def test_stack4_lmhead_full():
    T, tp = 4096, 4
    d = S.stack(T)
    hq, hkv, hd = 32, 8, 128
    layers = []
    for L in d["layers"]:
        layers.append(dict(
            qkv=tpl.tp_shard_qkv(dev(L["Wq"]), dev(L["Wk"]), dev(L["Wv"]), hq, hkv, hd, tp),
            o=tpl.tp_shard_weights(dev(L["Wo"]), tp, "row"),
            g=tpl.tp_shard_weights(dev(L["Wg"]), tp, "col"), u=tpl.tp_shard_weights(dev(L["Wu"]), tp, "col"),
            d=tpl.tp_shard_weights(dev(L["Wd"]), tp, "row")))
    lm = tpl.tp_shard_weights(dev(d["W_lm"]), tp, "col")
    x = torch.from_numpy(d["X"]).to("cuda")          # fp32 residual stream
    x1 = torch.empty_like(x)
    h = torch.empty(x.shape, dtype=B, device="cuda")  # bf16 GEMM input
    rows = sample_rows(T, 48)
    block_io = []  # the GPU's fp32 residual stream into and out of each block, sampled rows
    for Lw in layers:   # the same call sequence bench.py times
        x_in = host(x[rows])
        tpl.tp_rmsnorm(x, out=h)
        tpl.tp_attn_proj(h, Lw["qkv"], Lw["o"], residual=x, out=x1)
        tpl.tp_rmsnorm(x1, out=h)
        tpl.tp_mlp_block(h, Lw["g"], Lw["d"], W_up=Lw["u"], residual=x1, act="swiglu", out=x1)
        x = x1
        block_io.append((x_in, host(x[rows])))
    tpl.tp_rmsnorm(x, out=h)
    logits = tpl.tp_column_linear(h, lm, concat=True)
    assert tpl.tp_get_error() == 0
    Ls = [{k: f64(v) for k, v in L.items()} for L in d["layers"]]
    # Each block on its own, inside the real stack: the oracle's block fed the
    # GPU's own fp32 input to that block holds the GPU block's output to the
    # bf16 bound (rows are independent through a block).
    for b, (x_in, x_out) in enumerate(block_io):
        ref_b = O.transformer_block(x_in, Ls[b], tp, hq, hkv, hd)
        assert_close(x_out, ref_b, TOL_BF16, f"stack block {b} on its own input")
    ref = O.stack_forward(f64(d["X"][rows]), Ls, f64(d["W_lm"]), tp, hq, hkv, hd)
    # Four blocks compound the bf16 rounding of every GEMM input (the normed
    # activations, V, Hs; logits are stored bf16). The model below rounds just
    # those tensors on the same rows, with no GPU involved: it lands above 2e-2
    # on its own, so the end-to-end bound is 5e-2 (each block alone meets 2e-2
    # in the checks above).
    model_err = bf16_storage_model_error(f64(d["X"][rows]), Ls, f64(d["W_lm"]), ref, hq, hkv, hd)
    assert model_err > TOL_BF16
    assert_close(logits[rows], ref, TOL_STACK, "4-block stack + LM head")


TOL_STACK = 5e-2


def bf16_storage_model_error(X, Ls, Wlm, ref, hq, hkv, hd):
    """max|model - oracle| / RMS(oracle) for a model that computes exactly but
    rounds to bf16 the tensors a bf16 pipeline must store in bf16."""
    def bf(a):
        a = np.asarray(a, np.float32).copy()
        return S.to_bf16_inplace(a).astype(np.float64)
    x = X.copy()
    group = hq // hkv
    for L in Ls:
        h = bf(O.rmsnorm(x))
        V = bf(O.linear(h, L["Wv"]))
        ctx = np.concatenate([V[:, (q // group) * hd:(q // group + 1) * hd] for q in range(hq)], 1)
        x = x + O.linear(ctx, L["Wo"])
        h = bf(O.rmsnorm(x))
        g, u = O.linear(h, L["Wg"]), O.linear(h, L["Wu"])
        x = x + O.linear(bf(O.swiglu(g, u)), L["Wd"])
    y = bf(O.linear(bf(O.rmsnorm(x)), Wlm))
    return float(np.abs(y - ref).max() / np.sqrt(np.mean(ref ** 2)))
