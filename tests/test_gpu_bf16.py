"""GPU parity of the bf16 tensor-core path against the fp64 oracle, element by
element, at sizes the oracle finishes in seconds. Shapes are chosen to span
several 128x256 tiles and 64-wide k-blocks and to leave ragged tails in every
dimension (tokens, output columns per shard, K per shard).
Tolerance: max|gpu - oracle| <= 2e-2 * RMS(oracle)."""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_BF16, TOL_F32, assert_close, assert_close_stored, dev, f64, host

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")

B = torch.bfloat16


def nb(seed, shape, std=1.0):
    return S.normal(seed, shape, std)


@pytest.mark.parametrize("act", ["none", "relu", "gelu", "silu"])
@pytest.mark.parametrize("concat", [False, True])
def test_column_linear_acts_tails(act, concat):
    T, K, N, tp = 300, 200, 3 * 344, 3      # M tail 44, K tail 8, shard tail 88
    X, W, b = nb(1, (T, K)), nb(2, (K, N), 0.05), nb(3, (N,), 0.5)
    Sc = tpl.tp_shard_weights(dev(W), tp, "col")
    Y = tpl.tp_column_linear(dev(X), Sc, bias=dev(b), act=act, concat=concat)
    ref = O.column_parallel(f64(X), f64(W), tp, f64(b), O.ACTIVATIONS[act])
    assert_close(Y, O.all_gather(ref) if concat else np.stack(ref), TOL_BF16, f"col {act}")


@pytest.mark.parametrize("T,K,I,tp", [(257, 256, 2 * 1376, 2), (129, 64, 8 * 136, 8), (64, 512, 4 * 256, 4)])
def test_column_swiglu(T, K, I, tp):
    X, Wg, Wu = nb(4, (T, K)), nb(5, (K, I), 0.05), nb(6, (K, I), 0.05)
    bg, bu = nb(7, (I,), 0.3), nb(8, (I,), 0.3)
    Sg = tpl.tp_shard_weights(dev(Wg), tp, "col")
    Su = tpl.tp_shard_weights(dev(Wu), tp, "col")
    Y = tpl.tp_column_linear(dev(X), Sg, W_up=Su, bias=dev(bg), bias_up=dev(bu), act="swiglu")
    G = O.column_parallel(f64(X), f64(Wg), tp, f64(bg))
    U = O.column_parallel(f64(X), f64(Wu), tp, f64(bu))
    assert_close_stored(Y, np.stack([O.swiglu(G[s], U[s]) for s in range(tp)]), TOL_BF16, "swiglu")


@pytest.mark.parametrize("T,K,N,tp", [(200, 3 * 344, 264, 3), (130, 8 * 72, 512, 8), (5, 2 * 64, 256, 2)])
def test_row_linear_fused_and_partials(T, K, N, tp):
    Xf, W = nb(9, (T, K)), nb(10, (K, N), 0.05)
    b, R = nb(11, (N,), 0.5), nb(12, (T, N))
    Xs_np = np.ascontiguousarray(Xf.reshape(T, tp, K // tp).transpose(1, 0, 2))  # [tp][T][K/tp]
    Sr = tpl.tp_shard_weights(dev(W), tp, "row")
    Xs = dev(Xs_np)
    parts = O.row_parallel_partials([f64(x) for x in Xs_np], f64(W), tp)
    ref = O.all_reduce(parts) + f64(b) + f64(R)
    assert_close(tpl.tp_row_linear(Xs, Sr, bias=dev(b), residual=dev(R)), ref, TOL_BF16, "row fused")
    P = tpl.tp_row_linear_partials(Xs, Sr)
    assert_close(P, np.stack(parts), TOL_F32, "row partials (fp32 accumulation of bf16 products)")
    assert_close(tpl.tp_shard_reduce(P, bias=dev(b), residual=dev(R), out_dtype=B), ref, TOL_BF16, "reduce")
    if T % tp == 0:
        rs = tpl.tp_shard_reduce(P, op="scatter", out_dtype=torch.float32)
        assert_close(rs, np.stack(O.reduce_scatter(parts, tp)), TOL_F32, "reduce-scatter")


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_mlp_block_swiglu_small(tp):
    T, H, I = 333, 256, 8 * 344
    d = S.swiglu_mlp(T, H, I, seeds=(21, 22, 23, 24))
    R = nb(25, (T, H))
    Sg, Su = (tpl.tp_shard_weights(dev(d[k]), tp, "col") for k in ("Wg", "Wu"))
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    Y = tpl.tp_mlp_block(dev(d["X"]), Sg, Sd, W_up=Su, residual=dev(R), act="swiglu")
    _, ref = O.mlp_block(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, "swiglu", W_up=f64(d["Wu"]), residual=f64(R))
    assert_close(Y, ref, TOL_BF16, f"mlp swiglu tp={tp}")


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_mlp_block_plain_acts_bias(act):
    T, H, I, tp = 150, 128, 4 * 96, 4
    X, W1, W2 = nb(31, (T, H)), nb(32, (H, I), 0.05), nb(33, (I, H), 0.05)
    b1, b2 = nb(34, (I,), 0.3), nb(35, (H,), 0.3)
    S1 = tpl.tp_shard_weights(dev(W1), tp, "col")
    S2 = tpl.tp_shard_weights(dev(W2), tp, "row")
    Y = tpl.tp_mlp_block(dev(X), S1, S2, b1=dev(b1), b2=dev(b2), act=act)
    _, ref = O.mlp_block(f64(X), f64(W1), f64(W2), tp, act, b1=f64(b1), b2=f64(b2))
    assert_close(Y, ref, TOL_BF16, f"mlp {act}")


@pytest.mark.parametrize("tp", [1, 2, 4, 8, 16])
def test_attn_proj_gqa_small(tp):
    T, H, hq, hkv, hd = 260, 256, 16, 4, 64   # hkv < tp replicates KV at tp 8, 16
    d = S.gqa_proj(T, H, hq, hkv, hd, seeds=(41, 42, 43, 44, 45))
    R = nb(46, (T, H))
    Sqkv = tpl.tp_shard_qkv(dev(d["Wq"]), dev(d["Wk"]), dev(d["Wv"]), hq, hkv, hd, tp)
    So = tpl.tp_shard_weights(dev(d["Wo"]), tp, "row")
    qkv_ref, ctx_ref, Y_ref = O.attn_proj(*(f64(d[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), hq, hkv, hd, tp,
                                          residual=f64(R))
    qkv = torch.empty((tp, T, qkv_ref[0].shape[1]), dtype=B, device="cuda")
    Y = tpl.tp_attn_proj(dev(d["X"]), Sqkv, So, residual=dev(R), qkv_out=qkv)
    assert_close(qkv, np.stack(qkv_ref), TOL_BF16, f"qkv tp={tp}")
    assert_close(Y, Y_ref, TOL_BF16, f"attn tp={tp}")
    # an explicit per-shard context replaces the stand-in
    ctx = nb(47, (tp, T, hq // tp * hd))
    Y2 = tpl.tp_attn_proj(dev(d["X"]), Sqkv, So, ctx=dev(ctx))
    _, _, Y2_ref = O.attn_proj(*(f64(d[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), hq, hkv, hd, tp,
                               ctx=[f64(c) for c in ctx])
    assert_close(Y2, Y2_ref, TOL_BF16, "attn explicit ctx")


def test_rmsnorm_and_gather():
    X, g = nb(51, (77, 4096)), nb(52, (4096,), 1.0)
    assert_close_stored(tpl.tp_rmsnorm(dev(X), dev(g)), O.rmsnorm(f64(X), f64(g)), TOL_BF16, "rmsnorm bf16")
    assert_close(tpl.tp_rmsnorm(dev(X)), O.rmsnorm(f64(X)), TOL_BF16, "rmsnorm bf16, unit gain")
    assert_close(tpl.tp_rmsnorm(dev(X, torch.float32)), O.rmsnorm(f64(X)), TOL_F32, "rmsnorm f32")
    sh = nb(53, (4, 33, 80))
    ref = O.all_gather(list(sh))
    np.testing.assert_array_equal(host(tpl.tp_shard_gather(dev(sh))), ref)
    np.testing.assert_array_equal(host(tpl.tp_shard_gather(dev(sh, torch.float32))), ref)


def test_shard_layouts_bitwise():
    """Sharded storage is a pure copy: compare bits with the oracle's shards."""
    K, N, tp = 96, 160, 4
    W = nb(54, (K, N))
    c = host(tpl.tp_shard_weights(dev(W), tp, "col").storage).reshape(tp, N // tp, K)
    r = host(tpl.tp_shard_weights(dev(W), tp, "row").storage).reshape(tp, N, K // tp)
    for s in range(tp):
        np.testing.assert_array_equal(c[s], O.column_shards(f64(W), tp)[s].T)
        np.testing.assert_array_equal(r[s], O.row_shards(f64(W), tp)[s].T)
    H, hq, hkv, hd = 64, 8, 2, 16
    Wq, Wk, Wv = nb(55, (H, hq * hd)), nb(56, (H, hkv * hd)), nb(57, (H, hkv * hd))
    for tp in (1, 2, 4, 8):
        q = tpl.tp_shard_qkv(dev(Wq), dev(Wk), dev(Wv), hq, hkv, hd, tp)
        got = host(q.storage).reshape(tp, -1, H)
        for s, ws in enumerate(O.qkv_shards(f64(Wq), f64(Wk), f64(Wv), hq, hkv, hd, tp)):
            np.testing.assert_array_equal(got[s], ws.T)


@pytest.mark.parametrize("T", [1, 8, 32, 64, 100])
def test_small_token_counts(T):
    H, I, tp = 512, 8 * 136, 8
    d = S.decode_mlp(T, H, I, seed=60)
    Sg, Su = (tpl.tp_shard_weights(dev(d[k]), tp, "col") for k in ("Wg", "Wu"))
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    R = nb(61, (T, H))
    Y = tpl.tp_mlp_block(dev(d["X"]), Sg, Sd, W_up=Su, residual=dev(R), act="swiglu")
    _, ref = O.mlp_block(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, "swiglu", W_up=f64(d["Wu"]), residual=f64(R))
    assert_close(Y, ref, TOL_BF16, f"decode-shaped T={T}")
    assert tpl.tp_get_error() == 0


@pytest.mark.parametrize("hq,hkv,tp", [(32, 8, 16), (32, 2, 32), (32, 4, 8)])
def test_attn_proj_replica_dedup(hq, hkv, tp):
    """kv heads replicated over tp/hkv shards: their K|V tiles are computed once
    and stored to every shard of the group (hd 128 makes whole K|V tiles)."""
    T, H, hd = 260, 256, 128
    d = S.gqa_proj(T, H, hq, hkv, hd, seeds=(71, 72, 73, 74, 75))
    Sqkv = tpl.tp_shard_qkv(dev(d["Wq"]), dev(d["Wk"]), dev(d["Wv"]), hq, hkv, hd, tp)
    So = tpl.tp_shard_weights(dev(d["Wo"]), tp, "row")
    qkv_ref, _, Y_ref = O.attn_proj(*(f64(d[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), hq, hkv, hd, tp)
    qkv = torch.full((tp, T, qkv_ref[0].shape[1]), float("nan"), dtype=B, device="cuda")
    Y = tpl.tp_attn_proj(dev(d["X"]), Sqkv, So, qkv_out=qkv)
    assert_close(qkv, np.stack(qkv_ref), TOL_BF16, "qkv with replicas")
    g = qkv.float().cpu().numpy()
    rep = tp // hkv
    kv0 = hq // tp * hd
    c0 = -(-kv0 // 256) * 256   # first column of the whole-K|V tiles (computed once per group)
    for s in range(0, tp, rep):  # deduped tiles: replicas hold bitwise the primary's values
        for r in range(1, rep):
            np.testing.assert_array_equal(g[s][:, c0:], g[s + r][:, c0:])
    assert_close(Y, Y_ref, TOL_BF16, "attn with replicas")
    # the standalone call (whole tiles, no workspace) dedups the same way; its
    # summation order differs from the split-tile schedule, so compare within rounding
    qkv2 = tpl.tp_column_linear(dev(d["X"]), Sqkv)
    assert_close(qkv2, np.stack(qkv_ref), TOL_BF16, "standalone qkv with replicas")
    g2 = qkv2.float().cpu().numpy()
    for s in range(0, tp, rep):
        for r in range(1, rep):
            np.testing.assert_array_equal(g2[s][:, c0:], g2[s + r][:, c0:])


@pytest.mark.parametrize("T", [1, 17, 64, 65, 300])
def test_linears_with_workspace_schedules(T):
    """With a workspace and T <= 64 the column/row linears use the
    weight-streaming arrangement (split tiles); results match the oracle and
    agree with the whole-tile schedule within rounding."""
    K, N, tp = 512, 4 * 520, 4          # shard width 520: a 8-column tail past two 256 tiles
    X, W, b = nb(81, (T, K)), nb(82, (K, N), 0.05), nb(83, (N,), 0.5)
    Sc = tpl.tp_shard_weights(dev(W), tp, "col")
    ws = torch.empty(max(tpl.tp_gemm_workspace_bytes(T, Sc), 256), dtype=torch.uint8, device="cuda")
    ref = np.stack(O.column_parallel(f64(X), f64(W), tp, f64(b), O.gelu))
    Y1 = tpl.tp_column_linear(dev(X), Sc, bias=dev(b), act="gelu", workspace=ws)
    Y0 = tpl.tp_column_linear(dev(X), Sc, bias=dev(b), act="gelu")
    assert_close(Y1, ref, TOL_BF16, f"col T={T} with workspace")
    assert_close(Y0, ref, TOL_BF16, f"col T={T} whole tiles")
    Wr = nb(84, (N, 264), 0.05)
    Sr = tpl.tp_shard_weights(dev(Wr), tp, "row")
    R = nb(85, (T, 264))
    wsr = torch.empty(max(tpl.tp_gemm_workspace_bytes(T, Sr), 256), dtype=torch.uint8, device="cuda")
    parts = O.row_parallel_partials([f64(x) for x in np.ascontiguousarray(
        host(Y1).reshape(tp, T, N // tp))], f64(Wr), tp)
    refr = O.all_reduce(parts) + f64(R)
    Z1 = tpl.tp_row_linear(Y1, Sr, residual=dev(R), workspace=wsr)
    Z0 = tpl.tp_row_linear(Y1, Sr, residual=dev(R))
    assert_close(Z1, refr, TOL_BF16, f"row T={T} with workspace")
    assert_close(Z0, refr, TOL_BF16, f"row T={T} whole tiles")
    Zi = dev(R)                                       # residual aliasing the output
    tpl.tp_row_linear(Y1, Sr, residual=Zi, out=Zi, workspace=wsr)
    assert_close(Zi, refr, TOL_BF16, "row residual in place")
    assert tpl.tp_get_error() == 0


def test_swiglu_swap_many_shards_and_tails():
    """Weight-streaming arrangement with a shard width that is not a multiple
    of 128 and a K that is not a multiple of 64."""
    T, H, I, tp = 5, 200, 16 * 104, 16
    d = S.swiglu_mlp(T, H, I, seeds=(86, 87, 88, 89))
    Sg, Su = (tpl.tp_shard_weights(dev(d[k]), tp, "col") for k in ("Wg", "Wu"))
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    Y = tpl.tp_mlp_block(dev(d["X"]), Sg, Sd, W_up=Su, act="swiglu")
    _, ref = O.mlp_block(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, "swiglu", W_up=f64(d["Wu"]))
    assert_close(Y, ref, TOL_BF16, "swap swiglu tails")


def test_fp32_residual_stream_outputs():
    """bf16 GEMM operands with fp32 bias / residual / output: the row linear's
    output is not rounded to bf16, so it meets the fp32 tolerance; blocks whose
    intermediate (Hs, qkv) is bf16 meet the bf16 tolerance."""
    F = torch.float32
    rng = np.random.default_rng(120)
    for T in (200, 9):   # whole tiles; weight-streaming arrangement (with workspace)
        K, N, tp = 4 * 344, 264, 4
        Xf, W = nb(121, (T, K)), nb(122, (K, N), 0.05)
        b = rng.standard_normal(N).astype(np.float32)          # not bf16-representable
        R = rng.standard_normal((T, N)).astype(np.float32)
        Xs = np.ascontiguousarray(Xf.reshape(T, tp, K // tp).transpose(1, 0, 2))
        Sr = tpl.tp_shard_weights(dev(W), tp, "row")
        ws = torch.empty(max(tpl.tp_gemm_workspace_bytes(T, Sr), 256), dtype=torch.uint8, device="cuda")
        ref = O.all_reduce(O.row_parallel_partials([f64(x) for x in Xs], f64(W), tp)) + f64(b) + f64(R)
        Rd = dev(R, F)
        Y = tpl.tp_row_linear(dev(Xs), Sr, bias=dev(b, F), residual=Rd, workspace=ws)
        assert Y.dtype == F
        assert_close(Y, ref, TOL_F32, f"row linear fp32 out T={T}")
        tpl.tp_row_linear(dev(Xs), Sr, bias=dev(b, F), residual=Rd, out=Rd, workspace=ws)  # in place
        assert_close(Rd, ref, TOL_F32, f"row linear fp32 in place T={T}")
    T, H, I, tp = 130, 256, 4 * 344, 4
    d = S.swiglu_mlp(T, H, I, seeds=(123, 124, 125, 126))
    R = rng.standard_normal((T, H)).astype(np.float32)
    Sg, Su = (tpl.tp_shard_weights(dev(d[k]), tp, "col") for k in ("Wg", "Wu"))
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    Y = tpl.tp_mlp_block(dev(d["X"]), Sg, Sd, W_up=Su, residual=dev(R, F), act="swiglu")
    assert Y.dtype == F
    _, ref = O.mlp_block(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, "swiglu", W_up=f64(d["Wu"]), residual=f64(R))
    assert_close(Y, ref, TOL_BF16, "mlp fp32 residual")
    hq, hkv, hd = 8, 2, 32
    g = S.gqa_proj(T, H, hq, hkv, hd, seeds=(127, 128, 129, 130, 131))
    Sq = tpl.tp_shard_qkv(dev(g["Wq"]), dev(g["Wk"]), dev(g["Wv"]), hq, hkv, hd, tp)
    So = tpl.tp_shard_weights(dev(g["Wo"]), tp, "row")
    Ya = tpl.tp_attn_proj(dev(g["X"]), Sq, So, residual=dev(R, F))
    _, _, ref = O.attn_proj(*(f64(g[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), hq, hkv, hd, tp, residual=f64(R))
    assert Ya.dtype == F
    assert_close(Ya, ref, TOL_BF16, "attn fp32 residual")
    h = tpl.tp_rmsnorm(dev(R, F), out_dtype=B)     # fp32 stream -> bf16 GEMM input
    assert h.dtype == B
    assert_close(h, O.rmsnorm(f64(R)), TOL_BF16, "rmsnorm fp32 -> bf16")
    assert tpl.tp_get_error() == 0


@pytest.mark.parametrize("T,hq,hkv,hd,tp", [(260, 32, 8, 128, 16), (260, 16, 4, 64, 4), (130, 32, 2, 128, 32),
                                            (24, 32, 8, 128, 16), (64, 16, 16, 64, 4), (1, 8, 2, 64, 8)])
def test_attn_fused_context(T, hq, hkv, hd, tp):
    """Without a caller context the bf16 QKV epilogue writes the single-key
    stand-in itself: every query head's block of the context (in the caller
    workspace, after the qkv region) holds bitwise the V columns of its kv
    head on the same shard. T <= 64 runs the weight-streaming arrangement,
    hkv < tp the replica-dedup tiles."""
    H = 256
    d = S.gqa_proj(T, H, hq, hkv, hd, seeds=(81, 82, 83, 84, 85))
    Sqkv = tpl.tp_shard_qkv(dev(d["Wq"]), dev(d["Wk"]), dev(d["Wv"]), hq, hkv, hd, tp)
    So = tpl.tp_shard_weights(dev(d["Wo"]), tp, "row")
    Ns = Sqkv.shard_width
    ws = torch.zeros(tpl.tp_attn_workspace_bytes(T, hq, hkv, hd, tp, B), dtype=torch.uint8, device="cuda")
    qkv = torch.empty((tp, T, Ns), dtype=B, device="cuda")
    Y = tpl.tp_attn_proj(dev(d["X"]), Sqkv, So, qkv_out=qkv, workspace=ws)
    assert tpl.tp_get_error() == 0
    c0 = -(-(T * tp * Ns * 2) // 256) * 256   # the context follows the (256-aligned) qkv region
    nc = hq // tp * hd
    ctx = ws[c0:c0 + tp * T * nc * 2].view(B).view(tp, T, nc)
    g = host(qkv)
    layout = O.qkv_head_layout(hq, hkv, tp)
    for s in range(tp):
        want = O.context_standin(g[s], layout[s][0], layout[s][1], hq, hkv, hd)
        np.testing.assert_array_equal(host(ctx[s]), want, err_msg=f"context of shard {s}")
    qkv_ref, _, Y_ref = O.attn_proj(*(f64(d[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), hq, hkv, hd, tp)
    assert_close(qkv, np.stack(qkv_ref), TOL_BF16, "qkv")
    assert_close(Y, Y_ref, TOL_BF16, "attn with the fused context")


@pytest.mark.parametrize("T", [256, 1100])
def test_cluster_pairs(T):
    """Token-major launches with an even number of token blocks, or at least
    eight, run as CTA pairs (2-SM MMA, 256-token units, each CTA staging half
    of every weight tile). 1100 tokens make 9 blocks, so the odd CTA of the
    last unit has no token rows (its A tile is zero fill, it stores nothing)."""
    H, I, tp = 384, 4 * 320, 4
    d = S.swiglu_mlp(T, H, I, seeds=(91, 92, 93, 94))
    Sg, Su = (tpl.tp_shard_weights(dev(d[k]), tp, "col") for k in ("Wg", "Wu"))
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    Hs_ref, Y_ref = O.mlp_block(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, "swiglu", W_up=f64(d["Wu"]))
    Hs = tpl.tp_column_linear(dev(d["X"]), Sg, W_up=Su, act="swiglu")
    assert_close_stored(Hs, np.stack(Hs_ref), TOL_BF16, f"paired SwiGLU column T={T}")
    assert_close(tpl.tp_row_linear(Hs, Sd), Y_ref, TOL_BF16, f"paired row sum T={T}")
    P = tpl.tp_row_linear_partials(Hs, Sd)
    P_ref = O.row_parallel_partials([f64(h) for h in host(Hs)], f64(d["Wd"]), tp)
    assert_close(P, np.stack(P_ref), TOL_F32, f"paired row partials T={T}")
    b = nb(95, (I,), 0.3)
    Yc = tpl.tp_column_linear(dev(d["X"]), Sg, bias=dev(b), act="gelu", concat=True)
    ref = np.concatenate(O.column_parallel(f64(d["X"]), f64(d["Wg"]), tp, bias=f64(b), act=O.gelu), axis=1)
    assert_close_stored(Yc, ref, TOL_BF16, f"paired column, bias + GELU, concatenated T={T}")
    g = S.gqa_proj(T, H, 16, 2, 128, seeds=(96, 97, 98, 99, 100))   # kv replicated over 4 shards of 8
    Sqkv = tpl.tp_shard_qkv(dev(g["Wq"]), dev(g["Wk"]), dev(g["Wv"]), 16, 2, 128, 8)
    So = tpl.tp_shard_weights(dev(g["Wo"]), 8, "row")
    qkv_ref, _, Ya_ref = O.attn_proj(*(f64(g[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), 16, 2, 128, 8)
    qkv = torch.empty((8, T, qkv_ref[0].shape[1]), dtype=B, device="cuda")
    Ya = tpl.tp_attn_proj(dev(g["X"]), Sqkv, So, qkv_out=qkv)
    assert_close(qkv, np.stack(qkv_ref), TOL_BF16, f"paired QKV with replicas T={T}")
    assert_close(Ya, Ya_ref, TOL_BF16, f"paired attention projections T={T}")
    assert tpl.tp_get_error() == 0


@pytest.mark.parametrize("T", [256, 1100])
def test_split_last_round(T):
    """With a workspace, a paired row-GEMM launch whose units leave pairs of
    SMs idle in the last round cuts those units along K into pieces (one per
    pair) and combines them in a fixed order. Checked against the oracle; the
    column launches (which run whole with or without a workspace) against the
    oracle and the call without a workspace. Row GEMM: 6 units at 256 tokens,
    cut 4 ways (and the O projection's 8); at 1100 tokens (5 token units, the
    last one half empty) 30 units, cut 2 ways."""
    tp, K, Nc = 2, 2048, 2 * 768         # column: 3 units of 256 columns per shard, per 256 tokens
    X, W, b = nb(121, (T, K)), nb(122, (K, Nc), 0.02), nb(123, (Nc,), 0.3)
    Sc = tpl.tp_shard_weights(dev(W), tp, "col")
    ws = torch.empty(tpl.tp_gemm_workspace_bytes(T, Sc), dtype=torch.uint8, device="cuda")
    ref = np.concatenate(O.column_parallel(f64(X), f64(W), tp, bias=f64(b), act=O.gelu), axis=1)
    Y1 = tpl.tp_column_linear(dev(X), Sc, bias=dev(b), act="gelu", concat=True, workspace=ws)
    Y0 = tpl.tp_column_linear(dev(X), Sc, bias=dev(b), act="gelu", concat=True)
    assert_close_stored(Y1, ref, TOL_BF16, f"split column T={T}")
    assert_close_stored(Y1, host(Y0), TOL_BF16, f"split vs whole column T={T}")

    Wg, Wu = nb(124, (K, Nc), 0.02), nb(125, (K, Nc), 0.02)
    Sg, Su = tpl.tp_shard_weights(dev(Wg), tp, "col"), tpl.tp_shard_weights(dev(Wu), tp, "col")
    Hs = tpl.tp_column_linear(dev(X), Sg, W_up=Su, act="swiglu", workspace=ws)
    Hs_ref = O.column_parallel(f64(X), f64(Wg), tp)
    Up_ref = O.column_parallel(f64(X), f64(Wu), tp)
    assert_close_stored(Hs, np.stack([O.swiglu(g, u) for g, u in zip(Hs_ref, Up_ref)]), TOL_BF16,
                        f"split SwiGLU T={T}")
    Kr, Nr = 2048, 1536                   # row: 6 column blocks of 256, per 256 tokens
    Wr = nb(126, (Kr, Nr), 0.02)
    Sr = tpl.tp_shard_weights(dev(Wr), tp, "row")
    Xs = nb(127, (tp, T, Kr // tp))
    br, R = nb(128, (Nr,), 0.3), nb(129, (T, Nr))
    wsr = torch.empty(tpl.tp_gemm_workspace_bytes(T, Sr), dtype=torch.uint8, device="cuda")
    Yr = tpl.tp_row_linear(dev(Xs), Sr, bias=dev(br, torch.float32), residual=dev(R, torch.float32),
                           workspace=wsr)
    ref_r = O.all_reduce(O.row_parallel_partials([f64(x) for x in Xs], f64(Wr), tp)) + f64(br) + f64(R)
    assert_close(Yr, ref_r, TOL_BF16, f"split row sum, fp32 residual T={T}")
    Yr2 = tpl.tp_row_linear(dev(Xs), Sr, bias=dev(br, torch.float32), residual=dev(R, torch.float32),
                            workspace=wsr)
    np.testing.assert_array_equal(host(Yr2), host(Yr))   # fixed combine order: run to run identical
    Yr0 = tpl.tp_row_linear(dev(Xs), Sr, bias=dev(br, torch.float32), residual=dev(R, torch.float32))
    assert_close(Yr, host(Yr0), TOL_F32 * 10, f"split vs whole row sum T={T}")
    # attention projections: QKV (with replicas) and O both split
    g = S.gqa_proj(T, 2048, 16, 4, 128, seeds=(130, 131, 132, 133, 134))
    Sqkv = tpl.tp_shard_qkv(dev(g["Wq"]), dev(g["Wk"]), dev(g["Wv"]), 16, 4, 128, 8)
    So = tpl.tp_shard_weights(dev(g["Wo"]), 8, "row")
    qkv_ref, _, Ya_ref = O.attn_proj(*(f64(g[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), 16, 4, 128, 8)
    qkv = torch.empty((8, T, qkv_ref[0].shape[1]), dtype=B, device="cuda")
    Ya = tpl.tp_attn_proj(dev(g["X"]), Sqkv, So, qkv_out=qkv)
    assert_close(qkv, np.stack(qkv_ref), TOL_BF16, f"split QKV T={T}")
    assert_close(Ya, Ya_ref, TOL_BF16, f"split attention projections T={T}")
    assert tpl.tp_get_error() == 0


@pytest.mark.parametrize("T", [8, 256])
def test_graph_replay_matches_direct_calls(T):
    """The API calls can be recorded into a CUDA graph and replayed: launch
    arguments (including the split-tile epoch) are then frozen, and every
    launch returns its synchronisation words to zero, so each replay
    recombines its own pieces. 8 tokens: weight streaming with stream-K
    tiles; 256 tokens: the row GEMM's split last round. Each replay must
    reproduce the direct call bit for bit (fixed combine order)."""
    H, I, tp = 2048, 8 * 768, 8
    d = S.swiglu_mlp(T, H, I, seeds=(141, 142, 143, 144))
    Sg, Su = (tpl.tp_shard_weights(dev(d[k]), tp, "col") for k in ("Wg", "Wu"))
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    X = dev(d["X"])
    ws = torch.empty(tpl.tp_mlp_workspace_bytes(T, H, I, tp, B), dtype=torch.uint8, device="cuda")
    Y_direct = tpl.tp_mlp_block(X, Sg, Sd, W_up=Su, act="swiglu", workspace=ws)
    torch.cuda.synchronize()
    Y = torch.empty_like(Y_direct)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tpl.tp_mlp_block(X, Sg, Sd, W_up=Su, act="swiglu", workspace=ws, out=Y)
    for rep in range(3):
        Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert tpl.tp_get_error() == 0
        np.testing.assert_array_equal(host(Y), host(Y_direct), err_msg=f"replay {rep}")
    _, ref = O.mlp_block(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, "swiglu", W_up=f64(d["Wu"]))
    assert_close(Y, ref, TOL_BF16, f"graph replay T={T}")
