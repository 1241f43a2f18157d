"""Attention core between the QKV and O projections (tcgen05 kernel) against
the oracle: scaled dot-product attention of every local head, causal or
unmasked, with the GQA head map and kv replicas.

Inputs to the core are bf16 qkv buffers; the oracle takes the same bf16
values as exact reals. The kernel keeps scores, the softmax and P V in
fp32, rounds each weight P_k to bf16 before P V and divides by the row sum
of the unrounded weights, then stores the context in bf16. With w_k the
oracle's weights and O = sum_k w_k v_k its context, the GPU computes
sum_k w_k (1 + d_k) v_k with |d_k| <= 2^-8 (half an ulp of bf16, relative),
to fp32 accuracy, and rounds that to bf16 (at most 2^-8 of the value). So
each element is held to
    |gpu - O| <= 2^-8 * 1.01 * sum_k w_k |v_k| + 2^-8 * |O| + 1e-6,
the 1% and the 1e-6 covering fp32 sums and the MUFU exponential. This
follows the rows' own scale: causal rows that average a few keys are large,
and a row of two keys whose values nearly cancel has a small context but an
error set by its two values. The projection output Y of the block is held
to the plain 2e-2 * RMS.
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_BF16, assert_close, dev, f64, host

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")
B = torch.bfloat16


def qkv_input(seed, tp, T, hq, hkv, hd=128):
    nq, nkv = hq // tp, (hkv // tp if hkv >= tp else 1)
    return S.normal(seed, (tp, T, (nq + 2 * nkv) * hd))


def oracle_ctx_bound(qkv, hq, hkv, hd, causal, rows=None):
    """The oracle's context [tp][rows][nq * hd] and the per-element bound of
    the module docstring, for query rows a..b (all rows by default) of every
    shard, each row against all the keys it sees."""
    tp, T = qkv.shape[0], qkv.shape[1]
    a, b = rows if rows is not None else (0, T)
    layout = O.qkv_head_layout(hq, hkv, tp)
    ctx, bound = [], []
    for s in range(tp):
        q_heads, kv_heads = layout[s]
        nq, nkv = len(q_heads), len(kv_heads)
        x = f64(qkv[s])
        c_s, b_s = [], []
        for i, h in enumerate(q_heads):
            g = kv_heads.index(h // (hq // hkv))
            k0, v0 = (nq + g) * hd, (nq + nkv + g) * hd
            w = O.attention_weights(x[a:b, i * hd:(i + 1) * hd], x[:, k0:k0 + hd], causal, q_offset=a)
            v = x[:, v0:v0 + hd]
            o = O.attention_head(x[a:b, i * hd:(i + 1) * hd], x[:, k0:k0 + hd], v, causal, q_offset=a)
            c_s.append(o)
            b_s.append(2.0 ** -8 * 1.01 * (w @ np.abs(v)) + 2.0 ** -8 * np.abs(o) + 1e-6)
        ctx.append(np.concatenate(c_s, 1))
        bound.append(np.concatenate(b_s, 1))
    return np.stack(ctx), np.stack(bound)


def assert_within(gpu, ref, bound, what):
    g = host(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    excess = np.abs(g - ref) - bound
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess[i] <= 0, f"{what}: at {i} err {abs(g[i] - ref[i]):.4g} > bound {bound[i]:.4g}"


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("tp,T,hq,hkv,hd", [
    (1, 128, 1, 1, 128),      # one query block: the unit's second tile is empty
    (2, 200, 4, 2, 128),      # two q heads of one kv head per unit, ragged last block
    (4, 384, 8, 2, 128),      # kv heads replicated over two shards each
    (2, 1, 2, 2, 128),        # a single token
    (2, 300, 4, 4, 128),      # one q head per kv head: units of two query blocks, an odd count
    (16, 2200, 32, 8, 128),   # 18 x 16 = 288 units over 148 CTAs, pairs of heads
    (16, 2200, 32, 32, 128),  # 9 x 32 = 288 units of two query blocks
    (2, 300, 4, 2, 64),       # head size 64, pairs of heads
    (1, 520, 2, 2, 64),       # head size 64, pairs of query blocks, five blocks
    (8, 1100, 16, 4, 64),     # head size 64, nine blocks
])
def test_attention_core(tp, T, hq, hkv, hd, causal):
    """Several key blocks, ragged last blocks, replicated kv heads, a single
    token, both ways of pairing query tiles into a work unit (two q heads
    of one kv head; two query blocks of one head, whose causal key ranges
    differ by one block), more units than SMs (so that each CTA of the
    persistent kernel runs several units of different lengths), and both
    head sizes."""
    qkv = qkv_input(301 + T, tp, T, hq, hkv, hd)
    ctx = tpl.tp_attention(dev(qkv), hq, hkv, hd, causal=causal)
    assert tpl.tp_get_error() == 0
    assert_within(ctx, *oracle_ctx_bound(qkv, hq, hkv, hd, causal),
                  f"attention tp={tp} T={T} hq={hq} hkv={hkv} hd={hd} causal={causal}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv,hd", [(2, 1, 128), (1, 1, 128), (2, 1, 64), (1, 1, 64)])
def test_attention_growing_keys_move_the_exponent_base(causal, hq, hkv, hd):
    """Key rows scaled by 1 + t/40, so that the exponentials of later key
    blocks, taken with the running base, sum above 2^16 and the base moves,
    with O rescaled in TMEM (T = 700: six blocks, the last ragged), in units
    of two heads and in units of two query blocks."""
    tp, T = 1, 700
    qkv = qkv_input(341, tp, T, hq, hkv, hd)
    k0 = hq * hd
    qkv[:, :, k0:k0 + hd] *= (1.0 + np.arange(T) / 40.0)[None, :, None]
    S.to_bf16_inplace(qkv)  # the kernel's inputs, exactly
    ctx = tpl.tp_attention(dev(qkv), hq, hkv, hd, causal=causal)
    assert tpl.tp_get_error() == 0
    assert_within(ctx, *oracle_ctx_bound(qkv, hq, hkv, hd, causal), f"growing keys hq={hq} hd={hd} causal={causal}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv,hd", [(2, 1, 128), (1, 1, 128), (2, 1, 64)])
def test_attention_outlier_keys_move_the_exponent_base(causal, hq, hkv, hd):
    """Single keys scaled by 40 in the second half of the first block (key
    100: the base moves while O holds only the first half's P V), in a first
    half (key 300) and in a second half later on (key 500): every row that
    sees one takes the slow path there, the others keep their base."""
    tp, T = 1, 600
    qkv = qkv_input(361, tp, T, hq, hkv, hd)
    k0 = hq * hd
    for key in (100, 300, 500):
        qkv[:, key, k0:k0 + hd] *= 40.0
    S.to_bf16_inplace(qkv)
    ctx = tpl.tp_attention(dev(qkv), hq, hkv, hd, causal=causal)
    assert tpl.tp_get_error() == 0
    assert_within(ctx, *oracle_ctx_bound(qkv, hq, hkv, hd, causal), f"outlier keys hq={hq} hd={hd} causal={causal}")


@pytest.mark.parametrize("hd", [64, 128])
def test_attention_single_token_is_v(hd):
    """One token: the softmax weight is exactly 1, so the context is V."""
    qkv = qkv_input(311, 2, 1, 4, 2, hd)
    ctx = host(tpl.tp_attention(dev(qkv), 4, 2, hd, causal=True))
    layout = O.qkv_head_layout(4, 2, 2)
    want = np.stack([O.context_standin(f64(qkv[s]), layout[s][0], layout[s][1], 4, 2, hd) for s in range(2)])
    np.testing.assert_array_equal(ctx, want)


def test_attention_validation():
    with pytest.raises(tpl.TpError):     # head size 96: not served by the kernel
        tpl.tp_attention(torch.zeros((2, 8, 4 * 96), dtype=B, device="cuda"), 2, 2, 96)
    with pytest.raises(tpl.TpError):     # 3 q heads over 2 shards
        tpl.tp_attention(torch.zeros((2, 8, 6 * 128), dtype=B, device="cuda"), 3, 1, 128)


@pytest.mark.parametrize("attention", ["causal", "full"])
@pytest.mark.parametrize("hd", [128, 64])
def test_attn_block_with_core(attention, hd):
    """X -> QKV by heads -> attention core -> O + sum + residual."""
    T, H, hkv, tp = 260, 512, 2, 4
    hq = 2 * H // hd
    d = S.gqa_proj(T, H, hq, hkv, hd, seeds=(321, 322, 323, 324, 325))
    R = S.normal(326, (T, H))
    Sqkv = tpl.tp_shard_qkv(dev(d["Wq"]), dev(d["Wk"]), dev(d["Wv"]), hq, hkv, hd, tp)
    So = tpl.tp_shard_weights(dev(d["Wo"]), tp, "row")
    qkv = torch.empty((tp, T, Sqkv.shard_width), dtype=B, device="cuda")
    Y = tpl.tp_attn_block(dev(d["X"]), Sqkv, So, attention=attention, residual=dev(R), qkv_out=qkv)
    assert tpl.tp_get_error() == 0
    _, _, Y_ref = O.attn_proj(*(f64(d[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), hq, hkv, hd, tp,
                              residual=f64(R), attention=attention)
    assert_close(Y, Y_ref, TOL_BF16, f"attention block ({attention}, hd {hd})")
    # the core alone on the block's own qkv
    ctx = tpl.tp_attention(qkv, hq, hkv, hd, causal=attention == "causal")
    assert_within(ctx, *oracle_ctx_bound(host(qkv), hq, hkv, hd, attention == "causal"), "core on block qkv")


def test_attention_full_size_gqa_sampled_rows():
    """The GQA workload (T = 4096, 32 q / 8 kv heads, tp = 16): causal
    context of windows of query rows spread over the sequence -- the first
    256, windows that straddle query-block boundaries in the middle, the
    last 128 -- against the oracle (each row against all the keys it sees)."""
    T, hq, hkv, tp = 4096, 32, 8, 16
    qkv = qkv_input(331, tp, T, hq, hkv)
    ctx = host(tpl.tp_attention(dev(qkv), hq, hkv, 128, causal=True))
    assert tpl.tp_get_error() == 0
    for a, b in ((0, 256), (1000, 1100), (2040, 2180), (3071, 3137), (T - 128, T)):
        assert_within(ctx[:, a:b], *oracle_ctx_bound(qkv, hq, hkv, 128, True, rows=(a, b)), f"rows {a}..{b}")
