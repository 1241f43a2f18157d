"""Attention core between the QKV and O projections (tcgen05 kernel) against
the oracle: scaled dot-product attention of every local head, causal or
unmasked, with the GQA head map and kv replicas.

Inputs to the core are bf16 qkv buffers; the oracle takes the same bf16
values as exact reals. The kernel keeps scores, the softmax and P V in
fp32 and rounds P to bf16 before P V. The context is stored in bf16 and,
under the causal mask, its early rows average only a few values, so they
are several times larger than the rows that set the RMS: the context is
held to the bound for bf16-stored outputs, 2e-2 * RMS plus the storage
rounding of each element (2^-8 of its magnitude). The projection output Y
is held to the plain 2e-2 * RMS.
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_BF16, assert_close, assert_close_stored, dev, f64, host

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")
B = torch.bfloat16


def qkv_input(seed, tp, T, hq, hkv, hd=128):
    nq, nkv = hq // tp, (hkv // tp if hkv >= tp else 1)
    return S.normal(seed, (tp, T, (nq + 2 * nkv) * hd))


def oracle_ctx(qkv, hq, hkv, hd, causal, rows=None):
    tp = qkv.shape[0]
    layout = O.qkv_head_layout(hq, hkv, tp)
    if rows is None:
        return np.stack([O.context_attention(f64(qkv[s]), layout[s][0], layout[s][1], hq, hkv, hd, causal)
                         for s in range(tp)])
    # rows a..b of a long sequence: the queries at those positions against all keys
    a, b = rows
    out = []
    for s in range(tp):
        q_heads, kv_heads = layout[s]
        nq, nkv = len(q_heads), len(kv_heads)
        x = f64(qkv[s])
        cols = []
        for i, h in enumerate(q_heads):
            g = kv_heads.index(h // (hq // hkv))
            k0, v0 = (nq + g) * hd, (nq + nkv + g) * hd
            cols.append(O.attention_head(x[a:b, i * hd:(i + 1) * hd], x[:, k0:k0 + hd], x[:, v0:v0 + hd],
                                         causal, q_offset=a))
        out.append(np.concatenate(cols, 1))
    return np.stack(out)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("tp,T,hq,hkv", [(1, 128, 1, 1), (2, 200, 4, 2), (4, 384, 8, 2), (2, 1, 2, 2),
                                         (2, 300, 4, 4), (16, 1100, 32, 8)])
def test_attention_core(tp, T, hq, hkv, causal):
    """Several key blocks, a ragged last block (200, 300, 1100), replicated kv
    heads (tp 4 with 2 kv heads), a single token, and more work units
    (shard, q head, query block) than SMs (16 x 2 x 9 = 288), so that each
    CTA of the persistent kernel runs several units of different lengths."""
    qkv = qkv_input(301 + T, tp, T, hq, hkv)
    ctx = tpl.tp_attention(dev(qkv), hq, hkv, 128, causal=causal)
    assert tpl.tp_get_error() == 0
    assert_close_stored(ctx, oracle_ctx(qkv, hq, hkv, 128, causal), TOL_BF16,
                        f"attention tp={tp} T={T} causal={causal}")


@pytest.mark.parametrize("causal", [True, False])
def test_attention_growing_keys_move_the_exponent_base(causal):
    """Key rows scaled by 1 + t/40, so that the scores of later key blocks
    exceed the running base by more than 2^8 and O is rescaled in TMEM after
    the first block of each key-block parity (T = 700: six blocks, the last
    ragged)."""
    tp, T, hq, hkv, hd = 1, 700, 2, 1, 128
    qkv = qkv_input(341, tp, T, hq, hkv)
    k0 = hq * hd
    qkv[:, :, k0:k0 + hd] *= (1.0 + np.arange(T) / 40.0)[None, :, None]
    S.to_bf16_inplace(qkv)  # the kernel's inputs, exactly
    ctx = tpl.tp_attention(dev(qkv), hq, hkv, hd, causal=causal)
    assert tpl.tp_get_error() == 0
    assert_close_stored(ctx, oracle_ctx(qkv, hq, hkv, hd, causal), TOL_BF16, f"growing keys causal={causal}")


def test_attention_single_token_is_v():
    """One token: the softmax weight is exactly 1, so the context is V."""
    qkv = qkv_input(311, 2, 1, 4, 2)
    ctx = host(tpl.tp_attention(dev(qkv), 4, 2, 128, causal=True))
    layout = O.qkv_head_layout(4, 2, 2)
    want = np.stack([O.context_standin(f64(qkv[s]), layout[s][0], layout[s][1], 4, 2, 128) for s in range(2)])
    np.testing.assert_array_equal(ctx, want)


def test_attention_validation():
    qkv = torch.zeros((2, 8, 4 * 64), dtype=B, device="cuda")
    with pytest.raises(tpl.TpError):     # head size 64: not served by this kernel
        tpl.tp_attention(qkv, 2, 2, 64)
    with pytest.raises(tpl.TpError):     # 3 q heads over 2 shards
        tpl.tp_attention(torch.zeros((2, 8, 6 * 128), dtype=B, device="cuda"), 3, 1, 128)


@pytest.mark.parametrize("attention", ["causal", "full"])
def test_attn_block_with_core(attention):
    """X -> QKV by heads -> attention core -> O + sum + residual."""
    T, H, hq, hkv, hd, tp = 260, 512, 8, 2, 128, 4
    d = S.gqa_proj(T, H, hq, hkv, hd, seeds=(321, 322, 323, 324, 325))
    R = S.normal(326, (T, H))
    Sqkv = tpl.tp_shard_qkv(dev(d["Wq"]), dev(d["Wk"]), dev(d["Wv"]), hq, hkv, hd, tp)
    So = tpl.tp_shard_weights(dev(d["Wo"]), tp, "row")
    qkv = torch.empty((tp, T, Sqkv.shard_width), dtype=B, device="cuda")
    Y = tpl.tp_attn_block(dev(d["X"]), Sqkv, So, attention=attention, residual=dev(R), qkv_out=qkv)
    assert tpl.tp_get_error() == 0
    _, _, Y_ref = O.attn_proj(*(f64(d[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")), hq, hkv, hd, tp,
                              residual=f64(R), attention=attention)
    assert_close(Y, Y_ref, TOL_BF16, f"attention block ({attention})")
    # the core alone on the block's own qkv
    ctx = tpl.tp_attention(qkv, hq, hkv, hd, causal=attention == "causal")
    assert_close_stored(ctx, oracle_ctx(host(qkv), hq, hkv, hd, attention == "causal"), TOL_BF16,
                        "core on block qkv")


def test_attention_full_size_gqa_sampled_rows():
    """The GQA workload (T = 4096, 32 q / 8 kv heads, tp = 16): causal
    context of the first 256 and the last 128 query rows against the oracle
    (each row against all the keys it sees)."""
    T, hq, hkv, tp = 4096, 32, 8, 16
    qkv = qkv_input(331, tp, T, hq, hkv)
    ctx = host(tpl.tp_attention(dev(qkv), hq, hkv, 128, causal=True))
    assert tpl.tp_get_error() == 0
    for a, b in ((0, 256), (T - 128, T)):
        assert_close_stored(ctx[:, a:b], oracle_ctx(qkv, hq, hkv, 128, True, rows=(a, b)), TOL_BF16,
                            f"rows {a}..{b}")
