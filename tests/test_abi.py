"""C-ABI checks that need no GPU: the library loads, exports every function
include/tp.h declares, and rejects bad arguments before launching anything
(validation runs on the host and returns its status before any CUDA call)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

import tensor_transformer_linear_tma_b300 as tpl  # noqa: E402

HEADER = os.path.join(ROOT, "include", "tp.h")

# constants from tp.h
OK, NULL, SHAPE, DTYPE, MODE, ALIGN, WORKSPACE, CUDA, TIMEOUT, UNSUP, INDEX = range(11)
F32, BF16 = 0, 1
COL, ROW = 0, 1

FAKE = 0x10000  # a 64 KiB-aligned non-null address; never dereferenced by validation


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_pipeline_calls():
    names = declared_functions()
    for n in ["tp_shard_weights", "tp_shard_qkv", "tp_column_linear", "tp_row_linear",
              "tp_row_linear_partials", "tp_shard_reduce", "tp_shard_gather", "tp_mlp_block",
              "tp_attn_proj", "tp_rmsnorm", "tp_get_error"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(tpl.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version():
    for s in range(11):
        assert tpl.tp_status_string(s) != "unknown status"
    assert tpl.tp_status_string(1234) == "unknown status"
    assert tpl.lib.tp_abi_version() == 1


def view(K=64, N=256, tp=2, mode=COL, dtype=F32, data=FAKE, hq=0, hkv=0, hd=0):
    return tpl.TpShardsC(data, K, N, tp, mode, dtype, hq, hkv, hd)


def col(X=FAKE, T=16, W=None, Wu=None, bias=None, bias_up=None, act=0, concat=0, Y=FAKE):
    W = view() if W is None else W
    return tpl.lib.tp_column_linear(X, T, ctypes.byref(W), ctypes.byref(Wu) if Wu else None,
                                    bias, bias_up, act, concat, Y, None, 0, None)


def test_column_linear_validation():
    assert col(X=None) == NULL
    assert col(Y=None) == NULL
    assert col(W=view(data=None)) == NULL
    assert col(T=-1) == SHAPE
    assert col(W=view(N=255, tp=2)) == SHAPE          # N % tp != 0
    assert col(W=view(tp=0)) == SHAPE
    assert col(W=view(K=0)) == SHAPE
    assert col(W=view(mode=ROW)) == MODE
    assert col(W=view(dtype=7)) == DTYPE
    assert col(act=9) == MODE
    assert col(concat=2) == MODE
    assert col(act=4) == NULL                          # SwiGLU needs W_up
    assert col(act=4, Wu=view(N=128)) == SHAPE         # W_up must match W
    assert col(act=4, Wu=view(dtype=BF16)) in (SHAPE, ALIGN)
    assert col(Wu=view()) == MODE                      # W_up without SwiGLU
    assert col(W=view(dtype=BF16), X=FAKE + 4) == ALIGN  # bf16 needs 16-byte pointers
    assert col(W=view(dtype=BF16, K=60)) == ALIGN        # bf16 rows % 8
    assert col(W=view(dtype=BF16, N=2 * 100)) == ALIGN   # N/tp % 8
    assert col(W=view(data=FAKE + 2)) == ALIGN           # fp32 needs 4-byte pointers


def test_row_linear_validation():
    W = view(K=256, N=64, tp=2, mode=ROW)
    f = tpl.lib.tp_row_linear
    assert f(None, 16, ctypes.byref(W), None, None, FAKE, F32, None, 0, None) == NULL
    assert f(FAKE, 16, ctypes.byref(view(K=255, N=64, tp=2, mode=ROW)), None, None, FAKE, F32, None, 0, None) == SHAPE
    assert f(FAKE, 16, ctypes.byref(view(mode=COL)), None, None, FAKE, F32, None, 0, None) == MODE
    assert f(FAKE, -3, ctypes.byref(W), None, None, FAKE, F32, None, 0, None) == SHAPE
    Wb = view(K=256, N=64, tp=4, mode=ROW, dtype=BF16)   # K/tp = 64
    assert f(FAKE, 16, ctypes.byref(Wb), FAKE + 8, None, FAKE, BF16, None, 0, None) == ALIGN
    Wb = view(K=4 * 12, N=64, tp=4, mode=ROW, dtype=BF16)  # K/tp = 12, not % 8
    assert f(FAKE, 16, ctypes.byref(Wb), None, None, FAKE, BF16, None, 0, None) == ALIGN
    Wb = view(K=256, N=64, tp=4, mode=ROW, dtype=BF16)
    assert f(FAKE, 16, ctypes.byref(Wb), None, None, FAKE, BF16, FAKE + 16, 1 << 40, None) == ALIGN      # workspace 256-aligned
    assert f(FAKE, 16, ctypes.byref(Wb), None, None, FAKE, BF16, FAKE, 1024, None) == WORKSPACE
    assert f(FAKE, 16, ctypes.byref(Wb), None, None, FAKE, 7, None, 0, None) == DTYPE             # bad out dtype
    assert f(FAKE, 16, ctypes.byref(W), None, None, FAKE, BF16, None, 0, None) == DTYPE            # fp32 path writes fp32          # too small
    assert tpl.lib.tp_gemm_workspace_bytes(16, ctypes.byref(Wb)) > 0
    assert tpl.lib.tp_gemm_workspace_bytes(16, ctypes.byref(W)) == 0                              # fp32: none
    g = tpl.lib.tp_row_linear_partials
    assert g(FAKE, 16, ctypes.byref(W), None, None) == NULL


def test_reduce_and_gather_validation():
    r = tpl.lib.tp_shard_reduce
    assert r(None, 2, 4, 8, 0, None, None, F32, FAKE, None) == NULL
    assert r(FAKE, 2, 4, 8, 5, None, None, F32, FAKE, None) == MODE
    assert r(FAKE, 2, 4, 8, 0, None, None, 3, FAKE, None) == DTYPE
    assert r(FAKE, 0, 4, 8, 0, None, None, F32, FAKE, None) == SHAPE
    assert r(FAKE, 3, 4, 8, 1, None, None, F32, FAKE, None) == SHAPE   # scatter needs T % tp == 0
    assert r(FAKE + 4, 2, 4, 8, 0, None, None, F32, FAKE, None) == ALIGN
    assert r(FAKE, 2, 0, 8, 0, None, None, F32, FAKE, None) == OK      # empty: no launch
    g = tpl.lib.tp_shard_gather
    assert g(None, 2, 4, 8, F32, FAKE, None) == NULL
    assert g(FAKE, 3, 4, 8, F32, FAKE, None) == SHAPE
    assert g(FAKE, 2, 4, 8, 9, FAKE, None) == DTYPE
    assert g(FAKE, 2, 0, 8, F32, FAKE, None) == OK


def test_shard_weights_validation():
    f = tpl.lib.tp_shard_weights
    v = tpl.TpShardsC()
    big = 1 << 40
    assert f(None, 64, 256, F32, 2, COL, FAKE, big, ctypes.byref(v), None) == NULL
    assert f(FAKE, 64, 256, F32, 3, COL, FAKE, big, ctypes.byref(v), None) == SHAPE
    assert f(FAKE, 63, 256, F32, 2, ROW, FAKE, big, ctypes.byref(v), None) == SHAPE
    assert f(FAKE, 64, 256, F32, 2, 5, FAKE, big, ctypes.byref(v), None) == MODE
    assert f(FAKE, 64, 256, 2, 2, COL, FAKE, big, ctypes.byref(v), None) == DTYPE
    assert f(FAKE, 64, 256, F32, 2, COL, FAKE, 64 * 256 * 4 - 1, ctypes.byref(v), None) == WORKSPACE
    assert f(FAKE, 64, 200, BF16, 4, COL, FAKE, big, ctypes.byref(v), None) == ALIGN  # 50 % 8


def test_qkv_sizes_and_validation():
    e = tpl.tp_qkv_shard_elems
    # 32 q / 8 kv heads, hd 128, H 4096: per-shard columns (hq/tp + 2*nkv) * hd
    assert e(4096, 32, 8, 128, 2) == 2 * (16 + 8) * 128 * 4096
    assert e(4096, 32, 8, 128, 8) == 8 * (4 + 2) * 128 * 4096
    assert e(4096, 32, 8, 128, 16) == 16 * (2 + 2) * 128 * 4096   # one replicated kv head
    assert e(4096, 32, 8, 128, 3) == 0
    assert e(4096, 32, 6, 128, 4) == 0
    f = tpl.lib.tp_shard_qkv
    v = tpl.TpShardsC()
    assert f(FAKE, FAKE, FAKE, 4096, 32, 8, 128, 3, BF16, FAKE, 1 << 40, ctypes.byref(v), None) == SHAPE
    assert f(FAKE, None, FAKE, 4096, 32, 8, 128, 2, BF16, FAKE, 1 << 40, ctypes.byref(v), None) == NULL
    assert f(FAKE, FAKE, FAKE, 4096, 32, 8, 128, 2, BF16, FAKE, 10, ctypes.byref(v), None) == WORKSPACE


def test_mlp_and_attn_validation_and_workspace():
    ws = tpl.lib.tp_mlp_workspace_bytes(2048, 4096, 11008, 8, BF16)
    assert ws >= 2048 * 11008 * 2 and ws % 256 == 0
    assert tpl.lib.tp_mlp_workspace_bytes(2048, 4096, 11008, 0, BF16) == 0
    W1, W2 = view(K=64, N=256), view(K=256, N=64, mode=ROW)
    f = tpl.lib.tp_mlp_block
    args = lambda **k: dict(dict(X=FAKE, T=16, W1=W1, Wu=None, W2=W2, ws=FAKE, wsb=1 << 30, Y=FAKE, act=1), **k)

    def call(**k):
        a = args(**k)
        return f(a["X"], a["T"], ctypes.byref(a["W1"]), ctypes.byref(a["Wu"]) if a["Wu"] else None,
                 ctypes.byref(a["W2"]), None, None, None, None, a["act"], a.get("odt", F32), a["ws"], a["wsb"],
                 a["Y"], None)
    assert call(ws=None) == NULL
    assert call(wsb=16) == WORKSPACE
    assert call(W2=view(K=256, N=64, tp=4, mode=ROW)) == SHAPE        # tp mismatch
    assert call(W2=view(K=128, N=64, mode=ROW)) == SHAPE              # K of W2 != I
    assert call(W2=view(K=256, N=64, mode=COL)) == MODE
    assert call(ws=FAKE + 16) == ALIGN                                # workspace 256-aligned
    assert call(odt=BF16) == DTYPE                                    # fp32 path writes fp32
    aw = tpl.lib.tp_attn_workspace_bytes(4096, 32, 8, 128, 16, BF16)
    assert aw >= 4096 * (16 * 4 * 128) * 2 + 4096 * 4096 * 2
    Wqkv = view(K=4096, N=16 * 4 * 128, tp=16, mode=COL, dtype=BF16, hq=32, hkv=8, hd=128)
    Wo = view(K=4096, N=4096, tp=16, mode=ROW, dtype=BF16)
    a = tpl.lib.tp_attn_proj
    assert a(FAKE, 64, ctypes.byref(Wqkv), ctypes.byref(Wo), None, None, BF16, None, None, 1 << 40, FAKE, None) == NULL
    assert a(FAKE, 64, ctypes.byref(Wqkv), ctypes.byref(Wo), None, None, BF16, None, FAKE, 10, FAKE, None) == WORKSPACE
    Wplain = view(K=4096, N=16 * 4 * 128, tp=16, mode=COL, dtype=BF16)
    assert a(FAKE, 64, ctypes.byref(Wplain), ctypes.byref(Wo), None, None, BF16, None, FAKE, 1 << 40, FAKE, None) == MODE
    Wo_bad = view(K=2048, N=4096, tp=16, mode=ROW, dtype=BF16)
    assert a(FAKE, 64, ctypes.byref(Wqkv), ctypes.byref(Wo_bad), None, None, BF16, None, FAKE, 1 << 40, FAKE, None) == SHAPE


def test_rmsnorm_validation():
    f = tpl.lib.tp_rmsnorm
    assert f(None, None, 4, 8, 1e-5, F32, FAKE, F32, None) == NULL
    assert f(FAKE, None, 4, 0, 1e-5, F32, FAKE, F32, None) == SHAPE
    assert f(FAKE, None, 4, 8, -1.0, F32, FAKE, F32, None) == SHAPE
    assert f(FAKE, None, 4, 8, 1e-5, 5, FAKE, F32, None) == DTYPE
    assert f(FAKE, None, 4, 8, 1e-5, F32, FAKE, 5, None) == DTYPE
    assert f(FAKE + 2, None, 4, 8, 1e-5, F32, FAKE, BF16, None) == ALIGN
    assert f(FAKE, None, 0, 8, 1e-5, F32, FAKE, BF16, None) == OK


def test_binding_raises_on_error_status():
    with pytest.raises(tpl.TpError) as e:
        tpl._check("tp_column_linear", SHAPE)
    assert e.value.status == SHAPE and "shape" in str(e.value)


def test_backward_validation():
    L = tpl.lib
    rowv, colv = view(K=256, N=128, mode=ROW, dtype=BF16), view(K=128, N=256, mode=COL, dtype=BF16)
    # row layer
    assert L.tp_row_linear_backward(FAKE + 2, 8, ctypes.byref(view(mode=ROW)), FAKE, FAKE, FAKE, None) == ALIGN  # fp32
    assert L.tp_row_linear_backward(FAKE, 8, ctypes.byref(colv), FAKE, FAKE, FAKE, None) == MODE
    assert L.tp_row_linear_backward(FAKE, -1, ctypes.byref(rowv), FAKE, FAKE, FAKE, None) == SHAPE
    assert L.tp_row_linear_backward(FAKE, 8, ctypes.byref(rowv), None, FAKE, FAKE, None) == NULL
    assert L.tp_row_linear_backward(None, 8, ctypes.byref(rowv), FAKE, FAKE, FAKE, None) == NULL  # dW needs Xs
    assert L.tp_row_linear_backward(FAKE + 2, 8, ctypes.byref(rowv), FAKE, FAKE, FAKE, None) == ALIGN
    assert L.tp_row_linear_backward(FAKE, 0, ctypes.byref(rowv), FAKE, FAKE, FAKE, None) == OK
    # column layer
    assert L.tp_column_linear_backward(FAKE, 8, ctypes.byref(rowv), FAKE, None, FAKE, FAKE, None, 0, None) == MODE
    assert L.tp_column_linear_backward(FAKE, 8, ctypes.byref(colv), None, None, FAKE, FAKE, None, 0, None) == NULL
    assert L.tp_column_linear_backward(FAKE, 8, ctypes.byref(colv), FAKE, None, FAKE, FAKE, FAKE, 16, None) == WORKSPACE
    assert L.tp_column_linear_backward(FAKE, 0, ctypes.byref(colv), FAKE, None, FAKE, FAKE, None, 0, None) == OK
    # MLP block
    W1, W2 = view(K=128, N=256, mode=COL, dtype=BF16), view(K=256, N=128, mode=ROW, dtype=BF16)
    need = L.tp_mlp_backward_workspace_bytes(8, 128, 256, 2, 4, BF16)
    assert need > L.tp_mlp_backward_workspace_bytes(8, 128, 256, 2, 1, BF16) > 0
    assert L.tp_mlp_backward_workspace_bytes(8, 128, 256, 2, 4, F32) > 0
    assert L.tp_mlp_backward_workspace_bytes(8, 128, 256, 2, 4, 7) == 0
    args = lambda act, Wu, U, ws_bytes, T=8: (FAKE, T, ctypes.byref(W1), Wu, ctypes.byref(W2), act, FAKE, U, FAKE,
                                              FAKE, None, FAKE, ws_bytes, FAKE, FAKE, None, FAKE, None)
    assert L.tp_mlp_backward(*args(9, None, None, need)) == MODE
    assert L.tp_mlp_backward(*args(1, ctypes.byref(W1), None, need)) == MODE  # W_up without SwiGLU
    assert L.tp_mlp_backward(*args(4, None, FAKE, need)) == NULL               # SwiGLU needs W_up
    assert L.tp_mlp_backward(*args(4, ctypes.byref(W1), None, need)) == NULL  # and U
    assert L.tp_mlp_backward(*args(4, ctypes.byref(W1), FAKE, need - 1)) == WORKSPACE
    assert L.tp_mlp_backward(*args(4, ctypes.byref(W1), FAKE, need, T=0)) == OK
    W2f = view(K=256, N=128, mode=ROW, dtype=F32)   # an fp32 row layer under a bf16 column layer
    assert L.tp_mlp_backward(FAKE, 8, ctypes.byref(W1), None, ctypes.byref(W2f), 1, FAKE, None, FAKE, FAKE, None,
                             FAKE, need, FAKE, FAKE, None, FAKE, None) == DTYPE
    # the bf16 path keeps dG and dU token-major in 16-byte vectors: I/tp a
    # multiple of 8, and T * I/tp under 2^34
    def mlp_bwd(T, I):
        Wc, Wr = view(K=128, N=I, mode=COL, dtype=BF16), view(K=I, N=128, mode=ROW, dtype=BF16)
        ws = L.tp_mlp_backward_workspace_bytes(T, 128, I, 2, 4, BF16)
        return L.tp_mlp_backward(FAKE, T, ctypes.byref(Wc), ctypes.byref(Wc), ctypes.byref(Wr), 4, FAKE, FAKE,
                                 FAKE, FAKE, None, FAKE, ws, FAKE, FAKE, FAKE, FAKE, None)
    assert mlp_bwd(8, 260) == ALIGN              # I/tp = 130
    assert mlp_bwd((1 << 34) // 1024, 2048) == UNSUP  # T * I/tp = 2^34


def test_vocab_validation():
    L = tpl.lib
    assert L.tp_vocab_embedding(FAKE, 8, FAKE, 1000, 64, 3, BF16, FAKE, None) == SHAPE  # V % tp
    assert L.tp_vocab_embedding(FAKE, 8, FAKE, 1024, 64, 4, 7, FAKE, None) == DTYPE
    assert L.tp_vocab_embedding(None, 8, FAKE, 1024, 64, 4, BF16, FAKE, None) == NULL
    assert L.tp_vocab_embedding(FAKE + 1, 8, FAKE, 1024, 64, 4, BF16, FAKE, None) == ALIGN
    assert L.tp_vocab_embedding(FAKE, 0, FAKE, 1024, 64, 4, BF16, FAKE, None) == OK
    need = L.tp_cross_entropy_workspace_bytes(16, 32000, 4)
    assert need > 0
    ce = lambda T, V, tp, dt, ws_bytes, labels=FAKE: L.tp_vocab_cross_entropy(
        FAKE, labels, T, V, tp, dt, FAKE, None, None, ctypes.c_float(1.0), FAKE, ws_bytes, None)
    assert ce(16, 32001, 4, BF16, need) == SHAPE
    assert ce(16, 32000, 4, 9, need) == DTYPE
    assert ce(16, 32000, 4, BF16, need - 1) == WORKSPACE
    assert ce(16, 32000, 4, BF16, need, labels=None) == NULL
    assert ce(0, 32000, 4, BF16, need) == OK


def test_lm_head_cross_entropy_validation():
    """The fused LM head and loss: the column-linear checks, then labels,
    workspace and alignment, none of which reaches a launch."""
    L = tpl.lib
    W = view(K=256, N=4 * 512, tp=4, mode=COL, dtype=BF16)
    need = L.tp_lm_head_ce_workspace_bytes(300, ctypes.byref(W))
    assert need > L.tp_lm_head_ce_workspace_bytes(100, ctypes.byref(W)) > 0
    assert L.tp_lm_head_ce_workspace_bytes(300, None) == 0
    f = lambda T=300, w=W, labels=FAKE, logits=FAKE, ws=need, wsp=FAKE, dl=None: L.tp_lm_head_cross_entropy(
        FAKE, T, ctypes.byref(w), labels, logits, FAKE, None, dl, ctypes.c_float(1.0), wsp, ws, None)
    assert f(w=view(K=256, N=4 * 512, tp=4, mode=ROW, dtype=BF16)) == MODE   # a row view
    assert f(logits=None) == NULL
    assert f(labels=None) == NULL
    assert f(wsp=None) == NULL
    assert f(ws=need - 1) == WORKSPACE
    assert f(labels=FAKE + 2) == ALIGN
    assert f(dl=FAKE + 1) == ALIGN
    assert f(T=-1) == SHAPE
    assert f(T=0, labels=None, wsp=None, ws=0, logits=None) == OK


def test_moe_validation():
    L = tpl.lib
    Wg, Wd = view(K=128, N=256, mode=COL, dtype=BF16), view(K=256, N=128, mode=ROW, dtype=BF16)
    need = L.tp_moe_workspace_bytes(64, 128, 256, 2, 4, 2)
    assert need > L.tp_moe_workspace_bytes(64, 128, 256, 1, 4, 2) > 0
    moe = lambda T=64, k=2, E=4, g=Wg, d=Wd, ws=need, ids=FAKE: L.tp_moe_block(
        FAKE, T, ids, FAKE, k, E, ctypes.byref(g), ctypes.byref(g), ctypes.byref(d), None, FAKE, ws, FAKE, None)
    assert moe(g=view(K=128, N=256, mode=COL, dtype=F32), d=view(K=256, N=128, mode=ROW, dtype=F32)) == DTYPE
    assert moe(d=view(K=256, N=256, mode=ROW, dtype=BF16)) == SHAPE  # down does not match gate/up
    assert moe(E=0) == SHAPE
    assert moe(k=0) == SHAPE
    assert moe(E=2000) == SHAPE
    assert moe(ws=need - 1) == WORKSPACE
    assert moe(ids=None) == NULL
    assert moe(T=0) == OK


def test_attention_validation():
    """The attention core's checks, in the order the entry point runs them,
    none of which reaches a launch."""
    L = tpl.lib
    att = lambda qkv=FAKE, T=8, tp=2, hq=4, hkv=2, hd=128, mode=1, ctx=FAKE: L.tp_attention(
        qkv, T, tp, hq, hkv, hd, mode, ctx, None)
    assert att(qkv=None) == NULL
    assert att(ctx=None) == NULL
    assert att(mode=0) == MODE        # the single-key stand-in is not a core mode
    assert att(mode=3) == MODE
    assert att(hq=3) == SHAPE         # 3 q heads over 2 shards
    assert att(T=-1) == SHAPE
    assert att(hd=96, hq=4, hkv=2) == UNSUP   # head sizes 64 and 128 only
    assert att(hd=256, hq=4, hkv=2) == UNSUP
    assert att(T=2 ** 31) == UNSUP
    # query tiles (shard, q head, block of 128 queries) past the kernel's int range
    assert att(T=2 ** 31 - 1, tp=64, hq=64, hkv=64) == UNSUP
    assert att(qkv=FAKE + 1) == ALIGN
    assert att(T=0) == OK
    assert att(T=0, qkv=None, ctx=None) == OK


def test_binding_refuses_host_tensors():
    """The binding hands the library device pointers only: a host tensor is
    refused before any call into it."""
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        tpl._ptr(torch.zeros(4))
    assert tpl._ptr(None) is None
    with pytest.raises(ValueError):
        tpl.tp_attention(torch.zeros((2, 8, 512), dtype=torch.bfloat16), 4, 2, 128)
    with pytest.raises(ValueError):
        tpl.tp_rmsnorm(torch.zeros((4, 64), dtype=torch.bfloat16))
