"""Python binding of the tensor-parallel sharded linear library (libtp_b300.so).

Argument marshalling only: torch tensors supply device memory and the
current CUDA stream; each function passes pointers and sizes to the C entry
point of the same name (declared in include/tp.h) and raises TpError on a
non-zero status. Every step of the computation runs in the library's CUDA
kernels. There is no CPU fallback: importing this package fails if the
library has not been built, and the kernels need a CUDA device.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "TpError", "Shards", "lib", "LIB_PATH",
    "TP_F32", "TP_BF16", "TP_COL", "TP_ROW", "ACTS", "REDUCE_OPS",
    "tp_shard_weights", "tp_shard_qkv", "tp_qkv_shard_elems", "tp_column_linear",
    "tp_row_linear", "tp_row_linear_partials", "tp_gemm_workspace_bytes", "tp_shard_reduce", "tp_shard_gather",
    "tp_mlp_workspace_bytes", "tp_mlp_block", "tp_mlp_block_static", "tp_attn_workspace_bytes",
    "tp_attn_proj", "tp_attn_block", "tp_attention", "ATTN_MODES", "TP_STATIC_WORKSPACE_BYTES",
    "tp_rmsnorm", "tp_get_error", "tp_debug_set_wait_limit_ns", "tp_debug_inject",
    "tp_status_string", "tp_row_linear_backward", "tp_column_linear_backward",
    "tp_mlp_backward_workspace_bytes", "tp_mlp_backward", "tp_vocab_embedding",
    "tp_cross_entropy_workspace_bytes", "tp_vocab_cross_entropy", "tp_shard_experts",
    "tp_moe_workspace_bytes", "tp_moe_block",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtp_b300.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python tensor_transformer_linear_tma_b300/build.py`")
lib = ctypes.CDLL(LIB_PATH)

TP_F32, TP_BF16 = 0, 1
TP_COL, TP_ROW = 0, 1
ACTS = {"none": 0, "relu": 1, "gelu": 2, "silu": 3, "swiglu": 4}
REDUCE_OPS = {"sum": 0, "scatter": 1}
ATTN_MODES = {"single_key": 0, "causal": 1, "full": 2}

_vp, _i64, _i32, _sz, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_float


class TpShardsC(ctypes.Structure):
    _fields_ = [("data", _vp), ("K", _i64), ("N", _i64), ("tp", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("dtype", ctypes.c_int32), ("hq", ctypes.c_int32),
                ("hkv", ctypes.c_int32), ("hd", ctypes.c_int32)]


_P = ctypes.POINTER(TpShardsC)
_SIGS = {
    "tp_status_string": (ctypes.c_char_p, [_i32]),
    "tp_abi_version": (_i32, []),
    "tp_shard_weights": (_i32, [_vp, _i64, _i64, _i32, _i32, _i32, _vp, _sz, _P, _vp]),
    "tp_shard_qkv": (_i32, [_vp, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _P, _vp]),
    "tp_qkv_shard_elems": (_sz, [_i64, _i32, _i32, _i32, _i32]),
    "tp_column_linear": (_i32, [_vp, _i64, _P, _P, _vp, _vp, _i32, _i32, _vp, _vp, _sz, _vp]),
    "tp_row_linear": (_i32, [_vp, _i64, _P, _vp, _vp, _vp, _i32, _vp, _sz, _vp]),
    "tp_gemm_workspace_bytes": (_sz, [_i64, _P]),
    "tp_row_linear_partials": (_i32, [_vp, _i64, _P, _vp, _vp]),
    "tp_shard_reduce": (_i32, [_vp, _i32, _i64, _i64, _i32, _vp, _vp, _i32, _vp, _vp]),
    "tp_shard_gather": (_i32, [_vp, _i32, _i64, _i64, _i32, _vp, _vp]),
    "tp_mlp_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32, _i32]),
    "tp_mlp_block": (_i32, [_vp, _i64, _P, _P, _P, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _sz, _vp, _vp]),
    "tp_mlp_block_static": (_i32, [_vp, _i64, _P, _P, _P, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp]),
    "tp_attn_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32, _i32, _i32]),
    "tp_attn_proj": (_i32, [_vp, _i64, _P, _P, _vp, _vp, _i32, _vp, _vp, _sz, _vp, _vp]),
    "tp_attn_block": (_i32, [_vp, _i64, _P, _P, _i32, _vp, _i32, _vp, _vp, _sz, _vp, _vp]),
    "tp_attention": (_i32, [_vp, _i64, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "tp_rmsnorm": (_i32, [_vp, _vp, _i64, _i64, _f32, _i32, _vp, _i32, _vp]),
    "tp_get_error": (_i32, [_vp]),
    "tp_last_cuda_error": (_i32, []),
    "tp_cuda_error_name": (ctypes.c_char_p, [_i32]),
    "tp_row_linear_backward": (_i32, [_vp, _i64, _P, _vp, _vp, _vp, _vp]),
    "tp_column_linear_backward": (_i32, [_vp, _i64, _P, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tp_mlp_backward_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32, _i32, _i32]),
    "tp_mlp_backward": (_i32, [_vp, _i64, _P, _P, _P, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                               _vp, _vp, _vp, _vp, _vp]),
    "tp_vocab_embedding": (_i32, [_vp, _i64, _vp, _i64, _i64, _i32, _i32, _vp, _vp]),
    "tp_cross_entropy_workspace_bytes": (_sz, [_i64, _i64, _i32]),
    "tp_vocab_cross_entropy": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _f32, _vp, _sz, _vp]),
    "tp_lm_head_ce_workspace_bytes": (_sz, [_i64, _P]),
    "tp_lm_head_cross_entropy": (_i32, [_vp, _i64, _P, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _sz, _vp]),
    "tp_moe_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32, _i32, _i32]),
    "tp_moe_block": (_i32, [_vp, _i64, _vp, _vp, _i32, _i32, _P, _P, _P, _vp, _vp, _sz, _vp, _vp]),
    "tp_debug_set_wait_limit_ns": (_i32, [ctypes.c_uint64]),
    "tp_debug_inject": (_i32, [_i32]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype, _f.argtypes = _res, _args


class TpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn}: status {status} ({tp_status_string(status)})"
        if status == 7:  # TP_ERR_CUDA: name the failing CUDA call's code
            code = lib.tp_last_cuda_error()
            msg += f": CUDA code {code} ({lib.tp_cuda_error_name(code).decode()})"
        super().__init__(msg)


def tp_status_string(status: int) -> str:
    return lib.tp_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise TpError(fn, status)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return TP_BF16
    if t.dtype == torch.float32:
        return TP_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _torch_dt(code: int):
    return torch.bfloat16 if code == TP_BF16 else torch.float32


def _out_dtype(default, out=None, residual=None, out_dtype=None):
    """Output dtype: explicit, else that of `out`, else of `residual`, else `default`."""
    if out_dtype is not None:
        return out_dtype
    if out is not None:
        return out.dtype
    if residual is not None:
        return residual.dtype
    return default


def _ptr(t):
    """Device address of a tensor. The library takes pointers into the
    current CUDA device's memory and launches on that device, so a host
    tensor, or one on another device, is refused here rather than handed to
    a kernel."""
    if t is None:
        return None
    if t.device.type != "cuda":
        raise ValueError(f"tensors must be in CUDA device memory (got one on {t.device})")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensors must be on the current CUDA device "
                         f"(cuda:{torch.cuda.current_device()}), got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(device=None):
    if not torch.cuda.is_available():
        return None
    return torch.cuda.current_stream(device).cuda_stream


class Shards:
    """Sharded weights: the storage tensor plus its C view (tp_shards)."""

    def __init__(self, storage: torch.Tensor, view: TpShardsC):
        self.storage = storage
        self.view = view

    @property
    def tp(self):
        return self.view.tp

    @property
    def K(self):
        return self.view.K

    @property
    def N(self):
        return self.view.N

    @property
    def shard_width(self):
        """Output columns per shard (column mode) or N (row mode)."""
        return self.view.N // self.view.tp if self.view.mode == TP_COL else self.view.N

    def ref(self):
        return ctypes.byref(self.view)


def tp_shard_weights(W: torch.Tensor, tp: int, mode: str) -> Shards:
    """Shard W [K, N] (in, out) into tp column ("col") or row ("row") shards."""
    K, N = W.shape
    m = TP_COL if mode == "col" else TP_ROW
    out = torch.empty(K * N, dtype=W.dtype, device=W.device)
    view = TpShardsC()
    _check("tp_shard_weights", lib.tp_shard_weights(
        _ptr(W), K, N, _dt(W), tp, m, _ptr(out), out.numel() * out.element_size(),
        ctypes.byref(view), _stream(W.device)))
    return Shards(out, view)


def tp_qkv_shard_elems(H: int, hq: int, hkv: int, hd: int, tp: int) -> int:
    return lib.tp_qkv_shard_elems(H, hq, hkv, hd, tp)


def tp_shard_qkv(Wq, Wk, Wv, hq: int, hkv: int, hd: int, tp: int) -> Shards:
    H = Wq.shape[0]
    n = tp_qkv_shard_elems(H, hq, hkv, hd, tp)
    out = torch.empty(max(n, 1), dtype=Wq.dtype, device=Wq.device)
    view = TpShardsC()
    _check("tp_shard_qkv", lib.tp_shard_qkv(
        _ptr(Wq), _ptr(Wk), _ptr(Wv), H, hq, hkv, hd, tp, _dt(Wq), _ptr(out),
        out.numel() * out.element_size(), ctypes.byref(view), _stream(Wq.device)))
    return Shards(out, view)


def tp_gemm_workspace_bytes(T: int, W: Shards) -> int:
    return lib.tp_gemm_workspace_bytes(T, W.ref())


def _ws_args(workspace):
    if workspace is None:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def tp_column_linear(X, W: Shards, W_up: Shards | None = None, bias=None, bias_up=None,
                     act: str = "none", concat: bool = False, out=None, workspace=None):
    """Column-parallel linear; returns [tp, T, N/tp] or, with concat, [T, N].
    `workspace` (optional, tp_gemm_workspace_bytes) enables the balanced schedule."""
    T = X.shape[0]
    Ns = W.shard_width
    if out is None:
        shape = (T, W.N) if concat else (W.tp, T, Ns)
        out = torch.empty(shape, dtype=X.dtype, device=X.device)
    ws, wsb = _ws_args(workspace)
    _check("tp_column_linear", lib.tp_column_linear(
        _ptr(X), T, W.ref(), W_up.ref() if W_up is not None else None, _ptr(bias), _ptr(bias_up),
        ACTS[act], int(concat), _ptr(out), ws, wsb, _stream(X.device)))
    return out


def tp_row_linear(Xs, W: Shards, bias=None, residual=None, out=None, workspace=None, out_dtype=None):
    """Row-parallel linear with the shard sum fused; Xs is [tp, T, K/tp].
    bias, residual and the output share out_dtype (default Xs.dtype)."""
    T = Xs.shape[1]
    odt = _out_dtype(Xs.dtype, out, residual, out_dtype)
    if out is None:
        out = torch.empty((T, W.N), dtype=odt, device=Xs.device)
    ws, wsb = _ws_args(workspace)
    _check("tp_row_linear", lib.tp_row_linear(
        _ptr(Xs), T, W.ref(), _ptr(bias), _ptr(residual), _ptr(out), _dt(out), ws, wsb,
        _stream(Xs.device)))
    return out


def tp_row_linear_partials(Xs, W: Shards, out=None):
    """Per-shard fp32 contributions [tp, T, N]."""
    T = Xs.shape[1]
    if out is None:
        out = torch.empty((W.tp, T, W.N), dtype=torch.float32, device=Xs.device)
    _check("tp_row_linear_partials", lib.tp_row_linear_partials(
        _ptr(Xs), T, W.ref(), _ptr(out), _stream(Xs.device)))
    return out


def tp_shard_reduce(partials, op: str = "sum", bias=None, residual=None, out_dtype=None, out=None):
    """Sum [tp, T, N] fp32 partials; "scatter" returns the [tp, T/tp, N] view."""
    tp, T, N = partials.shape
    odt = out_dtype if out_dtype is not None else (out.dtype if out is not None else torch.float32)
    if out is None:
        out = torch.empty((T, N), dtype=odt, device=partials.device)
    _check("tp_shard_reduce", lib.tp_shard_reduce(
        _ptr(partials), tp, T, N, REDUCE_OPS[op], _ptr(bias), _ptr(residual),
        TP_BF16 if odt == torch.bfloat16 else TP_F32, _ptr(out), _stream(partials.device)))
    return out.view(tp, T // tp, N) if op == "scatter" else out


def tp_shard_gather(shards, out=None):
    """Concatenate [tp, T, N/tp] shards into [T, N]."""
    tp, T, Ns = shards.shape
    if out is None:
        out = torch.empty((T, tp * Ns), dtype=shards.dtype, device=shards.device)
    _check("tp_shard_gather", lib.tp_shard_gather(
        _ptr(shards), tp, T, tp * Ns, _dt(shards), _ptr(out), _stream(shards.device)))
    return out


def tp_mlp_workspace_bytes(T: int, H: int, I: int, tp: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (TP_BF16 if dtype == torch.bfloat16 else TP_F32)
    return lib.tp_mlp_workspace_bytes(T, H, I, tp, code)


def _workspace(nbytes: int, device):
    # 256-byte aligned by the caching allocator; at least one element
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def tp_mlp_block(X, W1: Shards, W2: Shards, W_up: Shards | None = None, b1=None, b1_up=None,
                 b2=None, residual=None, act: str = "relu", workspace=None, out=None, out_dtype=None):
    """column -> local activation -> row -> sum; returns Y [T, H] (b2, residual
    and Y in out_dtype, default X.dtype)."""
    T, H = X.shape
    need = tp_mlp_workspace_bytes(T, H, W1.N, W1.tp, _dt(X))
    if workspace is None:
        workspace = _workspace(need, X.device)
    odt = _out_dtype(X.dtype, out, residual, out_dtype)
    if out is None:
        out = torch.empty((T, W2.N), dtype=odt, device=X.device)
    _check("tp_mlp_block", lib.tp_mlp_block(
        _ptr(X), T, W1.ref(), W_up.ref() if W_up is not None else None, W2.ref(), _ptr(b1),
        _ptr(b1_up), _ptr(b2), _ptr(residual), ACTS[act], _dt(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _stream(X.device)))
    return out


def tp_row_linear_backward(Xs, W: Shards, dY, want_dX: bool = True, want_dW: bool = True):
    """Backward of Y = sum_s Xs[s] @ W_s: returns (dXs [tp][T][K/tp], dW
    [tp][N][K/tp] in W's storage layout); an output not wanted is None."""
    T = dY.shape[0]
    tp, Ks = W.tp, W.K // W.tp
    dXs = torch.empty((tp, T, Ks), dtype=dY.dtype, device=dY.device) if want_dX else None
    dW = torch.empty((tp, W.N, Ks), dtype=dY.dtype, device=dY.device) if want_dW else None
    _check("tp_row_linear_backward", lib.tp_row_linear_backward(
        _ptr(Xs), T, W.ref(), _ptr(dY), _ptr(dXs), _ptr(dW), _stream(dY.device)))
    return dXs, dW


def tp_column_linear_backward(X, W: Shards, dYs, dR=None, want_dX: bool = True, want_dW: bool = True,
                              workspace=None):
    """Backward of Y_s = X @ W_s: returns (dX [T][K] = sum_s dYs[s] @ W_s^T (+ dR),
    dW [tp][N/tp][K] in W's storage layout); an output not wanted is None."""
    T = dYs.shape[1]
    dX = torch.empty((T, W.K), dtype=dYs.dtype, device=dYs.device) if want_dX else None
    dW = torch.empty((W.tp, W.N // W.tp, W.K), dtype=dYs.dtype, device=dYs.device) if want_dW else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("tp_column_linear_backward", lib.tp_column_linear_backward(
        _ptr(X), T, W.ref(), _ptr(dYs), _ptr(dR), _ptr(dX), _ptr(dW), _ptr(workspace), ws_bytes,
        _stream(dYs.device)))
    return dX, dW


def tp_mlp_backward_workspace_bytes(T: int, H: int, I: int, tp: int, act: str = "swiglu",
                                    dtype=torch.bfloat16) -> int:
    return lib.tp_mlp_backward_workspace_bytes(T, H, I, tp, ACTS[act], TP_F32 if dtype == torch.float32 else TP_BF16)


def tp_mlp_backward(X, W1: Shards, W2: Shards, G, Hs, dY, W_up: Shards | None = None, U=None, dR=None,
                    act: str = "relu", workspace=None, want=("dX", "dW1", "dW_up", "dW2"), out=None):
    """Backward of tp_mlp_block (no biases) given the saved forward values G
    (pre-activation), U (up projection, SwiGLU) and Hs (activation output),
    each [tp][T][I/tp]. Returns a dict with dX [T][H], dW1 and dW_up
    [tp][I/tp][H], dW2 [tp][H][I/tp] (the shards' storage layouts); `out`
    may supply those tensors (a missing key is skipped)."""
    T, H = X.shape
    tp, Is = W1.tp, W1.N // W1.tp
    gated = act == "swiglu"
    need = tp_mlp_backward_workspace_bytes(T, H, W1.N, tp, act, X.dtype)
    if workspace is None:
        workspace = _workspace(need, X.device)
    if out is None:
        mk = lambda name, shape: torch.empty(shape, dtype=X.dtype, device=X.device) if name in want else None
        out = {"dX": mk("dX", (T, H)), "dW1": mk("dW1", (tp, Is, H)),
               "dW_up": mk("dW_up", (tp, Is, H)) if gated else None, "dW2": mk("dW2", (tp, H, Is))}
    else:
        out = {k: out.get(k) for k in ("dX", "dW1", "dW_up", "dW2")}
    _check("tp_mlp_backward", lib.tp_mlp_backward(
        _ptr(X), T, W1.ref(), W_up.ref() if W_up is not None else None, W2.ref(), ACTS[act], _ptr(G),
        _ptr(U), _ptr(Hs), _ptr(dY), _ptr(dR), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out["dX"]), _ptr(out["dW1"]), _ptr(out["dW_up"]), _ptr(out["dW2"]), _stream(X.device)))
    return out


def tp_vocab_embedding(ids, E, tp: int, out=None):
    """Y[t] = E[ids[t]] from the vocabulary-row shards of E [V][H] (ids int32)."""
    if ids.dtype != torch.int32:
        raise TypeError("ids must be int32")
    V, H = E.shape
    T = ids.numel()
    if out is None:
        out = torch.empty((T, H), dtype=E.dtype, device=E.device)
    _check("tp_vocab_embedding", lib.tp_vocab_embedding(
        _ptr(ids), T, _ptr(E), V, H, tp, _dt(E), _ptr(out), _stream(E.device)))
    return out


def tp_cross_entropy_workspace_bytes(T: int, V: int, tp: int) -> int:
    return lib.tp_cross_entropy_workspace_bytes(T, V, tp)


def tp_vocab_cross_entropy(logits, labels, want_loss: bool = True, want_mean: bool = True, dlogits=None,
                           grad_scale: float | None = None, workspace=None, loss=None, mean_loss=None):
    """Cross-entropy of vocabulary-sharded logits [tp][T][V/tp] with int32
    labels [T]. Returns (loss [T] fp32 or None, mean [1] fp32 or None); if
    `dlogits` is a tensor (it may be `logits` itself) it receives the
    gradient of grad_scale * sum(loss) (grad_scale defaults to 1/T)."""
    if labels.dtype != torch.int32:
        raise TypeError("labels must be int32")
    tp, T, v = logits.shape
    dev = logits.device
    if workspace is None:
        workspace = _workspace(tp_cross_entropy_workspace_bytes(T, tp * v, tp), dev)
    if loss is None and want_loss:
        loss = torch.empty(T, dtype=torch.float32, device=dev)
    if mean_loss is None and want_mean:
        mean_loss = torch.empty(1, dtype=torch.float32, device=dev)
    scale = (1.0 / max(T, 1)) if grad_scale is None else grad_scale
    _check("tp_vocab_cross_entropy", lib.tp_vocab_cross_entropy(
        _ptr(logits), _ptr(labels), T, tp * v, tp, _dt(logits), _ptr(loss), _ptr(mean_loss), _ptr(dlogits),
        scale, _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(dev)))
    return loss, mean_loss


def tp_lm_head_cross_entropy(X, W_lm: Shards, labels, logits=None, want_loss: bool = True,
                             want_mean: bool = True, dlogits=None, grad_scale: float | None = None,
                             workspace=None, loss=None, mean_loss=None):
    """LM head and vocabulary-parallel loss in one call: logits [tp][T][V/tp]
    (returned, or written into `logits`), losses [T] fp32, their mean [1]
    fp32, and, if `dlogits` is a tensor (it may be the logits), the gradient
    of grad_scale * sum(loss) (grad_scale defaults to 1/T). Returns
    (logits, loss, mean)."""
    if labels.dtype != torch.int32:
        raise TypeError("labels must be int32")
    T = X.shape[0]
    tp, V = W_lm.tp, W_lm.N
    dev = X.device
    if logits is None:
        logits = torch.empty((tp, T, V // tp), dtype=X.dtype, device=dev)
    if workspace is None:
        workspace = _workspace(lib.tp_lm_head_ce_workspace_bytes(T, W_lm.ref()), dev)
    if loss is None and want_loss:
        loss = torch.empty(T, dtype=torch.float32, device=dev)
    if mean_loss is None and want_mean:
        mean_loss = torch.empty(1, dtype=torch.float32, device=dev)
    scale = (1.0 / max(T, 1)) if grad_scale is None else grad_scale
    _check("tp_lm_head_cross_entropy", lib.tp_lm_head_cross_entropy(
        _ptr(X), T, W_lm.ref(), _ptr(labels), _ptr(logits), _ptr(loss), _ptr(mean_loss), _ptr(dlogits), scale,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(dev)))
    return logits, loss, mean_loss


def tp_shard_experts(Ws, tp: int, mode: str) -> Shards:
    """Shard each expert's W [K, N] like tp_shard_weights and store the E
    shard sets one after another; the view describes one expert."""
    K, N = Ws[0].shape
    m = TP_COL if mode == "col" else TP_ROW
    out = torch.empty(len(Ws) * K * N, dtype=Ws[0].dtype, device=Ws[0].device)
    view = TpShardsC()
    per = K * N * out.element_size()
    for e, W in enumerate(Ws):
        if tuple(W.shape) != (K, N):
            raise ValueError("experts must share one shape")
        _check("tp_shard_weights", lib.tp_shard_weights(
            _ptr(W), K, N, _dt(W), tp, m, out.data_ptr() + e * per, per, ctypes.byref(view), _stream(W.device)))
    view.data = out.data_ptr()
    return Shards(out, view)


def tp_moe_workspace_bytes(T: int, H: int, I: int, k: int, E: int, tp: int) -> int:
    return lib.tp_moe_workspace_bytes(T, H, I, k, E, tp)


def tp_moe_block(X, ids, weights, Wg: Shards, Wu: Shards, Wd: Shards, E: int, residual=None, workspace=None,
                 out=None):
    """Mixture of TP-sharded SwiGLU experts: ids [T, k] int32, weights [T, k]
    fp32; returns Y [T, H] (bf16)."""
    if ids.dtype != torch.int32 or weights.dtype != torch.float32:
        raise TypeError("ids must be int32 and weights fp32")
    T, H = X.shape
    k = ids.shape[1]
    need = tp_moe_workspace_bytes(T, H, Wg.N, k, E, Wg.tp)
    if workspace is None:
        workspace = _workspace(need, X.device)
    if out is None:
        out = torch.empty((T, H), dtype=X.dtype, device=X.device)
    _check("tp_moe_block", lib.tp_moe_block(
        _ptr(X), T, _ptr(ids), _ptr(weights), k, E, Wg.ref(), Wu.ref(), Wd.ref(), _ptr(residual),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _stream(X.device)))
    return out


TP_STATIC_WORKSPACE_BYTES = 32 << 20


def tp_mlp_block_static(X, W1: Shards, W2: Shards, W_up: Shards | None = None, b1=None, b1_up=None,
                        b2=None, residual=None, act: str = "relu", out=None, out_dtype=None):
    """tp_mlp_block with the library's static device workspace (no caller
    workspace; sizes beyond TP_STATIC_WORKSPACE_BYTES are refused)."""
    T = X.shape[0]
    odt = _out_dtype(X.dtype, out, residual, out_dtype)
    if out is None:
        out = torch.empty((T, W2.N), dtype=odt, device=X.device)
    _check("tp_mlp_block_static", lib.tp_mlp_block_static(
        _ptr(X), T, W1.ref(), W_up.ref() if W_up is not None else None, W2.ref(), _ptr(b1),
        _ptr(b1_up), _ptr(b2), _ptr(residual), ACTS[act], _dt(out), _ptr(out), _stream(X.device)))
    return out


def tp_attn_workspace_bytes(T: int, hq: int, hkv: int, hd: int, tp: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (TP_BF16 if dtype == torch.bfloat16 else TP_F32)
    return lib.tp_attn_workspace_bytes(T, hq, hkv, hd, tp, code)


def tp_attn_proj(X, Wqkv: Shards, Wo: Shards, ctx=None, residual=None, qkv_out=None,
                 workspace=None, out=None, out_dtype=None):
    """QKV by heads -> local heads (ctx, or the single-key stand-in) -> O + sum.
    residual and the output share out_dtype (default X.dtype)."""
    T = X.shape[0]
    v = Wqkv.view
    need = tp_attn_workspace_bytes(T, v.hq, v.hkv, v.hd, v.tp, _dt(X))
    if workspace is None:
        workspace = _workspace(need, X.device)
    odt = _out_dtype(X.dtype, out, residual, out_dtype)
    if out is None:
        out = torch.empty((T, Wo.N), dtype=odt, device=X.device)
    _check("tp_attn_proj", lib.tp_attn_proj(
        _ptr(X), T, Wqkv.ref(), Wo.ref(), _ptr(ctx), _ptr(residual), _dt(out), _ptr(qkv_out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _stream(X.device)))
    return out


def tp_attn_block(X, Wqkv: Shards, Wo: Shards, attention: str = "causal", residual=None, qkv_out=None,
                  workspace=None, out=None, out_dtype=None):
    """QKV by heads -> attention core ("causal", "full" or "single_key") -> O + sum."""
    T = X.shape[0]
    v = Wqkv.view
    need = tp_attn_workspace_bytes(T, v.hq, v.hkv, v.hd, v.tp, _dt(X))
    if workspace is None:
        workspace = _workspace(need, X.device)
    odt = _out_dtype(X.dtype, out, residual, out_dtype)
    if out is None:
        out = torch.empty((T, Wo.N), dtype=odt, device=X.device)
    _check("tp_attn_block", lib.tp_attn_block(
        _ptr(X), T, Wqkv.ref(), Wo.ref(), ATTN_MODES[attention], _ptr(residual), _dt(out), _ptr(qkv_out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _stream(X.device)))
    return out


def tp_attention(qkv, hq: int, hkv: int, hd: int, causal: bool = True, out=None):
    """Attention core of every local head: qkv [tp, T, (nq + 2 nkv) * hd] ->
    ctx [tp, T, nq * hd] (bf16, hd 64 or 128)."""
    tp, T, _ = qkv.shape
    if out is None:
        out = torch.empty((tp, T, hq // tp * hd), dtype=qkv.dtype, device=qkv.device)
    _check("tp_attention", lib.tp_attention(
        _ptr(qkv), T, tp, hq, hkv, hd, ATTN_MODES["causal" if causal else "full"], _ptr(out),
        _stream(qkv.device)))
    return out


def tp_rmsnorm(X, gamma=None, eps: float = 1e-5, out=None, out_dtype=None):
    """RMSNorm over the hidden; the output dtype may differ from X's."""
    T, H = X.shape
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype or X.dtype, device=X.device)
    _check("tp_rmsnorm", lib.tp_rmsnorm(
        _ptr(X), _ptr(gamma), T, H, eps, _dt(X), _ptr(out), _dt(out), _stream(X.device)))
    return out


def tp_get_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status."""
    return lib.tp_get_error(_stream(device))


def tp_debug_set_wait_limit_ns(ns: int) -> None:
    _check("tp_debug_set_wait_limit_ns", lib.tp_debug_set_wait_limit_ns(ns))


def tp_debug_inject(kind: int) -> None:
    _check("tp_debug_inject", lib.tp_debug_inject(kind))
