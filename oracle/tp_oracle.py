"""Oracle for the tensor-parallel sharded linear pipeline (TEST INFRASTRUCTURE).

This is a plain, slow, CPU-only statement of what the pipeline computes. Only
the tests, the smoke check and the bench's CPU-baseline leg may import it; the
product path (the CUDA library and its Python binding) never does, and the
oracle imports nothing from the product.

Arithmetic: whatever numpy dtype the caller passes. The tests pass float64
(inputs are the bf16 / fp32 values the GPU sees, treated as exact reals; no
intermediate is re-rounded) or int64 for integer-valued inputs, where every
result is exact. A library matmul (``@``) is the only primitive used for a
product; there is no blocking, fusion or reordering beyond what each
definition states.

Pages cited (by title and section):
  [CTP]  "CUDA tensor parallel computations" learning notes (jokeuncle.github.io):
         sections "minimal math foundation" (the X=[10,20], 2x4 W example),
         "Column Parallel: split by output columns", "Row Parallel: split by
         input rows", "cross-GPU communication" (all-gather, all-reduce,
         reduce-scatter, broadcast), "local elementwise computation",
         "putting it into a Transformer" (QKV, heads, O projection, MLP),
         and the summary table.
  [TUT]  "Tensor parallelism: splitting Transformer layers" tutorial
         (freeguideonline.com): "column-wise sharding", "row-wise sharding",
         "MLP block sharding", "self-attention block sharding",
         "input and output layers", and the two-GPU PyTorch MLP sample.
  [WIT]  "What is tensor parallelism" (aiug.cn): basic principle (column and
         row parallel linear).
  [TRT]  "Parallel strategies in TensorRT LLM" (developer.aliyun.com):
         attention module, tensor parallel, GQA/MQA exception (KV replicated).

Readings where the pages are silent or ambiguous (each is listed with its
reason in the design notes of the repository):
  * W is [in, out] and Y = X @ W  ([TUT] sample, [CTP] example).
  * shard s is the s-th contiguous block; a dimension not divisible by tp is
    an error ([CTP] column/row sections; [TUT] sample uses integer division).
  * row-parallel bias is added once, after the sum.
  * GELU is the exact erf form; SiLU(x) = x / (1 + exp(-x)); SwiGLU applies
    SiLU to the gate and multiplies by the up projection.
  * reduce-scatter splits the summed result along tokens into tp equal slices.
  * KV heads are replicated when num_kv_heads < tp; q head h uses kv head
    floor(h / (hq / hkv)).
  * Between QKV and O, the default attention core is the single-key case:
    each query attends only to its own token, so the softmax weight is 1 and
    the context of q head h is V of its kv head. The full core is scaled
    dot-product attention of each local head, softmax(q k^T / sqrt(hd)) v,
    either causal (query t sees keys 0..t, the decoder reading) or
    unmasked.
  * RMSNorm: x * g / sqrt(mean(x^2) + eps), eps = 1e-5, statistics over the
    full (replicated) hidden.
  * Block wiring: x += O(ctx(QKV(norm(x)))); x += MLP(norm(x)); after the
    last block a final norm and the column-split LM head, gathered.
  * Backward of the column/row pair ([TUT] column-wise sharding, MLP block
    sharding and "forward and backward communication symmetry"): the
    pages state the pattern loosely and in part contradict each other
    (identity versus reduce-scatter for the row layer). The reading here
    is the chain rule of the forward as written: the all-reduce after the
    row layer hands the same dY to every shard (identity); each shard's
    row and activation gradients are local; each shard's column layer
    produces a partial input gradient dY_s W_s^T and the input gradient
    is their sum in shard order (an all-reduce, or a reduce-scatter when
    the caller wants it split along tokens). Weight gradients are local:
    dW_s = (layer input)^T (output gradient). The ReLU derivative at 0 is
    taken as 0.
  * Vocabulary-parallel input and output layers ([TUT] input and output
    layers; [WIT] loss computed sharded over the class dimension): the
    embedding table [V, H] is split by vocabulary rows, shard s holding
    rows [s*V/tp, (s+1)*V/tp); a lookup is each shard's masked lookup (a
    zero row for ids it does not own) summed over shards (all-reduce). The
    LM head is column-split over the vocabulary (column_parallel). The
    cross-entropy of vocabulary-sharded logits is the plain cross-entropy of
    the gathered logits, loss[t] = log sum_v exp(z[t, v]) - z[t, y[t]]: the
    pages name the sharded computation without its steps, and any correct
    sharded method reaches that value up to rounding.
  * Mixture of experts under TP ([TRT] FFN module, mixture of experts: the
    TP mode splits every expert's weights across all shards and every shard
    sees all tokens): each expert is an MLP block sharded as above (gate and
    up by columns, down by rows, shard sum); token t's output is
    sum_k w[t, k] * MLP_{e[t, k]}(x_t) for its top-k experts e[t, :] with
    weights w[t, :]. The router's choice is an input (synthetic routing):
    the pages describe the selection but not the router.

Parity pins: every function here is checked, without the GPU, against the
worked example's printed values, brute force on tiny integer inputs, closed
forms and library routines (see tests/test_oracle_pins.py). GELU and SiLU are
pinned to scipy's normal CDF and logistic function; beyond that the float
activations are "parity unpinned" against the pages, which print no values
for them.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "linear", "column_shards", "row_shards", "split_columns",
    "column_parallel", "all_gather", "row_parallel_partials", "all_reduce",
    "reduce_scatter", "relu", "gelu", "silu", "swiglu", "ACTIVATIONS",
    "mlp_block", "qkv_head_layout", "qkv_shards", "context_standin",
    "attention_weights", "attention_head", "context_attention", "attn_proj", "rmsnorm",
    "transformer_block", "stack_forward",
    "activation_backward", "column_linear_backward", "row_linear_backward",
    "mlp_backward_saved", "mlp_backward", "vocab_shards", "vocab_embedding", "log_softmax_normaliser",
    "cross_entropy", "cross_entropy_grad", "vocab_parallel_cross_entropy", "moe_tp",
]


# ---------------------------------------------------------------------------
# The linear layer and its two splits
# ---------------------------------------------------------------------------

def linear(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Y = X @ W; y[t, n] = sum_k x[t, k] * w[k, n].  [CTP] minimal math
    foundation: each output is a sum of products over the input dimension."""
    return X @ W


def _block(n: int, tp: int, what: str) -> int:
    if tp < 1 or n % tp != 0:
        raise ValueError(f"{what}={n} is not divisible by tp={tp}")
    return n // tp


def column_shards(W: np.ndarray, tp: int) -> list[np.ndarray]:
    """W[:, s*N/tp:(s+1)*N/tp] for s = 0..tp-1.  [CTP] Column Parallel: GPU 0
    holds the first block of output columns, GPU 1 the next; [TUT]
    column-wise sharding."""
    n = _block(W.shape[1], tp, "N")
    return [W[:, s * n:(s + 1) * n] for s in range(tp)]


def row_shards(W: np.ndarray, tp: int) -> list[np.ndarray]:
    """W[s*K/tp:(s+1)*K/tp, :] for s = 0..tp-1.  [CTP] Row Parallel: the rows
    of W (input dimension) are split; [TUT] row-wise sharding."""
    k = _block(W.shape[0], tp, "K")
    return [W[s * k:(s + 1) * k, :] for s in range(tp)]


def split_columns(X: np.ndarray, tp: int) -> list[np.ndarray]:
    """The input blocks matching row shards: X[:, s*K/tp:(s+1)*K/tp].
    [CTP] Row Parallel: X is split along with the rows of W."""
    k = _block(X.shape[1], tp, "K")
    return [X[:, s * k:(s + 1) * k] for s in range(tp)]


def column_parallel(X, W, tp, bias=None, act=None):
    """Per-shard outputs Y_s = act(X @ W_s + b_s), X replicated on every shard.
    [CTP] Column Parallel (each GPU computes X @ W_s) and local elementwise
    computation (activation and bias are applied shard-locally); the bias is
    split with its columns."""
    Ws = column_shards(W, tp)
    bs = column_shards(bias.reshape(1, -1), tp) if bias is not None else [None] * tp
    out = []
    for s in range(tp):
        y = linear(X, Ws[s])
        if bs[s] is not None:
            y = y + bs[s]
        if act is not None:
            y = act(y)
        out.append(y)
    return out


def all_gather(parts: list[np.ndarray]) -> np.ndarray:
    """Concatenate shard outputs along the last (column) dimension.
    [CTP] all-gather ("every GPU ends with [110, 140, 170, 200]") and the
    Column Parallel merge: concatenation, not addition; [TUT] sample
    torch.cat(dim=-1)."""
    return np.concatenate(parts, axis=-1)


def row_parallel_partials(Xs: list[np.ndarray], W: np.ndarray, tp: int) -> list[np.ndarray]:
    """P_s = X_s @ W_s: each shard's contribution to the full output.
    [CTP] Row Parallel ("GPU 0 computes a local contribution")."""
    Ws = row_shards(W, tp)
    if len(Xs) != tp:
        raise ValueError("need one input block per shard")
    return [linear(Xs[s], Ws[s]) for s in range(tp)]


def all_reduce(partials: list[np.ndarray]) -> np.ndarray:
    """Elementwise sum of the partials, taken in shard order s = 0..tp-1.
    [CTP] all-reduce ("add the subtotals into the total") and the Row
    Parallel merge: addition, not concatenation."""
    total = np.zeros_like(partials[0])
    for p in partials:
        total = total + p
    return total


def reduce_scatter(partials: list[np.ndarray], tp: int) -> list[np.ndarray]:
    """Sum the partials, then cut the total into tp slices; shard s keeps
    token rows [s*T/tp, (s+1)*T/tp).  [CTP] reduce-scatter ("sum first,
    then split the result, each GPU keeps the slice it needs"). The split
    axis (tokens) is a reading: the page does not name it."""
    total = all_reduce(partials)
    rows = _block(total.shape[0], tp, "T")
    return [total[s * rows:(s + 1) * rows] for s in range(tp)]


# ---------------------------------------------------------------------------
# Local elementwise operations ([CTP] local elementwise computation)
# ---------------------------------------------------------------------------

def relu(x):
    """max(0, x)."""
    return np.maximum(x, 0)


def gelu(x):
    """0.5 * x * (1 + erf(x / sqrt(2))): the exact GELU ([TUT] sample uses
    nn.GELU(), whose default is this erf form)."""
    erf = np.vectorize(math.erf, otypes=[np.float64])
    return 0.5 * x * (1.0 + erf(np.asarray(x, np.float64) / math.sqrt(2.0)))


def silu(x):
    """x / (1 + exp(-x))."""
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(-x))


def swiglu(g, u):
    """SwiGLU gate: silu(gate) * up.  [TUT] MLP block sharding: gate and up
    projections multiplied elementwise, then the down projection; [CTP]
    "multiply by a gate" is listed as a local elementwise op."""
    return silu(g) * u


ACTIVATIONS = {"none": None, "relu": relu, "gelu": gelu, "silu": silu}


# ---------------------------------------------------------------------------
# The MLP block: column -> local activation -> row -> sum
# ---------------------------------------------------------------------------

def mlp_block(X, W1, W2, tp, act="relu", W_up=None, b1=None, b1_up=None,
              b2=None, residual=None):
    """[CTP] "MLP: expand then contract, exactly Column + Row": the first
    layer is column-split, the activation is applied locally to each
    intermediate shard, the second layer is row-split on that same shard,
    and the partial results are summed (all-reduce). [TUT] MLP block
    sharding, steps 1-4. With act == "swiglu", W1 is the gate projection
    and W_up the up projection; both are column-split the same way.

    Returns (Hs, Y): the per-shard intermediate activations and the
    combined output Y = sum_s Hs[s] @ W2_s (+ b2, once) (+ residual).
    """
    if act == "swiglu":
        G = column_parallel(X, W1, tp, b1)
        U = column_parallel(X, W_up, tp, b1_up)
        Hs = [swiglu(G[s], U[s]) for s in range(tp)]
    else:
        Hs = column_parallel(X, W1, tp, b1, ACTIVATIONS[act])
    partials = row_parallel_partials(Hs, W2, tp)
    Y = all_reduce(partials)
    if b2 is not None:
        Y = Y + b2.reshape(1, -1)
    if residual is not None:
        Y = Y + residual
    return Hs, Y


# ---------------------------------------------------------------------------
# Attention projections: QKV column-split by heads, O row-split
# ---------------------------------------------------------------------------

def qkv_head_layout(hq: int, hkv: int, tp: int):
    """Heads held by each shard.  [CTP] QKV projection: each GPU takes a
    subset of the attention heads; [TUT] split by number of heads, whole
    heads per device; [TRT] GQA/MQA: when the KV heads cannot be split
    (fewer KV heads than tp) they are replicated.

    Returns a list over shards of (q_heads, kv_heads). q heads are split
    evenly. If hkv >= tp the kv heads are split evenly too; otherwise shard
    s holds the single kv head floor(s * hkv / tp), shared (replicated)
    with the other shards of its group.
    """
    if hq % tp != 0:
        raise ValueError("hq must be divisible by tp")
    if hq % hkv != 0:
        raise ValueError("hq must be a multiple of hkv")
    if hkv >= tp:
        if hkv % tp != 0:
            raise ValueError("hkv must be divisible by tp when hkv >= tp")
    elif tp % hkv != 0:
        raise ValueError("tp must be a multiple of hkv when hkv < tp")
    nq = hq // tp
    out = []
    for s in range(tp):
        q = list(range(s * nq, (s + 1) * nq))
        if hkv >= tp:
            nk = hkv // tp
            kv = list(range(s * nk, (s + 1) * nk))
        else:
            kv = [s * hkv // tp]
        out.append((q, kv))
    return out


def _head_cols(W, heads, hd):
    return np.concatenate([W[:, h * hd:(h + 1) * hd] for h in heads], axis=1)


def qkv_shards(Wq, Wk, Wv, hq, hkv, hd, tp):
    """Per-shard column weights [H, (nq + 2*nkv) * hd]: the shard's q head
    columns, then its k head columns, then its v head columns."""
    layout = qkv_head_layout(hq, hkv, tp)
    return [np.concatenate([_head_cols(Wq, q, hd), _head_cols(Wk, kv, hd),
                            _head_cols(Wv, kv, hd)], axis=1)
            for q, kv in layout]


def context_standin(qkv_s, q_heads, kv_heads, hq, hkv, hd):
    """Attention context of one shard under the single-key reading: each
    query attends only to its own token, the softmax over one score is 1,
    and the context of q head h is V of kv head floor(h / (hq / hkv)).
    [CTP] attention heads are local once Q/K/V of a head sit on one GPU.
    Returns [T, len(q_heads) * hd]."""
    nq, nkv = len(q_heads), len(kv_heads)
    v0 = (nq + nkv) * hd
    group = hq // hkv
    cols = []
    for h in q_heads:
        j = kv_heads.index(h // group)
        cols.append(qkv_s[:, v0 + j * hd:v0 + (j + 1) * hd])
    return np.concatenate(cols, axis=1)


def attention_weights(q, k, causal=True, q_offset=0):
    """The attention weights of one head, softmax(q k^T / sqrt(hd)) over the
    keys, with query t restricted to keys 0..t when causal (a key it may not
    see has weight 0). q is [Tq, hd] holding the queries at positions
    q_offset..q_offset+Tq-1; k is [T, hd]. Returns [Tq, T]."""
    Tq, hd = q.shape
    s = (q @ k.T) / math.sqrt(hd)
    if causal:
        pos = np.arange(Tq)[:, None] + q_offset
        s = np.where(np.arange(k.shape[0])[None, :] <= pos, s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return p / p.sum(axis=1, keepdims=True)


def attention_head(q, k, v, causal=True, q_offset=0):
    """Scaled dot-product attention of one head: the attention weights times
    v ([T, hd]). [CTP] attention heads (each GPU runs the attention of its
    own heads); [TUT] self-attention block sharding (heads are local between
    the QKV and output projections)."""
    return attention_weights(q, k, causal, q_offset) @ v


def context_attention(qkv_s, q_heads, kv_heads, hq, hkv, hd, causal=True):
    """Attention core of one shard: every local q head h attends with the
    K and V of kv head floor(h / (hq / hkv)), which the shard holds (a
    replica when hkv < tp). qkv_s is [T, (nq + 2*nkv) * hd] (q | k | v).
    Returns [T, len(q_heads) * hd]."""
    nq, nkv = len(q_heads), len(kv_heads)
    k0, v0 = nq * hd, (nq + nkv) * hd
    group = hq // hkv
    cols = []
    for i, h in enumerate(q_heads):
        j = kv_heads.index(h // group)
        cols.append(attention_head(qkv_s[:, i * hd:(i + 1) * hd],
                                   qkv_s[:, k0 + j * hd:k0 + (j + 1) * hd],
                                   qkv_s[:, v0 + j * hd:v0 + (j + 1) * hd], causal))
    return np.concatenate(cols, axis=1)


def attn_proj(X, Wq, Wk, Wv, Wo, hq, hkv, hd, tp, ctx=None, residual=None, attention=None):
    """[CTP] QKV projection (column parallel by heads), local attention
    heads, output projection (row parallel, then all-reduce); [TUT]
    self-attention block sharding.

    ctx, if given, is the per-shard attention output [tp][T, hq/tp*hd];
    otherwise attention = "causal" or "full" runs the attention core of each
    shard's heads, and None the single-key stand-in. Returns
    (qkv per shard, ctx per shard, Y)."""
    layout = qkv_head_layout(hq, hkv, tp)
    Wqkv = qkv_shards(Wq, Wk, Wv, hq, hkv, hd, tp)
    qkv = [linear(X, Wqkv[s]) for s in range(tp)]
    if ctx is None and attention is not None:
        if attention not in ("causal", "full"):
            raise ValueError("attention must be 'causal', 'full' or None")
        ctx = [context_attention(qkv[s], layout[s][0], layout[s][1], hq, hkv, hd, attention == "causal")
               for s in range(tp)]
    if ctx is None:
        ctx = [context_standin(qkv[s], layout[s][0], layout[s][1], hq, hkv, hd)
               for s in range(tp)]
    partials = row_parallel_partials(ctx, Wo, tp)
    Y = all_reduce(partials)
    if residual is not None:
        Y = Y + residual
    return qkv, ctx, Y


# ---------------------------------------------------------------------------
# Norm and the block stack
# ---------------------------------------------------------------------------

def rmsnorm(x, gamma=None, eps=1e-5):
    """y = x * g / sqrt(mean over hidden of x^2 + eps). [CTP] local
    elementwise computation: a norm needs statistics over the hidden
    dimension and is local when run on the replicated hidden."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    y = x / np.sqrt(ms + eps)
    if gamma is not None:
        y = y * gamma
    return y


def transformer_block(x, L, tp, hq, hkv, hd, eps=1e-5):
    """Pre-norm block: x + O(ctx(QKV(norm(x)))), then + MLP(norm(x)).
    Weights L: Wq, Wk, Wv, Wo, Wg, Wu, Wd."""
    h = rmsnorm(x, None, eps)
    _, _, x = attn_proj(h, L["Wq"], L["Wk"], L["Wv"], L["Wo"], hq, hkv, hd, tp,
                        residual=x)
    h = rmsnorm(x, None, eps)
    _, x = mlp_block(h, L["Wg"], L["Wd"], tp, "swiglu", W_up=L["Wu"], residual=x)
    return x


def stack_forward(X, layers, W_lm, tp, hq, hkv, hd, eps=1e-5):
    """Blocks in order, a final norm, then the LM head column-split over
    the vocabulary and gathered ([TUT] input and output layers: the output
    projection is split by columns and the logits gathered)."""
    x = np.asarray(X, np.float64)
    for L in layers:
        x = transformer_block(x, L, tp, hq, hkv, hd, eps)
    h = rmsnorm(x, None, eps)
    return all_gather(column_parallel(h, W_lm, tp))


# ---------------------------------------------------------------------------
# Backward of the column/row pair
# ---------------------------------------------------------------------------

def activation_backward(act, G, dH, U=None):
    """Gradient through the local activation ([CTP] local elementwise
    computation; [TUT] MLP block sharding, step 2): given dL/dH for
    H = act(G), or H = silu(G) * U for SwiGLU, return (dL/dG, dL/dU), the
    second None except for SwiGLU. Derivatives written out:
    relu'(g) = [g > 0]; gelu'(g) = Phi(g) + g phi(g) with Phi the normal CDF
    and phi its density; silu'(g) = s (1 + g (1 - s)), s = 1 / (1 + e^-g)."""
    G = np.asarray(G)
    if act == "none":
        return dH, None
    if act == "relu":
        return dH * (G > 0), None
    if act == "gelu":
        erf = np.vectorize(math.erf, otypes=[np.float64])
        g = np.asarray(G, np.float64)
        Phi = 0.5 * (1.0 + erf(g / math.sqrt(2.0)))
        phi = np.exp(-0.5 * g * g) / math.sqrt(2.0 * math.pi)
        return dH * (Phi + g * phi), None
    g = np.asarray(G, np.float64)
    sg = 1.0 / (1.0 + np.exp(-g))
    dsilu = sg * (1.0 + g * (1.0 - sg))
    if act == "silu":
        return dH * dsilu, None
    if act == "swiglu":
        if U is None:
            raise ValueError("swiglu needs the up projection U")
        return dH * U * dsilu, dH * g * sg
    raise ValueError(f"unknown activation {act}")


def column_linear_backward(X, W, tp, dYs, dR=None):
    """Backward of the column-parallel layer Y_s = X @ W_s (X replicated on
    every shard). [TUT] column-wise sharding: X is a copy on each device,
    so each shard's input gradient dY_s @ W_s^T is only its share; the input
    gradient is their sum in shard order (all_reduce), plus the gradient
    dR reaching X by any other path (a residual branch). The weight
    gradient of shard s is local: X^T @ dY_s.
    Returns (dX, [dW_s])."""
    Ws = column_shards(W, tp)
    if len(dYs) != tp:
        raise ValueError("need one output gradient per shard")
    dX = all_reduce([dYs[s] @ Ws[s].T for s in range(tp)])
    if dR is not None:
        dX = dX + dR
    return dX, [X.T @ dYs[s] for s in range(tp)]


def row_linear_backward(Xs, W, tp, dY):
    """Backward of the row-parallel layer Y = sum_s X_s @ W_s. [TUT]
    communication symmetry: the forward all-reduce is an identity in the
    backward, so every shard receives the same dY; then dX_s = dY @ W_s^T
    and dW_s = X_s^T @ dY, both local. Returns ([dX_s], [dW_s])."""
    Ws = row_shards(W, tp)
    if len(Xs) != tp:
        raise ValueError("need one input block per shard")
    return [dY @ Ws[s].T for s in range(tp)], [Xs[s].T @ dY for s in range(tp)]


def mlp_backward_saved(X, W1, W2, tp, dY, G, Hs, act="relu", W_up=None, U=None, dR=None):
    """Backward of mlp_block (no biases) given the forward's saved per-shard
    values, as a training step runs it: G[s] the pre-activation X @ W1_s,
    U[s] the up projection X @ Wu_s (SwiGLU only), Hs[s] the activation
    output that fed W2. The forward steps in reverse ([TUT] MLP block
    sharding, steps 4 to 1):
      row layer:   dHs_s = dY @ W2_s^T, dW2_s = Hs_s^T @ dY (dY on every shard)
      activation:  dG_s, dU_s from dHs_s, G_s, U_s
      column layer(s): dX = sum_s dG_s @ W1_s^T (+ sum_s dU_s @ Wu_s^T) (+ dR),
                   dW1_s = X^T @ dG_s, dWu_s = X^T @ dU_s
    Returns a dict: dX [T, H]; dW1, dW_up (SwiGLU) lists over shards of
    [H, I/tp]; dW2 a list of [I/tp, H]; dHs, dG, dU per shard."""
    gated = act == "swiglu"
    U = U if gated else [None] * tp
    dHs, dW2 = row_linear_backward(Hs, W2, tp, dY)
    grads = [activation_backward(act, G[s], dHs[s], U[s]) for s in range(tp)]
    dG = [g for g, _ in grads]
    dU = [u for _, u in grads]
    dX, dW1 = column_linear_backward(X, W1, tp, dG, dR)
    dWu = None
    if gated:
        dX2, dWu = column_linear_backward(X, W_up, tp, dU)
        dX = dX + dX2
    return {"dX": dX, "dW1": dW1, "dW_up": dWu, "dW2": dW2, "dHs": dHs, "dG": dG, "dU": dU}


def mlp_backward(X, W1, W2, tp, dY, act="relu", W_up=None, dR=None):
    """Backward of mlp_block (no biases) for the output gradient dY: the
    forward recomputed in full precision (G, U, Hs per shard), then
    mlp_backward_saved. Returns its dict plus G, U and Hs."""
    gated = act == "swiglu"
    G = column_parallel(X, W1, tp)
    U = column_parallel(X, W_up, tp) if gated else [None] * tp
    if gated:
        Hs = [swiglu(G[s], U[s]) for s in range(tp)]
    else:
        f = ACTIVATIONS[act]
        Hs = [G[s] if f is None else f(G[s]) for s in range(tp)]
    out = mlp_backward_saved(X, W1, W2, tp, dY, G, Hs, act, W_up=W_up, U=U, dR=dR)
    out.update(G=G, U=U, Hs=Hs)
    return out


# ---------------------------------------------------------------------------
# Vocabulary-parallel input and output layers
# ---------------------------------------------------------------------------

def vocab_shards(E: np.ndarray, tp: int) -> list[np.ndarray]:
    """Row blocks of the embedding table E [V, H]: shard s holds the vectors
    of ids s*V/tp .. (s+1)*V/tp - 1. [TUT] input and output layers: the
    embedding is split along the vocabulary dimension."""
    v = _block(E.shape[0], tp, "V")
    return [E[s * v:(s + 1) * v] for s in range(tp)]


def vocab_embedding(ids, E, tp):
    """Embedding lookup from vocabulary shards: each shard returns the rows
    of the ids it holds and zero rows for the others; the shard results are
    summed (all_reduce). [TUT] input and output layers (each device keeps
    part of the embedding vectors, then all-reduce)."""
    ids = np.asarray(ids)
    shards = vocab_shards(E, tp)
    v = shards[0].shape[0]
    parts = []
    for s in range(tp):
        local = ids - s * v
        own = (local >= 0) & (local < v)
        p = np.zeros((len(ids), E.shape[1]), dtype=E.dtype)
        p[own] = shards[s][local[own]]
        parts.append(p)
    return all_reduce(parts)


def log_softmax_normaliser(z):
    """log sum_v exp(z[t, v]) per row, computed as m + log sum exp(z - m)
    with m the row maximum (the shift changes nothing mathematically and
    keeps exp in range)."""
    z = np.asarray(z, np.float64)
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def cross_entropy(z, labels):
    """loss[t] = log sum_v exp(z[t, v]) - z[t, labels[t]]: the negative log
    of the softmax probability of the label."""
    z = np.asarray(z, np.float64)
    labels = np.asarray(labels)
    return log_softmax_normaliser(z) - z[np.arange(z.shape[0]), labels]


def cross_entropy_grad(z, labels, scale=1.0):
    """Gradient of scale * sum_t loss[t] with respect to the logits:
    scale * (softmax(z[t]) - onehot(labels[t]))."""
    z = np.asarray(z, np.float64)
    p = np.exp(z - log_softmax_normaliser(z)[:, None])
    p[np.arange(z.shape[0]), np.asarray(labels)] -= 1.0
    return scale * p


def vocab_parallel_cross_entropy(logit_shards, labels):
    """Cross-entropy of logits split by vocabulary columns into shards
    [T, V/tp] ([TUT] output layer split by columns; [WIT] loss sharded on
    the class dimension): by definition, the cross-entropy of the gathered
    logits."""
    return cross_entropy(all_gather(logit_shards), labels)


# ---------------------------------------------------------------------------
# Mixture of experts with tensor-parallel experts
# ---------------------------------------------------------------------------

def moe_tp(X, experts, ids, weights, tp, act="swiglu", residual=None):
    """[TRT] FFN module, mixture of experts, TP mode: the router has chosen
    top-k experts ids[t, :] with weights weights[t, :] for token t; every
    expert's MLP is column/row sharded over tp shards (mlp_block) and sees
    the tokens routed to it; token t's output is the weighted sum of its
    experts' outputs, in k order (+ residual).
    experts: list of dicts with W1 (gate, [H, I]), W_up ([H, I], SwiGLU) and
    W2 ([I, H])."""
    X = np.asarray(X)
    ids = np.asarray(ids)
    T, k = ids.shape
    Y = np.zeros((T, experts[0]["W2"].shape[1]), dtype=np.result_type(X, experts[0]["W2"], np.asarray(weights)))
    for j in range(k):
        for e, ex in enumerate(experts):
            rows = np.nonzero(ids[:, j] == e)[0]
            if rows.size == 0:
                continue
            _, ye = mlp_block(X[rows], ex["W1"], ex["W2"], tp, act, W_up=ex.get("W_up"))
            Y[rows] = Y[rows] + np.asarray(weights)[rows, j][:, None] * ye
    if residual is not None:
        Y = Y + residual
    return Y
