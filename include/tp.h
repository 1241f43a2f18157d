/*
 * tp.h - C ABI of the tensor-parallel sharded linear pipeline, B300 (sm_103a).
 *
 * The pipeline (a Transformer block's linears under tensor parallelism) as
 * described on the "CUDA tensor parallel computations" learning-notes page
 * (jokeuncle.github.io) and the "Tensor parallelism: splitting Transformer
 * layers" tutorial (freeguideonline.com):
 *   - a column-parallel linear splits W by output columns; shard s computes
 *     X @ W_s from a replicated X; results are CONCATENATED (all-gather);
 *   - a row-parallel linear splits W by input rows and X by the matching
 *     columns; shard s computes X_s @ W_s, a contribution to the full output;
 *     contributions are SUMMED (all-reduce) or summed and split
 *     (reduce-scatter);
 *   - activations, gates and biases between them are shard-local;
 *   - the MLP is column -> local activation -> row -> sum; attention is QKV
 *     column-split by heads (KV heads replicated when there are fewer than
 *     tp, per the "Parallel strategies in TensorRT LLM" page), local heads,
 *     and an O projection row-split then summed.
 *
 * All tp shards live in ONE device's memory. Each "communication" step is
 * an on-device combine: a reduction folded into a GEMM accumulator, a
 * reduction kernel, or a strided copy.
 *
 * Conventions for every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller. The
 *     library keeps no pointer after a call returns and allocates nothing.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Arguments are validated before anything is launched:
 *     a validation error returns a non-zero status and leaves every output
 *     untouched.
 *   - Row-major layouts. Weights are given as W[K][N] ("[in, out]",
 *     Y = X @ W). Sharded weights are stored K-major per shard (see
 *     tp_shards).
 *   - dtype TP_BF16: bf16 storage, fp32 accumulation, fp32 epilogue math,
 *     one rounding to bf16 at the output. Pointers must be 16-byte aligned
 *     and every row width (K, K/tp, N/tp, N) a multiple of 8 elements
 *     (TP_ERR_ALIGN otherwise). Runs on tcgen05 tensor cores fed by TMA.
 *   - dtype TP_F32: fp32 storage and FFMA arithmetic in a fixed summation
 *     order (exact for integer-valued data whose partial sums stay below
 *     2^24). Pointers 4-byte aligned; any widths.
 *   - T == 0 is a valid empty call (returns TP_OK, launches nothing).
 *   - A failed CUDA launch returns TP_ERR_CUDA. Every device-side wait is
 *     bounded; an expired wait is reported by tp_get_error().
 */
#ifndef TP_B300_TP_H
#define TP_B300_TP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes: every entry point that can fail returns one. */
typedef enum tp_status {
  TP_OK = 0,
  TP_ERR_NULL = 1,        /* a required pointer is NULL */
  TP_ERR_SHAPE = 2,       /* bad size: < 1, not divisible by tp, or mismatched */
  TP_ERR_DTYPE = 3,       /* unknown dtype or dtypes that disagree */
  TP_ERR_MODE = 4,        /* unknown/wrong shard mode, activation, reduce op or flag */
  TP_ERR_ALIGN = 5,       /* pointer or row width breaks the alignment rule */
  TP_ERR_WORKSPACE = 6,   /* workspace or output buffer too small */
  TP_ERR_CUDA = 7,        /* a CUDA runtime/driver call failed */
  TP_ERR_TIMEOUT = 8,     /* a bounded device-side wait expired */
  TP_ERR_UNSUPPORTED = 9, /* valid request outside the library's limits */
  TP_ERR_INDEX = 10       /* (from tp_get_error) a token id or label outside [0, V) */
} tp_status;

/* Storage types. */
enum { TP_F32 = 0, TP_BF16 = 1 };

/* Shard modes ("partition dim" of the [in, out] weight). */
enum { TP_COL = 0, TP_ROW = 1 };

/* Shard-local activations (TP_ACT_SWIGLU = silu(gate) * up). */
enum { TP_ACT_NONE = 0, TP_ACT_RELU = 1, TP_ACT_GELU = 2, TP_ACT_SILU = 3, TP_ACT_SWIGLU = 4 };

/* Combine of row-parallel partials. */
enum { TP_REDUCE_SUM = 0, TP_REDUCE_SCATTER = 1 };

/* Attention core between the QKV and O projections (tp_attn_block): the
 * single-key stand-in (each query attends only to its own token), or scaled
 * dot-product attention of each local head, causal or unmasked. */
enum { TP_ATTN_SINGLE_KEY = 0, TP_ATTN_CAUSAL = 1, TP_ATTN_FULL = 2 };

/*
 * Non-owning view of sharded weights, filled in by tp_shard_weights /
 * tp_shard_qkv. K and N are the FULL weight's in/out features.
 *   mode TP_COL: data is [tp][N/tp][K]: shard s is W[:, s*N/tp:(s+1)*N/tp]
 *                transposed (K contiguous). The whole buffer equals W^T.
 *   mode TP_ROW: data is [tp][N][K/tp]: shard s is W[s*K/tp:(s+1)*K/tp, :]
 *                transposed.
 *   hq, hkv, hd: non-zero only for QKV views (tp_shard_qkv); then N is
 *                tp * (hq/tp + 2*nkv) * hd, with nkv = hkv/tp if hkv >= tp,
 *                else 1 (a replicated kv head).
 */
typedef struct tp_shards {
  void* data;
  int64_t K;
  int64_t N;
  int32_t tp;
  int32_t mode;
  int32_t dtype;
  int32_t hq;
  int32_t hkv;
  int32_t hd;
} tp_shards;

/* Human-readable name of a status code. Never NULL. */
const char* tp_status_string(tp_status status);

/* ABI version of this header (increments on incompatible change). */
int tp_abi_version(void);

/*
 * tp_shard_weights - re-shard a full weight into tp column or row shards.
 * Weight re-sharding and distribution, step 3 of the "AutoTP" page's
 * automatic derivation; the split itself is the Column Parallel / Row
 * Parallel split of the "CUDA tensor parallel computations" page.
 *   W        [K][N] row-major, dtype `dtype`.
 *   mode     TP_COL (N % tp == 0) or TP_ROW (K % tp == 0).
 *   out      K*N elements; layout as in tp_shards. out_bytes is its size.
 *   view     filled on success (may be NULL).
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE (K, N < 1 or not divisible),
 * TP_ERR_MODE, TP_ERR_DTYPE, TP_ERR_WORKSPACE (out_bytes < K*N*elem),
 * TP_ERR_ALIGN (bf16: K/tp, N/tp must be multiples of 8; 16-byte pointers).
 */
tp_status tp_shard_weights(const void* W, int64_t K, int64_t N, int dtype, int tp, int mode, void* out,
                           size_t out_bytes, tp_shards* view, void* stream);

/*
 * tp_shard_qkv - shard the Q, K, V projections by whole heads.
 * QKV projection split across GPUs by attention heads ("CUDA tensor parallel
 * computations" page, QKV projection section; tutorial page, self-attention
 * block sharding); KV heads replicated when hkv < tp ("Parallel strategies
 * in TensorRT LLM" page, attention tensor parallelism, GQA/MQA exception).
 *   Wq [H][hq*hd], Wk [H][hkv*hd], Wv [H][hkv*hd], row-major.
 *   Shard s holds q heads [s*hq/tp, (s+1)*hq/tp); kv heads [s*hkv/tp, ...)
 *   when hkv >= tp, else the single kv head floor(s*hkv/tp). Its storage is
 *   [Nqkv_s][H] (K-major) with rows: its q heads, then its kv heads' K
 *   columns, then their V columns; out is [tp][Nqkv_s][H].
 *   Requires hq % tp == 0, hq % hkv == 0, and hkv % tp == 0 (hkv >= tp) or
 *   tp % hkv == 0 (hkv < tp).
 * Errors as tp_shard_weights.
 */
tp_status tp_shard_qkv(const void* Wq, const void* Wk, const void* Wv, int64_t H, int hq, int hkv, int hd,
                       int tp, int dtype, void* out, size_t out_bytes, tp_shards* view, void* stream);

/* Elements of tp_shard_qkv's output, or 0 if the head counts are invalid. */
size_t tp_qkv_shard_elems(int64_t H, int hq, int hkv, int hd, int tp);

/*
 * tp_column_linear - column-parallel linear with the shard-local epilogue.
 * Y_s = act(X @ W_s + b_s) for s = 0..tp-1 ("CUDA tensor parallel
 * computations" page: Column Parallel, local elementwise computation).
 *   X       [T][K], replicated input, dtype W->dtype.
 *   W       TP_COL shards. W_up: TP_COL shards of the up projection, required
 *           iff act == TP_ACT_SWIGLU (then Y_s = silu(X@Wg_s + b_s) *
 *           (X@Wu_s + bu_s)), same K, N, tp, dtype.
 *   bias    [N] or NULL (shard s uses bias[s*N/tp ...]); bias_up likewise.
 *   concat  0: Y is [tp][T][N/tp] (each shard's own output);
 *           1: Y is [T][N], the all-gather result, written in place.
 *   For a QKV view (tp_shard_qkv) with replicated kv heads and no bias, the
 *   K|V columns of each group of tp/hkv shards are computed once and stored
 *   to every shard of the group (they are identical).
 *   workspace, ws_bytes: optional scratch (NULL/0 allowed) of at least
 *           tp_gemm_workspace_bytes(T, W) bytes, 256-byte aligned. With it, a
 *           bf16 call with T <= 64 uses the weight-streaming arrangement
 *           (weights as the 128-row MMA operand, their K loops split evenly
 *           over all SMs), and a larger row-parallel call whose last round
 *           of 256-token units leaves pairs of SMs idle cuts those units
 *           along K into pieces run side by side. Split tiles and pieces are combined in a
 *           fixed order, so results do not depend on timing. Without it every
 *           tile runs whole. The two agree within rounding.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_MODE, TP_ERR_DTYPE, TP_ERR_ALIGN,
 * TP_ERR_WORKSPACE, TP_ERR_CUDA.
 */
tp_status tp_column_linear(const void* X, int64_t T, const tp_shards* W, const tp_shards* W_up,
                           const void* bias, const void* bias_up, int act, int concat, void* Y,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * tp_row_linear - row-parallel linear with the combine fused:
 * Y = sum_{s=0..tp-1} Xs[s] @ W_s (+ bias, once) (+ residual).
 * ("CUDA tensor parallel computations" page: Row Parallel, all-reduce.)
 * The shard sum is accumulated in fp32 inside the GEMM; partials never
 * reach memory.
 *   Xs        [tp][T][K/tp] (shard s's input block), dtype W->dtype.
 *   W         TP_ROW shards.
 *   bias      [N] or NULL.  residual [T][N] or NULL (may alias Y: each
 *             element is read before it is written, by the same thread).
 *   Y         [T][N].
 *   out_dtype dtype of bias, residual and Y: W->dtype, or TP_F32 with bf16
 *             shards (an fp32 residual stream; the shard sum, bias and
 *             residual are added in fp32 and stored without rounding to bf16).
 *   workspace, ws_bytes: as tp_column_linear.
 * Errors as tp_column_linear.
 */
tp_status tp_row_linear(const void* Xs, int64_t T, const tp_shards* W, const void* bias,
                        const void* residual, void* Y, int out_dtype, void* workspace, size_t ws_bytes,
                        void* stream);

/* Scratch bytes that let tp_column_linear / tp_row_linear over W at T
 * tokens split tiles (the weight-streaming arrangement at T <= 64, the split
 * last round above): about 21 MB; 0 for fp32 views or invalid arguments. */
size_t tp_gemm_workspace_bytes(int64_t T, const tp_shards* W);

/*
 * tp_row_linear_partials - the per-shard contributions P_s = Xs[s] @ W_s,
 * kept apart ("Row Parallel": each GPU computes one contribution).
 *   partials  [tp][T][N] fp32 (always fp32, whatever W->dtype).
 * Errors as tp_column_linear.
 */
tp_status tp_row_linear_partials(const void* Xs, int64_t T, const tp_shards* W, float* partials,
                                 void* stream);

/*
 * tp_shard_reduce - combine row-parallel partials.
 *   op TP_REDUCE_SUM:     out[T][N] = sum_s partials[s] (+ bias) (+ residual)
 *                         (all-reduce: every shard's copy is this one buffer).
 *   op TP_REDUCE_SCATTER: the same sum, read as out[tp][T/tp][N]: shard s
 *                         keeps token rows [s*T/tp, (s+1)*T/tp). Requires
 *                         T % tp == 0. (The split axis, tokens, is a reading:
 *                         the page says only "sum, then split".)
 *   The sum is taken in fp32 in shard order 0..tp-1; bias [N] is added once;
 *   residual is [T][N] and may alias out. bias, residual and out have dtype
 *   out_dtype.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_MODE, TP_ERR_DTYPE, TP_ERR_ALIGN
 * (16-byte pointers when N % 4 == 0), TP_ERR_CUDA.
 */
tp_status tp_shard_reduce(const float* partials, int tp, int64_t T, int64_t N, int op, const void* bias,
                          const void* residual, int out_dtype, void* out, void* stream);

/*
 * tp_shard_gather - all-gather by concatenation:
 * out[t][s*N/tp + j] = shards[s][t][j] ("Column Parallel": concatenate, do
 * not add). shards [tp][T][N/tp], out [T][N], dtype `dtype`.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_DTYPE, TP_ERR_CUDA.
 */
tp_status tp_shard_gather(const void* shards, int tp, int64_t T, int64_t N, int dtype, void* out,
                          void* stream);

/* Workspace bytes tp_mlp_block needs for T tokens, hidden H, intermediate I. */
size_t tp_mlp_workspace_bytes(int64_t T, int64_t H, int64_t I, int tp, int dtype);

/*
 * tp_mlp_block - the MLP block: column -> local activation -> row -> sum
 * ("CUDA tensor parallel computations" page, MLP section; tutorial page,
 * MLP block sharding steps 1-4):
 *   Hs[s] = act(X @ W1_s + b1_s)            (SwiGLU: silu(X@Wg_s+b) * (X@Wu_s+bu))
 *   Y     = sum_s Hs[s] @ W2_s (+ b2, once) (+ residual)
 *   X [T][H]; W1, W_up: TP_COL shards (K=H, N=I); W2: TP_ROW shards (K=I,
 *   N=H); all the same tp and dtype. Y [T][H]; residual may alias Y.
 *   out_dtype: dtype of b2, residual and Y (as tp_row_linear).
 *   workspace: >= tp_mlp_workspace_bytes(T, H, I, tp, dtype) bytes, 256-byte
 *   aligned; holds Hs ([tp][T][I/tp], dtype) and, for bf16, the split-tile
 *   scratch (see tp_column_linear). Its contents on return are unspecified.
 * Errors: as tp_column_linear, plus TP_ERR_WORKSPACE.
 */
tp_status tp_mlp_block(const void* X, int64_t T, const tp_shards* W1, const tp_shards* W_up,
                       const tp_shards* W2, const void* b1, const void* b1_up, const void* b2,
                       const void* residual, int act, int out_dtype, void* workspace, size_t ws_bytes,
                       void* Y, void* stream);

/*
 * tp_mlp_block_static - tp_mlp_block without a caller workspace.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory at the point of the call -- for example a
 * plug-in whose host process owns the whole device-memory budget and forbids
 * further cudaMalloc calls, or a caller on a path where the driver's
 * allocator must not be entered. It takes the same arguments as tp_mlp_block
 * minus workspace/ws_bytes; Hs and the split-tile scratch live in one
 * array of TP_STATIC_WORKSPACE_BYTES in the library's static device memory,
 * which every GPU that loads the library holds until the process exits.
 *   Limit: tp_mlp_workspace_bytes(T, H, I, tp, dtype) must not exceed
 *   TP_STATIC_WORKSPACE_BYTES (32 MiB), else TP_ERR_WORKSPACE and nothing is
 *   launched. For bf16 that covers T * I up to about 6.2M, whatever T
 *   (Hs plus about 21 MB of scratch; e.g. the 70B-shaped decode block at
 *   T = 64).
 *   The array belongs to the library's device code. CUDA loads that code,
 *   and reserves the array with it, on a device the first time anything of
 *   the library runs there: a kernel launch from any entry point, or the
 *   first tp_mlp_block_static call, which also looks up the array's device
 *   address (with that device current) and caches it. Make one call of any
 *   entry point on each device before the point where allocation is
 *   forbidden, and make that first tp_mlp_block_static call before any
 *   stream capture. Every later call allocates nothing: no
 *   cudaMalloc/cudaFree and no allocating library routine.
 *   Every call shares the one array and the array keeps the last call's
 *   contents. Leftover contents are harmless: Hs is rewritten before it is
 *   read, and the split-tile synchronisation words are tagged with each
 *   launch's own epoch (a word left by an earlier call reads as "not
 *   arrived") and returned to zero by the kernel that used them; this is
 *   also why calls in a row can share the array. Calls that overlap on the
 *   GPU -- on different streams, or from different host threads without
 *   ordering -- race on the array; serialise them.
 * Errors: as tp_mlp_block.
 */
#define TP_STATIC_WORKSPACE_BYTES ((size_t)32 << 20)
tp_status tp_mlp_block_static(const void* X, int64_t T, const tp_shards* W1, const tp_shards* W_up,
                              const tp_shards* W2, const void* b1, const void* b1_up, const void* b2,
                              const void* residual, int act, int out_dtype, void* Y, void* stream);

/*
 * Backward of the column/row pair ("Tensor parallelism: splitting
 * Transformer layers" tutorial page: column-wise sharding, MLP block
 * sharding, and forward/backward communication symmetry). The forward
 * all-reduce after a row layer is an identity in the backward: every shard
 * receives the same dY. A column layer's shards each hold a share
 * dY_s @ W_s^T of its input gradient, and the input gradient is their sum
 * (all-reduce), taken in fp32 inside the accumulator in shard order.
 * Weight gradients are local. Every GEMM reads the forward's shard storage
 * as it is (MN-major operands on the tensor cores): nothing is transposed
 * in memory, and each weight gradient comes out in the layout of the shards
 * it belongs to, so an optimizer can update them in place.
 * bf16 views run on the tensor cores; fp32 views on an FFMA GEMM in which
 * every element is a fixed-order chain of fmaf, so integer-valued inputs
 * whose partial sums stay below 2^24 give exact results. All pointers are
 * device pointers, 16-byte aligned for bf16 and 4-byte aligned for fp32;
 * every tensor has the view's dtype. T >= 1 (T == 0 returns TP_OK and
 * launches nothing).
 */

/*
 * tp_row_linear_backward - backward of Y = sum_s Xs[s] @ W_s.
 *   W: TP_ROW view (shards [tp][N][K/tp]); Xs [tp][T][K/tp] (the forward
 *   input, needed for dW); dY [T][N].
 *   dXs [tp][T][K/tp] = dY @ W_s^T for every shard, or NULL to skip;
 *   dW  [tp][N][K/tp] (the view's layout) = (Xs[s]^T @ dY)^T, or NULL.
 * Errors: TP_ERR_NULL, TP_ERR_MODE, TP_ERR_SHAPE, TP_ERR_DTYPE, TP_ERR_ALIGN,
 * TP_ERR_CUDA.
 */
tp_status tp_row_linear_backward(const void* Xs, int64_t T, const tp_shards* W, const void* dY, void* dXs,
                                 void* dW, void* stream);

/*
 * tp_column_linear_backward - backward of Y_s = X @ W_s (X replicated).
 *   W: TP_COL view (shards [tp][N/tp][K]); X [T][K] (the forward input,
 *   needed for dW); dYs [tp][T][N/tp].
 *   dX [T][K] = sum_s dYs[s] @ W_s^T (+ dR), or NULL to skip. dR [T][K]
 *   (the gradient reaching X by another path, e.g. a residual branch) may
 *   be NULL. Token rows [s*T/tp, (s+1)*T/tp) of dX are shard s's slice of
 *   the reduce-scatter form.
 *   dW [tp][N/tp][K] (the view's layout) = (X^T @ dYs[s])^T, or NULL.
 *   workspace (optional, 256-byte aligned, >= tp_gemm_workspace_bytes(T,
 *   W)): scratch that lets the dX GEMM split its last round; NULL runs
 *   whole tiles only.
 * Errors: as tp_row_linear_backward, plus TP_ERR_WORKSPACE.
 */
tp_status tp_column_linear_backward(const void* X, int64_t T, const tp_shards* W, const void* dYs,
                                    const void* dR, void* dX, void* dW, void* workspace, size_t ws_bytes,
                                    void* stream);

/* Workspace bytes tp_mlp_backward needs (act decides whether dU is kept). */
size_t tp_mlp_backward_workspace_bytes(int64_t T, int64_t H, int64_t I, int tp, int act, int dtype);

/*
 * tp_mlp_backward - backward of tp_mlp_block without biases (the tutorial
 * page's MLP block steps 4 to 1 in reverse):
 *   dHs[s] = dY @ W2_s^T                         (row layer, dY on every shard)
 *   dW2_s  = Hs[s]^T @ dY                        -> dW2 [tp][H][I/tp]
 *   dG, dU = activation gradients of dHs         (dU for SwiGLU only)
 *   dW1_s  = X^T @ dG[s], dWu_s = X^T @ dU[s]    -> dW1, dW_up [tp][I/tp][H]
 *   dX     = sum_s dG[s] @ W1_s^T (+ sum_s dU[s] @ Wu_s^T) (+ dR)
 *   Five to six launches: five GEMMs (for SwiGLU the gate and up sums of dX
 *   share one accumulator) and the activation gradient, an HBM-bound
 *   elementwise pass over dHs.
 *   X [T][H]; W1 (gate for SwiGLU), W_up: TP_COL views (K=H, N=I); W2:
 *   TP_ROW view (K=I, N=H). Saved forward values, [tp][T][I/tp] each: G =
 *   X @ W1_s (the pre-activation), U = X @ Wu_s (SwiGLU only, else NULL),
 *   Hs = the activation output that fed W2. dY, dR, dX [T][H]; dR may be
 *   NULL. Any of dX, dW1, dW_up, dW2 may be NULL to skip it (dW_up must be
 *   NULL unless SwiGLU).
 *   workspace: >= tp_mlp_backward_workspace_bytes(T, H, I, tp, act, dtype) bytes,
 *   256-byte aligned: dHs, dG and dU (T * I elements each) plus the
 *   split-tile scratch. Contents on return are unspecified. (On the bf16
 *   path dG and dU are kept token-major, [T][I] with the shards side by
 *   side, so that dX is one contraction over I and dW1, dW_up one [I][H]
 *   product each: the same sums, with no tile cut at a shard's end.)
 * Errors: as tp_column_linear_backward, plus TP_ERR_MODE for an unknown act
 *   and, on the bf16 path, TP_ERR_ALIGN if I/tp is not a multiple of 8 and
 *   TP_ERR_UNSUPPORTED if T * I/tp >= 2^34.
 */
tp_status tp_mlp_backward(const void* X, int64_t T, const tp_shards* W1, const tp_shards* W_up,
                          const tp_shards* W2, int act, const void* G, const void* U, const void* Hs,
                          const void* dY, const void* dR, void* workspace, size_t ws_bytes, void* dX,
                          void* dW1, void* dW_up, void* dW2, void* stream);

/*
 * Vocabulary-parallel input and output layers ("Tensor parallelism:
 * splitting Transformer layers" tutorial page, input and output layers;
 * "What is tensor parallelism" page, loss sharded over the class dimension).
 * The embedding table is split by vocabulary rows and the LM head by
 * vocabulary columns (tp_shard_weights in TP_COL mode, then
 * tp_column_linear with concat = 0 gives the logits [tp][T][V/tp]).
 */

/*
 * tp_vocab_embedding - Y[t] = E[ids[t]] from a table split by vocabulary
 * rows: shard s holds ids [s*V/tp, (s+1)*V/tp) as rows s*V/tp.. of E, so
 * the shards stored one after another are E [V][H] itself. A lookup is each
 * shard's masked lookup summed over shards (all-reduce); one shard owns
 * each id, so the kernel copies the owner's row.
 *   ids [T] int32 (device); E [V][H] and Y [T][H] of dtype `dtype`.
 *   An id outside [0, V) gives a zero row and makes the next tp_get_error
 *   return TP_ERR_INDEX.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE (V % tp != 0, sizes < 1), TP_ERR_DTYPE,
 * TP_ERR_ALIGN (4-byte ids and element-aligned tables), TP_ERR_CUDA.
 */
tp_status tp_vocab_embedding(const int32_t* ids, int64_t T, const void* E, int64_t V, int64_t H, int tp,
                             int dtype, void* Y, void* stream);

/* Workspace bytes tp_vocab_cross_entropy needs (T tokens, vocabulary V). */
size_t tp_cross_entropy_workspace_bytes(int64_t T, int64_t V, int tp);

/*
 * tp_vocab_cross_entropy - loss[t] = log sum_v exp(z[t][v]) - z[t][labels[t]]
 * over logits split by vocabulary columns, z_s = logits[s] [T][V/tp].
 * Each shard reduces its own columns, in chunks of 2048, to (max, sum of
 * exp(z - max), the label's logit where it holds the label, else 0); the
 * per-token combine of those statistics in shard and chunk order (max,
 * rescaled sum, the sum of the masked label logits) is the all-reduce of a
 * vocabulary-parallel loss. fp32 arithmetic.
 *   logits [tp][T][V/tp], dtype `dtype`; labels [T] int32 (device).
 *   loss [T] fp32 per-token losses, or NULL; mean_loss [1] fp32 (their mean,
 *   summed in a fixed order), or NULL.
 *   dlogits [tp][T][V/tp] (dtype), or NULL: the gradient of
 *   grad_scale * sum_t loss[t], grad_scale * (softmax(z[t]) - onehot(label));
 *   it may be the logits buffer itself (written in place). grad_scale =
 *   1/T gives the gradient of the mean loss.
 *   workspace >= tp_cross_entropy_workspace_bytes(T, V, tp), 256-byte
 *   aligned.
 *   A label outside [0, V) gives a NaN loss and makes the next
 *   tp_get_error return TP_ERR_INDEX.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_DTYPE, TP_ERR_ALIGN,
 * TP_ERR_WORKSPACE, TP_ERR_CUDA.
 */
tp_status tp_vocab_cross_entropy(const void* logits, const int32_t* labels, int64_t T, int64_t V, int tp,
                                 int dtype, float* loss, float* mean_loss, void* dlogits, float grad_scale,
                                 void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes tp_lm_head_cross_entropy needs (T tokens, the LM head's view). */
size_t tp_lm_head_ce_workspace_bytes(int64_t T, const tp_shards* W_lm);

/*
 * tp_lm_head_cross_entropy - the column-parallel LM head and the
 * vocabulary-parallel loss in one call (same pages as above): logits
 * z_s = X W_s for every vocabulary shard s, then the losses, their mean and
 * optionally the gradient, as tp_vocab_cross_entropy defines them. On the
 * bf16 path with T > 64 the GEMM's epilogue reduces each (shard, token,
 * 256-column tile) of logits to (max, sum of exp(z - max), the label's
 * logit) from its fp32 accumulator while it stores the bf16 logits, so no
 * pass re-reads the logits for the loss; the statistics are then combined
 * per token in shard and tile order. The loss is thus that of the fp32
 * logits; the gradient is computed from the stored logits. With T <= 64
 * (the weight-streaming GEMM) or fp32 views the logits are reduced by a
 * separate pass, as in tp_vocab_cross_entropy.
 *   X [T][K] (K = W_lm->K); W_lm a TP_COL view of the [K][V] head, V = W_lm->N;
 *   labels [T] int32 (device).
 *   logits [tp][T][V/tp] (the view's dtype), written.
 *   loss, mean_loss, dlogits (may be `logits`), grad_scale: as
 *   tp_vocab_cross_entropy.
 *   workspace >= tp_lm_head_ce_workspace_bytes(T, W_lm), 256-byte aligned.
 *   A label outside [0, V) gives a NaN loss and makes the next
 *   tp_get_error return TP_ERR_INDEX.
 * Ownership: every buffer belongs to the caller; nothing is allocated.
 * Errors: as tp_column_linear (no activation, no bias), plus TP_ERR_NULL
 * for missing labels or workspace and TP_ERR_WORKSPACE.
 */
tp_status tp_lm_head_cross_entropy(const void* X, int64_t T, const tp_shards* W_lm, const int32_t* labels,
                                   void* logits, float* loss, float* mean_loss, void* dlogits, float grad_scale,
                                   void* workspace, size_t ws_bytes, void* stream);

/*
 * Mixture of experts with tensor-parallel experts ("Parallel strategies in
 * TensorRT LLM" page, FFN module, mixture of experts, TP mode: each expert's
 * weights are split across all shards; every shard sees all tokens).
 */

/* Workspace bytes tp_moe_block needs (T tokens, top-k of E experts). */
size_t tp_moe_workspace_bytes(int64_t T, int64_t H, int64_t I, int k, int E, int tp);

/*
 * tp_moe_block - Y[t] = sum_j weights[t][j] * MLP_{ids[t][j]}(X[t]) (+ residual)
 * with SwiGLU experts, each an MLP block under TP (gate and up column-split,
 * down row-split, shard sum). The router's choice is an input.
 *   X [T][H] bf16; ids [T][k] int32 in [0, E); weights [T][k] fp32.
 *   Wg, Wu: TP_COL views of ONE expert's shape (K = H, N = I) whose data
 *   holds the E experts' shard sets one after another ([E][tp][I/tp][H]);
 *   Wd: TP_ROW view (K = I, N = H), data [E][tp][H][I/tp]. bf16. E <= 1024.
 *   residual [T][H] or NULL; Y [T][H] bf16.
 *   The tokens of each expert are gathered, in token order, into a segment
 *   padded to 256 rows; the gate/up and down GEMMs each run as one grouped
 *   launch over all segments (the expert rows kept in fp32); Y sums a
 *   token's k slots in order in fp32.
 *   workspace >= tp_moe_workspace_bytes(...), 256-byte aligned.
 *   An id outside [0, E) drops that slot and makes the next tp_get_error
 *   return TP_ERR_INDEX.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_MODE, TP_ERR_DTYPE, TP_ERR_ALIGN,
 * TP_ERR_WORKSPACE, TP_ERR_UNSUPPORTED, TP_ERR_CUDA.
 */
tp_status tp_moe_block(const void* X, int64_t T, const int32_t* ids, const float* weights, int k, int E,
                       const tp_shards* Wg, const tp_shards* Wu, const tp_shards* Wd, const void* residual,
                       void* workspace, size_t ws_bytes, void* Y, void* stream);

/* Workspace bytes tp_attn_proj needs. */
size_t tp_attn_workspace_bytes(int64_t T, int hq, int hkv, int hd, int tp, int dtype);

/*
 * tp_attn_proj - attention projections under TP: QKV column-parallel by
 * heads, the local attention heads, O row-parallel then summed ("CUDA tensor
 * parallel computations" page, QKV projection, attention heads and output
 * projection sections).
 *   X        [T][H]. Wqkv: the view from tp_shard_qkv (K=H). Wo: TP_ROW
 *            shards of the O projection (K = hq*hd, N = H), same tp/dtype.
 *   ctx      [tp][T][hq/tp*hd]: the attention output of each shard's heads,
 *            or NULL for the single-key stand-in (each query attends only to
 *            its own token, so the context of q head h is V of its kv head).
 *   residual [T][H] or NULL; may alias Y. out_dtype: dtype of residual and Y
 *            (as tp_row_linear).
 *   qkv_out  [tp][T][Nqkv_s] (each shard's q | k | v), or NULL to keep it in
 *            the workspace.
 *   Y        [T][H] = sum_s ctx[s] @ Wo_s (+ residual).
 *   When kv heads are replicated (hkv < tp) the K|V columns of each group of
 *   tp/hkv shards are computed once and stored to every shard of the group.
 *   Requires H <= 4 * hq * hd (TP_ERR_UNSUPPORTED otherwise).
 * Errors: as tp_mlp_block.
 */
tp_status tp_attn_proj(const void* X, int64_t T, const tp_shards* Wqkv, const tp_shards* Wo,
                       const void* ctx, const void* residual, int out_dtype, void* qkv_out, void* workspace,
                       size_t ws_bytes, void* Y, void* stream);

/*
 * tp_attention - the attention core of every local head of every shard
 * ("CUDA tensor parallel computations" page, attention heads: each GPU runs
 * the attention of its own heads; tutorial page, self-attention block
 * sharding): for q head h of shard s and its kv head g = h / (hq / hkv)
 * (a replica when hkv < tp),
 *   ctx[s][:, h_local] = softmax(Q_h K_g^T / sqrt(hd)) V_g,
 * with query t restricted to keys 0..t under TP_ATTN_CAUSAL (the decoder
 * reading) and unmasked under TP_ATTN_FULL.
 *   qkv   [tp][T][(nq + 2 nkv) * hd] bf16, the layout tp_column_linear writes
 *         for a tp_shard_qkv view (q heads | k heads | v heads per shard).
 *   ctx   [tp][T][nq * hd] bf16, written.
 *   hd must be 64 or 128 (TP_ERR_UNSUPPORTED otherwise). Scores, the
 *   softmax and the P V accumulation are fp32; P is rounded to bf16 before
 *   P V.
 *   T = 0 is a no-op (null pointers allowed). The launch is persistent, one
 *   CTA per SM; a work unit is two tiles of 128 queries that read the same
 *   keys (two q heads of one kv head, or two query blocks of one head), so
 *   there are about hq * ceil(T / 128) / 2 units; hq * ceil(T / 128) above
 *   2^30 - 1 is TP_ERR_UNSUPPORTED.
 * Ownership: both buffers belong to the caller; nothing is allocated. The
 * call is asynchronous on `stream`; a bounded device wait that expired shows
 * as TP_ERR_TIMEOUT from tp_get_error.
 * Errors: TP_ERR_NULL, TP_ERR_MODE, TP_ERR_SHAPE (T < 0, or head counts that
 * tp_shard_qkv rejects), TP_ERR_UNSUPPORTED, TP_ERR_ALIGN, TP_ERR_CUDA.
 */
tp_status tp_attention(const void* qkv, int64_t T, int tp, int hq, int hkv, int hd, int mode, void* ctx, void* stream);

/*
 * tp_attn_block - tp_attn_proj with the attention core chosen by `mode`:
 * TP_ATTN_SINGLE_KEY (as tp_attn_proj without ctx), TP_ATTN_CAUSAL or
 * TP_ATTN_FULL (tp_attention between the QKV and O launches; bf16, hd 64 or 128).
 * Arguments otherwise as tp_attn_proj; the workspace holds qkv (unless
 * qkv_out is given), the context and the split-tile scratch
 * (tp_attn_workspace_bytes).
 * Errors: as tp_attn_proj, plus TP_ERR_MODE for an unknown mode and
 * TP_ERR_UNSUPPORTED for a core other than the single-key one on fp32 views,
 * hd other than 64 and 128, or too many query blocks (as tp_attention).
 */
tp_status tp_attn_block(const void* X, int64_t T, const tp_shards* Wqkv, const tp_shards* Wo, int mode,
                        const void* residual, int out_dtype, void* qkv_out, void* workspace, size_t ws_bytes, void* Y,
                        void* stream);

/*
 * tp_rmsnorm - RMSNorm on the replicated hidden ("CUDA tensor parallel
 * computations" page, local elementwise section: a norm is local when it
 * runs on the replicated hidden): Y = X * gamma / sqrt(mean(X^2) + eps),
 * fp32 statistics. X [T][H] and gamma [H] (or NULL = 1) in `dtype`; Y [T][H]
 * in `out_dtype` (e.g. an fp32 residual stream normalised into bf16 GEMM
 * input).
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_DTYPE, TP_ERR_ALIGN, TP_ERR_CUDA.
 */
tp_status tp_rmsnorm(const void* X, const void* gamma, int64_t T, int64_t H, float eps, int dtype, void* Y,
                     int out_dtype, void* stream);

/*
 * tp_last_cuda_error - the error code of the most recent CUDA call made by
 * this library on the calling host thread that failed (a cudaError_t, or
 * the CUresult of a tensor-map encoding), 0 if none has failed. A call that
 * returned TP_ERR_CUDA has set it; it is not cleared by later successes.
 * tp_cuda_error_name - the runtime's name for such a code (a static
 * string). The pages have no counterpart: these say why TP_ERR_CUDA was
 * returned.
 */
int tp_last_cuda_error(void);
const char* tp_cuda_error_name(int code);

/*
 * tp_get_error - synchronise `stream`, then report and clear the device
 * error word: TP_ERR_TIMEOUT if a kernel's bounded wait expired since the
 * last call (that kernel's outputs are then undefined), TP_ERR_CUDA if the
 * stream reported an error, else TP_OK.
 */
tp_status tp_get_error(void* stream);

/*
 * Test hooks (synchronous; they change device-global state used by every
 * later launch on the current device):
 *   tp_debug_set_wait_limit_ns: limit of every bounded device wait
 *     (default 2e9 ns).
 *   tp_debug_inject(1): the next tensor-core GEMM launch's first block
 *     withholds one operand load, so its consumer's wait expires and the
 *     kernel takes its abort path; tp_debug_inject(2): the same in its
 *     second block (in a launch of CTA pairs, the odd CTA of the first
 *     pair). tp_debug_inject(0) disarms.
 */
tp_status tp_debug_set_wait_limit_ns(uint64_t ns);
tp_status tp_debug_inject(int kind);

#ifdef __cplusplus
}
#endif

#endif /* TP_B300_TP_H */
