// C ABI of the tensor-parallel sharded linear pipeline (declared in tp.h).
//
// Each entry point validates its arguments on the host (no CUDA call before
// validation passes), then launches the kernels of its step on the caller's
// stream. Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <random>

#include "tp.h"
#include "tp_attention.cuh"
#include "tp_elementwise.cuh"
#include "tp_gemm.cuh"
#include "tp_simt.cuh"
#include "tp_moe.cuh"
#include "tp_vocab.cuh"

namespace {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------------------
// Host helpers
// ---------------------------------------------------------------------------
inline size_t elem_size(int dtype) { return dtype == TP_BF16 ? 2 : 4; }
inline bool dtype_ok(int dtype) { return dtype == TP_F32 || dtype == TP_BF16; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }
// a status computed as an int (a helper's result) as the public return type
inline tp_status as_status(int r) { return static_cast<tp_status>(r); }

// Pointer alignment each dtype path needs (bf16 feeds TMA / 16-byte vectors).
inline bool ptr_ok(const void* p, int dtype) {
  return p == nullptr || aligned(p, dtype == TP_BF16 ? 16 : 4);
}

// The code of the last CUDA runtime or driver call of this library that
// failed on the calling host thread (tp_last_cuda_error).
thread_local int g_last_cuda_error = 0;

// Records a failed call's code; true when the call succeeded.
inline bool cuda_ok(cudaError_t e) {
  if (e == cudaSuccess) return true;
  g_last_cuda_error = static_cast<int>(e);
  return false;
}

int launch_status() { return cuda_ok(cudaGetLastError()) ? TP_OK : TP_ERR_CUDA; }

int num_sms() {
  static int cache[128] = {0};
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev))) return 0;
  if (dev < 0 || dev >= 128) return 0;
  if (cache[dev] == 0) {
    int v = 0;
    if (!cuda_ok(cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev))) return 0;
    cache[dev] = v;
  }
  return cache[dev];
}

int grid_for(int64_t work, int threads) {
  const int sms = std::max(1, num_sms());
  const int64_t want = cdiv(std::max<int64_t>(work, 1), threads);
  return static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sms) * 16));
}

// --- TMA tensor maps ---------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D bf16 map over [d2][d1][d0] (d0 contiguous), box {64, box1, 1}, 128-byte
// swizzle, zero fill outside the tensor.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {64, box1, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) g_last_cuda_error = static_cast<int>(r);
  return r == CUDA_SUCCESS;
}

// 3-D map for bulk tensor stores of an output [d2][d1][d0] (d0 contiguous)
// with byte strides s1 (dim 1) and s2 (dim 2): box {128 bytes of elements,
// 32 rows, 1}, 128-byte swizzle (the epilogue's staging layout).
bool make_store_map(CUtensorMap* m, void* base, bool f32, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                    uint64_t s2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {f32 ? 32u : 64u, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) g_last_cuda_error = static_cast<int>(r);
  return r == CUDA_SUCCESS;
}

// Output maps of a token-major launch (unused by the weight-streaming one).
struct OutMaps {
  CUtensorMap y;  // the output
  CUtensorMap c;  // the attention context (QKV launches that write it)
};

// --- shard-view checks -------------------------------------------------------
int check_view(const tp_shards* W, int mode) {
  if (!W || !W->data) return TP_ERR_NULL;
  if (W->mode != mode) return TP_ERR_MODE;
  if (!dtype_ok(W->dtype)) return TP_ERR_DTYPE;
  if (W->tp < 1 || W->K < 1 || W->N < 1) return TP_ERR_SHAPE;
  if (mode == TP_COL && W->N % W->tp != 0) return TP_ERR_SHAPE;
  if (mode == TP_ROW && W->K % W->tp != 0) return TP_ERR_SHAPE;
  if (W->K > INT32_MAX || W->N > INT32_MAX) return TP_ERR_UNSUPPORTED;
  if (W->dtype == TP_BF16) {
    const int64_t inner = mode == TP_COL ? W->K : W->K / W->tp;
    const int64_t outw = mode == TP_COL ? W->N / W->tp : W->N;
    if (inner % 8 != 0 || outw % 8 != 0 || !aligned(W->data, 16)) return TP_ERR_ALIGN;
  } else if (!aligned(W->data, 4)) {
    return TP_ERR_ALIGN;
  }
  return TP_OK;
}

bool same_shape(const tp_shards* a, const tp_shards* b) {
  return a->K == b->K && a->N == b->N && a->tp == b->tp && a->mode == b->mode && a->dtype == b->dtype;
}

// ---------------------------------------------------------------------------
// Tensor-core GEMM launchers (bf16)
// ---------------------------------------------------------------------------
// Scratch for the stream-K schedule: fp32 workspace slots for split tiles
// and one counter per split tile. Without scratch every tile runs whole.
struct Scratch {
  float* partials;
  size_t partial_bytes;
  unsigned long long* words;  // epoch-tagged synchronisation words
  size_t nwords;
};

constexpr int SK_MAX_CTAS = 160;  // grid cap of the stream-K schedule (>= SMs of a B300)
constexpr int SWAP_MAX_T = 64;    // token counts served by the weight-streaming (swap) arrangement

// fp32 slots for split tiles of the weight-streaming arrangement: two per CTA,
// each 128 rows x up to 128 accumulator columns.
constexpr size_t SK_PARTIAL_BYTES = static_cast<size_t>(2) * SK_MAX_CTAS * 128 * 128 * sizeof(float);

// Epoch of a launch that splits tiles: a per-process random value and a
// launch counter, so no earlier launch (and no leftover workspace contents,
// except with vanishing probability) carries the same value.
unsigned long long next_epoch() {
  static std::atomic<unsigned long long> counter{0};
  static const unsigned long long salt = [] {
    std::random_device rd;
    return (static_cast<unsigned long long>(rd()) << 32) ^ static_cast<unsigned long long>(
        std::chrono::steady_clock::now().time_since_epoch().count());
  }();
  return salt ^ (counter.fetch_add(1, std::memory_order_relaxed) + 1);
}

// Work split. Token-major tiles (normal arrangement) run whole, round-robin:
// CTAs of one wave then walk the same K range in step, so the weight blocks
// they share are read from L2 rather than HBM (splitting their K loops
// measured a 4x rise in DRAM reads on the row GEMM). The weight-streaming
// arrangement reads each weight byte once whatever the order, so there the
// k-iterations of all tiles are spread evenly over the SMs (stream-K).
// Returns the grid size.
int plan_schedule(tpk::GemmArgs& a, bool swap, const Scratch* sc) {
  const int sms = std::max(1, std::min(num_sms(), SK_MAX_CTAS));
  a.dp_tiles = a.num_tiles;
  a.sk_iters = 0;
  const int grid = std::min(a.num_tiles, sms);
  if (!sc || !swap) return grid;
  const int dp = 0;
  const long long sk = static_cast<long long>(a.num_tiles - dp) * a.kpt;
  if (sk < 2 || static_cast<size_t>(a.num_tiles - dp) > sc->nwords) return grid;
  a.dp_tiles = dp;
  a.sk_iters = sk;
  a.partials = sc->partials;
  a.sync_words = sc->words;
  a.epoch = next_epoch();
  return sms;  // the launcher clamps it to sk_iters so that no stream-K range is empty
}

// The kernel's dynamic shared memory limit, raised once per device (not on
// every launch, so that launches can also be recorded into CUDA graphs).
template <int KIND, bool SWAP, bool PAIR, int MN = 0>
bool smem_attr_set() {
  using Cfg = tpk::GemmCfg<KIND, SWAP, PAIR>;
  static bool done[128] = {};
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev)) || dev < 0 || dev >= 128) return false;
  if (!done[dev]) {
    if (!cuda_ok(cudaFuncSetAttribute(tpk::tp_gemm_kernel<KIND, SWAP, PAIR, MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES)))
      return false;
    done[dev] = true;
  }
  return true;
}

// CTA pairs of the 2-SM kernel that fit on the device at once (the
// persistent grid of a paired launch), looked up once per device; the
// kernel's shared-memory limit must have been raised first.
template <int KIND, int MN = 0>
int max_cluster_pairs() {
  using Cfg = tpk::GemmCfg<KIND, false, true>;
  static int cache[128] = {0};
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev)) || dev < 0 || dev >= 128) return 0;
  if (cache[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * std::max(1, num_sms() / 2));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (!cuda_ok(cudaOccupancyMaxActiveClusters(&n, tpk::tp_gemm_kernel<KIND, false, true, MN>, &cfg)) ||
        n < 1) {
      cudaGetLastError();
      n = -1;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

// Pieces per unit of a split last round: as many as the idle pairs allow,
// at most 4 (each piece beyond the owner costs a 128 KB fp32 round trip per
// CTA), each at least 8 k-blocks long. 1: no split. Only row GEMMs split:
// the column GEMMs' heavier epilogues (SwiGLU, QKV replicas and context)
// make the owner's combine the longer tail, and splitting them measured
// slower.
template <int KIND>
int split_ways_for(int rem_units, int pairs, int kpt) {
  if (KIND != tpk::GK_ROW_SUM || rem_units <= 0) return 1;
  int ways = std::min(4, pairs / rem_units);
  while (ways > 1 && kpt / ways < 8) --ways;
  return std::max(1, ways);
}

// Paired launch: clusters of two CTAs, one pair per two SMs, each pair
// walking the 256-token tile units round-robin. With scratch, a partial last
// round is split along K (see the kernel's header).
template <int KIND, int MN = 0>
int pair_launch(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0, const CUtensorMap& b1,
                const OutMaps& om, tpk::GemmArgs args, const Scratch* sc, cudaStream_t st) {
  using Cfg = tpk::GemmCfg<KIND, false, true>;
  if (!smem_attr_set<KIND, false, true, MN>()) return TP_ERR_CUDA;
  const int pairs = max_cluster_pairs<KIND, MN>();
  if (pairs < 1) return TP_ERR_UNSUPPORTED;
  args.dp_tiles = args.num_tiles;
  args.sk_iters = 0;
  int grid_pairs = std::min(args.num_tiles, pairs);
  const int rem = args.num_tiles % pairs;
  const int ways = split_ways_for<KIND>(rem, pairs, args.kpt);
  if (ways > 1 && sc != nullptr &&
      static_cast<size_t>(rem) * (ways - 1) * 2 * (128 * 256 * sizeof(float)) <= sc->partial_bytes &&
      static_cast<size_t>(rem) * (ways - 1) * 2 <= sc->nwords) {
    args.dp_tiles = args.num_tiles - rem;
    args.split_units = rem;
    args.split_ways = ways;
    args.partials = sc->partials;
    args.sync_words = sc->words;
    args.epoch = next_epoch();
    grid_pairs = args.dp_tiles > 0 ? pairs : rem * ways;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * grid_pairs));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // setup may overlap the previous kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (!cuda_ok(cudaLaunchKernelEx(&cfg, tpk::tp_gemm_kernel<KIND, false, true, MN>, a0, a1, b0, b1, om.y, om.c, args)))
    return TP_ERR_CUDA;
  return launch_status();
}

template <int KIND, bool SWAP, int MN = 0>
int gemm_launch(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0, const CUtensorMap& b1,
                const OutMaps& om, tpk::GemmArgs args, const Scratch* sc, cudaStream_t st) {
  using Cfg = tpk::GemmCfg<KIND, SWAP>;
  if (args.num_tiles <= 0) return TP_OK;
  if constexpr (MN != 0) {
    static_assert(!SWAP, "MN-major operands run as CTA pairs");
    return args.cluster == 2 ? pair_launch<KIND, MN>(a0, a1, b0, b1, om, args, sc, st) : TP_ERR_UNSUPPORTED;
  }
  if constexpr (!SWAP) {
    if (args.cluster > 1) return pair_launch<KIND>(a0, a1, b0, b1, om, args, sc, st);
  }
  if (!smem_attr_set<KIND, SWAP, false>()) return TP_ERR_CUDA;
  int grid = plan_schedule(args, SWAP, sc);
  if (args.sk_iters > 0) {
    // every stream-K range must be non-empty: grid <= sk_iters
    grid = static_cast<int>(std::min<long long>(grid, args.sk_iters));
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // setup may overlap the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!cuda_ok(cudaLaunchKernelEx(&cfg, tpk::tp_gemm_kernel<KIND, SWAP, false>, a0, a1, b0, b1, om.y, om.c, args)))
    return TP_ERR_CUDA;
  return launch_status();
}

// Token-major launches run as CTA pairs (2-SM MMA, 256-token units) when
// there are at least two token blocks and pairing wastes little: an even
// count, or enough blocks that one empty half-unit is a small fraction.
inline int cluster_for(int64_t m_blocks) {
  return (m_blocks >= 2 && (m_blocks % 2 == 0 || m_blocks >= 8)) ? 2 : 1;
}

inline int tpad_of(int64_t T) { return static_cast<int>(cdiv(std::max<int64_t>(T, 1), 16) * 16); }

// Column-parallel bf16 GEMM. `rep` > 1 computes replicated K|V column blocks
// once per group of rep shards (QKV views with kv heads < tp). A non-null
// `ctx` (QKV views only) also receives the single-key attention context.
// With ce_stats, the token-major launch also writes the cross-entropy
// statistics of every (shard, token, 256-column tile) (GemmArgs::ce_stats);
// the caller keeps such launches out of the weight-streaming arrangement.
int col_bf16(const void* X, int64_t T, const tp_shards* W, const tp_shards* Wu, const void* bias,
             const void* bias_up, int act, int concat, void* Y, const Scratch* sc, int rep, int64_t kv_col0,
             void* ctx, cudaStream_t st, const int32_t* ce_labels = nullptr, float* ce_stats = nullptr) {
  const int tp = W->tp;
  const int64_t K = W->K, Ns = W->N / tp;
  const bool swiglu = act == TP_ACT_SWIGLU;
  const bool swap = sc != nullptr && T <= SWAP_MAX_T && !ce_stats;
  if (ce_stats && (swiglu || act != TP_ACT_NONE || ctx)) return TP_ERR_MODE;
  tpk::GemmArgs a{};
  a.M = static_cast<int>(T);
  a.Ns = static_cast<int>(Ns);
  a.tp = tp;
  a.rep = 1;
  a.cluster = 1;
  a.kb_per_shard = static_cast<int>(cdiv(K, 64));
  a.kpt = a.kb_per_shard;
  a.act = act;
  a.out_concat = concat;
  a.bias = bias;
  a.bias_up = static_cast<const bf16*>(bias_up);
  a.out = Y;
  a.ce_labels = ce_labels;
  a.ce_stats = ce_stats;
  if (ctx) {
    a.ctx = static_cast<bf16*>(ctx);
    a.hq = W->hq;
    a.hkv = W->hkv;
    a.hd = W->hd;
  }
  CUtensorMap mx, mw, mu;
  if (swap) {
    a.Tpad = tpad_of(T);
    if (!make_map_bf16(&mx, X, K, T, 1, a.Tpad)) return TP_ERR_CUDA;
    if (!make_map_bf16(&mw, W->data, K, Ns, tp, 128)) return TP_ERR_CUDA;
    if (swiglu && !make_map_bf16(&mu, Wu->data, K, Ns, tp, 128)) return TP_ERR_CUDA;
    if (!swiglu) mu = mw;
    a.m_tiles = static_cast<int>(cdiv(Ns, 128));
    a.n_tiles = 1;
    a.num_tiles = a.m_tiles * tp;
    a.r1_tiles = a.num_tiles;
    static const OutMaps none{};
    return swiglu ? gemm_launch<tpk::GK_COL_SWIGLU, true>(mw, mu, mx, mx, none, a, sc, st)
                  : gemm_launch<tpk::GK_COL, true>(mw, mu, mx, mx, none, a, sc, st);
  }
  const int nout = swiglu ? 128 : 256;
  a.cluster = cluster_for(cdiv(T, 128));
  // each CTA of a pair stages half of each 256-row B block
  if (!make_map_bf16(&mx, X, K, T, 1, 128)) return TP_ERR_CUDA;
  if (!make_map_bf16(&mw, W->data, K, Ns, tp, (swiglu || a.cluster > 1) ? 128 : 256)) return TP_ERR_CUDA;
  if (swiglu && !make_map_bf16(&mu, Wu->data, K, Ns, tp, 128)) return TP_ERR_CUDA;
  if (!swiglu) mu = mw;
  a.m_tiles = static_cast<int>(cdiv(cdiv(T, 128), a.cluster));
  a.n_tiles = static_cast<int>(cdiv(Ns, nout));
  int nq = a.n_tiles;
  if (rep > 1 && !swiglu && tp % rep == 0) {
    nq = static_cast<int>(cdiv(kv_col0, nout));
    if (nq < a.n_tiles) {
      a.rep = rep;
      a.n_q_tiles = nq;
    } else {
      nq = a.n_tiles;
    }
  }
  a.r1_tiles = a.m_tiles * nq * tp;
  a.num_tiles = a.r1_tiles + (a.rep > 1 ? a.m_tiles * (a.n_tiles - nq) * (tp / a.rep) : 0);
  // outputs through staging + bulk tensor stores: per shard [tp][T][Ns] or
  // concatenated [T][tp*Ns] (the same (n, t, s) coordinates, other strides);
  // a context needs whole 64-column chunks inside a head (hd % 64 == 0)
  OutMaps om{};
  const uint64_t es = 2;
  bool ok = a.out_concat
                ? make_store_map(&om.y, Y, false, Ns, T, tp, tp * Ns * es, Ns * es)
                : make_store_map(&om.y, Y, false, Ns, T, tp, Ns * es, T * Ns * es);
  if (ok && ctx) {
    const uint64_t nc = static_cast<uint64_t>(W->hq / tp) * W->hd;
    ok = W->hd % 64 == 0 && make_store_map(&om.c, ctx, false, nc, T, tp, nc * es, T * nc * es);
  }
  a.tma_store = ok ? 1 : 0;
  if (swiglu) return gemm_launch<tpk::GK_COL_SWIGLU, false>(mx, mx, mw, mu, om, a, sc, st);
  return ce_stats ? gemm_launch<tpk::GK_COL_CE, false>(mx, mx, mw, mu, om, a, sc, st)
                  : gemm_launch<tpk::GK_COL, false>(mx, mx, mw, mu, om, a, sc, st);
}

// Row-parallel bf16 GEMM: fused shard sum (partials_out == nullptr) or
// per-shard fp32 contributions.
int row_bf16(const void* Xs, int64_t T, const tp_shards* W, const void* bias, const void* residual,
             void* Y, int out_dtype, float* partials_out, const Scratch* sc, cudaStream_t st) {
  const int tp = W->tp;
  const int64_t Ks = W->K / tp, N = W->N;
  const bool swap = sc != nullptr && T <= SWAP_MAX_T && partials_out == nullptr;
  tpk::GemmArgs a{};
  a.M = static_cast<int>(T);
  a.Ns = static_cast<int>(N);
  a.tp = tp;
  a.rep = 1;
  a.cluster = 1;
  a.kb_per_shard = static_cast<int>(cdiv(Ks, 64));
  a.bias = bias;
  a.residual = residual;
  a.out_f32 = (out_dtype == TP_F32 && partials_out == nullptr) ? 1 : 0;
  CUtensorMap mx, mw;
  if (swap) {
    a.Tpad = tpad_of(T);
    if (!make_map_bf16(&mx, Xs, Ks, T, tp, a.Tpad)) return TP_ERR_CUDA;
    if (!make_map_bf16(&mw, W->data, Ks, N, tp, 128)) return TP_ERR_CUDA;
    a.m_tiles = static_cast<int>(cdiv(N, 128));
    a.n_tiles = 1;
    a.num_tiles = a.m_tiles;
    a.r1_tiles = a.num_tiles;
    a.kpt = a.kb_per_shard * tp;
    a.out = Y;
    static const OutMaps none{};
    return gemm_launch<tpk::GK_ROW_SUM, true>(mw, mw, mx, mx, none, a, sc, st);
  }
  a.cluster = cluster_for(cdiv(T, 128));
  if (!make_map_bf16(&mx, Xs, Ks, T, tp, 128)) return TP_ERR_CUDA;
  if (!make_map_bf16(&mw, W->data, Ks, N, tp, a.cluster > 1 ? 128 : 256)) return TP_ERR_CUDA;
  a.m_tiles = static_cast<int>(cdiv(cdiv(T, 128), a.cluster));
  a.n_tiles = static_cast<int>(cdiv(N, 256));
  if (partials_out) {
    a.num_tiles = a.m_tiles * a.n_tiles * tp;
    a.kpt = a.kb_per_shard;
    a.r1_tiles = a.num_tiles;
    a.out = partials_out;
    OutMaps om{};
    a.tma_store = make_store_map(&om.y, partials_out, true, N, T, tp, N * 4, T * N * 4) ? 1 : 0;
    return gemm_launch<tpk::GK_ROW_PARTIAL, false>(mx, mx, mw, mw, om, a, sc, st);
  }
  a.num_tiles = a.m_tiles * a.n_tiles;
  a.kpt = a.kb_per_shard * tp;
  a.r1_tiles = a.num_tiles;
  a.out = Y;
  OutMaps om{};
  const uint64_t oes = a.out_f32 ? 4 : 2;
  a.tma_store = make_store_map(&om.y, Y, a.out_f32 != 0, N, T, 1, N * oes, T * N * oes) ? 1 : 0;
  return gemm_launch<tpk::GK_ROW_SUM, false>(mx, mx, mw, mw, om, a, sc, st);
}

// GEMMs of the backward (bf16, CTA pairs, operands in either order):
//   COL:     out[s][m][n] = sum_k A_s[m][k] B_s[n][k]  -> [tp][M][Ns]
//   ROW_SUM: out[m][n]    = sum_s sum_k A_s[m][k] B_s[n][k] (+ residual) -> [M][Ns]
// ma / mb are the operands' maps (K-major: box {64, 128}; MN-major: box
// {64, 64}); k_ext is the K extent of one shard. With a_sharded (COL) A is
// per shard and B shared. ma1 / mb1 (ROW_SUM) add a second (A, B) pair
// whose sum goes into the same accumulator.

template <int KIND, int MN>
int gemm_bwd(const CUtensorMap& ma, const CUtensorMap& mb, int64_t M, int64_t Ns, int tp, int64_t k_ext,
             int a_sharded, const void* residual, void* out, const Scratch* sc, cudaStream_t st,
             const CUtensorMap* ma1 = nullptr, const CUtensorMap* mb1 = nullptr) {
  tpk::GemmArgs a{};
  a.M = static_cast<int>(M);
  a.Ns = static_cast<int>(Ns);
  a.tp = tp;
  a.rep = 1;
  a.cluster = 2;
  a.act = TP_ACT_NONE;
  a.two_src = ma1 != nullptr ? 1 : 0;
  a.a_sharded = a_sharded;
  a.residual = residual;
  a.out = out;
  a.kb_per_shard = static_cast<int>(cdiv(k_ext, 64));
  a.kpt = KIND == tpk::GK_ROW_SUM ? a.kb_per_shard * tp * (a.two_src ? 2 : 1) : a.kb_per_shard;
  a.m_tiles = static_cast<int>(cdiv(cdiv(M, 128), 2));
  a.n_tiles = static_cast<int>(cdiv(Ns, 256));
  a.num_tiles = a.m_tiles * a.n_tiles * (KIND == tpk::GK_ROW_SUM ? 1 : tp);
  a.r1_tiles = a.num_tiles;
  OutMaps om{};
  const int d2 = KIND == tpk::GK_ROW_SUM ? 1 : tp;
  a.tma_store = make_store_map(&om.y, out, false, Ns, M, d2, Ns * 2, M * Ns * 2) ? 1 : 0;
  return gemm_launch<KIND, false, MN>(ma, ma1 ? *ma1 : ma, mb, mb1 ? *mb1 : mb, om, a, sc, st);
}

template <int KIND>
int simt_launch(const tpk::SimtArgs& a, int s_tiles, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(cdiv(a.Ns, tpk::SK_BN)), static_cast<unsigned>(cdiv(a.M, tpk::SK_BM)),
                  static_cast<unsigned>(s_tiles));
  tpk::simt_gemm_kernel<KIND><<<grid, tpk::SK_THREADS, 0, st>>>(a);
  return launch_status();
}

int col_f32(const void* X, int64_t T, const tp_shards* W, const tp_shards* Wu, const void* bias,
            const void* bias_up, int act, int concat, void* Y, cudaStream_t st) {
  tpk::SimtArgs a{};
  a.M = static_cast<int>(T);
  a.Ns = static_cast<int>(W->N / W->tp);
  a.Ks = static_cast<int>(W->K);
  a.tp = W->tp;
  a.k_shards = 1;
  a.act = act;
  a.out_concat = concat;
  a.A = static_cast<const float*>(X);
  a.a_shard_stride = 0;
  a.B0 = static_cast<const float*>(W->data);
  a.B1 = Wu ? static_cast<const float*>(Wu->data) : nullptr;
  a.bias = static_cast<const float*>(bias);
  a.bias_up = static_cast<const float*>(bias_up);
  a.out = static_cast<float*>(Y);
  return act == TP_ACT_SWIGLU ? simt_launch<tpk::SK_COL_SWIGLU>(a, W->tp, st)
                              : simt_launch<tpk::SK_COL>(a, W->tp, st);
}

int row_f32(const void* Xs, int64_t T, const tp_shards* W, const void* bias, const void* residual,
            void* Y, float* partials, cudaStream_t st) {
  tpk::SimtArgs a{};
  a.M = static_cast<int>(T);
  a.Ns = static_cast<int>(W->N);
  a.Ks = static_cast<int>(W->K / W->tp);
  a.tp = W->tp;
  a.A = static_cast<const float*>(Xs);
  a.a_shard_stride = T * a.Ks;
  a.B0 = static_cast<const float*>(W->data);
  a.bias = static_cast<const float*>(bias);
  a.residual = static_cast<const float*>(residual);
  if (partials) {
    a.k_shards = 1;
    a.out = partials;
    return simt_launch<tpk::SK_ROW_PARTIAL>(a, W->tp, st);
  }
  a.k_shards = W->tp;
  a.out = static_cast<float*>(Y);
  return simt_launch<tpk::SK_ROW_SUM>(a, 1, st);
}

// Shared validation of a column-linear request.
int check_col(const void* X, int64_t T, const tp_shards* W, const tp_shards* Wu, const void* bias,
              const void* bias_up, int act, int concat, const void* Y) {
  if ((!X || !Y) && T != 0) return TP_ERR_NULL;  // an empty call may pass empty (null) buffers
  int r = check_view(W, TP_COL);
  if (r) return r;
  if (T < 0) return TP_ERR_SHAPE;
  if (T > INT32_MAX) return TP_ERR_UNSUPPORTED;
  if (act < TP_ACT_NONE || act > TP_ACT_SWIGLU) return TP_ERR_MODE;
  if (concat != 0 && concat != 1) return TP_ERR_MODE;
  if (act == TP_ACT_SWIGLU) {
    if (!Wu) return TP_ERR_NULL;
    if ((r = check_view(Wu, TP_COL))) return r;
    if (!same_shape(W, Wu)) return TP_ERR_SHAPE;
  } else if (Wu || bias_up) {
    return TP_ERR_MODE;
  }
  const int dt = W->dtype;
  if (!ptr_ok(X, dt) || !ptr_ok(Y, dt) || !ptr_ok(bias, dt) || !ptr_ok(bias_up, dt)) return TP_ERR_ALIGN;
  return TP_OK;
}

// bias, residual and out are in out_dt: bf16, or fp32 (a residual stream kept
// in fp32 while the GEMM operands are bf16); the fp32 path writes fp32 only.
int check_out_dtype(const tp_shards* W, int out_dt) {
  if (!dtype_ok(out_dt)) return TP_ERR_DTYPE;
  if (W->dtype == TP_F32 && out_dt != TP_F32) return TP_ERR_DTYPE;
  return TP_OK;
}

int check_row(const void* Xs, int64_t T, const tp_shards* W, const void* bias, const void* residual,
              const void* out, int out_dt) {
  if ((!Xs || !out) && T != 0) return TP_ERR_NULL;
  int r = check_view(W, TP_ROW);
  if (r) return r;
  if ((r = check_out_dtype(W, out_dt))) return r;
  if (T < 0) return TP_ERR_SHAPE;
  if (T > INT32_MAX) return TP_ERR_UNSUPPORTED;
  const int dt = W->dtype;
  if (!ptr_ok(Xs, dt) || !ptr_ok(bias, dt) || !ptr_ok(residual, dt) || !ptr_ok(out, dt))
    return TP_ERR_ALIGN;  // bf16 path: 16-byte vectors for every dtype of out
  return TP_OK;
}

int run_col(const void* X, int64_t T, const tp_shards* W, const tp_shards* Wu, const void* bias,
            const void* bias_up, int act, int concat, void* Y, cudaStream_t st, const Scratch* sc = nullptr,
            void* ctx = nullptr) {
  if (T == 0) return TP_OK;
  if (W->dtype != TP_BF16) return col_f32(X, T, W, Wu, bias, bias_up, act, concat, Y, st);
  // A QKV view whose kv heads are replicated (hkv < tp): without a bias the
  // replicas' K|V columns are identical, so each group of tp/hkv shards
  // computes them once and stores them to every shard of the group.
  int rep = 1;
  int64_t kv_col0 = 0;
  if (W->hd > 0 && W->hkv > 0 && W->hkv < W->tp && !bias && !bias_up) {
    rep = W->tp / W->hkv;
    kv_col0 = static_cast<int64_t>(W->hq / W->tp) * W->hd;
  }
  return col_bf16(X, T, W, Wu, bias, bias_up, act, concat, Y, sc, rep, kv_col0, ctx, st);
}

int run_row(const void* Xs, int64_t T, const tp_shards* W, const void* bias, const void* residual,
            void* Y, int out_dtype, float* partials, cudaStream_t st, const Scratch* sc = nullptr) {
  if (T == 0) return TP_OK;
  return W->dtype == TP_BF16 ? row_bf16(Xs, T, W, bias, residual, Y, out_dtype, partials, sc, st)
                             : row_f32(Xs, T, W, bias, residual, Y, partials, st);
}

// Split-tile scratch carved from a caller workspace after `used` bytes:
// fp32 slots and epoch-tagged synchronisation words (no clearing needed) for
// the stream-K schedule of the weight-streaming arrangement (T <= SWAP_MAX_T)
// and for the split last round of paired row GEMMs (larger T).
size_t scratch_bytes(int64_t T, size_t max_tiles) {
  (void)T;
  return align256(SK_PARTIAL_BYTES) + align256(sizeof(unsigned long long) * max_tiles);
}
Scratch carve_scratch(void* ws, size_t used, size_t max_tiles) {
  Scratch sc{};
  char* base = static_cast<char*>(ws) + used;
  sc.partial_bytes = SK_PARTIAL_BYTES;
  sc.partials = reinterpret_cast<float*>(base);
  sc.words = reinterpret_cast<unsigned long long*>(base + align256(sc.partial_bytes));
  sc.nwords = max_tiles;
  return sc;
}
// Counters the MLP's two GEMMs can need: the stream-K part of a normal
// schedule stays under 2 * SK_MAX_CTAS tiles; the swap schedule splits all
// of its tiles.
size_t mlp_max_tiles(int64_t H, int64_t I, int tp) {
  const size_t swap_col = static_cast<size_t>(tp) * cdiv(I / std::max(tp, 1), 128);
  const size_t swap_row = cdiv(H, 128);
  return std::max<size_t>(2 * SK_MAX_CTAS, std::max(swap_col, swap_row));
}
// Attention core over qkv [tp][T][(nq + 2 nkv) * hd] (q | k | v per
// shard) into ctx [tp][T][nq * hd]; mode TP_ATTN_CAUSAL or TP_ATTN_FULL,
// hd 64 or 128.
template <int HD>
int attention_launch_hd(const void* qkv, int64_t T, int tp, int hq, int hkv, int mode, void* ctx, cudaStream_t st) {
  using Cfg = tpk::AttnCfg<HD>;
  const int nq = hq / tp, nkv = hkv >= tp ? hkv / tp : 1;
  const int64_t nqkv = static_cast<int64_t>(nq + 2 * nkv) * HD;
  CUtensorMap m, mc;
  if (!make_map_bf16(&m, qkv, nqkv, T, tp, 128)) return TP_ERR_CUDA;
  const uint64_t nc = static_cast<uint64_t>(nq) * HD;  // context columns of a shard
  if (!make_store_map(&mc, ctx, false, nc, static_cast<uint64_t>(T), static_cast<uint64_t>(tp), nc * 2,
                      nc * 2 * static_cast<uint64_t>(T)))
    return TP_ERR_CUDA;
  tpk::AttnArgs a{};
  a.ctx = static_cast<bf16*>(ctx);
  a.T = static_cast<int>(T);
  a.tp = tp;
  a.hq = hq;
  a.hkv = hkv;
  a.nq = nq;
  a.nkv = nkv;
  a.group = hq / hkv;
  a.causal = mode == TP_ATTN_CAUSAL ? 1 : 0;
  a.q_blocks = static_cast<int>(cdiv(T, 128));
  // two q heads of one kv head share a unit when the shard's heads pair up
  // that way (an even group, an even count per shard); else two query blocks
  a.pair_heads = (a.group % 2 == 0 && nq % 2 == 0) ? 1 : 0;
  a.units = a.pair_heads ? a.q_blocks * tp * (nq / 2) : static_cast<int>((a.q_blocks + 1) / 2) * tp * nq;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HD)));
  static bool attr_done[128] = {};
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev)) || dev < 0 || dev >= 128) return TP_ERR_CUDA;
  if (!attr_done[dev]) {
    if (!cuda_ok(cudaFuncSetAttribute(tpk::tp_attn_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM)))
      return TP_ERR_CUDA;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  // persistent: one CTA per SM (each holds all of its SM's TMEM), none idle
  cfg.gridDim = dim3(static_cast<unsigned>(std::min(a.units, std::max(1, num_sms()))));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!cuda_ok(cudaLaunchKernelEx(&cfg, tpk::tp_attn_kernel<HD>, m, mc, a))) return TP_ERR_CUDA;
  return launch_status();
}

inline bool attention_hd_ok(int hd) { return hd == 64 || hd == 128; }

int attention_launch(const void* qkv, int64_t T, int tp, int hq, int hkv, int hd, int mode, void* ctx,
                     cudaStream_t st) {
  if (hd == 64) return attention_launch_hd<64>(qkv, T, tp, hq, hkv, mode, ctx, st);
  if (hd == 128) return attention_launch_hd<128>(qkv, T, tp, hq, hkv, mode, ctx, st);
  return TP_ERR_UNSUPPORTED;
}

size_t attn_max_tiles(int64_t H, int hq, int hkv, int hd, int tp) {
  const int64_t nkv = hkv >= tp ? hkv / tp : 1;
  const size_t swap_col = static_cast<size_t>(tp) * cdiv((hq / tp + 2 * nkv) * hd, 128);
  return std::max<size_t>(2 * SK_MAX_CTAS, std::max(swap_col, static_cast<size_t>(cdiv(H, 128))));
}

}  // namespace

// ===========================================================================
// Exported C ABI
// ===========================================================================
extern "C" {

const char* tp_status_string(tp_status s) {
  switch (s) {
    case TP_OK: return "ok";
    case TP_ERR_NULL: return "null pointer";
    case TP_ERR_SHAPE: return "bad shape (size < 1, not divisible by tp, or mismatched)";
    case TP_ERR_DTYPE: return "bad or mismatched dtype";
    case TP_ERR_MODE: return "bad mode, activation, reduce op or flag";
    case TP_ERR_ALIGN: return "alignment rule broken (bf16: 16-byte pointers, widths % 8)";
    case TP_ERR_WORKSPACE: return "workspace or output buffer too small";
    case TP_ERR_CUDA: return "CUDA error";
    case TP_ERR_TIMEOUT: return "bounded device wait expired";
    case TP_ERR_UNSUPPORTED: return "unsupported size";
    case TP_ERR_INDEX: return "token id or label outside [0, V)";
    default: return "unknown status";
  }
}

int tp_abi_version(void) { return 1; }

tp_status tp_shard_weights(const void* W, int64_t K, int64_t N, int dtype, int tp, int mode, void* out,
                           size_t out_bytes, tp_shards* view, void* stream) {
  if (!W || !out) return TP_ERR_NULL;
  if (!dtype_ok(dtype)) return TP_ERR_DTYPE;
  if (mode != TP_COL && mode != TP_ROW) return TP_ERR_MODE;
  if (tp < 1 || K < 1 || N < 1) return TP_ERR_SHAPE;
  if ((mode == TP_COL && N % tp) || (mode == TP_ROW && K % tp)) return TP_ERR_SHAPE;
  if (K > INT32_MAX || N > INT32_MAX) return TP_ERR_UNSUPPORTED;
  const size_t need = static_cast<size_t>(K) * static_cast<size_t>(N) * elem_size(dtype);
  if (out_bytes < need) return TP_ERR_WORKSPACE;
  if (dtype == TP_BF16) {
    const int64_t inner = mode == TP_COL ? K : K / tp, outw = mode == TP_COL ? N / tp : N;
    if (inner % 8 || outw % 8 || !aligned(W, 16) || !aligned(out, 16)) return TP_ERR_ALIGN;
  } else if (!aligned(W, 4) || !aligned(out, 4)) {
    return TP_ERR_ALIGN;
  }
  const dim3 grid(static_cast<unsigned>(cdiv(N, 32)), static_cast<unsigned>(cdiv(K, 32)));
  const int64_t Ks = mode == TP_ROW ? K / tp : K;
  if (dtype == TP_BF16)
    tpk::shard_weights_kernel<bf16><<<grid, 256, 0, as_stream(stream)>>>(
        static_cast<const bf16*>(W), K, N, Ks, mode == TP_ROW, static_cast<bf16*>(out));
  else
    tpk::shard_weights_kernel<float><<<grid, 256, 0, as_stream(stream)>>>(
        static_cast<const float*>(W), K, N, Ks, mode == TP_ROW, static_cast<float*>(out));
  const int r = launch_status();
  if (r == TP_OK && view) {
    *view = tp_shards{};
    view->data = out;
    view->K = K;
    view->N = N;
    view->tp = tp;
    view->mode = mode;
    view->dtype = dtype;
  }
  return as_status(r);
}

size_t tp_qkv_shard_elems(int64_t H, int hq, int hkv, int hd, int tp) {
  if (H < 1 || hq < 1 || hkv < 1 || hd < 1 || tp < 1) return 0;
  if (hq % tp || hq % hkv) return 0;
  if (hkv >= tp ? (hkv % tp != 0) : (tp % hkv != 0)) return 0;
  const int64_t nkv = hkv >= tp ? hkv / tp : 1;
  return static_cast<size_t>(tp) * static_cast<size_t>((hq / tp + 2 * nkv) * hd) * static_cast<size_t>(H);
}

tp_status tp_shard_qkv(const void* Wq, const void* Wk, const void* Wv, int64_t H, int hq, int hkv, int hd,
                       int tp, int dtype, void* out, size_t out_bytes, tp_shards* view, void* stream) {
  if (!Wq || !Wk || !Wv || !out) return TP_ERR_NULL;
  if (!dtype_ok(dtype)) return TP_ERR_DTYPE;
  const size_t elems = tp_qkv_shard_elems(H, hq, hkv, hd, tp);
  if (elems == 0) return TP_ERR_SHAPE;
  if (H > INT32_MAX) return TP_ERR_UNSUPPORTED;
  if (out_bytes < elems * elem_size(dtype)) return TP_ERR_WORKSPACE;
  const int64_t nkv = hkv >= tp ? hkv / tp : 1;
  const int64_t Ns = (hq / tp + 2 * nkv) * hd;
  if (dtype == TP_BF16) {
    if (H % 8 || Ns % 8 || hd % 8) return TP_ERR_ALIGN;
    for (const void* p : {Wq, Wk, Wv, static_cast<const void*>(out)})
      if (!aligned(p, 16)) return TP_ERR_ALIGN;
  } else {
    for (const void* p : {Wq, Wk, Wv, static_cast<const void*>(out)})
      if (!aligned(p, 4)) return TP_ERR_ALIGN;
  }
  const dim3 grid(static_cast<unsigned>(cdiv(Ns, 32)), static_cast<unsigned>(cdiv(H, 32)),
                  static_cast<unsigned>(tp));
  if (dtype == TP_BF16)
    tpk::shard_qkv_kernel<bf16><<<grid, 256, 0, as_stream(stream)>>>(
        static_cast<const bf16*>(Wq), static_cast<const bf16*>(Wk), static_cast<const bf16*>(Wv), H,
        hq, hkv, hd, tp, static_cast<bf16*>(out));
  else
    tpk::shard_qkv_kernel<float><<<grid, 256, 0, as_stream(stream)>>>(
        static_cast<const float*>(Wq), static_cast<const float*>(Wk), static_cast<const float*>(Wv),
        H, hq, hkv, hd, tp, static_cast<float*>(out));
  const int r = launch_status();
  if (r == TP_OK && view) {
    *view = tp_shards{};
    view->data = out;
    view->K = H;
    view->N = tp * Ns;
    view->tp = tp;
    view->mode = TP_COL;
    view->dtype = dtype;
    view->hq = hq;
    view->hkv = hkv;
    view->hd = hd;
  }
  return as_status(r);
}

size_t tp_gemm_workspace_bytes(int64_t T, const tp_shards* W) {
  if (!W || T < 0 || W->dtype != TP_BF16 || W->tp < 1 || W->K < 1 || W->N < 1) return 0;
  size_t tiles;
  if (W->mode == TP_COL) tiles = static_cast<size_t>(W->tp) * cdiv(W->N / W->tp, 128);
  else if (W->mode == TP_ROW) tiles = cdiv(W->N, 128);
  else return 0;
  return scratch_bytes(T, std::max<size_t>(2 * SK_MAX_CTAS, tiles));
}

// Optional caller scratch for a single linear: NULL -> whole tiles only.
int linear_scratch(const tp_shards* W, int64_t T, void* ws, size_t ws_bytes, Scratch* sc, const Scratch** scp) {
  *scp = nullptr;
  if (!ws || W->dtype != TP_BF16) return TP_OK;
  if (!aligned(ws, 256)) return TP_ERR_ALIGN;
  const size_t need = tp_gemm_workspace_bytes(T, W);
  if (ws_bytes < need) return TP_ERR_WORKSPACE;
  const size_t tiles = W->mode == TP_COL ? static_cast<size_t>(W->tp) * cdiv(W->N / W->tp, 128)
                                         : static_cast<size_t>(cdiv(W->N, 128));
  *sc = carve_scratch(ws, 0, std::max<size_t>(2 * SK_MAX_CTAS, tiles));
  *scp = sc;
  return TP_OK;
}

tp_status tp_column_linear(const void* X, int64_t T, const tp_shards* W, const tp_shards* W_up,
                           const void* bias, const void* bias_up, int act, int concat, void* Y,
                           void* workspace, size_t ws_bytes, void* stream) {
  int r = check_col(X, T, W, W_up, bias, bias_up, act, concat, Y);
  if (r) return as_status(r);
  Scratch sc{};
  const Scratch* scp;
  if ((r = linear_scratch(W, T, workspace, ws_bytes, &sc, &scp))) return as_status(r);
  return as_status(run_col(X, T, W, W_up, bias, bias_up, act, concat, Y, as_stream(stream), scp));
}

tp_status tp_row_linear(const void* Xs, int64_t T, const tp_shards* W, const void* bias,
                        const void* residual, void* Y, int out_dtype, void* workspace, size_t ws_bytes,
                        void* stream) {
  int r = check_row(Xs, T, W, bias, residual, Y, out_dtype);
  if (r) return as_status(r);
  Scratch sc{};
  const Scratch* scp;
  if ((r = linear_scratch(W, T, workspace, ws_bytes, &sc, &scp))) return as_status(r);
  return as_status(run_row(Xs, T, W, bias, residual, Y, out_dtype, nullptr, as_stream(stream), scp));
}

tp_status tp_row_linear_partials(const void* Xs, int64_t T, const tp_shards* W, float* partials,
                                 void* stream) {
  const int r = check_row(Xs, T, W, nullptr, nullptr, partials, TP_F32);
  if (r) return as_status(r);
  return as_status(run_row(Xs, T, W, nullptr, nullptr, nullptr, TP_F32, partials, as_stream(stream)));
}

tp_status tp_shard_reduce(const float* partials, int tp, int64_t T, int64_t N, int op, const void* bias,
                          const void* residual, int out_dtype, void* out, void* stream) {
  if (!partials || !out) return TP_ERR_NULL;
  if (op != TP_REDUCE_SUM && op != TP_REDUCE_SCATTER) return TP_ERR_MODE;
  if (!dtype_ok(out_dtype)) return TP_ERR_DTYPE;
  if (tp < 1 || T < 0 || N < 1) return TP_ERR_SHAPE;
  if (op == TP_REDUCE_SCATTER && T % tp) return TP_ERR_SHAPE;
  if (T == 0) return TP_OK;
  const bool vec = (N % 4 == 0);
  if (vec) {
    if (!aligned(partials, 16)) return TP_ERR_ALIGN;
  } else if (!aligned(partials, 4)) {
    return TP_ERR_ALIGN;
  }
  for (const void* p : {bias, residual, static_cast<const void*>(out)})
    if (p && !aligned(p, elem_size(out_dtype))) return TP_ERR_ALIGN;
  const cudaStream_t st = as_stream(stream);
  const int64_t work = vec ? T * N / 4 : T * N;
  const int grid = grid_for(work, 256);
  if (out_dtype == TP_BF16) {
    auto b = static_cast<const bf16*>(bias);
    auto rr = static_cast<const bf16*>(residual);
    auto o = static_cast<bf16*>(out);
    if (vec) tpk::reduce_kernel<bf16><<<grid, 256, 0, st>>>(partials, tp, T, N, b, rr, o);
    else tpk::reduce_kernel_scalar<bf16><<<grid, 256, 0, st>>>(partials, tp, T, N, b, rr, o);
  } else {
    auto b = static_cast<const float*>(bias);
    auto rr = static_cast<const float*>(residual);
    auto o = static_cast<float*>(out);
    if (vec) tpk::reduce_kernel<float><<<grid, 256, 0, st>>>(partials, tp, T, N, b, rr, o);
    else tpk::reduce_kernel_scalar<float><<<grid, 256, 0, st>>>(partials, tp, T, N, b, rr, o);
  }
  return as_status(launch_status());
}

tp_status tp_shard_gather(const void* shards, int tp, int64_t T, int64_t N, int dtype, void* out,
                          void* stream) {
  if (!shards || !out) return TP_ERR_NULL;
  if (!dtype_ok(dtype)) return TP_ERR_DTYPE;
  if (tp < 1 || T < 0 || N < 1 || N % tp) return TP_ERR_SHAPE;
  if (T == 0) return TP_OK;
  const int64_t Ns = N / tp;
  const size_t es = elem_size(dtype);
  const bool vec = (Ns * es) % 16 == 0 && aligned(shards, 16) && aligned(out, 16);
  if (!aligned(shards, es) || !aligned(out, es)) return TP_ERR_ALIGN;
  const cudaStream_t st = as_stream(stream);
  if (dtype == TP_BF16) {
    auto in = static_cast<const bf16*>(shards);
    auto o = static_cast<bf16*>(out);
    if (vec) tpk::gather_kernel<bf16, 8><<<grid_for(tp * T * Ns / 8, 256), 256, 0, st>>>(in, tp, T, Ns, o);
    else tpk::gather_kernel<bf16, 1><<<grid_for(tp * T * Ns, 256), 256, 0, st>>>(in, tp, T, Ns, o);
  } else {
    auto in = static_cast<const float*>(shards);
    auto o = static_cast<float*>(out);
    if (vec) tpk::gather_kernel<float, 4><<<grid_for(tp * T * Ns / 4, 256), 256, 0, st>>>(in, tp, T, Ns, o);
    else tpk::gather_kernel<float, 1><<<grid_for(tp * T * Ns, 256), 256, 0, st>>>(in, tp, T, Ns, o);
  }
  return as_status(launch_status());
}

size_t tp_mlp_workspace_bytes(int64_t T, int64_t H, int64_t I, int tp, int dtype) {
  if (T < 0 || H < 1 || I < 1 || tp < 1 || !dtype_ok(dtype)) return 0;
  size_t b = align256(static_cast<size_t>(T) * static_cast<size_t>(I) * elem_size(dtype));
  if (dtype == TP_BF16) b += scratch_bytes(T, mlp_max_tiles(H, I, tp));
  return b;
}

tp_status tp_mlp_block(const void* X, int64_t T, const tp_shards* W1, const tp_shards* W_up,
                       const tp_shards* W2, const void* b1, const void* b1_up, const void* b2,
                       const void* residual, int act, int out_dtype, void* workspace, size_t ws_bytes,
                       void* Y, void* stream) {
  if (!W2 || (!workspace && T != 0)) return TP_ERR_NULL;
  int r = check_col(X, T, W1, W_up, b1, b1_up, act, 0, Y);
  if (r) return as_status(r);
  if ((r = check_view(W2, TP_ROW))) return as_status(r);
  if ((r = check_out_dtype(W2, out_dtype))) return as_status(r);
  if (W2->dtype != W1->dtype) return TP_ERR_DTYPE;
  if (W2->tp != W1->tp || W2->K != W1->N || W2->N != W1->K) return TP_ERR_SHAPE;
  const int dt = W1->dtype;
  if (!ptr_ok(b2, dt) || !ptr_ok(residual, dt) || !aligned(workspace, 256)) return TP_ERR_ALIGN;
  if (ws_bytes < tp_mlp_workspace_bytes(T, W1->K, W1->N, W1->tp, dt)) return TP_ERR_WORKSPACE;
  if (T == 0) return TP_OK;
  const cudaStream_t st = as_stream(stream);
  void* Hs = workspace;  // [tp][T][I/tp]
  const size_t hs_bytes = align256(static_cast<size_t>(T) * W1->N * elem_size(dt));
  Scratch sc{};
  const Scratch* scp = nullptr;
  if (dt == TP_BF16) {
    sc = carve_scratch(workspace, hs_bytes, mlp_max_tiles(W1->K, W1->N, W1->tp));
    scp = &sc;
  }
  if ((r = run_col(X, T, W1, W_up, b1, b1_up, act, 0, Hs, st, scp))) return as_status(r);
  return as_status(run_row(Hs, T, W2, b2, residual, Y, out_dtype, nullptr, st, scp));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Static workspace for tp_mlp_block_static (callers that cannot allocate)
// ---------------------------------------------------------------------------
// The array lives in this module's static device memory. In host code its
// name is only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and cached.
static __device__ __align__(256) unsigned char g_static_workspace[TP_STATIC_WORKSPACE_BYTES];

namespace {
std::mutex g_static_mu;
void* g_static_ptr[128] = {};

int static_workspace(void** out) {
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev))) return TP_ERR_CUDA;
  if (dev < 0 || dev >= 128) return TP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (!cuda_ok(cudaGetSymbolAddress(&p, g_static_workspace)) || !p) return TP_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return TP_OK;
}
}  // namespace

extern "C" {

tp_status tp_mlp_block_static(const void* X, int64_t T, const tp_shards* W1, const tp_shards* W_up,
                              const tp_shards* W2, const void* b1, const void* b1_up, const void* b2,
                              const void* residual, int act, int out_dtype, void* Y, void* stream) {
  if (!W1 || !W2) return TP_ERR_NULL;
  // sizes beyond the static array are refused before anything else happens
  if (tp_mlp_workspace_bytes(T, W1->K, W1->N, W1->tp, W1->dtype) > TP_STATIC_WORKSPACE_BYTES)
    return TP_ERR_WORKSPACE;
  void* ws = nullptr;
  const int r = static_workspace(&ws);
  if (r) return as_status(r);
  return tp_mlp_block(X, T, W1, W_up, W2, b1, b1_up, b2, residual, act, out_dtype, ws,
                      TP_STATIC_WORKSPACE_BYTES, Y, stream);
}

size_t tp_attn_workspace_bytes(int64_t T, int hq, int hkv, int hd, int tp, int dtype) {
  if (T < 0 || !dtype_ok(dtype)) return 0;
  const size_t qkv = tp_qkv_shard_elems(1, hq, hkv, hd, tp);  // per token, all shards
  if (qkv == 0) return 0;
  const size_t es = elem_size(dtype);
  const size_t ctx = static_cast<size_t>(hq) * hd;  // per token, all shards
  size_t b = align256(static_cast<size_t>(T) * qkv * es) + align256(static_cast<size_t>(T) * ctx * es);
  // the stream-K scratch is sized for the largest hidden size the O projection may have
  if (dtype == TP_BF16) b += scratch_bytes(T, attn_max_tiles(static_cast<int64_t>(hq) * hd * 4, hq, hkv, hd, tp));
  return b;
}

}  // extern "C"

namespace {
// QKV by heads -> attention core (caller context, single-key stand-in or the
// causal / full core) -> O and the shard sum.
int attn_block_impl(const void* X, int64_t T, const tp_shards* Wqkv, const tp_shards* Wo, const void* ctx,
                    int mode, const void* residual, int out_dtype, void* qkv_out, void* workspace,
                    size_t ws_bytes, void* Y, void* stream) {
  if (!Wo || !Wqkv || (!workspace && T != 0)) return TP_ERR_NULL;
  int r = check_col(X, T, Wqkv, nullptr, nullptr, nullptr, TP_ACT_NONE, 0, Y);
  if (r) return r;
  if (Wqkv->hd < 1 || Wqkv->hq < 1 || Wqkv->hkv < 1) return TP_ERR_MODE;  // not a QKV view
  const int tp = Wqkv->tp, hq = Wqkv->hq, hkv = Wqkv->hkv, hd = Wqkv->hd;
  if (tp_qkv_shard_elems(Wqkv->K, hq, hkv, hd, tp) != static_cast<size_t>(Wqkv->K) * Wqkv->N)
    return TP_ERR_SHAPE;
  if ((r = check_view(Wo, TP_ROW))) return r;
  if (Wo->dtype != Wqkv->dtype) return TP_ERR_DTYPE;
  if ((r = check_out_dtype(Wo, out_dtype))) return r;
  if (Wo->tp != tp || Wo->K != static_cast<int64_t>(hq) * hd || Wo->N != Wqkv->K) return TP_ERR_SHAPE;
  const int dt = Wqkv->dtype;
  if (!ptr_ok(ctx, dt) || !ptr_ok(residual, dt) || !ptr_ok(qkv_out, dt) || !aligned(workspace, 256))
    return TP_ERR_ALIGN;
  if (dt == TP_BF16 && hd % 8) return TP_ERR_ALIGN;
  if (Wqkv->K > static_cast<int64_t>(hq) * hd * 4) return TP_ERR_UNSUPPORTED;  // scratch sizing bound
  if (mode != TP_ATTN_SINGLE_KEY && mode != TP_ATTN_CAUSAL && mode != TP_ATTN_FULL) return TP_ERR_MODE;
  if (mode != TP_ATTN_SINGLE_KEY && (dt != TP_BF16 || !attention_hd_ok(hd))) return TP_ERR_UNSUPPORTED;
  if (mode != TP_ATTN_SINGLE_KEY && static_cast<int64_t>(hq) * cdiv(T, 128) > INT32_MAX / 2)
    return TP_ERR_UNSUPPORTED;  // the core counts its work units in int
  if (ws_bytes < tp_attn_workspace_bytes(T, hq, hkv, hd, tp, dt)) return TP_ERR_WORKSPACE;
  if (T == 0) return TP_OK;
  const cudaStream_t st = as_stream(stream);
  const size_t es = elem_size(dt);
  const size_t qkv_bytes = align256(static_cast<size_t>(T) * tp_qkv_shard_elems(1, hq, hkv, hd, tp) * es);
  const size_t ctx_bytes = align256(static_cast<size_t>(T) * hq * hd * es);
  void* qkv = qkv_out ? qkv_out : workspace;
  void* ctx_ws = static_cast<char*>(workspace) + qkv_bytes;
  Scratch sc{};
  const Scratch* scp = nullptr;
  if (dt == TP_BF16) {
    sc = carve_scratch(workspace, qkv_bytes + ctx_bytes,
                       attn_max_tiles(static_cast<int64_t>(hq) * hd * 4, hq, hkv, hd, tp));
    scp = &sc;
  }
  if (mode != TP_ATTN_SINGLE_KEY) {
    if ((r = run_col(X, T, Wqkv, nullptr, nullptr, nullptr, TP_ACT_NONE, 0, qkv, st, scp))) return r;
    if ((r = attention_launch(qkv, T, tp, hq, hkv, hd, mode, ctx_ws, st))) return r;
    return run_row(ctx_ws, T, Wo, nullptr, residual, Y, out_dtype, nullptr, st, scp);
  }
  // Without a caller context the single-key stand-in is used: on the bf16
  // path the QKV epilogue writes it from the V columns it has just computed;
  // the fp32 path copies it from qkv with a separate kernel.
  const bool fused_ctx = !ctx && dt == TP_BF16;
  if ((r = run_col(X, T, Wqkv, nullptr, nullptr, nullptr, TP_ACT_NONE, 0, qkv, st, scp,
                   fused_ctx ? ctx_ws : nullptr)))
    return r;
  if (!ctx && !fused_ctx) {
    const dim3 block(32, 8);
    const dim3 grid(static_cast<unsigned>(cdiv(static_cast<int64_t>(tp) * T, 8)));
    tpk::ctx_standin_kernel<float><<<grid, block, 0, st>>>(
        static_cast<const float*>(qkv), tp, T, hq, hkv, hd, static_cast<float*>(ctx_ws));
    if ((r = launch_status())) return r;
  }
  if (!ctx) ctx = ctx_ws;
  return run_row(ctx, T, Wo, nullptr, residual, Y, out_dtype, nullptr, st, scp);
}

}  // namespace

extern "C" {

tp_status tp_attn_proj(const void* X, int64_t T, const tp_shards* Wqkv, const tp_shards* Wo,
                       const void* ctx, const void* residual, int out_dtype, void* qkv_out, void* workspace,
                       size_t ws_bytes, void* Y, void* stream) {
  return as_status(attn_block_impl(X, T, Wqkv, Wo, ctx, TP_ATTN_SINGLE_KEY, residual, out_dtype,
                                                qkv_out, workspace, ws_bytes, Y, stream));
}

tp_status tp_attn_block(const void* X, int64_t T, const tp_shards* Wqkv, const tp_shards* Wo, int mode,
                        const void* residual, int out_dtype, void* qkv_out, void* workspace, size_t ws_bytes, void* Y,
                        void* stream) {
  return as_status(attn_block_impl(X, T, Wqkv, Wo, nullptr, mode, residual, out_dtype, qkv_out,
                                                workspace, ws_bytes, Y, stream));
}

tp_status tp_attention(const void* qkv, int64_t T, int tp, int hq, int hkv, int hd, int mode, void* ctx, void* stream) {
  if ((!qkv || !ctx) && T != 0) return TP_ERR_NULL;
  if (mode != TP_ATTN_CAUSAL && mode != TP_ATTN_FULL) return TP_ERR_MODE;
  if (T < 0 || tp < 1 || hq < 1 || hkv < 1 || hd < 1 || tp_qkv_shard_elems(1, hq, hkv, hd, tp) == 0)
    return TP_ERR_SHAPE;
  // (work units, one per shard, q head and 128 queries, are counted in int)
  if (!attention_hd_ok(hd) || T > INT32_MAX || static_cast<int64_t>(hq) * cdiv(T, 128) > INT32_MAX / 2)
    return TP_ERR_UNSUPPORTED;
  if (!ptr_ok(qkv, TP_BF16) || !ptr_ok(ctx, TP_BF16)) return TP_ERR_ALIGN;
  if (T == 0) return TP_OK;
  return as_status(attention_launch(qkv, T, tp, hq, hkv, hd, mode, ctx, as_stream(stream)));
}

tp_status tp_rmsnorm(const void* X, const void* gamma, int64_t T, int64_t H, float eps, int dtype, void* Y,
                     int out_dtype, void* stream) {
  if ((!X || !Y) && T != 0) return TP_ERR_NULL;
  if (!dtype_ok(dtype) || !dtype_ok(out_dtype)) return TP_ERR_DTYPE;
  if (T < 0 || H < 1 || !(eps >= 0.0f)) return TP_ERR_SHAPE;
  if (T > INT32_MAX) return TP_ERR_UNSUPPORTED;
  for (const void* p : {X, gamma})
    if (p && !aligned(p, elem_size(dtype))) return TP_ERR_ALIGN;
  if (Y && !aligned(Y, elem_size(out_dtype))) return TP_ERR_ALIGN;
  if (T == 0) return TP_OK;
  const cudaStream_t st = as_stream(stream);
  const unsigned grid = static_cast<unsigned>(T);
  if (dtype == TP_BF16 && out_dtype == TP_BF16)
    tpk::rmsnorm_kernel<bf16, bf16><<<grid, 256, 0, st>>>(
        static_cast<const bf16*>(X), static_cast<const bf16*>(gamma), H, eps, static_cast<bf16*>(Y));
  else if (dtype == TP_BF16)
    tpk::rmsnorm_kernel<bf16, float><<<grid, 256, 0, st>>>(
        static_cast<const bf16*>(X), static_cast<const bf16*>(gamma), H, eps, static_cast<float*>(Y));
  else if (out_dtype == TP_BF16)
    tpk::rmsnorm_kernel<float, bf16><<<grid, 256, 0, st>>>(
        static_cast<const float*>(X), static_cast<const float*>(gamma), H, eps, static_cast<bf16*>(Y));
  else
    tpk::rmsnorm_kernel<float, float><<<grid, 256, 0, st>>>(
        static_cast<const float*>(X), static_cast<const float*>(gamma), H, eps, static_cast<float*>(Y));
  return as_status(launch_status());
}

int tp_last_cuda_error(void) { return g_last_cuda_error; }

const char* tp_cuda_error_name(int code) {
  const char* name = cudaGetErrorName(static_cast<cudaError_t>(code));
  return name ? name : "unrecognised CUDA error code";
}

tp_status tp_get_error(void* stream) {
  if (!cuda_ok(cudaStreamSynchronize(as_stream(stream)))) return TP_ERR_CUDA;
  int err = 0;
  if (!cuda_ok(cudaMemcpyFromSymbol(&err, tpk::g_tp_error, sizeof(int)))) return TP_ERR_CUDA;
  if (err != 0) {
    const int zero = 0;
    if (!cuda_ok(cudaMemcpyToSymbol(tpk::g_tp_error, &zero, sizeof(int)))) return TP_ERR_CUDA;
    return err == tpk::TP_DEVERR_WAIT_TIMEOUT ? TP_ERR_TIMEOUT
           : err == tpk::TP_DEVERR_INDEX      ? TP_ERR_INDEX
                                              : TP_ERR_CUDA;
  }
  return TP_OK;
}

tp_status tp_debug_set_wait_limit_ns(uint64_t ns) {
  const unsigned long long v = ns;
  return cuda_ok(cudaMemcpyToSymbol(tpk::g_tp_wait_limit_ns, &v, sizeof(v))) ? TP_OK : TP_ERR_CUDA;
}

tp_status tp_debug_inject(int kind) {
  if (kind < 0 || kind > 2) return TP_ERR_MODE;
  return cuda_ok(cudaMemcpyToSymbol(tpk::g_tp_inject, &kind, sizeof(int))) ? TP_OK : TP_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward of the column/row pair (bf16, tensor cores, CTA pairs)
// ---------------------------------------------------------------------------
namespace {

int check_bwd_view(const tp_shards* W, int mode) { return check_view(W, mode); }

// --- fp32 backward: the strided FFMA GEMM (exact on integer inputs) ---------
int simt_g_launch(const tpk::SimtGArgs& a, int z, cudaStream_t st) {
  if (a.M <= 0 || a.N <= 0 || z <= 0) return TP_OK;
  const dim3 grid(static_cast<unsigned>(cdiv(a.N, tpk::SK_BN)), static_cast<unsigned>(cdiv(a.M, tpk::SK_BM)),
                  static_cast<unsigned>(z));
  tpk::simt_gemm_strided_kernel<<<grid, tpk::SK_THREADS, 0, st>>>(a);
  return launch_status();
}
// Row layer on fp32 (view [tp][N][Ks], dY [T][N], Xs [tp][T][Ks]):
// dXs_s = dY W_s^T, dW_s = (Xs_s^T dY)^T in the view's storage layout.
int row_bwd_f32(const void* Xs, int64_t T, const tp_shards* W, const void* dY, void* dXs, void* dW,
                cudaStream_t st) {
  const int tp = W->tp;
  const int64_t N = W->N, Ks = W->K / tp;
  int r;
  if (dXs) {
    tpk::SimtGArgs a{};
    a.M = static_cast<int>(T), a.N = static_cast<int>(Ks), a.K = static_cast<int>(N), a.Q = 1;
    a.A = static_cast<const float*>(dY), a.a_m = N, a.a_k = 1;
    a.B = static_cast<const float*>(W->data), a.b_k = Ks, a.b_n = 1, a.b_z = N * Ks;
    a.C = static_cast<float*>(dXs), a.c_m = Ks, a.c_n = 1, a.c_z = T * Ks;
    if ((r = simt_g_launch(a, tp, st))) return r;
  }
  if (dW) {
    tpk::SimtGArgs a{};
    a.M = static_cast<int>(N), a.N = static_cast<int>(Ks), a.K = static_cast<int>(T), a.Q = 1;
    a.A = static_cast<const float*>(dY), a.a_m = 1, a.a_k = N;
    a.B = static_cast<const float*>(Xs), a.b_k = Ks, a.b_n = 1, a.b_z = T * Ks;
    a.C = static_cast<float*>(dW), a.c_m = Ks, a.c_n = 1, a.c_z = N * Ks;
    if ((r = simt_g_launch(a, tp, st))) return r;
  }
  return TP_OK;
}
// Column layer on fp32 (view [tp][Ns][K], dYs [tp][T][Ns], X [T][K]):
// dX = sum_s dYs_s W_s^T (+ add, which may be dX itself), dW_s = (X^T dYs_s)^T.
int col_bwd_f32(const void* X, int64_t T, const tp_shards* W, const void* dYs, const void* add, void* dX,
                void* dW, cudaStream_t st) {
  const int tp = W->tp;
  const int64_t K = W->K, Ns = W->N / tp;
  int r;
  if (dX) {
    tpk::SimtGArgs a{};
    a.M = static_cast<int>(T), a.N = static_cast<int>(K), a.K = static_cast<int>(Ns), a.Q = tp;
    a.A = static_cast<const float*>(dYs), a.a_m = Ns, a.a_k = 1, a.a_q = T * Ns;
    a.B = static_cast<const float*>(W->data), a.b_k = K, a.b_n = 1, a.b_q = Ns * K;
    a.C = static_cast<float*>(dX), a.c_m = K, a.c_n = 1;
    a.add = static_cast<const float*>(add);
    if ((r = simt_g_launch(a, 1, st))) return r;
  }
  if (dW) {
    tpk::SimtGArgs a{};
    a.M = static_cast<int>(Ns), a.N = static_cast<int>(K), a.K = static_cast<int>(T), a.Q = 1;
    a.A = static_cast<const float*>(dYs), a.a_m = 1, a.a_k = Ns, a.a_z = T * Ns;
    a.B = static_cast<const float*>(X), a.b_k = K, a.b_n = 1;
    a.C = static_cast<float*>(dW), a.c_m = K, a.c_n = 1, a.c_z = Ns * K;
    if ((r = simt_g_launch(a, tp, st))) return r;
  }
  return TP_OK;
}
// Pointer alignment of the backward's buffers: 16 bytes on the bf16
// (tensor-map) path, the element on the fp32 one.
bool bwd_ptrs_ok(std::initializer_list<const void*> ps, int dtype) {
  for (const void* p : ps)
    if (!ptr_ok(p, dtype)) return false;
  return true;
}

bool ptrs16(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p && !aligned(p, 16)) return false;
  return true;
}

// dXs[s] = dY @ W_s^T and dW_s = (Xs[s]^T @ dY)^T for a row view W
// (shards [tp][N][Ks]). Both read W's storage, or Xs and dY, MN-major.
int row_bwd_bf16(const void* Xs, int64_t T, const tp_shards* W, const void* dY, void* dXs, void* dW,
                 const Scratch* sc, cudaStream_t st) {
  const int tp = W->tp;
  const int64_t Ks = W->K / tp, N = W->N;
  CUtensorMap ma, mb;
  int r = TP_OK;
  if (dXs) {  // COL over shards: A = dY [T][N] (K = N), B_s[k][n] = W storage [tp][N][Ks] (MN-major)
    if (!make_map_bf16(&ma, dY, N, T, 1, 128) || !make_map_bf16(&mb, W->data, Ks, N, tp, 64)) return TP_ERR_CUDA;
    if ((r = gemm_bwd<tpk::GK_COL, 2>(ma, mb, T, Ks, tp, N, 0, nullptr, dXs, sc, st))) return r;
  }
  if (dW) {  // COL over shards, K = T: A = dY^T (M = N), B_s = Xs[s]^T (N = Ks), both MN-major
    if (!make_map_bf16(&ma, dY, N, T, 1, 64) || !make_map_bf16(&mb, Xs, Ks, T, tp, 64)) return TP_ERR_CUDA;
    if ((r = gemm_bwd<tpk::GK_COL, 3>(ma, mb, N, Ks, tp, T, 0, nullptr, dW, sc, st))) return r;
  }
  return r;
}

// dX = sum_s dYs[s] @ W_s^T (+ dR) and dW_s = (X^T @ dYs[s])^T for a column
// view W (shards [tp][Ns][K]).
int col_bwd_bf16(const void* X, int64_t T, const tp_shards* W, const void* dYs, const void* dR, void* dX,
                 void* dW, const Scratch* sc, cudaStream_t st) {
  const int tp = W->tp;
  const int64_t K = W->K, Ns = W->N / tp;
  CUtensorMap ma, mb;
  int r = TP_OK;
  if (dX) {  // ROW_SUM: A_s = dYs[s] [T][Ns] (K = Ns), B_s[k][n] = W storage [tp][Ns][K] (MN-major)
    if (!make_map_bf16(&ma, dYs, Ns, T, tp, 128) || !make_map_bf16(&mb, W->data, K, Ns, tp, 64)) return TP_ERR_CUDA;
    if ((r = gemm_bwd<tpk::GK_ROW_SUM, 2>(ma, mb, T, K, tp, Ns, 0, dR, dX, sc, st))) return r;
  }
  if (dW) {  // COL with A per shard, K = T: A_s = dYs[s]^T (M = Ns), B = X^T (N = K), both MN-major
    if (!make_map_bf16(&ma, dYs, Ns, T, tp, 64) || !make_map_bf16(&mb, X, K, T, 1, 64)) return TP_ERR_CUDA;
    if ((r = gemm_bwd<tpk::GK_COL, 3>(ma, mb, Ns, K, tp, T, 1, nullptr, dW, sc, st))) return r;
  }
  return r;
}

// tok_rows > 0 (bf16 only): dG and dU token-major [tok_rows][tp * Is] (see
// act_backward_kernel; Is % 8 == 0, tok_rows * Is / 8 < 2^31 and tp < 2^16,
// checked by the caller).
int act_bwd_launch(const void* dH, const void* G, const void* U, int64_t n, int act, void* dG, void* dU,
                   cudaStream_t st, int dtype = TP_BF16, int64_t tok_rows = 0, int tp = 1, int64_t Is = 0) {
  if (dtype == TP_F32) {
    if (n == 0) return TP_OK;
    tpk::act_backward_f32_kernel<<<grid_for(n, 256), 256, 0, st>>>(
        static_cast<const float*>(dH), static_cast<const float*>(G), static_cast<const float*>(U), n, act,
        static_cast<float*>(dG), static_cast<float*>(dU));
    return launch_status();
  }
  const int64_t n8 = n / 8;
  if (n8 == 0) return TP_OK;
  if (tok_rows > 0) {  // a grid row per shard; T * Is / 8 vectors each
    const uint32_t d = static_cast<uint32_t>(Is / 8);
    int shift = 0;
    while ((1ull << shift) < d) ++shift;
    const uint32_t magic = static_cast<uint32_t>((1ull << (32 + shift)) / d - (1ull << 32) + 1);
    const int64_t per = tok_rows * d;
    const dim3 grid(static_cast<unsigned>(std::max(1, std::min<int>(grid_for(per, 256), grid_for(n8, 256) / tp))),
                    static_cast<unsigned>(tp));
    tpk::act_backward_kernel<<<grid, 256, 0, st>>>(
        static_cast<const bf16*>(dH), static_cast<const bf16*>(G), static_cast<const bf16*>(U), per, act,
        static_cast<bf16*>(dG), static_cast<bf16*>(dU), d, magic, shift, tp);
    return launch_status();
  }
  tpk::act_backward_kernel<<<grid_for(n8, 256), 256, 0, st>>>(
      static_cast<const bf16*>(dH), static_cast<const bf16*>(G), static_cast<const bf16*>(U), n8, act,
      static_cast<bf16*>(dG), static_cast<bf16*>(dU));
  return launch_status();
}

size_t bwd_max_tiles(int64_t H, int64_t I, int tp) {
  return std::max<size_t>(mlp_max_tiles(H, I, tp), 2 * SK_MAX_CTAS);
}

}  // namespace

extern "C" {

tp_status tp_row_linear_backward(const void* Xs, int64_t T, const tp_shards* W, const void* dY, void* dXs,
                                 void* dW, void* stream) {
  int r = check_bwd_view(W, TP_ROW);
  if (r) return as_status(r);
  if (T < 0) return TP_ERR_SHAPE;
  if (T > INT32_MAX) return TP_ERR_UNSUPPORTED;
  if (T > 0 && (!dY || (dW && !Xs))) return TP_ERR_NULL;
  if (!bwd_ptrs_ok({Xs, dY, dXs, dW}, W->dtype)) return TP_ERR_ALIGN;
  if (T == 0) return TP_OK;
  if (W->dtype == TP_F32) return as_status(row_bwd_f32(Xs, T, W, dY, dXs, dW, as_stream(stream)));
  return as_status(row_bwd_bf16(Xs, T, W, dY, dXs, dW, nullptr, as_stream(stream)));
}

tp_status tp_column_linear_backward(const void* X, int64_t T, const tp_shards* W, const void* dYs,
                                    const void* dR, void* dX, void* dW, void* workspace, size_t ws_bytes,
                                    void* stream) {
  int r = check_bwd_view(W, TP_COL);
  if (r) return as_status(r);
  if (T < 0) return TP_ERR_SHAPE;
  if (T > INT32_MAX) return TP_ERR_UNSUPPORTED;
  if (T > 0 && (!dYs || (dW && !X))) return TP_ERR_NULL;
  if (!bwd_ptrs_ok({X, dYs, dR, dX, dW}, W->dtype)) return TP_ERR_ALIGN;
  if (W->dtype == TP_F32) {
    if (T == 0) return TP_OK;
    return as_status(col_bwd_f32(X, T, W, dYs, dR, dX, dW, as_stream(stream)));
  }
  if (W->K % 8 != 0) return TP_ERR_ALIGN;
  Scratch sc{};
  const Scratch* scp = nullptr;
  if ((r = linear_scratch(W, T, workspace, ws_bytes, &sc, &scp))) return as_status(r);
  if (T == 0) return TP_OK;
  return as_status(col_bwd_bf16(X, T, W, dYs, dR, dX, dW, scp, as_stream(stream)));
}

size_t tp_mlp_backward_workspace_bytes(int64_t T, int64_t H, int64_t I, int tp, int act, int dtype) {
  if (T < 0 || H < 1 || I < 1 || tp < 1 || !dtype_ok(dtype)) return 0;
  const size_t inter = align256(static_cast<size_t>(T) * I * elem_size(dtype));
  const bool gated = act == TP_ACT_SWIGLU;
  // dHs, dG (, dU); the bf16 (tcgen05) path also takes the split-tile scratch
  return (gated ? 3 : 2) * inter + (dtype == TP_BF16 ? scratch_bytes(T, bwd_max_tiles(H, I, tp)) : 0);
}

tp_status tp_mlp_backward(const void* X, int64_t T, const tp_shards* W1, const tp_shards* W_up,
                          const tp_shards* W2, int act, const void* G, const void* U, const void* Hs,
                          const void* dY, const void* dR, void* workspace, size_t ws_bytes, void* dX,
                          void* dW1, void* dW_up, void* dW2, void* stream) {
  if (!W1 || !W2) return TP_ERR_NULL;
  if (act < TP_ACT_NONE || act > TP_ACT_SWIGLU) return TP_ERR_MODE;
  const bool gated = act == TP_ACT_SWIGLU;
  int r;
  if ((r = check_bwd_view(W1, TP_COL)) || (r = check_bwd_view(W2, TP_ROW))) return as_status(r);
  if (gated) {
    if (!W_up) return TP_ERR_NULL;
    if ((r = check_bwd_view(W_up, TP_COL))) return as_status(r);
    if (!same_shape(W1, W_up)) return TP_ERR_SHAPE;
  } else if (W_up || U || dW_up) {
    return TP_ERR_MODE;
  }
  if (W2->tp != W1->tp || W2->K != W1->N || W2->N != W1->K) return TP_ERR_SHAPE;
  if (T < 0) return TP_ERR_SHAPE;
  if (T > INT32_MAX) return TP_ERR_UNSUPPORTED;
  if (W2->dtype != W1->dtype || (gated && W_up->dtype != W1->dtype)) return TP_ERR_DTYPE;
  if (T > 0 && (!X || !G || !Hs || !dY || (gated && !U) || !workspace)) return TP_ERR_NULL;
  const int dt = W1->dtype;
  if (!bwd_ptrs_ok({X, G, U, Hs, dY, dR, dX, dW1, dW_up, dW2}, dt) || !aligned(workspace, 256)) return TP_ERR_ALIGN;
  const int64_t H = W1->K, I = W1->N;
  const int tp = W1->tp;
  if (ws_bytes < tp_mlp_backward_workspace_bytes(T, H, I, tp, act, dt)) return TP_ERR_WORKSPACE;
  if (T == 0) return TP_OK;
  const cudaStream_t st = as_stream(stream);
  char* ws = static_cast<char*>(workspace);
  if (dt == TP_F32) {
    // the same steps on the FFMA GEMM: row layer, activation, column layer(s)
    // with the input gradient accumulated over gate and up, plus dR
    const size_t inter = align256(static_cast<size_t>(T) * I * sizeof(float));
    void* dHs = ws;
    void* dG = ws + inter;
    void* dU = gated ? ws + 2 * inter : nullptr;
    if ((r = row_bwd_f32(Hs, T, W2, dY, dHs, dW2, st))) return as_status(r);
    if ((r = act_bwd_launch(dHs, G, U, static_cast<int64_t>(T) * I, act, dG, dU, st, TP_F32))) return as_status(r);
    if ((r = col_bwd_f32(X, T, W1, dG, dR, dX, dW1, st))) return as_status(r);
    if (gated) r = col_bwd_f32(X, T, W_up, dU, dX, dX, dW_up, st);
    return as_status(r);
  }
  const size_t inter = align256(static_cast<size_t>(T) * I * 2);
  void* dHs = ws;
  void* dG = ws + inter;
  void* dU = gated ? ws + 2 * inter : nullptr;
  const int64_t Is = I / tp;
  if (Is % 8 != 0) return TP_ERR_ALIGN;  // (16-byte rows, as every tensor map here needs)
  if (static_cast<int64_t>(T) * (Is / 8) > INT32_MAX || tp > 65535) return TP_ERR_UNSUPPORTED;
  const Scratch sc = carve_scratch(workspace, (gated ? 3 : 2) * inter, bwd_max_tiles(H, I, tp));
  // row layer (every shard gets dY): dHs and dW2; then the local activation,
  // which writes dG (and dU) token-major, [T][I] with the shards side by side
  if ((r = row_bwd_bf16(Hs, T, W2, dY, dHs, dW2, &sc, st))) return as_status(r);
  if ((r = act_bwd_launch(dHs, G, U, static_cast<int64_t>(T) * I, act, dG, dU, st, TP_BF16, T, tp, Is)))
    return as_status(r);
  // Column layer(s), each over all of I at once: the shards' contributions
  // to dX are terms of one contraction over I, and their weight gradients
  // are row blocks of one [I][H] product, so no tile is cut at a shard's
  // ragged end (the column shards' storage [tp][Is][H] is [I][H]).
  // dX: one accumulator over gate and up for SwiGLU, plus dR.
  if (dX) {
    CUtensorMap ma0, mb0, ma1, mb1;
    if (!make_map_bf16(&ma0, dG, I, T, 1, 128) || !make_map_bf16(&mb0, W1->data, H, I, 1, 64) ||
        (gated && (!make_map_bf16(&ma1, dU, I, T, 1, 128) || !make_map_bf16(&mb1, W_up->data, H, I, 1, 64))))
      return TP_ERR_CUDA;
    if ((r = gemm_bwd<tpk::GK_ROW_SUM, 2>(ma0, mb0, T, H, 1, I, 0, dR, dX, &sc, st, gated ? &ma1 : nullptr,
                                          gated ? &mb1 : nullptr)))
      return as_status(r);
  }
  // dW = (X^T dG)^T: A = dG^T (M = I), B = X^T (N = H), both MN-major, K = T
  auto dw = [&](const void* dA, void* dW) -> int {
    if (!dW) return TP_OK;
    CUtensorMap ma, mb;
    if (!make_map_bf16(&ma, dA, I, T, 1, 64) || !make_map_bf16(&mb, X, H, T, 1, 64)) return TP_ERR_CUDA;
    return gemm_bwd<tpk::GK_COL, 3>(ma, mb, I, H, 1, T, 1, nullptr, dW, &sc, st);
  };
  if ((r = dw(dG, dW1))) return as_status(r);
  return as_status(gated ? dw(dU, dW_up) : TP_OK);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Vocabulary-parallel embedding and cross-entropy
// ---------------------------------------------------------------------------
extern "C" {

tp_status tp_vocab_embedding(const int32_t* ids, int64_t T, const void* E, int64_t V, int64_t H, int tp,
                             int dtype, void* Y, void* stream) {
  if (!dtype_ok(dtype)) return TP_ERR_DTYPE;
  if (T < 0 || V < 1 || H < 1 || tp < 1 || V % tp != 0) return TP_ERR_SHAPE;
  if (T == 0) return TP_OK;
  if (!ids || !E || !Y) return TP_ERR_NULL;
  const size_t es = elem_size(dtype);
  if (!aligned(ids, 4) || !aligned(E, es) || !aligned(Y, es)) return TP_ERR_ALIGN;
  const int vec = (H * static_cast<int64_t>(es)) % 16 == 0 && aligned(E, 16) && aligned(Y, 16);
  const int grid = static_cast<int>(std::min<int64_t>(cdiv(T, 8), static_cast<int64_t>(std::max(1, num_sms())) * 16));
  const cudaStream_t st = as_stream(stream);
  if (dtype == TP_BF16)
    tpk::vocab_embed_kernel<bf16><<<grid, 256, 0, st>>>(ids, T, static_cast<const bf16*>(E), V, H, V / tp, vec,
                                                          static_cast<bf16*>(Y));
  else
    tpk::vocab_embed_kernel<float><<<grid, 256, 0, st>>>(ids, T, static_cast<const float*>(E), V, H, V / tp, vec,
                                                           static_cast<float*>(Y));
  return as_status(launch_status());
}

// Partial statistics of the cross-entropy's first pass: 3 floats per
// (shard, token, chunk of CE_CHUNK logits) unit.
size_t ce_stats_bytes(int64_t T, int64_t V, int tp) {
  const int64_t v = V / std::max(tp, 1), nchunk = cdiv(std::max<int64_t>(v, 1), tpk::CE_CHUNK);
  return align256(static_cast<size_t>(T) * tp * nchunk * 3 * sizeof(float));
}

size_t tp_cross_entropy_workspace_bytes(int64_t T, int64_t V, int tp) {
  if (T < 0 || V < 1 || tp < 1) return 0;
  return ce_stats_bytes(T, V, tp) + 2 * align256(static_cast<size_t>(T) * sizeof(float));
}

tp_status tp_vocab_cross_entropy(const void* logits, const int32_t* labels, int64_t T, int64_t V, int tp,
                                 int dtype, float* loss, float* mean_loss, void* dlogits, float grad_scale,
                                 void* workspace, size_t ws_bytes, void* stream) {
  if (!dtype_ok(dtype)) return TP_ERR_DTYPE;
  if (T < 0 || V < 1 || tp < 1 || V % tp != 0) return TP_ERR_SHAPE;
  if (ws_bytes < tp_cross_entropy_workspace_bytes(T, V, tp)) return TP_ERR_WORKSPACE;
  if (T == 0) {
    if (mean_loss && !cuda_ok(cudaMemsetAsync(mean_loss, 0, sizeof(float), as_stream(stream))))
      return TP_ERR_CUDA;
    return TP_OK;
  }
  if (!logits || !labels || !workspace) return TP_ERR_NULL;
  const size_t es = elem_size(dtype);
  if (!aligned(labels, 4) || !aligned(logits, es) || !aligned(workspace, 256) || (loss && !aligned(loss, 4)) ||
      (mean_loss && !aligned(mean_loss, 4)) || (dlogits && !aligned(dlogits, es)))
    return TP_ERR_ALIGN;
  const int64_t v = V / tp;
  const int vec = (v % 8 == 0) && aligned(logits, 16) && (!dlogits || aligned(dlogits, 16));
  const cudaStream_t st = as_stream(stream);
  char* ws = static_cast<char*>(workspace);
  float* stats = reinterpret_cast<float*>(ws);
  float* lse = reinterpret_cast<float*>(ws + ce_stats_bytes(T, V, tp));
  float* loss_ws = lse + align256(static_cast<size_t>(T) * sizeof(float)) / sizeof(float);
  float* per_tok = loss ? loss : loss_ws;
  const int sms = std::max(1, num_sms());
  const int64_t nchunk = cdiv(v, tpk::CE_CHUNK);  // units of pass 1: (shard, token, chunk)
  const int64_t units = T * tp * nchunk;            // one warp per unit, 8 per CTA
  const int grid_rows = static_cast<int>(std::min<int64_t>(cdiv(units, 8), static_cast<int64_t>(sms) * 16));
  if (dtype == TP_BF16)
    tpk::ce_stats_kernel<bf16><<<grid_rows, 256, 0, st>>>(static_cast<const bf16*>(logits), labels, T, tp, v, vec,
                                                            stats);
  else
    tpk::ce_stats_kernel<float><<<grid_rows, 256, 0, st>>>(static_cast<const float*>(logits), labels, T, tp, v,
                                                             vec, stats);
  int r = launch_status();
  if (r) return as_status(r);
  tpk::ce_combine_kernel<<<static_cast<int>(std::min<int64_t>(cdiv(T, 8), static_cast<int64_t>(sms) * 16)), 256, 0,
                           st>>>(stats, labels, T, tp, V, nchunk, lse, per_tok);
  if ((r = launch_status())) return as_status(r);
  if (mean_loss) {
    tpk::ce_mean_kernel<<<1, 1024, 0, st>>>(per_tok, T, mean_loss);
    if ((r = launch_status())) return as_status(r);
  }
  if (dlogits) {
    const int grid_g = vec ? grid_rows : grid_for(T * V, 256);
    if (dtype == TP_BF16)
      tpk::ce_grad_kernel<bf16><<<grid_g, 256, 0, st>>>(
          static_cast<const bf16*>(logits), labels, lse, T, tp, v, grad_scale, vec, static_cast<bf16*>(dlogits));
    else
      tpk::ce_grad_kernel<float><<<grid_g, 256, 0, st>>>(
          static_cast<const float*>(logits), labels, lse, T, tp, v, grad_scale, vec, static_cast<float*>(dlogits));
    r = launch_status();
  }
  return as_status(r);
}

// Statistics of the fused LM head: one (max, sum, label logit) triple per
// (shard, token, 256-column tile of the shard's vocabulary).
size_t lm_ce_stats_bytes(int64_t T, int64_t V, int tp) {
  const int64_t v = V / std::max(tp, 1);
  return align256(static_cast<size_t>(T) * tp * cdiv(std::max<int64_t>(v, 1), 256) * 3 * sizeof(float));
}

size_t tp_lm_head_ce_workspace_bytes(int64_t T, const tp_shards* W_lm) {
  if (!W_lm || T < 0 || W_lm->tp < 1 || W_lm->N < 1 || W_lm->K < 1) return 0;
  const int tp = W_lm->tp;
  const int64_t V = W_lm->N;
  const size_t head = std::max(lm_ce_stats_bytes(T, V, tp), ce_stats_bytes(T, V, tp)) +
                      2 * align256(static_cast<size_t>(T) * sizeof(float));
  return head + tp_gemm_workspace_bytes(T, W_lm);
}

tp_status tp_lm_head_cross_entropy(const void* X, int64_t T, const tp_shards* W_lm, const int32_t* labels,
                                   void* logits, float* loss, float* mean_loss, void* dlogits, float grad_scale,
                                   void* workspace, size_t ws_bytes, void* stream) {
  int r = check_col(X, T, W_lm, nullptr, nullptr, nullptr, TP_ACT_NONE, 0, logits);
  if (r) return as_status(r);
  const int tp = W_lm->tp, dt = W_lm->dtype;
  const int64_t V = W_lm->N, v = V / tp;
  if (T == 0) {  // an empty call needs no labels or workspace
    if (mean_loss && !cuda_ok(cudaMemsetAsync(mean_loss, 0, sizeof(float), as_stream(stream))))
      return TP_ERR_CUDA;
    return TP_OK;
  }
  if (!labels || !workspace) return TP_ERR_NULL;
  if (ws_bytes < tp_lm_head_ce_workspace_bytes(T, W_lm)) return TP_ERR_WORKSPACE;
  const size_t es = elem_size(dt);
  if (!aligned(labels, 4) || !aligned(workspace, 256) || (loss && !aligned(loss, 4)) ||
      (mean_loss && !aligned(mean_loss, 4)) || (dlogits && !aligned(dlogits, es)))
    return TP_ERR_ALIGN;
  const cudaStream_t st = as_stream(stream);
  char* ws = static_cast<char*>(workspace);
  const size_t stats_bytes = std::max(lm_ce_stats_bytes(T, V, tp), ce_stats_bytes(T, V, tp));
  float* stats = reinterpret_cast<float*>(ws);
  float* lse = reinterpret_cast<float*>(ws + stats_bytes);
  float* loss_ws = lse + align256(static_cast<size_t>(T) * sizeof(float)) / sizeof(float);
  float* per_tok = loss ? loss : loss_ws;
  const size_t head = stats_bytes + 2 * align256(static_cast<size_t>(T) * sizeof(float));
  const int sms = std::max(1, num_sms());
  const int vec = (v % 8 == 0) && aligned(logits, 16) && (!dlogits || aligned(dlogits, 16));
  int64_t nchunk;
  if (dt == TP_BF16 && T > SWAP_MAX_T) {
    // the statistics come out of the GEMM's epilogue, per 256-column tile
    Scratch sc = carve_scratch(ws, head, std::max<size_t>(2 * SK_MAX_CTAS, static_cast<size_t>(tp) * cdiv(v, 128)));
    if ((r = col_bf16(X, T, W_lm, nullptr, nullptr, nullptr, TP_ACT_NONE, 0, logits, &sc, 1, 0, nullptr, st,
                      labels, stats)))
      return as_status(r);
    nchunk = cdiv(v, 256);
  } else {
    // few tokens (weight-streaming GEMM) or fp32: the logits, then a pass over them
    Scratch sc{};
    const Scratch* scp = nullptr;
    if (dt == TP_BF16) {
      sc = carve_scratch(ws, head, std::max<size_t>(2 * SK_MAX_CTAS, static_cast<size_t>(tp) * cdiv(v, 128)));
      scp = &sc;
    }
    if ((r = run_col(X, T, W_lm, nullptr, nullptr, nullptr, TP_ACT_NONE, 0, logits, st, scp))) return as_status(r);
    nchunk = cdiv(v, tpk::CE_CHUNK);
    const int64_t units = T * tp * nchunk;
    const int grid_rows = static_cast<int>(std::min<int64_t>(cdiv(units, 8), static_cast<int64_t>(sms) * 16));
    if (dt == TP_BF16)
      tpk::ce_stats_kernel<bf16><<<grid_rows, 256, 0, st>>>(static_cast<const bf16*>(logits), labels, T, tp, v,
                                                              vec, stats);
    else
      tpk::ce_stats_kernel<float><<<grid_rows, 256, 0, st>>>(static_cast<const float*>(logits), labels, T, tp, v,
                                                               vec, stats);
    if ((r = launch_status())) return as_status(r);
  }
  tpk::ce_combine_kernel<<<static_cast<int>(std::min<int64_t>(cdiv(T, 8), static_cast<int64_t>(sms) * 16)), 256, 0,
                           st>>>(stats, labels, T, tp, V, nchunk, lse, per_tok);
  if ((r = launch_status())) return as_status(r);
  if (mean_loss) {
    tpk::ce_mean_kernel<<<1, 1024, 0, st>>>(per_tok, T, mean_loss);
    if ((r = launch_status())) return as_status(r);
  }
  if (dlogits) {
    const int64_t units = T * tp * cdiv(v, tpk::CE_CHUNK);
    const int grid_g = vec ? static_cast<int>(std::min<int64_t>(cdiv(units, 8), static_cast<int64_t>(sms) * 16))
                           : grid_for(T * V, 256);
    if (dt == TP_BF16)
      tpk::ce_grad_kernel<bf16><<<grid_g, 256, 0, st>>>(
          static_cast<const bf16*>(logits), labels, lse, T, tp, v, grad_scale, vec, static_cast<bf16*>(dlogits));
    else
      tpk::ce_grad_kernel<float><<<grid_g, 256, 0, st>>>(
          static_cast<const float*>(logits), labels, lse, T, tp, v, grad_scale, vec, static_cast<float*>(dlogits));
    r = launch_status();
  }
  return as_status(r);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Mixture of experts with tensor-parallel experts (grouped GEMMs)
// ---------------------------------------------------------------------------
namespace {

struct MoeLayout {
  int64_t units, rows;  // 256-row units of the permuted buffers, and their rows
  size_t xp, hs, yp, pos, inv, counts, off, unit_expert, unit_seg, total;
};

MoeLayout moe_layout(int64_t T, int64_t H, int64_t I, int k, int E) {
  MoeLayout L{};
  L.units = cdiv(T * k, tpk::MOE_UNIT) + E;  // each expert's padding adds at most one unit
  L.rows = L.units * tpk::MOE_UNIT;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  L.xp = take(static_cast<size_t>(L.rows) * H * 2);   // bf16
  L.hs = take(static_cast<size_t>(L.rows) * I * 2);   // bf16 [tp][rows][I/tp]
  L.yp = take(static_cast<size_t>(L.rows) * H * 4);   // fp32
  L.pos = take(static_cast<size_t>(T) * k * 4);
  L.inv = take(static_cast<size_t>(T) * k * 4);
  L.counts = take(static_cast<size_t>(E) * 4);
  L.off = take(static_cast<size_t>(E) * 4);
  L.unit_expert = take(static_cast<size_t>(L.units) * 4);
  L.unit_seg = take(static_cast<size_t>(L.units) * 8);
  L.total = o;
  return L;
}

}  // namespace

extern "C" {

size_t tp_moe_workspace_bytes(int64_t T, int64_t H, int64_t I, int k, int E, int tp) {
  if (T < 0 || H < 1 || I < 1 || k < 1 || E < 1 || tp < 1) return 0;
  return moe_layout(T, H, I, k, E).total;
}

tp_status tp_moe_block(const void* X, int64_t T, const int32_t* ids, const float* weights, int k, int E,
                       const tp_shards* Wg, const tp_shards* Wu, const tp_shards* Wd, const void* residual,
                       void* workspace, size_t ws_bytes, void* Y, void* stream) {
  if (!Wg || !Wu || !Wd) return TP_ERR_NULL;
  int r;
  if ((r = check_view(Wg, TP_COL)) || (r = check_view(Wu, TP_COL)) || (r = check_view(Wd, TP_ROW))) return as_status(r);
  if (Wg->dtype != TP_BF16 || !same_shape(Wg, Wu) || Wd->dtype != TP_BF16) return TP_ERR_DTYPE;
  if (Wd->tp != Wg->tp || Wd->K != Wg->N || Wd->N != Wg->K) return TP_ERR_SHAPE;
  if (T < 0 || k < 1 || E < 1 || E > 1024) return TP_ERR_SHAPE;
  if (T * k > INT32_MAX / 2) return TP_ERR_UNSUPPORTED;
  const int64_t H = Wg->K, I = Wg->N;
  const int tp = Wg->tp;
  const MoeLayout L = moe_layout(T, H, I, k, E);
  if (ws_bytes < L.total) return TP_ERR_WORKSPACE;
  if (T == 0) return TP_OK;
  if (!X || !ids || !weights || !workspace || !Y) return TP_ERR_NULL;
  if (!ptrs16({X, residual, Y}) || !aligned(workspace, 256) || !aligned(ids, 4) || !aligned(weights, 4))
    return TP_ERR_ALIGN;
  const cudaStream_t st = as_stream(stream);
  char* ws = static_cast<char*>(workspace);
  bf16* Xp = reinterpret_cast<bf16*>(ws + L.xp);
  bf16* Hs = reinterpret_cast<bf16*>(ws + L.hs);
  float* Yp = reinterpret_cast<float*>(ws + L.yp);
  int32_t* pos = reinterpret_cast<int32_t*>(ws + L.pos);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + L.inv);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
  int32_t* unit_expert = reinterpret_cast<int32_t*>(ws + L.unit_expert);
  int2* unit_seg = reinterpret_cast<int2*>(ws + L.unit_seg);
  const int64_t n = T * k;
  const int64_t grid_cap = static_cast<int64_t>(std::max(1, num_sms())) * 16;
  // 1. dispatch
  tpk::moe_route_kernel<<<E, 1024, 0, st>>>(ids, n, E, pos, counts);
  if ((r = launch_status())) return as_status(r);
  tpk::moe_units_kernel<<<1, 256, 0, st>>>(counts, E, static_cast<int>(L.units), off, unit_expert, unit_seg);
  if ((r = launch_status())) return as_status(r);
  tpk::moe_gather_kernel<<<static_cast<int>(std::min<int64_t>(cdiv(n, 8), grid_cap)), 256, 0, st>>>(
      static_cast<const bf16*>(X), ids, pos, off, n, k, E, H, Xp, inv);
  if ((r = launch_status())) return as_status(r);
  // 2. the experts' MLP blocks over all units: gate/up + SwiGLU per shard,
  // then down + the shard sum; each tile takes its expert's shard set
  const int64_t Is = I / tp;
  {
    CUtensorMap mx, mg, mu;
    if (!make_map_bf16(&mx, Xp, H, L.rows, 1, 128) ||
        !make_map_bf16(&mg, Wg->data, H, Is, static_cast<uint64_t>(E) * tp, 128) ||
        !make_map_bf16(&mu, Wu->data, H, Is, static_cast<uint64_t>(E) * tp, 128))
      return TP_ERR_CUDA;
    tpk::GemmArgs a{};
    a.M = static_cast<int>(L.rows);
    a.Ns = static_cast<int>(Is);
    a.tp = tp;
    a.rep = 1;
    a.cluster = 2;
    a.kb_per_shard = static_cast<int>(cdiv(H, 64));
    a.kpt = a.kb_per_shard;
    a.act = TP_ACT_SWIGLU;
    a.out = Hs;
    a.m_tiles = static_cast<int>(L.units);
    a.n_tiles = static_cast<int>(cdiv(Is, 128));
    a.num_tiles = a.m_tiles * a.n_tiles * tp;
    a.r1_tiles = a.num_tiles;
    a.unit_expert = unit_expert;
    // groups of 8 pairs within each expert: a weight tile's few readers
    // (the expert's units) fall within 8 tiles of each other
    a.unit_group = 8;
    a.unit_seg = unit_seg;
    OutMaps om{};
    a.tma_store = make_store_map(&om.y, Hs, false, Is, L.rows, tp, Is * 2, L.rows * Is * 2) ? 1 : 0;
    if ((r = gemm_launch<tpk::GK_COL_SWIGLU, false>(mx, mx, mg, mu, om, a, nullptr, st))) return as_status(r);
  }
  {
    CUtensorMap mx, mw;
    if (!make_map_bf16(&mx, Hs, Is, L.rows, tp, 128) ||
        !make_map_bf16(&mw, Wd->data, Is, H, static_cast<uint64_t>(E) * tp, 128))
      return TP_ERR_CUDA;
    tpk::GemmArgs a{};
    a.M = static_cast<int>(L.rows);
    a.Ns = static_cast<int>(H);
    a.tp = tp;
    a.rep = 1;
    a.cluster = 2;
    a.kb_per_shard = static_cast<int>(cdiv(Is, 64));
    a.kpt = a.kb_per_shard * tp;
    a.out = Yp;
    a.out_f32 = 1;  // the expert rows stay fp32 until the weighted combine
    a.m_tiles = static_cast<int>(L.units);
    a.n_tiles = static_cast<int>(cdiv(H, 256));
    a.num_tiles = a.m_tiles * a.n_tiles;
    a.r1_tiles = a.num_tiles;
    a.unit_expert = unit_expert;
    // one column block at a time, the expert's units fastest: the few
    // units that read a weight block do so side by side (the 16 blocks in one
    // group spread them over two rounds, and the second read missed L2)
    a.unit_group = 1;
    a.unit_seg = unit_seg;
    OutMaps om{};
    a.tma_store = make_store_map(&om.y, Yp, true, H, L.rows, 1, H * 4, L.rows * H * 4) ? 1 : 0;
    if ((r = gemm_launch<tpk::GK_ROW_SUM, false>(mx, mx, mw, mw, om, a, nullptr, st))) return as_status(r);
  }
  // 3. combine
  tpk::moe_combine_kernel<<<static_cast<int>(std::min<int64_t>(cdiv(T, 8), grid_cap)), 256, 0, st>>>(
      Yp, inv, weights, T, k, H, static_cast<const bf16*>(residual), static_cast<bf16*>(Y));
  return as_status(launch_status());
}

}  // extern "C"
