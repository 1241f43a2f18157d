// Persistent tcgen05 GEMM for the sharded column / row linears (bf16 in,
// fp32 accumulation in tensor memory, fused epilogues).
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: streams operand tiles through an mbarrier ring;
//   warp 1      TMEM owner and MMA issuer (one thread issues tcgen05.mma into
//               one of two TMEM accumulators, so the epilogue of one work
//               unit overlaps the main loop of the next);
//   warps 2..5  epilogue (tcgen05.ld, fused elementwise work, stores).
//
// Two operand arrangements:
//   normal   A = 128 token rows, B = 256 weight rows (MMA 128x256x16). For
//            large token counts.
//   SWAP     A = 128 weight rows (two tiles, gate and up, for SwiGLU), B = the
//            token rows padded to Tpad in {16,32,48,64} (MMA 128xTpadx16). For
//            few tokens: the weights are the big operand and are streamed
//            once, so this regime is bound by HBM bandwidth, not the MMA.
//
// Tile kinds (what one output tile is and how its K loop runs):
//   COL         column-parallel linear, Y_s = act(X @ W_s + b_s) for each
//               output-column shard s ("CUDA tensor parallel computations"
//               page, Column Parallel and local elementwise sections); X is
//               replicated, so every shard's tiles read the same A rows.
//   COL_SWIGLU  gate and up shards together; the epilogue writes
//               silu(gate) * up ("Tensor parallelism" tutorial page, MLP block).
//   ROW_SUM     row-parallel linear with the all-reduce folded into the
//               accumulator: the K loop runs over (shard, k-block), so
//               sum_s X_s @ W_s never leaves TMEM; bias once, then residual
//               ("Row Parallel": contributions are added).
//   ROW_PARTIAL per-shard contributions P_s = X_s @ W_s stored as fp32.
//
// Work schedule. A work unit is a tile's K loop or a contiguous piece of it.
// The first dp_tiles tiles go round-robin to the CTAs, whole. The remaining
// tiles' k-iterations are split evenly over the grid (stream-K), which
// removes the last-wave imbalance. A tile split over several CTAs is
// combined deterministically: each piece is stored as fp32 in a workspace
// slot, and the CTA that finishes last (an atomic counter per tile) sums the
// pieces in k order and runs the tile's epilogue. No CTA ever waits for
// another, so the schedule cannot deadlock.
//
// CTA pairs (normal mode, PAIR): a cluster of two CTAs on two SMs computes a
// 256 x 256 tile with the 2-SM MMA. The even CTA holds token block 2u, the
// odd one block 2u+1 (A), and each holds one 128-row half of the weight
// block (B: gate / up for SwiGLU, else rows [128 r, 128 r + 128)). Per SM a
// k-step then stages 32 KB instead of 48 KB and the tensor core reads half
// of B from each SM's shared memory, which leaves room for six stages. One
// thread of the even CTA issues the MMAs; both CTAs' TMA loads count on the
// even CTA's "full" barrier; its commits release the stage in both CTAs and
// hand each CTA's accumulator half (its own tensor memory) to that CTA's
// epilogue; both epilogues report a drained accumulator to the even CTA.
//
// Split last round (CTA pairs, row GEMMs): when the units do not fill the pairs evenly,
// the first dp_tiles units run whole, round-robin, and each of the
// split_units remaining ones is cut along K into split_ways equal pieces,
// one piece per pair, so that the last round is 1/split_ways as long. Pair q
// of that round takes piece j = q / split_units of unit q % split_units, so
// the pieces running together cover the same K range of their operands.
// Pieces j < split_ways - 1 park their fp32 accumulator in a workspace slot
// and then set their flag (per unit, CTA rank and piece) to this launch's
// epoch (see GemmArgs::sync_words). The last piece (the owner, every pair's
// final item) waits for the others' flags, adds their slots in j order to
// its own accumulator and runs the epilogue. The sum order is fixed, so
// results do not depend on timing.
//
// QKV replica dedup (normal COL): when kv heads are replicated across rep
// consecutive shards, the tiles holding only replicated K|V columns are
// computed once, on the first shard of each group, and stored to all rep
// shards.
//
// Operand order (CTA pairs, COL and ROW_SUM; the template argument MN):
// bit 0 set means A is given MN-major ([K][M] in memory, M contiguous),
// bit 1 the same for B. An MN-major tile is loaded as two 64-wide panels
// (64 K rows x 128 bytes each) and described to the tensor core with the
// MN-major shared-memory descriptor and the instruction's transpose bit, so
// no operand is ever transposed in memory. This serves the backward of the
// column/row pair: data gradients read the forward's K-major weight shards
// as MN-major B, and weight gradients contract over tokens with both
// operands MN-major. With GemmArgs::a_sharded a COL launch takes A per shard
// and B replicated (the weight gradient of a column layer).
#pragma once

#include "tp_epilogue.cuh"
#include "tp_ptx.cuh"

namespace tpk {

// GK_COL_CE: GK_COL whose epilogue also reduces each token row to cross-
// entropy statistics (GemmArgs::ce_stats); an instance of its own, so that
// the plain column GEMM's epilogue carries none of that code.
enum GemmKind : int { GK_COL = 0, GK_COL_SWIGLU = 1, GK_ROW_SUM = 2, GK_ROW_PARTIAL = 3, GK_COL_CE = 4 };


template <int KIND_, bool SWAP_, bool PAIR_ = false>
struct GemmCfg {
  static constexpr int KIND = KIND_;
  static constexpr bool SWAP = SWAP_;
  static constexpr bool PAIR = PAIR_;  // normal mode only: 2-SM MMA over a CTA pair
  static constexpr bool SWIGLU = KIND_ == GK_COL_SWIGLU;
  static constexpr bool IS_COL = KIND_ == GK_COL || KIND_ == GK_COL_SWIGLU || KIND_ == GK_COL_CE;
  static constexpr int NACC = (SWAP_ && SWIGLU) ? 2 : 1;  // A tiles per stage in swap mode
  static constexpr int BM = 128;
  static constexpr int BK = 64;
  static constexpr int A_TILE = BM * BK * 2;               // 16 KB
  static constexpr int A_BYTES = NACC * A_TILE;
  static constexpr int B_ROWS = SWAP_ ? 64 : (PAIR_ ? 128 : 256);  // rows staged by this CTA
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = SWAP_ ? (NACC == 2 ? 5 : 8) : (PAIR_ ? 6 : 4);
  static constexpr int ACC_COLS = SWAP_ ? 128 : 256;      // TMEM columns per accumulator buffer
  static constexpr int TMEM_COLS = 2 * ACC_COLS;
  static constexpr int SLOT_FLOATS = 128 * ACC_COLS;       // one fp32 partial tile
  static constexpr int THREADS = 192;
  static constexpr int OUT_STAGE_BYTES = SWAP_ ? 0 : 4 * 2 * 4096;  // epilogue warps x 2 x (32 rows x 128 B)
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_STAGE_BYTES + 1024 + 512;
};

struct GemmArgs {
  int M;             // tokens
  int Ns;            // normal: output columns of a tile's shard; swap: weight rows per shard
  int tp;
  int Tpad;          // swap: MMA N (tokens padded to a multiple of 16)
  int m_tiles;       // normal: token-block units (pairs of blocks when cluster = 2); swap: weight-row blocks
  int n_tiles;       // normal: output-column blocks per shard; swap: 1
  int num_tiles;
  int r1_tiles;      // tiles enumerated over all shards (the rest: first shard of each replica group)
  int n_q_tiles;     // with rep > 1: column blocks before the replicated K|V columns
  int rep;           // shards sharing one computed K|V tile (1 = no dedup)
  int kb_per_shard;  // ceil(K extent of one shard / 64)
  int kpt;           // k-iterations per tile: kb_per_shard * (ROW_SUM ? tp : 1)
  int dp_tiles;      // tiles processed whole, round-robin
  long long sk_iters;  // k-iterations of tiles [dp_tiles, num_tiles), split evenly over the grid
  int cluster;       // CTAs per cluster: 2 for a CTA-pair launch, else 1
  int act;
  int out_concat;    // COL: 1 -> Y[T][tp*Ns]; 0 -> Y[tp][T][Ns]
  int out_f32;       // ROW_SUM: bias, residual and Y are fp32 (else bf16)
  int tma_store;     // normal mode: outputs go through staging + bulk tensor stores (mapY, mapC)
  const void* bias;               // COL: [tp*Ns]; ROW_SUM: [N]; may be null
  const __nv_bfloat16* bias_up;   // COL_SWIGLU up bias [tp*Ns]; may be null
  const void* residual;           // ROW_SUM: [M][N]; may be null
  void* out;
  float* partials;   // [2 * gridDim.x][SLOT_FLOATS] when sk_iters > 0; split pieces' slots
  // Synchronisation words in the workspace, tagged with this launch's epoch
  // (a 64-bit value no earlier launch used), so that leftover contents read
  // as "not arrived"; the kernel also returns each word it used to zero, so a
  // replayed launch (same epoch, e.g. from a CUDA graph) starts clean:
  // stream-K: [num_tiles - dp_tiles] arrival counters, (epoch << 16) | count;
  // split pieces: [split_units][2][split_ways - 1] flags, equal to epoch when set.
  unsigned long long* sync_words;
  unsigned long long epoch;
  int split_units;   // CTA pairs: units after dp_tiles, each cut into split_ways K pieces
  int split_ways;    // 0 or 1: no split
  // COL on a QKV view: also write the single-key attention context
  // ctx [tp][M][hq/tp * hd] from the V columns (null: no context)
  __nv_bfloat16* ctx;
  int hq, hkv, hd;   // the view's heads (global) and head size
  int a_sharded;     // COL with MN != 0: A is [tp][..] (per shard) and B is shared
  // ROW_SUM: the K loop also runs over a second (A, B) pair (mapA1, mapB1),
  // so that out = sum_s A_s B_s^T + sum_s A'_s B'_s^T in one accumulator
  int two_src;
  // GK_COL_CE (no activation, a vocabulary-split LM head): the epilogue also
  // reduces each token row of the tile to cross-entropy statistics of its
  // logits (taken from the fp32 accumulator), ce_stats[((s * M + t) * n_tiles
  // + n) * 3 + {0, 1, 2}] = {max, sum exp(z - max), the label's logit where
  // the tile holds column labels[t] - s * Ns, else 0}. Null: no statistics.
  const int32_t* ce_labels;
  float* ce_stats;
  // Grouped experts (CTA pairs, whole tiles only): the token rows are the
  // experts' routed tokens, each expert's segment padded to 256-row units;
  // unit_expert[u] is the expert of unit u (see tile_unit_pair), or -1 for an
  // unused unit, which every warp role skips. The weight maps hold the
  // experts' shard sets one after another: shard coordinate e * tp + s.
  const int* unit_expert;
  // Grouped experts: the tile order takes the (column block, shard) pairs in
  // groups of unit_group, every unit per group with the group's pairs
  // fastest, so that a unit's permuted tokens serve unit_group tiles while
  // they are in L2 and no more than that many tiles read them at once
  // (0: units fastest over all pairs).
  int unit_group;
  // Grouped experts: unit_seg[u] = {first unit, units} of the segment that
  // holds unit u (an expert's units; an unused unit is a segment of its
  // own). With it the grouped order runs segment by segment (every group of
  // one expert before the next expert), so an expert's tokens stay in L2
  // across its groups. Null: one segment of all units.
  const int2* unit_seg;
};

// normal mode: the tile's unit (token-block unit, before the cluster rank)
// and its (column block, shard) pair index, in the tile order above
__device__ __forceinline__ void tile_unit_pair(const GemmArgs& a, int tile, int& mu, int& pr) {
  if (a.unit_group > 0 && tile < a.r1_tiles) {
    const int P = a.r1_tiles / a.m_tiles;               // pairs per unit
    // a segment of units u0 .. u0 + nu - 1 owns tiles u0 * P .. (u0 + nu) * P - 1,
    // so the unit tile / P lies in the tile's own segment
    int u0 = 0, nu = a.m_tiles;
    if (a.unit_seg) {
      const int2 sg = __ldg(a.unit_seg + tile / P);
      u0 = sg.x;
      nu = sg.y;
    }
    const int rem = tile - u0 * P;
    const int g = rem / (nu * a.unit_group);
    const int base = g * a.unit_group;
    const int gl = min(a.unit_group, P - base);         // the last group may be partial
    const int r2 = rem - g * nu * a.unit_group;
    mu = u0 + r2 / gl;
    pr = base + r2 % gl;
  } else {
    mu = tile % a.m_tiles;
    pr = tile / a.m_tiles;
  }
}

// ---------------------------------------------------------------------------
// Schedule helpers (identical in every role, so all roles see one sequence)
// ---------------------------------------------------------------------------
struct Seg {
  int tile, kb0, kb1;
};

__device__ __forceinline__ long long sk_begin(const GemmArgs& a, int c) {
  return a.sk_iters * c / gridDim.x;
}
// The CTA whose stream-K range holds iteration i (every range is non-empty).
__device__ __forceinline__ int sk_cta_of(const GemmArgs& a, long long i) {
  return static_cast<int>(((i + 1) * gridDim.x - 1) / a.sk_iters);
}

struct SegIter {
  int dp_next;
  bool piece_left;
  long long i, i_end;
  __device__ explicit SegIter(const GemmArgs& a) {
    dp_next = blockIdx.x / a.cluster;  // the CTAs of a cluster walk the same tiles
    piece_left = a.split_ways > 1 && static_cast<int>(blockIdx.x / a.cluster) < a.split_units * a.split_ways;
    i = sk_begin(a, blockIdx.x);
    i_end = sk_begin(a, blockIdx.x + 1);
  }
  __device__ bool next(const GemmArgs& a, Seg& s) {
    while (dp_next < a.dp_tiles) {
      const int t = dp_next;
      dp_next += gridDim.x / a.cluster;
      if (a.unit_expert) {  // an unused expert unit
        int mu, pr;
        tile_unit_pair(a, t, mu, pr);
        if (__ldg(a.unit_expert + mu) < 0) continue;
      }
      s.tile = t;
      s.kb0 = 0;
      s.kb1 = a.kpt;
      return true;
    }
    if (piece_left) {  // this pair's piece of the split last round
      piece_left = false;
      const int q = static_cast<int>(blockIdx.x / a.cluster);
      const int j = q / a.split_units;
      s.tile = a.dp_tiles + q % a.split_units;
      s.kb0 = static_cast<int>(static_cast<long long>(j) * a.kpt / a.split_ways);
      s.kb1 = static_cast<int>(static_cast<long long>(j + 1) * a.kpt / a.split_ways);
      return true;
    }
    if (i < i_end) {
      const long long t = i / a.kpt;
      s.tile = a.dp_tiles + static_cast<int>(t);
      s.kb0 = static_cast<int>(i - t * a.kpt);
      const long long left = i_end - i;
      s.kb1 = static_cast<int>(left < a.kpt - s.kb0 ? s.kb0 + left : a.kpt);
      i += s.kb1 - s.kb0;
      return true;
    }
    return false;
  }
};

// normal mode: tile -> (token block m, column block n, shard s); `rank` is
// the CTA's rank in its cluster (token block m = unit * cluster + rank)
__device__ __forceinline__ void decode_tile_normal(const GemmArgs& a, int tile, int rank, int& m, int& n,
                                                   int& s) {
  if (tile < a.r1_tiles) {
    const int nq = a.rep > 1 ? a.n_q_tiles : a.n_tiles;
    int r;
    tile_unit_pair(a, tile, m, r);
    n = r % nq;
    s = r / nq;
  } else {
    const int t2 = tile - a.r1_tiles;
    const int nk = a.n_tiles - a.n_q_tiles;
    m = t2 % a.m_tiles;
    const int r = t2 / a.m_tiles;
    n = a.n_q_tiles + r % nk;
    s = (r / nk) * a.rep;
  }
  m = m * a.cluster + rank;
}

// swap mode: tile -> (weight-row block m, shard s); ROW_SUM has s = 0
__device__ __forceinline__ void decode_tile_swap(const GemmArgs& a, int tile, int& m, int& s) {
  m = tile % a.m_tiles;
  s = tile / a.m_tiles;
}

// Count one arrival on an epoch-tagged counter ((epoch << 16) | count; a
// word left by any other launch reads as zero arrivals) and return the count
// including this one.
__device__ __forceinline__ int arrive_tagged(unsigned long long* word, unsigned long long epoch) {
  const unsigned long long tag = epoch & ((1ull << 48) - 1);
  unsigned long long cur = atomicAdd(word, 0ull);
  for (;;) {
    const unsigned long long nv = ((cur >> 16) == tag) ? cur + 1 : ((tag << 16) | 1ull);
    const unsigned long long prev = atomicCAS(word, cur, nv);
    if (prev == cur) return static_cast<int>(nv & 0xFFFFull);
    cur = prev;
  }
}

// Named barrier 1 over the 128 epilogue threads (warps 2..5).
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Barrier over the 128 epilogue threads that also ORs a predicate across
// them, so every epilogue warp takes the same branch (no warp can be left
// waiting at a later named barrier for one that gave up).
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void load_bf16x8_f(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
  v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
}
__device__ __forceinline__ void store_bf16x8_f(__nv_bfloat16* p, const float* v) {
  uint4 q;
  q.x = pack_bf16x2(v[0], v[1]); q.y = pack_bf16x2(v[2], v[3]);
  q.z = pack_bf16x2(v[4], v[5]); q.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = q;
}

// ---------------------------------------------------------------------------
// Accumulator sources for the epilogue: TMEM, or the sum of workspace pieces.
// Partial slot layout: float4 index (col/4) * 128 + row, so a warp's 32 rows
// read and write 512 contiguous bytes.
// ---------------------------------------------------------------------------
struct TmemSrc {
  uint32_t t_acc;  // lane quadrant + accumulator buffer already applied
  template <int N>
  __device__ __forceinline__ void fetch(int col, float* v) const {
    if constexpr (N == 32) {
      uint32_t r[32];
      tmem_ld32(t_acc + col, r);
      tmem_ld_wait_regs(r);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    } else {
      uint32_t r[16];
      tmem_ld16(t_acc + col, r);
      tmem_ld_wait_regs(r);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
    }
  }
};

struct PartialSrc {
  const float* ws;  // partial workspace base
  int slot_floats;
  int c_first, c_last;  // CTAs whose pieces make up this tile, in k order
  int row;              // this thread's row within the tile
  const GemmArgs* a;
  int tile_local;       // tile - dp_tiles
  __device__ __forceinline__ const float4* slot_ptr(int c) const {
    const long long f = a->sk_iters * c / gridDim.x;
    const int first_local = static_cast<int>(f / a->kpt);
    const int slot = 2 * c + (first_local == tile_local ? 0 : 1);
    return reinterpret_cast<const float4*>(ws + static_cast<size_t>(slot) * slot_floats);
  }
  template <int N>
  __device__ __forceinline__ void fetch(int col, float* v) const {
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] = 0.0f;
    for (int c = c_first; c <= c_last; ++c) {
      const float4* p = slot_ptr(c);
#pragma unroll
      for (int j4 = 0; j4 < N / 4; ++j4) {
        const float4 q = __ldcg(p + static_cast<size_t>(col / 4 + j4) * 128 + row);
        v[4 * j4 + 0] += q.x; v[4 * j4 + 1] += q.y; v[4 * j4 + 2] += q.z; v[4 * j4 + 3] += q.w;
      }
    }
  }
};

// The owner piece of a split unit: the other pieces' slots (j = 0..ways-2,
// this CTA rank, in that order) summed, then this CTA's own accumulator.
struct SplitSrc {
  uint32_t t_acc;
  const float* slot0;   // slot of piece 0; piece j's slot is 2 * j slots further
  int row;
  int others;           // split_ways - 1
  template <int N>
  __device__ __forceinline__ void fetch(int col, float* v) const {
    float own[N];
    TmemSrc{t_acc}.template fetch<N>(col, own);
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] = 0.0f;
    for (int p = 0; p < others; ++p) {
      const float4* sp = reinterpret_cast<const float4*>(slot0 + static_cast<size_t>(2 * p) * (128 * 256));
#pragma unroll
      for (int j4 = 0; j4 < N / 4; ++j4) {
        const float4 q = __ldcg(sp + static_cast<size_t>(col / 4 + j4) * 128 + row);
        v[4 * j4 + 0] += q.x; v[4 * j4 + 1] += q.y; v[4 * j4 + 2] += q.z; v[4 * j4 + 3] += q.w;
      }
    }
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] += own[j];
  }
};

// Store this thread's accumulator row (ncols columns) from TMEM into a slot.
template <int CHUNK>
__device__ __forceinline__ void store_partial(uint32_t t_acc, float* slot, int row, int ncols) {
  float4* p = reinterpret_cast<float4*>(slot);
  for (int c = 0; c < ncols; c += CHUNK) {
    float v[CHUNK];
    TmemSrc{t_acc}.template fetch<CHUNK>(c, v);
#pragma unroll
    for (int j4 = 0; j4 < CHUNK / 4; ++j4)
      __stcg(p + static_cast<size_t>(c / 4 + j4) * 128 + row,
             make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]));
  }
}

// ---------------------------------------------------------------------------
// Single-key attention context, written from the QKV epilogue. With every
// query attending only to its own token the softmax weight is 1, so the
// context of query head g is V of its kv head g / (hq / hkv). A V column of
// shard s (shard-local column n in the V block) is copied to each query head
// that reads it, on each of the `copies` shards s, s+1, ... that hold it.
// ---------------------------------------------------------------------------
struct CtxMap {
  int nq, nkv, group, vcol0, hd;
  __device__ explicit CtxMap(const GemmArgs& a) {
    nq = a.hq / a.tp;
    nkv = a.hkv >= a.tp ? a.hkv / a.tp : 1;
    group = a.hq / a.hkv;
    vcol0 = (nq + nkv) * a.hd;
    hd = a.hd;
  }
  __device__ int kv_first(const GemmArgs& a, int s) const {
    return a.hkv >= a.tp ? s * nkv : (s * a.hkv) / a.tp;
  }
};

// W elements (W = 8: one 16-byte vector; W = 1: one element) at V column n.
template <int W>
__device__ __forceinline__ void store_ctx(const GemmArgs& a, const CtxMap& cm, int s, int copies, int row,
                                          int n, const float* v) {
  const int i = (n - cm.vcol0) / cm.hd;        // kv head within the shard's V block
  const int d = n - cm.vcol0 - i * cm.hd;      // position in the head
  const int kvh = cm.kv_first(a, s) + i;       // global kv head (the same on every replica)
  const size_t nc = static_cast<size_t>(cm.nq) * cm.hd;
  for (int r = 0; r < copies; ++r) {
    const int s2 = s + r;
    const int g0 = max(s2 * cm.nq, kvh * cm.group);
    const int g1 = min((s2 + 1) * cm.nq, (kvh + 1) * cm.group);
    __nv_bfloat16* base = a.ctx + (static_cast<size_t>(s2) * a.M + row) * nc + d;
    for (int g = g0; g < g1; ++g) {
      __nv_bfloat16* p = base + static_cast<size_t>(g - s2 * cm.nq) * cm.hd;
      if constexpr (W == 8) store_bf16x8_f(p, v);
      else *p = __float2bfloat16_rn(v[0]);
    }
  }
}

// ---------------------------------------------------------------------------
// Tile epilogues
// ---------------------------------------------------------------------------
// Output staging for TMA stores (normal mode). Each epilogue warp owns 32
// token rows of the tile and two 4 KB buffers. A chunk of 128 bytes per row
// (64 bf16 or 32 fp32 columns) is written by its 32 threads, one row each,
// into a buffer in the 128-byte-swizzled layout of the output tensor map,
// then one thread stores the 32 x 128 B box with a bulk tensor copy (to
// every destination: replica shards, context slots). The copy engine writes
// whole lines and clips rows and columns outside the output.
struct OutStage {
  uint8_t* buf;              // this warp's two staging buffers (null: per-thread stores)
  const CUtensorMap* mapY;   // output
  const CUtensorMap* mapC;   // attention context (COL with a context)
  int next;                  // buffer filled next
  int row0;                  // first token row of the warp's 32 rows
  int lane;
};

// Wait until the buffer about to be filled has been read by its last store.
__device__ __forceinline__ uint8_t* stage_acquire(OutStage& o) {
  if (o.lane == 0) tma_store_wait_read<1>();
  __syncwarp();
  return o.buf + o.next * 4096;
}
// 16-byte piece c16 (0..7) of this thread's 128-byte row, swizzled.
__device__ __forceinline__ void stage_put(uint8_t* b, int lane, int c16, uint4 v) {
  *reinterpret_cast<uint4*>(b + lane * 128 + ((c16 ^ (lane & 7)) << 4)) = v;
}
// Make the warp's staged rows visible to the copy engine.
__device__ __forceinline__ void stage_ready() {
  fence_proxy_async_smem();
  __syncwarp();
}
__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// Online cross-entropy statistics of one token row over a tile's columns:
// the running maximum m, the sum S of exp(z - m), and the label's logit.
struct CeAcc {
  float m, S, zy;
};
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(x) = 2^(x log2 e)
// 32 logits at once (columns past the shard hold -inf): one maximum and at
// most one rescale per 32, each exponential one FMA and a MUFU 2^x.
__device__ __forceinline__ void ce_add32(CeAcc& c, const float* z) {
  float mx = z[0];
#pragma unroll
  for (int j = 1; j < 32; ++j) mx = fmaxf(mx, z[j]);
  if (mx > c.m) {
    c.S *= ex2_approx((c.m - mx) * kLog2e);  // 2^-inf = 0 on the first chunk
    c.m = mx;
  }
  if (c.m == -INFINITY) return;  // no column of this row seen yet
  const float mb = c.m * kLog2e;
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    s0 += ex2_approx(fmaf(z[j], kLog2e, -mb));
    s1 += ex2_approx(fmaf(z[j + 1], kLog2e, -mb));
  }
  c.S += s0 + s1;
}

// normal mode: this thread owns token row `row`; columns are output features.
template <class Cfg, class Src>
__device__ __forceinline__ void epilogue_normal(const GemmArgs& a, const Src& src, int row, int n_blk, int s,
                                                OutStage& os) {
  const bool row_ok = row < a.M;
  if constexpr (Cfg::IS_COL) {
    constexpr int NOUT = Cfg::SWIGLU ? 128 : 256;
    const int n0 = n_blk * NOUT;
    const int copies = (a.rep > 1 && n_blk >= a.n_q_tiles) ? a.rep : 1;
    __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.out);
    const __nv_bfloat16* bias =
        a.bias ? static_cast<const __nv_bfloat16*>(a.bias) + static_cast<size_t>(s) * a.Ns : nullptr;
    const __nv_bfloat16* bias_up = a.bias_up ? a.bias_up + static_cast<size_t>(s) * a.Ns : nullptr;
    const bool with_ctx = !Cfg::SWIGLU && a.ctx != nullptr;
    const bool with_ce = Cfg::KIND == GK_COL_CE && a.ce_stats != nullptr;
    CeAcc ce{-INFINITY, 0.0f, 0.0f};
    const int ce_loc = (with_ce && row_ok) ? __ldg(a.ce_labels + row) - s * a.Ns : -1;  // the label's shard column
#pragma unroll 1
    for (int cc = 0; cc < NOUT; cc += 64) {  // one 128-byte chunk of bf16 per row
      uint8_t* sb = os.buf ? stage_acquire(os) : nullptr;
#pragma unroll 1
      for (int h = 0; h < 64; h += 32) {
        const int c = cc + h;
        float g[32];
        src.template fetch<32>(c, g);
        float u[Cfg::SWIGLU ? 32 : 1];
        if constexpr (Cfg::SWIGLU) src.template fetch<32>(NOUT + c, u);
#pragma unroll
        for (int j8 = 0; j8 < 32; j8 += 8) {
          const int n = n0 + c + j8;
          const bool col_ok = n < a.Ns;
          float v[8], b[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = g[j8 + j];
          if (bias && col_ok) {
            load_bf16x8_f(bias + n, b);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] += b[j];
          }
          if constexpr (Cfg::SWIGLU) {
            float w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = u[j8 + j];
            if (bias_up && col_ok) {
              load_bf16x8_f(bias_up + n, b);
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] += b[j];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = act_silu(v[j]) * w[j];
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = apply_act(a.act, v[j]);
            if (with_ce) {  // the chunk's logits, kept for its statistics below
#pragma unroll
              for (int j = 0; j < 8; ++j) g[j8 + j] = col_ok ? v[j] : -INFINITY;
              if (col_ok && ce_loc >= n && ce_loc < n + 8) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (ce_loc == n + j) ce.zy = v[j];
              }
            }
          }
          if (sb) {
            stage_put(sb, os.lane, (h + j8) >> 3, pack_bf16x8(v));
          } else if (row_ok && col_ok) {
            for (int r = 0; r < copies; ++r) {
              const size_t sr = static_cast<size_t>(s + r);
              const size_t off = a.out_concat
                                     ? static_cast<size_t>(row) * (static_cast<size_t>(a.tp) * a.Ns) + sr * a.Ns + n
                                     : (sr * a.M + row) * static_cast<size_t>(a.Ns) + n;
              store_bf16x8_f(Y + off, v);
            }
            if constexpr (!Cfg::SWIGLU) {
              if (with_ctx) {
                const CtxMap cm(a);
                if (n >= cm.vcol0) store_ctx<8>(a, cm, s, copies, row, n, v);
              }
            }
          }
        }
        if constexpr (!Cfg::SWIGLU) {
          if (with_ce) ce_add32(ce, g);
        }
      }
      if (sb) {
        stage_ready();
        if (os.lane == 0) {
          const int n = n0 + cc;
          if (n < a.Ns && os.row0 < a.M) {  // boxes wholly outside the output are not issued
            for (int r = 0; r < copies; ++r) tma_store_3d(os.mapY, sb, n, os.row0, s + r);
            if constexpr (!Cfg::SWIGLU) {
              if (with_ctx) {
                // the chunk lies in one head (hd % 64 == 0 on this path): store it to
                // every query head that reads it, on every replica shard
                const CtxMap cm(a);
                if (n >= cm.vcol0) {
                  const int i = (n - cm.vcol0) / cm.hd;
                  const int d = n - cm.vcol0 - i * cm.hd;
                  const int kvh = cm.kv_first(a, s) + i;
                  for (int r = 0; r < copies; ++r) {
                    const int s2 = s + r;
                    const int g0 = max(s2 * cm.nq, kvh * cm.group);
                    const int g1 = min((s2 + 1) * cm.nq, (kvh + 1) * cm.group);
                    for (int gq = g0; gq < g1; ++gq)
                      tma_store_3d(os.mapC, sb, (gq - s2 * cm.nq) * cm.hd + d, os.row0, s2);
                  }
                }
              }
            }
          }
          tma_store_commit();
        }
        os.next ^= 1;
      }
    }
    if (with_ce && row_ok) {
      float* o = a.ce_stats + ((static_cast<size_t>(s) * a.M + row) * a.n_tiles + n_blk) * 3;
      o[0] = ce.m;
      o[1] = ce.S;
      o[2] = ce.zy;
    }
  } else if constexpr (Cfg::KIND == GK_ROW_SUM) {
    const int n0 = n_blk * 256;
    const size_t row_off = static_cast<size_t>(row) * a.Ns;
    if (a.out_f32) {  // fp32 bias / residual / output (an fp32 residual stream)
      const float* bias = static_cast<const float*>(a.bias);
      const float* res = static_cast<const float*>(a.residual);
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {  // one 128-byte chunk of fp32 per row
        uint8_t* sb = os.buf ? stage_acquire(os) : nullptr;
        float g[32];
        src.template fetch<32>(c, g);
#pragma unroll
        for (int j4 = 0; j4 < 32; j4 += 4) {
          const int n = n0 + c + j4;
          const bool col_ok = n < a.Ns;
          float4 v = make_float4(g[j4], g[j4 + 1], g[j4 + 2], g[j4 + 3]);
          if (bias && col_ok) {
            const float4 p = __ldg(reinterpret_cast<const float4*>(bias + n));
            v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
          }
          if (res && row_ok && col_ok) {  // may alias Y: read here, before this chunk is stored
            const float4 p = *reinterpret_cast<const float4*>(res + row_off + n);
            v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
          }
          if (sb) {
            stage_put(sb, os.lane, j4 >> 2,
                      make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                                 __float_as_uint(v.w)));
          } else if (row_ok && col_ok) {
            *reinterpret_cast<float4*>(static_cast<float*>(a.out) + row_off + n) = v;
          }
        }
        if (sb) {
          stage_ready();
          if (os.lane == 0) {
            if (n0 + c < a.Ns && os.row0 < a.M) tma_store_3d(os.mapY, sb, n0 + c, os.row0, 0);
            tma_store_commit();
          }
          os.next ^= 1;
        }
      }
    } else {
      const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(a.bias);
      const __nv_bfloat16* res = static_cast<const __nv_bfloat16*>(a.residual);
#pragma unroll 1
      for (int cc = 0; cc < 256; cc += 64) {  // one 128-byte chunk of bf16 per row
        uint8_t* sb = os.buf ? stage_acquire(os) : nullptr;
#pragma unroll 1
        for (int h = 0; h < 64; h += 32) {
          const int c = cc + h;
          float g[32];
          src.template fetch<32>(c, g);
#pragma unroll
          for (int j8 = 0; j8 < 32; j8 += 8) {
            const int n = n0 + c + j8;
            const bool col_ok = n < a.Ns;
            float v[8], b[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = g[j8 + j];
            if (bias && col_ok) {
              load_bf16x8_f(bias + n, b);
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] += b[j];
            }
            if (res && row_ok && col_ok) {  // plain load: may alias Y (read before this chunk is stored)
              const uint4 q = *reinterpret_cast<const uint4*>(res + row_off + n);
              v[0] += bf16_lo(q.x); v[1] += bf16_hi(q.x); v[2] += bf16_lo(q.y); v[3] += bf16_hi(q.y);
              v[4] += bf16_lo(q.z); v[5] += bf16_hi(q.z); v[6] += bf16_lo(q.w); v[7] += bf16_hi(q.w);
            }
            if (sb) stage_put(sb, os.lane, (h + j8) >> 3, pack_bf16x8(v));
            else if (row_ok && col_ok) store_bf16x8_f(static_cast<__nv_bfloat16*>(a.out) + row_off + n, v);
          }
        }
        if (sb) {
          stage_ready();
          if (os.lane == 0) {
            if (n0 + cc < a.Ns && os.row0 < a.M) tma_store_3d(os.mapY, sb, n0 + cc, os.row0, 0);
            tma_store_commit();
          }
          os.next ^= 1;
        }
      }
    }
  } else {  // GK_ROW_PARTIAL: fp32 [tp][M][N]
    const int n0 = n_blk * 256;
    float* P = static_cast<float*>(a.out);
    const size_t row_off = (static_cast<size_t>(s) * a.M + row) * static_cast<size_t>(a.Ns);
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
      uint8_t* sb = os.buf ? stage_acquire(os) : nullptr;
      float g[32];
      src.template fetch<32>(c, g);
#pragma unroll
      for (int j4 = 0; j4 < 32; j4 += 4) {
        const int n = n0 + c + j4;
        if (sb)
          stage_put(sb, os.lane, j4 >> 2,
                    make_uint4(__float_as_uint(g[j4]), __float_as_uint(g[j4 + 1]), __float_as_uint(g[j4 + 2]),
                               __float_as_uint(g[j4 + 3])));
        else if (row_ok && n < a.Ns)
          *reinterpret_cast<float4*>(P + row_off + n) = make_float4(g[j4], g[j4 + 1], g[j4 + 2], g[j4 + 3]);
      }
      if (sb) {
        stage_ready();
        if (os.lane == 0) {
          if (n0 + c < a.Ns && os.row0 < a.M) tma_store_3d(os.mapY, sb, n0 + c, os.row0, s);
          tma_store_commit();
        }
        os.next ^= 1;
      }
    }
  }
}

// swap mode: this thread owns weight row `wrow` (an output feature); the
// accumulator columns are tokens (gate at [0, Tpad), up at [Tpad, 2*Tpad)).
template <class Cfg, class Src>
__device__ __forceinline__ void epilogue_swap(const GemmArgs& a, const Src& src, int wrow, int s) {
  const bool ok = wrow < a.Ns;
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.out);
  float bg = 0.0f, bu = 0.0f;
  if constexpr (Cfg::IS_COL) {
    if (ok && a.bias)
      bg = __bfloat162float(static_cast<const __nv_bfloat16*>(a.bias)[static_cast<size_t>(s) * a.Ns + wrow]);
    if constexpr (Cfg::SWIGLU)
      if (ok && a.bias_up) bu = __bfloat162float(a.bias_up[static_cast<size_t>(s) * a.Ns + wrow]);
  } else {
    if (ok && a.bias)
      bg = a.out_f32 ? static_cast<const float*>(a.bias)[wrow]
                     : __bfloat162float(static_cast<const __nv_bfloat16*>(a.bias)[wrow]);
  }
#pragma unroll 1
  for (int t0 = 0; t0 < a.M; t0 += 16) {
    float g[16];
    src.template fetch<16>(t0, g);
    float u[Cfg::SWIGLU ? 16 : 1];
    if constexpr (Cfg::SWIGLU) src.template fetch<16>(a.Tpad + t0, u);
    if (!ok) continue;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int t = t0 + j;
      if (t >= a.M) break;
      float v = g[j] + bg;
      if constexpr (Cfg::IS_COL) {
        if constexpr (Cfg::SWIGLU) v = act_silu(v) * (u[j] + bu);
        else v = apply_act(a.act, v);
        const size_t off = a.out_concat
                               ? static_cast<size_t>(t) * (static_cast<size_t>(a.tp) * a.Ns) +
                                     static_cast<size_t>(s) * a.Ns + wrow
                               : (static_cast<size_t>(s) * a.M + t) * static_cast<size_t>(a.Ns) + wrow;
        Y[off] = __float2bfloat16_rn(v);
        if constexpr (!Cfg::SWIGLU) {
          if (a.ctx) {
            const CtxMap cm(a);
            if (wrow >= cm.vcol0) store_ctx<1>(a, cm, s, 1, t, wrow, &v);
          }
        }
      } else {  // ROW_SUM
        const size_t off = static_cast<size_t>(t) * a.Ns + wrow;
        if (a.out_f32) {
          if (a.residual) v += static_cast<const float*>(a.residual)[off];
          static_cast<float*>(a.out)[off] = v;
        } else {
          if (a.residual) v += __bfloat162float(static_cast<const __nv_bfloat16*>(a.residual)[off]);
          Y[off] = __float2bfloat16_rn(v);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int KIND, bool SWAP, bool PAIR, int MN = 0>
__global__ void __launch_bounds__(192, 1)
    tp_gemm_kernel(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapA1,
                   const __grid_constant__ CUtensorMap mapB0, const __grid_constant__ CUtensorMap mapB1,
                   const __grid_constant__ CUtensorMap mapY, const __grid_constant__ CUtensorMap mapC,
                   const GemmArgs args) {
  using Cfg = GemmCfg<KIND, SWAP, PAIR>;
  static_assert(!(PAIR && SWAP), "CTA pairs are a token-major arrangement");
  static_assert(MN == 0 || (PAIR && (KIND == GK_COL || KIND == GK_ROW_SUM)),
                "MN-major operands: CTA pairs, COL or ROW_SUM");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* out_stage = smem + Cfg::STAGES * Cfg::STAGE_BYTES;  // epilogue staging (normal mode)
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + Cfg::OUT_STAGE_BYTES);
  uint64_t* full = bars;                        // [STAGES]  TMA -> MMA
  uint64_t* empty = bars + Cfg::STAGES;         // [STAGES]  MMA -> TMA
  uint64_t* tfull = bars + 2 * Cfg::STAGES;     // [2]       MMA -> epilogue
  uint64_t* tempty = tfull + 2;                 // [2]       epilogue -> MMA
  uint64_t* drain = tempty + 2;                 // [1]       abort path only
  uint64_t* xch = drain + 1;                    // [1]       abort path, CTA pairs: odd -> even (counts written)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xch + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;
  // abort path, CTA pairs: the odd CTA's last issued use of each stage,
  // written into the even CTA
  volatile int* peer_issued = last_flag + 1;    // [STAGES]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;  // 0: the pair's MMA issuer

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], PAIR ? 8 : 4);  // the epilogue warps of both CTAs of a pair
    }
    mbar_init(drain, 1);
    mbar_init(xch, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mapA0);
    tma_prefetch_desc(&mapB0);
    if (Cfg::SWIGLU) {
      tma_prefetch_desc(&mapA1);
      tma_prefetch_desc(&mapB1);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before either signals the other
  // Setup above may overlap the previous kernel of the stream; every global
  // memory access below comes after it has completed. The next kernel may
  // begin its own setup on SMs this launch leaves idle.
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer ------------------------------
      // The pair's full barrier counts both CTAs' bytes; only the even CTA arms it.
      const uint32_t stage_tx = SWAP ? static_cast<uint32_t>(Cfg::A_BYTES + args.Tpad * 128)
                                     : static_cast<uint32_t>((PAIR ? 2 : 1) * Cfg::STAGE_BYTES);
      int stage = 0;
      uint32_t phase = 0;
      int round = 0;            // passes over the ring so far: the use index of each stage this pass
      int issued[Cfg::STAGES];  // per stage: the use index of the last load issued, or -1
#pragma unroll
      for (int i = 0; i < Cfg::STAGES; ++i) issued[i] = -1;
      // test-only: withhold one load (the flag is consumed by the first launch that sees it)
      // (kind 1: block 0, the even CTA of a pair; kind 2: block 1, the odd one)
      const int inj = g_tp_inject;
      bool skip_one = (inj == 1 || inj == 2) && static_cast<int>(blockIdx.x) == inj - 1 &&
                      atomicExch(&g_tp_inject, 0) == inj;
      bool ok = true;

      SegIter it(args);
      Seg sg;
      while (ok && it.next(args, sg)) {
        int m, n = 0, s;
        if constexpr (SWAP) decode_tile_swap(args, sg.tile, m, s);
        else decode_tile_normal(args, sg.tile, rank, m, n, s);
        // grouped experts: the tile's expert selects its shard set
        int wks = 0;
        if (args.unit_expert) {
          int mu, pr;
          tile_unit_pair(args, sg.tile, mu, pr);
          wks = __ldg(args.unit_expert + mu) * args.tp;
        }
        for (int kb_i = sg.kb0; kb_i < sg.kb1; ++kb_i) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (skip_one) {
            skip_one = false;
          } else {
            int ks, kb;
            bool src1 = false;  // ROW_SUM with two sources: the second (A, B) pair
            if constexpr (KIND == GK_ROW_SUM) {
              ks = kb_i / args.kb_per_shard;
              kb = kb_i - ks * args.kb_per_shard;
              if (ks >= args.tp) {
                src1 = true;
                ks -= args.tp;
              }
            } else {
              ks = s;
              kb = kb_i;
            }
            uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
            uint8_t* sb = sa + Cfg::A_BYTES;
            if constexpr (PAIR) {
              if (rank == 0) mbar_arrive_expect_tx(&full[stage], stage_tx);
              const uint32_t fb = mapa_shared(&full[stage], 0);
              const int a_s = Cfg::IS_COL ? (args.a_sharded ? s : 0) : ks;
              const int b_s = (args.a_sharded ? 0 : ks) + wks;
              const CUtensorMap* ma = src1 ? &mapA1 : &mapA0;
              if constexpr (MN & 1) {  // [K][M]: M columns m*128 .. +127 as two panels
                tma_load_3d_pair(sa, ma, fb, m * 128, kb * 64, a_s);
                tma_load_3d_pair(sa + Cfg::A_TILE / 2, ma, fb, m * 128 + 64, kb * 64, a_s);
              } else {
                tma_load_3d_pair(sa, ma, fb, kb * 64, m * 128, a_s);
              }
              if constexpr (Cfg::SWIGLU) {
                tma_load_3d_pair(sb, rank ? &mapB1 : &mapB0, fb, kb * 64, n * 128, ks + wks);
              } else if constexpr ((MN & 2) != 0) {  // [K][N]: this CTA's 128 of the 256 N columns
                const CUtensorMap* mb = src1 ? &mapB1 : &mapB0;
                const int n0 = n * 256 + rank * 128;
                tma_load_3d_pair(sb, mb, fb, n0, kb * 64, b_s);
                tma_load_3d_pair(sb + Cfg::B_BYTES / 2, mb, fb, n0 + 64, kb * 64, b_s);
              } else {
                tma_load_3d_pair(sb, src1 ? &mapB1 : &mapB0, fb, kb * 64, n * 256 + rank * 128, b_s);
              }
            } else {
              mbar_arrive_expect_tx(&full[stage], stage_tx);
              if constexpr (SWAP) {
                // A: weight rows of shard ks; B: token rows (X for COL, Hs[ks] for ROW)
                // L2 priorities: each weight byte is read once here, so its lines
                // go first and the token rows stay (token-major tiles reuse both
                // operands across a round; hints measured no gain there)
                const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
                tma_load_3d_hint(sa, &mapA0, &full[stage], kb * 64, m * 128, ks, pol_w);
                if constexpr (Cfg::NACC == 2)
                  tma_load_3d_hint(sa + Cfg::A_TILE, &mapA1, &full[stage], kb * 64, m * 128, ks, pol_w);
                tma_load_3d_hint(sb, &mapB0, &full[stage], kb * 64, 0, Cfg::IS_COL ? 0 : ks, pol_x);
              } else {
                tma_load_3d(sa, &mapA0, &full[stage], kb * 64, m * 128, Cfg::IS_COL ? 0 : ks);
                if constexpr (Cfg::SWIGLU) {
                  tma_load_3d(sb, &mapB0, &full[stage], kb * 64, n * 128, ks);
                  tma_load_3d(sb + Cfg::B_BYTES / 2, &mapB1, &full[stage], kb * 64, n * 128, ks);
                } else {
                  tma_load_3d(sb, &mapB0, &full[stage], kb * 64, n * 256, ks);
                }
              }
            }
            issued[stage] = round;
          }
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
            ++round;
          }
        }
      }
      if constexpr (PAIR) {
        // wait until the pair's MMAs have released every stage, so that no
        // commit from the even CTA is still on its way to this CTA's barriers
        for (int i = 0; ok && i < Cfg::STAGES; ++i) {
          ok = mbar_wait(&empty[stage], phase ^ 1u, abort_flag);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let every copy this block started land before it exits
        if constexpr (!PAIR) {
          for (int i = 0; i < Cfg::STAGES; ++i)
            if (issued[i] >= 0) mbar_wait_drain(&full[i], static_cast<uint32_t>(issued[i]) & 1u);
        } else if (rank != 0) {
          // The odd CTA's copies count on the even CTA's full barriers, which
          // it cannot poll: it hands the even CTA its last issued use of each
          // stage, then waits (bounded) until the even CTA reports that every
          // such copy has landed.
          for (int i = 0; i < Cfg::STAGES; ++i)
            st_cluster_u32(mapa_shared(const_cast<int*>(peer_issued + i), 0), static_cast<uint32_t>(issued[i]));
          mbar_arrive_cluster(mapa_shared(xch, 0));  // release: the words above are visible first
          mbar_wait_drain(drain, 0);
        } else {
          // The even CTA: with the odd CTA's counts (if they come within the
          // limit; else the odd CTA is taken to have issued what this one
          // did), make the pending phase of each stage completable and wait
          // for it. At most one phase per stage is pending (a CTA issues use
          // k only once use k - 1 has been consumed): a use the odd CTA
          // issued and this one did not is armed for the odd half alone; a
          // use this one armed that the odd CTA never issued has the odd
          // half counted as arrived. Then the odd CTA may leave.
          const bool got = mbar_wait_drain(xch, 0);
          const uint32_t half = static_cast<uint32_t>(Cfg::STAGE_BYTES);
          for (int i = 0; i < Cfg::STAGES; ++i) {
            const int e = issued[i], o = got ? peer_issued[i] : issued[i];
            const int last = e > o ? e : o;
            if (last < 0) continue;
            if (o == last && e < last) mbar_arrive_expect_tx(&full[i], half);
            else if (e == last && o < last) mbar_complete_tx(&full[i], half);
            mbar_wait_drain(&full[i], static_cast<uint32_t>(last) & 1u);
          }
          if (got) mbar_arrive_cluster(mapa_shared(drain, 1));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------ MMA issuer ------------------------------
      // MN-major operands set the instruction's transpose bits (15: A, 16: B)
      const uint32_t idesc = (SWAP ? idesc_bf16_f32(128, args.Tpad) : idesc_bf16_f32(PAIR ? 256 : 128, 256)) |
                             ((MN & 1) ? (1u << 15) : 0u) | ((MN & 2) ? (1u << 16) : 0u);
      // a K step of 16: +32 bytes inside a K-major row, +16 rows (2048 bytes)
      // of an MN-major panel; descriptor addresses count 16-byte units
      constexpr uint32_t a_step = (MN & 1) ? 128u : 2u, b_step = (MN & 2) ? 128u : 2u;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued_any = false;
      SegIter it(args);
      Seg sg;
      while (ok && it.next(args, sg)) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::ACC_COLS);
        for (int kb_i = sg.kb0; kb_i < sg.kb1; ++kb_i) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint64_t bdesc = (MN & 2) ? smem_desc_mn_sw128(sa + Cfg::A_BYTES, Cfg::B_BYTES / 2, 1024)
                                          : smem_desc_k_sw128(sa + Cfg::A_BYTES);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t accumulate = (kb_i > sg.kb0 || k > 0) ? 1u : 0u;
#pragma unroll
            for (int q = 0; q < Cfg::NACC; ++q) {
              const uint64_t adesc = (MN & 1) ? smem_desc_mn_sw128(sa, Cfg::A_TILE / 2, 1024)
                                              : smem_desc_k_sw128(sa + q * Cfg::A_TILE);
              if constexpr (PAIR)
                tc_mma_bf16_pair(d_tmem, adesc + a_step * k, bdesc + b_step * k, idesc, accumulate);
              else
                tc_mma_bf16(d_tmem + static_cast<uint32_t>(q * args.Tpad), adesc + 2 * k, bdesc + 2 * k,
                            idesc, accumulate);
            }
          }
          if constexpr (PAIR) tc_commit_pair_both(&empty[stage]);
          else tc_commit(&empty[stage]);
          issued_any = true;
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR) tc_commit_pair_both(&tfull[acc]);
        else tc_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok && issued_any) {  // wait for MMAs in flight before TMEM is freed
        if constexpr (PAIR) tc_commit_pair_local(drain);
        else tc_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;        // TMEM lane quadrant this warp may access
    const int row = q * 32 + lane; // row of the 128-row tile
    OutStage os{(!SWAP && args.tma_store) ? out_stage + (warp - 2) * 8192 : nullptr, &mapY, &mapC, 0, 0, lane};
    int acc = 0;
    uint32_t acc_phase = 0;
    SegIter it(args);
    Seg sg;
    while (it.next(args, sg)) {
      const bool waited = mbar_wait(&tfull[acc], acc_phase, abort_flag);
      if (epi_any(!waited || *abort_flag)) break;  // uniform over the four epilogue warps
      tc_fence_after();
      const uint32_t t_acc =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * Cfg::ACC_COLS);
      int m, n = 0, s;
      if constexpr (SWAP) decode_tile_swap(args, sg.tile, m, s);
      else decode_tile_normal(args, sg.tile, rank, m, n, s);
      os.row0 = m * 128 + q * 32;
      const bool whole = sg.kb0 == 0 && sg.kb1 == args.kpt;
      if constexpr (PAIR && KIND == GK_ROW_SUM) {  // only row GEMMs split their last round
        if (!whole) {
          // a piece of a split unit: slots per (unit u, piece j < ways-1, rank),
          // counters per (unit u, rank)
          const int q = static_cast<int>(blockIdx.x / 2);
          const int u = q % args.split_units, j = q / args.split_units;
          const int others = args.split_ways - 1;
          float* slot0 = args.partials + (static_cast<size_t>(u) * others * 2 + rank) * (128 * 256);
          volatile unsigned long long* flags = args.sync_words + (static_cast<size_t>(u) * 2 + rank) * others;
          if (j < others) {
            store_partial<32>(t_acc, slot0 + static_cast<size_t>(2 * j) * (128 * 256), row, 256);
            tc_fence_before();
            __syncwarp();
            __threadfence();
            epi_bar();
            if (threadIdx.x == 64) {
              __threadfence();
              flags[j] = args.epoch;
            }
          } else {
            // the owner: wait (bounded) until the other pieces have parked their slots
            if (threadIdx.x == 64) {
              const uint64_t t0 = globaltimer_ns();
              const uint64_t limit = g_tp_wait_limit_ns;
              bool ok = true;
              for (int p = 0; ok && p < others; ++p) {
                while (flags[p] != args.epoch) {
                  if (*abort_flag || globaltimer_ns() - t0 > limit) {
                    atomicCAS(&g_tp_error, TP_DEVERR_NONE, TP_DEVERR_WAIT_TIMEOUT);
                    *abort_flag = 1;
                    ok = false;
                    break;
                  }
                }
              }
              __threadfence();
              *last_flag = ok ? 1 : 0;
            }
            epi_bar();
            if (*last_flag) {
              SplitSrc src{t_acc, slot0, row, others};
              epilogue_normal<Cfg>(args, src, m * 128 + row, n, s, os);
              if (threadIdx.x == 64)
                for (int p = 0; p < others; ++p) flags[p] = 0ull;  // every piece has arrived: clear for a replay
            }
            tc_fence_before();
            __syncwarp();
          }
          if (lane == 0) {
            if (rank != 0) mbar_arrive_cluster(mapa_shared(&tempty[acc], 0));
            else mbar_arrive(&tempty[acc]);
          }
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
          continue;
        }
      }
      if (PAIR || whole) {
        TmemSrc src{t_acc};
        if constexpr (SWAP) epilogue_swap<Cfg>(args, src, m * 128 + row, s);
        else epilogue_normal<Cfg>(args, src, m * 128 + row, n, s, os);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && rank != 0) mbar_arrive_cluster(mapa_shared(&tempty[acc], 0));
          else mbar_arrive(&tempty[acc]);
        }
      } else {
        // a piece of a split tile: park it in this CTA's workspace slot
        const int tile_local = sg.tile - args.dp_tiles;
        const long long f = sk_begin(args, blockIdx.x);
        const int slot = 2 * blockIdx.x + (static_cast<int>(f / args.kpt) == tile_local ? 0 : 1);
        float* slot_ptr = args.partials + static_cast<size_t>(slot) * Cfg::SLOT_FLOATS;
        if constexpr (SWAP) store_partial<16>(t_acc, slot_ptr, row, Cfg::NACC * args.Tpad);
        else store_partial<32>(t_acc, slot_ptr, row, 256);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        // count the pieces; the CTA adding the last one combines them
        const long long i0 = static_cast<long long>(tile_local) * args.kpt;
        const int c_first = sk_cta_of(args, i0);
        const int c_last = sk_cta_of(args, i0 + args.kpt - 1);
        __threadfence();
        epi_bar();
        if (threadIdx.x == 64) {
          *last_flag = arrive_tagged(args.sync_words + tile_local, args.epoch) == c_last - c_first + 1 ? 1 : 0;
        }
        epi_bar();
        if (*last_flag) {
          __threadfence();
          PartialSrc src{args.partials, Cfg::SLOT_FLOATS, c_first, c_last, row, &args, tile_local};
          if constexpr (SWAP) epilogue_swap<Cfg>(args, src, m * 128 + row, s);
          else epilogue_normal<Cfg>(args, src, m * 128 + row, n, s, os);
          if (threadIdx.x == 64) args.sync_words[tile_local] = 0ull;  // all pieces arrived: clear for a replay
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (os.buf && lane == 0) tma_store_wait_all();  // the staged outputs have landed
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    else tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace tpk
