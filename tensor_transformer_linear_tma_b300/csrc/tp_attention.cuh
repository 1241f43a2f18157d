// Attention core of each local head, between the QKV and O projections:
// ctx_h = softmax(q_h k_g^T / sqrt(hd)) v_g for every q head h of a shard,
// g = h / (hq / hkv) its kv head ("CUDA tensor parallel computations" page,
// attention heads; tutorial page, self-attention block sharding), causal
// (query t sees keys 0..t) or unmasked. Head size 64 or 128 (template HD).
//
// A work unit is two query tiles of 128 rows that read the same keys and
// values: two q heads of one kv head over one block of queries (when the
// heads of a shard pair up that way), else two consecutive query blocks of
// one head. The tiles share every K and V tile the ring brings in, and the
// tensor core alternates between them: while the softmax of one tile runs,
// it computes the other tile's P V and next scores, so the exponentials
// and the MMAs overlap.
//
// The kernel is persistent: one CTA per SM (all of TMEM is allocated)
// walks its units, the longest (latest, under the causal mask) first, in
// alternating directions from wave to wave. 320 threads:
//   warp 0      TMA producer: each unit's two Q tiles (tile t once the last
//               unit's scores of tile t are computed), then the K and V
//               tiles of each block of 128 keys through a ring, K(j), V(j),
//               K(j+1), ... (the ring runs on across units);
//   warp 1      TMEM owner and MMA issuer (all lanes run the loop, one
//               elected lane issues): S_t = Q_t K^T with both operands in
//               shared memory, into tile t's score buffer, and
//               O_t += P_t V with P_t in TMEM (over the first half of its
//               scores) and V an MN-major operand straight from its TMA
//               tile. Per key block the order is P_0 V, S_0(next),
//               P_1 V, S_1(next), each P_t V in two halves of 64 keys:
//               the first as soon as the softmax has stored P_t for them;
//   warps 2..5  softmax of tile 0, warps 6..9 of tile 1, one thread per
//               query row: the row's 128 scores from TMEM, exp2 with the
//               log2(e)/sqrt(hd) scale and the base folded into one paired
//               FMA, the row sum, P packed to bf16 and stored over the
//               scores, handed over a half at a time (the first half's P V
//               runs while the second half's exponentials are computed);
//               at the end of a unit O / l to the context.
// The exponent base m is any value that keeps P from overflowing: the
// softmax is the same for every m, and P's bf16 rounding is relative at any
// magnitude. It is set to the row maximum of a unit's first 64 keys; after
// that no maximum is taken: each half-block's P is computed with the current
// m, and only when the half's row sum exceeds 2^16 (some P above 2^16, or
// an overflow) is its maximum taken, m moved there, the half's P computed
// again and O and l rescaled. S_t(j) is issued after P_t(j-1) V, and a
// commit arrives once every earlier MMA of the issuer is complete, so the
// scores of block j reaching the softmax mean that O_t holds blocks
// 0..j-1 and no MMA writes it: a move in a block's first half needs no
// other wait. A move in its second half waits until the first half's P V
// is complete, then rescales O_t, which holds that half too.
// The tensor core runs tcgen05 operations in issue order, so S_t(j+1) may be
// issued into the buffer that holds P_t(j) right after P_t(j) V.
// Every wait is bounded as in the GEMM kernel.
#pragma once

#include "tp_gemm.cuh"  // store_bf16x8_f
#include "tp_ptx.cuh"

namespace tpk {

// Two fp32 values in one 64-bit register pair (the first in the low half),
// for the paired fp32 instructions: one instruction, two results.
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c). (Written with two fmaxf: the three-input max.f32 of inline
// PTX returned about 0 for all-negative inputs on this toolchain, so it is
// not used.)
__device__ __forceinline__ float fmax3(float a, float b, float c) { return fmaxf(fmaxf(a, b), c); }

struct AttnArgs {
  __nv_bfloat16* ctx;  // [tp][T][nq * hd]
  int T, tp, hq, hkv, nq, nkv, group;
  int causal;
  int q_blocks;        // ceil(T / 128)
  int pair_heads;      // 1: a unit's tiles are q heads 2i, 2i+1 (one kv head) over one query block;
                       // 0: query blocks 2i, 2i+1 of one head
  int units;           // work units; the grid has at most this many CTAs
  float scale_log2;    // log2(e) / sqrt(hd)
};

template <int HD>
struct AttnCfg {
  static_assert(HD == 64 || HD == 128, "head size 64 or 128");
  static constexpr int ROWS = 128;                  // queries per tile, keys per block
  static constexpr int PANEL = ROWS * 128;          // 128 rows x 128 bytes (64 bf16 columns)
  static constexpr int PANELS = HD / 64;
  static constexpr int TILE = PANELS * PANEL;       // 128 x HD bf16
  static constexpr int SLOTS = HD == 128 ? 4 : 8;   // K/V ring
  static constexpr int STAGE = 8 * 4096;            // output staging: 4 KB per softmax warp
  static constexpr int THREADS = 320;
  static constexpr int AUX = 512;                   // barriers, TMEM address, abort flag
  static constexpr int SMEM = (2 + SLOTS) * TILE + STAGE + AUX + 1024;  // Q tiles, ring, staging, aux; alignment
  static constexpr uint32_t TM_S = 0;               // scores / P of tile t at column 128 t
  static constexpr uint32_t TM_O = 256;             // O of tile t at 256 + HD t
};
constexpr float AT_SUM_LIMIT = 65536.0f;  // a half-block's row sum of P above this moves the base

// The w-th unit of CTA c in a grid of g CTAs, or -1 past its last one.
// Units are numbered longest first; wave w covers units w*g .. w*g + g - 1,
// taken in reverse on odd waves, which keeps every CTA's total within a
// unit's length of the mean.
__device__ __forceinline__ int at_unit(int c, int g, int w, int units) {
  const int u = w * g + ((w & 1) ? g - 1 - c : c);
  return u < units ? u : -1;
}

struct AtUnit {
  int s;                     // shard
  int qb[2], j[2];           // per tile: query block, q head within the shard
  int nkb[2];                // key blocks the tile's queries see (0: no such tile)
  int nkb_max;
  int kcol, vcol;            // columns of the shared kv head in the shard's qkv rows
};

__device__ __forceinline__ AtUnit at_decode(const AttnArgs& a, int u, int hd) {
  AtUnit w;
  if (a.pair_heads) {
    const int half = a.nq >> 1;
    const int hp = a.tp * half;
    const int qb = a.q_blocks - 1 - u / hp;
    const int hh = u % hp;
    w.s = hh / half;
    w.j[0] = 2 * (hh % half);
    w.j[1] = w.j[0] + 1;
    w.qb[0] = w.qb[1] = qb;
  } else {
    const int heads = a.tp * a.nq;
    const int qp = (a.q_blocks + 1) / 2 - 1 - u / heads;
    const int hh = u % heads;
    w.s = hh / a.nq;
    w.j[0] = w.j[1] = hh % a.nq;
    w.qb[0] = 2 * qp;
    w.qb[1] = 2 * qp + 1;
  }
  const int kv0 = a.hkv >= a.tp ? w.s * a.nkv : (w.s * a.hkv) / a.tp;
  const int kvi = (w.s * a.nq + w.j[0]) / a.group - kv0;  // the kv head within the shard's block
  w.kcol = (a.nq + kvi) * hd;
  w.vcol = (a.nq + a.nkv + kvi) * hd;
#pragma unroll
  for (int t = 0; t < 2; ++t) w.nkb[t] = w.qb[t] >= a.q_blocks ? 0 : (a.causal ? w.qb[t] + 1 : a.q_blocks);
  w.nkb_max = max(w.nkb[0], w.nkb[1]);
  return w;
}

// A moved exponent base (rare): this warp's rows of O_t are multiplied by
// alpha (1 for rows whose base stayed). The caller has made sure that no MMA
// writes O_t meanwhile. Kept out of line: its registers are paid for only
// when it runs.
template <int HD>
__device__ __noinline__ void at_rescale(uint32_t tO, float alpha) {
#pragma unroll 1
  for (int c = 0; c < HD; c += 32) {
    uint32_t rr[32];
    tmem_ld32(tO + static_cast<uint32_t>(c), rr);
    tmem_ld_wait_regs(rr);
#pragma unroll
    for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
    tmem_st32(tO + static_cast<uint32_t>(c), rr);
  }
}

template <int HD>
__global__ void __launch_bounds__(320, 1)
    tp_attn_kernel(const __grid_constant__ CUtensorMap mapQKV, const __grid_constant__ CUtensorMap mapCtx,
                   const AttnArgs a) {
  using Cfg = AttnCfg<HD>;
  constexpr int SLOTS = Cfg::SLOTS, TILE = Cfg::TILE, PANEL = Cfg::PANEL;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                // [2] Q tiles
  uint8_t* ring = smem + 2 * TILE;   // [SLOTS]: K(j) is item 2j, V(j) item 2j+1
  uint8_t* stage = ring + SLOTS * TILE;  // [8] a softmax warp's output staging buffer
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + Cfg::STAGE);
  uint64_t* q_full = bars;                // [2] TMA -> MMA (a unit's Q tile t landed)
  uint64_t* q_free = bars + 2;            // [2] MMA -> TMA (the unit's last S_t is computed: Q_t tile free)
  uint64_t* r_full = bars + 4;            // [SLOTS] TMA -> MMA
  uint64_t* r_empty = r_full + SLOTS;     // [SLOTS] MMA -> TMA
  uint64_t* s_full = r_empty + SLOTS;     // [2] MMA -> softmax t (scores of tile t)
  uint64_t* p_full = s_full + 2;          // [2] softmax t -> MMA (all of P_t stored)
  uint64_t* o_done = p_full + 2;          // [2] MMA -> softmax t (the unit's last P_t V complete)
  uint64_t* o_free = o_done + 2;          // [2] softmax t -> MMA (O_t read out)
  uint64_t* drain = o_free + 2;           // abort path only
  uint64_t* p_half = drain + 1;           // [2] softmax t -> MMA (P_t of keys 0..63 stored, O_t rescaled)
  uint64_t* o_half = p_half + 2;          // [2] MMA -> softmax t (P_t V of keys 0..63 complete)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_half + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the 1024-byte alignment of the tiles must leave room for the barriers (a
  // dynamic shared-memory base is 1024-aligned in practice; otherwise the
  // block reports an error instead of overrunning)
  if ((smem - smem_raw) + (2 + SLOTS) * TILE + Cfg::STAGE + Cfg::AUX > Cfg::SMEM) {
    if (threadIdx.x == 0) atomicCAS(&g_tp_error, TP_DEVERR_NONE, TP_DEVERR_LAYOUT);
    return;
  }

  const int cta = static_cast<int>(blockIdx.x), grid = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_free[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&p_half[t], 4);
      mbar_init(&o_half[t], 1);
      mbar_init(&o_done[t], 1);
      mbar_init(&o_free[t], 4);
    }
    for (int i = 0; i < SLOTS; ++i) {
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mapQKV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer ------------------------------
      uint32_t issued = 0, issued_ph = 0;  // per ring slot: a copy was started, its phase
      int it = 0;                          // ring items of all units so far
      int ua[2] = {0, 0};                  // units that had a tile t so far (= Q_t loads)
      bool ok = true;
      for (int w = 0; ok; ++w) {
        const int u = at_unit(cta, grid, w, a.units);
        if (u < 0) break;
        const AtUnit wu = at_decode(a, u, HD);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || wu.nkb[t] == 0) continue;
          if (ua[t] > 0 && !mbar_wait(&q_free[t], static_cast<uint32_t>(ua[t] - 1) & 1u, abort_flag)) {
            ok = false;
            continue;
          }
          mbar_arrive_expect_tx(&q_full[t], TILE);
#pragma unroll
          for (int p = 0; p < Cfg::PANELS; ++p)
            tma_load_3d(sQ + t * TILE + p * PANEL, &mapQKV, &q_full[t], wu.j[t] * HD + 64 * p, wu.qb[t] * 128, wu.s);
          ++ua[t];
        }
        for (int i = 0; ok && i < 2 * wu.nkb_max; ++i, ++it) {  // K(j), V(j), K(j+1), ...
          const int slot = it % SLOTS;
          const uint32_t ph = static_cast<uint32_t>(it / SLOTS) & 1u;
          if (!mbar_wait(&r_empty[slot], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const int col = (i & 1) ? wu.vcol : wu.kcol;
          uint8_t* dst = ring + slot * TILE;
          mbar_arrive_expect_tx(&r_full[slot], TILE);
#pragma unroll
          for (int p = 0; p < Cfg::PANELS; ++p)
            tma_load_3d(dst + p * PANEL, &mapQKV, &r_full[slot], col + 64 * p, (i >> 1) * 128, wu.s);
          issued |= 1u << slot;
          issued_ph = (issued_ph & ~(1u << slot)) | (ph << slot);
        }
      }
      if (!ok) {  // let every copy this block started land before it exits
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (ua[t] > 0) mbar_wait_drain(&q_full[t], static_cast<uint32_t>(ua[t] - 1) & 1u);
        for (int i = 0; i < SLOTS; ++i)
          if ((issued >> i) & 1u) mbar_wait_drain(&r_full[i], (issued_ph >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    const uint32_t idesc_s = idesc_bf16_f32(128, 128);
    const uint32_t idesc_o = idesc_bf16_f32_bmn(128, HD);
    const uint64_t q_desc = smem_desc_k_sw128(smem_u32(sQ));
    const uint64_t ring_k = smem_desc_k_sw128(smem_u32(ring));
    const uint64_t ring_mn = smem_desc_mn_sw128(smem_u32(ring), PANEL, 1024);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    auto wait_item = [&](int item) {
      return wait_all(&r_full[item % SLOTS], static_cast<uint32_t>(item / SLOTS) & 1u);
    };
    bool ok = true, issued_any = false;
    // S_t = Q_t K^T: M = 128 queries, N = 128 keys, K = HD in steps of 16
    // (both operands K-major in 64-wide panels: +32 bytes a step inside a
    // panel; descriptor start addresses count 16-byte units). The caller has
    // waited for Q_t and the K tile.
    auto issue_s = [&](int t, int item) {
      const uint64_t qd = q_desc + static_cast<uint64_t>((t * TILE) >> 4);
      const uint64_t kd = ring_k + static_cast<uint64_t>(((item % SLOTS) * TILE) >> 4);
      const uint32_t tS = tmem_base + Cfg::TM_S + static_cast<uint32_t>(t * 128);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint64_t off = static_cast<uint64_t>(((k >> 2) * PANEL + (k & 3) * 32) >> 4);
        tc_mma_bf16_warp(tS, qd + off, kd + off, idesc_s, k > 0 ? 1u : 0u);
      }
      issued_any = true;
    };
    // O_t (+)= P_t V over keys 64 h .. 64 h + 63: M = 128 queries, N = HD,
    // K = 64 keys in 4 steps; P_t sits in TMEM (key pairs at the first 64
    // columns of tile t's scores), V is MN-major (rows = keys, 64 hd values a
    // row, the next 64 hd values one panel further). A unit's first block
    // overwrites O_t. The caller has waited for the V tile and that half of
    // P_t.
    auto issue_pv = [&](int t, int item, bool first, int h) {
      const uint32_t tP = tmem_base + Cfg::TM_S + static_cast<uint32_t>(t * 128);
      const uint32_t tO = tmem_base + Cfg::TM_O + static_cast<uint32_t>(t * HD);
      const uint64_t vd = ring_mn + static_cast<uint64_t>(((item % SLOTS) * TILE) >> 4);
#pragma unroll
      for (int k = 4 * h; k < 4 * h + 4; ++k)
        tc_mma_bf16_ts_warp(tO, tP + static_cast<uint32_t>(k * 8), vd + static_cast<uint64_t>((k * 16 * 128) >> 4),
                            idesc_o, (!first || k > 0) ? 1u : 0u);
      issued_any = true;
    };
    int it0 = 0;                          // ring items of the earlier units
    int ua[2] = {0, 0}, pg[2] = {0, 0};   // units with tile t, P_t blocks consumed
    for (int w = 0; ok; ++w) {
      const int u = at_unit(cta, grid, w, a.units);
      if (u < 0) break;
      const AtUnit wu = at_decode(a, u, HD);
      // first scores of each tile (right behind the last unit's final P V)
      ok = wait_item(it0);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok || wu.nkb[t] == 0) continue;
        ok = wait_all(&q_full[t], static_cast<uint32_t>(ua[t]) & 1u);
        if (!ok) continue;
        tc_fence_after();
        issue_s(t, it0);
        tc_commit_warp(&s_full[t]);
        if (wu.nkb[t] == 1) tc_commit_warp(&q_free[t]);
      }
      if (!ok) break;
      tc_commit_warp(&r_empty[it0 % SLOTS]);  // K(0) read
      // per key block: P_0 V, S_0(next), P_1 V, S_1(next). The ring waits
      // come before the waits for P, off the path from the softmax to the
      // tensor core; a unit's first P_t V also waits until the softmax has
      // read the last unit's O_t out of TMEM.
      for (int jb = 0; ok && jb < wu.nkb_max; ++jb) {
        const bool next = jb + 1 < wu.nkb_max;
        const int iv = it0 + 2 * jb + 1, ik = iv + 1;
        ok = wait_item(iv) && (!next || wait_item(ik));
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || jb >= wu.nkb[t]) continue;
          ok = wait_all(&p_half[t], static_cast<uint32_t>(pg[t]) & 1u) &&
               (jb > 0 || ua[t] == 0 || wait_all(&o_free[t], static_cast<uint32_t>(ua[t] - 1) & 1u));
          if (!ok) continue;
          tc_fence_after();
          issue_pv(t, iv, jb == 0, 0);
          tc_commit_warp(&o_half[t]);
          ok = wait_all(&p_full[t], static_cast<uint32_t>(pg[t]) & 1u);
          if (!ok) continue;
          ++pg[t];
          tc_fence_after();
          issue_pv(t, iv, jb == 0, 1);
          if (jb + 1 < wu.nkb[t]) {
            issue_s(t, ik);
            tc_commit_warp(&s_full[t]);
            if (jb + 2 == wu.nkb[t]) tc_commit_warp(&q_free[t]);  // that was the unit's last S_t
          } else {
            tc_commit_warp(&o_done[t]);
          }
        }
        if (!ok) break;
        tc_commit_warp(&r_empty[iv % SLOTS]);          // V(jb) read
        if (next) tc_commit_warp(&r_empty[ik % SLOTS]);  // K(jb + 1) read
      }
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (wu.nkb[t] > 0) ++ua[t];
      it0 += 2 * wu.nkb_max;
    }
    if (!ok && issued_any) {  // wait for MMAs in flight before TMEM is freed
      tc_commit_warp(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------ softmax ------------------------------
    const int t = (warp - 2) >> 2;     // query tile
    const int q = warp & 3;            // TMEM lane quadrant
    const int r = q * 32 + lane;       // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t tS = tmem_base + Cfg::TM_S + static_cast<uint32_t>(t * 128) + lane_off;
    const uint32_t tO = tmem_base + Cfg::TM_O + static_cast<uint32_t>(t * HD) + lane_off;
    const uint64_t scale2 = f2_make(a.scale_log2, a.scale_log2);
    bool ok = true;
    int ua = 0, sg = 0;  // units with this tile, score blocks consumed
    for (int w = 0; ok; ++w) {
      const int u = at_unit(cta, grid, w, a.units);
      if (u < 0) break;
      const AtUnit wu = at_decode(a, u, HD);
      const int nkb = t ? wu.nkb[1] : wu.nkb[0];
      if (nkb == 0) continue;
      const int qb = t ? wu.qb[1] : wu.qb[0];
      const int jq = t ? wu.j[1] : wu.j[0];
      const int tq = qb * 128 + r;                             // query index
      const int kmax = a.causal ? min(tq, a.T - 1) : a.T - 1;  // last key this query sees
      float m = -INFINITY;  // exponent base, in log2 units of the scaled scores
      float l = 0.0f;       // row sum of the exponentials
      for (int jb = 0; jb < nkb; ++jb, ++sg) {
        const bool waited = mbar_wait(&s_full[t], static_cast<uint32_t>(sg) & 1u, abort_flag);
        if (__any_sync(0xffffffffu, !waited)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // The block's 128 keys in two halves of 64, each a step of the online
        // softmax: its scores from TMEM, its maximum, a move of the base if
        // needed, its exponentials packed to bf16 over the score columns the
        // first half has already consumed (P keys 0..63 at columns 0..31,
        // keys 64..127 at 32..63), then the half handed to the MMA. A base
        // that moves in the second half (rarely: only when the half's P sum
        // exceeds 2^16) rescales O, once the first half's P V has been added
        // to it, and l.
        const bool masked = (a.causal && jb == qb) || jb * 128 + 128 > a.T;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float sv[64];
          {
            uint32_t ra[32], rb[32];
            tmem_ld32(tS + static_cast<uint32_t>(h * 64), ra);
            tmem_ld32(tS + static_cast<uint32_t>(h * 64 + 32), rb);
            tmem_ld_wait_regs(ra);
            reg_fence32(rb);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              sv[i] = __uint_as_float(ra[i]);
              sv[32 + i] = __uint_as_float(rb[i]);
            }
          }
          // only the diagonal block (causal) and a ragged last block need a mask
          if (masked) {
            const int kb = jb * 128 + h * 64;
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (kb + i > kmax) sv[i] = -INFINITY;
          }
          // the half's maximum of the scaled scores (-inf if no key is visible)
          auto half_max = [&]() -> float {
            float mx4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) mx4[i] = sv[i];
#pragma unroll
            for (int i = 4; i < 64; i += 8) {
              mx4[0] = fmax3(mx4[0], sv[i], sv[i + 1]);
              mx4[1] = fmax3(mx4[1], sv[i + 2], sv[i + 3]);
              mx4[2] = fmax3(mx4[2], sv[i + 4], sv[i + 5]);
              mx4[3] = fmax3(mx4[3], sv[i + 6], sv[i + 7]);
            }
            return fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]) * a.scale_log2;  // (the scale is positive)
          };
          // P = 2^(s * scale - m), two at a time, packed; the half's row sum
          uint32_t pk[32];
          auto half_exp = [&]() -> float {
            const uint64_t negm = f2_make(-m, -m);
            uint64_t acc[2] = {f2_make(0.0f, 0.0f), f2_make(0.0f, 0.0f)};
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float x0, x1;
              f2_split(f2_fma(f2_make(sv[2 * i], sv[2 * i + 1]), scale2, negm), x0, x1);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              acc[i & 1] = f2_add(acc[i & 1], f2_make(p0, p1));
              pk[i] = pack_bf16x2(p0, p1);
            }
            float s0, s1, s2, s3;
            f2_split(acc[0], s0, s1);
            f2_split(acc[1], s2, s3);
            return (s0 + s1) + (s2 + s3);
          };
          const bool unit_first = jb == 0 && h == 0;
          if (unit_first) {  // key 0 is visible to every row, so the maximum is finite
            const float mx = half_max();
            m = mx > -INFINITY ? mx : 0.0f;
          }
          float lh = half_exp();
          if (!unit_first) {
            const bool big = !(lh <= AT_SUM_LIMIT);  // (also an overflow to inf)
            if (__any_sync(0xffffffffu, big)) {
              // rare: move the base to the half's maximum (above m: some P
              // exceeded 1), recompute the half, rescale O and l (rows whose
              // base stayed use alpha = 1). O holds the blocks before this one
              // (and, in the second half, the first half's P V once done).
              float alpha = 1.0f;
              if (big) {
                const float mx = half_max();
                alpha = ex2_approx(m - mx);
                m = mx;
                l *= alpha;
                lh = half_exp();
              }
              const bool go = h == 0 || __all_sync(0xffffffffu, mbar_wait(&o_half[t], static_cast<uint32_t>(sg) & 1u,
                                                                           abort_flag));
              if (go) {
                tc_fence_after();
                at_rescale<HD>(tO, alpha);
              }
            }
          }
          tmem_st32(tS + static_cast<uint32_t>(h * 32), pk);
          l += lh;
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(h == 0 ? &p_half[t] : &p_full[t]);
        }
      }
      if (!ok) break;
      const bool done = mbar_wait(&o_done[t], static_cast<uint32_t>(ua) & 1u, abort_flag);
      if (__any_sync(0xffffffffu, !done)) {
        ok = false;
        break;
      }
      ++ua;
      tc_fence_after();
      const float inv = 1.0f / l;
      // 64 columns at a time: the warp's 32 rows of O / l as bf16 into its
      // staging buffer (128-byte-swizzled rows), then one bulk tensor store of
      // the 32 x 64 box (rows past the sequence are clipped by the copy
      // engine; a box wholly past it is not issued)
      const int row0 = qb * 128 + q * 32;
      uint8_t* sb = stage + (warp - 2) * 4096;
#pragma unroll 1
      for (int c = 0; c < HD; c += 64) {
        if (lane == 0) tma_store_wait_read<0>();  // the buffer's last store has read it
        __syncwarp();
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t rr[32];
          tmem_ld32(tO + static_cast<uint32_t>(c + 32 * hh), rr);
          tmem_ld_wait_regs(rr);
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(rr[i + e]) * inv;
            stage_put(sb, lane, 4 * hh + (i >> 3), pack_bf16x8(v));
          }
        }
        stage_ready();
        if (lane == 0 && row0 < a.T) {
          tma_store_3d(&mapCtx, sb, jq * HD + c, row0, wu.s);
          tma_store_commit();
        }
      }
      // O_t is read out (each load waited for): the next unit's first P_t V
      // may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[t]);
    }
    if (lane == 0) tma_store_wait_all();  // the context is written before the block exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace tpk
