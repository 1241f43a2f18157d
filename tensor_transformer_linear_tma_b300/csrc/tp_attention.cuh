// Attention core of each local head, between the QKV and O projections:
// ctx_h = softmax(q_h k_g^T / sqrt(hd)) v_g for every q head h of a shard,
// g = h / (hq / hkv) its kv head ("CUDA tensor parallel computations" page,
// attention heads; tutorial page, self-attention block sharding), causal
// (query t sees keys 0..t) or unmasked.
//
// Work units are (shard, q head, block of 128 queries), head size 128. The
// kernel is persistent: one CTA per SM (all of TMEM is allocated) walks its
// units, the longest (latest, under the causal mask) first, in alternating
// directions from wave to wave. Within a CTA the ring, the score buffers and
// their barriers run on across units, so the next unit's Q, K and V tiles
// are loaded, and its first scores computed, while the softmax warps write
// the last unit's output. 320 threads:
//   warp 0      TMA producer: the Q tile once, then the K and V tiles of
//               each block of 128 keys through a ring of six 32 KB slots (a
//               K slot is released as soon as Q K^T has read it, a V slot
//               after P V), three key blocks of lookahead;
//   warp 1      TMEM owner and MMA issuer (one elected lane issues):
//               S = Q K^T into one of two TMEM score buffers (one key
//               block ahead of the softmax), then
//               O += P V into the TMEM output accumulator. Q and P are the
//               A operands and sit in TMEM; only K and V are read from
//               shared memory (V as an MN-major operand straight from its
//               TMA tile), which halves the tensor core's shared-memory
//               traffic against staging Q and P there;
//   warps 2..9  softmax, two threads per query row (warps w and w+4 share
//               a TMEM lane quadrant; each takes 64 of the block's 128
//               keys and the matching 64 output columns). They copy each
//               unit's Q from its TMA tile into TMEM, the next unit's as
//               soon as the last scores of the current one are in (every
//               S MMA that read the old Q is then complete), before they
//               write the current unit's output. Per key block: scores from
//               TMEM, online maximum (exchanged between the two halves of a
//               row through shared memory) and sum in fp32, exp2 with the
//               log2(e)/sqrt(hd) scale folded into one FFMA, P packed to
//               bf16 and stored over the first half of its own scores; at
//               the end O / l.
// The exponent base m only moves when a row's maximum exceeds it by more
// than 2^8 (P then stays below 256, exact enough in bf16), so O and l are
// rescaled in TMEM only on such jumps.
// The tensor core runs tcgen05 operations in issue order, so S(j + 2) may be
// issued into the buffer that holds P(j) as soon as P(j) V has been issued.
// P V of block j commits to the barrier of buffer j & 1: a softmax thread
// waits on it only to rescale O or to read the result, and since S(j) was
// issued after P(j - 2) V, each wait's barrier is at most one phase behind.
// Every wait is bounded as in the GEMM kernel.
#pragma once

#include "tp_gemm.cuh"  // epi_any, store_bf16x8_f
#include "tp_ptx.cuh"

namespace tpk {

// 2^x with the MUFU approximation (flushes subnormals; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Barrier over the two softmax warps of TMEM lane quadrant q (named barriers
// 2..5) that ORs a predicate, so that both take the same branch.
__device__ __forceinline__ bool pair_any(int q, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %2, 0;\n\t"
      "bar.red.or.pred po, %1, 64, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}\n"
      : "=r"(r)
      : "r"(2 + q), "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

struct AttnArgs {
  __nv_bfloat16* ctx;  // [tp][T][nq * hd]
  int T, tp, hq, hkv, nq, nkv, group;
  int causal;
  int q_blocks;        // ceil(T / 128)
  int units;           // tp * nq * q_blocks work units; the grid has at most this many CTAs
  float scale_log2;    // log2(e) / sqrt(hd)
};

constexpr int AT_ROWS = 128;                   // queries per CTA, keys per block
constexpr int AT_HD = 128;                     // head size
constexpr int AT_PANEL = AT_ROWS * 128;        // 128 rows x 128 bytes (64 bf16 columns)
constexpr int AT_TILE = 2 * AT_PANEL;          // 128 x 128 bf16 as two 64-column panels
constexpr int AT_THREADS = 320;
constexpr int AT_SOFTMAX_THREADS = 256;
constexpr int AT_SLOTS = 6;                        // K/V ring slots
constexpr int AT_SMEM = (1 + AT_SLOTS) * AT_TILE + 1024 + 2048;  // Q, ring; alignment; barriers, row exchange
constexpr int AT_AUX = 512 + 2048;  // barriers, then the row exchange [2 blocks][2 halves][128] floats
constexpr float AT_RESCALE_LOG2 = 8.0f;            // move the exponent base only on a jump above 2^8
// TMEM columns (512 allocated): two score buffers, O, Q as packed bf16
constexpr uint32_t AT_TM_S = 0, AT_TM_O = 256, AT_TM_Q = 384;

// The w-th unit of CTA c in a grid of g CTAs, or -1 past its last one.
// Units are numbered longest first; wave w covers units w*g .. w*g + g - 1,
// taken in reverse on odd waves, which keeps every CTA's total within a
// unit's length of the mean.
__device__ __forceinline__ int at_unit(int c, int g, int w, int units) {
  const int u = w * g + ((w & 1) ? g - 1 - c : c);
  return u < units ? u : -1;
}

struct AtUnit {
  int qb, s, j;          // query block, shard, q head within the shard
  int qcol, kcol, vcol;  // columns of its q, k and v head in the shard's qkv rows
  int nkb;               // key blocks its queries see
};

__device__ __forceinline__ AtUnit at_decode(const AttnArgs& a, int u) {
  AtUnit w;
  const int heads = a.tp * a.nq;
  w.qb = a.q_blocks - 1 - u / heads;
  const int hh = u % heads;
  w.s = hh / a.nq;
  w.j = hh % a.nq;
  const int kv0 = a.hkv >= a.tp ? w.s * a.nkv : (w.s * a.hkv) / a.tp;
  const int kvi = (w.s * a.nq + w.j) / a.group - kv0;  // the kv head within the shard's block
  w.qcol = w.j * AT_HD;
  w.kcol = (a.nq + kvi) * AT_HD;
  w.vcol = (a.nq + a.nkv + kvi) * AT_HD;
  w.nkb = a.causal ? w.qb + 1 : a.q_blocks;
  return w;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    tp_attn_kernel(const __grid_constant__ CUtensorMap mapQKV, const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* ring = smem + AT_TILE;  // [AT_SLOTS]: K(j) is item 2j, V(j) item 2j+1
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (1 + AT_SLOTS) * AT_TILE);
  uint64_t* q_full = bars;                // TMA -> softmax (a unit's Q tile landed)
  uint64_t* q_tm = bars + 1;              // softmax -> MMA, TMA (that Q copied into TMEM; its tile free)
  uint64_t* o_free = bars + 2;            // softmax -> MMA (a unit's O read out)
  uint64_t* r_full = bars + 3;            // [AT_SLOTS] TMA -> MMA
  uint64_t* r_empty = r_full + AT_SLOTS;  // [AT_SLOTS] MMA -> TMA
  uint64_t* s_full = r_empty + AT_SLOTS;  // [2] MMA -> softmax (S of block gb in buffer gb & 1)
  uint64_t* p_full = s_full + 2;          // [2] softmax -> MMA (P stored, O rescaled)
  uint64_t* o_done = p_full + 2;          // [2] MMA -> softmax (P V of block gb complete, barrier gb & 1)
  uint64_t* drain = o_done + 2;           // abort path only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* xrow = reinterpret_cast<float*>(smem + (1 + AT_SLOTS) * AT_TILE + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the 1024-byte alignment of the tiles must leave room for the barriers
  // and the row exchange (a dynamic shared-memory base is 1024-aligned in
  // practice; otherwise the block reports an error instead of overrunning)
  if ((smem - smem_raw) + (1 + AT_SLOTS) * AT_TILE + AT_AUX > AT_SMEM) {
    if (threadIdx.x == 0) atomicCAS(&g_tp_error, TP_DEVERR_NONE, TP_DEVERR_LAYOUT);
    return;
  }

  const int cta = static_cast<int>(blockIdx.x), grid = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_tm, 8);
    mbar_init(o_free, 8);
    for (int i = 0; i < AT_SLOTS; ++i) {
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&o_done[i], 1);
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
      // Per unit: its Q tile (once the last unit's Q has been copied out of
      // the tile), then its K and V tiles through the ring.
      uint32_t issued = 0, issued_ph = 0;  // per slot: a copy was started, its phase
      int it = 0;                          // ring items of all units so far
      int q_loads = 0;
      bool ok = true;
      for (int w = 0; ok; ++w) {
        const int u = at_unit(cta, grid, w, a.units);
        if (u < 0) break;
        const AtUnit wu = at_decode(a, u);
        if (w > 0 && !mbar_wait(q_tm, static_cast<uint32_t>(w - 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, AT_TILE);
        tma_load_3d(sQ, &mapQKV, q_full, wu.qcol, wu.qb * AT_ROWS, wu.s);
        tma_load_3d(sQ + AT_PANEL, &mapQKV, q_full, wu.qcol + 64, wu.qb * AT_ROWS, wu.s);
        ++q_loads;
        for (int i = 0; i < 2 * wu.nkb; ++i, ++it) {  // K(j), V(j), K(j+1), ...
          const int slot = it % AT_SLOTS;
          const uint32_t ph = static_cast<uint32_t>(it / AT_SLOTS) & 1u;
          if (!mbar_wait(&r_empty[slot], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const int col = (i & 1) ? wu.vcol : wu.kcol;
          uint8_t* dst = ring + slot * AT_TILE;
          mbar_arrive_expect_tx(&r_full[slot], AT_TILE);
          tma_load_3d(dst, &mapQKV, &r_full[slot], col, (i >> 1) * AT_ROWS, wu.s);
          tma_load_3d(dst + AT_PANEL, &mapQKV, &r_full[slot], col + 64, (i >> 1) * AT_ROWS, wu.s);
          issued |= 1u << slot;
          issued_ph = (issued_ph & ~(1u << slot)) | (ph << slot);
        }
      }
      if (!ok) {  // let every copy this block started land before it exits
        if (q_loads > 0) mbar_wait_drain(q_full, static_cast<uint32_t>(q_loads - 1) & 1u);
        for (int i = 0; i < AT_SLOTS; ++i)
          if ((issued >> i) & 1u) mbar_wait_drain(&r_full[i], (issued_ph >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // The whole warp runs the loop (waits and descriptors are warp-uniform);
    // one elected lane issues each MMA and commit.
    const uint32_t idesc_s = idesc_bf16_f32(128, 128);
    const uint32_t idesc_o = idesc_bf16_f32_bmn(128, 128);
    const uint32_t tO = tmem_base + AT_TM_O, tQ = tmem_base + AT_TM_Q;
    const uint64_t ring_k = smem_desc_k_sw128(smem_u32(ring));
    const uint64_t ring_mn = smem_desc_mn_sw128(smem_u32(ring), AT_PANEL, 1024);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    bool ok = true, issued_any = false;
    // Block gb counts the key blocks of all this CTA's units so far: it
    // picks the score buffer (gb & 1) and the phases of its barriers. Ring
    // item `item` holds a K tile (S) or a V tile (P V).
    //
    // S(gb) = Q K^T: M = 128 queries, N = 128 keys, K = hd in 8 steps of 16
    // (Q: 8 TMEM columns a step; K: two 64-wide panels, +32 bytes a step
    // inside a panel; descriptor start addresses count 16-byte units). The
    // caller has waited for the K tile.
    auto issue_s = [&](int gb, int item) {
      const int st = gb & 1;
      const int slot = item % AT_SLOTS;
      const uint64_t kd = ring_k + static_cast<uint64_t>((slot * AT_TILE) >> 4);
      const uint32_t tS = tmem_base + AT_TM_S + static_cast<uint32_t>(st * 128);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        tc_mma_bf16_ts_warp(tS, tQ + static_cast<uint32_t>(k * 8),
                            kd + static_cast<uint64_t>(((k >> 2) * AT_PANEL + (k & 3) * 32) >> 4), idesc_s,
                            k > 0 ? 1u : 0u);
      tc_commit_warp(&s_full[st]);
      tc_commit_warp(&r_empty[slot]);  // K read
      issued_any = true;
    };
    // O (+)= P(gb) V: M = 128 queries, N = hd, K = 128 keys in 8 steps; P
    // sits in TMEM (keys 0..63 at score columns 0..31 of its buffer, keys
    // 64..127 at 64..95), V is MN-major (rows = keys, each row 64 hd values;
    // the second 64 hd values one panel further). A unit's first block
    // overwrites O. The caller has waited for the V tile and P.
    auto issue_pv = [&](int gb, int item, bool first) {
      const int st = gb & 1;
      const int slot = item % AT_SLOTS;
      const uint32_t tP = tmem_base + AT_TM_S + static_cast<uint32_t>(st * 128);
      const uint64_t vd = ring_mn + static_cast<uint64_t>((slot * AT_TILE) >> 4);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        tc_mma_bf16_ts_warp(tO, tP + static_cast<uint32_t>((k >> 2) * 64 + (k & 3) * 8),
                            vd + static_cast<uint64_t>((k * 16 * 128) >> 4), idesc_o, (!first || k > 0) ? 1u : 0u);
      tc_commit_warp(&o_done[st]);
      tc_commit_warp(&r_empty[slot]);  // V read
    };
    auto wait_item = [&](int item) {
      return wait_all(&r_full[item % AT_SLOTS], static_cast<uint32_t>(item / AT_SLOTS) & 1u);
    };
    // Per unit: once its Q is in TMEM, S(0) and S(1) fill both score
    // buffers (right behind the last unit's final P V, which the tensor
    // core runs first); then, per block, P(jb) V and S(jb + 2) are issued
    // back to back as soon as the softmax hands over P(jb): S(jb + 2) reuses
    // P(jb)'s buffer, and the tensor core runs them in issue order. The
    // ring waits come before the wait for P, off the path from the softmax
    // to the tensor core. The unit's first P V also waits until the softmax
    // has read the last unit's O out of TMEM.
    int it0 = 0, g0 = 0;  // ring items and key blocks of the earlier units
    for (int w = 0; ok; ++w) {
      const int u = at_unit(cta, grid, w, a.units);
      if (u < 0) break;
      const int nkb = at_decode(a, u).nkb;
      ok = wait_all(q_tm, static_cast<uint32_t>(w) & 1u);
      for (int jb = 0; ok && jb < 2 && jb < nkb; ++jb) {
        ok = wait_item(it0 + 2 * jb);
        if (ok) {
          tc_fence_after();
          issue_s(g0 + jb, it0 + 2 * jb);
        }
      }
      for (int jb = 0; ok && jb < nkb; ++jb) {
        const bool next = jb + 2 < nkb;
        const int gb = g0 + jb;
        ok = wait_item(it0 + 2 * jb + 1) && (!next || wait_item(it0 + 2 * jb + 4)) &&
             wait_all(&p_full[gb & 1], static_cast<uint32_t>(gb >> 1) & 1u) &&
             (jb > 0 || w == 0 || wait_all(o_free, static_cast<uint32_t>(w - 1) & 1u));
        if (!ok) break;
        tc_fence_after();
        issue_pv(gb, it0 + 2 * jb + 1, jb == 0);
        if (next) issue_s(gb + 2, it0 + 2 * jb + 4);
      }
      it0 += 2 * nkb;
      g0 += nkb;
    }
    if (!ok && issued_any) {  // wait for MMAs in flight before TMEM is freed
      tc_commit_warp(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------ softmax ------------------------------
    const int q = warp & 3;            // TMEM lane quadrant
    const int half = (warp - 2) >> 2;  // which 64 keys / output columns of the row
    const int r = q * 32 + lane;       // query row within the block
    const int c0 = half * 64;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t tO = tmem_base + AT_TM_O + lane_off + static_cast<uint32_t>(c0);
    // Q of unit w into TMEM: this thread's row, hd values 64 * half .. + 63,
    // read from the 128-byte-swizzled TMA tile. Returns false (for both
    // warps of the quadrant) if the wait gave up.
    auto copy_q = [&](int w) -> bool {
      const bool q_ok = mbar_wait(q_full, static_cast<uint32_t>(w) & 1u, abort_flag);
      if (pair_any(q, !q_ok || *abort_flag)) return false;
      const uint8_t* qrow = sQ + half * AT_PANEL + r * 128;
      uint32_t rr[32];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + ((ch ^ (r & 7)) << 4));
        rr[ch * 4 + 0] = v.x;
        rr[ch * 4 + 1] = v.y;
        rr[ch * 4 + 2] = v.z;
        rr[ch * 4 + 3] = v.w;
      }
      tmem_st32(tmem_base + AT_TM_Q + lane_off + static_cast<uint32_t>(half * 32), rr);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_tm);
      return true;
    };
    // (the grid has no more CTAs than units, so every CTA has a first one)
    bool ok = copy_q(0);
    int g0 = 0;  // key blocks of the earlier units
    for (int w = 0; ok; ++w) {
      const int u = at_unit(cta, grid, w, a.units);
      if (u < 0) break;
      const AtUnit wu = at_decode(a, u);
      const int nkb = wu.nkb, qb = wu.qb;
      const int t = qb * AT_ROWS + r;                         // query index
      const int kmax = a.causal ? min(t, a.T - 1) : a.T - 1;  // last key this query sees
      float m = -INFINITY;  // exponent base, in log2 units of the scaled scores
      float l = 0.0f;       // this half's share of the row sum
      for (int jb = 0; ok && jb < nkb; ++jb) {
        const int gb = g0 + jb;  // block count over this CTA's units: buffer and phases
        const int st = gb & 1;
        const uint32_t ph = static_cast<uint32_t>(gb >> 1) & 1u;
        // (a wait that gave up leaves garbage in the scores, which the vote at
        // the exchange below discards)
        const bool waited = mbar_wait(&s_full[st], ph, abort_flag);
        tc_fence_after();
        float sv[64];
        const uint32_t tS = tmem_base + AT_TM_S + static_cast<uint32_t>(st * 128 + c0) + lane_off;
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t rr[32];
          tmem_ld32(tS + static_cast<uint32_t>(c), rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[c + i] = __uint_as_float(rr[i]);
        }
        tmem_ld_wait();
        const int kbase = jb * AT_ROWS + c0;
        // only the diagonal block (causal) and a ragged last block need a mask
        if ((a.causal && jb == qb) || jb * AT_ROWS + AT_ROWS > a.T) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (kbase + i > kmax) sv[i] = -INFINITY;
        }
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = sv[i];
#pragma unroll
        for (int i = 8; i < 64; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], sv[i]);
        float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                         fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        // the row's other half: exchange the maxima, in one of two slots by
        // block parity (the partner's write two blocks on comes after the next
        // exchange, which this thread reaches only after this read); the
        // barrier also takes both halves out together if a wait gave up
        float* xr = xrow + st * 256;
        xr[half * 128 + r] = mx;
        if (pair_any(q, !waited || *abort_flag)) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, xr[(half ^ 1) * 128 + r]);
        const float m_cand = mx * a.scale_log2;  // the scale is positive: same order
        bool rescale = false;
        float alpha = 1.0f;
        if (m_cand > m + AT_RESCALE_LOG2) {  // also the first visible block (m = -inf)
          alpha = ex2_approx(m - m_cand);    // 0 on the first block
          rescale = jb > 0;
          m = m_cand;
          l *= alpha;
        }
        float sum8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) sum8[i] = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          sv[i] = ex2_approx(fmaf(sv[i], a.scale_log2, -m));
          sum8[i & 7] += sv[i];
        }
        l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        if (__any_sync(0xffffffffu, rescale)) {
          // the base moved: once P V of block jb - 1 is done, this half's 64
          // columns of O are rescaled. A wait that gives up (the abort flag is
          // then set) skips the rescale; the next exchange takes both halves
          // of the row out of the loop together.
          const bool done = mbar_wait(&o_done[st ^ 1], static_cast<uint32_t>((gb - 1) >> 1) & 1u, abort_flag);
          if (__all_sync(0xffffffffu, done)) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 64; c += 32) {
              uint32_t rr[32];
              tmem_ld32(tO + static_cast<uint32_t>(c), rr);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
              tmem_st32(tO + static_cast<uint32_t>(c), rr);
            }
          }
        }
        // this half's 64 P values as bf16 pairs over its first 32 score columns
        // (already read into registers)
        {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(sv[2 * i], sv[2 * i + 1]);
          tmem_st32(tS, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[st]);
      }
      // ok is uniform over the two warps of a quadrant
      const int gl = g0 + nkb - 1;  // the unit's last block
      g0 += nkb;
      if (!ok) break;
      // The next unit's Q into TMEM now: every S MMA of this unit is complete
      // (its last scores are in), so the next unit's first scores are computed
      // while this unit's output is written.
      if (at_unit(cta, grid, w + 1, a.units) >= 0 && !copy_q(w + 1)) {
        ok = false;
        break;
      }
      // (S(gl) was issued after P V of block gl - 2, so the barrier of block
      // gl is at most one phase behind: its parity is unambiguous)
      const bool done = mbar_wait(&o_done[gl & 1], static_cast<uint32_t>(gl >> 1) & 1u, abort_flag);
      // The row sum is the two halves' shares (same exponent base), exchanged
      // in the slot that the next block's maxima use; the second barrier keeps
      // those out until both halves have read.
      float* xr = xrow + ((gl + 1) & 1) * 256;
      xr[half * 128 + r] = l;
      if (pair_any(q, !done || *abort_flag)) {
        ok = false;
        break;
      }
      l += xr[(half ^ 1) * 128 + r];
      pair_any(q, false);
      tc_fence_after();
      const float inv = 1.0f / l;
      const int nc = a.nq * AT_HD;
      __nv_bfloat16* out = a.ctx + (static_cast<size_t>(wu.s) * a.T + t) * nc + wu.j * AT_HD + c0;
#pragma unroll 1
      for (int c = 0; c < 64; c += 32) {
        uint32_t rr[32];
        tmem_ld32(tO + static_cast<uint32_t>(c), rr);
        tmem_ld_wait();
        if (t < a.T) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(rr[i + e]) * inv;
            store_bf16x8_f(out + c + i, v);
          }
        }
      }
      // O is read out (each load waited for): the next unit's first P V may
      // overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace tpk
