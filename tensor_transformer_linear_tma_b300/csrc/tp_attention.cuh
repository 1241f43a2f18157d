// Attention core of each local head, between the QKV and O projections:
// ctx_h = softmax(q_h k_g^T / sqrt(hd)) v_g for every q head h of a shard,
// g = h / (hq / hkv) its kv head ("CUDA tensor parallel computations" page,
// attention heads; tutorial page, self-attention block sharding), causal
// (query t sees keys 0..t) or unmasked.
//
// One CTA per (shard, q head, block of 128 queries), head size 128, 192
// threads:
//   warp 0      TMA producer: the Q tile once, then the K and V tiles of
//               each block of 128 keys through a ring of five 32 KB slots (a
//               K slot is released as soon as Q K^T has read it, a V slot
//               after P V), 2.5 key blocks of lookahead;
//   warp 1      TMEM owner and MMA issuer: S = Q K^T into one of two TMEM
//               score buffers (one key block ahead of the softmax), then
//               O += P V into the TMEM output accumulator, with V read as an
//               MN-major operand straight from its TMA tile;
//   warps 2..5  softmax, one query row per thread: scores from TMEM, online
//               maximum and sum in fp32 (exp2 with the log2(e)/sqrt(hd)
//               scale folded into one FFMA), P written as bf16 into a
//               128-byte-swizzled shared-memory tile (the next MMA's A
//               operand) once P V of the previous block has read it; at the
//               end O / l is stored.
// The exponent base m only moves when a row's maximum exceeds it by more
// than 2^8 (P then stays below 256, exact enough in bf16), so O and l are
// rescaled in TMEM only on such jumps.
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

struct AttnArgs {
  __nv_bfloat16* ctx;  // [tp][T][nq * hd]
  int T, tp, hq, hkv, nq, nkv, group;
  int causal;
  int q_blocks;        // ceil(T / 128)
  float scale_log2;    // log2(e) / sqrt(hd)
};

constexpr int AT_ROWS = 128;                   // queries per CTA, keys per block
constexpr int AT_HD = 128;                     // head size
constexpr int AT_PANEL = AT_ROWS * 128;        // 128 rows x 128 bytes (64 bf16 columns)
constexpr int AT_TILE = 2 * AT_PANEL;          // 128 x 128 bf16 as two 64-column panels
constexpr int AT_THREADS = 192;
constexpr int AT_SLOTS = 5;                        // K/V ring slots
constexpr int AT_SMEM = (2 + AT_SLOTS) * AT_TILE + 1024 + 512;  // Q, P, ring; alignment; barriers
constexpr float AT_RESCALE_LOG2 = 8.0f;            // move the exponent base only on a jump above 2^8

__global__ void __launch_bounds__(AT_THREADS, 1)
    tp_attn_kernel(const __grid_constant__ CUtensorMap mapQKV, const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sP = smem + AT_TILE;
  uint8_t* ring = smem + 2 * AT_TILE;  // [AT_SLOTS]: K(j) is item 2j, V(j) item 2j+1
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (2 + AT_SLOTS) * AT_TILE);
  uint64_t* q_full = bars;              // TMA -> MMA
  uint64_t* r_full = bars + 1;          // [AT_SLOTS] TMA -> MMA
  uint64_t* r_empty = r_full + AT_SLOTS;  // [AT_SLOTS] MMA -> TMA
  uint64_t* s_full = r_empty + AT_SLOTS;  // [2] MMA -> softmax
  uint64_t* s_empty = s_full + 2;       // [2] softmax -> MMA
  uint64_t* p_full = s_empty + 2;       // softmax -> MMA (P written, O rescaled)
  uint64_t* o_done = p_full + 1;        // MMA -> softmax (P V of a block complete)
  uint64_t* drain = o_done + 1;         // abort path only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // work unit; the longest (latest, under the causal mask) query blocks first
  const int heads = a.tp * a.nq;
  const int qb = a.q_blocks - 1 - static_cast<int>(blockIdx.x) / heads;
  const int hh = static_cast<int>(blockIdx.x) % heads;
  const int s = hh / a.nq, j = hh % a.nq;
  const int kv0 = a.hkv >= a.tp ? s * a.nkv : (s * a.hkv) / a.tp;
  const int kvi = (s * a.nq + j) / a.group - kv0;  // the kv head within the shard's block
  const int qcol = j * AT_HD, kcol = (a.nq + kvi) * AT_HD, vcol = (a.nq + a.nkv + kvi) * AT_HD;
  const int q0 = qb * AT_ROWS;
  const int nkb = a.causal ? qb + 1 : (a.T + AT_ROWS - 1) / AT_ROWS;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < AT_SLOTS; ++i) {
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
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
      int issued[AT_SLOTS];
#pragma unroll
      for (int i = 0; i < AT_SLOTS; ++i) issued[i] = -1;
      bool ok = true;
      mbar_arrive_expect_tx(q_full, AT_TILE);
      tma_load_3d(sQ, &mapQKV, q_full, qcol, q0, s);
      tma_load_3d(sQ + AT_PANEL, &mapQKV, q_full, qcol + 64, q0, s);
      for (int it = 0; it < 2 * nkb; ++it) {  // K(j), V(j), K(j+1), ...
        const int slot = it % AT_SLOTS;
        const uint32_t ph = static_cast<uint32_t>(it / AT_SLOTS) & 1u;
        if (!mbar_wait(&r_empty[slot], ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const int col = (it & 1) ? vcol : kcol;
        uint8_t* dst = ring + slot * AT_TILE;
        mbar_arrive_expect_tx(&r_full[slot], AT_TILE);
        tma_load_3d(dst, &mapQKV, &r_full[slot], col, (it >> 1) * AT_ROWS, s);
        tma_load_3d(dst + AT_PANEL, &mapQKV, &r_full[slot], col + 64, (it >> 1) * AT_ROWS, s);
        issued[slot] = static_cast<int>(ph);
      }
      if (!ok) {  // let every copy this block started land before it exits
        mbar_wait_drain(q_full, 0);
        for (int i = 0; i < AT_SLOTS; ++i)
          if (issued[i] >= 0) mbar_wait_drain(&r_full[i], static_cast<uint32_t>(issued[i]));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------ MMA issuer ------------------------------
      const uint32_t idesc_s = idesc_bf16_f32(128, 128);
      const uint32_t idesc_o = idesc_bf16_f32_bmn(128, 128);
      const uint32_t tO = tmem_base + 256;
      bool ok = mbar_wait(q_full, 0, abort_flag), issued_any = false;
      // S(jb) = Q K(jb)^T: M = 128 queries, N = 128 keys, K = hd in 8 steps
      // of 16 (two 64-wide panels, +32 bytes per step inside a panel)
      auto issue_s = [&](int jb) -> bool {
        const int st = jb & 1;
        const uint32_t ph = static_cast<uint32_t>(jb >> 1) & 1u;
        const int slot = (2 * jb) % AT_SLOTS;
        if (!mbar_wait(&r_full[slot], static_cast<uint32_t>(2 * jb / AT_SLOTS) & 1u, abort_flag)) return false;
        if (!mbar_wait(&s_empty[st], ph ^ 1u, abort_flag)) return false;
        tc_fence_after();
        const uint32_t q_a = smem_u32(sQ), k_a = smem_u32(ring + slot * AT_TILE);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = static_cast<uint32_t>((k >> 2) * AT_PANEL + (k & 3) * 32);
          tc_mma_bf16(tmem_base + static_cast<uint32_t>(st * 128), smem_desc_k_sw128(q_a + off),
                      smem_desc_k_sw128(k_a + off), idesc_s, k > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[st]);
        tc_commit(&r_empty[slot]);  // K(jb) read
        issued_any = true;
        return true;
      };
      // O += P(jb) V(jb): M = 128 queries, N = hd, K = 128 keys in 8 steps;
      // P is K-major (two 64-key panels), V MN-major (rows = keys, each row
      // 64 hd values; the second 64 hd values one panel further)
      auto issue_pv = [&](int jb) -> bool {
        const int slot = (2 * jb + 1) % AT_SLOTS;
        if (!mbar_wait(p_full, static_cast<uint32_t>(jb) & 1u, abort_flag)) return false;
        if (!mbar_wait(&r_full[slot], static_cast<uint32_t>((2 * jb + 1) / AT_SLOTS) & 1u, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t p_a = smem_u32(sP), v_a = smem_u32(ring + slot * AT_TILE);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t poff = static_cast<uint32_t>((k >> 2) * AT_PANEL + (k & 3) * 32);
          tc_mma_bf16(tO, smem_desc_k_sw128(p_a + poff),
                      smem_desc_mn_sw128(v_a + static_cast<uint32_t>(k * 16 * 128), AT_PANEL, 1024), idesc_o,
                      (jb > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(o_done);
        tc_commit(&r_empty[slot]);  // V(jb) read
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int jb = 0; ok && jb < nkb; ++jb) {
        if (jb + 1 < nkb && !issue_s(jb + 1)) {
          ok = false;
          break;
        }
        ok = issue_pv(jb);
      }
      if (!ok && issued_any) {  // wait for MMAs in flight before TMEM is freed
        tc_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // ------------------------------ softmax ------------------------------
    const int q = warp & 3;            // TMEM lane quadrant
    const int r = q * 32 + lane;       // query row within the block
    const int t = q0 + r;              // query index
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t tO = tmem_base + 256 + lane_off;
    const int kmax = a.causal ? min(t, a.T - 1) : a.T - 1;  // last key this query sees
    float m = -INFINITY;  // exponent base, in log2 units of the scaled scores
    float l = 0.0f;
    bool ok = true;
    for (int jb = 0; jb < nkb; ++jb) {
      const int st = jb & 1;
      const uint32_t ph = static_cast<uint32_t>(jb >> 1) & 1u;
      const bool waited = mbar_wait(&s_full[st], ph, abort_flag);
      if (epi_any(!waited || *abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[128];
      const uint32_t tS = tmem_base + static_cast<uint32_t>(st * 128) + lane_off;
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        uint32_t rr[32];
        tmem_ld32(tS + static_cast<uint32_t>(c), rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c + i] = __uint_as_float(rr[i]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[st]);  // S(jb + 2) may overwrite this buffer
      const int kbase = jb * AT_ROWS;
      // only the diagonal block (causal) and a ragged last block need a mask
      if ((a.causal && jb == qb) || kbase + AT_ROWS > a.T) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (kbase + i > kmax) sv[i] = -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = sv[i];
#pragma unroll
      for (int i = 8; i < 128; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], sv[i]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
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
      for (int i = 0; i < 128; ++i) {
        sv[i] = ex2_approx(fmaf(sv[i], a.scale_log2, -m));
        sum8[i & 7] += sv[i];
      }
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      // P V of the previous block has read P and finished with O
      if (jb >= 1) {
        const bool freed = mbar_wait(o_done, static_cast<uint32_t>(jb - 1) & 1u, abort_flag);
        if (epi_any(!freed || *abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // the base moved: O (all P V up to block jb - 1) is rescaled first
        {
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            uint32_t rr[32];
            tmem_ld32(tO + static_cast<uint32_t>(c), rr);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            tmem_st32(tO + static_cast<uint32_t>(c), rr);
          }
          tmem_st_wait();
        }
      }
      // P row in bf16: keys 0..63 in panel 0, 64..127 in panel 1, 16-byte
      // chunks at the 128-byte swizzle position of this row
      uint8_t* pb = sP;
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        const int panel = c8 >> 3, ch = c8 & 7;
        uint4 v;
        v.x = pack_bf16x2(sv[c8 * 8 + 0], sv[c8 * 8 + 1]);
        v.y = pack_bf16x2(sv[c8 * 8 + 2], sv[c8 * 8 + 3]);
        v.z = pack_bf16x2(sv[c8 * 8 + 4], sv[c8 * 8 + 5]);
        v.w = pack_bf16x2(sv[c8 * 8 + 6], sv[c8 * 8 + 7]);
        *reinterpret_cast<uint4*>(pb + panel * AT_PANEL + r * 128 + ((ch ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();  // the tensor core reads P through the async proxy
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && !*abort_flag) {
      const bool done = mbar_wait(o_done, static_cast<uint32_t>(nkb - 1) & 1u, abort_flag);
      if (!epi_any(!done || *abort_flag)) {
        tc_fence_after();
        const float inv = 1.0f / l;
        const int nc = a.nq * AT_HD;
        __nv_bfloat16* out = a.ctx + (static_cast<size_t>(s) * a.T + t) * nc + j * AT_HD;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
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
      }
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
