// Mixture of experts with tensor-parallel experts ("Parallel strategies in
// TensorRT LLM" page, FFN module, mixture of experts, TP mode: every expert's
// weights are split across all shards and every shard sees all tokens).
//
// The router's choice is an input: ids [T][k] (expert of each of a token's k
// slots) and weights [T][k]. The block runs
//   1. dispatch: every (token, slot) entry gets a row in a permuted buffer
//      Xp, the experts' segments one after another in expert order, each
//      segment in token order and padded to a multiple of 256 rows (one
//      CTA-pair unit); unit_expert[u] names the expert of each 256-row unit
//      (-1 past the last one);
//   2. the experts' MLP blocks as two grouped GEMM launches over all units
//      (gate/up with the SwiGLU epilogue per shard, then down with the shard
//      sum, written as fp32 rows Yp), each tile taking its expert's shard set;
//   3. combine: Y[t] = sum_j weights[t][j] * Yp[row of (t, j)] (+ residual),
//      in slot order, fp32 accumulation, one bf16 rounding at the end.
// Everything is deterministic: positions come from ordered scans, not from
// atomics. An id outside [0, E) records TP_DEVERR_INDEX; that entry is left
// out of the sum.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tp_epilogue.cuh"
#include "tp_ptx.cuh"

namespace tpk {

constexpr int MOE_UNIT = 256;  // rows per CTA-pair unit

// 1a. One CTA (1024 threads) per expert e: the position of every entry routed
// to e among e's entries, in entry order (t * k + j); counts[e].
__global__ void __launch_bounds__(1024) moe_route_kernel(const int32_t* __restrict__ ids, int64_t n, int E,
                                                          int32_t* __restrict__ pos, int32_t* __restrict__ counts) {
  __shared__ int warp_tot[32];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int base = 0;
  for (int64_t c = 0; c < n; c += 1024) {
    const int64_t i = c + threadIdx.x;
    const int id = i < n ? ids[i] : -1;
    if (e == 0 && i < n && (id < 0 || id >= E)) atomicCAS(&g_tp_error, TP_DEVERR_NONE, TP_DEVERR_INDEX);
    const bool mine = id == e;
    const unsigned bal = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) warp_tot[w] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
    for (int q = 0; q < 32; ++q) {  // warps before this one, then all
      const int v = warp_tot[q];
      before += q < w ? v : 0;
      total += v;
    }
    if (mine) pos[i] = base + before + __popc(bal & ((1u << lane) - 1u));
    base += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) counts[e] = base;
}

// 1b. One CTA: segment offsets (each count padded to a multiple of 256), the
// unit -> expert table for n_units units (-1 past the last segment) and each
// unit's segment {first unit, units} (an unused unit: itself alone), which
// orders the grouped GEMMs' tiles. E <= 1024.
__global__ void moe_units_kernel(const int32_t* __restrict__ counts, int E, int n_units, int32_t* __restrict__ off,
                                 int32_t* __restrict__ unit_expert, int2* __restrict__ unit_seg) {
  __shared__ int s_off[1025];
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_off[e] = acc;
      acc += (counts[e] + MOE_UNIT - 1) / MOE_UNIT * MOE_UNIT;
    }
    s_off[E] = acc;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) off[e] = s_off[e];
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
    const int row = u * MOE_UNIT;
    int ex = -1;
    for (int e = 0; e < E; ++e)
      if (row >= s_off[e] && row < s_off[e + 1]) ex = e;
    unit_expert[u] = ex;
    unit_seg[u] = ex >= 0 ? make_int2(s_off[ex] / MOE_UNIT, (s_off[ex + 1] - s_off[ex]) / MOE_UNIT) : make_int2(u, 1);
  }
}

// 1c. One warp per entry: its row in Xp (inv), and the token's row copied
// there in 16-byte vectors (H * 2 bytes is a multiple of 16).
__global__ void moe_gather_kernel(const __nv_bfloat16* __restrict__ X, const int32_t* __restrict__ ids,
                                  const int32_t* __restrict__ pos, const int32_t* __restrict__ off, int64_t n,
                                  int k, int E, int64_t H, __nv_bfloat16* __restrict__ Xp,
                                  int32_t* __restrict__ inv) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); i < n; i += warps) {
    const int e = ids[i];
    if (e < 0 || e >= E) {
      if (lane == 0) inv[i] = -1;
      continue;
    }
    const int64_t dst = static_cast<int64_t>(off[e]) + pos[i];
    if (lane == 0) inv[i] = static_cast<int32_t>(dst);
    const uint4* src = reinterpret_cast<const uint4*>(X + (i / k) * H);
    uint4* d = reinterpret_cast<uint4*>(Xp + dst * H);
    for (int64_t v = lane; v < H / 8; v += 32) d[v] = __ldg(src + v);
  }
}

// 3. One warp per token: Y[t] = sum_j w[t][j] * Yp[inv[t][j]] (+ residual),
// slot order, fp32 (Yp is fp32); 8 columns per lane and step.
__global__ void moe_combine_kernel(const float* __restrict__ Yp, const int32_t* __restrict__ inv,
                                   const float* __restrict__ wts, int64_t T, int k, int64_t H,
                                   const __nv_bfloat16* __restrict__ residual, __nv_bfloat16* __restrict__ Y) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
    for (int64_t c = static_cast<int64_t>(lane) * 8; c < H; c += 32 * 8) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
      for (int j = 0; j < k; ++j) {
        const int r = inv[t * k + j];
        if (r < 0) continue;
        const float w = wts[t * k + j];
        const float4* src = reinterpret_cast<const float4*>(Yp + static_cast<int64_t>(r) * H + c);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(w, v[q], acc[q]);
      }
      if (residual) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(residual + t * H + c));
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] += bf16_lo(wd[q]);
          acc[2 * q + 1] += bf16_hi(wd[q]);
        }
      }
      *reinterpret_cast<uint4*>(Y + t * H + c) = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                            pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

}  // namespace tpk
