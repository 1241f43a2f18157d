// Vocabulary-parallel input and output layers ("Tensor parallelism:
// splitting Transformer layers" tutorial page, input and output layers;
// "What is tensor parallelism" page, loss sharded over the class dimension):
//
//   embedding     the table E [V][H] is split by vocabulary rows, shard s
//                 holding ids [s*V/tp, (s+1)*V/tp) as the row block
//                 E[s*V/tp ..] (so the shards, stored one after another, are
//                 E itself). A lookup is every shard's masked lookup summed
//                 over shards; exactly one shard owns an id, so the sum is
//                 that shard's row, which this kernel copies directly (x + 0
//                 is x): one warp per token, 16-byte vectors.
//   cross-entropy logits [tp][T][V/tp] split by vocabulary columns (the
//                 column-parallel LM head's per-shard output). Pass 1: per
//                 (shard, token) row the maximum m_s, the sum of exp(z - m_s)
//                 and, on the shard that owns the label, its logit. Pass 2:
//                 per token, the all-reduce of those statistics
//                 (m = max m_s, S = sum_s S_s exp(m_s - m)) and
//                 loss = m + log S - z_label; then the mean over tokens in a
//                 fixed order. Pass 3 (optional): the gradient of
//                 scale * sum_t loss[t], scale * (exp(z - lse) - [v == label]),
//                 written over the logits or to another buffer.
// Ids and labels outside [0, V) record TP_DEVERR_INDEX in the device error
// word; their rows read as zeros and their losses as NaN.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tp_epilogue.cuh"
#include "tp_ptx.cuh"

namespace tpk {

// ---------------------------------------------------------------------------
// Embedding lookup. Y [T][H]; E [V][H]; v = V / tp rows per shard.
// vec: H * sizeof(T) is a multiple of 16 and both pointers are 16-aligned.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void vocab_embed_kernel(const int32_t* __restrict__ ids, int64_t n_tok, const T* __restrict__ E,
                                   int64_t V, int64_t H, int64_t v, int vec, T* __restrict__ Y) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_tok;
       t += warps) {
    const int64_t id = ids[t];
    const bool ok = id >= 0 && id < V;
    if (!ok && lane == 0) atomicCAS(&g_tp_error, TP_DEVERR_NONE, TP_DEVERR_INDEX);
    // the owning shard and the row inside it
    const int64_t s = ok ? id / v : 0, local = ok ? id - s * v : 0;
    const T* src = E + (s * v + local) * H;
    T* dst = Y + t * H;
    if (vec) {
      constexpr int PER = 16 / sizeof(T);
      const int64_t n16 = H / PER;
      for (int64_t i = lane; i < n16; i += 32) {
        const uint4 q = ok ? __ldg(reinterpret_cast<const uint4*>(src) + i) : make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(dst)[i] = q;
      }
    } else {
      for (int64_t i = lane; i < H; i += 32) dst[i] = ok ? src[i] : from_f32<T>(0.0f);
    }
  }
}

// ---------------------------------------------------------------------------
// Cross-entropy, pass 1: one warp per (shard, token) row of v logits.
// stats[(s * T + t) * 3 + {0, 1, 2}] = {max, sum exp(z - max), label logit
// or 0 when shard s does not own the label}.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void lse_merge(float& m, float& S, float m2, float S2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  S = S * __expf(m - mn) + S2 * __expf(m2 - mn);
  m = mn;
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&x)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_lo(w[i]);
    x[2 * i + 1] = bf16_hi(w[i]);
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&x)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <typename T>
__global__ void ce_stats_kernel(const T* __restrict__ logits, const int32_t* __restrict__ labels, int64_t n_tok,
                                int tp, int64_t v, int vec, float* __restrict__ stats) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = n_tok * tp;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const int64_t s = r / n_tok, t = r - s * n_tok;
    const T* z = logits + r * v;
    float m = -INFINITY, S = 0.0f;
    if (vec) {  // 8 logits per step, v % 8 == 0
      for (int64_t i = static_cast<int64_t>(lane) * 8; i < v; i += 32 * 8) {
        float x[8];
        load8<T>(z + i, x);
        float mx = x[0];
#pragma unroll
        for (int j = 1; j < 8; ++j) mx = fmaxf(mx, x[j]);
        float acc = 0.0f;
        const float mn = fmaxf(m, mx);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc += __expf(x[j] - mn);
        S = (m == -INFINITY ? 0.0f : S * __expf(m - mn)) + acc;
        m = mn;
      }
    } else {
      for (int64_t i = lane; i < v; i += 32) {
        const float x = to_f32<T>(z[i]);
        const float mn = fmaxf(m, x);
        S = (m == -INFINITY ? 0.0f : S * __expf(m - mn)) + __expf(x - mn);
        m = mn;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), S2 = __shfl_xor_sync(0xffffffffu, S, o);
      lse_merge(m, S, m2, S2);
    }
    if (lane == 0) {
      const int64_t y = labels[t];
      const int64_t loc = y - s * v;
      const float zy = (loc >= 0 && loc < v) ? to_f32<T>(z[loc]) : 0.0f;
      float* o = stats + r * 3;
      o[0] = m;
      o[1] = S;
      o[2] = zy;
    }
  }
}

// ---------------------------------------------------------------------------
// Pass 2: per token, combine the tp shards' statistics in shard order.
// lse[t] = m + log S (kept for the gradient); loss[t] = lse[t] - z_label.
// ---------------------------------------------------------------------------
__global__ void ce_combine_kernel(const float* __restrict__ stats, const int32_t* __restrict__ labels,
                                  int64_t n_tok, int tp, int64_t V, float* __restrict__ lse,
                                  float* __restrict__ loss) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n_tok; t += stride) {
    const int64_t y = labels[t];
    const bool ok = y >= 0 && y < V;
    if (!ok) atomicCAS(&g_tp_error, TP_DEVERR_NONE, TP_DEVERR_INDEX);
    const int64_t v = V / tp;
    const int owner = ok ? static_cast<int>(y / v) : 0;
    float m = -INFINITY, S = 0.0f, zy = 0.0f;
    for (int s = 0; s < tp; ++s) {
      const float* st = stats + (static_cast<int64_t>(s) * n_tok + t) * 3;
      lse_merge(m, S, st[0], st[1]);
      if (s == owner) zy = st[2];
    }
    const float l = m + __logf(S);
    lse[t] = l;
    loss[t] = ok ? l - zy : __int_as_float(0x7fc00000);
  }
}

// Mean of loss[0..n) in a fixed order: one CTA of 1024 threads, each a
// strided partial sum, then a tree.
__global__ void ce_mean_kernel(const float* __restrict__ loss, int64_t n, float* __restrict__ out) {
  __shared__ float part[1024];
  float acc = 0.0f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) acc += loss[i];
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[0] = n > 0 ? part[0] / static_cast<float>(n) : 0.0f;
}

// ---------------------------------------------------------------------------
// Pass 3: dz = scale * (exp(z - lse[t]) - [global column == label]) over the
// [tp][T][v] logits; out may alias logits (each element is read, then
// written, by the same thread). 8 elements per step when vec.
// ---------------------------------------------------------------------------
// Plain (coherent) loads for the gradient pass, whose output may be the
// logits themselves.
template <typename T>
__device__ __forceinline__ void load8_rw(const T* p, float (&x)[8]);
template <>
__device__ __forceinline__ void load8_rw<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_lo(w[i]);
    x[2 * i + 1] = bf16_hi(w[i]);
  }
}
template <>
__device__ __forceinline__ void load8_rw<float>(const float* p, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <typename T>
__global__ void ce_grad_kernel(const T* logits, const int32_t* __restrict__ labels, const float* __restrict__ lse,
                               int64_t n_tok, int tp, int64_t v, float scale, int vec, T* out) {
  const int64_t total = n_tok * tp * v;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (vec) {
    const int64_t n8 = total / 8;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
      const int64_t e = i * 8, r = e / v, c = e - r * v;  // r = s * T + t; 8 | v, so the 8 share a row
      const int64_t s = r / n_tok, t = r - s * n_tok;
      const float l = lse[t];
      const int64_t loc = static_cast<int64_t>(labels[t]) - s * v;
      float x[8], g[8];
      load8_rw<T>(logits + e, x);
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = scale * (__expf(x[j] - l) - (c + j == loc ? 1.0f : 0.0f));
      if constexpr (sizeof(T) == 2) {
        *reinterpret_cast<uint4*>(out + e) = make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                                                        pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7]));
      } else {
        reinterpret_cast<float4*>(out + e)[0] = make_float4(g[0], g[1], g[2], g[3]);
        reinterpret_cast<float4*>(out + e)[1] = make_float4(g[4], g[5], g[6], g[7]);
      }
    }
  } else {
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += stride) {
      const int64_t r = e / v, c = e - r * v;
      const int64_t s = r / n_tok, t = r - s * n_tok;
      const int64_t loc = static_cast<int64_t>(labels[t]) - s * v;
      out[e] = from_f32<T>(scale * (__expf(to_f32<T>(logits[e]) - lse[t]) - (c == loc ? 1.0f : 0.0f)));
    }
  }
}

}  // namespace tpk
