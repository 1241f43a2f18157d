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
//                 (shard, token) row, in chunks of 2048 logits, the maximum,
//                 the sum of exp(z - max) and the label's logit where the
//                 chunk holds it (else 0). Pass 2: per token, the all-reduce
//                 of those statistics over shards and chunks
//                 (m = max m_i, S = sum_i S_i exp(m_i - m), z_label = the
//                 sum of the masked label logits) and
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

// Units of work: a row (shard s, token t) of v logits in chunks of CE_CHUNK;
// one warp per (row, chunk). On the vector path each lane keeps CE_NV
// packed 16-byte vectors in flight (bf16: 8 x 8 logits, the whole 2048-logit
// chunk in one step; fp32: two steps of 8 x 4), all loads issued before the
// arithmetic. Partial statistics per unit:
// stats[((s * T + t) * nchunk + c) * 3 + {0, 1, 2}] = {max, sum exp(z - max),
// label logit if this chunk holds the label, else 0}.
constexpr int CE_CHUNK = 2048;
constexpr int CE_NV = 8;

// Element j of a 16-byte vector of T.
template <typename T>
__device__ __forceinline__ float vec_elem(const uint4& q, int j);
template <>
__device__ __forceinline__ float vec_elem<__nv_bfloat16>(const uint4& q, int j) {
  const uint32_t w = j < 2 ? q.x : j < 4 ? q.y : j < 6 ? q.z : q.w;
  return (j & 1) ? bf16_hi(w) : bf16_lo(w);
}
template <>
__device__ __forceinline__ float vec_elem<float>(const uint4& q, int j) {
  return __uint_as_float(j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w);
}

template <typename T>
__global__ void ce_stats_kernel(const T* __restrict__ logits, const int32_t* __restrict__ labels, int64_t n_tok,
                                int tp, int64_t v, int vec, float* __restrict__ stats) {
  const int lane = threadIdx.x & 31;
  const int64_t nchunk = (v + CE_CHUNK - 1) / CE_CHUNK;
  const int64_t units = n_tok * tp * nchunk;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t un = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); un < units;
       un += warps) {
    const int64_t r = un / nchunk, c0 = (un - r * nchunk) * CE_CHUNK;
    const int64_t c1 = min(v, c0 + CE_CHUNK);
    const int64_t s = r / n_tok, t = r - s * n_tok;
    const T* z = logits + r * v;
    // the label and, where this chunk holds it, its logit: loaded with the
    // data rather than after the reduction
    const int64_t loc = static_cast<int64_t>(labels[t]) - s * v;
    const bool has_label = loc >= c0 && loc < c1;
    const float zy = (has_label && lane == 0) ? to_f32<T>(z[loc]) : 0.0f;
    float m = -INFINITY, S = 0.0f;
    if (vec) {  // v % 8 == 0, so every 16-byte vector is whole and aligned
      constexpr int EPV = 16 / sizeof(T);
      for (int64_t base = c0; base < c1; base += CE_NV * 32 * EPV) {
        uint4 q[CE_NV];
#pragma unroll
        for (int u = 0; u < CE_NV; ++u) {
          const int64_t i = base + (u * 32 + lane) * EPV;
          q[u] = i < c1 ? __ldg(reinterpret_cast<const uint4*>(z + i)) : make_uint4(0, 0, 0, 0);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < CE_NV; ++u)
          if (base + (u * 32 + lane) * EPV < c1)
#pragma unroll
            for (int j = 0; j < EPV; ++j) mx = fmaxf(mx, vec_elem<T>(q[u], j));
        if (mx != -INFINITY) {
          float acc = 0.0f;
#pragma unroll
          for (int u = 0; u < CE_NV; ++u)
            if (base + (u * 32 + lane) * EPV < c1)
#pragma unroll
              for (int j = 0; j < EPV; ++j) acc += __expf(vec_elem<T>(q[u], j) - mx);
          lse_merge(m, S, mx, acc);
        }
      }
    } else {
      for (int64_t i = c0 + lane; i < c1; i += 32) {
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
      float* o = stats + un * 3;
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
                                  int64_t n_tok, int tp, int64_t V, int64_t nchunk, float* __restrict__ lse,
                                  float* __restrict__ loss) {
  // one warp per token: lane i merges units i, i + 32, ... (shard-major,
  // then chunk), then the lanes merge in a fixed butterfly; the label logit
  // is the sum of the units' entries, all zero but the owner's (a masked
  // value summed)
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t nu = tp * nchunk;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_tok;
       t += warps) {
    float m = -INFINITY, S = 0.0f, zy = 0.0f;
    for (int64_t i = lane; i < nu; i += 32) {
      const int64_t s = i / nchunk, c = i - s * nchunk;
      const float* st = stats + ((s * n_tok + t) * nchunk + c) * 3;
      lse_merge(m, S, st[0], st[1]);
      zy += st[2];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), S2 = __shfl_xor_sync(0xffffffffu, S, o);
      lse_merge(m, S, m2, S2);
      zy += __shfl_xor_sync(0xffffffffu, zy, o);
    }
    if (lane == 0) {
      const int64_t y = labels[t];
      const bool ok = y >= 0 && y < V;
      if (!ok) atomicCAS(&g_tp_error, TP_DEVERR_NONE, TP_DEVERR_INDEX);
      const float l = m + __logf(S);
      lse[t] = l;
      loss[t] = ok ? l - zy : __int_as_float(0x7fc00000);
    }
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
template <typename T>
__global__ void ce_grad_kernel(const T* logits, const int32_t* __restrict__ labels, const float* __restrict__ lse,
                               int64_t n_tok, int tp, int64_t v, float scale, int vec, T* out) {
  const int64_t total = n_tok * tp * v;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (vec) {  // one warp per (row, chunk) unit as in pass 1; v % 8 == 0
    const int lane = threadIdx.x & 31;
    const int64_t nchunk = (v + CE_CHUNK - 1) / CE_CHUNK;
    const int64_t units = n_tok * tp * nchunk;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t un = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); un < units;
         un += warps) {
      const int64_t r = un / nchunk, c0 = (un - r * nchunk) * CE_CHUNK;
      const int64_t c1 = min(v, c0 + CE_CHUNK);
      const int64_t s = r / n_tok, t = r - s * n_tok;
      const float l = lse[t];
      const int64_t loc = static_cast<int64_t>(labels[t]) - s * v;
      const T* z = logits + r * v;
      T* o = out + r * v;
      constexpr int EPV = 16 / sizeof(T);
      for (int64_t base = c0; base < c1; base += CE_NV * 32 * EPV) {
        uint4 q[CE_NV];
#pragma unroll
        for (int u = 0; u < CE_NV; ++u) {
          const int64_t i = base + (u * 32 + lane) * EPV;
          if (i < c1) q[u] = *reinterpret_cast<const uint4*>(z + i);  // coherent: o may be z
        }
#pragma unroll
        for (int u = 0; u < CE_NV; ++u) {
          const int64_t i = base + (u * 32 + lane) * EPV;
          if (i >= c1) break;
          float g[EPV];
#pragma unroll
          for (int j = 0; j < EPV; ++j)
            g[j] = scale * (__expf(vec_elem<T>(q[u], j) - l) - (i + j == loc ? 1.0f : 0.0f));
          if constexpr (sizeof(T) == 2) {
            *reinterpret_cast<uint4*>(o + i) = make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                                                          pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7]));
          } else {
            *reinterpret_cast<float4*>(o + i) = make_float4(g[0], g[1], g[2], g[3]);
          }
        }
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
