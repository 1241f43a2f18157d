// Memory-bound kernels of the pipeline: weight sharding, the on-device
// combines (concatenation = all-gather, sum = all-reduce, reduce-scatter),
// RMSNorm on the replicated hidden, and the attention-context stand-in.
#pragma once

#include "tp_epilogue.cuh"

namespace tpk {

// ---------------------------------------------------------------------------
// Weight sharding. Input W is [K][N] row-major (the [in, out] orientation,
// Y = X @ W). Output shards are stored K-major so that a GEMM tile of one
// shard is a block of contiguous rows:
//   column mode: shard s = W[:, s*N/tp:(s+1)*N/tp]^T, stored [tp][N/tp][K]
//                (the whole output equals W^T);
//   row mode:    shard s = W[s*K/tp:(s+1)*K/tp, :]^T, stored [tp][N][K/tp].
// A 32x32 shared-memory transpose; grid (ceil(N/32), ceil(K/32)).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void shard_weights_kernel(const T* __restrict__ W, int64_t K, int64_t N, int64_t Ks,
                                     int row_mode, T* __restrict__ out) {
  __shared__ T tile[32][33];
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 32, k0 = static_cast<int64_t>(blockIdx.y) * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
  for (int r = ty; r < 32; r += 8) {
    const int64_t k = k0 + r, n = n0 + tx;
    if (k < K && n < N) tile[r][tx] = W[k * N + n];
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int64_t n = n0 + r, k = k0 + tx;
    if (k < K && n < N) {
      int64_t dst;
      if (!row_mode) {
        dst = n * K + k;
      } else {
        const int64_t s = k / Ks, kl = k - s * Ks;
        dst = (s * N + n) * Ks + kl;
      }
      out[dst] = tile[tx][r];
    }
  }
}

// QKV sharded by heads. Shard s holds its q heads, then its kv heads' K
// columns, then their V columns, stored K-major: out [tp][Nqkv_s][H].
// kv_first(s) is s*nkv when hkv >= tp, else the replicated head
// floor(s*hkv/tp). grid (ceil(Nqkv_s/32), ceil(H/32), tp).
template <typename T>
__global__ void shard_qkv_kernel(const T* __restrict__ Wq, const T* __restrict__ Wk,
                                 const T* __restrict__ Wv, int64_t H, int hq, int hkv, int hd, int tp,
                                 T* __restrict__ out) {
  __shared__ T tile[32][33];
  const int s = blockIdx.z;
  const int nq = hq / tp;
  const int nkv = hkv >= tp ? hkv / tp : 1;
  const int kv0 = hkv >= tp ? s * nkv : (s * hkv) / tp;
  const int64_t Nq = static_cast<int64_t>(nq) * hd, Nkv = static_cast<int64_t>(nkv) * hd;
  const int64_t Ns = Nq + 2 * Nkv;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32, k0 = static_cast<int64_t>(blockIdx.y) * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int i = ty; i < 32; i += 8) {
    const int64_t k = k0 + i, r = r0 + tx;
    if (k < H && r < Ns) {
      T v;
      if (r < Nq) {
        v = Wq[k * hq * hd + static_cast<int64_t>(s) * Nq + r];
      } else if (r < Nq + Nkv) {
        v = Wk[k * hkv * hd + static_cast<int64_t>(kv0) * hd + (r - Nq)];
      } else {
        v = Wv[k * hkv * hd + static_cast<int64_t>(kv0) * hd + (r - Nq - Nkv)];
      }
      tile[i][tx] = v;
    }
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int64_t r = r0 + i, k = k0 + tx;
    if (k < H && r < Ns) out[(static_cast<int64_t>(s) * Ns + r) * H + k] = tile[tx][i];
  }
}

// ---------------------------------------------------------------------------
// Gather (all-gather semantics): shards [tp][T][Ns] -> Y[T][tp*Ns].
// VEC elements per thread (16-byte copies when the widths allow).
// ---------------------------------------------------------------------------
template <typename T, int VEC>
__global__ void gather_kernel(const T* __restrict__ in, int tp, int64_t Tn, int64_t Ns,
                              T* __restrict__ out) {
  const int64_t nv = Ns / VEC;
  const int64_t total = static_cast<int64_t>(tp) * Tn * nv;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t j = i % nv;
    const int64_t t = (i / nv) % Tn;
    const int64_t s = i / (nv * Tn);
    const T* src = in + (s * Tn + t) * Ns + j * VEC;
    T* dst = out + t * tp * Ns + s * Ns + j * VEC;
    if constexpr (VEC * sizeof(T) == 16) {
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    } else {
#pragma unroll
      for (int v = 0; v < VEC; ++v) dst[v] = src[v];
    }
  }
}

// ---------------------------------------------------------------------------
// Reduce (all-reduce / reduce-scatter semantics): out[t][n] = sum over
// s = 0..tp-1 of P[s][t][n], in that order, in fp32, then + bias[n] once and
// + residual[t][n]. For reduce-scatter the output buffer is read as
// [tp][T/tp][N]: shard s's slice holds token rows [s*T/tp, (s+1)*T/tp),
// which is the same memory as [T][N]. 4 elements per thread.
// ---------------------------------------------------------------------------
template <typename TO>
__global__ void reduce_kernel(const float* __restrict__ P, int tp, int64_t Tn, int64_t N,
                              const TO* __restrict__ bias, const TO* __restrict__ residual,
                              TO* __restrict__ out) {
  const int64_t total4 = Tn * N / 4;
  const int64_t plane = Tn * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i * 4;
    float4 acc = *reinterpret_cast<const float4*>(P + e);
    for (int s = 1; s < tp; ++s) {
      const float4 p = *reinterpret_cast<const float4*>(P + s * plane + e);
      acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
    }
    float v[4] = {acc.x, acc.y, acc.z, acc.w};
    const int64_t n = e % N;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (bias) v[j] += to_f32(bias[n + j]);
      if (residual) v[j] += to_f32(residual[e + j]);
      out[e + j] = from_f32<TO>(v[j]);
    }
  }
}

// Scalar variant for widths that are not a multiple of 4.
template <typename TO>
__global__ void reduce_kernel_scalar(const float* __restrict__ P, int tp, int64_t Tn, int64_t N,
                                     const TO* __restrict__ bias, const TO* __restrict__ residual,
                                     TO* __restrict__ out) {
  const int64_t total = Tn * N;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float v = P[e];
    for (int s = 1; s < tp; ++s) v += P[s * total + e];
    if (bias) v += to_f32(bias[e % N]);
    if (residual) v += to_f32(residual[e]);
    out[e] = from_f32<TO>(v);
  }
}

// ---------------------------------------------------------------------------
// RMSNorm over the replicated hidden: y = x * g / sqrt(mean(x^2) + eps),
// fp32 statistics. One 256-thread block per token row.
// ---------------------------------------------------------------------------
template <typename T, typename TO>
__global__ void rmsnorm_kernel(const T* __restrict__ X, const T* __restrict__ gamma, int64_t H,
                               float eps, TO* __restrict__ Y) {
  const int64_t row = blockIdx.x;
  const T* x = X + row * H;
  TO* y = Y + row * H;
  float ss = 0.0f;
  for (int64_t i = threadIdx.x; i < H; i += blockDim.x) {
    const float v = to_f32(x[i]);
    ss = fmaf(v, v, ss);
  }
  __shared__ float red[32];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / static_cast<float>(H) + eps);
  for (int64_t i = threadIdx.x; i < H; i += blockDim.x) {
    float v = to_f32(x[i]) * inv;
    if (gamma) v *= to_f32(gamma[i]);
    y[i] = from_f32<TO>(v);
  }
}

// ---------------------------------------------------------------------------
// Attention-context stand-in as a separate copy (the fp32 path; the bf16
// QKV GEMM writes the same context from its epilogue): with each query
// attending only to its own token, the softmax weight is 1 and the context
// of local q head j is V of its kv head. qkv [tp][T][Nqkv_s] (q | k | v per
// shard) -> ctx [tp][T][nq*hd]. Block (32, 8): eight (shard, token) rows per
// block, the 32 lanes stride over the row in 16-byte chunks (bf16, hd % 8 ==
// 0) or single elements (fp32); 32-bit index math inside a row.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void ctx_standin_kernel(const T* __restrict__ qkv, int tp, int64_t Tn, int hq, int hkv,
                                   int hd, T* __restrict__ ctx) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.y + threadIdx.y;  // s * T + t
  if (row >= static_cast<int64_t>(tp) * Tn) return;
  const int s = static_cast<int>(row / Tn);
  const int nq = hq / tp;
  const int nkv = hkv >= tp ? hkv / tp : 1;
  const int group = hq / hkv;
  const int kv0 = hkv >= tp ? s * nkv : (s * hkv) / tp;
  const int Nqkv = (nq + 2 * nkv) * hd;
  const int Nc = nq * hd;
  const T* src_row = qkv + row * Nqkv + (nq + nkv) * hd;  // start of this shard-row's V block
  T* dst_row = ctx + row * Nc;
  constexpr int CH = sizeof(T) == 2 ? 8 : 1;  // bf16: 16-byte chunks (hd % 8 == 0); fp32: elements
  for (int c = threadIdx.x * CH; c < Nc; c += 32 * CH) {
    const int j = c / hd;
    const int g = (s * nq + j) / group;  // kv head of global q head s*nq + j
    const T* src = src_row + (g - kv0) * hd + (c - j * hd);
    if constexpr (CH == 8) {
      *reinterpret_cast<uint4*>(dst_row + c) = *reinterpret_cast<const uint4*>(src);
    } else {
      dst_row[c] = *src;
    }
  }
}

// ---------------------------------------------------------------------------
// Gradient through the MLP's local activation (the backward of the tutorial
// page's MLP block step 2), per element of the shards' intermediate
// [tp][T][I/tp]: dG = dH * act'(G), and for SwiGLU dG = dH * U * silu'(G),
// dU = dH * silu(G) (act_grad). bf16 in and out, fp32 arithmetic, eight
// elements (16 bytes) per step; n8 = elements / 8. HBM-bound: per element 2
// (SwiGLU 3) bf16 reads and 1 (2) bf16 writes.
// With rows8 > 0, dG and dU are written token-major, [T][tp * I/tp] (the
// shards side by side in each token row, so that the backward's GEMMs run
// over all of I at once): vector t * rows8 + c of shard s (rows8 = I/tp / 8,
// blockIdx.y = s, n8 = T * rows8 < 2^31 vectors a shard) goes to
// (t * tp + s) * rows8 + c. t = i / rows8 is taken as
// (umulhi(magic, i) + i) >> shift, the round-up method of Granlund and
// Montgomery ("Division by invariant integers using multiplication", 1994),
// with shift = ceil(log2 rows8) and magic = floor(2^(32 + shift) / rows8) -
// 2^32 + 1, exact for every i < 2^31.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void act_backward_vec(const __nv_bfloat16* __restrict__ dH,
                                                 const __nv_bfloat16* __restrict__ G,
                                                 const __nv_bfloat16* __restrict__ U, int act, int64_t i, int64_t o,
                                                 __nv_bfloat16* __restrict__ dG, __nv_bfloat16* __restrict__ dU) {
  const uint4 h4 = reinterpret_cast<const uint4*>(dH)[i];
  const uint4 g4 = reinterpret_cast<const uint4*>(G)[i];
  const uint4 u4 = act == ACT_SWIGLU ? reinterpret_cast<const uint4*>(U)[i] : make_uint4(0, 0, 0, 0);
  const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w}, gw[4] = {g4.x, g4.y, g4.z, g4.w},
                 uw[4] = {u4.x, u4.y, u4.z, u4.w};
  uint32_t og[4], ou[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float dg0, du0, dg1, du1;
    // element 2w is the low half of a 32-bit word, 2w + 1 the high half
    act_grad(act, __uint_as_float(hw[w] << 16), __uint_as_float(gw[w] << 16), __uint_as_float(uw[w] << 16), dg0,
             du0);
    act_grad(act, __uint_as_float(hw[w] & 0xFFFF0000u), __uint_as_float(gw[w] & 0xFFFF0000u),
             __uint_as_float(uw[w] & 0xFFFF0000u), dg1, du1);
    __nv_bfloat162 a = __floats2bfloat162_rn(dg0, dg1), b = __floats2bfloat162_rn(du0, du1);
    og[w] = *reinterpret_cast<uint32_t*>(&a);
    ou[w] = *reinterpret_cast<uint32_t*>(&b);
  }
  reinterpret_cast<uint4*>(dG)[o] = make_uint4(og[0], og[1], og[2], og[3]);
  if (act == ACT_SWIGLU) reinterpret_cast<uint4*>(dU)[o] = make_uint4(ou[0], ou[1], ou[2], ou[3]);
}

__global__ void act_backward_kernel(const __nv_bfloat16* __restrict__ dH, const __nv_bfloat16* __restrict__ G,
                                    const __nv_bfloat16* __restrict__ U, int64_t n8, int act,
                                    __nv_bfloat16* __restrict__ dG, __nv_bfloat16* __restrict__ dU,
                                    uint32_t rows8 = 0, uint32_t magic = 0, int shift = 0, int tp = 1) {
  if (rows8 > 0) {
    const uint32_t per = static_cast<uint32_t>(n8);
    const int64_t sh = blockIdx.y;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < per; i += stride) {
      const uint32_t t = (__umulhi(magic, i) + i) >> shift;
      const uint32_t c = i - t * rows8;
      act_backward_vec(dH, G, U, act, sh * per + i, (static_cast<int64_t>(t) * tp + sh) * rows8 + c, dG, dU);
    }
    return;
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride)
    act_backward_vec(dH, G, U, act, i, i, dG, dU);
}

// fp32 form of act_backward_kernel: one element per step, any count.
__global__ void act_backward_f32_kernel(const float* __restrict__ dH, const float* __restrict__ G,
                                        const float* __restrict__ U, int64_t n, int act, float* __restrict__ dG,
                                        float* __restrict__ dU) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    float dg, du;
    act_grad(act, dH[i], G[i], act == ACT_SWIGLU ? U[i] : 0.0f, dg, du);
    dG[i] = dg;
    if (act == ACT_SWIGLU) dU[i] = du;
  }
}

}  // namespace tpk
