// fp32 path of the sharded linears: a plain shared-memory-tiled FFMA GEMM.
//
// Used for fp32 tensors (the exact-integer workload among them). Each output
// element accumulates its products in a fixed order (shard ascending, then k
// ascending) with fmaf, so integer-valued inputs whose partial sums stay
// below 2^24 give exact results. TF32 tensor cores are not used here: they
// round fp32 inputs to 10 mantissa bits.
#pragma once

#include "tp_epilogue.cuh"

namespace tpk {

enum SimtKind : int { SK_COL = 0, SK_COL_SWIGLU = 1, SK_ROW_SUM = 2, SK_ROW_PARTIAL = 3 };

constexpr int SK_BM = 64, SK_BN = 64, SK_BK = 16, SK_THREADS = 256;

struct SimtArgs {
  int M, Ns, Ks, tp;
  int k_shards;            // ROW_SUM: tp, else 1
  int act, out_concat;
  const float* A;          // COL: X [M][Ks]; ROW: Xs [tp][M][Ks]
  int64_t a_shard_stride;  // 0 for COL, M*Ks for ROW
  const float* B0;         // shards, K-major: [tp][Ns][Ks]
  const float* B1;         // up shards for SwiGLU
  const float* bias;
  const float* bias_up;
  const float* residual;
  float* out;
};

// grid: (ceil(Ns/64), ceil(M/64), tp for COL/ROW_PARTIAL or 1 for ROW_SUM)
template <int KIND>
__global__ void __launch_bounds__(SK_THREADS) simt_gemm_kernel(const SimtArgs a) {
  __shared__ float As[SK_BK][SK_BM + 4];
  __shared__ float Bs[SK_BK][SK_BN + 4];
  __shared__ float Us[KIND == SK_COL_SWIGLU ? SK_BK : 1][SK_BN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * SK_BM, n0 = blockIdx.x * SK_BN;
  const int s = blockIdx.z;
  float acc[4][4] = {}, accu[4][4] = {};

  for (int kk_sh = 0; kk_sh < a.k_shards; ++kk_sh) {
    const int ks = (KIND == SK_ROW_SUM) ? kk_sh : s;
    const float* A = a.A + static_cast<int64_t>(ks) * a.a_shard_stride;
    const float* B = a.B0 + static_cast<int64_t>(ks) * a.Ns * a.Ks;
    const float* U = (KIND == SK_COL_SWIGLU) ? a.B1 + static_cast<int64_t>(ks) * a.Ns * a.Ks : nullptr;
    for (int k0 = 0; k0 < a.Ks; k0 += SK_BK) {
      for (int i = threadIdx.x; i < SK_BK * SK_BM; i += SK_THREADS) {
        const int kk = i % SK_BK, r = i / SK_BK;
        const int gm = m0 + r, gk = k0 + kk;
        As[kk][r] = (gm < a.M && gk < a.Ks) ? A[static_cast<int64_t>(gm) * a.Ks + gk] : 0.0f;
        const int gn = n0 + r;
        const bool okb = gn < a.Ns && gk < a.Ks;
        Bs[kk][r] = okb ? B[static_cast<int64_t>(gn) * a.Ks + gk] : 0.0f;
        if constexpr (KIND == SK_COL_SWIGLU) Us[kk][r] = okb ? U[static_cast<int64_t>(gn) * a.Ks + gk] : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < SK_BK; ++kk) {
        float av[4], bv[4], uv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
        if constexpr (KIND == SK_COL_SWIGLU) {
#pragma unroll
          for (int j = 0; j < 4; ++j) uv[j] = Us[kk][tx * 4 + j];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            if constexpr (KIND == SK_COL_SWIGLU) accu[i][j] = fmaf(av[i], uv[j], accu[i][j]);
          }
      }
      __syncthreads();
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.Ns) continue;
      float v = acc[i][j];
      if constexpr (KIND == SK_COL || KIND == SK_COL_SWIGLU) {
        if (a.bias) v += a.bias[static_cast<int64_t>(s) * a.Ns + n];
        if constexpr (KIND == SK_COL_SWIGLU) {
          float u = accu[i][j];
          if (a.bias_up) u += a.bias_up[static_cast<int64_t>(s) * a.Ns + n];
          v = act_silu(v) * u;
        } else {
          v = apply_act(a.act, v);
        }
        const int64_t off = a.out_concat
                                ? static_cast<int64_t>(m) * a.tp * a.Ns + static_cast<int64_t>(s) * a.Ns + n
                                : (static_cast<int64_t>(s) * a.M + m) * a.Ns + n;
        a.out[off] = v;
      } else if constexpr (KIND == SK_ROW_SUM) {
        if (a.bias) v += a.bias[n];
        if (a.residual) v += a.residual[static_cast<int64_t>(m) * a.Ns + n];
        a.out[static_cast<int64_t>(m) * a.Ns + n] = v;
      } else {
        a.out[(static_cast<int64_t>(s) * a.M + m) * a.Ns + n] = v;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Strided fp32 GEMM for the backward of the column/row pair on fp32 tensors:
//   C_z(m, n) = sum_{q < Q} sum_{k < K} A_{q,z}(m, k) * B_{q,z}(k, n)  (+ add_z(m, n))
// with every operand given by strides, so that the data and weight
// gradients read the forward's tensors and shard layouts as they are
// (A_{q,z}(m, k) = A[q * a_q + z * a_z + m * a_m + k * a_k], likewise B, C).
// Each element is a fixed-order chain of fmaf (q ascending, then k
// ascending), so integer-valued inputs whose partial sums stay below 2^24
// give exact results. `add` has C's strides and may be C itself (each
// element is read, then written, by one thread).
// grid: (ceil(N / 64), ceil(M / 64), Z)
// ---------------------------------------------------------------------------
struct SimtGArgs {
  int M, N, K, Q;
  const float* A;
  int64_t a_m, a_k, a_q, a_z;
  const float* B;
  int64_t b_k, b_n, b_q, b_z;
  float* C;
  int64_t c_m, c_n, c_z;
  const float* add;
};

__global__ void __launch_bounds__(SK_THREADS) simt_gemm_strided_kernel(const SimtGArgs a) {
  __shared__ float As[SK_BK][SK_BM + 4];
  __shared__ float Bs[SK_BK][SK_BN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * SK_BM, n0 = blockIdx.x * SK_BN;
  const int64_t z = blockIdx.z;
  float acc[4][4] = {};
  for (int q = 0; q < a.Q; ++q) {
    const float* A = a.A + q * a.a_q + z * a.a_z;
    const float* B = a.B + q * a.b_q + z * a.b_z;
    for (int k0 = 0; k0 < a.K; k0 += SK_BK) {
      for (int i = threadIdx.x; i < SK_BK * SK_BM; i += SK_THREADS) {
        const int kk = i % SK_BK, r = i / SK_BK;
        const int gk = k0 + kk, gm = m0 + r, gn = n0 + r;
        As[kk][r] = (gm < a.M && gk < a.K) ? A[gm * a.a_m + gk * a.a_k] : 0.0f;
        Bs[kk][r] = (gn < a.N && gk < a.K) ? B[gk * a.b_k + gn * a.b_n] : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < SK_BK; ++kk) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      const int64_t off = z * a.c_z + m * a.c_m + n * a.c_n;
      float v = acc[i][j];
      if (a.add) v += a.add[off];
      a.C[off] = v;
    }
  }
}

}  // namespace tpk
