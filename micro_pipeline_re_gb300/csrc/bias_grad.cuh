// Bias gradient of a weight-gradient GEMM, shared by the tcgen05 kernels so
// that every path gives the same bits: for C = A B^T accumulated into the fp32
// weight gradient, the bias gradient is dbias[m] += sum_k A(m, k).
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"

namespace gp {

// Rows m0..m0+127: dbias[m] += sum_k A(m, k), by the 8
// epilogue warps (warp w owns rows m0 + 16w .. +15) in a fixed order: each
// lane sums a fixed residue class of k in fp32, in increasing k, then the
// lanes are folded by xor-shuffles.  One thread adds each row's sum; rows >= M
// are skipped.  Loads are issued kU at a time before any of them is added
// (same order of additions), so a lane keeps kU 16-byte loads in flight.
constexpr int kU = 8;

template <bool A_K>
__device__ __noinline__ void bias_grad_rows(const __nv_bfloat16* __restrict__ A, int64_t lda, int M, int K,
                                            float* dbias, int m0, int ew, int lane) {
  const int mb = m0 + 16 * ew;
  if (A_K) {
    // row-major rows of K: lane = (row r = lane >> 1, half h = lane & 1); h sums chunks 2j + h of 8
    const int m = mb + (lane >> 1), h = lane & 1;
    float s = 0.f;
    if (m < M) {
      const __nv_bfloat16* row = A + static_cast<int64_t>(m) * lda;
      const int full = K / 8;
      for (int j0 = h; j0 < full; j0 += 2 * kU) {
        float v[kU][8];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int j = j0 + 2 * u;
          if (j < full) {
            load8(row + 8 * j, v[u]);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[u][e] = 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (j0 + 2 * u < full)
#pragma unroll
            for (int e = 0; e < 8; ++e) s += v[u][e];
      }
      if (h == 0)
        for (int k = 8 * full; k < K; ++k) s += bf2f(row[k]);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    if (h == 0 && m < M) dbias[m] += s;
  } else {
    // rows of A are k: lane = (row class g = lane >> 1, 8-column chunk c = lane & 1)
    const int g = lane >> 1, c = lane & 1;
    const int mc = mb + 8 * c;
    float s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] = 0.f;
    if (mc + 8 <= M) {
      for (int k0 = g; k0 < K; k0 += 16 * kU) {
        float v[kU][8];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int k = k0 + 16 * u;
          if (k < K) {
            load8(A + static_cast<int64_t>(k) * lda + mc, v[u]);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[u][e] = 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (k0 + 16 * u < K)
#pragma unroll
            for (int e = 0; e < 8; ++e) s[e] += v[u][e];
      }
    } else {
      for (int k = g; k < K; k += 16) {
        const __nv_bfloat16* p = A + static_cast<int64_t>(k) * lda + mc;
        for (int e = 0; e < 8; ++e)
          if (mc + e < M) s[e] += bf2f(p[e]);
      }
    }
#pragma unroll
    for (int o = 2; o < 32; o <<= 1)
#pragma unroll
      for (int e = 0; e < 8; ++e) s[e] += __shfl_xor_sync(0xffffffffu, s[e], o);
    if (g == 0)
      for (int e = 0; e < 8; ++e)
        if (mc + e < M) dbias[mc + e] += s[e];
  }
}

}  // namespace gp
