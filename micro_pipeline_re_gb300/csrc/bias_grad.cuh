// Bias gradient of a weight-gradient GEMM, shared by the tcgen05 kernels so
// that every path gives the same bits: for C = A B^T accumulated into the fp32
// weight gradient, the bias gradient is dbias[m] += sum_k A(m, k).
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"

namespace gp {

// Rows m0..m0+127: dbias[m] += sum_k A(m, k), by the 8
// epilogue warps (warp w owns rows m0 + 16w .. +15) in a fixed order: each
// lane sums a fixed residue class of k in fp32, then the lanes are folded by
// xor-shuffles.  One thread adds each row's sum; rows >= M are skipped.
template <bool A_K>
__device__ __noinline__ void bias_grad_rows(const __nv_bfloat16* A, int64_t lda, int M, int K, float* dbias, int m0,
                                            int ew, int lane) {
  const int mb = m0 + 16 * ew;
  if (A_K) {
    // row-major rows of K: lane = (row r = lane >> 1, half h = lane & 1); h sums chunks 2j + h of 8
    const int m = mb + (lane >> 1), h = lane & 1;
    float s = 0.f;
    if (m < M) {
      const __nv_bfloat16* row = A + static_cast<int64_t>(m) * lda;
      const int full = K / 8;
      for (int j = h; j < full; j += 2) {
        float v[8];
        load8(row + 8 * j, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += v[e];
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
    const bool vec = mc + 8 <= M;
    for (int k = g; k < K; k += 16) {
      const __nv_bfloat16* p = A + static_cast<int64_t>(k) * lda + mc;
      if (vec) {
        float v[8];
        load8(p, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) s[e] += v[e];
      } else {
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
