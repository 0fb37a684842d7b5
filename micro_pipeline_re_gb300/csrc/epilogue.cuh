// GEMM epilogues shared by the tensor-core and the FFMA GEMM kernels.
//   EPI_STORE      C = acc (+bias[n]) (+resid[m,n])          (forward projections)
//   EPI_BIAS_GELU  C = z = acc + bias[n]; C2 = GELU(z)         (FFN first layer)
//   EPI_GELU_BWD   C = acc * GELU'(aux[m,n])                   (FFN input gradient)
//   EPI_ACC_F32    C(fp32) += acc                              (weight gradients,
//                  accumulated across micro-batches in the fp32 gradient buffer)
//   EPI_STORE_F32  C(fp32) = acc                               (logits)
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace gp {

struct EpiArgs {
  void* C;
  int64_t ldc;
  const float* bias;
  const void* resid;
  int64_t ldr;
  void* C2;
  const void* aux;
  int64_t ldaux;
  int M, N;
};

// One output element.
template <typename T, int EPI>
__device__ __forceinline__ void epi_scalar(const EpiArgs& ep, int m, int n, float acc) {
  if (EPI == EPI_ACC_F32) {
    float* c = static_cast<float*>(ep.C) + (int64_t)m * ep.ldc + n;
    *c += acc;
    return;
  }
  if (EPI == EPI_STORE_F32) {
    static_cast<float*>(ep.C)[(int64_t)m * ep.ldc + n] = acc;
    return;
  }
  if (ep.bias) acc += ep.bias[n];
  if (EPI == EPI_STORE) {
    if (ep.resid) acc += Elem<T>::ld(static_cast<const T*>(ep.resid) + (int64_t)m * ep.ldr + n);
    Elem<T>::st(static_cast<T*>(ep.C) + (int64_t)m * ep.ldc + n, acc);
  } else if (EPI == EPI_BIAS_GELU) {
    Elem<T>::st(static_cast<T*>(ep.C) + (int64_t)m * ep.ldc + n, acc);
    Elem<T>::st(static_cast<T*>(ep.C2) + (int64_t)m * ep.ldc + n, gelu_f(acc));
  } else if (EPI == EPI_GELU_BWD) {
    float z = Elem<T>::ld(static_cast<const T*>(ep.aux) + (int64_t)m * ep.ldaux + n);
    Elem<T>::st(static_cast<T*>(ep.C) + (int64_t)m * ep.ldc + n, acc * gelu_grad_f(z));
  }
}

// 32 consecutive columns n0..n0+31 of row m held by one thread (tensor-core
// epilogue).  Vectorised when the whole chunk is in range; leading dimensions
// are multiples of 8 elements and n0 a multiple of 32, so 16-B accesses align.
template <int EPI>
__device__ __forceinline__ void epi_row32_bf16(const EpiArgs& ep, int m, int n0, float* v) {
  const int ncols = min(32, ep.N - n0);
  if (ncols < 32) {
    for (int j = 0; j < ncols; ++j) epi_scalar<__nv_bfloat16, EPI>(ep, m, n0 + j, v[j]);
    return;
  }
  if (EPI == EPI_ACC_F32) {
    float* c = static_cast<float*>(ep.C) + (int64_t)m * ep.ldc + n0;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      float4 x = *reinterpret_cast<float4*>(c + j);
      x.x += v[j]; x.y += v[j + 1]; x.z += v[j + 2]; x.w += v[j + 3];
      *reinterpret_cast<float4*>(c + j) = x;
    }
    return;
  }
  if (EPI == EPI_STORE_F32) {
    float* c = static_cast<float*>(ep.C) + (int64_t)m * ep.ldc + n0;
#pragma unroll
    for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    return;
  }
  if (ep.bias) {
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      float4 b = *reinterpret_cast<const float4*>(ep.bias + n0 + j);
      v[j] += b.x; v[j + 1] += b.y; v[j + 2] += b.z; v[j + 3] += b.w;
    }
  }
  __nv_bfloat16* c = static_cast<__nv_bfloat16*>(ep.C) + (int64_t)m * ep.ldc + n0;
  if (EPI == EPI_STORE) {
    if (ep.resid) {
      const __nv_bfloat16* r = static_cast<const __nv_bfloat16*>(ep.resid) + (int64_t)m * ep.ldr + n0;
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        float t[8];
        load8(r + j, t);
#pragma unroll
        for (int q = 0; q < 8; ++q) v[j + q] += t[q];
      }
    }
#pragma unroll
    for (int j = 0; j < 32; j += 8) store8(c + j, v + j);
  } else if (EPI == EPI_BIAS_GELU) {
    __nv_bfloat16* c2 = static_cast<__nv_bfloat16*>(ep.C2) + (int64_t)m * ep.ldc + n0;
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      store8(c + j, v + j);
      float t[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) t[q] = gelu_f(v[j + q]);
      store8(c2 + j, t);
    }
  } else if (EPI == EPI_GELU_BWD) {
    const __nv_bfloat16* a = static_cast<const __nv_bfloat16*>(ep.aux) + (int64_t)m * ep.ldaux + n0;
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      float z[8];
      load8(a + j, z);
#pragma unroll
      for (int q = 0; q < 8; ++q) v[j + q] *= gelu_grad_f(z[q]);
      store8(c + j, v + j);
    }
  }
}

}  // namespace gp
