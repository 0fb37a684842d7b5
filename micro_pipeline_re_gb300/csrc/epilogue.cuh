// Per-element GEMM epilogues of the FFMA GEMM kernel (the tensor-core kernel
// applies the same operations on 128B-swizzled shared tiles).
//   EPI_STORE      C = acc (+bias[n]) (+resid[m,n])          (forward projections)
//   EPI_BIAS_GELU  C = z = acc + bias[n]; C2 = GELU(z)         (FFN first layer)
//   EPI_GELU_BWD   C = acc * GELU'(aux[m,n])                   (FFN input gradient)
//   EPI_ACC_F32    C(fp32) += acc                              (weight gradients,
//                  accumulated across micro-batches in the fp32 gradient buffer)
//   EPI_STORE_F32  C(fp32) = acc                               (logits)
//   EPI_RESID_F32  C(fp32) = (acc + bias[n]) + resid(fp32)[m,n] (residual adds
//                  that keep the residual stream in fp32)
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
  if (EPI == EPI_RESID_F32) {
    if (ep.resid) acc += static_cast<const float*>(ep.resid)[(int64_t)m * ep.ldr + n];
    static_cast<float*>(ep.C)[(int64_t)m * ep.ldc + n] = acc;
    return;
  }
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

}  // namespace gp
