// FFMA GEMM (fp32 accumulation) for the fp32 configuration, with the same
// operand layouts and epilogues as the tensor-core kernel.  fp32 tensor-core
// math (TF32) would miss an fp32-level tolerance, so the fp32 path stays on
// the FMA pipes.  Each output sums over k in ascending order, so results are
// bit-reproducible.
//
// Tile 64 x 64, k-step 16, 256 threads, 4 x 4 outputs per thread.
#include "../../include/gpipe.h"
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "launch_util.cuh"

namespace gp {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <typename T, int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const T* __restrict__ A, int64_t lda, int a_k,
                                                        const T* __restrict__ B, int64_t ldb, int b_k, int M, int N,
                                                        int K, EpiArgs ep, float* __restrict__ dbias) {
  griddep_wait();
  griddep_launch();
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  float acc[4][4] = {};
  float rowsum[4] = {0.f, 0.f, 0.f, 0.f};  // sum_k A(m,k) for the bias gradient (first N tile)
  const bool do_db = dbias != nullptr && blockIdx.x == 0 && tx == 0;
  for (int k0 = 0; k0 < K; k0 += TK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * 256;
      // K-major: consecutive threads walk k (contiguous); MN-major: walk m/n.
      int mm, kk;
      if (a_k) { kk = idx % TK; mm = idx / TK; } else { mm = idx % TM; kk = idx / TM; }
      int m = m0 + mm, k = k0 + kk;
      float va = 0.f;
      if (m < M && k < K) va = Elem<T>::ld(A + (a_k ? (int64_t)m * lda + k : (int64_t)k * lda + m));
      As[kk][mm] = va;
      int nn;
      if (b_k) { kk = idx % TK; nn = idx / TK; } else { nn = idx % TN; kk = idx / TN; }
      int n = n0 + nn;
      k = k0 + kk;
      float vb = 0.f;
      if (n < N && k < K) vb = Elem<T>::ld(B + (b_k ? (int64_t)n * ldb + k : (int64_t)k * ldb + n));
      Bs[kk][nn] = vb;
    }
    __syncthreads();
    if (do_db) {
#pragma unroll
      for (int kk = 0; kk < TK; ++kk)
#pragma unroll
        for (int i = 0; i < 4; ++i) rowsum[i] += As[kk][ty * 4 + i];
    }
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  if (do_db) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (m0 + ty * 4 + i < M) dbias[m0 + ty * 4 + i] += rowsum[i];
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) epi_scalar<T, EPI>(ep, m, n, acc[i][j]);
    }
  }
}

template <typename T>
int run_simt(const GemmDesc& g, cudaStream_t s) {
  EpiArgs ep{g.C, g.ldc, g.bias, g.resid, g.ldr, g.C2, g.aux, g.ldaux, g.M, g.N};
  dim3 grid((g.N + TN - 1) / TN, (g.M + TM - 1) / TM);
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B);
  int ak = g.a_kmajor ? 1 : 0, bk = g.b_kmajor ? 1 : 0;
  float* db = g.epi == EPI_ACC_F32 ? g.dbias : nullptr;
  switch (g.epi) {
    case EPI_STORE: (void)launch_k(simt_gemm_kernel<T, EPI_STORE>, grid, 256, 0, s, A, g.lda, ak, B, g.ldb, bk, g.M, g.N, g.K, ep, db); break;
    case EPI_BIAS_GELU: (void)launch_k(simt_gemm_kernel<T, EPI_BIAS_GELU>, grid, 256, 0, s, A, g.lda, ak, B, g.ldb, bk, g.M, g.N, g.K, ep, db); break;
    case EPI_GELU_BWD: (void)launch_k(simt_gemm_kernel<T, EPI_GELU_BWD>, grid, 256, 0, s, A, g.lda, ak, B, g.ldb, bk, g.M, g.N, g.K, ep, db); break;
    case EPI_ACC_F32: (void)launch_k(simt_gemm_kernel<T, EPI_ACC_F32>, grid, 256, 0, s, A, g.lda, ak, B, g.ldb, bk, g.M, g.N, g.K, ep, db); break;
    case EPI_STORE_F32: (void)launch_k(simt_gemm_kernel<T, EPI_STORE_F32>, grid, 256, 0, s, A, g.lda, ak, B, g.ldb, bk, g.M, g.N, g.K, ep, db); break;
    case EPI_RESID_F32: (void)launch_k(simt_gemm_kernel<T, EPI_RESID_F32>, grid, 256, 0, s, A, g.lda, ak, B, g.ldb, bk, g.M, g.N, g.K, ep, db); break;
    default: return set_error(GPIPE_ERR_INVALID_ARG, "gemm: unknown epilogue %d", g.epi);
  }
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "gemm (simt) launch: %s", cudaGetErrorString(e));
  return GPIPE_OK;
}

}  // namespace

int launch_gemm_simt(const GemmDesc& g, cudaStream_t s) {
  if (g.M < 1 || g.N < 1 || g.K < 1) return set_error(GPIPE_ERR_INVALID_ARG, "gemm: M, N, K must be >= 1");
  if (!g.A || !g.B || !g.C) return set_error(GPIPE_ERR_INVALID_ARG, "gemm: NULL operand");
  if (g.epi == EPI_BIAS_GELU && !g.C2) return set_error(GPIPE_ERR_INVALID_ARG, "gemm: GELU epilogue needs C2");
  if (g.epi == EPI_GELU_BWD && !g.aux) return set_error(GPIPE_ERR_INVALID_ARG, "gemm: GELU backward needs aux");
  if (g.dtype == DT_F32) return run_simt<float>(g, s);
  return run_simt<__nv_bfloat16>(g, s);
}

int launch_gemm(const GemmDesc& g, cudaStream_t s) {
  if (g.dtype == DT_F32) return launch_gemm_simt(g, s);
  if (g.dtype == DT_BF16) return launch_gemm_tc(g, s);
  return set_error(GPIPE_ERR_INVALID_ARG, "gemm: unknown dtype %d", g.dtype);
}

}  // namespace gp
