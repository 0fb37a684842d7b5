// bf16 GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a.
//
// C[m,n] = epilogue( sum_k A(m,k) B(n,k) ) with A and B each K-major or
// MN-major in global memory.  One CTA computes a 128 x BN output tile:
//   warp 0 / lane 0   TMA producer: 128-byte-swizzled tiles of A and B into a
//                     ring of STAGES shared-memory stages (mbarrier complete_tx)
//   warp 1 / lane 0   MMA issuer: tcgen05.mma kind::f16, M=128, N=BN, K=16,
//                     accumulator in tensor memory (BN fp32 columns x 128 lanes),
//                     tcgen05.commit frees each stage and finally signals the
//                     epilogue
//   warps 0..3        epilogue: tcgen05.ld of their 32 TMEM lanes (= 32 rows),
//                     fused bias / residual / GELU / fp32 accumulate, stores.
// Every mbarrier wait is bounded (2 s); a timed-out wait sets the library's
// device error flag and the CTA still releases its tensor memory and waits for
// its own in-flight copies before exiting.
//
// Shared-memory tile layouts (both 128 B swizzle, 1024-B aligned):
//   K-major operand: row r holds k = 0..63 of that row (128 B); 8-row groups
//     are 1024 B apart (stride byte offset 1024).  The k-th 16-wide slice
//     starts 32 B into each row.
//   MN-major operand: 64-wide MN chunks, each [64 k-rows][64 mn] (8 KB);
//     chunks 8192 B apart (leading byte offset), 8-k-row groups 1024 B apart
//     (stride byte offset); the k-th 16-deep slice starts 2048 B further.
#include <cuda.h>

#include "../../include/gpipe.h"
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace gp {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;

template <int BN>
struct TcCfg {
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + STAGES * (A_BYTES + B_BYTES) + BAR_BYTES;
};

template <bool A_K, bool B_K, int BN, int EPI>
__global__ void __launch_bounds__(128, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, EpiArgs ep,
                   int K, int* err) {
  using Cfg = TcCfg<BN>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * Cfg::B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accb = empty + STAGES;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM;
  const int n0 = blockIdx.x * BN;
  const int nk = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0 && lane == 0) {
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1, err, DERR_TMA_WAIT)) break;
      mbar_arrive_expect_tx(&full[s], Cfg::A_BYTES + Cfg::B_BYTES);
      const int k0 = kb * BK;
      uint8_t* a = sA + s * Cfg::A_BYTES;
      uint8_t* b = sB + s * Cfg::B_BYTES;
      if (A_K) {
        tma_load_2d(a, &tmA, k0, m0, &full[s]);
      } else {
        tma_load_2d(a, &tmA, m0, k0, &full[s]);
        tma_load_2d(a + 8192, &tmA, m0 + 64, k0, &full[s]);
      }
      if (B_K) {
        tma_load_2d(b, &tmB, k0, n0, &full[s]);
      } else {
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) tma_load_2d(b + j * 8192, &tmB, n0 + 64 * j, k0, &full[s]);
      }
      issued = kb + 1;
    }
    // No copy may still be landing in shared memory when the CTA exits.
    for (int kb = (issued > STAGES ? issued - STAGES : 0); kb < issued; ++kb)
      mbar_wait_bounded(&full[kb % STAGES], (kb / STAGES) & 1, err, DERR_DRAIN_WAIT);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = mma_idesc_bf16(BM, BN, !A_K, !B_K);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait_bounded(&full[s], ph, err, DERR_MMA_WAIT)) break;
      tc_fence_after();
      const uint32_t a = smem_u32(sA + s * Cfg::A_BYTES);
      const uint32_t b = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint64_t ad = A_K ? sw128_desc(a + kk * 32, 16, 1024) : sw128_desc(a + kk * 2048, 8192, 1024);
        const uint64_t bd = B_K ? sw128_desc(b + kk * 32, 16, 1024) : sw128_desc(b + kk * 2048, 8192, 1024);
        tc_mma_f16(tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      tc_commit(&empty[s]);
    }
    tc_commit(accb);  // fires once every MMA issued above has completed
  }
  __syncwarp();

  // Epilogue: warp w owns TMEM lanes 32w..32w+31, i.e. tile rows 32w + lane.
  const bool ok = mbar_wait_bounded(accb, 0, err, DERR_ACC_WAIT);
  tc_fence_after();
  if (ok) {
    const int row = m0 + warp * 32 + lane;
    const uint32_t tbase = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col0 = n0 + c * 32;
      if (col0 >= ep.N) break;  // uniform across the warp
      uint32_t r[32];
      tmem_ld32(tbase + c * 32, r);
      tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
      if (row < ep.M) epi_row32_bf16<EPI>(ep, row, col0, v);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and dispatch
// ---------------------------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor [outer][inner] with row stride ld elements; box {64, box_outer}.
bool make_tmap(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld, int box_outer) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool A_K, bool B_K, int BN, int EPI>
int set_attr() {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<A_K, B_K, BN, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<BN>::SMEM);
    if (e != cudaSuccess) return set_error(-3, "gemm: smem attribute: %s", cudaGetErrorString(e));
    attr_set = true;
  }
  return 0;
}

template <bool A_K, bool B_K, int BN, int EPI>
int run(const GemmDesc& g, cudaStream_t stream) {
  using Cfg = TcCfg<BN>;
  CUtensorMap ta, tb;
  bool ok = A_K ? make_tmap(&ta, g.A, g.K, g.M, g.lda, BM) : make_tmap(&ta, g.A, g.M, g.K, g.lda, 64);
  ok = ok && (B_K ? make_tmap(&tb, g.B, g.K, g.N, g.ldb, BN) : make_tmap(&tb, g.B, g.N, g.K, g.ldb, 64));
  if (!ok) return set_error(-3, "gemm: cuTensorMapEncodeTiled failed");
  int rc = set_attr<A_K, B_K, BN, EPI>();
  if (rc) return rc;
  auto kern = tc_gemm_kernel<A_K, B_K, BN, EPI>;
  EpiArgs ep{g.C, g.ldc, g.bias, g.resid, g.ldr, g.C2, g.aux, g.ldaux, g.M, g.N};
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM);
  kern<<<grid, 128, Cfg::SMEM, stream>>>(ta, tb, ep, g.K, device_error_ptr());
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(-3, "gemm launch: %s", cudaGetErrorString(e));
  return 0;
}

// Instantiated combinations: the forward projections and logits (K-major A
// and B), input gradients (K-major A, MN-major B) and weight gradients
// (MN-major A and B); a plain store / fp32 accumulate for each, so every
// operand layout can be checked with the simplest epilogue.
int run_epi(const GemmDesc& g, cudaStream_t s) {
  if (g.a_kmajor && g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE: return run<true, true, 128, EPI_STORE>(g, s);
      case EPI_BIAS_GELU: return run<true, true, 128, EPI_BIAS_GELU>(g, s);
      case EPI_STORE_F32: return run<true, true, 128, EPI_STORE_F32>(g, s);
      case EPI_ACC_F32: return run<true, true, 128, EPI_ACC_F32>(g, s);
    }
  } else if (g.a_kmajor && !g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE: return run<true, false, 128, EPI_STORE>(g, s);
      case EPI_GELU_BWD: return run<true, false, 128, EPI_GELU_BWD>(g, s);
      case EPI_ACC_F32: return run<true, false, 128, EPI_ACC_F32>(g, s);
    }
  } else if (!g.a_kmajor && !g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE: return run<false, false, 128, EPI_STORE>(g, s);
      case EPI_ACC_F32: return run<false, false, 128, EPI_ACC_F32>(g, s);
    }
  }
  return set_error(GPIPE_ERR_UNSUPPORTED, "gemm (tensor core): layout a_kmajor=%d b_kmajor=%d with epilogue %d not built",
                   (int)g.a_kmajor, (int)g.b_kmajor, g.epi);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int prepare_gemm_tc() {
  if (!encode_fn()) return set_error(GPIPE_ERR_CUDA, "gemm: cuTensorMapEncodeTiled entry point not found");
  int rc = 0;
  rc = rc ? rc : set_attr<true, true, 128, EPI_STORE>();
  rc = rc ? rc : set_attr<true, true, 128, EPI_BIAS_GELU>();
  rc = rc ? rc : set_attr<true, true, 128, EPI_STORE_F32>();
  rc = rc ? rc : set_attr<true, true, 128, EPI_ACC_F32>();
  rc = rc ? rc : set_attr<true, false, 128, EPI_STORE>();
  rc = rc ? rc : set_attr<true, false, 128, EPI_GELU_BWD>();
  rc = rc ? rc : set_attr<true, false, 128, EPI_ACC_F32>();
  rc = rc ? rc : set_attr<false, false, 128, EPI_STORE>();
  rc = rc ? rc : set_attr<false, false, 128, EPI_ACC_F32>();
  return rc;
}

int launch_gemm_tc(const GemmDesc& g, cudaStream_t stream) {
  if (g.M < 1 || g.N < 1 || g.K < 1) return set_error(GPIPE_ERR_INVALID_ARG, "gemm: M, N, K must be >= 1");
  if (!g.A || !g.B || !g.C) return set_error(GPIPE_ERR_INVALID_ARG, "gemm: NULL operand");
  if ((g.lda % 8) || (g.ldb % 8) || (g.ldc % 8) || !aligned16(g.A) || !aligned16(g.B) || !aligned16(g.C))
    return set_error(GPIPE_ERR_INVALID_ARG, "gemm: leading dimensions must be multiples of 8 and bases 16-B aligned");
  if (g.lda < (g.a_kmajor ? g.K : g.M) || g.ldb < (g.b_kmajor ? g.K : g.N) || g.ldc < g.N)
    return set_error(GPIPE_ERR_INVALID_ARG, "gemm: leading dimension smaller than the matrix");
  if (g.epi == EPI_BIAS_GELU && (!g.C2 || !aligned16(g.C2)))
    return set_error(GPIPE_ERR_INVALID_ARG, "gemm: GELU epilogue needs an aligned C2");
  if (g.epi == EPI_GELU_BWD && (!g.aux || g.ldaux % 8 || !aligned16(g.aux)))
    return set_error(GPIPE_ERR_INVALID_ARG, "gemm: GELU backward needs an aligned aux");
  if (g.resid && (g.ldr % 8 || !aligned16(g.resid)))
    return set_error(GPIPE_ERR_INVALID_ARG, "gemm: residual must be aligned");
  if (g.bias && !aligned16(g.bias)) return set_error(GPIPE_ERR_INVALID_ARG, "gemm: bias must be 16-B aligned");
  return run_epi(g, stream);
}

}  // namespace gp
