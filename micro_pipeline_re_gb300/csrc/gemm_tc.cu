// bf16 GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a.
//
// C[m,n] = epilogue( sum_k A(m,k) B(n,k) ) with A and B each K-major or
// MN-major in global memory.  One CTA computes a 128 x BN output tile:
//   warp 0 / lane 0   TMA producer: 128-byte-swizzled tiles of A and B into a
//                     ring of STAGES shared-memory stages (mbarrier complete_tx);
//                     first it also loads the epilogue's input tile (residual or
//                     GELU pre-activation) so it lands during the main loop
//   warp 1 / lane 0   MMA issuer: tcgen05.mma kind::f16, M=128, N=BN, K=16,
//                     fp32 accumulator in tensor memory; tcgen05.commit frees
//                     each stage and finally signals the epilogue.  For the
//                     weight-gradient GEMM of the first N tile it also issues
//                     an M=128, N=16 MMA against a tile of ones, which leaves
//                     sum_k A(m,k) (the bias gradient) in TMEM column BN
//   warps 0..3        epilogue: tcgen05.ld of their 32 TMEM lanes (= rows),
//                     fused bias / residual / GELU, written into a 128B-swizzled
//                     shared tile that one thread sends out with TMA stores
//                     (or, for the fp32 gradient, TMA reduce-add, so the
//                     read-modify-write happens in L2 and the SM never waits on
//                     a global read)
// Every mbarrier wait is bounded (2 s); a timed-out wait sets the library's
// device error flag and the CTA still releases its tensor memory and waits for
// its own in-flight copies before exiting.
//
// Shared-memory tile layouts (128 B swizzle, 1024-B aligned):
//   K-major operand: row r holds k = 0..63 of that row (128 B); 8-row groups
//     are 1024 B apart (stride byte offset 1024).  The k-th 16-wide slice
//     starts 32 B into each row.
//   MN-major operand: 64-wide MN chunks, each [64 k-rows][64 mn] (8 KB);
//     chunks 8192 B apart (leading byte offset), 8-k-row groups 1024 B apart
//     (stride byte offset); the k-th 16-deep slice starts 2048 B further.
//   Epilogue tile: boxes of [128 rows][128 B] (64 bf16 or 32 fp32 columns),
//     16 KB each; the 16-B unit u of row r sits at r*128 + ((u ^ (r&7)) * 16).
#include <cuda.h>

#include "../../include/gpipe.h"
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "launch_util.cuh"

namespace gp {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BOX = 16384;  // one epilogue box: 128 rows x 128 B

template <int BN, int EPI>
struct TcCfg {
  static constexpr int STAGES = BN == 64 ? 3 : 4;  // BN=64: two CTAs fit on one SM
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr bool F32_OUT = (EPI == EPI_ACC_F32 || EPI == EPI_STORE_F32 || EPI == EPI_RESID_F32);
  static constexpr int OUT_BOXES = F32_OUT ? BN / 32 : BN / 64;            // boxes of one output tile
  static constexpr int EPI_BYTES = (EPI == EPI_BIAS_GELU ? 2 : 1) * OUT_BOXES * BOX;
  static constexpr int ONES_BYTES = (EPI == EPI_ACC_F32) ? 2048 : 0;
  static constexpr int OFF_B = STAGES * A_BYTES;
  static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_ONES = OFF_EPI + EPI_BYTES;
  static constexpr int OFF_BIAS = OFF_ONES + ONES_BYTES;
  static constexpr int OFF_BAR = OFF_BIAS + BN * 4;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
};

struct TcArgs {
  const float* bias;  // forward epilogues: fp32 [N] or NULL
  float* dbias;       // EPI_ACC_F32: fp32 [M] accumulator of sum_k A(m,k), or NULL
  int M, N, K;
  int has_x;          // the epilogue input tile (residual / GELU pre-activation) is used
  // split-K epilogue (plain global accesses): output, its leading dimension,
  // and the residual / GELU pre-activation matrix (or NULL) with its own
  void* C;
  int64_t ldc;
  const void* xsrc;
  int64_t ldx;
};

__device__ __forceinline__ uint32_t swz(int r, int unit) {
  return static_cast<uint32_t>(r * 128 + ((unit ^ (r & 7)) << 4));
}

constexpr int THREADS = 256;  // 8 warps: producer (w0), MMA issuer (w1), all 8 share the epilogue

// SPLIT: the S = gridDim.z CTAs of a (1,1,S) cluster split K; each keeps its
// fp32 partial tile in shared memory, and after a cluster barrier CTA rank q
// sums rows [q*128/S, (q+1)*128/S) of all S partials in rank order (through
// distributed shared memory), applies the epilogue and stores.  Deterministic,
// no workspace, one launch.
template <bool A_K, bool B_K, int BN, int EPI, bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
                   const __grid_constant__ CUtensorMap tmX, TcArgs args, int* err) {
  using Cfg = TcCfg<BN, EPI>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + Cfg::OFF_B;
  uint8_t* sE = smem + Cfg::OFF_EPI;
  uint8_t* sOnes = smem + Cfg::OFF_ONES;
  float* sBias = reinterpret_cast<float*>(smem + Cfg::OFF_BIAS);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* accb = empty + STAGES;
  uint64_t* epib = accb + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(epib + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM;
  const int n0 = blockIdx.x * BN;
  const int nk_all = (args.K + BK - 1) / BK;
  const int S = SPLIT ? static_cast<int>(gridDim.z) : 1;
  const int kb_begin = SPLIT ? static_cast<int>(blockIdx.z) * nk_all / S : 0;
  const int nk = (SPLIT ? (static_cast<int>(blockIdx.z) + 1) * nk_all / S : nk_all) - kb_begin;
  const bool do_db = (EPI == EPI_ACC_F32) && args.dbias != nullptr && blockIdx.x == 0;
  const uint32_t tcols = do_db ? static_cast<uint32_t>(BN == 64 ? 128 : 256) : static_cast<uint32_t>(BN);

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    mbar_init(epib, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, tcols);
    tmem_relinquish();
  }
  griddep_wait();  // the previous kernel in the stream has completed; global reads from here on
  if (EPI != EPI_ACC_F32 && EPI != EPI_STORE_F32 && EPI != EPI_GELU_BWD) {
    if (threadIdx.x < BN) {
      const int n = n0 + threadIdx.x;
      sBias[threadIdx.x] = (args.bias != nullptr && n < args.N) ? args.bias[n] : 0.f;
    }
  }
  if (do_db && threadIdx.x < 128) {  // 16 rows x 64 bf16 of 1.0
    reinterpret_cast<uint4*>(sOnes)[threadIdx.x] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0 && lane == 0) {
    // Epilogue input tile first: it has the whole main loop to arrive.
    if (args.has_x) {
      mbar_arrive_expect_tx(epib, (BN / 64) * BOX);
      for (int b = 0; b < BN / 64; ++b) tma_load_2d(sE + b * BOX, &tmX, n0 + 64 * b, m0, epib);
    }
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1, err, DERR_TMA_WAIT)) break;
      mbar_arrive_expect_tx(&full[s], Cfg::A_BYTES + Cfg::B_BYTES);
      const int k0 = (kb_begin + kb) * BK;
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
    if (args.has_x) mbar_wait_bounded(epib, 0, err, DERR_DRAIN_WAIT);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = mma_idesc_bf16(BM, BN, !A_K, !B_K);
    constexpr uint32_t idesc_db = mma_idesc_bf16(BM, 16, !A_K, false);
    const uint32_t ones = smem_u32(sOnes);
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
        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
        tc_mma_f16(tmem, ad, bd, idesc, acc);
        if (do_db) tc_mma_f16(tmem + BN, ad, sw128_desc(ones + kk * 32, 16, 1024), idesc_db, acc);
      }
      tc_commit(&empty[s]);
    }
    tc_commit(accb);  // fires once every MMA issued above has completed
  }
  __syncwarp();
  griddep_launch();  // main loop issued: the next kernel may start its prologue

  // ---- epilogue: warp w reads TMEM lanes 32(w%4).. (tile rows 32(w%4) + lane);
  //      warps w and w+4 split the tile's 32-column chunks ----
  const int r = (warp & 3) * 32 + lane;
  if (SPLIT) {
    constexpr int PLD = BN + 4;  // padded fp32 row of the partial tile (in the now idle stage buffers)
    float* P = reinterpret_cast<float*>(sA);
    const bool okp = mbar_wait_bounded(accb, 0, err, DERR_ACC_WAIT);
    tc_fence_after();
    if (okp) {
      const uint32_t tb = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
#pragma unroll 1
      for (int c = warp >> 2; c < BN / 32; c += 2) {
        uint32_t rr[32];
        tmem_ld32(tb + c * 32, rr);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<float4*>(P + r * PLD + c * 32 + 4 * u) =
              make_float4(__uint_as_float(rr[4 * u]), __uint_as_float(rr[4 * u + 1]), __uint_as_float(rr[4 * u + 2]),
                          __uint_as_float(rr[4 * u + 3]));
      }
    }
    tc_fence_before();
    cluster_sync();  // every partial of the cluster is in place
    const int R = BM / S;
    const int rank = static_cast<int>(cluster_ctarank());
    uint32_t peer[8];
    for (int q = 0; q < S; ++q) peer[q] = map_peer(smem_u32(P), static_cast<uint32_t>(q));
    const int groups = R * (BN / 8);
    for (int gi = threadIdx.x; gi < groups; gi += THREADS) {
      const int rr = rank * R + gi / (BN / 8);
      const int cc = (gi % (BN / 8)) * 8;
      const int m = m0 + rr, n = n0 + cc;
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      const uint32_t off = static_cast<uint32_t>((rr * PLD + cc) * 4);
      for (int q = 0; q < S; ++q) {
        const float4 a = ld_peer_f4(peer[q] + off), b = ld_peer_f4(peer[q] + off + 16);
        v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
        v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
      }
      if (m < args.M && n < args.N) {
        if (EPI == EPI_STORE && args.bias) {
          float bb[8];
          load8(args.bias + n, bb);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] += bb[j];
        }
        if (args.xsrc) {  // residual (store) or GELU pre-activation (GELU backward)
          float t[8];
          load8(static_cast<const __nv_bfloat16*>(args.xsrc) + static_cast<int64_t>(m) * args.ldx + n, t);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (EPI == EPI_GELU_BWD) v[j] *= gelu_grad_f(t[j]);
            else v[j] += t[j];
          }
        }
        store8(static_cast<__nv_bfloat16*>(args.C) + static_cast<int64_t>(m) * args.ldc + n, v);
      }
    }
    cluster_sync();  // peers have finished reading this CTA's partial
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, tcols);
    }
    return;
  }
  const bool ok = mbar_wait_bounded(accb, 0, err, DERR_ACC_WAIT);
  tc_fence_after();
  bool ok_x = true;
  if (args.has_x) ok_x = mbar_wait_bounded(epib, 0, err, DERR_ACC_WAIT);
  const uint32_t tbase = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  if (ok && ok_x) {
#pragma unroll 1
    for (int c = warp >> 2; c < BN / 32; c += 2) {
      uint32_t rr[32];
      tmem_ld32(tbase + c * 32, rr);
      tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(rr[j]);
      if (Cfg::F32_OUT) {
        if (EPI == EPI_RESID_F32) {  // + bias + the fp32 residual, read straight from global memory
          const int m = m0 + r, n = n0 + c * 32;  // (acc + bias) + residual
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += sBias[c * 32 + j];
          if (m < args.M) {
            const float* xr = static_cast<const float*>(args.xsrc) + static_cast<int64_t>(m) * args.ldx + n;
            if (n + 32 <= args.N) {
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                float t[8];
                load8(xr + j, t);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[j + e] += t[e];
              }
            } else {
              for (int j = 0; j < 32; ++j)
                if (n + j < args.N) v[j] += xr[j];
            }
          }
        }
        uint8_t* box = sE + c * BOX;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<float4*>(box + swz(r, u)) = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      } else {
        uint8_t* box = sE + (c >> 1) * BOX;
        const int u0 = (c & 1) * 4;
        if (EPI == EPI_STORE || EPI == EPI_BIAS_GELU) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += sBias[c * 32 + j];
        }
        if (args.has_x) {  // residual (store) or GELU pre-activation (GELU backward)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float t[8];
            load8(reinterpret_cast<const __nv_bfloat16*>(box + swz(r, u0 + u)), t);
            if (EPI == EPI_GELU_BWD) {  // two lanes at a time
#pragma unroll
              for (int q = 0; q < 8; q += 2) {
                float g0, g1;
                gelu_grad2(t[q], t[q + 1], g0, g1);
                fmul2(v[8 * u + q], v[8 * u + q + 1], v[8 * u + q], v[8 * u + q + 1], g0, g1);
              }
            } else {
#pragma unroll
              for (int q = 0; q < 8; ++q) v[8 * u + q] += t[q];
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) store8(reinterpret_cast<__nv_bfloat16*>(box + swz(r, u0 + u)), v + 8 * u);
        if (EPI == EPI_BIAS_GELU) {
          uint8_t* box2 = sE + (Cfg::OUT_BOXES + (c >> 1)) * BOX;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float t[8];
#pragma unroll
            for (int q = 0; q < 8; q += 2) gelu2(v[8 * u + q], v[8 * u + q + 1], t[q], t[q + 1]);
            store8(reinterpret_cast<__nv_bfloat16*>(box2 + swz(r, u0 + u)), t);
          }
        }
      }
    }
    if (do_db && warp < 4) {
      uint32_t rr[32];
      tmem_ld32(tbase + BN, rr);
      tmem_ld_wait();
      const int m = m0 + r;
      if (m < args.M) args.dbias[m] += __uint_as_float(rr[0]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && ok && ok_x) {
    constexpr int COLS = Cfg::F32_OUT ? 32 : 64;
    for (int b = 0; b < Cfg::OUT_BOXES; ++b) {
      const int x = n0 + b * COLS;
      if (x >= args.N) break;
      if (EPI == EPI_ACC_F32) tma_reduce_add_2d(&tmC, x, m0, sE + b * BOX);
      else tma_store_2d(&tmC, x, m0, sE + b * BOX);
      if (EPI == EPI_BIAS_GELU) tma_store_2d(&tmC2, x, m0, sE + (Cfg::OUT_BOXES + b) * BOX);
    }
    bulk_commit();
    bulk_wait_read_all();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
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

// 2-D tensor [outer][inner] (row stride ld elements) with a box of
// box_inner x box_outer elements, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, bool f32, int64_t inner, int64_t outer, int64_t ld, int box_inner,
               int box_outer) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  const int es = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool A_K, bool B_K, int BN, int EPI, bool SPLIT = false>
int set_attr() {
  static std::atomic<unsigned long long> done{0};
  return once_per_device(done, [] {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<A_K, B_K, BN, EPI, SPLIT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<BN, EPI>::SMEM);
    return e == cudaSuccess ? GPIPE_OK
                            : set_error(GPIPE_ERR_CUDA, "gemm: smem attribute: %s", cudaGetErrorString(e));
  });
}

template <bool A_K, bool B_K, int BN, int EPI, bool SPLIT = false>
int run(const GemmDesc& g, cudaStream_t stream, int S = 1) {
  using Cfg = TcCfg<BN, EPI>;
  CUtensorMap ta, tb, tc, tc2, tx;
  bool ok = A_K ? make_tmap(&ta, g.A, false, g.K, g.M, g.lda, 64, BM) : make_tmap(&ta, g.A, false, g.M, g.K, g.lda, 64, 64);
  ok = ok && (B_K ? make_tmap(&tb, g.B, false, g.K, g.N, g.ldb, 64, BN)
                  : make_tmap(&tb, g.B, false, g.N, g.K, g.ldb, 64, 64));
  ok = ok && make_tmap(&tc, g.C, Cfg::F32_OUT, g.N, g.M, g.ldc, Cfg::F32_OUT ? 32 : 64, BM);
  tc2 = tc;
  tx = tc;
  if (EPI == EPI_BIAS_GELU) ok = ok && make_tmap(&tc2, g.C2, false, g.N, g.M, g.ldc, 64, BM);
  int has_x = 0;
  const void* xsrc = nullptr;
  int64_t ldx = 0;
  if ((EPI == EPI_STORE || EPI == EPI_RESID_F32) && g.resid) {
    xsrc = g.resid;
    ldx = g.ldr;
  }
  if (EPI == EPI_GELU_BWD) {
    xsrc = g.aux;
    ldx = g.ldaux;
  }
  if (xsrc && !SPLIT && EPI != EPI_RESID_F32) {  // the fp32 residual is read in the epilogue itself
    ok = ok && make_tmap(&tx, xsrc, false, g.N, g.M, ldx, 64, BM);
    has_x = 1;
  }
  if (!ok) return set_error(GPIPE_ERR_CUDA, "gemm: cuTensorMapEncodeTiled failed");
  int rc = set_attr<A_K, B_K, BN, EPI, SPLIT>();
  if (rc) return rc;
  TcArgs args{g.bias, g.dbias, g.M, g.N, g.K, has_x, g.C, g.ldc, xsrc, ldx};
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, SPLIT ? S : 1);
  cudaError_t e;
  if (SPLIT) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = S;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 0;  // heavy: never launched early
    set_priority_attr(attr[2], stream);
    cfg.attrs = attr;
    cfg.numAttrs = 3;
    e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<A_K, B_K, BN, EPI, SPLIT>, ta, tb, tc, tc2, tx, args,
                           device_error_ptr());
  } else {
    (void)launch_k<true>(tc_gemm_kernel<A_K, B_K, BN, EPI, SPLIT>, grid, THREADS, Cfg::SMEM, stream, ta, tb, tc, tc2, tx, args,
                                                                                  device_error_ptr());
    e = cudaGetLastError();
  }
  count_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
  return GPIPE_OK;
}

// Split-K factor for a bf16-output GEMM: only K long enough that every split
// keeps at least 32 k-blocks (so the per-CTA set-up stays small against its
// work), up to 8 (a portable cluster) and never more CTAs than two per SM.
// Split K across S (<= 8) CTAs of a cluster while each split keeps at least
// kMinSplitBlocks k-blocks and the tiles x S stay within two waves, and only
// for GEMMs of at most 64 tiles of 128 x 64: in the concurrent step cluster
// launches wait for co-resident SMs that other lanes hold, so only very long
// K with few tiles (the head's dh = dz E, K = vocab) gains.  (Measured: splits
// of mid-length K (2048) slowed the small LM's step, and splitting the wide
// LM's 128-tile 1024 x 1024 x 8192 GEMMs cost it 16%.)
constexpr int kMinSplitBlocks = 32;
constexpr int64_t kMaxSplitTiles = 64;

int split_factor(const GemmDesc& g, int BN) {
  const int64_t tiles = static_cast<int64_t>((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
  const int nk = (g.K + BK - 1) / BK;
  int S = 1;
  if (tiles > kMaxSplitTiles) return 1;
  while (S < 8 && nk / (S * 2) >= kMinSplitBlocks && tiles * S * 2 <= 2 * static_cast<int64_t>(num_sms())) S *= 2;
  return S;
}

// S: K split across a cluster of S CTAs (1: none), for the bf16-output
// epilogues that have a split variant.
template <int BN>
int run_epi_bn(const GemmDesc& g, cudaStream_t s, int S) {
  if (g.a_kmajor && g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE:
        return S > 1 ? run<true, true, BN, EPI_STORE, true>(g, s, S) : run<true, true, BN, EPI_STORE>(g, s);
      case EPI_BIAS_GELU: return run<true, true, BN, EPI_BIAS_GELU>(g, s);
      case EPI_STORE_F32: return run<true, true, BN, EPI_STORE_F32>(g, s);
      case EPI_ACC_F32: return run<true, true, BN, EPI_ACC_F32>(g, s);
      case EPI_RESID_F32: return run<true, true, BN, EPI_RESID_F32>(g, s);
    }
  } else if (g.a_kmajor && !g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE:
        return S > 1 ? run<true, false, BN, EPI_STORE, true>(g, s, S) : run<true, false, BN, EPI_STORE>(g, s);
      case EPI_GELU_BWD:
        return S > 1 ? run<true, false, BN, EPI_GELU_BWD, true>(g, s, S) : run<true, false, BN, EPI_GELU_BWD>(g, s);
      case EPI_ACC_F32: return run<true, false, BN, EPI_ACC_F32>(g, s);
    }
  } else if (!g.a_kmajor && !g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE: return run<false, false, BN, EPI_STORE>(g, s);
      case EPI_ACC_F32: return run<false, false, BN, EPI_ACC_F32>(g, s);
    }
  }
  return set_error(GPIPE_ERR_UNSUPPORTED,
                   "gemm (tensor core): layout a_kmajor=%d b_kmajor=%d with epilogue %d not built",
                   (int)g.a_kmajor, (int)g.b_kmajor, g.epi);
}

// Instantiated combinations: the forward projections and logits (K-major A
// and B), input gradients (K-major A, MN-major B) and weight gradients
// (MN-major A and B); a plain store / fp32 accumulate for each, so every
// operand layout can be checked with the simplest epilogue.  Tile width:
// 128 columns when that already gives at least one CTA per SM, else 64
// (twice the CTAs, each with half the operand traffic and epilogue work).
int run_epi(const GemmDesc& g, cudaStream_t s) {
  // More tiles than this GEMM's share of the machine (at 128 x 256 / 128 x 128
  // tiles): the persistent kernel, one CTA per SM of the share, overlapping
  // each tile's epilogue with the next tile's MMAs.  Otherwise one tile per
  // CTA, 128 columns when that gives at least one CTA per SM of the share,
  // else 64 (twice the CTAs, each with half the operand traffic and epilogue).
  // The split-K choice depends on the shape alone (never on the SM share), so
  // that a GEMM sums in the same order whatever the schedule around it.
  const bool has_split = g.a_kmajor && (g.epi == EPI_STORE || (!g.b_kmajor && g.epi == EPI_GELU_BWD));
  const int S = has_split ? split_factor(g, 64) : 1;
  if (S > 1) return run_epi_bn<64>(g, s, S);
  const int budget = g.sm_budget > 0 ? g.sm_budget : num_sms();
  if (wide_bias_grad_gemm(g)) {
    // 256-wide tiles leave no tensor memory for the ones-MMA, and summing A
    // inside the GEMM's epilogue cost it up to 40%: the GEMM runs without the
    // bias gradient and one reduction kernel adds it (shape-only choice, so
    // every schedule sums it the same way)
    GemmDesc w = g;
    w.dbias = nullptr;
    const int rc = launch_gemm_persistent(w, s, budget);
    return rc ? rc : launch_dbias(g.a_kmajor, g.M, g.K, g.A, g.lda, g.dbias, s);
  }
  if (persistent_tiles(g) > budget) return launch_gemm_persistent(g, s, budget);
  const int64_t tiles128 = static_cast<int64_t>((g.M + BM - 1) / BM) * ((g.N + 127) / 128);
  if (tiles128 >= budget) return run_epi_bn<128>(g, s, 1);
  // A long mainloop (K >= 2048) repays the wider tile even on as few as half
  // the share's SMs: 128-wide products read 128 B of operands per 64 MMA
  // clocks, 64-wide ones 96 B per 32 (above what shared memory feeds an SM),
  // and two 64-wide CTAs on one SM share its tensor core anyway.
  if (g.K >= 2048 && 2 * tiles128 >= budget) return run_epi_bn<128>(g, s, 1);
  return run_epi_bn<64>(g, s, 1);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

template <int BN>
int prepare_bn() {
  int rc = GPIPE_OK;
  rc = rc ? rc : set_attr<true, true, BN, EPI_STORE>();
  rc = rc ? rc : set_attr<true, true, BN, EPI_BIAS_GELU>();
  rc = rc ? rc : set_attr<true, true, BN, EPI_STORE_F32>();
  rc = rc ? rc : set_attr<true, true, BN, EPI_ACC_F32>();
  rc = rc ? rc : set_attr<true, true, BN, EPI_RESID_F32>();
  rc = rc ? rc : set_attr<true, false, BN, EPI_STORE>();
  rc = rc ? rc : set_attr<true, false, BN, EPI_GELU_BWD>();
  rc = rc ? rc : set_attr<true, false, BN, EPI_ACC_F32>();
  rc = rc ? rc : set_attr<false, false, BN, EPI_STORE>();
  rc = rc ? rc : set_attr<false, false, BN, EPI_ACC_F32>();
  rc = rc ? rc : set_attr<true, true, BN, EPI_STORE, true>();
  rc = rc ? rc : set_attr<true, false, BN, EPI_STORE, true>();
  rc = rc ? rc : set_attr<true, false, BN, EPI_GELU_BWD, true>();
  return rc;
}

int prepare_gemm_tc() {
  if (!encode_fn()) return set_error(GPIPE_ERR_CUDA, "gemm: cuTensorMapEncodeTiled entry point not found");
  int rc = prepare_bn<128>();
  rc = rc ? rc : prepare_bn<64>();
  return rc ? rc : prepare_gemm_persistent();
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
  if (g.epi == EPI_GELU_BWD && (!g.aux || g.ldaux % 8 || g.ldaux < g.N || !aligned16(g.aux)))
    return set_error(GPIPE_ERR_INVALID_ARG, "gemm: GELU backward needs an aligned aux");
  if (g.resid && (g.ldr % 8 || g.ldr < g.N || !aligned16(g.resid)))
    return set_error(GPIPE_ERR_INVALID_ARG, "gemm: residual must be aligned");
  if (g.epi == EPI_RESID_F32 && (!g.resid || !g.a_kmajor || !g.b_kmajor))
    return set_error(GPIPE_ERR_INVALID_ARG, "gemm: the fp32 residual epilogue needs a residual and K-major operands");
  return run_epi(g, stream);
}

}  // namespace gp
