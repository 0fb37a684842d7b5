// Causal multi-head attention on the 5th-generation tensor cores (tcgen05),
// head width 64, bf16 operands, fp32 softmax.  Scale 1/sqrt(64) = 0.125;
// query i sees keys j <= i.
//
// Every matrix product runs as tcgen05.mma kind::f16 (bf16 in, fp32 in tensor
// memory), issued by one thread; Q, K, V and dO tiles arrive by TMA with the
// 128-byte swizzle (no multicast); the softmax-side tiles (P, dS) are written
// by the threads into shared memory in the same swizzled layout and fed back
// to the tensor cores.  Thread r of the CTA's 128 owns row r of every
// accumulator (tensor-memory lane r): no cross-thread reductions.
//
// Forward: a CTA per (128-query block, head, sequence).  For each 128-key
// block: S = Q K^T into TMEM; the threads read their row of S, update the
// running maximum (log2 domain), rescale their row of O in TMEM when it
// grows, write P = exp2(S - m) as bf16 and add its row sum; then
// O += P V.  Saves the natural-log log-sum-exp per (row, head).
//
// Backward, without atomics (bit-reproducible): D = rowsum(dO o O) for every
// (row, head) by a small kernel, then one launch of two CTA kinds:
//   dQ CTA    per (128-query block, head, sequence): for every visible
//             64-key block S = Q K^T, dP = dO V^T, P = exp2(S - LSE),
//             dS = P o (dP - D), dQ += dS K.
//   dK/dV CTA per (128-key block, head, sequence): for every 64-query block
//             that sees it, S^T = K Q^T, dP^T = V dO^T, P^T, dS^T (with the
//             same D), dV += P^T dO, dK += dS^T Q.
//
// Shared-memory tiles (1024-B aligned, 128-B rows, 16-B unit u of row r at
// r*128 + ((u ^ (r&7)) * 16)):
//   as a K-major operand (rows = M or N, 64 head columns or 64 keys per row):
//     the 16-wide k slice kk starts 32*kk bytes into each row; 8-row groups
//     are 1024 B apart;
//   as an MN-major operand (rows = K, 64 head columns = N per row): the
//     16-deep k slice kk starts 2048*kk bytes further.
// Every mbarrier wait is bounded (2 s); a wait that gives up sets the
// library's device error word, the CTA leaves its loop at the next barrier
// (the decision is made uniform with __syncthreads_and), waits (bounded) for
// its own copies and products in flight, and frees its tensor memory.
#include <cuda.h>

#include <atomic>

#include "../../include/gpipe.h"
#include "common.cuh"
#include "kernels.h"
#include "launch_util.cuh"

namespace gp {
namespace {

constexpr int HD = 64;                                      // head width
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;  // scale * log2(e)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int T128 = 128 * 128;  // bytes of a 128-row tile (128 B per row)
constexpr int T64 = 64 * 128;    // bytes of a 64-row tile

__device__ __forceinline__ uint32_t swz(int r, int u) { return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4)); }
// K-major operand tile, 16-wide k slice kk (0..3)
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int kk) { return sw128_desc(tile + kk * 32, 16, 1024); }
// MN-major operand tile (64 wide), 16-deep k slice kk
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int kk) { return sw128_desc(tile + kk * 2048, 8192, 1024); }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Load 32 fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void ld_row32(uint32_t taddr, float* v) {
  uint32_t u[32];
  tmem_ld32(taddr, u);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
}

// Load 32 * N fp32 columns of this thread's lane from the column addresses
// a[0..N-1]: every load is issued before the one wait, so their latencies
// overlap (a TMEM load takes a few hundred cycles to return).
template <int N>
__device__ __forceinline__ void ld_rows(const uint32_t* a, float* v) {
  uint32_t u[32 * N];
#pragma unroll
  for (int c = 0; c < N; ++c) tmem_ld32(a[c], u + 32 * c);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32 * N; ++i) v[i] = __uint_as_float(u[i]);
}


// Write 32 values of row r as bf16 into a swizzled tile at units u0..u0+3.
__device__ __forceinline__ void st_row32_bf16(uint8_t* tile, int r, int u0, const float* v) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * u + 0], v[8 * u + 1]);
    w.y = pack_bf16x2(v[8 * u + 2], v[8 * u + 3]);
    w.z = pack_bf16x2(v[8 * u + 4], v[8 * u + 5]);
    w.w = pack_bf16x2(v[8 * u + 6], v[8 * u + 7]);
    *reinterpret_cast<uint4*>(tile + swz(r, u0 + u)) = w;
  }
}

// Store 64 fp32 TMEM columns of this thread's lane, times scale, as bf16 to
// dst when `valid`.  Every thread of the warp calls it (the TMEM loads are
// warp-collective); only the stores depend on `valid`.
__device__ __forceinline__ void store_row64(uint32_t taddr, __nv_bfloat16* dst, float scale, bool valid) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float v[32];
    ld_row32(taddr + 32 * h, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= scale;
    if (valid) {
#pragma unroll
      for (int u = 0; u < 4; ++u) store8(dst + 32 * h + 8 * u, v + 8 * u);
    }
  }
}

// rowsum(dO o O) of one 64-wide head row, in a fixed order (shared by the dQ
// and dK/dV CTAs, so both see the same bits).
__device__ __forceinline__ float row_dot64(const __nv_bfloat16* o, const __nv_bfloat16* d) {
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < HD; c += 8) {
    float ov[8], dv[8];
    load8(o + c, ov);
    load8(d + c, dv);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = fmaf(ov[j], dv[j], acc);
  }
  return acc;
}

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
// Warps 0-3 (128 threads) own the rows; warp 4's lane 0 issues every TMA copy
// and every MMA, so that waiting on a copy never stalls the softmax.  Per key
// block j, hand-offs through mbarriers:
//   issuer:  S_{j+1} = Q K_{j+1}^T as soon as the rows have read S_j out of
//            TMEM -> commit bs;  K_{j+2} into S_j's K buffer;
//            O += P_j V_j (once the rows wrote P_j and rescaled O, and
//            O += P_{j-1} V_{j-1} is done) -> commit bo;  V_{j+1}.
//   rows:    wait bs; read S_j; arrive bsc (S consumed); the running max;
//            wait bo (the previous O product, which reads P and writes O);
//            rescale O; write P_j; arrive bp.
// So S_{j+1} computes while the rows work on block j.
constexpr int FWD_THREADS = 160;
// Two CTAs of five warps put three warps on some of an SM's four sub-partitions,
// each of which holds a quarter of the register file (16384): at most 170
// registers a thread (168 after the allocation granularity) keep two CTAs per SM.
constexpr int ATTN_MAXNREG = 168;
// Q, K x2, V x2, P (2 sub-tiles), barriers.  No slack for aligning the base:
// with no static shared memory the dynamic window starts 1024-byte aligned
// (checked at run time), and without the slack two CTAs fit on an SM.
constexpr int FWD_SMEM = 7 * T128 + 128;

// Bounded wait that gives up at once after any earlier give-up in the CTA.
__device__ __forceinline__ bool await(uint64_t* bar, uint32_t parity, int* err, int code, volatile int* abort) {
  if (*abort) return false;
  if (mbar_wait_bounded(bar, parity, err, code)) return true;
  *abort = 1;
  return false;
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __maxnreg__(ATTN_MAXNREG) attn_fwd_kernel(const __grid_constant__ CUtensorMap tq,
                                                               __nv_bfloat16* __restrict__ out,
                                                               float* __restrict__ lse, int seq, int heads, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (reinterpret_cast<uintptr_t>(smem_raw) & 1023u) {  // the tiles' swizzle needs 1024-byte alignment
    if (threadIdx.x == 0) atomicExch(err, DERR_ALIGN);
    return;
  }
  uint8_t* sm = smem_raw;
  uint8_t* sQ = sm;
  uint8_t* sK = sm + T128;      // two buffers
  uint8_t* sV = sm + 3 * T128;  // two buffers
  uint8_t* sP = sm + 5 * T128;  // keys 0..63 | keys 64..127
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 7 * T128);
  uint64_t *bq = bar, *bk = bar + 1, *bv = bar + 3, *bs = bar + 5, *bsc = bar + 6, *bp = bar + 7, *bo = bar + 8,
           *bfin = bar + 9;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 10);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

  const int r = threadIdx.x, warp = r >> 5;
  const int nqb = (seq + 127) / 128;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x);  // the longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int D = heads * HD;
  const int row0 = b * seq;  // the sequence's first row
  const int q0 = qb * 128;
  const int nkb = qb + 1;    // key blocks 0..qb (the last one holds the diagonal)
  const int qi = q0 + r;     // the query of row thread r (r < 128)

  if (r == 0) {
    prefetch_tmap(&tq);
    for (int i = 0; i < 6; ++i) mbar_init(&bar[i], 1);
    mbar_init(bsc, 128);
    mbar_init(bp, 128);
    mbar_init(bo, 1);
    mbar_init(bfin, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem, tO = tmem + 128;

  if (warp == 4) {
    if (r == 128) {  // ---- issuer ----
      constexpr uint32_t idS = mma_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idO = mma_idesc_bf16(128, 64, false, true);
      int nk[2] = {0, 0}, nv[2] = {0, 0};
      mbar_arrive_expect_tx(bq, T128);
      tma_load_2d(sQ, &tq, h * HD, row0 + q0, bq);
      for (int j = 0; j < 2 && j < nkb; ++j) {
        mbar_arrive_expect_tx(&bk[j], T128);
        tma_load_2d(sK + j * T128, &tq, D + h * HD, row0 + j * 128, &bk[j]);
        ++nk[j];
        mbar_arrive_expect_tx(&bv[j], T128);
        tma_load_2d(sV + j * T128, &tq, 2 * D + h * HD, row0 + j * 128, &bv[j]);
        ++nv[j];
      }
      auto issue_s = [&](int jj) {  // S_jj = Q K_jj^T into TMEM (K_jj loaded, S_{jj-1} read out)
        const uint32_t q = smem_u32(sQ), k = smem_u32(sK + (jj & 1) * T128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tS, kdesc(q, kk), kdesc(k, kk), idS, kk ? 1u : 0u);
        tc_commit(bs);
      };
      bool go = await(bq, 0, err, DERR_MMA_WAIT, abort) && await(&bk[0], 0, err, DERR_MMA_WAIT, abort);
      if (go) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; j < nkb && go; ++j) {
        const int kb = j & 1;
        if (j + 1 < nkb) {  // S_{j+1} as soon as the rows have read S_j: it computes during block j's softmax
          if (!await(&bk[(j + 1) & 1], ((j + 1) >> 1) & 1, err, DERR_MMA_WAIT, abort)) break;
          if (!await(bsc, j & 1, err, DERR_MMA_WAIT, abort)) break;
          tc_fence_after();
          issue_s(j + 1);
          if (j + 2 < nkb) {  // K buffer of block j: S_j is done
            mbar_arrive_expect_tx(&bk[kb], T128);
            tma_load_2d(sK + kb * T128, &tq, D + h * HD, row0 + (j + 2) * 128, &bk[kb]);
            ++nk[kb];
          }
        }
        if (!await(bp, j & 1, err, DERR_MMA_WAIT, abort)) break;                 // P_j written, O rescaled
        if (j > 0 && !await(bo, (j - 1) & 1, err, DERR_MMA_WAIT, abort)) break;  // O += P_{j-1} V_{j-1} done
        if (j >= 1 && j + 1 < nkb) {  // V buffer of block j-1 is free
          const int nb = (j + 1) & 1;
          mbar_arrive_expect_tx(&bv[nb], T128);
          tma_load_2d(sV + nb * T128, &tq, 2 * D + h * HD, row0 + (j + 1) * 128, &bv[nb]);
          ++nv[nb];
        }
        if (!await(&bv[kb], (j >> 1) & 1, err, DERR_MMA_WAIT, abort)) break;
        tc_fence_after();
        {
          const uint32_t p = smem_u32(sP), v = smem_u32(sV + kb * T128);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_f16(tO, kdesc(p + (kk >> 2) * T128, kk & 3), mndesc(v, kk), idO, (j | kk) ? 1u : 0u);
          tc_commit(bo);
        }
      }
      // no copy may still be landing, and no product still running, when the CTA exits
      tc_commit(bfin);
      mbar_wait_bounded(bfin, 0, err, DERR_DRAIN_WAIT);
      for (int bb = 0; bb < 2; ++bb) {
        if (nk[bb]) mbar_wait_bounded(&bk[bb], (nk[bb] - 1) & 1, err, DERR_DRAIN_WAIT);
        if (nv[bb]) mbar_wait_bounded(&bv[bb], (nv[bb] - 1) & 1, err, DERR_DRAIN_WAIT);
      }
      mbar_wait_bounded(bq, 0, err, DERR_DRAIN_WAIT);
    }
  } else {  // ---- rows ----
    const uint32_t lane = static_cast<uint32_t>(warp * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb && ok; ++j) {
      ok = __all_sync(0xffffffffu, await(bs, j & 1, err, DERR_ACC_WAIT, abort));
      if (!ok) break;
      tc_fence_after();
      const bool diag = j == qb;
      // this row of S, all 128 columns in one round trip
      float sv[128];
      {
        const uint32_t a[4] = {tS + lane, tS + lane + 32, tS + lane + 64, tS + lane + 96};
        ld_rows<4>(a, sv);
      }
      tc_fence_before();
      mbar_arrive1(bsc);  // S may be overwritten by the next block's product
      if (diag) {         // the causal mask: only the block on the diagonal has hidden keys
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (j * 128 + i > qi) sv[i] = -INFINITY;
      }
      // the row maximum of the raw scores (scaling by a positive constant keeps
      // it the maximum) over 8 independent partial maxima
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; i += 2) mx8[(i >> 1) & 7] = fmax3(mx8[(i >> 1) & 7], sv[i], sv[i + 1]);
      const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      const float mn = fmaxf(m, mx * kScaleLog2);  // the running maximum, log2 domain
      const float alpha = ex2_approx(m - mn);       // 0 for the first block
      m = mn;
      if (j > 0) {  // the previous O product reads P and writes O
        ok = __all_sync(0xffffffffu, await(bo, (j - 1) & 1, err, DERR_ACC_WAIT, abort));
        if (!ok) break;
        tc_fence_after();
      }
      // P = exp2(s * scale log2(e) - m) as bf16 into shared memory, and its row
      // sum (8 partial sums, added pairwise at the end)
      float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float* pc = sv + 32 * c;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          ffma2(pc[i], pc[i + 1], pc[i], pc[i + 1], kScaleLog2, kScaleLog2, -m, -m);
          pc[i] = ex2_approx(pc[i]);
          pc[i + 1] = ex2_approx(pc[i + 1]);
          const int e = (i >> 1) & 3;
          fadd2(rs8[2 * e], rs8[2 * e + 1], rs8[2 * e], rs8[2 * e + 1], pc[i], pc[i + 1]);
        }
        st_row32_bf16(sP + (c >> 1) * T128, r, (c & 1) * 4, pc);
      }
      const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
      // then O *= alpha, with S's registers free again
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // warp-uniform: tcgen05 loads/stores are per warp
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t u[32];
          tmem_ld32(tO + lane + 32 * c, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float a0, a1;
            fmul2(a0, a1, __uint_as_float(u[i]), __uint_as_float(u[i + 1]), alpha, alpha);
            u[i] = __float_as_uint(a0);
            u[i + 1] = __float_as_uint(a1);
          }
          tmem_st32(tO + lane + 32 * c, u);
        }
        tmem_st_wait();
      }
      l = l * alpha + rs;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive1(bp);
    }
    if (ok) ok = __all_sync(0xffffffffu, await(bo, (nkb - 1) & 1, err, DERR_ACC_WAIT, abort));
    tc_fence_after();
    if (ok) {
      // rows past the sequence end (a last block of 64) are computed, not stored
      const int64_t row = static_cast<int64_t>(row0) + qi;
      store_row64(tO + lane, out + row * D + h * HD, 1.0f / l, qi < seq);
      if (qi < seq) lse[row * heads + h] = (m + log2f(l)) * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  griddep_launch();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------
// Backward
// ---------------------------------------------------------------------------
// D = rowsum(dO o O) for every (row, head), once, before the backward kernel
// (stream order): both kinds of backward CTA read the same values.
__global__ void __launch_bounds__(256) attn_dvec_kernel(const __nv_bfloat16* __restrict__ out,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ dvec, int64_t n, int heads) {
  griddep_wait();
  griddep_launch();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // (row, head) = (i / heads, i % heads)
  if (i >= n) return;
  const int64_t off = i * HD;  // row * heads * 64 + head * 64
  dvec[i] = row_dot64(out + off, dout + off);
}

// dQ CTA: Q, dO (128 rows), K and V blocks of 64 keys (two buffers each), dS
// (128 x 64).  dK/dV CTA: K, V (128 rows), Q and dO blocks of 64 queries (two
// buffers each), P^T and dS^T (128 x 64), LSE and D of two query blocks.
// Both: warps 0-3 the rows, warp 4's lane 0 the issuer of every copy and
// product, hand-offs through mbarriers as in the forward:
//   issuer:  the products S, dP of block t+1 as soon as the rows have read
//            block t's out of TMEM -> commit bs;  the gradient product of
//            block t (once the rows wrote its dS, or P^T and dS^T) -> commit
//            bo;  block t+2's tiles into block t's buffers (after bo(t)).
//   rows:    wait bs; read S, dP; arrive bsc; the elementwise gradient; wait
//            bo(t-1) (the previous gradient product reads the same shared
//            tile); write it; arrive bp.
constexpr int BWD_THREADS = 160;
constexpr int BWD_TILES = 4 * T128 + 4 * T64;  // the larger of the two kinds' tiles (dK/dV: 96 KB)
constexpr int BWD_LD = BWD_TILES;               // dK/dV: LSE and D of two query blocks (1 KB)
constexpr int BWD_BAR = BWD_LD + 4 * 64 * 4;
constexpr int BWD_SMEM = 1024 + BWD_BAR + 128;
__device__ void attn_bwd_dq(const CUtensorMap* tq64, const CUtensorMap* tq128, const CUtensorMap* td128,
                            const float* __restrict__ lse, const float* __restrict__ dvec,
                            __nv_bfloat16* __restrict__ dqkv, int seq, int heads, int b, int* err, uint8_t* sm) {
  uint8_t* sQ = sm;
  uint8_t* sdO = sm + T128;
  uint8_t* sK = sm + 2 * T128;        // two 64-row buffers
  uint8_t* sV = sK + 2 * T64;         // two 64-row buffers
  uint8_t* sdS = sV + 2 * T64;        // 128 rows x 64 keys (ends at 80 KB)
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + BWD_BAR);
  uint64_t *bq = bar, *bkv = bar + 1, *bs = bar + 3, *bsc = bar + 4, *bp = bar + 5, *bo = bar + 6, *bfin = bar + 7;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

  const int r = threadIdx.x, warp = r >> 5;
  const int nqb = (seq + 127) / 128;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x);
  const int h = blockIdx.y;
  const int D = heads * HD;
  const int64_t ld = 3 * static_cast<int64_t>(D);
  const int row0 = b * seq;
  const int q0 = qb * 128;
  const int qi = q0 + r;
  const int nkb = (min(q0 + 127, seq - 1)) / 64 + 1;  // 64-key blocks that any row of the block sees

  if (r == 0) {
    prefetch_tmap(tq64);
    prefetch_tmap(tq128);
    prefetch_tmap(td128);
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    mbar_init(bsc, 128);
    mbar_init(bp, 128);
    mbar_init(bo, 1);
    mbar_init(bfin, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem, tP = tmem + 64, tQ = tmem + 128;

  if (warp == 4) {
    if (r == 128) {  // ---- issuer ----
      constexpr uint32_t idSP = mma_idesc_bf16(128, 64, false, false);
      constexpr uint32_t idQ = mma_idesc_bf16(128, 64, false, true);
      int nkv[2] = {0, 0};
      mbar_arrive_expect_tx(bq, 2 * T128);
      tma_load_2d(sQ, tq128, h * HD, row0 + q0, bq);
      tma_load_2d(sdO, td128, h * HD, row0 + q0, bq);
      for (int j = 0; j < 2 && j < nkb; ++j) {
        mbar_arrive_expect_tx(&bkv[j], 2 * T64);
        tma_load_2d(sK + j * T64, tq64, D + h * HD, row0 + j * 64, &bkv[j]);
        tma_load_2d(sV + j * T64, tq64, 2 * D + h * HD, row0 + j * 64, &bkv[j]);
        ++nkv[j];
      }
      auto issue_sp = [&](int jj) {  // S = Q K_jj^T, dP = dO V_jj^T (block jj loaded, block jj-1's read out)
        const int kb = jj & 1;
        const uint32_t q = smem_u32(sQ), dO = smem_u32(sdO), k = smem_u32(sK + kb * T64), v = smem_u32(sV + kb * T64);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tS, kdesc(q, kk), kdesc(k, kk), idSP, kk ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tP, kdesc(dO, kk), kdesc(v, kk), idSP, kk ? 1u : 0u);
        tc_commit(bs);
      };
      bool go = await(bq, 0, err, DERR_MMA_WAIT, abort) && await(&bkv[0], 0, err, DERR_MMA_WAIT, abort);
      if (go) {
        tc_fence_after();
        issue_sp(0);
      }
      for (int j = 0; j < nkb && go; ++j) {
        const int kb = j & 1;
        if (j + 1 < nkb) {  // the next block's S, dP as soon as the rows have read block j's
          if (!await(&bkv[(j + 1) & 1], ((j + 1) >> 1) & 1, err, DERR_MMA_WAIT, abort)) break;
          if (!await(bsc, j & 1, err, DERR_MMA_WAIT, abort)) break;
          tc_fence_after();
          issue_sp(j + 1);
        }
        if (!await(bp, j & 1, err, DERR_MMA_WAIT, abort)) break;  // dS_j written
        tc_fence_after();
        {
          const uint32_t ds = smem_u32(sdS), k = smem_u32(sK + kb * T64);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tQ, kdesc(ds, kk), mndesc(k, kk), idQ, (j | kk) ? 1u : 0u);
          tc_commit(bo);
        }
        if (j + 2 < nkb) {  // block j's buffers, once dQ += dS_j K_j is done
          if (!await(bo, j & 1, err, DERR_MMA_WAIT, abort)) break;
          mbar_arrive_expect_tx(&bkv[kb], 2 * T64);
          tma_load_2d(sK + kb * T64, tq64, D + h * HD, row0 + (j + 2) * 64, &bkv[kb]);
          tma_load_2d(sV + kb * T64, tq64, 2 * D + h * HD, row0 + (j + 2) * 64, &bkv[kb]);
          ++nkv[kb];
        }
      }
      tc_commit(bfin);
      mbar_wait_bounded(bfin, 0, err, DERR_DRAIN_WAIT);
      for (int bb = 0; bb < 2; ++bb)
        if (nkv[bb]) mbar_wait_bounded(&bkv[bb], (nkv[bb] - 1) & 1, err, DERR_DRAIN_WAIT);
      mbar_wait_bounded(bq, 0, err, DERR_DRAIN_WAIT);
    }
  } else {  // ---- rows ----
    const uint32_t lane = static_cast<uint32_t>(warp * 32) << 16;
    // this row's log-sum-exp (log2 domain) and D = rowsum(dO o O)
    float L2 = 0.f, Dr = 0.f;
    if (qi < seq) {
      const int64_t row = static_cast<int64_t>(row0) + qi;
      L2 = lse[row * heads + h] * kLog2e;
      Dr = dvec[row * heads + h];
    }
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      ok = __all_sync(0xffffffffu, await(bs, j & 1, err, DERR_ACC_WAIT, abort));
      if (!ok) break;
      tc_fence_after();
      float v[128];  // S (64 columns), then dP (64 columns), one round trip
      {
        const uint32_t a[4] = {tS + lane, tS + lane + 32, tP + lane, tP + lane + 32};
        ld_rows<4>(a, v);
      }
      tc_fence_before();
      mbar_arrive1(bsc);
      // P = exp2(s * scale log2(e) - LSE) (hidden keys: 2^-inf = 0), then
      // dS = P o (dP - D), two lanes per instruction
#pragma unroll
      for (int i = 0; i < 64; i += 2) ffma2(v[i], v[i + 1], v[i], v[i + 1], kScaleLog2, kScaleLog2, -L2, -L2);
      if (j * 64 + 63 > q0) {  // a block that some row of this CTA sees only in part
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (j * 64 + i > qi) v[i] = -INFINITY;
      }
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        float d0, d1;
        fadd2(d0, d1, v[64 + i], v[65 + i], -Dr, -Dr);
        fmul2(v[i], v[i + 1], ex2_approx(v[i]), ex2_approx(v[i + 1]), d0, d1);  // dS
      }
      if (j > 0) {  // the previous dQ product reads the dS tile
        ok = __all_sync(0xffffffffu, await(bo, (j - 1) & 1, err, DERR_ACC_WAIT, abort));
        if (!ok) break;
      }
      st_row32_bf16(sdS, r, 0, v);
      st_row32_bf16(sdS, r, 4, v + 32);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive1(bp);
    }
    if (ok) ok = __all_sync(0xffffffffu, await(bo, (nkb - 1) & 1, err, DERR_ACC_WAIT, abort));
    tc_fence_after();
    if (ok) {
      const int64_t row = static_cast<int64_t>(row0) + qi;
      store_row64(tQ + lane, dqkv + row * ld + h * HD, 0.125f, qi < seq);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

__device__ void attn_bwd_dkv(const CUtensorMap* tq64, const CUtensorMap* tq128, const CUtensorMap* td64,
                             const float* __restrict__ lse, const float* __restrict__ dvec,
                             __nv_bfloat16* __restrict__ dqkv, int seq, int heads, int b, int* err, uint8_t* sm) {
  uint8_t* sK = sm;
  uint8_t* sV = sm + T128;
  uint8_t* sQ = sm + 2 * T128;     // two 64-row buffers
  uint8_t* sdO = sQ + 2 * T64;     // two 64-row buffers
  uint8_t* sPt = sdO + 2 * T64;    // 128 keys x 64 queries
  uint8_t* sdSt = sPt + T128;      // 128 keys x 64 queries (ends at 96 KB)
  float* sL = reinterpret_cast<float*>(sm + BWD_LD);  // [2][64], negated
  float* sD = sL + 128;                               // [2][64], negated
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + BWD_BAR);
  uint64_t *bkv = bar, *bq = bar + 1, *bs = bar + 3, *bsc = bar + 4, *bp = bar + 5, *bo = bar + 6, *bfin = bar + 7,
           *bld = bar + 8;  // bld[2]: the LSE and D of a block are in their slot (64 writers)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 10);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

  const int r = threadIdx.x, warp = r >> 5;
  const int kb = blockIdx.x;  // the key blocks with the most queries first
  const int h = blockIdx.y;
  const int D = heads * HD;
  const int64_t ld = 3 * static_cast<int64_t>(D);
  const int row0 = b * seq;
  const int k0 = kb * 128;
  const int kr = k0 + r;  // the key of row thread r
  const int i0 = k0 / 64, nq = seq / 64;  // 64-query blocks i0..nq-1 see this key block
  const int niter = nq - i0;

  if (r == 0) {
    prefetch_tmap(tq64);
    prefetch_tmap(tq128);
    prefetch_tmap(td64);
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    mbar_init(bsc, 128);
    mbar_init(bp, 128);
    mbar_init(bo, 1);
    mbar_init(bfin, 1);
    mbar_init(&bld[0], 64);
    mbar_init(&bld[1], 64);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem, tP = tmem + 64, tV = tmem + 128, tK = tmem + 192;

  if (warp == 4) {
    if (r == 128) {  // ---- issuer ----
      constexpr uint32_t idSP = mma_idesc_bf16(128, 64, false, false);
      constexpr uint32_t idKV = mma_idesc_bf16(128, 64, false, true);
      int nqi[2] = {0, 0};
      mbar_arrive_expect_tx(bkv, 2 * T128);
      tma_load_2d(sK, tq128, D + h * HD, row0 + k0, bkv);
      tma_load_2d(sV, tq128, 2 * D + h * HD, row0 + k0, bkv);
      for (int t = 0; t < 2 && t < niter; ++t) {
        mbar_arrive_expect_tx(&bq[t], 2 * T64);
        tma_load_2d(sQ + t * T64, tq64, h * HD, row0 + (i0 + t) * 64, &bq[t]);
        tma_load_2d(sdO + t * T64, td64, h * HD, row0 + (i0 + t) * 64, &bq[t]);
        ++nqi[t];
      }
      auto issue_sp = [&](int tt) {  // S^T = K Q_tt^T, dP^T = V dO_tt^T
        const int qb2 = tt & 1;
        const uint32_t k = smem_u32(sK), v = smem_u32(sV), q = smem_u32(sQ + qb2 * T64),
                       dO = smem_u32(sdO + qb2 * T64);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tS, kdesc(k, kk), kdesc(q, kk), idSP, kk ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tP, kdesc(v, kk), kdesc(dO, kk), idSP, kk ? 1u : 0u);
        tc_commit(bs);
      };
      bool go = await(bkv, 0, err, DERR_MMA_WAIT, abort) && await(&bq[0], 0, err, DERR_MMA_WAIT, abort);
      if (go) {
        tc_fence_after();
        issue_sp(0);
      }
      for (int t = 0; t < niter && go; ++t) {
        const int qbuf = t & 1;
        if (t + 1 < niter) {  // the next block's S^T, dP^T as soon as the rows have read block t's
          if (!await(&bq[(t + 1) & 1], ((t + 1) >> 1) & 1, err, DERR_MMA_WAIT, abort)) break;
          if (!await(bsc, t & 1, err, DERR_MMA_WAIT, abort)) break;
          tc_fence_after();
          issue_sp(t + 1);
        }
        if (!await(bp, t & 1, err, DERR_MMA_WAIT, abort)) break;  // P^T, dS^T of block t written
        tc_fence_after();
        {
          const uint32_t pt = smem_u32(sPt), dst = smem_u32(sdSt), q = smem_u32(sQ + qbuf * T64),
                         dO = smem_u32(sdO + qbuf * T64);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tV, kdesc(pt, kk), mndesc(dO, kk), idKV, (t | kk) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tK, kdesc(dst, kk), mndesc(q, kk), idKV, (t | kk) ? 1u : 0u);
          tc_commit(bo);
        }
        if (t + 2 < niter) {  // block t's buffers, once dV, dK of block t are done
          if (!await(bo, t & 1, err, DERR_MMA_WAIT, abort)) break;
          mbar_arrive_expect_tx(&bq[qbuf], 2 * T64);
          tma_load_2d(sQ + qbuf * T64, tq64, h * HD, row0 + (i0 + t + 2) * 64, &bq[qbuf]);
          tma_load_2d(sdO + qbuf * T64, td64, h * HD, row0 + (i0 + t + 2) * 64, &bq[qbuf]);
          ++nqi[qbuf];
        }
      }
      tc_commit(bfin);
      mbar_wait_bounded(bfin, 0, err, DERR_DRAIN_WAIT);
      for (int bb = 0; bb < 2; ++bb)
        if (nqi[bb]) mbar_wait_bounded(&bq[bb], (nqi[bb] - 1) & 1, err, DERR_DRAIN_WAIT);
      mbar_wait_bounded(bkv, 0, err, DERR_DRAIN_WAIT);
    }
  } else {  // ---- rows ----
    const uint32_t lane = static_cast<uint32_t>(warp * 32) << 16;
    // -LSE (log2 domain) and -D of the 64 queries of a block: block i0's now,
    // each next block's read one block ahead; block t sits in slot t & 1 and
    // is published by the (t >> 1)-th phase of bld[t & 1]
    if (r < 64) {
      const int64_t row = static_cast<int64_t>(row0) + i0 * 64 + r;
      sL[r] = -(lse[row * heads + h] * kLog2e);
      sD[r] = -dvec[row * heads + h];
      mbar_arrive1(&bld[0]);
    }
    bool ok = true;
    for (int t = 0; t < niter; ++t) {
      const int i = i0 + t, qbuf = t & 1;
      ok = __all_sync(0xffffffffu, await(&bld[qbuf], (t >> 1) & 1, err, DERR_ACC_WAIT, abort));
      if (!ok) break;
      float nL = 0.f, nD = 0.f;
      if (r < 64 && t + 1 < niter) {
        const int64_t row = static_cast<int64_t>(row0) + (i + 1) * 64 + r;
        nL = -(lse[row * heads + h] * kLog2e);
        nD = -dvec[row * heads + h];
      }
      ok = __all_sync(0xffffffffu, await(bs, t & 1, err, DERR_ACC_WAIT, abort));
      if (!ok) break;
      tc_fence_after();
      float v[128];  // S^T (64 columns), then dP^T (64 columns), one round trip
      {
        const uint32_t a[4] = {tS + lane, tS + lane + 32, tP + lane, tP + lane + 32};
        ld_rows<4>(a, v);
      }
      tc_fence_before();
      mbar_arrive1(bsc);
      const float* L = sL + qbuf * 64;
      const float* Dq = sD + qbuf * 64;
      // P^T = exp2(s * scale log2(e) - LSE) (hidden pairs: 2^-inf = 0) and
      // dS^T = P^T o (dP^T - D), two lanes per instruction; the slots hold
      // -LSE and -D
#pragma unroll
      for (int q = 0; q < 64; q += 2) ffma2(v[q], v[q + 1], v[q], v[q + 1], kScaleLog2, kScaleLog2, L[q], L[q + 1]);
      if (i * 64 < k0 + 127) {  // a query block that some key of this CTA precedes only in part
#pragma unroll
        for (int q = 0; q < 64; ++q)
          if (i * 64 + q < kr) v[q] = -INFINITY;
      }
#pragma unroll
      for (int q = 0; q < 64; q += 2) {
        v[q] = ex2_approx(v[q]);  // P^T
        v[q + 1] = ex2_approx(v[q + 1]);
        float d0, d1;
        fadd2(d0, d1, v[64 + q], v[65 + q], Dq[q], Dq[q + 1]);
        fmul2(v[64 + q], v[65 + q], v[q], v[q + 1], d0, d1);  // dS^T
      }
      if (t > 0) {  // the previous dV, dK products read the P^T and dS^T tiles
        ok = __all_sync(0xffffffffu, await(bo, (t - 1) & 1, err, DERR_ACC_WAIT, abort));
        if (!ok) break;
      }
      st_row32_bf16(sPt, r, 0, v);
      st_row32_bf16(sPt, r, 4, v + 32);
      st_row32_bf16(sdSt, r, 0, v + 64);
      st_row32_bf16(sdSt, r, 4, v + 96);
      if (r < 64 && t + 1 < niter) {  // the next block's
        sL[(qbuf ^ 1) * 64 + r] = nL;
        sD[(qbuf ^ 1) * 64 + r] = nD;
        mbar_arrive1(&bld[qbuf ^ 1]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive1(bp);
    }
    if (ok) ok = __all_sync(0xffffffffu, await(bo, (niter - 1) & 1, err, DERR_ACC_WAIT, abort));
    tc_fence_after();
    if (ok) {
      const int64_t row = static_cast<int64_t>(row0) + kr;
      store_row64(tK + lane, dqkv + row * ld + D + h * HD, 0.125f, kr < seq);
      store_row64(tV + lane, dqkv + row * ld + 2 * D + h * HD, 1.0f, kr < seq);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// One launch for both kinds: blocks with z < nseq compute dQ of sequence z,
// the others dK/dV of sequence z - nseq; the two kinds share no data.
__global__ void __maxnreg__(ATTN_MAXNREG) attn_bwd_kernel(const __grid_constant__ CUtensorMap tq64,
                                                       const __grid_constant__ CUtensorMap tq128,
                                                       const __grid_constant__ CUtensorMap td64,
                                                       const __grid_constant__ CUtensorMap td128,
                                                       const float* __restrict__ lse, const float* __restrict__ dvec,
                                                       __nv_bfloat16* __restrict__ dqkv, int seq, int heads, int nseq,
                                                       int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int z = blockIdx.z;
  if (z < nseq)
    attn_bwd_dq(&tq64, &tq128, &td128, lse, dvec, dqkv, seq, heads, z, err, sm);
  else
    attn_bwd_dkv(&tq64, &tq128, &td64, lse, dvec, dqkv, seq, heads, z - nseq, err, sm);
  griddep_launch();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static std::atomic<EncodeFn> fn{nullptr};
  EncodeFn f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeFn>(p);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

// bf16 matrix [rows][cols] (row stride ld elements), boxes of 64 columns x
// box_rows rows, 128-byte swizzle.
bool amake_tmap(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld, int box_rows) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_args(int nseq, int seq, int heads) {
  if (nseq < 1 || seq < 64 || seq % 64 || heads < 1 || heads > 65535)
    return set_error(GPIPE_ERR_INVALID_ARG, "attention: need nseq >= 1, seq %% 64 == 0, heads >= 1");
  if (static_cast<int64_t>(nseq) * seq > (int64_t(1) << 30))
    return set_error(GPIPE_ERR_INVALID_ARG, "attention: nseq * seq must be at most 2^30");
  return GPIPE_OK;
}

}  // namespace

int prepare_attention() {
  static std::atomic<unsigned long long> done{0};
  return once_per_device(done, []() -> int {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BWD_SMEM);
    if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "attention: shared-memory attribute failed");
    if (!encode_fn()) return set_error(GPIPE_ERR_CUDA, "attention: cuTensorMapEncodeTiled entry point not found");
    return static_cast<int>(GPIPE_OK);
  });
}

int launch_attention_fwd(int nseq, int seq, int heads, const void* qkv, void* o, float* lse, cudaStream_t s) {
  int rc = check_args(nseq, seq, heads);
  if (rc) return rc;
  if (!al16(qkv) || !al16(o)) return set_error(GPIPE_ERR_INVALID_ARG, "attention: pointers must be 16-B aligned");
  rc = prepare_attention();
  if (rc) return rc;
  int* err = device_error_ptr();
  if (!err) return set_error(GPIPE_ERR_CUDA, "attention: no device error word");
  const int64_t D = static_cast<int64_t>(heads) * HD, rows = static_cast<int64_t>(nseq) * seq;
  CUtensorMap tq;
  if (!amake_tmap(&tq, qkv, 3 * D, rows, 3 * D, 128))
    return set_error(GPIPE_ERR_CUDA, "attention_fwd: tensor map creation failed");
  dim3 grid((seq + 127) / 128, heads, nseq);
  (void)launch_k<true>(attn_fwd_kernel, grid, FWD_THREADS, FWD_SMEM, s, tq, static_cast<__nv_bfloat16*>(o), lse, seq,
                       heads, err);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "attention_fwd launch: %s", cudaGetErrorString(e));
  return GPIPE_OK;
}

int launch_attention_bwd(int nseq, int seq, int heads, const void* qkv, const void* o, const void* dout,
                         const float* lse, float* dvec, void* dqkv, cudaStream_t s) {
  int rc = check_args(nseq, seq, heads);
  if (rc) return rc;
  if (!al16(qkv) || !al16(o) || !al16(dout) || !al16(dqkv))
    return set_error(GPIPE_ERR_INVALID_ARG, "attention: pointers must be 16-B aligned");
  if (nseq > 32767) return set_error(GPIPE_ERR_INVALID_ARG, "attention: nseq must be <= 32767");
  rc = prepare_attention();
  if (rc) return rc;
  int* err = device_error_ptr();
  if (!err) return set_error(GPIPE_ERR_CUDA, "attention: no device error word");
  const int64_t D = static_cast<int64_t>(heads) * HD, rows = static_cast<int64_t>(nseq) * seq;
  CUtensorMap tq64, tq128, td64, td128;
  bool ok = amake_tmap(&tq64, qkv, 3 * D, rows, 3 * D, 64) && amake_tmap(&tq128, qkv, 3 * D, rows, 3 * D, 128) &&
            amake_tmap(&td64, dout, D, rows, D, 64) && amake_tmap(&td128, dout, D, rows, D, 128);
  if (!ok) return set_error(GPIPE_ERR_CUDA, "attention_bwd: tensor map creation failed");
  const int64_t nd = rows * heads;
  (void)launch_k(attn_dvec_kernel, static_cast<int>((nd + 255) / 256), 256, 0, s, static_cast<const __nv_bfloat16*>(o),
                 static_cast<const __nv_bfloat16*>(dout), dvec, nd, heads);
  count_launch();
  cudaError_t e0 = cudaGetLastError();
  if (e0 != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "attention_bwd (D) launch: %s", cudaGetErrorString(e0));
  dim3 grid((seq + 127) / 128, heads, 2 * nseq);
  (void)launch_k<true>(attn_bwd_kernel, grid, BWD_THREADS, BWD_SMEM, s, tq64, tq128, td64, td128, lse,
                       static_cast<const float*>(dvec), static_cast<__nv_bfloat16*>(dqkv), seq, heads, nseq, err);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "attention_bwd launch: %s", cudaGetErrorString(e));
  return GPIPE_OK;
}

}  // namespace gp
