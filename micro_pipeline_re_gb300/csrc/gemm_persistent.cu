// Persistent bf16 GEMM on tcgen05 for GEMMs with more output tiles than SMs.
//
// One CTA per SM walks tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...
// Tiles are numbered in groups of PGROUP row tiles (m fastest within a group,
// then n), so the tiles in flight at one time read a band of A and a band of B
// that stay in L2 together.  Each tile is computed by exactly one CTA:
// deterministic.
//   warp 0 / lane 0   TMA producer over all (tile, k-block) pairs, through a
//                     ring of STAGES operand stages
//   warp 1            allocates TMEM; lane 0 issues tcgen05.mma into one of two
//                     accumulators (2 x BN columns), so the MMAs of tile i+1
//                     run while the epilogue drains tile i
//   warps 2..9        epilogue, each warp on its own (no barrier between
//                     them): TMEM lane quarter warp % 4 (the lanes a warp may
//                     read), column half (warp - 2) / 4; per 32-column chunk it
//                     loads the accumulator (the next chunk's load in flight),
//                     applies bias / residual / GELU, writes its own swizzled
//                     32 x 32 staging box and TMA-stores it, or TMA-reduce-adds
//                     the fp32 gradient (the bias gradient, sum over k of A:
//                     with 128-wide tiles an M=128, N=16 MMA against a tile of
//                     ones into TMEM beside the accumulators; 256-wide tiles
//                     fill TMEM, so callers add it with a separate reduction)
// SM pairs (PAIR): clusters of two CTAs walk 256 x BN tiles, pair p taking
// tiles p, p + pairs, ...  Each CTA's producer loads its own 128 rows of A and
// BN/2 columns of B per stage, both completing on rank 0's stage barrier
// (rank 0 expects both halves' bytes); rank 0's lane issues 256-row
// cta_group::2 products that read both CTAs' stages and accumulate each CTA's
// rows in its own TMEM; its commits free both CTAs' stages and announce a
// finished accumulator to both CTAs' epilogues (multicast); the 16 epilogue
// warps of the pair arrive on rank 0's accumulator-free barrier.  A cluster
// barrier at the start (every barrier initialised) and at the end (no CTA
// leaves while the pair's products may still read its shared memory) frames
// the work.
// Bounded waits as in the single-tile kernel.
#include <cuda.h>

#include "../../include/gpipe.h"
#include "common.cuh"
#include "kernels.h"
#include "launch_util.cuh"

namespace gp {
namespace {

constexpr int PM = 128;
constexpr int PK = 64;
constexpr int P_THREADS = 320;      // 10 warps
constexpr int SMEM_BUDGET = 232448 - 1024 - 512;

// PAIR: a cluster of two CTAs computes 256 x BN tiles with 256-row MMAs
// (cta_group::2); each CTA holds 128 rows of A and BN/2 columns of B per stage
// and accumulates its own 128 rows in its tensor memory.
template <int BN, int EPI, bool PAIR = false>
struct PCfg {
  static constexpr bool F32_OUT = (EPI == EPI_ACC_F32 || EPI == EPI_STORE_F32 || EPI == EPI_RESID_F32);
  static constexpr int TM = PAIR ? 2 * PM : PM;  // rows of a tile
  static constexpr int BH = PAIR ? BN / 2 : BN;  // columns of B one CTA holds
  static constexpr int A_BYTES = PM * PK * 2;
  static constexpr int B_BYTES = BH * PK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // an epilogue warp's staging box: 32 rows x 32 columns (64-byte rows in bf16,
  // 128-byte rows in fp32); bias+GELU writes two (z and GELU(z))
  static constexpr int BOX_BYTES = 32 * 32 * (F32_OUT ? 4 : 2);
  static constexpr int BOXES = EPI == EPI_BIAS_GELU ? 2 : 1;
  // bias gradient by MMA against ones (2 x 16 TMEM columns beside the accumulators) when they fit
  static constexpr bool DB_MMA = !PAIR && EPI == EPI_ACC_F32 && 2 * BN + 32 <= 512;
  static constexpr int ONES_BYTES = DB_MMA ? 2048 : 0;
  static constexpr int fit(int nbuf) { return (SMEM_BUDGET - 8 * nbuf * BOXES * BOX_BYTES - ONES_BYTES) / STAGE_BYTES; }
  // two staging buffers per warp (a chunk's store drains while the next chunk
  // is computed) when four operand stages still fit, else one
  static constexpr int WNB = fit(2) >= 4 ? 2 : 1;
  static constexpr int WARP_STG = WNB * BOXES * BOX_BYTES;
  static constexpr int STAGING = 8 * WARP_STG;
  static constexpr int STAGES = fit(WNB) > 6 ? 6 : fit(WNB);
  static constexpr int OFF_STG = STAGES * STAGE_BYTES;
  static constexpr int OFF_ONES = OFF_STG + STAGING;
  static constexpr int OFF_BAR = OFF_ONES + ONES_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 512;
  static constexpr int MMA_M = PAIR ? 2 * PM : PM;
  // TMEM: two accumulators of BN columns (+ 2 x 16 bias-gradient columns)
  static constexpr int TCOLS = (2 * BN + (DB_MMA ? 32 : 0)) <= 256 ? 256 : 512;
  static_assert(STAGES >= 3, "not enough shared memory for three stages");
  static_assert(SMEM <= 232448, "over the 227 KB per-CTA shared memory limit");
  static_assert(2 * BN + (DB_MMA ? 32 : 0) <= 512, "accumulators exceed tensor memory");
};

constexpr int PGROUP = 16;  // row tiles per group of the tile order

struct PArgs {
  const float* bias;   // fp32 [N] (store / bias+GELU) or NULL
  float* dbias;        // EPI_ACC_F32: fp32 [M] += sum_k A(m,k), or NULL
  const void* xsrc;    // residual (store) or GELU pre-activation (GELU backward), bf16, or NULL
  int64_t ldx;
  int M, N, K;
  int m_tiles, n_tiles;
};

// Byte offset of 16-byte unit u of row r in a staging box, in the layout of the
// tensor map's swizzle: bf16 boxes (64-byte rows, 64-byte swizzle: unit bits
// 4-5 XOR address bits 7-8) and fp32 boxes (128-byte rows, 128-byte swizzle:
// unit bits 4-6 XOR address bits 7-9).  Lanes = rows, so a warp's 16-byte
// writes of one unit hit every bank once per 8 rows.
__device__ __forceinline__ uint32_t box_off_bf16(int r, int u) {
  return static_cast<uint32_t>(r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
}
__device__ __forceinline__ uint32_t box_off_f32(int r, int u) {
  return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Origin (row, column) of tile t in the grouped tile order.
template <int TM, int BN>
__device__ __forceinline__ void tile_origin(int t, const PArgs& a, int& m0, int& n0) {
  const int per_group = PGROUP * a.n_tiles;
  const int grp = t / per_group, r = t - grp * per_group;
  const int first = grp * PGROUP;
  const int gm = a.m_tiles - first < PGROUP ? a.m_tiles - first : PGROUP;
  m0 = (first + r % gm) * TM;
  n0 = (r / gm) * BN;
}

// Bounded wait that gives up at once after any earlier give-up in the CTA.
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, int* err, int code, volatile int* abort) {
  if (*abort) return false;
  if (mbar_wait_bounded(bar, parity, err, code)) return true;
  *abort = 1;
  return false;
}

template <bool A_K, bool B_K, int BN, int EPI, bool PAIR = false>
__global__ void __launch_bounds__(P_THREADS, 1)
    tc_gemm_persistent(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
                       PArgs args, int* err) {
  using Cfg = PCfg<BN, EPI, PAIR>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int TM = Cfg::TM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sStg = smem + Cfg::OFF_STG;
  uint8_t* sOnes = smem + Cfg::OFF_ONES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;  // accumulator b holds a finished tile
  uint64_t* acce = accf + 2;        // accumulator b has been drained
  uint64_t* bfin = acce + 2;        // every MMA of the CTA (pair) has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bfin + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = args.m_tiles * args.n_tiles;
  const int nk = (args.K + PK - 1) / PK;
  // PAIR: rank 0 of the pair issues the MMAs; both load their halves and run
  // their epilogues; the pair walks tiles pair, pair + pairs, ...
  const int rank = PAIR ? static_cast<int>(cluster_ctarank() & 1u) : 0;
  const int first_tile = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], PAIR ? 16 : 8);  // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(bfin, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (Cfg::DB_MMA && threadIdx.x < 128) {  // 16 rows x 64 bf16 of 1.0
    reinterpret_cast<uint4*>(sOnes)[threadIdx.x] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tslot, Cfg::TCOLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tslot, Cfg::TCOLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR) cluster_sync();  // both CTAs' barriers exist before any copy or arrival names them
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  griddep_wait();  // the previous kernel in the stream has completed; global reads from here on

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      for (int t = first_tile; t < total && !*abort; t += tile_step) {
        int m0, n0;
        tile_origin<TM, BN>(t, args, m0, n0);
        const int am = m0 + rank * PM;        // this CTA's rows of A
        const int bn = n0 + rank * Cfg::BH;   // this CTA's columns of B
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          if (!pwait(&empty[s], ((it / STAGES) & 1) ^ 1, err, DERR_TMA_WAIT, abort)) break;
          uint8_t* a = smem + s * Cfg::STAGE_BYTES;
          uint8_t* b = a + Cfg::A_BYTES;
          const int k0 = kb * PK;
          if (PAIR) {
            // both CTAs' copies complete on rank 0's barrier, which expects the bytes of both
            const uint32_t fb = map_peer(smem_u32(&full[s]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * Cfg::STAGE_BYTES);
            if (A_K) {
              tma_load_2d_pair(a, &tmA, k0, am, fb);
            } else {
              tma_load_2d_pair(a, &tmA, am, k0, fb);
              tma_load_2d_pair(a + 8192, &tmA, am + 64, k0, fb);
            }
            if (B_K) {
              tma_load_2d_pair(b, &tmB, k0, bn, fb);
            } else {
#pragma unroll
              for (int j = 0; j < Cfg::BH / 64; ++j) tma_load_2d_pair(b + j * 8192, &tmB, bn + 64 * j, k0, fb);
            }
          } else {
            mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
            if (A_K) {
              tma_load_2d(a, &tmA, k0, am, &full[s]);
            } else {
              tma_load_2d(a, &tmA, am, k0, &full[s]);
              tma_load_2d(a + 8192, &tmA, am + 64, k0, &full[s]);
            }
            if (B_K) {
              tma_load_2d(b, &tmB, k0, bn, &full[s]);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_2d(b + j * 8192, &tmB, bn + 64 * j, k0, &full[s]);
            }
          }
        }
      }
      // no copy may still be landing in shared memory when the CTA exits (the
      // pair's copies all complete on rank 0's barriers; rank 1 is held by the
      // final cluster barrier until rank 0 has seen them)
      if (rank == 0)
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1, err, DERR_DRAIN_WAIT);
    }
    griddep_launch();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = mma_idesc_bf16(Cfg::MMA_M, BN, !A_K, !B_K);
      constexpr uint32_t idesc_db = mma_idesc_bf16(PM, 16, !A_K, false);
      const uint32_t ones = smem_u32(sOnes);
      int it = 0, i = 0;
      for (int t = first_tile; t < total; t += tile_step, ++i) {
        const int b = i & 1;
        if (PAIR) {  // the peer's epilogue warps arrive from the other CTA
          if (*abort || !mbar_wait_bounded_cluster(&acce[b], ((i >> 1) & 1) ^ 1, err, DERR_MMA_WAIT)) {
            *abort = 1;
            break;
          }
        } else if (!pwait(&acce[b], ((i >> 1) & 1) ^ 1, err, DERR_MMA_WAIT, abort)) {
          break;
        }
        tc_fence_after();
        int tm0, tn0;
        tile_origin<TM, BN>(t, args, tm0, tn0);
        const bool do_db = Cfg::DB_MMA && args.dbias != nullptr && tn0 == 0;
        const uint32_t dacc = tmem + b * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          if (!pwait(&full[s], (it / STAGES) & 1, err, DERR_MMA_WAIT, abort)) break;
          tc_fence_after();
          const uint32_t a = smem_u32(smem + s * Cfg::STAGE_BYTES);
          const uint32_t bb = a + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < PK / 16; ++kk) {
            const uint64_t ad = A_K ? sw128_desc(a + kk * 32, 16, 1024) : sw128_desc(a + kk * 2048, 8192, 1024);
            const uint64_t bd = B_K ? sw128_desc(bb + kk * 32, 16, 1024) : sw128_desc(bb + kk * 2048, 8192, 1024);
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            if (PAIR) {
              tc_mma_f16_pair(dacc, ad, bd, idesc, acc);
            } else {
              tc_mma_f16(dacc, ad, bd, idesc, acc);
              if (do_db) tc_mma_f16(tmem + 2 * BN + 16 * b, ad, sw128_desc(ones + kk * 32, 16, 1024), idesc_db, acc);
            }
          }
          if (PAIR) tc_commit_pair(&empty[s], 3);  // both CTAs' stage s is free again
          else tc_commit(&empty[s]);
        }
        // fires once this tile's MMAs have completed (in both CTAs of a pair)
        if (PAIR) tc_commit_pair(&accf[b], 3);
        else tc_commit(&accf[b]);
      }
      // every product issued has completed before the tensor memory is released
      if (PAIR) tc_commit_pair(bfin, 1);
      else tc_commit(bfin);
      mbar_wait_bounded(bfin, 0, err, DERR_DRAIN_WAIT);
    }
    griddep_launch();
  } else {
    // ---- epilogue warps 2..9, each independent of the others ----
    constexpr int HALF = BN / 2;     // columns of a warp per tile
    constexpr int CH = HALF / 32;    // its 32-column chunks
    constexpr bool X_F32 = EPI == EPI_RESID_F32;                                     // fp32 residual
    constexpr bool X_BF16 = EPI == EPI_STORE || EPI == EPI_GELU_BWD;                 // bf16 residual / z
    constexpr int XV = X_F32 ? 8 : 4;  // 16-byte words of a row's 32 inputs
    // the next chunk's accumulator load overlaps this chunk's work, except with
    // the fp32 residual, whose look-ahead already takes those registers
    constexpr bool LD_AHEAD = !X_F32;
    const int q = warp & 3;            // TMEM lane quarter this warp may read
    const int h = (warp - 2) >> 2;     // column half
    const int r = q * 32 + lane;       // row of the tile
    uint8_t* wst = sStg + (warp - 2) * Cfg::WARP_STG;
    int nst = 0;  // chunks this warp has staged (alternates its buffers)
    int i = 0;
    // rank 0's acce barrier (the MMA issuer's); a pair's epilogue warps arrive on it from both CTAs
    const uint32_t acce_leader = PAIR ? map_peer(smem_u32(acce), 0) : 0u;
    for (int t = first_tile; t < total; t += tile_step, ++i) {
      const int b = i & 1;
      int m0, n0;
      tile_origin<TM, BN>(t, args, m0, n0);
      m0 += rank * PM;  // this CTA's 128 rows of the tile
      const int m = m0 + r;
      const int c0 = n0 + h * HALF;  // the warp's first column
      int nch = (args.N - c0 + 31) / 32;  // its chunks inside the matrix
      nch = nch < 0 ? 0 : (nch > CH ? CH : nch);
      // The epilogue input (residual / GELU pre-activation) of this thread's
      // row is read one chunk ahead: chunk 0 before waiting for the accumulator.
      const bool has_x = (X_F32 || X_BF16) && args.xsrc != nullptr && m < args.M;
      const char* xrow = has_x ? static_cast<const char*>(args.xsrc) +
                                     static_cast<int64_t>(m) * args.ldx * (X_F32 ? 4 : 2)
                               : nullptr;
      uint4 xnext[XV];
      auto load_x = [&](int cc, uint4* dst) {
        const int col = c0 + cc * 32;
        if (has_x && col + 32 <= args.N) {
          const uint4* src = reinterpret_cast<const uint4*>(xrow + static_cast<int64_t>(col) * (X_F32 ? 4 : 2));
#pragma unroll
          for (int j = 0; j < XV; ++j) dst[j] = src[j];
        }
      };
      if (nch > 0) load_x(0, xnext);
      pwait(&accf[b], (i >> 1) & 1, err, DERR_ACC_WAIT, abort);
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * BN + h * HALF;
      uint32_t ra[32];
      if (LD_AHEAD && nch > 0) tmem_ld32(tb, ra);
#pragma unroll 1
      for (int c = 0; c < nch; ++c, ++nst) {
        if (!LD_AHEAD) tmem_ld32(tb + c * 32, ra);
        tmem_ld_wait32(ra);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(ra[j]);
        if (LD_AHEAD && c + 1 < nch) tmem_ld32(tb + (c + 1) * 32, ra);  // lands while this chunk is processed
        uint4 xcur[XV];
#pragma unroll
        for (int j = 0; j < XV; ++j) xcur[j] = xnext[j];
        if (c + 1 < nch) load_x(c + 1, xnext);
        const int ncol0 = c0 + c * 32;
        const bool full_cols = ncol0 + 32 <= args.N;
        // bias, then the residual / GELU derivative, in the single-tile kernel's order
        if ((EPI == EPI_STORE || EPI == EPI_BIAS_GELU || EPI == EPI_RESID_F32) && args.bias) {
          if (full_cols) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              float bb8[8];
              load8(args.bias + ncol0 + j, bb8);
#pragma unroll
              for (int e = 0; e < 8; ++e) v[j + e] += bb8[e];
            }
          } else {
            for (int j = 0; j < 32; ++j)
              if (ncol0 + j < args.N) v[j] += args.bias[ncol0 + j];
          }
        }
        if (has_x) {
          auto apply = [&](float& acc, float x) {
            if (EPI == EPI_GELU_BWD) acc *= gelu_grad_f(x);
            else acc += x;
          };
          if (full_cols) {
#pragma unroll
            for (int j = 0; j < XV; ++j) {
              const uint32_t w4[4] = {xcur[j].x, xcur[j].y, xcur[j].z, xcur[j].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (X_F32) {
                  apply(v[4 * j + e], __uint_as_float(w4[e]));
                } else if (EPI == EPI_GELU_BWD) {  // two lanes at a time
                  const float2 f = unpack_bf16x2(w4[e]);
                  float g0, g1;
                  gelu_grad2(f.x, f.y, g0, g1);
                  fmul2(v[8 * j + 2 * e], v[8 * j + 2 * e + 1], v[8 * j + 2 * e], v[8 * j + 2 * e + 1], g0, g1);
                } else {
                  const float2 f = unpack_bf16x2(w4[e]);
                  apply(v[8 * j + 2 * e], f.x);
                  apply(v[8 * j + 2 * e + 1], f.y);
                }
              }
            }
          } else {
            for (int j = 0; j < 32; ++j)
              if (ncol0 + j < args.N)
                apply(v[j], X_F32 ? reinterpret_cast<const float*>(xrow)[ncol0 + j]
                                  : bf2f(reinterpret_cast<const __nv_bfloat16*>(xrow)[ncol0 + j]));
          }
        }
        // stage the chunk (the store that last read this buffer has finished reading)
        uint8_t* stg = wst + (Cfg::WNB == 2 ? (nst & 1) : 0) * Cfg::BOXES * Cfg::BOX_BYTES;
        if (lane == 0) {
          if (Cfg::WNB == 2) bulk_wait_read_1();
          else bulk_wait_read_all();
        }
        __syncwarp();
        if (Cfg::F32_OUT) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(stg + box_off_f32(lane, u)) =
                make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) store8(reinterpret_cast<__nv_bfloat16*>(stg + box_off_bf16(lane, u)), v + 8 * u);
          if (EPI == EPI_BIAS_GELU) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float gv[8];
#pragma unroll
              for (int e = 0; e < 8; e += 2) gelu2(v[8 * u + e], v[8 * u + e + 1], gv[e], gv[e + 1]);
              store8(reinterpret_cast<__nv_bfloat16*>(stg + Cfg::BOX_BYTES + box_off_bf16(lane, u)), gv);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (!*abort) {
            if (EPI == EPI_ACC_F32) tma_reduce_add_2d(&tmC, ncol0, m0 + q * 32, stg);
            else tma_store_2d(&tmC, ncol0, m0 + q * 32, stg);
            if (EPI == EPI_BIAS_GELU) tma_store_2d(&tmC2, ncol0, m0 + q * 32, stg + Cfg::BOX_BYTES);
          }
          bulk_commit();  // (empty after a give-up: the buffer count stays in step)
        }
      }
      if (Cfg::DB_MMA && args.dbias != nullptr && n0 == 0 && h == 0) {
        uint32_t rr[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + 2 * BN + 16 * b, rr);
        tmem_ld_wait32(rr);
        if (m < args.M && !*abort) args.dbias[m] += __uint_as_float(rr[0]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // this warp has drained accumulator b
        if (PAIR) mbar_arrive_cluster(acce_leader + static_cast<uint32_t>(b * sizeof(uint64_t)));
        else mbar_arrive(&acce[b]);
      }
    }
    griddep_launch();
    if (lane == 0) bulk_wait_read_all();
  }
  tc_fence_before();
  if (PAIR) cluster_sync();  // neither CTA leaves while the pair's products may read its shared memory
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem, Cfg::TCOLS);
    else tmem_dealloc(tmem, Cfg::TCOLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool pmake_tmap(CUtensorMap* m, const void* base, bool f32, int64_t inner, int64_t outer, int64_t ld, int box_inner,
                int box_outer, bool swizzle64 = false) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn enc = nullptr;
  if (!enc) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<EncodeFn>(p);
  }
  const int es = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1u, 1u};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool A_K, bool B_K, int BN, int EPI, bool PAIR>
int pset_attr() {
  static std::atomic<unsigned long long> done{0};
  return once_per_device(done, [] {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_persistent<A_K, B_K, BN, EPI, PAIR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, PCfg<BN, EPI, PAIR>::SMEM);
    return e == cudaSuccess
               ? GPIPE_OK
               : set_error(GPIPE_ERR_CUDA, "persistent gemm: smem attribute: %s", cudaGetErrorString(e));
  });
}

template <bool A_K, bool B_K, int BN, int EPI, bool PAIR>
int prun(const GemmDesc& g, cudaStream_t stream, int ctas) {
  using Cfg = PCfg<BN, EPI, PAIR>;
  CUtensorMap ta, tb, tc, tc2;
  bool ok = A_K ? pmake_tmap(&ta, g.A, false, g.K, g.M, g.lda, 64, PM) : pmake_tmap(&ta, g.A, false, g.M, g.K, g.lda, 64, 64);
  ok = ok && (B_K ? pmake_tmap(&tb, g.B, false, g.K, g.N, g.ldb, 64, Cfg::BH)
                  : pmake_tmap(&tb, g.B, false, g.N, g.K, g.ldb, 64, 64));
  // output boxes: 32 x 32, one per epilogue warp and chunk (64-byte swizzle for
  // the 64-byte bf16 rows, 128-byte for the fp32 rows)
  ok = ok && pmake_tmap(&tc, g.C, Cfg::F32_OUT, g.N, g.M, g.ldc, 32, 32, !Cfg::F32_OUT);
  tc2 = tc;
  if (EPI == EPI_BIAS_GELU) ok = ok && pmake_tmap(&tc2, g.C2, false, g.N, g.M, g.ldc, 32, 32, true);
  if (!ok) return set_error(GPIPE_ERR_CUDA, "persistent gemm: cuTensorMapEncodeTiled failed");
  int rc = pset_attr<A_K, B_K, BN, EPI, PAIR>();
  if (rc) return rc;
  PArgs args{};
  args.bias = (EPI == EPI_STORE || EPI == EPI_BIAS_GELU || EPI == EPI_RESID_F32) ? g.bias : nullptr;
  args.dbias = EPI == EPI_ACC_F32 ? g.dbias : nullptr;
  if (EPI == EPI_ACC_F32 && !Cfg::DB_MMA && g.dbias)
    return set_error(GPIPE_ERR_UNSUPPORTED, "persistent gemm: no bias gradient with 256-wide tiles");
  const bool resid = EPI == EPI_STORE || EPI == EPI_RESID_F32;
  args.xsrc = resid ? g.resid : (EPI == EPI_GELU_BWD ? g.aux : nullptr);
  args.ldx = resid ? g.ldr : g.ldaux;
  args.M = g.M;
  args.N = g.N;
  args.K = g.K;
  args.m_tiles = (g.M + Cfg::TM - 1) / Cfg::TM;
  args.n_tiles = (g.N + BN - 1) / BN;
  const int tiles = args.m_tiles * args.n_tiles;
  if (!PAIR) {
    const int grid = ctas < tiles ? ctas : tiles;
    (void)launch_k<true>(tc_gemm_persistent<A_K, B_K, BN, EPI, PAIR>, grid, P_THREADS, Cfg::SMEM, stream, ta, tb, tc,
                         tc2, args, device_error_ptr());
  } else {
    // one cluster of two CTAs per pair of SMs of the share (an odd share rounded up)
    const int want = (ctas + 1) / 2;
    const int pairs = want < tiles ? want : tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(P_THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 0;  // heavy: never launched early
    set_priority_attr(attr[2], stream);
    cfg.attrs = attr;
    cfg.numAttrs = 3;
    (void)cudaLaunchKernelEx(&cfg, tc_gemm_persistent<A_K, B_K, BN, EPI, PAIR>, ta, tb, tc, tc2, args,
                             device_error_ptr());
  }
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "persistent gemm launch: %s", cudaGetErrorString(e));
  return GPIPE_OK;
}

// Output-tile width: 128 x 256 tiles read 96 B of operands per 128 clocks of
// MMA against 128 B per 64 clocks for 128 x 128 tiles, so they win unless
// the coarser tiles leave CTAs idle: take 256 when the rounds of tiles per CTA
// times the wider tile's relative time (1.5) is below the narrow tiles' rounds.
bool wide_tiles(const GemmDesc& g, int ctas) {
  const int64_t mt = (g.M + PM - 1) / PM;
  const int64_t r128 = (mt * ((g.N + 127) / 128) + ctas - 1) / ctas;
  const int64_t r256 = (mt * ((g.N + 255) / 256) + ctas - 1) / ctas;
  return 3 * r256 < 2 * r128;
}

template <int BN, bool PAIR = false>
int dispatch(const GemmDesc& g, cudaStream_t s, int ctas) {
  if (g.a_kmajor && g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE: return prun<true, true, BN, EPI_STORE, PAIR>(g, s, ctas);
      case EPI_BIAS_GELU: return prun<true, true, BN, EPI_BIAS_GELU, PAIR>(g, s, ctas);
      case EPI_STORE_F32: return prun<true, true, BN, EPI_STORE_F32, PAIR>(g, s, ctas);
      case EPI_ACC_F32: return prun<true, true, BN, EPI_ACC_F32, PAIR>(g, s, ctas);
      case EPI_RESID_F32: return prun<true, true, BN, EPI_RESID_F32, PAIR>(g, s, ctas);
    }
  } else if (g.a_kmajor && !g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE: return prun<true, false, BN, EPI_STORE, PAIR>(g, s, ctas);
      case EPI_GELU_BWD: return prun<true, false, BN, EPI_GELU_BWD, PAIR>(g, s, ctas);
      case EPI_ACC_F32: return prun<true, false, BN, EPI_ACC_F32, PAIR>(g, s, ctas);
    }
  } else if (!g.a_kmajor && !g.b_kmajor) {
    switch (g.epi) {
      case EPI_STORE: return prun<false, false, BN, EPI_STORE, PAIR>(g, s, ctas);
      case EPI_ACC_F32: return prun<false, false, BN, EPI_ACC_F32, PAIR>(g, s, ctas);
    }
  }
  return set_error(GPIPE_ERR_UNSUPPORTED, "persistent gemm: layout/epilogue not built");
}

template <int BN, bool PAIR = false>
int prepare_bn() {
  int rc = GPIPE_OK;
  rc = rc ? rc : pset_attr<true, true, BN, EPI_STORE, PAIR>();
  rc = rc ? rc : pset_attr<true, true, BN, EPI_BIAS_GELU, PAIR>();
  rc = rc ? rc : pset_attr<true, true, BN, EPI_STORE_F32, PAIR>();
  rc = rc ? rc : pset_attr<true, true, BN, EPI_ACC_F32, PAIR>();
  rc = rc ? rc : pset_attr<true, true, BN, EPI_RESID_F32, PAIR>();
  rc = rc ? rc : pset_attr<true, false, BN, EPI_STORE, PAIR>();
  rc = rc ? rc : pset_attr<true, false, BN, EPI_GELU_BWD, PAIR>();
  rc = rc ? rc : pset_attr<true, false, BN, EPI_ACC_F32, PAIR>();
  rc = rc ? rc : pset_attr<false, false, BN, EPI_STORE, PAIR>();
  rc = rc ? rc : pset_attr<false, false, BN, EPI_ACC_F32, PAIR>();
  return rc;
}

}  // namespace

// Output tiles at the finest persistent tiling (128 x 128).
int64_t persistent_tiles(const GemmDesc& g) {
  return static_cast<int64_t>((g.M + PM - 1) / PM) * ((g.N + 127) / 128);
}

// A weight-gradient GEMM with a bias gradient gets it by an MMA against ones
// beside 128-wide accumulators; for large ones (wide_bias_grad_gemm: M and N
// >= 1024, a shape-only rule) the caller runs the GEMM without it, on any
// tiles, and adds it with a separate reduction.
bool wide_bias_grad_gemm(const GemmDesc& g) { return g.epi == EPI_ACC_F32 && g.dbias && g.M >= 1024 && g.N >= 1024; }

// 128 x 256 tiles on SM pairs: 256 x 256 tiles computed by 256-row MMAs over
// two CTAs, each of which loads half the operand bytes per product of one
// 128 x 256 tile (the per-SM operand stream that bounds the single-CTA tiles).
// With K < 1024 a tile's mainloop is too short to repay the pair's hand-offs
// (measured: the small LM's vocabulary GEMMs, K = 512, ran slower on pairs).
constexpr int kPairMinK = 1024;
int launch_gemm_persistent(const GemmDesc& g, cudaStream_t s, int ctas) {
  if (g.epi == EPI_ACC_F32 && g.dbias) return dispatch<128>(g, s, ctas);  // bias gradient by ones-MMA
  if (!wide_tiles(g, ctas)) return dispatch<128>(g, s, ctas);
  return ctas >= 2 && g.K >= kPairMinK ? dispatch<256, true>(g, s, ctas) : dispatch<256>(g, s, ctas);
}

int prepare_gemm_persistent() {
  int rc = prepare_bn<128>();
  rc = rc ? rc : prepare_bn<256>();
  return rc ? rc : prepare_bn<256, true>();
}

}  // namespace gp
