// Causal multi-head attention, head width 64, bf16 operands, fp32 softmax.
//
// Forward: one CTA per (64-query block, head, sequence); 4 warps, 16 query
// rows each.  Key/value blocks of 64 stream through double-buffered shared
// memory (cp.async); S = Q K^T and O += P V run on the tensor cores
// (mma.sync m16n8k16, bf16 in, fp32 accumulate) with an online softmax in
// the log2 domain.  Saves the natural-log LSE per (row, head).
//
// Backward, without atomics (bit-reproducible):
//   dq kernel   per (query block, head, sequence): D = rowsum(dO o O), then for
//               every visible key block P = exp(S - LSE), dP = dO V^T,
//               dS = P o (dP - D), dQ += dS K.
//   dkv kernel  per (key block, head, sequence): for every query block that
//               sees it, P^T, dV += P^T dO, dP^T = V dO^T, dS^T, dK += dS^T Q.
// Scale 1/sqrt(64) = 0.125.  Causal: query i sees keys j <= i.
#include "../../include/gpipe.h"
#include "common.cuh"
#include "kernels.h"
#include "launch_util.cuh"

namespace gp {
namespace {

constexpr int HD = 64;         // head width
constexpr int BQ = 64;         // rows per block (queries or keys)
constexpr int LDS = HD + 8;    // padded shared row (bf16 elements)
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;  // scale * log2(e)
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldm_x4_t(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Copy a 64 x 64 bf16 tile (global row stride ld elements) into padded smem.
__device__ __forceinline__ void load_tile(__nv_bfloat16 (*dst)[LDS], const __nv_bfloat16* src, int64_t ld) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = threadIdx.x + i * 128;  // 512 16-B chunks
    const int r = idx >> 3, c = (idx & 7) * 8;
    cp_async16(&dst[r][c], src + (int64_t)r * ld + c);
  }
}

// A fragments (16 rows x 64) of rows r0.. from a smem tile: af[kk][4] for k16 step kk.
__device__ __forceinline__ void load_a_frags(uint32_t (*af)[4], __nv_bfloat16 (*t)[LDS], int r0) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    ldm_x4(af[kk], &t[r0 + (lane & 7) + ((lane >> 3) & 1) * 8][kk * 16 + ((lane >> 4) & 1) * 8]);
}

// acc[nt][4] (16 x 64) += A (16 x 64, fragments) * T^T where T is a 64 x 64
// smem tile whose rows are the n index (B "col" layout, non-transposed ldmatrix).
__device__ __forceinline__ void mma_abt(float (*acc)[4], const uint32_t (*af)[4], __nv_bfloat16 (*t)[LDS]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b[4];
      ldm_x4(b, &t[np * 16 + ((lane >> 4) & 1) * 8 + (lane & 7)][kk * 16 + ((lane >> 3) & 1) * 8]);
      mma16816(acc[2 * np], af[kk], b[0], b[1]);
      mma16816(acc[2 * np + 1], af[kk], b[2], b[3]);
    }
  }
}

// acc[nt][4] (16 x 64) += P (16 x 64 over k, as fp32 accumulator fragments
// converted to bf16) * T where T is a 64 x 64 smem tile with rows = k
// (transposed ldmatrix).
__device__ __forceinline__ void mma_pt(float (*acc)[4], const float (*p)[4], __nv_bfloat16 (*t)[LDS]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t a[4];
    a[0] = pack_bf16x2(p[2 * kk][0], p[2 * kk][1]);
    a[1] = pack_bf16x2(p[2 * kk][2], p[2 * kk][3]);
    a[2] = pack_bf16x2(p[2 * kk + 1][0], p[2 * kk + 1][1]);
    a[3] = pack_bf16x2(p[2 * kk + 1][2], p[2 * kk + 1][3]);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b[4];
      ldm_x4_t(b, &t[kk * 16 + (lane >> 3 & 1) * 8 + (lane & 7)][np * 16 + ((lane >> 4) & 1) * 8]);
      mma16816(acc[2 * np], a, b[0], b[1]);
      mma16816(acc[2 * np + 1], a, b[2], b[3]);
    }
  }
}

__device__ __forceinline__ void zero_acc(float (*a)[4]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i][0] = a[i][1] = a[i][2] = a[i][3] = 0.f;
}

// Store a 16 x 64 fp32 fragment block (rows r0.., scaled) as bf16 at dst (row stride ld).
__device__ __forceinline__ void store_frag(__nv_bfloat16* dst, int64_t ld, const float (*a)[4], float scale) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int c = nt * 8 + 2 * t;
    *reinterpret_cast<uint32_t*>(dst + (int64_t)g * ld + c) = pack_bf16x2(a[nt][0] * scale, a[nt][1] * scale);
    *reinterpret_cast<uint32_t*>(dst + (int64_t)(g + 8) * ld + c) = pack_bf16x2(a[nt][2] * scale, a[nt][3] * scale);
  }
}

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) attn_fwd_kernel(const __nv_bfloat16* __restrict__ qkv,
                                                       __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                       int seq, int heads) {
  griddep_wait();
  griddep_launch();
  __shared__ __align__(16) __nv_bfloat16 Qs[BQ][LDS];
  __shared__ __align__(16) __nv_bfloat16 Ks[2][BQ][LDS];
  __shared__ __align__(16) __nv_bfloat16 Vs[2][BQ][LDS];
  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int D = heads * HD;
  const int64_t ld = 3 * (int64_t)D;
  const __nv_bfloat16* base = qkv + (int64_t)b * seq * ld;
  const __nv_bfloat16* Qg = base + (int64_t)qb * BQ * ld + h * HD;
  const __nv_bfloat16* Kg = base + D + h * HD;
  const __nv_bfloat16* Vg = base + 2 * D + h * HD;

  load_tile(Qs, Qg, ld);
  load_tile(Ks[0], Kg, ld);
  load_tile(Vs[0], Vg, ld);
  cp_async_commit();

  uint32_t qf[4][4];
  float o[8][4];
  zero_acc(o);
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int qrow0 = warp * 16 + g;  // local query rows qrow0, qrow0 + 8

  for (int kb = 0; kb <= qb; ++kb) {
    if (kb + 1 <= qb) {
      load_tile(Ks[(kb + 1) & 1], Kg + (int64_t)(kb + 1) * BQ * ld, ld);
      load_tile(Vs[(kb + 1) & 1], Vg + (int64_t)(kb + 1) * BQ * ld, ld);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kb == 0) load_a_frags(qf, Qs, warp * 16);
    float s[8][4];
    zero_acc(s);
    mma_abt(s, qf, Ks[kb & 1]);
    // scale into the log2 domain, mask the diagonal block
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[nt][e] * kScaleLog2;
        if (kb == qb) {
          const int key = nt * 8 + 2 * t + (e & 1);
          const int q = qrow0 + (e >> 1) * 8;
          if (key > q) v = -INFINITY;
        }
        s[nt][e] = v;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
    const float c0 = exp2f(m0 - nm0), c1 = exp2f(m1 - nm1);
    m0 = nm0;
    m1 = nm1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - m0);
      s[nt][1] = exp2f(s[nt][1] - m0);
      s[nt][2] = exp2f(s[nt][2] - m1);
      s[nt][3] = exp2f(s[nt][3] - m1);
      rs0 += s[nt][0] + s[nt][1];
      rs1 += s[nt][2] + s[nt][3];
      o[nt][0] *= c0;
      o[nt][1] *= c0;
      o[nt][2] *= c1;
      o[nt][3] *= c1;
    }
    l0 = l0 * c0 + rs0;
    l1 = l1 * c1 + rs1;
    mma_pt(o, s, Vs[kb & 1]);
    __syncthreads();
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.0f / l0, inv1 = 1.0f / l1;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    o[nt][0] *= inv0;
    o[nt][1] *= inv0;
    o[nt][2] *= inv1;
    o[nt][3] *= inv1;
  }
  const int64_t row = (int64_t)b * seq + qb * BQ + warp * 16;
  store_frag(out + row * D + h * HD, D, o, 1.0f);
  if (t == 0) {
    lse[(row + g) * heads + h] = (m0 + log2f(l0)) * kLn2;
    lse[(row + g + 8) * heads + h] = (m1 + log2f(l1)) * kLn2;
  }
}

// Shared storage of the backward kernels (above the 48 KB static limit, so
// allocated dynamically).
struct DqSmem {
  __nv_bfloat16 Qs[BQ][LDS];
  __nv_bfloat16 dOs[BQ][LDS];
  __nv_bfloat16 Ks[2][BQ][LDS];
  __nv_bfloat16 Vs[2][BQ][LDS];
  float Ls[BQ], Ds[BQ];
};
struct DkvSmem {
  __nv_bfloat16 Ks[BQ][LDS];
  __nv_bfloat16 Vs[BQ][LDS];
  __nv_bfloat16 Qs[2][BQ][LDS];
  __nv_bfloat16 dOs[2][BQ][LDS];
  float Ls[2][BQ], Ds[2][BQ];
};

// D = rowsum(dO o O) of head h for the 64 rows row0..row0+63, by the block's
// 128 threads (two per row, 32 columns each, then one shuffle): the same
// arithmetic wherever it runs, so the dQ and dK/dV blocks agree bit for bit.
__device__ __forceinline__ float row_dot_o_do(const __nv_bfloat16* __restrict__ out,
                                              const __nv_bfloat16* __restrict__ dout, int64_t row0, int h, int D) {
  const int r = threadIdx.x >> 1, c0 = (threadIdx.x & 1) * 32;
  const __nv_bfloat16* orow = out + (row0 + r) * D + h * HD + c0;
  const __nv_bfloat16* drow = dout + (row0 + r) * D + h * HD + c0;
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < 32; c += 8) {
    float ov[8], dv[8];
    load8(orow + c, ov);
    load8(drow + c, dv);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = fmaf(ov[j], dv[j], acc);
  }
  return acc + __shfl_xor_sync(0xffffffffu, acc, 1);
}

// ---------------------------------------------------------------------------
// Backward: dQ (and D = rowsum(dO o O)) for sequence b
// ---------------------------------------------------------------------------
__device__ __forceinline__ void attn_bwd_dq(const __nv_bfloat16* __restrict__ qkv,
                                            const __nv_bfloat16* __restrict__ out,
                                            const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
                                            float* __restrict__ dvec, __nv_bfloat16* __restrict__ dqkv, int seq,
                                            int heads, int b, uint8_t* dyn_smem) {
  DqSmem& S = *reinterpret_cast<DqSmem*>(dyn_smem);
  auto& Qs = S.Qs;
  auto& dOs = S.dOs;
  auto& Ks = S.Ks;
  auto& Vs = S.Vs;
  auto& Ls = S.Ls;
  auto& Ds = S.Ds;
  const int qb = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int D = heads * HD;
  const int64_t ld = 3 * (int64_t)D;
  const int64_t row0 = (int64_t)b * seq + qb * BQ;  // first global row of this block
  const __nv_bfloat16* base = qkv + (int64_t)b * seq * ld;
  const __nv_bfloat16* Kg = base + D + h * HD;
  const __nv_bfloat16* Vg = base + 2 * D + h * HD;

  load_tile(Qs, qkv + row0 * ld + h * HD, ld);
  load_tile(dOs, dout + row0 * D + h * HD, D);
  load_tile(Ks[0], Kg, ld);
  load_tile(Vs[0], Vg, ld);
  cp_async_commit();

  // D for the block's rows
  {
    const int r = threadIdx.x >> 1;
    const float acc = row_dot_o_do(out, dout, row0, h, D);
    if ((threadIdx.x & 1) == 0) {
      Ds[r] = acc;
      dvec[(row0 + r) * heads + h] = acc;
      Ls[r] = lse[(row0 + r) * heads + h] * 1.4426950408889634f;
    }
  }

  uint32_t qf[4][4], df[4][4];
  float dq[8][4];
  zero_acc(dq);
  const int qr = warp * 16 + g;
  for (int kb = 0; kb <= qb; ++kb) {
    if (kb + 1 <= qb) {
      load_tile(Ks[(kb + 1) & 1], Kg + (int64_t)(kb + 1) * BQ * ld, ld);
      load_tile(Vs[(kb + 1) & 1], Vg + (int64_t)(kb + 1) * BQ * ld, ld);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kb == 0) {
      load_a_frags(qf, Qs, warp * 16);
      load_a_frags(df, dOs, warp * 16);
    }
    const float L0 = Ls[qr], L1 = Ls[qr + 8], D0 = Ds[qr], D1 = Ds[qr + 8];
    float p[8][4], dp[8][4];
    zero_acc(p);
    zero_acc(dp);
    mma_abt(p, qf, Ks[kb & 1]);
    mma_abt(dp, df, Vs[kb & 1]);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool lo = e < 2;
        float pv = exp2f(p[nt][e] * kScaleLog2 - (lo ? L0 : L1));
        if (kb == qb) {
          const int key = nt * 8 + 2 * t + (e & 1);
          if (key > qr + (lo ? 0 : 8)) pv = 0.f;
        }
        p[nt][e] = pv * (dp[nt][e] - (lo ? D0 : D1));  // dS
      }
    }
    mma_pt(dq, p, Ks[kb & 1]);
    __syncthreads();
  }
  store_frag(dqkv + (row0 + warp * 16) * ld + h * HD, ld, dq, 0.125f);
}

// ---------------------------------------------------------------------------
// Backward: dK, dV
// ---------------------------------------------------------------------------
// (D of the query rows recomputed here, so this part does not wait for the dQ part)
__device__ __forceinline__ void attn_bwd_dkv(const __nv_bfloat16* __restrict__ qkv,
                                             const __nv_bfloat16* __restrict__ out,
                                             const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
                                             __nv_bfloat16* __restrict__ dqkv, int seq, int heads, int b,
                                             uint8_t* dyn_smem) {
  DkvSmem& S = *reinterpret_cast<DkvSmem*>(dyn_smem);
  auto& Ks = S.Ks;
  auto& Vs = S.Vs;
  auto& Qs = S.Qs;
  auto& dOs = S.dOs;
  auto& Ls = S.Ls;
  auto& Ds = S.Ds;
  const int kb = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int D = heads * HD;
  const int64_t ld = 3 * (int64_t)D;
  const int nqb = seq / BQ;
  const int64_t srow = (int64_t)b * seq;  // first global row of the sequence
  const __nv_bfloat16* Qg = qkv + srow * ld + h * HD;
  const __nv_bfloat16* dOg = dout + srow * D + h * HD;

  load_tile(Ks, qkv + (srow + kb * BQ) * ld + D + h * HD, ld);
  load_tile(Vs, qkv + (srow + kb * BQ) * ld + 2 * D + h * HD, ld);
  load_tile(Qs[0], Qg + (int64_t)kb * BQ * ld, ld);
  load_tile(dOs[0], dOg + (int64_t)kb * BQ * D, D);
  cp_async_commit();
  {
    const float dd = row_dot_o_do(out, dout, srow + kb * BQ, h, D);
    if ((threadIdx.x & 1) == 0) Ds[0][threadIdx.x >> 1] = dd;
  }
  if (threadIdx.x < BQ) {
    const int64_t r = srow + kb * BQ + threadIdx.x;
    Ls[0][threadIdx.x] = lse[r * heads + h] * 1.4426950408889634f;
  }

  uint32_t kf[4][4], vf[4][4];
  float dk[8][4], dv[8][4];
  zero_acc(dk);
  zero_acc(dv);
  const int kr = warp * 16 + g;  // local key rows kr, kr + 8
  for (int qb = kb; qb < nqb; ++qb) {
    const int buf = (qb - kb) & 1;
    if (qb + 1 < nqb) {
      const int nb = buf ^ 1;
      load_tile(Qs[nb], Qg + (int64_t)(qb + 1) * BQ * ld, ld);
      load_tile(dOs[nb], dOg + (int64_t)(qb + 1) * BQ * D, D);
      cp_async_commit();
      {
        const float dd = row_dot_o_do(out, dout, srow + (qb + 1) * BQ, h, D);
        if ((threadIdx.x & 1) == 0) Ds[nb][threadIdx.x >> 1] = dd;
      }
      if (threadIdx.x < BQ) {
        const int64_t r = srow + (qb + 1) * BQ + threadIdx.x;
        Ls[nb][threadIdx.x] = lse[r * heads + h] * 1.4426950408889634f;
      }
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (qb == kb) {
      load_a_frags(kf, Ks, warp * 16);
      load_a_frags(vf, Vs, warp * 16);
    }
    float pt[8][4], dpt[8][4];
    zero_acc(pt);
    zero_acc(dpt);
    mma_abt(pt, kf, Qs[buf]);   // S^T (keys x queries)
    mma_abt(dpt, vf, dOs[buf]); // dP^T = V dO^T
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int q = nt * 8 + 2 * t + (e & 1);
        float pv = exp2f(pt[nt][e] * kScaleLog2 - Ls[buf][q]);
        if (qb == kb && q < kr + (e >= 2 ? 8 : 0)) pv = 0.f;
        pt[nt][e] = pv;
        dpt[nt][e] = pv * (dpt[nt][e] - Ds[buf][q]);  // dS^T
      }
    }
    mma_pt(dv, pt, dOs[buf]);
    mma_pt(dk, dpt, Qs[buf]);
    __syncthreads();
  }
  const int64_t row = srow + kb * BQ + warp * 16;
  store_frag(dqkv + row * ld + D + h * HD, ld, dk, 0.125f);
  store_frag(dqkv + row * ld + 2 * D + h * HD, ld, dv, 1.0f);
}

// One launch for both parts: blocks with z < nseq compute dQ of sequence z,
// the others dK/dV of sequence z - nseq; the two parts share no data.
constexpr size_t kBwdSmem = sizeof(DqSmem) > sizeof(DkvSmem) ? sizeof(DqSmem) : sizeof(DkvSmem);
__global__ void __launch_bounds__(128) attn_bwd_kernel(const __nv_bfloat16* __restrict__ qkv,
                                                       const __nv_bfloat16* __restrict__ out,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse, float* __restrict__ dvec,
                                                       __nv_bfloat16* __restrict__ dqkv, int seq, int heads, int nseq) {
  griddep_wait();
  griddep_launch();
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  const int z = blockIdx.z;
  if (z < nseq)
    attn_bwd_dq(qkv, out, dout, lse, dvec, dqkv, seq, heads, z, dyn_smem);
  else
    attn_bwd_dkv(qkv, out, dout, lse, dqkv, seq, heads, z - nseq, dyn_smem);
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int prepare_attention() {
  static std::atomic<unsigned long long> done{0};
  return once_per_device(done, [] {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBwdSmem);
    return e == cudaSuccess ? GPIPE_OK : set_error(GPIPE_ERR_CUDA, "attention_bwd: shared-memory attribute failed");
  });
}

int launch_attention_fwd(int nseq, int seq, int heads, const void* qkv, void* o, float* lse, cudaStream_t s) {
  if (nseq < 1 || seq < BQ || seq % BQ || heads < 1 || heads > 65535)
    return set_error(GPIPE_ERR_INVALID_ARG, "attention: need nseq >= 1, seq %% 64 == 0, heads >= 1");
  if (!al16(qkv) || !al16(o)) return set_error(GPIPE_ERR_INVALID_ARG, "attention: pointers must be 16-B aligned");
  dim3 grid(seq / BQ, heads, nseq);
  (void)launch_k(attn_fwd_kernel, grid, 128, 0, s, static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(o), lse,
                                       seq, heads);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "attention_fwd launch: %s", cudaGetErrorString(e));
  return GPIPE_OK;
}

int launch_attention_bwd(int nseq, int seq, int heads, const void* qkv, const void* o, const void* dout,
                         const float* lse, float* dvec, void* dqkv, cudaStream_t s) {
  if (nseq < 1 || seq < BQ || seq % BQ || heads < 1 || heads > 65535)
    return set_error(GPIPE_ERR_INVALID_ARG, "attention: need nseq >= 1, seq %% 64 == 0, heads >= 1");
  if (!al16(qkv) || !al16(o) || !al16(dout) || !al16(dqkv))
    return set_error(GPIPE_ERR_INVALID_ARG, "attention: pointers must be 16-B aligned");
  int rc = prepare_attention();
  if (rc) return rc;
  if (nseq > 32767) return set_error(GPIPE_ERR_INVALID_ARG, "attention: nseq must be <= 32767");
  dim3 grid(seq / BQ, heads, 2 * nseq);
  (void)launch_k(attn_bwd_kernel, grid, 128, kBwdSmem, s, static_cast<const __nv_bfloat16*>(qkv),
                 static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, dvec,
                 static_cast<__nv_bfloat16*>(dqkv), seq, heads, nseq);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "attention_bwd launch: %s", cudaGetErrorString(e));
  return GPIPE_OK;
}

}  // namespace gp
