// Memory-bound kernels of the step: LayerNorm forward/backward, column sums
// (bias gradients), next-token cross-entropy, MSE, embedding gather/scatter,
// the fused RMSProp update and small utilities.  All reductions run in a fixed
// order (no floating-point atomics), so every result is bit-reproducible and
// a re-computed forward equals the first one byte for byte.
#include <algorithm>
#include <atomic>

#include "../../include/gpipe.h"
#include "common.cuh"
#include "kernels.h"
#include "launch_util.cuh"

namespace gp {
namespace {

constexpr float kLnEps = 1e-5f;
constexpr int kMaxChunks = 4;       // d <= 4 * 256 = 1024 per warp-row
constexpr int kLnRowsPerWarp = 8;   // rows one block (8 warps) folds into one partial row
constexpr int kColRowsPerChunk = 32;

inline int blocks_for(size_t n, int per_block) { return static_cast<int>((n + per_block - 1) / per_block); }

int check_launch(const char* what) {
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  return GPIPE_OK;
}

// ---------------------------------------------------------------------------
// LayerNorm forward: one warp per row; lane owns 8-wide column groups
// (c*32 + lane)*8 for chunk c.  Two passes over registers (mean, then
// centred variance), fp32 statistics.
// ---------------------------------------------------------------------------
template <typename TI, typename TO>
__global__ void __launch_bounds__(256) ln_fwd_kernel(const TI* __restrict__ x, const float* __restrict__ g,
                                                     const float* __restrict__ b, TO* __restrict__ y,
                                                     float* __restrict__ mean, float* __restrict__ rstd, int rows,
                                                     int d) {
  griddep_wait();
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  if (row >= rows) return;
  const TI* xr = x + (int64_t)row * d;
  // every load of the row (x, and gamma / beta for the output) is issued
  // before the first reduction, so the row costs one memory round trip
  float v[kMaxChunks][8], gg[kMaxChunks][8], bb[kMaxChunks][8];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int col = (c * 32 + lane) * 8;
    if (col < d) {
      load8(xr + col, v[c]);
      load8(g + col, gg[c]);
      load8(b + col, bb[c]);
    }
  }
  // sums over 8 independent partials per lane (short dependency chains)
  float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int col = (c * 32 + lane) * 8;
    if (col < d) {
#pragma unroll
      for (int j = 0; j < 8; ++j) s8[j] += v[c][j];
    }
  }
  const float mu = warp_sum(((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]))) / d;
  float q8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int col = (c * 32 + lane) * 8;
    if (col < d) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float t = v[c][j] - mu;
        q8[j] = fmaf(t, t, q8[j]);
      }
    }
  }
  const float var = warp_sum(((q8[0] + q8[1]) + (q8[2] + q8[3])) + ((q8[4] + q8[5]) + (q8[6] + q8[7]))) / d;
  const float rs = 1.0f / sqrtf(var + kLnEps);
  TO* yr = y + (int64_t)row * d;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int col = (c * 32 + lane) * 8;
    if (col < d) {
      float o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = (v[c][j] - mu) * rs * gg[c][j] + bb[c][j];
      store8(yr + col, o);
    }
  }
  if (lane == 0) {
    mean[row] = mu;
    rstd[row] = rs;
  }
}

// ---------------------------------------------------------------------------
// LayerNorm backward.  Block b (8 warps) handles rows 8b .. 8b+7, one row per
// warp, with CH 256-column chunks per row (d <= 256*CH).  Each warp writes its
// row's dg and db terms (dy * x-hat, dy) to shared memory as soon as they are
// known; after one barrier every column is added over the warps in warp order
// into one partial row of scratch; col_reduce adds the partial rows in order.
// Both orders are fixed, so results are bit-reproducible.  Dynamic shared
// memory: 2 x 8 x d floats.
// ---------------------------------------------------------------------------
template <typename TD, typename TX, typename TO, int CH>
__global__ void __launch_bounds__(256) ln_bwd_kernel(const TD* __restrict__ dy, const TX* __restrict__ x,
                                                     const float* __restrict__ mean, const float* __restrict__ rstd,
                                                     const float* __restrict__ g, const TO* __restrict__ dres,
                                                     TO* __restrict__ dx, __nv_bfloat16* __restrict__ dx16,
                                                     float* __restrict__ partial, int rows, int d) {
  griddep_wait();
  griddep_launch();
  extern __shared__ __align__(16) float ln_stage[];  // [2][8][d]: dg terms, then db terms
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kLnRowsPerWarp + warp;
  float* sg = ln_stage + warp * d;
  float* sb = ln_stage + (kLnRowsPerWarp + warp) * d;
  if (r < rows) {
    const float mu = mean[r], rs = rstd[r];
    // every load of the row (x, dy, gamma and the residual gradient) is issued
    // before the first reduction: one memory round trip per row
    float xh[CH][8], gd[CH][8], rv[CH][8];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = (c * 32 + lane) * 8;
      if (col < d) {
        float dv[8];
        load8(x + (int64_t)r * d + col, xh[c]);
        load8(dy + (int64_t)r * d + col, dv);
        load8(g + col, gd[c]);
        if (dres) load8(dres + (int64_t)r * d + col, rv[c]);
        float tg[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          xh[c][j] = (xh[c][j] - mu) * rs;
          gd[c][j] = gd[c][j] * dv[j];  // gamma * dy
          tg[j] = dv[j] * xh[c][j];     // dg term
        }
        *reinterpret_cast<float4*>(sg + col) = make_float4(tg[0], tg[1], tg[2], tg[3]);
        *reinterpret_cast<float4*>(sg + col + 4) = make_float4(tg[4], tg[5], tg[6], tg[7]);
        *reinterpret_cast<float4*>(sb + col) = make_float4(dv[0], dv[1], dv[2], dv[3]);
        *reinterpret_cast<float4*>(sb + col + 4) = make_float4(dv[4], dv[5], dv[6], dv[7]);
      }
    }
    // the two row sums over 8 independent partials per lane
    float s1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, s2[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = (c * 32 + lane) * 8;
      if (col < d) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          s1[j] += gd[c][j];
          s2[j] += gd[c][j] * xh[c][j];
        }
      }
    }
    const float m1 = warp_sum(((s1[0] + s1[1]) + (s1[2] + s1[3])) + ((s1[4] + s1[5]) + (s1[6] + s1[7]))) / d;
    const float m2 = warp_sum(((s2[0] + s2[1]) + (s2[2] + s2[3])) + ((s2[4] + s2[5]) + (s2[6] + s2[7]))) / d;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = (c * 32 + lane) * 8;
      if (col < d) {
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = rs * (gd[c][j] - m1 - xh[c][j] * m2);
        if (dres) {
#pragma unroll
          for (int j = 0; j < 8; ++j) o[j] += rv[c][j];
        }
        store8(dx + (int64_t)r * d + col, o);
        if (dx16) store8(dx16 + (int64_t)r * d + col, o);  // the same values as bf16 (GEMM operands)
      }
    }
  } else {  // a row past the end adds nothing
    for (int col = lane * 4; col < d; col += 128) {
      *reinterpret_cast<float4*>(sg + col) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(sb + col) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();
  // fold the 8 rows' terms in warp order: dg into partial[0, d), db into [d, 2d)
  float* pr = partial + (int64_t)blockIdx.x * 2 * d;
  for (int col = threadIdx.x; col < 2 * d; col += 256) {
    const float* src = ln_stage + (col < d ? col : kLnRowsPerWarp * d + (col - d));
    float a = src[0];
#pragma unroll
    for (int w = 1; w < kLnRowsPerWarp; ++w) a += src[w * d];
    pr[col] = a;
  }
}

// out[c] += sum_{p < nparts} partial[p*ncols + c] in a fixed order: a block
// owns 32 columns, warp w adds the parts p = w, w + 8, ... (two alternating
// accumulators, loads of several parts in flight), and warp 0 adds the 8
// warps' sums in warp order.  Columns < split go to out_a, the rest to out_b.
constexpr int kColReduceWarps = 8;
__global__ void __launch_bounds__(32 * kColReduceWarps) col_reduce_kernel(const float* __restrict__ partial,
                                                                         int nparts, int ncols, float* out_a,
                                                                         int split, float* out_b) {
  griddep_wait();
  griddep_launch();
  __shared__ float wsum[kColReduceWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 32 + lane;
  float a0 = 0.f, a1 = 0.f;
  if (c < ncols) {
    int p = warp;
#pragma unroll 4
    for (; p + kColReduceWarps < nparts; p += 2 * kColReduceWarps) {
      a0 += partial[(int64_t)p * ncols + c];
      a1 += partial[(int64_t)(p + kColReduceWarps) * ncols + c];
    }
    if (p < nparts) a0 += partial[(int64_t)p * ncols + c];
  }
  wsum[warp][lane] = a0 + a1;
  __syncthreads();
  if (warp == 0 && c < ncols) {
    float t = wsum[0][lane];
#pragma unroll
    for (int w = 1; w < kColReduceWarps; ++w) t += wsum[w][lane];
    if (c < split) out_a[c] += t;
    else out_b[c - split] += t;
  }
}

// Column sums of a [rows, cols] matrix: block (x, y) sums rows
// y*kColRowsPerChunk.. of columns x*2048 + 8*tid .. +7 into partial row y.
template <typename T>
__global__ void __launch_bounds__(256) colsum_partial_kernel(const T* __restrict__ y, int64_t ldy, int rows,
                                                             int cols, float* __restrict__ partial) {
  griddep_wait();
  griddep_launch();
  const int col = (blockIdx.x * 256 + threadIdx.x) * 8;
  if (col >= cols) return;
  const int r0 = blockIdx.y * kColRowsPerChunk;
  const int r1 = min(r0 + kColRowsPerChunk, rows);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int r = r0; r < r1; ++r) {
    float v[8];
    load8(y + (int64_t)r * ldy + col, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] += v[j];
  }
  store8(partial + (int64_t)blockIdx.y * cols + col, acc);
}

// ---------------------------------------------------------------------------
// Bias gradient of a weight-gradient GEMM (db[m] += sum_k A(m, k)) in one
// launch without scratch, fixed order.
//  - A MN-major (stored [K][M], the step's dY): a cluster of kDbSplit CTAs
//    owns the 64 columns m = 64x .. 64x+63, CTA s of it the rows of its K
//    range; thread t sums the 8 columns 8(t%8).. over rows k = t/8, t/8 + 32,
//    ... of the range (16-B loads, 8 rows in flight, a row's 128 B read by 8
//    threads), the 32 row groups are added in order through shared memory,
//    and CTA 0 adds the kDbSplit range sums in rank order (distributed shared
//    memory) into db.
//  - A K-major (stored [M][K]): one warp per row m, lanes over k, shuffle fold.
// ---------------------------------------------------------------------------
constexpr int kDbSplit = 8;

__global__ void __launch_bounds__(256) dbias_mn_kernel(const __nv_bfloat16* __restrict__ a, int64_t lda, int M,
                                                        int K, float* __restrict__ db) {
  griddep_wait();
  griddep_launch();
  __shared__ float part[32][64 + 1];
  __shared__ __align__(16) float tot[64];
  const int c8 = (threadIdx.x & 7) * 8, g = threadIdx.x >> 3;
  const int m0 = blockIdx.x * 64;
  const int kper = ((K + kDbSplit - 1) / kDbSplit + 31) / 32 * 32;  // rows per CTA, a multiple of 32
  const int kb = static_cast<int>(blockIdx.y) * kper;
  const int ke = min(K, kb + kper);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (m0 + c8 + 8 <= M) {
    int k = kb + g;
    for (; k + 224 < ke; k += 256) {  // eight rows in flight
      float v[8][8];
#pragma unroll
      for (int u = 0; u < 8; ++u) load8(a + static_cast<int64_t>(k + 32 * u) * lda + m0 + c8, v[u]);
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += v[u][j];
    }
    for (; k < ke; k += 32) {
      float v[8];
      load8(a + static_cast<int64_t>(k) * lda + m0 + c8, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += v[j];
    }
  } else {
    for (int k = kb + g; k < ke; k += 32)
      for (int j = 0; j < 8; ++j)
        if (m0 + c8 + j < M) acc[j] += bf2f(a[static_cast<int64_t>(k) * lda + m0 + c8 + j]);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) part[g][c8 + j] = acc[j];
  __syncthreads();
  if (threadIdx.x < 64) {
    float t = part[0][threadIdx.x];
    for (int r = 1; r < 32; ++r) t += part[r][threadIdx.x];
    tot[threadIdx.x] = t;
  }
  cluster_sync();  // every range sum of the cluster is in place
  if (cluster_ctarank() == 0 && threadIdx.x < 64 && m0 + static_cast<int>(threadIdx.x) < M) {
    const uint32_t mine = smem_u32(&tot[threadIdx.x]);
    float t = ld_peer_f32(map_peer(mine, 0));
    for (int q = 1; q < kDbSplit; ++q) t += ld_peer_f32(map_peer(mine, static_cast<uint32_t>(q)));
    db[m0 + threadIdx.x] += t;
  }
  cluster_sync();  // the peers keep their shared memory until CTA 0 has read it
}

__global__ void __launch_bounds__(256) dbias_k_kernel(const __nv_bfloat16* __restrict__ a, int64_t lda, int M, int K,
                                                       float* __restrict__ db) {
  griddep_wait();
  griddep_launch();
  const int m = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (m >= M) return;
  const __nv_bfloat16* row = a + static_cast<int64_t>(m) * lda;
  float s = 0.f;
  const int full = K / 8;
  for (int j = lane; j < full; j += 32) {
    float v[8];
    load8(row + 8 * j, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) s += v[e];
  }
  if (lane == 0)
    for (int k = 8 * full; k < K; ++k) s += bf2f(row[k]);
  s = warp_sum(s);
  if (lane == 0) db[m] += s;
}

// ---------------------------------------------------------------------------
// Softmax cross-entropy on fp32 logits, one CTA (512 threads) per row.
// clip > 0: logit clipping ("GPipe technical review", "Training stability"):
// the softmax sees min(max(z, -clip), clip), and the gradient is zero where a
// logit lies outside [-clip, clip] (the derivative of the clamp).
// ---------------------------------------------------------------------------
constexpr int kCeThreads = 512;

// The clamp keeps a NaN a NaN (so a non-finite loss is still reported).
__device__ __forceinline__ float clip_logit(float x, float c) { return x < -c ? -c : (x > c ? c : x); }

__global__ void __launch_bounds__(kCeThreads) ce_kernel(float* __restrict__ logits, int vocab, int seq,
                                                        const int32_t* __restrict__ tokens, int row0,
                                                        float inv_count, float clip, float* __restrict__ loss_rows,
                                                        int want_grad, int* err) {
  griddep_wait();
  griddep_launch();
  __shared__ float sm_m[kCeThreads / 32], sm_s[kCeThreads / 32];
  __shared__ float sh_lse;
  const int r = blockIdx.x;
  const int gidx = row0 + r;
  const bool has_t = (gidx % seq) != seq - 1;
  int tgt = has_t ? tokens[gidx + 1] : -1;
  if (tgt >= vocab || (has_t && tgt < 0)) {  // invalid id: no target, flag it
    if (threadIdx.x == 0) atomicExch(err, DERR_BAD_TOKEN);
    tgt = -1;
  }
  float* z = logits + (int64_t)r * vocab;
  const float4* z4 = reinterpret_cast<const float4*>(z);
  const int n4 = vocab / 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const bool clipping = clip > 0.f;
  // pass 1: running max and rescaled sum of exp
  float m = -INFINITY, s = 0.f;
  for (int i = tid; i < n4; i += kCeThreads) {
    float4 v = z4[i];
    if (clipping) {
      v.x = clip_logit(v.x, clip);
      v.y = clip_logit(v.y, clip);
      v.z = clip_logit(v.z, clip);
      v.w = clip_logit(v.w, clip);
    }
    const float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (mx > m) {
      s *= expf(m - mx);
      m = mx;
    }
    s += expf(v.x - m) + expf(v.y - m) + expf(v.z - m) + expf(v.w - m);
  }
  // warp combine
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    const float nm = fmaxf(m, om);
    s = (m == -INFINITY ? 0.f : s * expf(m - nm)) + (om == -INFINITY ? 0.f : os * expf(om - nm));
    m = nm;
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_s[warp] = s;
  }
  __syncthreads();
  if (tid == 0) {
    float M = sm_m[0], S = sm_s[0];
    for (int w = 1; w < kCeThreads / 32; ++w) {
      const float nm = fmaxf(M, sm_m[w]);
      S = S * expf(M - nm) + sm_s[w] * expf(sm_m[w] - nm);
      M = nm;
    }
    const float lse = M + logf(S);
    sh_lse = lse;
    loss_rows[r] = tgt >= 0 ? (lse - (clipping ? clip_logit(z[tgt], clip) : z[tgt])) * inv_count : 0.f;
  }
  __syncthreads();
  if (!want_grad) return;
  const float lse = sh_lse;
  const float scale = tgt >= 0 ? inv_count : 0.f;
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(z);
  // pass 2: dz written in place.  Chunk c reads floats [4*512c, 4*512(c+1))
  // and then writes bf16 elements of the same indices, i.e. floats
  // [2*512c, 2*512(c+1)), all of which every thread has already read.
  for (int base = 0; base < n4; base += kCeThreads) {
    const int i = base + tid;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < n4) v = z4[i];
    __syncthreads();
    if (i < n4) {
      const float zv[4] = {v.x, v.y, v.z, v.w};
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = expf((clipping ? clip_logit(zv[e], clip) : zv[e]) - lse) * scale;
      const int c0 = 4 * i;
      if (tgt >= c0 && tgt < c0 + 4) p[tgt - c0] -= scale;
      if (clipping) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (!(fabsf(zv[e]) <= clip)) p[e] = 0.f;
      }
      uint2 u;
      u.x = pack_bf16x2(p[0], p[1]);
      u.y = pack_bf16x2(p[2], p[3]);
      *reinterpret_cast<uint2*>(dz + c0) = u;
    }
  }
}

// MSE: one warp per row.
__global__ void mse_kernel(const float* __restrict__ y, const float* __restrict__ t, int rows, int d,
                           float inv_count, float* __restrict__ loss_rows, float* __restrict__ dy) {
  griddep_wait();
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r >= rows) return;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float e = y[(int64_t)r * d + c] - t[(int64_t)r * d + c];
    s += e * e;
    dy[(int64_t)r * d + c] = 2.0f * e * inv_count;
  }
  s = warp_sum(s);
  if (lane == 0) loss_rows[r] = s * inv_count;
}

// ---------------------------------------------------------------------------
// Embedding
// ---------------------------------------------------------------------------
template <typename TO>
__global__ void embed_fwd_kernel(int rows, int d, int vocab, const int32_t* __restrict__ tokens,
                                 const __nv_bfloat16* __restrict__ emb, TO* __restrict__ x, int* err) {
  griddep_wait();
  griddep_launch();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // 8-element group
  const int groups = d / 8;
  if (i >= (int64_t)rows * groups) return;
  const int r = static_cast<int>(i / groups), c = static_cast<int>(i % groups) * 8;
  const int tok = tokens[r];
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (tok >= 0 && tok < vocab)
    load8(emb + (int64_t)tok * d + c, v);
  else if (c == 0)
    atomicExch(err, DERR_BAD_TOKEN);
  store8(x + (int64_t)r * d + c, v);  // exact: a bf16 value is an fp32 value
}

// CTA b owns embedding rows [b*vpc, (b+1)*vpc).  It scans the token list in
// order, compacts the positions whose token it owns (order kept), and adds
// each such dx row into its own embedding rows: one owner per row and a fixed
// order, hence no atomics and a deterministic result.
template <typename TI>
__global__ void __launch_bounds__(256) embed_bwd_kernel(int rows, int d, int vocab, int vpc,
                                                        const int32_t* __restrict__ tokens,
                                                        const TI* __restrict__ dx,
                                                        float* __restrict__ demb) {
  griddep_wait();
  griddep_launch();
  __shared__ int list[256];
  __shared__ int wcount[8];
  const int v0 = blockIdx.x * vpc, v1 = min(v0 + vpc, vocab);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int base = 0; base < rows; base += 256) {
    const int r = base + tid;
    const int t = r < rows ? tokens[r] : -1;
    const bool mine = t >= v0 && t < v1;
    const unsigned bal = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) wcount[warp] = __popc(bal);
    __syncthreads();
    int off = 0, total = 0;
    for (int w = 0; w < 8; ++w) {
      if (w < warp) off += wcount[w];
      total += wcount[w];
    }
    if (mine) list[off + __popc(bal & ((1u << lane) - 1u))] = r;
    __syncthreads();
    for (int i = 0; i < total; ++i) {
      const int rr = list[i];
      const int64_t vrow = tokens[rr];
      for (int c = tid * 8; c < d; c += 256 * 8) {
        float a[8], g[8];
        load8(demb + vrow * d + c, a);
        load8(dx + (int64_t)rr * d + c, g);
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] += g[j];
        store8(demb + vrow * d + c, a);
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------------------
// RMSProp, float4-vectorised, grid-stride; tail handled element-wise.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void rms_one(float& w, float& g, float& v, float lr, float decay, float omd, float eps) {
  v = decay * v + omd * (g * g);
  w = w - lr * g / (sqrtf(v) + eps);
}

__global__ void rmsprop_kernel(float* __restrict__ w, float* __restrict__ g, float* __restrict__ v,
                               __nv_bfloat16* __restrict__ wb, size_t n, float lr, float decay, float eps,
                               int zero_grad) {
  griddep_wait();
  griddep_launch();
  const float omd = 1.0f - decay;
  const size_t n4 = n / 4;
  float4* w4 = reinterpret_cast<float4*>(w);
  float4* g4 = reinterpret_cast<float4*>(g);
  float4* v4 = reinterpret_cast<float4*>(v);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 W = w4[i], G = g4[i], V = v4[i];
    rms_one(W.x, G.x, V.x, lr, decay, omd, eps);
    rms_one(W.y, G.y, V.y, lr, decay, omd, eps);
    rms_one(W.z, G.z, V.z, lr, decay, omd, eps);
    rms_one(W.w, G.w, V.w, lr, decay, omd, eps);
    w4[i] = W;
    v4[i] = V;
    if (zero_grad) g4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (wb) {
      uint2 u;
      u.x = pack_bf16x2(W.x, W.y);
      u.y = pack_bf16x2(W.z, W.w);
      *reinterpret_cast<uint2*>(wb + 4 * i) = u;
    }
  }
  if (blockIdx.x == 0) {
    for (size_t i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) {
      float W = w[i], G = g[i], V = v[i];
      rms_one(W, G, V, lr, decay, omd, eps);
      w[i] = W;
      v[i] = V;
      if (zero_grad) g[i] = 0.f;
      if (wb) wb[i] = f2bf(W);
    }
  }
}

__global__ void cast_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, size_t n) {
  griddep_wait();
  griddep_launch();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = f2bf(src[i]);
}

// One block of 1024 threads: fixed-order fp64 partial sums, fixed tree.
__global__ void __launch_bounds__(1024) sum_kernel(const float* __restrict__ x, size_t n, float* out) {
  griddep_wait();
  griddep_launch();
  __shared__ double sm[1024];
  double s = 0.0;
  for (size_t i = threadIdx.x; i < n; i += 1024) s += static_cast<double>(x[i]);
  sm[threadIdx.x] = s;
  __syncthreads();
  for (int o = 512; o > 0; o >>= 1) {
    if (threadIdx.x < o) sm[threadIdx.x] += sm[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = static_cast<float>(sm[0]);
}

// One thread writes the GPU's nanosecond clock (tracing of the step's phases).
__global__ void stamp_kernel(unsigned long long* out) {
  griddep_wait();
  griddep_launch();
  *out = globaltimer_ns();
}

__global__ void copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, size_t n16) {
  griddep_wait();
  griddep_launch();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
}

__global__ void count_diff_kernel(const uint32_t* __restrict__ a, const uint32_t* __restrict__ b, size_t n4,
                                  unsigned long long* counter) {
  griddep_wait();
  griddep_launch();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  unsigned int c = 0;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const uint32_t x = a[i] ^ b[i];
    c += ((x & 0xffu) != 0) + ((x & 0xff00u) != 0) + ((x & 0xff0000u) != 0) + ((x & 0xff000000u) != 0);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(counter, static_cast<unsigned long long>(c));
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// GELU and its derivative in fp32 (the epilogues' arithmetic, for checking it).
__global__ void gelu_kernel(size_t n, const float* __restrict__ z, float* __restrict__ y, float* __restrict__ dy) {
  griddep_wait();
  griddep_launch();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    if (y) y[i] = gelu_f(z[i]);
    if (dy) dy[i] = gelu_grad_f(z[i]);
  }
}

// Failure-detection probe: one thread waits, with the library's bounded wait,
// on an mbarrier that nothing will complete; the wait gives up after its limit
// and sets the device error word, and the kernel returns.
__global__ void wait_probe_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait_bounded(&bar, 0, err, DERR_PROBE);
  __syncthreads();
}

}  // namespace

int launch_wait_probe(cudaStream_t s) {
  (void)launch_k(wait_probe_kernel, 1, 32, 0, s, device_error_ptr());
  return check_launch("wait probe");
}

int launch_gelu(size_t n, const float* z, float* y, float* dy, cudaStream_t s) {
  if (n == 0) return GPIPE_OK;
  if (!z) return set_error(GPIPE_ERR_INVALID_ARG, "gelu: NULL input");
  const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, 65536));
  (void)launch_k(gelu_kernel, grid, 256, 0, s, n, z, y, dy);
  return check_launch("gelu");
}

size_t colred_scratch_floats(int rows, int cols) {
  const size_t parts = (rows + kLnRowsPerWarp - 1) / kLnRowsPerWarp;
  return parts * static_cast<size_t>(cols);
}

int launch_layernorm_fwd_io(int in_dtype, int out_dtype, int rows, int d, const void* x, const float* g,
                            const float* b, void* y, float* mean, float* rstd, cudaStream_t s) {
  if (rows < 1 || d < 8 || d % 8 || d > 32 * 8 * kMaxChunks)
    return set_error(GPIPE_ERR_INVALID_ARG, "layernorm: need rows >= 1, d %% 8 == 0, 8 <= d <= 1024");
  if (!al16(x) || !al16(y) || !al16(g) || !al16(b))
    return set_error(GPIPE_ERR_INVALID_ARG, "layernorm: pointers must be 16-B aligned");
  const int grid = blocks_for(rows, 8);
  using bf = __nv_bfloat16;
  if (in_dtype == DT_F32 && out_dtype == DT_F32)
    (void)launch_k(ln_fwd_kernel<float, float>, grid, 256, 0, s, static_cast<const float*>(x), g, b,
                   static_cast<float*>(y), mean, rstd, rows, d);
  else if (in_dtype == DT_F32 && out_dtype == DT_BF16)
    (void)launch_k(ln_fwd_kernel<float, bf>, grid, 256, 0, s, static_cast<const float*>(x), g, b,
                   static_cast<bf*>(y), mean, rstd, rows, d);
  else if (in_dtype == DT_BF16 && out_dtype == DT_BF16)
    (void)launch_k(ln_fwd_kernel<bf, bf>, grid, 256, 0, s, static_cast<const bf*>(x), g, b, static_cast<bf*>(y),
                   mean, rstd, rows, d);
  else
    return set_error(GPIPE_ERR_UNSUPPORTED, "layernorm: bf16 input with fp32 output is not built");
  return check_launch("layernorm_fwd");
}

int launch_layernorm_fwd(int dtype, int rows, int d, const void* x, const float* g, const float* b, void* y,
                         float* mean, float* rstd, cudaStream_t s) {
  return launch_layernorm_fwd_io(dtype, dtype, rows, d, x, g, b, y, mean, rstd, s);
}

namespace {
size_t ln_bwd_smem(int d) { return static_cast<size_t>(2 * kLnRowsPerWarp) * d * sizeof(float); }

template <typename TD, typename TX, typename TO>
cudaError_t ln_bwd_attr() {
  const int mx = static_cast<int>(ln_bwd_smem(32 * 8 * kMaxChunks));
  cudaError_t e = cudaFuncSetAttribute(ln_bwd_kernel<TD, TX, TO, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ln_bwd_kernel<TD, TX, TO, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ln_bwd_kernel<TD, TX, TO, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  return e;
}

template <typename TD, typename TX, typename TO>
void ln_bwd_launch(int grid, int d, cudaStream_t s, const void* dy, const void* x, const float* mean, const float* rstd,
                   const float* g, const void* dres, void* dx, void* dx16, float* scratch, int rows) {
  const TD* dyp = static_cast<const TD*>(dy);
  const TX* xp = static_cast<const TX*>(x);
  const TO* rp = static_cast<const TO*>(dres);
  TO* dxp = static_cast<TO*>(dx);
  __nv_bfloat16* d16 = static_cast<__nv_bfloat16*>(dx16);
  if (d <= 256)
    (void)launch_k(ln_bwd_kernel<TD, TX, TO, 1>, grid, 256, ln_bwd_smem(d), s, dyp, xp, mean, rstd, g, rp, dxp, d16, scratch, rows, d);
  else if (d <= 512)
    (void)launch_k(ln_bwd_kernel<TD, TX, TO, 2>, grid, 256, ln_bwd_smem(d), s, dyp, xp, mean, rstd, g, rp, dxp, d16, scratch, rows, d);
  else
    (void)launch_k(ln_bwd_kernel<TD, TX, TO, 4>, grid, 256, ln_bwd_smem(d), s, dyp, xp, mean, rstd, g, rp, dxp, d16, scratch, rows, d);
}
}  // namespace

int prepare_layernorm() {
  static std::atomic<unsigned long long> done{0};
  return once_per_device(done, []() -> int {
    using bf = __nv_bfloat16;
    cudaError_t e = ln_bwd_attr<float, float, float>();
    if (e == cudaSuccess) e = ln_bwd_attr<bf, bf, bf>();
    if (e == cudaSuccess) e = ln_bwd_attr<bf, float, float>();
    return e == cudaSuccess ? static_cast<int>(GPIPE_OK)
                            : set_error(GPIPE_ERR_CUDA, "layernorm_bwd: shared-memory attribute: %s", cudaGetErrorString(e));
  });
}

int launch_layernorm_bwd_rows_io(int dy_dtype, int x_dtype, int out_dtype, int rows, int d, const void* dy,
                                 const void* x, const float* mean, const float* rstd, const float* g, const void* dres,
                                 void* dx, void* dx16, float* scratch, cudaStream_t s) {
  if (rows < 1 || d < 8 || d % 8 || d > 32 * 8 * kMaxChunks)
    return set_error(GPIPE_ERR_INVALID_ARG, "layernorm_bwd: need rows >= 1, d %% 8 == 0, 8 <= d <= 1024");
  if (!al16(dy) || !al16(x) || !al16(dx) || !al16(g) || (dres && !al16(dres)) || (dx16 && !al16(dx16)) ||
      !al16(scratch))
    return set_error(GPIPE_ERR_INVALID_ARG, "layernorm_bwd: pointers must be 16-B aligned");
  const int rc = prepare_layernorm();
  if (rc) return rc;
  const int grid = (rows + kLnRowsPerWarp - 1) / kLnRowsPerWarp;
  using bf = __nv_bfloat16;
  if (dy_dtype == DT_F32 && x_dtype == DT_F32 && out_dtype == DT_F32)
    ln_bwd_launch<float, float, float>(grid, d, s, dy, x, mean, rstd, g, dres, dx, dx16, scratch, rows);
  else if (dy_dtype == DT_BF16 && x_dtype == DT_BF16 && out_dtype == DT_BF16)
    ln_bwd_launch<bf, bf, bf>(grid, d, s, dy, x, mean, rstd, g, dres, dx, dx16, scratch, rows);
  else if (dy_dtype == DT_BF16 && x_dtype == DT_F32 && out_dtype == DT_F32)
    ln_bwd_launch<bf, float, float>(grid, d, s, dy, x, mean, rstd, g, dres, dx, dx16, scratch, rows);
  else
    return set_error(GPIPE_ERR_UNSUPPORTED, "layernorm_bwd: this combination of element types is not built");
  return check_launch("layernorm_bwd");
}

int launch_layernorm_bwd_rows(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                              const float* rstd, const float* g, const void* dres, void* dx, float* scratch,
                              cudaStream_t s) {
  return launch_layernorm_bwd_rows_io(dtype, dtype, dtype, rows, d, dy, x, mean, rstd, g, dres, dx, nullptr, scratch,
                                      s);
}

int launch_layernorm_bwd_reduce(int rows, int d, const float* scratch, float* dg_acc, float* db_acc, cudaStream_t s) {
  const int parts = (rows + kLnRowsPerWarp - 1) / kLnRowsPerWarp;
  (void)launch_k(col_reduce_kernel, blocks_for(2 * d, 32), 32 * kColReduceWarps, 0, s, scratch, parts, 2 * d, dg_acc, d,
                 db_acc);
  return check_launch("layernorm_bwd reduce");
}

int launch_layernorm_bwd(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                         const float* rstd, const float* g, const void* dres, void* dx, float* dg_acc,
                         float* db_acc, float* scratch, cudaStream_t s) {
  const int rc = launch_layernorm_bwd_rows(dtype, rows, d, dy, x, mean, rstd, g, dres, dx, scratch, s);
  return rc ? rc : launch_layernorm_bwd_reduce(rows, d, scratch, dg_acc, db_acc, s);
}

int launch_dbias(bool a_kmajor, int M, int K, const void* a, int64_t lda, float* db, cudaStream_t s) {
  const __nv_bfloat16* ap = static_cast<const __nv_bfloat16*>(a);
  if (a_kmajor)
    (void)launch_k(dbias_k_kernel, blocks_for(M, 8), 256, 0, s, ap, lda, M, K, db);
  else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks_for(M, 64), kDbSplit, 1);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = kDbSplit;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    set_priority_attr(attr[2], s);
    cfg.attrs = attr;
    cfg.numAttrs = 3;
    (void)cudaLaunchKernelEx(&cfg, dbias_mn_kernel, ap, lda, M, K, db);
  }
  return check_launch("bias gradient");
}

int launch_colsum(int dtype, int rows, int cols, const void* y, int64_t ldy, float* out_acc, float* scratch,
                  cudaStream_t s) {
  if (rows < 1 || cols < 8 || cols % 8 || ldy % 8 || ldy < cols)
    return set_error(GPIPE_ERR_INVALID_ARG, "colsum: need rows >= 1, cols %% 8 == 0, ldy %% 8 == 0, ldy >= cols");
  if (!al16(y) || !al16(scratch)) return set_error(GPIPE_ERR_INVALID_ARG, "colsum: pointers must be 16-B aligned");
  const int chunks = (rows + kColRowsPerChunk - 1) / kColRowsPerChunk;
  dim3 grid(blocks_for(cols, 256 * 8), chunks);
  if (dtype == DT_F32)
    (void)launch_k(colsum_partial_kernel<float>, grid, 256, 0, s, static_cast<const float*>(y), ldy, rows, cols, scratch);
  else
    (void)launch_k(colsum_partial_kernel<__nv_bfloat16>, grid, 256, 0, s, static_cast<const __nv_bfloat16*>(y), ldy, rows,
                                                              cols, scratch);
  int rc = check_launch("colsum");
  if (rc) return rc;
  (void)launch_k(col_reduce_kernel, blocks_for(cols, 32), 32 * kColReduceWarps, 0, s, scratch, chunks, cols, out_acc,
                 cols, nullptr);
  return check_launch("colsum reduce");
}

int launch_cross_entropy(int rows, int vocab, int seq, const int32_t* tokens, int row0, float inv_count,
                         float* logits, float* loss_rows, int want_grad, cudaStream_t s, float clip) {
  if (rows < 1 || vocab < 4 || vocab % 4 || seq < 1 || row0 < 0)
    return set_error(GPIPE_ERR_INVALID_ARG, "cross_entropy: need rows >= 1, vocab %% 4 == 0, seq >= 1");
  if (!al16(logits)) return set_error(GPIPE_ERR_INVALID_ARG, "cross_entropy: logits must be 16-B aligned");
  if (!(clip >= 0.f)) return set_error(GPIPE_ERR_INVALID_ARG, "cross_entropy: clip must be >= 0 (0: none)");
  (void)launch_k(ce_kernel, rows, kCeThreads, 0, s, logits, vocab, seq, tokens, row0, inv_count, clip, loss_rows,
                 want_grad, device_error_ptr());
  return check_launch("cross_entropy");
}

int launch_mse(int rows, int d, const float* y, const float* t, float inv_count, float* loss_rows, float* dy,
               cudaStream_t s) {
  if (rows < 1 || d < 1) return set_error(GPIPE_ERR_INVALID_ARG, "mse: need rows, d >= 1");
  (void)launch_k(mse_kernel, blocks_for(rows, 8), 256, 0, s, y, t, rows, d, inv_count, loss_rows, dy);
  return check_launch("mse");
}

int launch_embedding_fwd_io(int out_dtype, int rows, int d, int vocab, const int32_t* tokens, const void* emb,
                            void* x, cudaStream_t s) {
  if (rows < 1 || d < 8 || d % 8 || vocab < 1 || !al16(emb) || !al16(x))
    return set_error(GPIPE_ERR_INVALID_ARG,
                     "embedding_fwd: need rows >= 1, d %% 8 == 0, vocab >= 1 and 16-B aligned rows");
  const int64_t n = (int64_t)rows * (d / 8);
  const __nv_bfloat16* e = static_cast<const __nv_bfloat16*>(emb);
  if (out_dtype == DT_F32)
    (void)launch_k(embed_fwd_kernel<float>, blocks_for(n, 256), 256, 0, s, rows, d, vocab, tokens, e,
                   static_cast<float*>(x), device_error_ptr());
  else
    (void)launch_k(embed_fwd_kernel<__nv_bfloat16>, blocks_for(n, 256), 256, 0, s, rows, d, vocab, tokens, e,
                   static_cast<__nv_bfloat16*>(x), device_error_ptr());
  return check_launch("embedding_fwd");
}

int launch_embedding_fwd(int rows, int d, int vocab, const int32_t* tokens, const void* emb, void* x,
                         cudaStream_t s) {
  return launch_embedding_fwd_io(DT_BF16, rows, d, vocab, tokens, emb, x, s);
}

int launch_embedding_bwd_io(int dx_dtype, int rows, int d, int vocab, const int32_t* tokens, const void* dx,
                            float* demb, cudaStream_t s) {
  if (rows < 1 || d < 8 || d % 8 || vocab < 1 || !al16(dx) || !al16(demb))
    return set_error(GPIPE_ERR_INVALID_ARG,
                     "embedding_bwd: need rows >= 1, d %% 8 == 0, vocab >= 1 and 16-B aligned rows");
  int ctas = 4 * num_sms();
  const int vpc = (vocab + ctas - 1) / ctas;
  ctas = (vocab + vpc - 1) / vpc;
  if (dx_dtype == DT_F32)
    (void)launch_k(embed_bwd_kernel<float>, ctas, 256, 0, s, rows, d, vocab, vpc, tokens, static_cast<const float*>(dx),
                   demb);
  else
    (void)launch_k(embed_bwd_kernel<__nv_bfloat16>, ctas, 256, 0, s, rows, d, vocab, vpc, tokens,
                   static_cast<const __nv_bfloat16*>(dx), demb);
  return check_launch("embedding_bwd");
}

int launch_embedding_bwd(int rows, int d, int vocab, const int32_t* tokens, const void* dx, float* demb,
                         cudaStream_t s) {
  return launch_embedding_bwd_io(DT_BF16, rows, d, vocab, tokens, dx, demb, s);
}

int launch_rmsprop(size_t n, float* w, float* g, float* v, void* wb, float lr, float decay, float eps,
                   int zero_grad, cudaStream_t s) {
  if (n == 0) return GPIPE_OK;
  if (!al16(w) || !al16(g) || !al16(v) || (wb && (reinterpret_cast<uintptr_t>(wb) & 7u)))
    return set_error(GPIPE_ERR_INVALID_ARG, "rmsprop: w, g, v must be 16-B aligned, w_bf16 8-B aligned");
  const int grid = std::min<int64_t>(blocks_for(n / 4 + 1, 256), (int64_t)num_sms() * 8);
  (void)launch_k(rmsprop_kernel, grid, 256, 0, s, w, g, v, static_cast<__nv_bfloat16*>(wb), n, lr, decay, eps, zero_grad);
  return check_launch("rmsprop");
}

int launch_cast_bf16(size_t n, const float* src, void* dst, cudaStream_t s) {
  if (n == 0) return GPIPE_OK;
  const int grid = std::min<int64_t>(blocks_for(n, 256), (int64_t)num_sms() * 8);
  (void)launch_k(cast_bf16_kernel, grid, 256, 0, s, src, static_cast<__nv_bfloat16*>(dst), n);
  return check_launch("cast_bf16");
}

int launch_sum(const float* x, size_t n, float* out, cudaStream_t s) {
  (void)launch_k(sum_kernel, 1, 1024, 0, s, x, n, out);
  return check_launch("sum");
}

int launch_stamp(unsigned long long* out, cudaStream_t s) {
  (void)launch_k(stamp_kernel, 1, 1, 0, s, out);
  return check_launch("stamp");
}

int launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (bytes % 16 || !al16(dst) || !al16(src))
    return set_error(GPIPE_ERR_INVALID_ARG, "copy: 16-B aligned buffers and sizes required");
  if (bytes == 0) return GPIPE_OK;
  const int grid = std::min<int64_t>(blocks_for(bytes / 16, 256), (int64_t)num_sms() * 8);
  (void)launch_k(copy_kernel, grid, 256, 0, s, static_cast<uint4*>(dst), static_cast<const uint4*>(src), bytes / 16);
  return check_launch("copy");
}

int launch_count_diff(const void* a, const void* b, size_t bytes, unsigned long long* counter, cudaStream_t s) {
  if (bytes % 4) return set_error(GPIPE_ERR_INVALID_ARG, "count_diff: size must be a multiple of 4");
  if (bytes == 0) return GPIPE_OK;
  const int grid = std::min<int64_t>(blocks_for(bytes / 4, 256), (int64_t)num_sms() * 8);
  (void)launch_k(count_diff_kernel, grid, 256, 0, s, static_cast<const uint32_t*>(a), static_cast<const uint32_t*>(b),
                                         bytes / 4, counter);
  return check_launch("count_diff");
}


// ---------------------------------------------------------------------------
// LayerNorm backward without caller-provided scratch.
//
// For callers that cannot allocate device memory at call time (for example a
// plugin whose host framework owns every byte of device memory through its
// own pool, or a latency-critical path that must not enter the CUDA
// allocator), the two-stage reduction's partial sums live in a fixed array in
// the library's device image instead of a caller buffer.  Every GPU that
// loads the library holds this array until the process exits.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocScratchFloats = size_t(1) << 20;  // 4 MiB of fp32 partial sums
static __device__ __align__(256) float g_ln_bwd_scratch[kNoAllocScratchFloats];
}  // namespace

size_t layernorm_bwd_noalloc_max_floats() { return kNoAllocScratchFloats; }

int launch_layernorm_bwd_noalloc(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                                 const float* rstd, const float* g, const void* dres, void* dx, float* dg_acc,
                                 float* db_acc, cudaStream_t s) {
  if (rows < 1 || d < 8 || d % 8 || d > 32 * 8 * kMaxChunks)
    return set_error(GPIPE_ERR_INVALID_ARG, "layernorm_bwd_noalloc: need rows >= 1, d %% 8 == 0, 8 <= d <= 1024");
  const size_t need = colred_scratch_floats(rows, 2 * d);
  if (need > kNoAllocScratchFloats)
    return set_error(GPIPE_ERR_INVALID_ARG,
                     "layernorm_bwd_noalloc: rows=%d, d=%d needs %zu scratch floats, more than the fixed %zu "
                     "(ceil(rows/8) * 2d must not exceed %zu)",
                     rows, d, need, kNoAllocScratchFloats, kNoAllocScratchFloats);
  // The array's host-side name is only a stand-in; its device address is
  // resolved on every call (no allocation, no stream work), so that a context
  // re-created after a device reset, whose module may sit elsewhere, is never
  // handed a stale address.
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_ln_bwd_scratch);
  if (e != cudaSuccess)
    return set_error(GPIPE_ERR_CUDA, "layernorm_bwd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
  float* scratch = static_cast<float*>(p);
  // Every partial row the reduction reads is written by this call, so nothing
  // needs clearing first.
  return launch_layernorm_bwd(dtype, rows, d, dy, x, mean, rstd, g, dres, dx, dg_acc, db_acc, scratch, s);
}

}  // namespace gp
