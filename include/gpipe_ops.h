/*
 * gpipe_ops.h - kernel-level entry points of libgpipe.
 *
 * Each call enqueues the kernel(s) of one operation of the GPipe step on
 * `stream` (a cudaStream_t passed as void*; NULL = legacy default stream) and
 * returns 0 or a negative GPIPE_ERR_* code from gpipe.h without launching on
 * invalid arguments.  All pointers are caller-owned device addresses unless
 * stated; nothing is allocated or freed.  They exist so that every kernel the
 * step uses can be checked on its own; gpipe_step calls the same launchers.
 * The operations are the pieces of the step of "GPipe technical review"
 * (zzz0906.github.io), section "Pipeline flow": the layers' forward and
 * backward, the loss, the gradient accumulation and the RMSProp update
 * ("Preliminaries 2: the memory wall").
 *
 * dtype: 0 = fp32 operands/activations, 1 = bf16 operands/activations (fp32
 * accumulation and fp32 statistics in both cases).
 */
#ifndef GPIPE_OPS_H
#define GPIPE_OPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  GPIPE_EPI_STORE = 0,     /* C = acc (+ bias[n]) (+ resid[m,n])                  */
  GPIPE_EPI_BIAS_GELU = 1, /* C = z = acc + bias[n];  C2 = GELU(z)  (exact erf)    */
  GPIPE_EPI_GELU_BWD = 2,  /* C = acc * GELU'(aux[m,n])                              */
  GPIPE_EPI_ACC_F32 = 3,   /* C (fp32) += acc                                        */
  GPIPE_EPI_STORE_F32 = 4, /* C (fp32) = acc                                         */
  GPIPE_EPI_RESID_F32 = 5  /* C (fp32) = (acc + bias[n]) + resid (fp32)[m,n]         */
};

/* C[m,n] = epilogue( sum_k A(m,k) B(n,k) ), 0 <= m < M, 0 <= n < N.
 * A(m,k) = A[m*lda + k] when a_kmajor, else A[k*lda + m];
 * B(n,k) = B[n*ldb + k] when b_kmajor, else B[k*ldb + n].
 * So x W^T (W [out,in]) is (a_kmajor=1, b_kmajor=1); dY W is (1, 0); the weight
 * gradient dY^T X is (0, 0).  C, C2, resid and aux are row-major with leading
 * dimension ldc (C, C2), ldr (resid), ldaux (aux); element type = dtype except
 * for the fp32 epilogues.  bias is fp32 [N] (read) or NULL for the forward
 * epilogues; for GPIPE_EPI_ACC_F32 a non-NULL bias is an fp32 [M] accumulator
 * that receives += sum_k A(m,k) (the bias gradient that goes with a weight
 * gradient dY^T X, computed by the same launch).  resid may be NULL.
 * dtype 1 runs the tcgen05/TMEM tensor-core kernel fed by TMA and needs every
 * leading dimension a multiple of 8 elements and 16-byte aligned bases; it is
 * built for (1,1) with STORE, BIAS_GELU, STORE_F32, ACC_F32, RESID_F32 (resid
 * required, fp32 like C); (1,0) with STORE,
 * GELU_BWD, ACC_F32; (0,0) with STORE, ACC_F32 (others: GPIPE_ERR_UNSUPPORTED).
 * dtype 0 runs an fp32 FFMA kernel (any layout and epilogue).
 * Requires M, N, K >= 1. */
int gpipe_op_gemm(int dtype, int M, int N, int K,
                  const void* A, int64_t lda, int a_kmajor,
                  const void* B, int64_t ldb, int b_kmajor,
                  int epi, void* C, int64_t ldc,
                  float* bias, const void* resid, int64_t ldr,
                  void* C2, const void* aux, int64_t ldaux, void* stream);

/* SM share of the GEMMs this host thread launches through gpipe_op_gemm from
 * now on: sms > 0 sizes their grids (and so the tile width and kernel) as the
 * step does for a GEMM given that many SMs; 0 (the default) gives each the
 * whole GPU.  Returns 0, or GPIPE_ERR_INVALID_ARG for sms < 0. */
int gpipe_op_gemm_set_sm_share(int sms);

/* Bytes of fp32 scratch the two-stage column reductions below need. */
size_t gpipe_op_scratch_bytes(int rows, int cols);

/* LayerNorm over rows of width d (eps 1e-5, biased variance):
 * y = (x - mean) * rstd * g + b; mean and rstd (fp32 [rows]) are saved.
 * d must be a multiple of 8 and at most 1024 (GPIPE_ERR_INVALID_ARG otherwise). */
int gpipe_op_layernorm_fwd(int dtype, int rows, int d, const void* x, const float* g,
                           const float* b, void* y, float* mean, float* rstd, void* stream);

/* LayerNorm backward: dx = rstd (g dy - mean(g dy) - xhat mean(g dy xhat)) + dres
 * (dres may be NULL); dg_acc += sum_rows dy xhat and db_acc += sum_rows dy,
 * accumulated in a fixed order (two stages through `scratch`, of
 * gpipe_op_scratch_bytes(rows, 2*d) bytes). */
int gpipe_op_layernorm_bwd(int dtype, int rows, int d, const void* dy, const void* x,
                           const float* mean, const float* rstd, const float* g,
                           const void* dres, void* dx, float* dg_acc, float* db_acc,
                           float* scratch, void* stream);

/* The same LayerNorm backward for callers that cannot allocate device memory
 * when they call it: for instance a plugin inside a host framework that owns
 * all device memory through its own pool, or a latency-critical path that must
 * never enter the CUDA allocator.  The paper has no counterpart; this is a
 * convenience of this library.  Instead of a caller `scratch` buffer it uses a
 * fixed array of 2^20 floats (4 MiB) inside the library's device image, which
 * every GPU that loads the library keeps until the process exits; it calls no
 * allocation routine.  Limit: ceil(rows / 8) * 2 * d <= 2^20 (for d = 1024,
 * rows <= 4096); larger sizes return GPIPE_ERR_INVALID_ARG with a message.
 * Every call looks up the array's device address in the current context (no
 * allocation and no stream work), so a context re-created after
 * cudaDeviceReset is served correctly; the first lookup on a device may load
 * the library's device image, so make the first call before any stream
 * capture.  All calls
 * share the one array: every partial sum the call reads is written by the
 * same call, so nothing needs clearing, but calls that overlap on the GPU (on
 * different streams, or from different threads) race on it. */
int gpipe_op_layernorm_bwd_noalloc(int dtype, int rows, int d, const void* dy, const void* x,
                                   const float* mean, const float* rstd, const float* g,
                                   const void* dres, void* dx, float* dg_acc, float* db_acc,
                                   void* stream);

/* out_acc[c] += sum_r y[r*ldy + c] in a fixed order (bias gradients); scratch
 * of gpipe_op_scratch_bytes(rows, cols) bytes. cols % 8 == 0, ldy % 8 == 0. */
int gpipe_op_colsum(int dtype, int rows, int cols, const void* y, int64_t ldy,
                    float* out_acc, float* scratch, void* stream);

/* Causal multi-head attention forward, bf16, head width 64, scale 1/8, on
 * the tcgen05 tensor cores (S and O accumulate in tensor memory).
 * qkv [nseq*seq, 3*heads*64] (query | key | value column blocks), output
 * o [nseq*seq, heads*64], lse [nseq*seq, heads] fp32 natural-log
 * log-sum-exp of the scaled scores.  seq % 64 == 0, nseq * seq <= 2^30. */
int gpipe_op_attention_fwd(int nseq, int seq, int heads, const void* qkv, void* o,
                           float* lse, void* stream);

/* Backward: dqkv [nseq*seq, 3*heads*64] gets dQ | dK | dV.  dvec is fp32
 * [nseq*seq, heads]: rowsum(dO o O), written first by a small kernel, then
 * read by one launch whose dQ blocks and dK/dV blocks run side by side; no
 * atomics, so results are bit-reproducible.  nseq <= 32767. */
int gpipe_op_attention_bwd(int nseq, int seq, int heads, const void* qkv, const void* o,
                           const void* dout, const float* lse, float* dvec, void* dqkv,
                           void* stream);

/* Next-token softmax cross-entropy on fp32 logits [rows, vocab].
 * Row r is token row0 + r of the mini-batch (tokens [N*seq] int32); its target
 * is tokens[row0 + r + 1] unless (row0 + r) % seq == seq - 1 (no target).
 * loss_rows[r] = (lse - z_target) * inv_count (0 without target).
 * want_grad: writes dz = (softmax - onehot) * inv_count as bf16 IN PLACE over
 * the logits, row r at bf16 offset r * 2 * vocab (so the gradient matrix has
 * leading dimension 2*vocab bf16 elements).  vocab % 4 == 0.  A target id
 * outside [0, vocab) is treated as "no target" and sets the device error flag. */
int gpipe_op_cross_entropy(int rows, int vocab, int seq, const int32_t* tokens, int row0,
                           float inv_count, float* logits, float* loss_rows, int want_grad,
                           void* stream);

/* The same with logit clipping ("GPipe technical review", "Training
 * stability": logits above a threshold are clipped before the softmax).
 * clip > 0: the softmax and the target term see min(max(z, -clip), clip), and
 * dz is zero where |z| > clip (the clamp's derivative; a NaN logit stays NaN in
 * the loss).  clip = 0: no clipping, exactly gpipe_op_cross_entropy.  A
 * negative or NaN clip is rejected (GPIPE_ERR_INVALID_ARG). */
int gpipe_op_cross_entropy_clip(int rows, int vocab, int seq, const int32_t* tokens, int row0,
                                float inv_count, float clip, float* logits, float* loss_rows,
                                int want_grad, void* stream);

/* MSE rows: loss_rows[r] = sum_j (y - t)^2 * inv_count; dy = 2 (y - t) inv_count. */
int gpipe_op_mse(int rows, int d, const float* y, const float* t, float inv_count,
                 float* loss_rows, float* dy, void* stream);

/* x[r,:] = emb[tokens[r],:] (bf16 rows of width d, d % 8 == 0, vocab rows).
 * A token id outside [0, vocab) gives a zero row and sets the device error
 * flag (read by gpipe_debug_counters) instead of reading out of bounds. */
int gpipe_op_embedding_fwd(int rows, int d, int vocab, const int32_t* tokens, const void* emb_bf16,
                           void* x, void* stream);

/* demb[tokens[r],:] += dx[r,:] (fp32 accumulator, bf16 dx).  Deterministic: each
 * embedding row is owned by one CTA, which adds its tokens in ascending r. */
int gpipe_op_embedding_bwd(int rows, int d, int vocab, const int32_t* tokens,
                           const void* dx_bf16, float* demb, void* stream);

/* RMSProp over n parameters: v = decay v + (1-decay) g^2; w -= lr g/(sqrt(v)+eps);
 * w_bf16 (may be NULL) receives the round-to-nearest-even bf16 copy of w;
 * zero_grad != 0 sets g = 0 afterwards. */
int gpipe_op_rmsprop(size_t n, float* w, float* g, float* v, void* w_bf16, float lr,
                     float decay, float eps, int zero_grad, void* stream);

/* dst[i] = bf16(src[i]) (round to nearest even). */
int gpipe_op_cast_bf16(size_t n, const float* src, void* dst, void* stream);

/* Failure detection.  Every wait of the library's kernels on another part of
 * the GPU is bounded (2 s); one that gives up, or a kernel that meets an
 * invalid input it skips (a token id outside [0, vocab)), sets the device error
 * word of the current device: 1-4 a bounded wait (TMA producer, MMA issuer,
 * epilogue, exit drain), 5 an invalid token id, 6 this probe, 7 a kernel whose
 * shared memory was less aligned than its swizzled tiles need (its work is
 * skipped).
 *   gpipe_op_wait_probe: launches one CTA whose bounded wait on an mbarrier
 *     that nothing completes gives up after the limit and sets code 6; the
 *     kernel returns normally and the context stays usable.
 *   gpipe_op_device_error: copies the word to *flag_out (synchronises
 *     `stream`); clear != 0 resets it to 0 afterwards. */
int gpipe_op_wait_probe(void* stream);
int gpipe_op_device_error(int* flag_out, int clear, void* stream);

/* The GELU arithmetic of the GEMM epilogues, in fp32 (for checking it):
 * gelu[i] = z Phi(z) and dgelu[i] = Phi(z) + z phi(z) for z = z_in[i] (exact-erf
 * GELU as the review's Transformer uses it; erf evaluated to within 1.5e-7, see
 * the kernels).  Either output may be NULL. */
int gpipe_op_gelu(size_t n, const float* z_in, float* gelu, float* dgelu, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GPIPE_OPS_H */
