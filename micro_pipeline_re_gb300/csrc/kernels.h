// Host-side declarations of the kernel launchers (one per operation of the
// step).  Every launcher validates its arguments, enqueues on `stream` and
// returns 0 or a negative GPIPE_ERR_* code, recording a message with
// set_error().  The step executor and the gpipe_op_* entry points call these.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gp {

enum { DT_F32 = 0, DT_BF16 = 1 };
// EPI_RESID_F32: C(fp32) = acc + bias[n] + resid(fp32)[m, n], the step's
// residual adds, which keep the residual stream in fp32.
enum { EPI_STORE = 0, EPI_BIAS_GELU = 1, EPI_GELU_BWD = 2, EPI_ACC_F32 = 3, EPI_STORE_F32 = 4, EPI_RESID_F32 = 5 };

// Error reporting (thread-local message; see launch.cu).
int set_error(int code, const char* fmt, ...);
const char* last_error_message();

// Device address of the library's error word (set by bounded device waits
// that give up; see common.cuh).
int* device_error_ptr();

// Counts kernel launches made through the launchers (host side).
void count_launch(int n = 1);
int64_t launch_count();

struct GemmDesc {
  int dtype = DT_BF16;
  int M = 0, N = 0, K = 0;
  const void* A = nullptr;
  int64_t lda = 0;
  bool a_kmajor = true;
  const void* B = nullptr;
  int64_t ldb = 0;
  bool b_kmajor = true;
  int epi = EPI_STORE;
  void* C = nullptr;
  int64_t ldc = 0;
  const float* bias = nullptr;  // forward epilogues: fp32 [N]
  float* dbias = nullptr;        // EPI_ACC_F32: fp32 [M] accumulator, += sum_k A(m,k)
  const void* resid = nullptr;
  int64_t ldr = 0;
  void* C2 = nullptr;
  const void* aux = nullptr;
  int64_t ldaux = 0;
  int sm_budget = 0;  // SMs this GEMM may expect to itself (0: all); picks tile width and split-K
};

int launch_gemm(const GemmDesc& g, cudaStream_t stream);       // dispatch by dtype
int launch_gemm_tc(const GemmDesc& g, cudaStream_t stream);    // bf16, tcgen05 + TMA
int launch_gemm_simt(const GemmDesc& g, cudaStream_t stream);  // fp32 or bf16, FFMA
// Persistent tcgen05 GEMM (one CTA per SM over many tiles, two TMEM
// accumulators); `ctas` caps the grid.  persistent_tiles: its tile count.
int launch_gemm_persistent(const GemmDesc& g, cudaStream_t stream, int ctas);
bool wide_bias_grad_gemm(const GemmDesc& g);
int64_t persistent_tiles(const GemmDesc& g);
int prepare_gemm_persistent();

size_t colred_scratch_floats(int rows, int cols);

int launch_layernorm_fwd(int dtype, int rows, int d, const void* x, const float* g, const float* b, void* y,
                         float* mean, float* rstd, cudaStream_t stream);
// The same with separate input and output element types: the step reads the
// fp32 residual stream and writes the bf16 GEMM operand (fp32 -> bf16;
// fp32 -> fp32 and bf16 -> bf16 as above).
int launch_layernorm_fwd_io(int in_dtype, int out_dtype, int rows, int d, const void* x, const float* g,
                            const float* b, void* y, float* mean, float* rstd, cudaStream_t stream);
// LayerNorm backward in two launches: the rows (dx, and one partial row of the
// gamma/beta column sums per 8 rows into scratch), then the fixed-order
// reduction of the partials into dg_acc / db_acc (+=).
int launch_layernorm_bwd_rows(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                              const float* rstd, const float* g, const void* dres, void* dx, float* scratch,
                              cudaStream_t s);
// The same with dy of dy_dtype, x of x_dtype, and dres and dx of out_dtype;
// dx16 (may be NULL) receives a bf16 copy of dx.  The step: a bf16 GEMM output
// dy, the fp32 residual stream x, the fp32 residual gradient dres -> dx in
// fp32 (the residual gradient stream) and in bf16 (the next GEMMs' operand).
int launch_layernorm_bwd_rows_io(int dy_dtype, int x_dtype, int out_dtype, int rows, int d, const void* dy,
                                 const void* x, const float* mean, const float* rstd, const float* g, const void* dres,
                                 void* dx, void* dx16, float* scratch, cudaStream_t s);
int launch_gelu(size_t n, const float* z, float* y, float* dy, cudaStream_t s);
// One CTA whose bounded wait on an mbarrier nothing completes gives up and
// sets the device error word (code 6): checks the failure path without a fault.
int launch_wait_probe(cudaStream_t s);
// db[m] += sum_k A(m, k) for a bf16 A, K-major ([M][K]) or MN-major ([K][M]);
// one launch, fixed order (the bias gradient of the wide weight-gradient GEMMs).
int launch_dbias(bool a_kmajor, int M, int K, const void* a, int64_t lda, float* db, cudaStream_t s);
int launch_layernorm_bwd_reduce(int rows, int d, const float* scratch, float* dg_acc, float* db_acc, cudaStream_t s);
int launch_layernorm_bwd(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                         const float* rstd, const float* g, const void* dres, void* dx, float* dg_acc,
                         float* db_acc, float* scratch, cudaStream_t stream);
// LayerNorm backward whose reduction scratch is a fixed static device array
// (no caller scratch); rejects sizes beyond layernorm_bwd_noalloc_max_floats().
int launch_layernorm_bwd_noalloc(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                                 const float* rstd, const float* g, const void* dres, void* dx, float* dg_acc,
                                 float* db_acc, cudaStream_t stream);
size_t layernorm_bwd_noalloc_max_floats();
int launch_colsum(int dtype, int rows, int cols, const void* y, int64_t ldy, float* out_acc, float* scratch,
                  cudaStream_t stream);

int launch_attention_fwd(int nseq, int seq, int heads, const void* qkv, void* o, float* lse, cudaStream_t stream);
int launch_attention_bwd(int nseq, int seq, int heads, const void* qkv, const void* o, const void* dout,
                         const float* lse, float* dvec, void* dqkv, cudaStream_t stream);

int launch_cross_entropy(int rows, int vocab, int seq, const int32_t* tokens, int row0, float inv_count,
                         float* logits, float* loss_rows, int want_grad, cudaStream_t stream, float clip = 0.f);
int launch_mse(int rows, int d, const float* y, const float* t, float inv_count, float* loss_rows, float* dy,
               cudaStream_t stream);

int launch_embedding_fwd(int rows, int d, int vocab, const int32_t* tokens, const void* emb_bf16, void* x,
                         cudaStream_t stream);
int launch_embedding_bwd(int rows, int d, int vocab, const int32_t* tokens, const void* dx_bf16, float* demb,
                         cudaStream_t stream);
// The same with the residual stream's element type (x written, dx read) given.
int launch_embedding_fwd_io(int out_dtype, int rows, int d, int vocab, const int32_t* tokens, const void* emb_bf16,
                            void* x, cudaStream_t stream);
int launch_embedding_bwd_io(int dx_dtype, int rows, int d, int vocab, const int32_t* tokens, const void* dx,
                            float* demb, cudaStream_t stream);

int launch_rmsprop(size_t n, float* w, float* g, float* v, void* w_bf16, float lr, float decay, float eps,
                   int zero_grad, cudaStream_t stream);
int launch_cast_bf16(size_t n, const float* src, void* dst, cudaStream_t stream);

// Deterministic sum of n floats into *out (one block, fixed order, fp64 partials).
int launch_sum(const float* x, size_t n, float* out, cudaStream_t stream);
// *out = the GPU's nanosecond clock (one thread), for tracing.
int launch_stamp(unsigned long long* out, cudaStream_t stream);
// Copy n bytes (device to device) with a kernel.
int launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t stream);
// counter[0] += number of bytes that differ between a and b.
int launch_count_diff(const void* a, const void* b, size_t bytes, unsigned long long* counter,
                      cudaStream_t stream);

// Sets the shared-memory attributes of every kernel that needs more than the
// default and resolves driver entry points, outside any stream capture.
int prepare_kernels();
int prepare_gemm_tc();
int prepare_attention();
int prepare_layernorm();

// Number of SMs of the current device (cached).
int num_sms();

}  // namespace gp
