// Library-wide launch plumbing (error messages, the device error word, the
// launch counter, SM count) and the gpipe_op_* kernel-level C entry points.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/gpipe.h"
#include "../../include/gpipe_ops.h"
#include "common.cuh"
#include "kernels.h"
#include "launch_util.cuh"

namespace gp {

namespace {
thread_local std::string g_last_error = "no error";
int64_t g_launches = 0;
__device__ int g_device_error = 0;
}  // namespace

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

const char* last_error_message() { return g_last_error.c_str(); }

void count_launch(int n) { g_launches += n; }

namespace {
thread_local bool g_pdl = true;
}
bool pdl_enabled() { return g_pdl; }
void set_pdl_enabled(bool on) { g_pdl = on; }
int64_t launch_count() { return g_launches; }

// Per-device caches (a process may drive several devices from several host
// threads): resolved once per device under a lock, then read without one.
namespace {
constexpr int kMaxDevices = 256;
std::mutex g_dev_mu;
std::atomic<int*> g_err_ptr[kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];
int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}
}  // namespace

int* device_error_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  int* p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  p = g_err_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_device_error) != cudaSuccess) return nullptr;
    p = static_cast<int*>(q);
    g_err_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 1;
  int n = g_sms[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  g_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

int prepare_kernels() {
  int rc = prepare_gemm_tc();
  if (rc) return rc;
  rc = prepare_attention();
  if (rc) return rc;
  rc = prepare_layernorm();
  if (rc) return rc;
  if (!device_error_ptr()) return set_error(GPIPE_ERR_CUDA, "cannot resolve the device error flag");
  num_sms();
  return GPIPE_OK;
}

}  // namespace gp

using gp::set_error;

extern "C" {

namespace {
thread_local int g_op_sm_share = 0;
}

int gpipe_op_gemm_set_sm_share(int sms) {
  if (sms < 0) return gp::set_error(GPIPE_ERR_INVALID_ARG, "gemm SM share must be >= 0");
  g_op_sm_share = sms;
  return GPIPE_OK;
}

int gpipe_op_gemm(int dtype, int M, int N, int K, const void* A, int64_t lda, int a_kmajor, const void* B,
                  int64_t ldb, int b_kmajor, int epi, void* C, int64_t ldc, float* bias, const void* resid,
                  int64_t ldr, void* C2, const void* aux, int64_t ldaux, void* stream) {
  gp::GemmDesc g;
  g.dtype = dtype;
  g.M = M;
  g.N = N;
  g.K = K;
  g.A = A;
  g.lda = lda;
  g.a_kmajor = a_kmajor != 0;
  g.B = B;
  g.ldb = ldb;
  g.b_kmajor = b_kmajor != 0;
  g.epi = epi;
  g.C = C;
  g.ldc = ldc;
  if (epi == gp::EPI_ACC_F32) g.dbias = bias;  // bias-gradient accumulator
  else g.bias = bias;
  g.resid = resid;
  g.ldr = ldr;
  g.C2 = C2;
  g.aux = aux;
  g.ldaux = ldaux;
  g.sm_budget = g_op_sm_share;
  return gp::launch_gemm(g, static_cast<cudaStream_t>(stream));
}

size_t gpipe_op_scratch_bytes(int rows, int cols) {
  if (rows < 1 || cols < 1) return 0;
  return gp::colred_scratch_floats(rows, cols) * sizeof(float);
}

int gpipe_op_layernorm_fwd(int dtype, int rows, int d, const void* x, const float* g, const float* b, void* y,
                           float* mean, float* rstd, void* stream) {
  return gp::launch_layernorm_fwd(dtype, rows, d, x, g, b, y, mean, rstd, static_cast<cudaStream_t>(stream));
}

int gpipe_op_layernorm_bwd(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                           const float* rstd, const float* g, const void* dres, void* dx, float* dg_acc,
                           float* db_acc, float* scratch, void* stream) {
  return gp::launch_layernorm_bwd(dtype, rows, d, dy, x, mean, rstd, g, dres, dx, dg_acc, db_acc, scratch,
                                  static_cast<cudaStream_t>(stream));
}

int gpipe_op_layernorm_bwd_noalloc(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                                   const float* rstd, const float* g, const void* dres, void* dx, float* dg_acc,
                                   float* db_acc, void* stream) {
  return gp::launch_layernorm_bwd_noalloc(dtype, rows, d, dy, x, mean, rstd, g, dres, dx, dg_acc, db_acc,
                                          static_cast<cudaStream_t>(stream));
}

int gpipe_op_colsum(int dtype, int rows, int cols, const void* y, int64_t ldy, float* out_acc, float* scratch,
                    void* stream) {
  return gp::launch_colsum(dtype, rows, cols, y, ldy, out_acc, scratch, static_cast<cudaStream_t>(stream));
}

int gpipe_op_attention_fwd(int nseq, int seq, int heads, const void* qkv, void* o, float* lse, void* stream) {
  return gp::launch_attention_fwd(nseq, seq, heads, qkv, o, lse, static_cast<cudaStream_t>(stream));
}

int gpipe_op_attention_bwd(int nseq, int seq, int heads, const void* qkv, const void* o, const void* dout,
                           const float* lse, float* dvec, void* dqkv, void* stream) {
  return gp::launch_attention_bwd(nseq, seq, heads, qkv, o, dout, lse, dvec, dqkv,
                                  static_cast<cudaStream_t>(stream));
}

int gpipe_op_cross_entropy(int rows, int vocab, int seq, const int32_t* tokens, int row0, float inv_count,
                           float* logits, float* loss_rows, int want_grad, void* stream) {
  return gp::launch_cross_entropy(rows, vocab, seq, tokens, row0, inv_count, logits, loss_rows, want_grad,
                                  static_cast<cudaStream_t>(stream));
}

int gpipe_op_cross_entropy_clip(int rows, int vocab, int seq, const int32_t* tokens, int row0, float inv_count,
                                float clip, float* logits, float* loss_rows, int want_grad, void* stream) {
  return gp::launch_cross_entropy(rows, vocab, seq, tokens, row0, inv_count, logits, loss_rows, want_grad,
                                  static_cast<cudaStream_t>(stream), clip);
}

int gpipe_op_mse(int rows, int d, const float* y, const float* t, float inv_count, float* loss_rows, float* dy,
                 void* stream) {
  return gp::launch_mse(rows, d, y, t, inv_count, loss_rows, dy, static_cast<cudaStream_t>(stream));
}

int gpipe_op_embedding_fwd(int rows, int d, int vocab, const int32_t* tokens, const void* emb_bf16, void* x,
                           void* stream) {
  return gp::launch_embedding_fwd(rows, d, vocab, tokens, emb_bf16, x, static_cast<cudaStream_t>(stream));
}

int gpipe_op_embedding_bwd(int rows, int d, int vocab, const int32_t* tokens, const void* dx_bf16, float* demb,
                           void* stream) {
  return gp::launch_embedding_bwd(rows, d, vocab, tokens, dx_bf16, demb, static_cast<cudaStream_t>(stream));
}

int gpipe_op_rmsprop(size_t n, float* w, float* g, float* v, void* w_bf16, float lr, float decay, float eps,
                     int zero_grad, void* stream) {
  return gp::launch_rmsprop(n, w, g, v, w_bf16, lr, decay, eps, zero_grad, static_cast<cudaStream_t>(stream));
}

int gpipe_op_cast_bf16(size_t n, const float* src, void* dst, void* stream) {
  return gp::launch_cast_bf16(n, src, dst, static_cast<cudaStream_t>(stream));
}

int gpipe_op_wait_probe(void* stream) { return gp::launch_wait_probe(static_cast<cudaStream_t>(stream)); }

int gpipe_op_device_error(int* flag_out, int clear, void* stream) {
  if (!flag_out) return gp::set_error(GPIPE_ERR_INVALID_ARG, "device_error: NULL output");
  int* dev = gp::device_error_ptr();
  if (!dev) return gp::set_error(GPIPE_ERR_CUDA, "device_error: cannot resolve the device error word");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flag_out, dev, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(dev, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return gp::set_error(GPIPE_ERR_CUDA, "device_error: %s", cudaGetErrorString(e));
  return GPIPE_OK;
}

int gpipe_op_gelu(size_t n, const float* z_in, float* gelu, float* dgelu, void* stream) {
  return gp::launch_gelu(n, z_in, gelu, dgelu, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
