// Host-only dry run of the step executor (test infrastructure).
//
// Built by tests/test_dryrun_executor.py with g++ together with the library's
// own gpipe.cpp and planner.cpp, against the stand-in cuda_runtime.h of this
// folder.  The CUDA runtime calls the executor makes are implemented here as a
// log: stream work items, event records and event waits, in host issue order.
// The kernel launchers of kernels.h are implemented as log entries that list
// the byte ranges each kernel reads ('R'), writes ('W') or accumulates into
// ('A'; 'I' for an integer atomic count, whose order does not matter),
// computed from the launcher's documented arguments.  Nothing runs and
// no memory is touched: the addresses the test passes are never dereferenced.
// The test then checks every range against the buffers it passed (bounds) and
// every pair of conflicting accesses for a happens-before order (races).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "kernels.h"

struct CUstream_st {
  int id;
  int prio;
};
struct CUevent_st {
  int id;
};
struct CUgraph_st {
  int id;
};
struct CUgraphExec_st {
  int id;
};

namespace {

struct Access {
  uint64_t lo, hi;
  char mode;
};
struct Entry {
  int type;    // 0 work item, 1 event record, 2 event wait
  int stream;  // stream id (0: the legacy default stream)
  int event;   // event id for records and waits
  std::string name;
  std::vector<Access> acc;
};

std::vector<Entry> g_log;
int g_next_stream = 1, g_next_event = 1;
int g_sms = 152;
int64_t g_launches = 0;
bool g_pdl = false;
cudaStream_t g_capturing = nullptr;
thread_local std::string g_err = "no error";

int sid(cudaStream_t s) { return s ? s->id : 0; }

void work(cudaStream_t s, const char* name, std::vector<Access> acc) {
  g_log.push_back(Entry{0, sid(s), 0, name, std::move(acc)});
  ++g_launches;
}

Access rng(const void* p, uint64_t bytes, char mode) {
  const uint64_t lo = reinterpret_cast<uint64_t>(p);
  return Access{lo, lo + bytes, mode};
}
// A row-major rows x cols matrix with leading dimension ld (elements of es bytes).
Access mat(const void* p, int64_t rows, int64_t cols, int64_t ld, int es, char mode) {
  const uint64_t n = rows > 0 && cols > 0 ? static_cast<uint64_t>((rows - 1) * ld + cols) * es : 0;
  return rng(p, n, mode);
}

}  // namespace

// ---------------------------------------------------------------- runtime
const char* cudaGetErrorString(cudaError_t e) { return e == cudaSuccess ? "no error" : "dry-run error"; }
cudaError_t cudaGetDevice(int* dev) {
  *dev = 0;
  return cudaSuccess;
}
cudaError_t cudaDeviceGetStreamPriorityRange(int* least, int* greatest) {
  *least = 0;
  *greatest = -5;
  return cudaSuccess;
}
cudaError_t cudaStreamCreateWithFlags(cudaStream_t* s, unsigned) {
  *s = new CUstream_st{g_next_stream++, 0};
  return cudaSuccess;
}
cudaError_t cudaStreamCreateWithPriority(cudaStream_t* s, unsigned, int priority) {
  *s = new CUstream_st{g_next_stream++, priority};
  return cudaSuccess;
}
cudaError_t cudaStreamGetPriority(cudaStream_t s, int* priority) {
  *priority = s ? s->prio : 0;
  return cudaSuccess;
}
cudaError_t cudaStreamDestroy(cudaStream_t s) {
  delete s;
  return cudaSuccess;
}
cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }
cudaError_t cudaStreamWaitEvent(cudaStream_t s, cudaEvent_t e, unsigned) {
  g_log.push_back(Entry{2, sid(s), e->id, "wait", {}});
  return cudaSuccess;
}
cudaError_t cudaStreamBeginCapture(cudaStream_t s, cudaStreamCaptureMode) {
  g_capturing = s;
  return cudaSuccess;
}
cudaError_t cudaStreamEndCapture(cudaStream_t, cudaGraph_t* g) {
  g_capturing = nullptr;
  *g = new CUgraph_st{1};
  return cudaSuccess;
}
cudaError_t cudaStreamIsCapturing(cudaStream_t, cudaStreamCaptureStatus* status) {
  *status = g_capturing ? cudaStreamCaptureStatusActive : cudaStreamCaptureStatusNone;
  return cudaSuccess;
}
cudaError_t cudaEventCreate(cudaEvent_t* e) {
  *e = new CUevent_st{g_next_event++};
  return cudaSuccess;
}
cudaError_t cudaEventCreateWithFlags(cudaEvent_t* e, unsigned) { return cudaEventCreate(e); }
cudaError_t cudaEventDestroy(cudaEvent_t e) {
  delete e;
  return cudaSuccess;
}
cudaError_t cudaEventRecord(cudaEvent_t e, cudaStream_t s) {
  g_log.push_back(Entry{1, sid(s), e->id, "record", {}});
  return cudaSuccess;
}
cudaError_t cudaEventRecordWithFlags(cudaEvent_t e, cudaStream_t s, unsigned) { return cudaEventRecord(e, s); }
cudaError_t cudaEventSynchronize(cudaEvent_t) { return cudaSuccess; }
cudaError_t cudaEventElapsedTime(float* ms, cudaEvent_t, cudaEvent_t) {
  *ms = 0.f;
  return cudaSuccess;
}
cudaError_t cudaGraphInstantiate(cudaGraphExec_t* exec, cudaGraph_t, unsigned long long) {
  *exec = new CUgraphExec_st{1};
  return cudaSuccess;
}
cudaError_t cudaGraphLaunch(cudaGraphExec_t, cudaStream_t) { return cudaSuccess; }
cudaError_t cudaGraphDestroy(cudaGraph_t g) {
  delete g;
  return cudaSuccess;
}
cudaError_t cudaGraphExecDestroy(cudaGraphExec_t exec) {
  delete exec;
  return cudaSuccess;
}
cudaError_t cudaMemsetAsync(void* p, int, size_t bytes, cudaStream_t s) {
  work(s, "memset", {rng(p, bytes, 'W')});
  return cudaSuccess;
}
cudaError_t cudaMemcpyAsync(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
  std::vector<Access> a;
  if (kind == cudaMemcpyDeviceToHost || kind == cudaMemcpyDeviceToDevice) a.push_back(rng(src, bytes, 'R'));
  if (kind == cudaMemcpyHostToDevice || kind == cudaMemcpyDeviceToDevice) a.push_back(rng(dst, bytes, 'W'));
  work(s, "memcpy", a);
  return cudaSuccess;
}

// ---------------------------------------------------------------- launchers
namespace gp {

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}
const char* last_error_message() { return g_err.c_str(); }
int* device_error_ptr() {
  static int word;
  return &word;
}
void count_launch(int n) { g_launches += n; }
int64_t launch_count() { return g_launches; }
bool pdl_enabled() { return g_pdl; }
void set_pdl_enabled(bool on) { g_pdl = on; }
int prepare_kernels() { return 0; }
int num_sms() { return g_sms; }

int launch_gemm(const GemmDesc& g, cudaStream_t s) {
  const int es = g.dtype == DT_BF16 ? 2 : 4;
  const bool f32_out = g.epi == EPI_ACC_F32 || g.epi == EPI_STORE_F32 || g.epi == EPI_RESID_F32;
  std::vector<Access> a;
  a.push_back(g.a_kmajor ? mat(g.A, g.M, g.K, g.lda, es, 'R') : mat(g.A, g.K, g.M, g.lda, es, 'R'));
  a.push_back(g.b_kmajor ? mat(g.B, g.N, g.K, g.ldb, es, 'R') : mat(g.B, g.K, g.N, g.ldb, es, 'R'));
  a.push_back(mat(g.C, g.M, g.N, g.ldc, f32_out ? 4 : es, g.epi == EPI_ACC_F32 ? 'A' : 'W'));
  if (g.bias) a.push_back(rng(g.bias, static_cast<uint64_t>(g.N) * 4, 'R'));
  if (g.dbias) a.push_back(rng(g.dbias, static_cast<uint64_t>(g.M) * 4, 'A'));
  if (g.resid) a.push_back(mat(g.resid, g.M, g.N, g.ldr, g.epi == EPI_RESID_F32 ? 4 : es, 'R'));
  if (g.C2) a.push_back(mat(g.C2, g.M, g.N, g.ldc, es, 'W'));
  if (g.aux) a.push_back(mat(g.aux, g.M, g.N, g.ldaux, es, 'R'));
  const std::string name = "gemm:" + std::to_string(g.M) + ":" + std::to_string(g.N) + ":" + std::to_string(g.K);
  work(s, name.c_str(), a);
  return 0;
}

int launch_layernorm_fwd_io(int in_dtype, int out_dtype, int rows, int d, const void* x, const float* g,
                            const float* b, void* y, float* mean, float* rstd, cudaStream_t s) {
  const uint64_t n = static_cast<uint64_t>(rows) * d;
  const int ei = in_dtype == DT_BF16 ? 2 : 4, eo = out_dtype == DT_BF16 ? 2 : 4;
  work(s, "layernorm_fwd",
       {rng(x, n * ei, 'R'), rng(g, d * 4ull, 'R'), rng(b, d * 4ull, 'R'), rng(y, n * eo, 'W'),
        rng(mean, rows * 4ull, 'W'), rng(rstd, rows * 4ull, 'W')});
  return 0;
}

int launch_layernorm_fwd(int dtype, int rows, int d, const void* x, const float* g, const float* b, void* y,
                         float* mean, float* rstd, cudaStream_t s) {
  return launch_layernorm_fwd_io(dtype, dtype, rows, d, x, g, b, y, mean, rstd, s);
}

int launch_layernorm_bwd_rows_io(int dy_dtype, int x_dtype, int out_dtype, int rows, int d, const void* dy,
                                 const void* x, const float* mean, const float* rstd, const float* g, const void* dres,
                                 void* dx, void* dx16, float* scratch, cudaStream_t s) {
  const uint64_t n = static_cast<uint64_t>(rows) * d;
  const int ed = dy_dtype == DT_BF16 ? 2 : 4, ex = x_dtype == DT_BF16 ? 2 : 4, eo = out_dtype == DT_BF16 ? 2 : 4;
  std::vector<Access> a{rng(dy, n * ed, 'R'),        rng(x, n * ex, 'R'),     rng(mean, rows * 4ull, 'R'),
                        rng(rstd, rows * 4ull, 'R'), rng(g, d * 4ull, 'R'), rng(dx, n * eo, 'W'),
                        rng(scratch, static_cast<uint64_t>((rows + 7) / 8) * 2 * d * 4, 'W')};
  if (dres) a.push_back(rng(dres, n * eo, 'R'));
  if (dx16) a.push_back(rng(dx16, n * 2, 'W'));
  work(s, "layernorm_bwd_rows", a);
  return 0;
}

int launch_layernorm_bwd_rows(int dtype, int rows, int d, const void* dy, const void* x, const float* mean,
                              const float* rstd, const float* g, const void* dres, void* dx, float* scratch,
                              cudaStream_t s) {
  return launch_layernorm_bwd_rows_io(dtype, dtype, dtype, rows, d, dy, x, mean, rstd, g, dres, dx, nullptr, scratch,
                                      s);
}

int launch_layernorm_bwd_reduce(int rows, int d, const float* scratch, float* dg, float* db, cudaStream_t s) {
  work(s, "layernorm_bwd_reduce",
       {rng(scratch, static_cast<uint64_t>((rows + 7) / 8) * 2 * d * 4, 'R'), rng(dg, d * 4ull, 'A'),
        rng(db, d * 4ull, 'A')});
  return 0;
}

int launch_attention_fwd(int nseq, int seq, int heads, const void* qkv, void* o, float* lse, cudaStream_t s) {
  const uint64_t T = static_cast<uint64_t>(nseq) * seq, d = static_cast<uint64_t>(heads) * 64;
  work(s, "attention_fwd", {rng(qkv, T * 3 * d * 2, 'R'), rng(o, T * d * 2, 'W'), rng(lse, T * heads * 4, 'W')});
  return 0;
}

int launch_attention_bwd(int nseq, int seq, int heads, const void* qkv, const void* o, const void* dout,
                         const float* lse, float* dvec, void* dqkv, cudaStream_t s) {
  const uint64_t T = static_cast<uint64_t>(nseq) * seq, d = static_cast<uint64_t>(heads) * 64;
  work(s, "attention_bwd",
       {rng(qkv, T * 3 * d * 2, 'R'), rng(o, T * d * 2, 'R'), rng(dout, T * d * 2, 'R'), rng(lse, T * heads * 4, 'R'),
        rng(dvec, T * heads * 4, 'W'), rng(dqkv, T * 3 * d * 2, 'W')});
  return 0;
}

int launch_cross_entropy(int rows, int vocab, int, const int32_t* tokens, int row0, float, float* logits,
                         float* loss_rows, int, cudaStream_t s, float) {
  work(s, "cross_entropy",
       {rng(tokens + row0, rows * 4ull, 'R'), rng(logits, static_cast<uint64_t>(rows) * vocab * 4, 'W'),
        rng(loss_rows, rows * 4ull, 'W')});
  return 0;
}

int launch_mse(int rows, int d, const float* y, const float* t, float, float* loss_rows, float* dy, cudaStream_t s) {
  const uint64_t n = static_cast<uint64_t>(rows) * d * 4;
  work(s, "mse", {rng(y, n, 'R'), rng(t, n, 'R'), rng(loss_rows, rows * 4ull, 'W'), rng(dy, n, 'W')});
  return 0;
}

int launch_embedding_fwd_io(int out_dtype, int rows, int d, int vocab, const int32_t* tokens, const void* emb, void* x,
                            cudaStream_t s) {
  work(s, "embedding_fwd",
       {rng(tokens, rows * 4ull, 'R'), rng(emb, static_cast<uint64_t>(vocab) * d * 2, 'R'),
        rng(x, static_cast<uint64_t>(rows) * d * (out_dtype == DT_BF16 ? 2 : 4), 'W')});
  return 0;
}

int launch_embedding_fwd(int rows, int d, int vocab, const int32_t* tokens, const void* emb, void* x,
                         cudaStream_t s) {
  return launch_embedding_fwd_io(DT_BF16, rows, d, vocab, tokens, emb, x, s);
}

int launch_embedding_bwd_io(int dx_dtype, int rows, int d, int vocab, const int32_t* tokens, const void* dx,
                            float* demb, cudaStream_t s) {
  work(s, "embedding_bwd",
       {rng(tokens, rows * 4ull, 'R'), rng(dx, static_cast<uint64_t>(rows) * d * (dx_dtype == DT_BF16 ? 2 : 4), 'R'),
        rng(demb, static_cast<uint64_t>(vocab) * d * 4, 'A')});
  return 0;
}

int launch_embedding_bwd(int rows, int d, int vocab, const int32_t* tokens, const void* dx, float* demb,
                         cudaStream_t s) {
  return launch_embedding_bwd_io(DT_BF16, rows, d, vocab, tokens, dx, demb, s);
}

int launch_rmsprop(size_t n, float* w, float* g, float* v, void* w16, float, float, float, int, cudaStream_t s) {
  std::vector<Access> a{rng(w, n * 4, 'W'), rng(g, n * 4, 'W'), rng(v, n * 4, 'W')};
  if (w16) a.push_back(rng(w16, n * 2, 'W'));
  work(s, "rmsprop", a);
  return 0;
}

int launch_cast_bf16(size_t n, const float* src, void* dst, cudaStream_t s) {
  work(s, "cast_bf16", {rng(src, n * 4, 'R'), rng(dst, n * 2, 'W')});
  return 0;
}

int launch_sum(const float* x, size_t n, float* out, cudaStream_t s) {
  work(s, "sum", {rng(x, n * 4, 'R'), rng(out, 4, 'W')});
  return 0;
}

int launch_stamp(unsigned long long* out, cudaStream_t s) {
  work(s, "stamp", {rng(out, 8, 'W')});
  return 0;
}

int launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  work(s, "copy", {rng(src, bytes, 'R'), rng(dst, bytes, 'W')});
  return 0;
}

int launch_count_diff(const void* a, const void* b, size_t bytes, unsigned long long* counter, cudaStream_t s) {
  work(s, "count_diff", {rng(a, bytes, 'R'), rng(b, bytes, 'R'), rng(counter, 8, 'I')});
  return 0;
}

}  // namespace gp

// ---------------------------------------------------------------- log access
extern "C" {

void dry_reset() {
  g_log.clear();
  g_launches = 0;
}
void dry_set_sms(int n) { g_sms = n; }
int dry_entries() { return static_cast<int>(g_log.size()); }
// Entry i: type, stream, event, number of accesses; its name into name (cap bytes).
int dry_entry(int i, int* type, int* stream, int* event, int* nacc, char* name, int cap) {
  if (i < 0 || i >= static_cast<int>(g_log.size())) return -1;
  const Entry& e = g_log[i];
  *type = e.type;
  *stream = e.stream;
  *event = e.event;
  *nacc = static_cast<int>(e.acc.size());
  std::snprintf(name, cap, "%s", e.name.c_str());
  return 0;
}
int dry_access(int i, int j, uint64_t* lo, uint64_t* hi, char* mode) {
  if (i < 0 || i >= static_cast<int>(g_log.size()) || j < 0 || j >= static_cast<int>(g_log[i].acc.size())) return -1;
  const Access& a = g_log[i].acc[j];
  *lo = a.lo;
  *hi = a.hi;
  *mode = a.mode;
  return 0;
}

}  // extern "C"
