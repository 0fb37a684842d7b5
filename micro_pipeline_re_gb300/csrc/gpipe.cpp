// Step executor and the gpipe_* C ABI.
//
// One synchronous GPipe step ("GPipe technical review", zzz0906.github.io,
// "Pipeline flow", phases 1-3) with all K cells on one GPU:
//   phase 1  for m in 0..M-1, for k in 0..K-1: cell k forwards micro-batch m
//            from the stashed cell input stash[k][m] and writes its output to
//            stash[k+1][m]; the cell's internals go to its lane's slots and
//            are overwritten by the next micro-batch (re-materialisation keeps
//            only the boundary activations).  Then the head (final LN, tied
//            logits, cross-entropy; MSE for the FFN model) computes micro-batch
//            m's loss and the gradient of the last cell's output, once.
//   phase 2  for m in 0..M-1, for k in K-1..0: re-compute cell k's forward
//            from stash[k][m] (its last layer's output projection is skipped:
//            that output is already stashed and not needed to differentiate
//            the cell), then differentiate it layer by layer in reverse; weight
//            gradients are added into the fp32 gradient buffer straight from
//            the GEMM epilogue (accumulation across micro-batches, no update in
//            between).
//   phase 3  the tied embedding's scatter-add for all tokens, then one RMSProp
//            update of every parameter (and the bf16 copy).
// The review's K accelerators become K concurrent lanes (a main and a side
// stream each, plus one lane for the head): cell k works on micro-batch m while
// cell k+1 works on m-1, with events carrying exactly the pipeline's
// dependencies; weight-gradient GEMMs run on each lane's side stream.  Each
// cell's gradient accumulation stays in micro-batch order on one stream, so the
// result is bit-identical to running the cells in turn on one stream
// (GPIPE_OPT_PIPELINE / GPIPE_OPT_CONCURRENT = 0).  GPIPE_OPT_SCHEDULE 1
// issues the same operations in the one-forward-one-backward order (each cell
// alternates forwards and backwards after a short warm-up), so a cell boundary
// is stashed for at most min(M, K+1) micro-batches: the stash becomes a ring
// whose slots are rewritten only after their reader released them (events).
// The whole step is captured once into a CUDA graph and replayed.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/gpipe.h"
#include "context_info.h"
#include "kernels.h"
#include "launch_util.cuh"
#include "planner.h"

namespace {

using namespace gp;

struct StepPtrs {
  float* p32;
  void* p16;
  float* g32;
  float* v32;
  const void* batch;
  const void* targets;
  char* ws;
};

struct GraphKey {
  StepPtrs p;
  int64_t opts[15];
  bool operator==(const GraphKey& o) const { return std::memcmp(this, &o, sizeof(GraphKey)) == 0; }
};

}  // namespace

struct gpipe_ctx {
  int L = 0, K = 0, M = 0;
  Dims dm{};
  std::vector<int64_t> cost;
  std::vector<int32_t> bounds;
  std::vector<int> ffn;    // per-layer FFN width (dm.ffn holds the widest, which sizes the workspace)
  int max_cell = 0;
  ParamLayout pl;
  Workspace ws;
  bool ws_stale = true;
  // options
  bool keep_grads = false, use_graph = true, no_remat = false, skip_update = false;
  int64_t remat_check_m = -1;
  // state
  std::string err = "no error";
  cudaStream_t cap_stream = nullptr;
  bool concurrent = true;  // weight gradients and the loss-only head on each lane's side stream
  bool pipelined = true;   // cells run as concurrent lanes (the review's pipeline on one GPU)
  bool pdl = false;        // kernels may launch while their predecessor drains (measured slower with lanes)
  bool trace = false;      // stamp the GPU clock at the end of every (cell, micro-batch, phase)
  int inflight = 0;        // with lanes: micro-batches each cell works on at once (1, 2; 0: by size)
  int schedule = 0;        // issue order: 0 GPipe (all forwards, then all backwards), 1 one-forward-one-backward
  int64_t clip_milli = 0;  // logit clipping threshold in thousandths (0: none)
  // Two in flight when a micro-batch's FFN GEMM is small enough (tokens x d x
  // ffn <= 2^30) that its kernels are bound by latency rather than throughput.
  int inflight_eff() const {
    if (inflight) return inflight;
    const double work = static_cast<double>(Tmb()) * dm.d * (dm.ffn > 0 ? dm.ffn : dm.d);
    return work <= 1073741824.0 ? 2 : 1;
  }
  int ktime = 0;           // e+1: time every GEMM launch with epilogue e (event pairs)
  int sm_share = 100;      // percent of a GEMM's fair share of the SMs (with lanes)
  int side_share = 100;    // percent of that share for GEMMs on the side streams
  int nside = 2;           // side streams per lane (parameter groups spread over them)
  std::vector<cudaEvent_t> kt_ev;  // 2 per timed launch, reused step to step
  std::vector<double> kt_flops;
  std::vector<int32_t> kt_mnk;
  int kt_n = 0;  // timed launches issued by the last issued (or captured) step
  bool layer_times = false;        // event pairs around every layer's forward and backward of micro-batch 0
  std::vector<cudaEvent_t> lt_ev;  // 4 per layer: forward start/end, backward start/end
  bool lt_valid = false;           // the last issued (or captured) step recorded them
  static constexpr int kMaxLanes = 128;
  static constexpr int kLaneEvents = 13;
  static constexpr int kSides = 4;  // most side streams per lane
  cudaStream_t lane_main[kMaxLanes] = {}, lane_side[kMaxLanes][kSides] = {};
  cudaEvent_t lane_ev[kMaxLanes][kLaneEvents] = {};
  static constexpr int kRing = 4;  // deepest gradient ring between neighbouring cells (= most in flight)
  cudaEvent_t ev_origin = nullptr, ev_bdone[kMaxLanes][kRing] = {}, ev_bfree[kMaxLanes][kRing] = {},
              ev_lane_end[kMaxLanes] = {};
  std::vector<cudaEvent_t> ev_hdone;  // per micro-batch: the head has written the last cell's output gradient
  std::vector<cudaEvent_t> ev_fwd;    // per (cell, stash slot): the cell has written its output
  std::vector<cudaEvent_t> ev_sfree;  // per (stash level, slot): its reader is done (stash ring shorter than M)
  std::vector<cudaEvent_t> ev_hfree;  // per slot: the last cell has read the head's output gradient (likewise)
  // streams in use: one pair per lane, plus the head's pair when the cells are pipelined
  int nstreams() const { return ws.nlanes > 1 ? ws.nlanes + ws.nheads : 1; }
  cudaGraphExec_t gexec = nullptr;
  cudaGraph_t graph = nullptr;
  GraphKey key{};
  bool have_key = false;
  int64_t launches_per_step = 0;

  size_t T() const { return static_cast<size_t>(dm.n) * (dm.kind == 1 ? dm.seq : 1); }
  size_t Tmb() const { return T() / M; }
  size_t es() const { return dm.dtype == 0 ? 4 : 2; }
  int fail(int code, const std::string& msg) {
    err = msg;
    return code;
  }
  int fail_from_launch(int code) {
    err = last_error_message();
    return code;
  }
  MemoryModel memory_model() const {
    return review_memory_model(dm, L, K, M, max_cell, stash_depth(K, M, schedule), !no_remat);
  }
  void refresh_ws() {
    if (ws_stale) {
      const int nin = inflight_eff();
      const bool lanes = pipelined && K * nin + 2 <= kMaxLanes;  // + the head lanes
      ws = make_workspace(dm, L, K, M, max_cell, !no_remat, remat_check_m >= 0 && !no_remat, lanes,
                          lanes ? nin : 1, stash_depth(K, M, schedule));
      ws_stale = false;
    }
  }
  // lane streams and events (created on first use, on the current device)
  int ensure_lanes() {
    auto mk_ev = [&](cudaEvent_t& e) {
      return e || cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    };
    // Priorities: the cells' main streams (the critical path) highest, the
    // head lanes next (two of them keep ahead of the last cell's backward),
    // the side streams (weight gradients and gamma/beta reductions, off the
    // critical path) lowest.
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) least = greatest = 0;
    auto mk_st = [&](cudaStream_t& st, int prio) {
      return st || cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, prio) == cudaSuccess;
    };
    bool ok = mk_ev(ev_origin);
    auto mk_evs = [&](std::vector<cudaEvent_t>& v, size_t n) {
      if (v.size() < n) v.resize(n, nullptr);
      bool r = true;
      for (size_t i = 0; i < n && r; ++i) r = mk_ev(v[i]);
      return r;
    };
    const size_t D = static_cast<size_t>(ws.depth);
    ok = ok && mk_evs(ev_hdone, M) && mk_evs(ev_fwd, K * D);
    if (ws.depth < M) ok = ok && mk_evs(ev_sfree, (K + 1) * D) && mk_evs(ev_hfree, D);
    for (int i = 0; i < nstreams() && ok; ++i) {
      const bool head = nstreams() > 1 && i >= ws.nlanes;
      ok = mk_st(lane_main[i], head ? (least + greatest) / 2 : greatest);
      for (int j = 0; j < nside && ok; ++j) ok = mk_st(lane_side[i][j], least);
      ok = ok && mk_ev(ev_lane_end[i]);
      for (int e = 0; e < kLaneEvents && ok; ++e) ok = mk_ev(lane_ev[i][e]);
    }
    for (int k = 0; k < K && k < kMaxLanes && ok; ++k)
      for (int r = 0; r < kRing && ok; ++r) ok = mk_ev(ev_bdone[k][r]) && mk_ev(ev_bfree[k][r]);
    return ok ? GPIPE_OK : fail(GPIPE_ERR_CUDA, "cannot create the lane streams/events");
  }
  // The event pair of the next timed launch (created on first use).
  int kt_next(int M, int N, int K, cudaEvent_t* e0, cudaEvent_t* e1) {
    while (kt_ev.size() < static_cast<size_t>(2 * kt_n + 2)) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreate(&e) != cudaSuccess) return fail(GPIPE_ERR_CUDA, "cannot create a timing event");
      kt_ev.push_back(e);
    }
    if (kt_flops.size() <= static_cast<size_t>(kt_n)) {
      kt_flops.resize(kt_n + 1);
      kt_mnk.resize(3 * (kt_n + 1));
    }
    kt_flops[kt_n] = 2.0 * M * N * K;
    kt_mnk[3 * kt_n] = M;
    kt_mnk[3 * kt_n + 1] = N;
    kt_mnk[3 * kt_n + 2] = K;
    *e0 = kt_ev[2 * kt_n];
    *e1 = kt_ev[2 * kt_n + 1];
    ++kt_n;
    return GPIPE_OK;
  }
  void drop_graph() {
    if (gexec) cudaGraphExecDestroy(gexec);
    if (graph) cudaGraphDestroy(graph);
    gexec = nullptr;
    graph = nullptr;
    have_key = false;
  }
};

namespace {

#define TRY(expr)                          \
  do {                                     \
    int _rc = (expr);                      \
    if (_rc != GPIPE_OK) return _rc;       \
  } while (0)

// Pointers of one layer's slot.
struct Slot {
  char *u, *qkv, *o, *h1, *u2, *z1, *g, *y;
  float *mean1, *rstd1, *mean2, *rstd2, *lse;
};

// Events that order a lane's side stream against its main stream.
enum {
  EV_FORK,
  EV_GF,  // EV_GF + b: side work has read gf[b] (likewise gh[b], gq[b])
  EV_GF1,
  EV_GH,
  EV_GH1,
  EV_GQ,
  EV_GQ1,
  EV_DY0,
  EV_DY1,
  EV_DYB,
  EV_HEAD,
  EV_LN0,
  EV_LN1,
  EV_COUNT
};
constexpr int BUF_EXT = 2;  // "dy lives outside the lane" (boundary ring / head output)

// Issues one step.  Host issue order is the step's issue order (the planner's
// issue_order): the GPipe order of the review's "Pipeline flow" (phase 1:
// micro-batch-major forward, each micro-batch's head right after its last
// cell; phase 2: micro-batch-major backward, cells K-1..0) or the
// one-forward-one-backward order; then phase 3, the update.  When the cells
// are pipelined, cell k's work for micro-batch m goes to the streams of lane
// k*S + m mod S (S micro-batches in flight per cell), the head's to head lane
// m mod 2, and events carry exactly the dependencies of the review's pipeline:
// cell k forwards micro-batch m after cell k-1 handed it m; cell k
// differentiates m after cell k+1 handed it the gradient of m; a lane
// processes its micro-batches in order; a ring slot is rewritten only after
// its reader released it.  So cell k can work on micro-batch m while cell k+1
// works on m-1, as the review's K accelerators do.  Each parameter's gradient
// accumulation stays in micro-batch order on one stream, in either order, so
// the result does not depend on the interleaving.
class Executor {
 public:
  Executor(gpipe_ctx* c, const StepPtrs& p, cudaStream_t origin) : c_(c), p_(p), origin_(origin) {}

  int run_step() {
    const Workspace& w = c_->ws;
    const int M = c_->M, K = c_->K;
    set_pdl_enabled(c_->pdl);
    c_->kt_n = 0;
    c_->lt_valid = false;
    if (c_->layer_times) {
      if (c_->lt_ev.size() < static_cast<size_t>(4) * c_->L) c_->lt_ev.resize(static_cast<size_t>(4) * c_->L, nullptr);
      for (cudaEvent_t& e : c_->lt_ev)
        if (!e && cudaEventCreate(&e) != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "cannot create a layer event");
    }
    std::vector<Op> ops;
    if (!issue_order(K, M, c_->schedule, w.ring, ops, w.head_depth))
      return set_error(GPIPE_ERR_INVALID_ARG, "no issue order");
    // cells busy at each tick of the order (ops of one tick can run at once)
    int ticks = 0;
    for (const Op& o : ops) ticks = std::max(ticks, o.tick + 1);
    std::vector<int> busy(ticks, 0);
    for (const Op& o : ops)
      if (o.kind != OP_HEAD) ++busy[o.tick];
    fwd_rec_.assign(static_cast<size_t>(K) * w.depth, 0);
    sfree_rec_.assign(static_cast<size_t>(K + 1) * w.depth, 0);
    hfree_rec_.assign(w.depth, 0);
    // zero the loss scalar and the debug counter, then start every lane
    if (cudaMemsetAsync(p_.ws + w.misc, 0, 16, origin_) != cudaSuccess)
      return set_error(GPIPE_ERR_CUDA, "memset of the step counters failed");
    if (c_->trace) TRY(launch_stamp(stamp(0), origin_));
    TRY(cuda_ok(cudaEventRecord(c_->ev_origin, origin_), "event record"));
    for (int i = 0; i < c_->nstreams(); ++i)
      TRY(cuda_ok(cudaStreamWaitEvent(c_->lane_main[i], c_->ev_origin, 0), "stream wait"));
    for (const Op& o : ops) {
      busy_ = std::max(1, busy[o.tick]);
      if (o.kind == OP_FWD)
        TRY(forward_op(o.k, o.m));
      else if (o.kind == OP_HEAD)
        TRY(head_op(o.m));
      else
        TRY(backward_op(o.k, o.m));
    }
    // every lane (and its side stream) back into the origin stream
    for (int i = 0; i < c_->nstreams(); ++i) {
      TRY(join_all(i));
      TRY(cuda_ok(cudaEventRecord(c_->ev_lane_end[i], c_->lane_main[i]), "event record"));
      TRY(cuda_ok(cudaStreamWaitEvent(origin_, c_->ev_lane_end[i], 0), "stream wait"));
    }
    // phase 3: the embedding scatter of all micro-batches (after the head's
    // contributions, in token order), then one update of every parameter
    if (c_->dm.kind == 1)
      TRY(launch_embedding_bwd_io(DT_F32, static_cast<int>(c_->T()), c_->dm.d, c_->dm.vocab,
                                  static_cast<const int32_t*>(p_.batch), dx0(0), grad(c_->pl.emb), origin_));
    if (!c_->skip_update)
      TRY(launch_rmsprop(c_->pl.total, p_.p32, p_.g32, p_.v32, c_->dm.dtype == 1 ? p_.p16 : nullptr, c_->dm.lr,
                         c_->dm.decay, c_->dm.eps, c_->keep_grads ? 0 : 1, origin_));
    TRY(launch_sum(reinterpret_cast<float*>(ws(w.loss_rows)), c_->T(), reinterpret_cast<float*>(ws(w.misc)),
                   origin_));
    if (c_->trace) TRY(launch_stamp(stamp(1), origin_));
    c_->lt_valid = c_->layer_times;
    return GPIPE_OK;
  }

 private:
  gpipe_ctx* c_;
  StepPtrs p_;
  cudaStream_t origin_;
  cudaStream_t cur_ = nullptr;  // stream override for gemm()/launch helpers (nullptr: the lane's main stream)
  int cur_lane_ = 0;            // lane whose main stream receives the current cell's work
  int busy_ = 1;                // cells busy at the current op's tick of the schedule
  int ln_buf_[gpipe_ctx::kMaxLanes] = {};  // per lane: the LayerNorm-backward partial buffer to use next
  int gbuf_[gpipe_ctx::kMaxLanes] = {};    // per lane: the gf/gh/gq set the next layer backward uses
  bool rec_[gpipe_ctx::kMaxLanes][EV_COUNT] = {};
  std::vector<char> fwd_rec_, sfree_rec_, hfree_rec_;  // per (cell or level, ring slot)
  bool bdone_rec_[gpipe_ctx::kMaxLanes][gpipe_ctx::kRing] = {};
  bool bfree_rec_[gpipe_ctx::kMaxLanes][gpipe_ctx::kRing] = {};

  // Forward of cell k for micro-batch m (the embedding first for k = 0),
  // handing its output to cell k+1 (or the head) through the stash.
  int forward_op(int k, int m) {
    const int M = c_->M;
    const int lk = lane_of(k, m);
    // one-forward-one-backward: side work of an earlier backward on this lane
    // may still read the slots that this forward overwrites (in the GPipe
    // order every forward comes before the first backward)
    if (c_->schedule != 0) TRY(join_all(lk));
    if (k == 0) {
      if (c_->dm.kind == 1) TRY(slot_free_wait(lk, 0, m));
      TRY(cell0_input(m));
    } else {
      TRY(cross_wait(k, m, fwd_ev(k - 1, m), fwd_rec_[fwd_i(k - 1, m)], k - 1));
    }
    TRY(slot_free_wait(lk, k + 1, m));
    TRY(cell_forward(k, m, /*recompute=*/false));
    if (c_->trace) TRY(launch_stamp(stamp(2 + (static_cast<size_t>(k) * M + m) * 2), st()));
    return cross_record(k, m, fwd_ev(k, m), fwd_rec_[fwd_i(k, m)]);
  }

  // The head of micro-batch m on its own lane: loss rows and the gradient of
  // the last cell's output.
  int head_op(int m) {
    const int M = c_->M, K = c_->K;
    const int hl = head_lane(m);
    if (hl != lane_of(K - 1, m))
      TRY(cuda_ok(cudaStreamWaitEvent(main_s(hl), fwd_ev(K - 1, m), 0), "stream wait"));
    const int D = c_->ws.depth;
    if (m >= D && c_->ws.nlanes > 1) {  // the previous user of this output-gradient slot has read it
      if (!hfree_rec_[(m - D) % D]) return set_error(GPIPE_ERR_INVALID_ARG, "issue order reuses a head slot early");
      TRY(cuda_ok(cudaStreamWaitEvent(main_s(hl), c_->ev_hfree[(m - D) % D], 0), "stream wait"));
    }
    TRY(head(m));
    if (c_->trace) TRY(launch_stamp(stamp(2 + (static_cast<size_t>(K) * M + m) * 2), st()));
    if (hl != lane_of(K - 1, m)) TRY(cuda_ok(cudaEventRecord(c_->ev_hdone[m], main_s(hl)), "event record"));
    return GPIPE_OK;
  }

  // Backward of cell k for micro-batch m with re-computation, handing the
  // gradient of its input to cell k-1 through the ring.
  int backward_op(int k, int m) {
    const int M = c_->M, K = c_->K;
    const int p = m % c_->ws.ring;
    const int lk = lane_of(k, m);
    cur_lane_ = lk;
    TRY(join_all(lk));  // side work still reading this lane's slots
    if (!c_->no_remat) TRY(cell_forward(k, m, /*recompute=*/true));
    // gradient of the cell's output (fp32, with its bf16 copy for the GEMMs)
    char *dy, *dy16;
    const int dy_buf = BUF_EXT;
    if (k == K - 1) {
      if (head_lane(m) != lk) TRY(cuda_ok(cudaStreamWaitEvent(main_s(lk), c_->ev_hdone[m], 0), "stream wait"));
      dy = hdy(m);
      dy16 = hdy16(m);
    } else {
      TRY(cross_wait(k, m, c_->ev_bdone[k + 1][p], bdone_rec_[k + 1][p], k + 1));
      dy = bgrad(k + 1, p);
      dy16 = bgrad16(k + 1, p);
    }
    int cur_buf = dy_buf;
    const int first = c_->bounds[k], n = c_->bounds[k + 1] - first;
    for (int j = n - 1; j >= 0; --j) {
      const void* x = j == 0 ? cell_input(k, m) : slot(k, m, j - 1).y;
      char *dx, *dx16;
      int dx_buf;
      if (j == 0 && k > 0) {
        // hand the input gradient to cell k-1 through the ring
        if (bfree_rec_[k][p]) TRY(cross_wait(k, m, c_->ev_bfree[k][p], bfree_rec_[k][p], k - 1));
        dx = bgrad(k, p);
        dx16 = bgrad16(k, p);
        dx_buf = BUF_EXT;
      } else if (j == 0 && c_->dm.kind == 1) {
        dx = dx0(m);  // the embedding's input gradient, scattered once at the end (fp32 only)
        dx16 = dx;
        dx_buf = BUF_EXT;
      } else {
        dx_buf = cur_buf == 0 ? 1 : 0;
        dx = lbuf(lk, dx_buf);
        dx16 = lbuf16(lk, dx_buf);
      }
      const bool timed = c_->layer_times && m == 0;
      if (timed) TRY(record_timed(c_->lt_ev[4 * (first + j) + 2]));
      TRY(layer_backward(first + j, x, slot(k, m, j), dy, dy16, cur_buf, dx, copy_of(dx16, dx), dx_buf));
      if (timed) TRY(record_timed(c_->lt_ev[4 * (first + j) + 3]));
      dy = dx;
      dy16 = dx16;
      cur_buf = dx_buf;
    }
    if (c_->trace) TRY(launch_stamp(stamp(2 + (static_cast<size_t>(k) * M + m) * 2 + 1), st()));
    if (k > 0) TRY(cross_record(k, m, c_->ev_bdone[k][p], bdone_rec_[k][p]));
    if (k < K - 1) {  // this cell has finished reading the ring slot of cell k+1
      TRY(join(lk, EV_DYB));
      TRY(cross_record(k, m, c_->ev_bfree[k + 1][p], bfree_rec_[k + 1][p]));
    }
    const int D = c_->ws.depth;
    if (D < M && c_->ws.nlanes > 1) {
      // with a stash ring shorter than M: release this micro-batch's stash
      // slot of the cell's input (read by the re-computation and the first
      // layer's LayerNorm backward, both on the main stream) and, for the last
      // cell, its slot of the head's output gradient (read on the side too)
      sfree_rec_[static_cast<size_t>(k) * D + m % D] = 1;
      TRY(cuda_ok(cudaEventRecord(c_->ev_sfree[static_cast<size_t>(k) * D + m % D], main_s(lk)), "event record"));
      if (k == K - 1) {
        TRY(join(lk, EV_DYB));
        hfree_rec_[m % D] = 1;
        TRY(cuda_ok(cudaEventRecord(c_->ev_hfree[m % D], main_s(lk)), "event record"));
      }
    }
    return GPIPE_OK;
  }

  // The stash ring: cell k's output event, and the wait, before a slot of
  // level lev is rewritten for micro-batch m, for its previous micro-batch's
  // reader (the backward of cell lev, or the head for lev = K).
  size_t fwd_i(int k, int m) const { return static_cast<size_t>(k) * c_->ws.depth + m % c_->ws.depth; }
  cudaEvent_t fwd_ev(int k, int m) const { return c_->ev_fwd[fwd_i(k, m)]; }
  int slot_free_wait(int lane, int lev, int m) {
    const int D = lev == c_->K ? c_->ws.head_depth : c_->ws.depth;
    if (m < D || c_->ws.nlanes == 1) return GPIPE_OK;
    cudaEvent_t e;
    if (lev == c_->K) {
      e = c_->ev_hdone[m - D];  // the head has read its input (recorded: the issue order put it earlier)
    } else {
      const size_t i = static_cast<size_t>(lev) * D + (m - D) % D;
      if (!sfree_rec_[i]) return set_error(GPIPE_ERR_INVALID_ARG, "issue order reuses a stash slot early");
      e = c_->ev_sfree[i];
    }
    return cuda_ok(cudaStreamWaitEvent(main_s(lane), e, 0), "stream wait");
  }

  // Lane of cell k for micro-batch m: with lanes, cell k owns lanes
  // k*inflight .. k*inflight + inflight-1 and takes its micro-batches in turn.
  int lane_of(int k, int m) const { return c_->ws.nlanes > 1 ? k * c_->ws.inflight + m % c_->ws.inflight : 0; }
  // Head lanes follow the cells' lanes and take the micro-batches in turn.
  int head_lane(int m) const { return c_->ws.nlanes > 1 ? c_->ws.nlanes + m % c_->ws.nheads : 0; }
  bool is_head_lane(int lane) const { return c_->ws.nlanes > 1 && lane >= c_->ws.nlanes; }
  // A cell's lanes share the side streams of its first lane (the head lanes
  // those of the first head lane), which receive the weight-gradient work in
  // micro-batch order.
  int side_of(int lane) const { return lane < c_->ws.nlanes ? lane - lane % c_->ws.inflight : c_->ws.nlanes; }
  char* hdy(int m) const { return ws(c_->ws.hdy) + static_cast<size_t>(m % c_->ws.depth) * c_->ws.stash_bytes; }
  // The GEMM operand of a residual gradient: its bf16 copy, or the fp32
  // buffer itself for the fp32 model (copy_bytes 0).
  char* hdy16(int m) const {
    if (!c_->ws.copy_bytes) return hdy(m);
    return ws(c_->ws.hdy16) + static_cast<size_t>(m % c_->ws.depth) * c_->ws.copy_bytes;
  }
  cudaStream_t main_s(int lane) const { return c_->lane_main[lane]; }
  // Weight-gradient work goes to a side stream when CONCURRENT is on, and
  // always when a cell or the head has more than one lane (its lanes must not
  // accumulate into the same gradients from two streams).
  bool use_side() const { return c_->concurrent || c_->ws.inflight > 1 || c_->ws.nheads > 1; }
  // The side stream of a parameter group: the group of the event that marks
  // its work (W2, W1, W_o, W_qkv weight gradients, LayerNorm reductions; the
  // head's dE with W2).  A group always goes to the same stream, so each
  // parameter's gradient still accumulates in micro-batch order.
  static int group_of(int e) {
    switch (e) {
      case EV_GF: case EV_GF1: return 1;
      case EV_GH: case EV_GH1: return 2;
      case EV_GQ: case EV_GQ1: return 3;
      case EV_LN0: case EV_LN1: return 4;
      default: return 0;
    }
  }
  cudaStream_t side(int lane, int e) const {
    return use_side() ? c_->lane_side[side_of(lane)][group_of(e) % c_->nside] : c_->lane_main[lane];
  }
  cudaStream_t st() const { return cur_ ? cur_ : c_->lane_main[cur_lane_]; }
  int cuda_ok(cudaError_t e, const char* what) {
    return e == cudaSuccess ? GPIPE_OK : set_error(GPIPE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  }
  // cross-lane handshakes (no-ops when both cells share a lane)
  template <typename Flag>
  int cross_record(int k, int m, cudaEvent_t e, Flag& rec) {
    if (c_->ws.nlanes == 1) return GPIPE_OK;
    rec = true;
    return cuda_ok(cudaEventRecord(e, main_s(lane_of(k, m))), "event record");
  }
  int cross_wait(int k, int m, cudaEvent_t e, bool rec, int from_k) {
    if (c_->ws.nlanes == 1 || !rec || lane_of(k, m) == lane_of(from_k, m)) return GPIPE_OK;
    return cuda_ok(cudaStreamWaitEvent(main_s(lane_of(k, m)), e, 0), "stream wait");
  }
  // a lane's side stream starts after everything issued so far on its main stream
  int fork(int lane, int e) {
    if (!use_side()) return GPIPE_OK;
    TRY(cuda_ok(cudaEventRecord(c_->lane_ev[lane][EV_FORK], main_s(lane)), "event record"));
    return cuda_ok(cudaStreamWaitEvent(side(lane, e), c_->lane_ev[lane][EV_FORK], 0), "stream wait");
  }
  int mark(int lane, int e) {
    if (!use_side()) return GPIPE_OK;
    rec_[lane][e] = true;
    return cuda_ok(cudaEventRecord(c_->lane_ev[lane][e], side(lane, e)), "event record");
  }
  int join(int lane, int e) {
    if (!use_side() || !rec_[lane][e]) return GPIPE_OK;
    return cuda_ok(cudaStreamWaitEvent(main_s(lane), c_->lane_ev[lane][e], 0), "stream wait");
  }
  int join_all(int lane) {
    for (int e = EV_GF; e < EV_COUNT; ++e) TRY(join(lane, e));
    return GPIPE_OK;
  }
  template <typename F>
  int on_side(int e, F&& f) {
    const int lane = cur_lane_;
    TRY(fork(lane, e));
    cur_ = side(lane, e);
    int rc = f();
    cur_ = nullptr;
    if (rc) return rc;
    return mark(lane, e);
  }

  // LayerNorm backward: the rows (dx, on the critical path) on the current
  // stream; the fixed-order reduction of the gamma/beta partial sums on the
  // side stream, in issue order like the weight gradients.  The two partial
  // buffers alternate, so the next LayerNorm backward need not wait for this
  // reduction, only for the one that read its buffer before.
  // dy: a GEMM output of the compute type (dt); x, dres and dx: the fp32
  // residual stream and its gradient; dx16: the bf16 copy of dx (or nullptr).
  int ln_backward(int dt, int T, int d, const void* dy, const void* x, const float* mean, const float* rstd,
                  const float* g, const void* dres, void* dx, void* dx16, float* dg, float* db, float* part0,
                  float* part1) {
    const int lane = cur_lane_;
    const int b = ln_buf_[lane];
    ln_buf_[lane] ^= 1;
    float* part = b ? part1 : part0;
    TRY(join(lane, EV_LN0 + b));
    TRY(launch_layernorm_bwd_rows_io(dt, DT_F32, DT_F32, T, d, dy, x, mean, rstd, g, dres, dx, dx16, part, st()));
    return on_side(EV_LN0 + b, [&] { return launch_layernorm_bwd_reduce(T, d, part, dg, db, st()); });
  }

  char* ws(size_t off) const { return p_.ws + off; }
  unsigned long long* stamp(size_t i) const {
    return reinterpret_cast<unsigned long long*>(ws(c_->ws.trace)) + i;
  }
  const float* p32(size_t off) const { return p_.p32 + off; }
  float* grad(size_t off) const { return p_.g32 + off; }
  // GEMM operand weights: the bf16 compute copy, or the fp32 master for dtype 0
  const void* wgt(size_t off) const {
    return c_->dm.dtype == 1 ? static_cast<const void*>(static_cast<const char*>(p_.p16) + off * 2)
                             : static_cast<const void*>(p_.p32 + off);
  }
  const int32_t* tokens(int m) const {
    return static_cast<const int32_t*>(p_.batch) + static_cast<size_t>(m) * c_->Tmb();
  }
  // cell k's input (k < K; level 0 is the embedding's output) or, for k = K,
  // the last cell's output in the head's shorter ring
  char* stash(int k, int m) const {
    const Workspace& w = c_->ws;
    const size_t i = k < c_->K ? static_cast<size_t>(k) * w.depth + m % w.depth
                               : static_cast<size_t>(c_->K) * w.depth + m % w.head_depth;
    return ws(w.stash) + i * w.stash_bytes;
  }
  char* dx0(int m) const { return ws(c_->ws.dx0) + static_cast<size_t>(m) * c_->ws.stash_bytes; }
  char* bgrad(int k, int p) const {
    return ws(c_->ws.bgrad) + (static_cast<size_t>(k) * c_->ws.ring + p) * c_->ws.stash_bytes;
  }
  char* bgrad16(int k, int p) const {
    if (!c_->ws.copy_bytes) return bgrad(k, p);
    return ws(c_->ws.bgrad16) + (static_cast<size_t>(k) * c_->ws.ring + p) * c_->ws.copy_bytes;
  }
  char* lane_base(int lane) const { return ws(c_->ws.lanes) + static_cast<size_t>(lane) * c_->ws.lane.bytes; }
  char* lbuf(int lane, int i) const { return lane_base(lane) + (i == 0 ? c_->ws.lane.g0 : c_->ws.lane.g1); }
  char* lbuf16(int lane, int i) const {
    if (!c_->ws.copy_bytes) return lbuf(lane, i);
    return lane_base(lane) + (i == 0 ? c_->ws.lane.g0b : c_->ws.lane.g1b);
  }
  // bf16 copy to write beside a residual gradient (nullptr for the fp32 model)
  void* copy_of(char* op, char* f32) const { return op == f32 ? nullptr : op; }
  const void* cell_input(int k, int m) const {
    if (k == 0 && c_->dm.kind == 0)
      return static_cast<const char*>(p_.batch) + static_cast<size_t>(m) * c_->Tmb() * c_->dm.d * 4;
    return stash(k, m);
  }
  Slot slot(int k, int m, int j) const {
    char* b;
    if (c_->no_remat)
      b = ws(c_->ws.noremat_slots) + (static_cast<size_t>(m) * c_->L + c_->bounds[k] + j) * c_->ws.slot_bytes;
    else
      b = lane_base(lane_of(k, m)) + c_->ws.lane.slots + static_cast<size_t>(j) * c_->ws.slot_bytes;
    const SlotLayout& s = c_->ws.slot;
    Slot r;
    r.u = b + s.u;
    r.qkv = b + s.qkv;
    r.o = b + s.o;
    r.h1 = b + s.h1;
    r.u2 = b + s.u2;
    r.z1 = b + s.z1;
    r.g = b + s.g;
    r.y = b + s.y;
    r.mean1 = reinterpret_cast<float*>(b + s.mean1);
    r.rstd1 = reinterpret_cast<float*>(b + s.rstd1);
    r.mean2 = reinterpret_cast<float*>(b + s.mean2);
    r.rstd2 = reinterpret_cast<float*>(b + s.rstd2);
    r.lse = reinterpret_cast<float*>(b + s.lse);
    return r;
  }

  int gemm(int M, int N, int K, const void* A, int64_t lda, bool ak, const void* B, int64_t ldb, bool bk, int epi,
           void* C, int64_t ldc, const float* bias = nullptr, const void* resid = nullptr, int64_t ldr = 0,
           void* C2 = nullptr, const void* aux = nullptr, int64_t ldaux = 0, float* dbias = nullptr) {
    GemmDesc g;
    g.dtype = c_->dm.dtype == 0 ? DT_F32 : DT_BF16;
    g.M = M;
    g.N = N;
    g.K = K;
    g.A = A;
    g.lda = lda;
    g.a_kmajor = ak;
    g.B = B;
    g.ldb = ldb;
    g.b_kmajor = bk;
    g.epi = epi;
    g.C = C;
    g.ldc = ldc;
    g.bias = bias;
    g.dbias = dbias;
    g.resid = resid;
    g.ldr = ldr;
    g.C2 = C2;
    g.aux = aux;
    g.ldaux = ldaux;
    // lanes share the machine: a GEMM gets the SMs of one lane among the cells
    // that the review's schedule has busy at this clock tick (plus the head)
    if (c_->nstreams() > 1) {
      // a GEMM of few output tiles is bound by latency, not by its share of
      // the tensor cores: let it spread over twice the share
      int share = num_sms() * c_->sm_share / (100 * (busy_ + 1));
      const int64_t tiles = static_cast<int64_t>((M + 127) / 128) * ((N + 127) / 128);
      if (cur_) {
        // side stream (weight gradients, off the critical path): a small grid
        // whose CTAs each take many tiles spends the least SM time
        share = share * c_->side_share / 100;
      } else if (is_head_lane(cur_lane_)) {
        share = num_sms() * c_->sm_share / 200;  // the head's GEMMs: half the machine
      } else if (tiles <= 4 * static_cast<int64_t>(share)) {
        share *= 2;
      }
      g.sm_budget = share < 1 ? 1 : (share > num_sms() ? num_sms() : share);
    } else {
      g.sm_budget = num_sms();
    }
    if (c_->ktime != epi + 1) return launch_gemm(g, st());
    cudaEvent_t e0, e1;
    TRY(c_->kt_next(M, N, K, &e0, &e1));
    TRY(record_timed(e0));
    TRY(launch_gemm(g, st()));
    return record_timed(e1);
  }

  // A timing event on the current stream; under capture it becomes an event
  // node of the graph, so it is recorded at every replay.
  int record_timed(cudaEvent_t e) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st(), &cs) != cudaSuccess) return set_error(GPIPE_ERR_CUDA, "cudaStreamIsCapturing failed");
    const cudaError_t ce = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(e, st(), cudaEventRecordExternal)
                                                               : cudaEventRecord(e, st());
    return cuda_ok(ce, "timing event record");
  }

  int cell0_input(int m) {
    if (c_->dm.kind != 1) return GPIPE_OK;  // kind 0 reads the caller's x directly
    cur_lane_ = lane_of(0, m);
    return launch_embedding_fwd_io(DT_F32, static_cast<int>(c_->Tmb()), c_->dm.d, c_->dm.vocab, tokens(m),
                                   wgt(c_->pl.emb), stash(0, m), st());
  }

  // Forward of cell k for micro-batch m.  recompute: re-materialisation pass
  // of the backward (the last layer's output projection is skipped since its
  // result, the cell output, is already stashed and not needed to
  // differentiate the cell).
  int cell_forward(int k, int m, bool recompute) {
    cur_lane_ = lane_of(k, m);
    const int first = c_->bounds[k], n = c_->bounds[k + 1] - first;
    for (int j = 0; j < n; ++j) {
      const void* x = j == 0 ? cell_input(k, m) : slot(k, m, j - 1).y;
      void* out = j == n - 1 ? static_cast<void*>(stash(k + 1, m)) : static_cast<void*>(slot(k, m, j).y);
      const bool timed = c_->layer_times && m == 0 && !recompute;
      if (timed) TRY(record_timed(c_->lt_ev[4 * (first + j)]));
      TRY(layer_forward(first + j, x, slot(k, m, j), out, recompute && j == n - 1));
      if (timed) TRY(record_timed(c_->lt_ev[4 * (first + j) + 1]));
    }
    if (c_->remat_check_m == m && !c_->no_remat) TRY(remat_check(k, m, n, recompute));
    return GPIPE_OK;
  }

  // Debug: keep the first forward's internals of micro-batch m and count the
  // bytes that the re-computation reproduces differently.
  int remat_check(int k, int m, int n, bool recompute) {
    const Workspace& w = c_->ws;
    char* saved = ws(w.check) + static_cast<size_t>(k) * c_->max_cell * w.slot_bytes;
    char* slots = lane_base(lane_of(k, m)) + w.lane.slots;
    for (int j = 0; j < n; ++j) {
      char* sl = slots + static_cast<size_t>(j) * w.slot_bytes;
      const size_t bytes = j == n - 1 ? w.slot.compare_bytes_last : w.slot_bytes;
      if (!recompute)
        TRY(launch_copy(saved + j * w.slot_bytes, sl, bytes, st()));
      else
        TRY(launch_count_diff(saved + j * w.slot_bytes, sl, bytes,
                              reinterpret_cast<unsigned long long*>(ws(w.misc) + 8), st()));
    }
    return GPIPE_OK;
  }

  int layer_forward(int l, const void* x, const Slot& s, void* out, bool skip_out_proj) {
    const Dims& dm = c_->dm;
    const LayerOff& o = c_->pl.layers[l];
    const int T = static_cast<int>(c_->Tmb()), d = dm.d, f = c_->ffn[l];
    const int dt = dm.dtype == 0 ? DT_F32 : DT_BF16;
    // the residual stream (x, h1, the layer's output) is fp32; the residual
    // adds happen in the output projections' epilogues, in fp32
    const int resid_epi = dt == DT_F32 ? EPI_STORE : EPI_RESID_F32;
    TRY(launch_layernorm_fwd_io(DT_F32, dt, T, d, x, p32(o.ln1_g), p32(o.ln1_b), s.u, s.mean1, s.rstd1, st()));
    const void* ffn_in = s.u;
    const void* resid2 = x;
    if (dm.kind == 1) {
      TRY(gemm(T, 3 * d, d, s.u, d, true, wgt(o.w_qkv), d, true, EPI_STORE, s.qkv, 3 * d, p32(o.b_qkv)));
      TRY(launch_attention_fwd(T / dm.seq, dm.seq, dm.heads, s.qkv, s.o, s.lse, st()));
      TRY(gemm(T, d, d, s.o, d, true, wgt(o.w_o), d, true, resid_epi, s.h1, d, p32(o.b_o), x, d));
      TRY(launch_layernorm_fwd_io(DT_F32, dt, T, d, s.h1, p32(o.ln2_g), p32(o.ln2_b), s.u2, s.mean2, s.rstd2, st()));
      ffn_in = s.u2;
      resid2 = s.h1;
    }
    TRY(gemm(T, f, d, ffn_in, d, true, wgt(o.w1), d, true, EPI_BIAS_GELU, s.z1, f, p32(o.b1), nullptr, 0, s.g));
    if (!skip_out_proj)
      TRY(gemm(T, d, f, s.g, f, true, wgt(o.w2), f, true, resid_epi, out, d, p32(o.b2), resid2, d));
    return GPIPE_OK;
  }

  // Backward of layer l: dy (the gradient of its output) lives in lane buffer
  // dy_buf (0/1) or outside the lane (BUF_EXT); writes the gradient of its
  // input into dx (lane buffer dx_buf, or outside).  Weight gradients run on
  // the lane's side stream; before the main stream overwrites a buffer that a
  // side GEMM reads, it joins that GEMM's event.
  // dy / dx: the fp32 residual gradient of the layer's output / input; dy16:
  // dy as the GEMMs read it (its bf16 copy, or dy itself for the fp32 model);
  // dx16: where to write dx's bf16 copy (nullptr: none).
  int layer_backward(int l, const void* x, const Slot& s, const void* dy, const void* dy16, int dy_buf, void* dx,
                     void* dx16, int dx_buf) {
    const Dims& dm = c_->dm;
    const LayerOff& o = c_->pl.layers[l];
    const LaneLayout& ll = c_->ws.lane;
    const int lane = cur_lane_;
    char* lb = lane_base(lane);
    const int T = static_cast<int>(c_->Tmb()), d = dm.d, f = c_->ffn[l];
    const int dt = dm.dtype == 0 ? DT_F32 : DT_BF16;
    float* scratch = reinterpret_cast<float*>(lb + ll.scratch);
    float* lnp0 = reinterpret_cast<float*>(lb + ll.lnp[0]);
    float* lnp1 = reinterpret_cast<float*>(lb + ll.lnp[1]);
    // the weight-gradient operands alternate between two sets by layer, so the
    // main stream waits only for side work of two layers back before reuse
    const int gb = gbuf_[lane];
    gbuf_[lane] ^= 1;
    char* gf = lb + ll.gf[gb];
    char* gt = lb + ll.gt;
    const void* ffn_in = dm.kind == 1 ? static_cast<const void*>(s.u2) : static_cast<const void*>(s.u);
    const int ev_dy = dy_buf == 0 ? EV_DY0 : (dy_buf == 1 ? EV_DY1 : EV_DYB);
    // FFN: y = r + W2 GELU(W1 u + b1) + b2
    TRY(on_side(ev_dy, [&] {
      return gemm(d, f, T, dy16, d, false, s.g, f, false, EPI_ACC_F32, grad(o.w2), f, nullptr, nullptr, 0, nullptr,
                  nullptr, 0, grad(o.b2));
    }));
    TRY(join(lane, EV_GF + gb));
    TRY(gemm(T, f, d, dy16, d, true, wgt(o.w2), f, false, EPI_GELU_BWD, gf, f, nullptr, nullptr, 0, nullptr, s.z1, f));
    TRY(on_side(EV_GF + gb, [&] {
      return gemm(f, d, T, gf, f, false, ffn_in, d, false, EPI_ACC_F32, grad(o.w1), d, nullptr, nullptr, 0, nullptr,
                  nullptr, 0, grad(o.b1));
    }));
    TRY(gemm(T, d, f, gf, f, true, wgt(o.w1), d, false, EPI_STORE, gt, d));
    if (dm.kind == 0) {
      if (dx_buf != BUF_EXT) TRY(join(lane, dx_buf == 0 ? EV_DY0 : EV_DY1));
      return ln_backward(dt, T, d, gt, x, s.mean1, s.rstd1, p32(o.ln1_g), dy, dx, dx16, grad(o.ln1_g),
                         grad(o.ln1_b), lnp0, lnp1);
    }
    char* gh = lb + ll.gh[gb];    // bf16 copy of dh1 (the GEMMs' operand)
    char* gh32 = lb + ll.gh32;    // dh1 in fp32 (the residual gradient)
    char* gq = lb + ll.gq[gb];
    // h1 -> LN2: dh1 = LN2'(du2) + dy
    TRY(join(lane, EV_GH + gb));
    TRY(ln_backward(dt, T, d, gt, s.h1, s.mean2, s.rstd2, p32(o.ln2_g), dy, gh32, gh, grad(o.ln2_g),
                    grad(o.ln2_b), lnp0, lnp1));
    // attention output projection
    TRY(on_side(EV_GH + gb, [&] {
      return gemm(d, d, T, gh, d, false, s.o, d, false, EPI_ACC_F32, grad(o.w_o), d, nullptr, nullptr, 0, nullptr,
                  nullptr, 0, grad(o.b_o));
    }));
    TRY(gemm(T, d, d, gh, d, true, wgt(o.w_o), d, false, EPI_STORE, gt, d));
    TRY(join(lane, EV_GQ + gb));
    TRY(launch_attention_bwd(T / dm.seq, dm.seq, dm.heads, s.qkv, s.o, gt, s.lse, scratch, gq, st()));
    TRY(on_side(EV_GQ + gb, [&] {
      return gemm(3 * d, d, T, gq, 3 * d, false, s.u, d, false, EPI_ACC_F32, grad(o.w_qkv), d, nullptr, nullptr, 0,
                  nullptr, nullptr, 0, grad(o.b_qkv));
    }));
    TRY(gemm(T, d, 3 * d, gq, 3 * d, true, wgt(o.w_qkv), d, false, EPI_STORE, gt, d));
    if (dx_buf != BUF_EXT) TRY(join(lane, dx_buf == 0 ? EV_DY0 : EV_DY1));
    return ln_backward(dt, T, d, gt, x, s.mean1, s.rstd1, p32(o.ln1_g), gh32, dx, dx16, grad(o.ln1_g),
                       grad(o.ln1_b), lnp0, lnp1);
  }

  // The head of micro-batch m, once: loss rows from the last cell's output
  // stash[K][m] and the gradient of that output into hdy[m] (final LN, tied
  // logits, cross-entropy and their backward; MSE for the FFN model).
  int head(int m) {
    const Dims& dm = c_->dm;
    const Workspace& w = c_->ws;
    cur_lane_ = head_lane(m);
    const Workspace::Head& hb = w.head[c_->ws.nlanes > 1 ? m % w.nheads : 0];
    const int T = static_cast<int>(c_->Tmb()), d = dm.d;
    float* loss_rows = reinterpret_cast<float*>(ws(w.loss_rows)) + static_cast<size_t>(m) * T;
    const char* xf = stash(c_->K, m);
    char* dy = hdy(m);
    if (dm.kind == 0) {
      const float inv = 1.0f / (static_cast<float>(dm.n) * d);
      const float* t = static_cast<const float*>(p_.targets) + static_cast<size_t>(m) * T * d;
      return launch_mse(T, d, reinterpret_cast<const float*>(xf), t, inv, loss_rows, reinterpret_cast<float*>(dy),
                        st());
    }
    TRY(join(cur_lane_, EV_HEAD));  // the previous micro-batch's dE GEMM has read the logits and hf
    const float inv = 1.0f / (static_cast<float>(dm.n) * (dm.seq - 1));
    float* logits = reinterpret_cast<float*>(ws(hb.logits));
    TRY(launch_layernorm_fwd_io(DT_F32, DT_BF16, T, d, xf, p32(c_->pl.lnf_g), p32(c_->pl.lnf_b), ws(hb.hf),
                                reinterpret_cast<float*>(ws(hb.meanf)), reinterpret_cast<float*>(ws(hb.rstdf)),
                                st()));
    TRY(gemm(T, dm.vocab, d, ws(hb.hf), d, true, wgt(c_->pl.emb), d, true, EPI_STORE_F32, logits, dm.vocab));
    TRY(launch_cross_entropy(T, dm.vocab, dm.seq, static_cast<const int32_t*>(p_.batch), m * T, inv, logits,
                             loss_rows, 1, st(), static_cast<float>(static_cast<double>(c_->clip_milli) / 1000.0)));
    // dz (bf16, in place over the logits, leading dimension 2*vocab)
    const int64_t ldz = 2 * static_cast<int64_t>(dm.vocab);
    char* gt = ws(hb.hgt);
    TRY(gemm(T, d, dm.vocab, logits, ldz, true, wgt(c_->pl.emb), d, false, EPI_STORE, gt, d));
    TRY(on_side(EV_HEAD, [&] {
      return gemm(dm.vocab, d, T, logits, ldz, false, ws(hb.hf), d, false, EPI_ACC_F32, grad(c_->pl.emb), d);
    }));
    return ln_backward(DT_BF16, T, d, gt, xf, reinterpret_cast<float*>(ws(hb.meanf)),
                       reinterpret_cast<float*>(ws(hb.rstdf)), p32(c_->pl.lnf_g), nullptr, dy, copy_of(hdy16(m), dy),
                       grad(c_->pl.lnf_g), grad(c_->pl.lnf_b), reinterpret_cast<float*>(ws(hb.hlnp[0])),
                       reinterpret_cast<float*>(ws(hb.hlnp[1])));
  }
};

int validate_ffn(int kind, int ffn, std::string& why) {
  if (kind == GPIPE_KIND_FFN) {
    if (ffn < 8 || ffn % 8) return why = "kind 0 needs ffn % 8 == 0 and ffn >= 8", GPIPE_ERR_INVALID_ARG;
  } else if (ffn < 64 || ffn % 64) {
    return why = "ffn must be a positive multiple of 64", GPIPE_ERR_INVALID_ARG;
  }
  return GPIPE_OK;
}

int validate(int L, int K, int M, const gpipe_dims* dm, std::string& why) {
  if (!dm) return why = "dims is NULL", GPIPE_ERR_INVALID_ARG;
  if (L < 1) return why = "L must be >= 1", GPIPE_ERR_INVALID_ARG;
  if (K < 1 || K > L) return why = "need 1 <= K <= L", GPIPE_ERR_INVALID_ARG;
  if (M < 1) return why = "M must be >= 1", GPIPE_ERR_INVALID_ARG;
  if (dm->n < 1 || dm->n % M) return why = "N must be a positive multiple of M", GPIPE_ERR_INVALID_ARG;
  if (!(dm->lr > 0) || !(dm->decay >= 0 && dm->decay < 1) || !(dm->eps > 0))
    return why = "need lr > 0, 0 <= decay < 1, eps > 0", GPIPE_ERR_INVALID_ARG;
  if (dm->kind == GPIPE_KIND_FFN) {
    if (dm->dtype != GPIPE_DTYPE_F32) return why = "the FFN-block model runs in fp32 (dtype 0)", GPIPE_ERR_UNSUPPORTED;
    if (dm->d < 8 || dm->d % 8 || dm->d > 1024)
      return why = "kind 0 needs d % 8 == 0, 8 <= d <= 1024", GPIPE_ERR_INVALID_ARG;
    return GPIPE_OK;
  }
  if (dm->kind != GPIPE_KIND_LM) return why = "unknown kind", GPIPE_ERR_INVALID_ARG;
  if (dm->dtype != GPIPE_DTYPE_BF16) return why = "the Transformer model runs in bf16 (dtype 1)", GPIPE_ERR_UNSUPPORTED;
  if (dm->d < 64 || dm->d % 64 || dm->d > 1024 || dm->heads < 1 || dm->d / dm->heads != 64 || dm->d % dm->heads)
    return why = "kind 1 needs d % 64 == 0, d <= 1024 and d/heads == 64", GPIPE_ERR_INVALID_ARG;
  if (dm->seq < 64 || dm->seq % 64) return why = "seq must be a positive multiple of 64", GPIPE_ERR_INVALID_ARG;
  if (dm->vocab < 8 || dm->vocab % 8) return why = "vocab must be a positive multiple of 8", GPIPE_ERR_INVALID_ARG;
  return GPIPE_OK;
}

}  // namespace

namespace gp {

void describe_context(const gpipe_ctx* c, Dims* dm, int* L, std::vector<int>* ffn, size_t* params) {
  *dm = c->dm;
  *L = c->L;
  *ffn = c->ffn;
  *params = c->pl.total;
}

int context_fail(gpipe_ctx* c, int code, const char* msg) { return c->fail(code, msg); }

}  // namespace gp

extern "C" {

int gpipe_create(gpipe_ctx** out, int L, int K, int M, const gpipe_dims* dims, const int64_t* cost) {
  return gpipe_create_layers(out, L, K, M, dims, nullptr, cost);
}

int gpipe_create_layers(gpipe_ctx** out, int L, int K, int M, const gpipe_dims* dims, const int32_t* ffn,
                        const int64_t* cost) {
  if (!out) return set_error(GPIPE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  std::string why;
  int rc = validate(L, K, M, dims, why);
  if (rc) return set_error(rc, "%s", why.c_str());
  std::vector<int> widths(L, dims->ffn);
  if (!ffn) {
    rc = validate_ffn(dims->kind, dims->ffn, why);
    if (rc) return set_error(rc, "%s", why.c_str());
  } else {
    for (int l = 0; l < L; ++l) {
      rc = validate_ffn(dims->kind, ffn[l], why);
      if (rc) return set_error(rc, "layer %d: %s", l, why.c_str());
      widths[l] = ffn[l];
    }
  }
  gpipe_ctx* c = new gpipe_ctx();
  c->L = L;
  c->K = K;
  c->M = M;
  c->ffn = widths;
  c->dm = Dims{dims->kind, dims->d, dims->heads, *std::max_element(widths.begin(), widths.end()), dims->seq,
               dims->vocab, dims->n, dims->dtype, dims->lr, dims->decay, dims->eps};
  // default cost: the layer's forward FLOPs per token
  const int64_t d = dims->d;
  c->cost.resize(L);
  for (int i = 0; i < L; ++i) {
    const int64_t f = widths[i];
    const int64_t default_cost =
        dims->kind == 1 ? 2 * (4 * d * d + 2 * d * f) + 2 * d * (dims->seq + 1) : 2 * (2 * d * f);
    c->cost[i] = cost ? cost[i] : default_cost;
    if (c->cost[i] < 1) {
      delete c;
      return set_error(GPIPE_ERR_INVALID_ARG, "layer costs must be >= 1");
    }
  }
  if (!partition_min_variance(c->cost, K, c->bounds)) {
    delete c;
    return set_error(GPIPE_ERR_INVALID_ARG, "partition failed");
  }
  c->max_cell = 0;
  for (int k = 0; k < K; ++k) c->max_cell = std::max(c->max_cell, c->bounds[k + 1] - c->bounds[k]);
  c->pl = make_param_layout(c->dm, L, c->ffn);
  c->refresh_ws();
  *out = c;
  return GPIPE_OK;
}

int gpipe_repartition(gpipe_ctx* c, const int64_t* cost) {
  if (!c || !cost) return GPIPE_ERR_INVALID_ARG;
  std::vector<int64_t> costs(cost, cost + c->L);
  for (int64_t x : costs)
    if (x < 1) return c->fail(GPIPE_ERR_INVALID_ARG, "layer costs must be >= 1");
  std::vector<int32_t> bounds;
  if (!partition_min_variance(costs, c->K, bounds)) return c->fail(GPIPE_ERR_INVALID_ARG, "partition failed");
  c->cost = costs;
  c->bounds = bounds;
  c->max_cell = 0;
  for (int k = 0; k < c->K; ++k) c->max_cell = std::max(c->max_cell, bounds[k + 1] - bounds[k]);
  c->ws_stale = true;
  c->drop_graph();
  return GPIPE_OK;
}

int gpipe_partition(gpipe_ctx* c, int32_t* bounds_out) {
  if (!c || !bounds_out) return GPIPE_ERR_INVALID_ARG;
  std::copy(c->bounds.begin(), c->bounds.end(), bounds_out);
  return GPIPE_OK;
}

int gpipe_sizes(const gpipe_ctx* cc, size_t* param_elems, size_t* workspace_bytes) {
  if (!cc) return GPIPE_ERR_INVALID_ARG;
  gpipe_ctx* c = const_cast<gpipe_ctx*>(cc);
  c->refresh_ws();
  if (param_elems) *param_elems = c->pl.total;
  if (workspace_bytes) *workspace_bytes = c->ws.total;
  return GPIPE_OK;
}

int gpipe_init_params(gpipe_ctx* c, const float* p32, void* p16, void* stream) {
  if (!c) return GPIPE_ERR_INVALID_ARG;
  if (c->dm.dtype != 1) return GPIPE_OK;
  if (!p32 || !p16) return c->fail(GPIPE_ERR_INVALID_ARG, "NULL parameter buffer");
  int rc = launch_cast_bf16(c->pl.total, p32, p16, static_cast<cudaStream_t>(stream));
  return rc ? c->fail_from_launch(rc) : GPIPE_OK;
}

static int check_ptr(const void* p, const char* what, std::string& err) {
  if (!p) {
    err = std::string(what) + " is NULL";
    return GPIPE_ERR_INVALID_ARG;
  }
  if (reinterpret_cast<uintptr_t>(p) & 15u) {
    err = std::string(what) + " must be 16-byte aligned";
    return GPIPE_ERR_INVALID_ARG;
  }
  return GPIPE_OK;
}

int gpipe_step(gpipe_ctx* c, float* p32, void* p16, float* g32, float* v32, const void* batch, const void* targets,
               void* workspace, void* stream, float* loss_out) {
  if (!c) return GPIPE_ERR_INVALID_ARG;
  std::string e;
  int rc = check_ptr(p32, "params_fp32", e);
  if (!rc && c->dm.dtype == 1) rc = check_ptr(p16, "params_bf16", e);
  if (!rc) rc = check_ptr(g32, "grads_fp32", e);
  if (!rc) rc = check_ptr(v32, "rms_v_fp32", e);
  if (!rc) rc = check_ptr(batch, "batch_in", e);
  if (!rc && c->dm.kind == 0) rc = check_ptr(targets, "targets", e);
  if (!rc) rc = check_ptr(workspace, "workspace", e);
  if (rc) return c->fail(rc, e);
  c->refresh_ws();
  rc = prepare_kernels();
  if (rc) return c->fail_from_launch(rc);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StepPtrs ptrs{p32, p16, g32, v32, batch, targets, static_cast<char*>(workspace)};
  if (!c->use_graph) {
    rc = c->ensure_lanes();
    if (rc) return rc;
    const int64_t before = launch_count();
    Executor ex(c, ptrs, s);
    rc = ex.run_step();
    if (rc) return c->fail_from_launch(rc);
    c->launches_per_step = launch_count() - before;
  } else {
    GraphKey key{};
    key.p = ptrs;
    key.opts[0] = c->keep_grads;
    key.opts[1] = c->no_remat;
    key.opts[2] = c->skip_update;
    key.opts[3] = c->remat_check_m;
    key.opts[4] = c->concurrent;
    key.opts[5] = c->pipelined;
    key.opts[6] = c->pdl;
    key.opts[7] = c->trace;
    key.opts[8] = c->ktime;
    key.opts[9] = c->sm_share;
    key.opts[10] = c->side_share;
    key.opts[11] = c->nside;
    key.opts[12] = c->schedule;
    key.opts[13] = c->clip_milli;
    key.opts[14] = c->layer_times;
    if (!c->have_key || !(key == c->key)) {
      c->drop_graph();
      if (!c->cap_stream && cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
        return c->fail(GPIPE_ERR_CUDA, "cannot create the capture stream");
      if (cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
        return c->fail(GPIPE_ERR_CUDA, "cudaStreamBeginCapture failed");
      rc = c->ensure_lanes();
      if (rc) return rc;
      const int64_t before = launch_count();
      Executor ex(c, ptrs, c->cap_stream);
      rc = ex.run_step();
      cudaGraph_t g = nullptr;
      cudaError_t ce = cudaStreamEndCapture(c->cap_stream, &g);
      if (rc) {
        if (g) cudaGraphDestroy(g);
        return c->fail_from_launch(rc);
      }
      if (ce != cudaSuccess || !g)
        return c->fail(GPIPE_ERR_CUDA, std::string("graph capture failed: ") + cudaGetErrorString(ce));
      c->launches_per_step = launch_count() - before;
      c->graph = g;
      ce = cudaGraphInstantiate(&c->gexec, g, cudaGraphInstantiateFlagUseNodePriority);
      if (ce != cudaSuccess) {
        c->drop_graph();
        return c->fail(GPIPE_ERR_CUDA, std::string("graph instantiate failed: ") + cudaGetErrorString(ce));
      }
      c->key = key;
      c->have_key = true;
    }
    cudaError_t ce = cudaGraphLaunch(c->gexec, s);
    if (ce != cudaSuccess) return c->fail(GPIPE_ERR_CUDA, std::string("graph launch failed: ") + cudaGetErrorString(ce));
  }
  if (loss_out) {
    float loss = 0.f;
    int derr = 0;
    cudaError_t ce = cudaMemcpyAsync(&loss, static_cast<char*>(workspace) + c->ws.misc, 4, cudaMemcpyDeviceToHost, s);
    if (ce == cudaSuccess) ce = cudaMemcpyAsync(&derr, device_error_ptr(), 4, cudaMemcpyDeviceToHost, s);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
    if (ce != cudaSuccess) return c->fail(GPIPE_ERR_CUDA, std::string("step failed: ") + cudaGetErrorString(ce));
    *loss_out = loss;
    if (derr) return c->fail(GPIPE_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up (device error flag " +
                                                           std::to_string(derr) + ")");
    if (!std::isfinite(loss)) return c->fail(GPIPE_ERR_NONFINITE_LOSS, "loss is not finite");
  }
  return GPIPE_OK;
}

double gpipe_bubble_fraction(const gpipe_ctx* c) {
  if (!c) return -1.0;
  return static_cast<double>(c->K - 1) / static_cast<double>(c->M + c->K - 1);
}

int gpipe_schedule_model(const gpipe_ctx* c, const double* t_f, const double* t_b, double* makespan, double* bubble) {
  if (!c) return GPIPE_ERR_INVALID_ARG;
  std::vector<double> tf(c->K), tb(c->K);
  for (int k = 0; k < c->K; ++k) {
    double cellcost = 0.0;
    for (int l = c->bounds[k]; l < c->bounds[k + 1]; ++l) cellcost += static_cast<double>(c->cost[l]);
    tf[k] = t_f ? t_f[k] : cellcost;
    tb[k] = t_b ? t_b[k] : 2.0 * cellcost;
  }
  double b = 0.0, ms = 0.0;
  if (c->schedule == 0) {
    ms = simulate_gpipe(c->K, c->M, tf.data(), tb.data(), &b);
  } else {
    std::vector<Op> ops;
    if (!issue_order(c->K, c->M, c->schedule, 2, ops)) return GPIPE_ERR_INVALID_ARG;
    ms = simulate_order(c->K, c->M, ops, tf.data(), tb.data(), &b);
  }
  if (makespan) *makespan = ms;
  if (bubble) *bubble = b;
  return GPIPE_OK;
}

int gpipe_issue_order(const gpipe_ctx* cc, int32_t* ops_out, int count) {
  if (!cc || count < 0 || (count > 0 && !ops_out)) return GPIPE_ERR_INVALID_ARG;
  gpipe_ctx* c = const_cast<gpipe_ctx*>(cc);
  c->refresh_ws();
  std::vector<Op> ops;
  if (!issue_order(c->K, c->M, c->schedule, c->ws.ring, ops, c->ws.head_depth))
    return c->fail(GPIPE_ERR_INVALID_ARG, "no issue order");
  for (int i = 0; i < count && i < static_cast<int>(ops.size()); ++i) {
    ops_out[4 * i] = ops[i].kind;
    ops_out[4 * i + 1] = ops[i].k;
    ops_out[4 * i + 2] = ops[i].m;
    ops_out[4 * i + 3] = ops[i].tick;
  }
  return static_cast<int>(ops.size());
}

int gpipe_memory_report(const gpipe_ctx* cc, size_t* peak_act_bytes, size_t* model_bound_bytes) {
  if (!cc) return GPIPE_ERR_INVALID_ARG;
  gpipe_ctx* c = const_cast<gpipe_ctx*>(cc);
  c->refresh_ws();
  if (peak_act_bytes) *peak_act_bytes = c->ws.act_bytes;
  if (model_bound_bytes) *model_bound_bytes = c->memory_model().total;
  return GPIPE_OK;
}

int gpipe_memory_model(const gpipe_ctx* cc, size_t* terms_out, int count) {
  if (!cc || count < 0 || (count > 0 && !terms_out)) return GPIPE_ERR_INVALID_ARG;
  gpipe_ctx* c = const_cast<gpipe_ctx*>(cc);
  c->refresh_ws();
  const MemoryModel mm = c->memory_model();
  const size_t t[GPIPE_MEMORY_TERMS] = {mm.boundary, mm.cell, mm.head, mm.grads, mm.rows, mm.align, mm.total,
                                        mm.survey, c->ws.act_bytes};
  for (int i = 0; i < count && i < GPIPE_MEMORY_TERMS; ++i) terms_out[i] = t[i];
  return GPIPE_MEMORY_TERMS;
}

int gpipe_set_option(gpipe_ctx* c, int option, int64_t value) {
  if (!c) return GPIPE_ERR_INVALID_ARG;
  switch (option) {
    case GPIPE_OPT_KEEP_GRADS: c->keep_grads = value != 0; break;
    case GPIPE_OPT_GRAPH: c->use_graph = value != 0; break;
    case GPIPE_OPT_NO_REMAT: c->no_remat = value != 0; c->ws_stale = true; break;
    case GPIPE_OPT_REMAT_CHECK:
      if (value >= c->M) return c->fail(GPIPE_ERR_INVALID_ARG, "remat check micro-batch out of range");
      c->remat_check_m = value < 0 ? -1 : value;
      c->ws_stale = true;
      break;
    case GPIPE_OPT_SKIP_UPDATE: c->skip_update = value != 0; break;
    case GPIPE_OPT_CONCURRENT: c->concurrent = value != 0; break;
    case GPIPE_OPT_PIPELINE: c->pipelined = value != 0; c->ws_stale = true; break;
    case GPIPE_OPT_PDL: c->pdl = value != 0; break;
    case GPIPE_OPT_TRACE: c->trace = value != 0; break;
    case GPIPE_OPT_LAYER_TIMES:
      c->layer_times = value != 0;
      c->lt_valid = false;
      break;
    case GPIPE_OPT_LOGIT_CLIP:
      if (value < 0 || value > 1000000000)
        return c->fail(GPIPE_ERR_INVALID_ARG, "logit clip must be 0 (none) or a threshold in thousandths up to 1e9");
      c->clip_milli = value;
      break;
    case GPIPE_OPT_SCHEDULE:
      if (value < 0 || value > 1) return c->fail(GPIPE_ERR_INVALID_ARG, "schedule must be 0 (GPipe) or 1 (1F1B)");
      c->schedule = static_cast<int>(value);
      c->ws_stale = true;
      break;
    case GPIPE_OPT_SIDE_STREAMS:
      if (value < 1 || value > gpipe_ctx::kSides)
        return c->fail(GPIPE_ERR_INVALID_ARG, "side streams per lane must be 1..4");
      c->nside = static_cast<int>(value);
      break;
    case GPIPE_OPT_SIDE_SHARE:
      if (value < 5 || value > 800) return c->fail(GPIPE_ERR_INVALID_ARG, "side SM share must be 5..800 percent");
      c->side_share = static_cast<int>(value);
      break;
    case GPIPE_OPT_INFLIGHT:
      if (value < 0 || value > gpipe_ctx::kRing)
        return c->fail(GPIPE_ERR_INVALID_ARG, "in-flight micro-batches per cell must be 0 (by size) or 1..4");
      c->inflight = static_cast<int>(value);
      c->ws_stale = true;
      break;
    case GPIPE_OPT_SM_SHARE:
      if (value < 25 || value > 800) return c->fail(GPIPE_ERR_INVALID_ARG, "SM share must be 25..800 percent");
      c->sm_share = static_cast<int>(value);
      break;
    case GPIPE_OPT_KERNEL_TIMES:
      if (value < 0 || value > 6) return c->fail(GPIPE_ERR_INVALID_ARG, "kernel-times selector out of range");
      c->ktime = static_cast<int>(value);
      break;
    default: return c->fail(GPIPE_ERR_INVALID_ARG, "unknown option");
  }
  c->drop_graph();
  return GPIPE_OK;
}

int gpipe_kernel_times(gpipe_ctx* c, float* ms_out, double* flops_out, int32_t* mnk_out, int count) {
  if (!c || count < 0) return GPIPE_ERR_INVALID_ARG;
  const int n = c->ktime ? c->kt_n : 0;
  for (int i = 0; i < n && i < count; ++i) {
    float t = 0.f;
    cudaError_t ce = cudaEventSynchronize(c->kt_ev[2 * i + 1]);
    if (ce == cudaSuccess) ce = cudaEventElapsedTime(&t, c->kt_ev[2 * i], c->kt_ev[2 * i + 1]);
    if (ce != cudaSuccess) return c->fail(GPIPE_ERR_CUDA, std::string("kernel times: ") + cudaGetErrorString(ce));
    if (ms_out) ms_out[i] = t;
    if (flops_out) flops_out[i] = c->kt_flops[i];
    if (mnk_out)
      for (int j = 0; j < 3; ++j) mnk_out[3 * i + j] = c->kt_mnk[3 * i + j];
  }
  return n;
}

int gpipe_layer_times(gpipe_ctx* c, float* fwd_ms, float* bwd_ms, int count) {
  if (!c || count < 0) return GPIPE_ERR_INVALID_ARG;
  if (!c->lt_valid) return 0;
  for (int l = 0; l < c->L && l < count; ++l) {
    float t[2] = {0.f, 0.f};
    for (int ph = 0; ph < 2; ++ph) {
      cudaError_t ce = cudaEventSynchronize(c->lt_ev[4 * l + 2 * ph + 1]);
      if (ce == cudaSuccess) ce = cudaEventElapsedTime(&t[ph], c->lt_ev[4 * l + 2 * ph], c->lt_ev[4 * l + 2 * ph + 1]);
      if (ce != cudaSuccess) return c->fail(GPIPE_ERR_CUDA, std::string("layer times: ") + cudaGetErrorString(ce));
    }
    if (fwd_ms) fwd_ms[l] = t[0];
    if (bwd_ms) bwd_ms[l] = t[1];
  }
  return c->L;
}

int gpipe_debug_counters(gpipe_ctx* c, void* workspace, void* stream, uint64_t* remat_mismatch, int* error_flag) {
  if (!c || !workspace) return GPIPE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long cnt = 0;
  int derr = 0;
  cudaError_t ce = cudaMemcpyAsync(&cnt, static_cast<char*>(workspace) + c->ws.misc + 8, 8, cudaMemcpyDeviceToHost, s);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(&derr, device_error_ptr(), 4, cudaMemcpyDeviceToHost, s);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
  if (ce == cudaSuccess && derr) ce = cudaMemsetAsync(device_error_ptr(), 0, 4, s);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
  if (ce != cudaSuccess) return c->fail(GPIPE_ERR_CUDA, cudaGetErrorString(ce));
  if (remat_mismatch) *remat_mismatch = cnt;
  if (error_flag) *error_flag = derr;
  return GPIPE_OK;
}

int gpipe_loss_rows(gpipe_ctx* c, void* workspace, void* stream, float* host_out, size_t count) {
  if (!c || !workspace || !host_out) return GPIPE_ERR_INVALID_ARG;
  if (count > c->T()) return c->fail(GPIPE_ERR_INVALID_ARG, "count exceeds the number of loss rows");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaMemcpyAsync(host_out, static_cast<char*>(workspace) + c->ws.loss_rows, count * 4,
                                   cudaMemcpyDeviceToHost, s);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
  if (ce != cudaSuccess) return c->fail(GPIPE_ERR_CUDA, cudaGetErrorString(ce));
  return GPIPE_OK;
}

int gpipe_trace(gpipe_ctx* c, void* workspace, void* stream, uint64_t* host_out, size_t count) {
  if (!c || !workspace || !host_out) return GPIPE_ERR_INVALID_ARG;
  c->refresh_ws();
  if (count > c->ws.trace_count) return c->fail(GPIPE_ERR_INVALID_ARG, "count exceeds the trace length");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaMemcpyAsync(host_out, static_cast<char*>(workspace) + c->ws.trace, count * 8,
                                   cudaMemcpyDeviceToHost, s);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
  if (ce != cudaSuccess) return c->fail(GPIPE_ERR_CUDA, cudaGetErrorString(ce));
  return GPIPE_OK;
}

int64_t gpipe_launches_per_step(const gpipe_ctx* c) { return c ? c->launches_per_step : -1; }

const char* gpipe_last_error(const gpipe_ctx* c) {
  if (!c) return last_error_message();
  return c->err.c_str();
}

void gpipe_destroy(gpipe_ctx* c) {
  if (!c) return;
  c->drop_graph();
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  for (int i = 0; i < gpipe_ctx::kMaxLanes; ++i) {
    if (c->lane_main[i]) cudaStreamDestroy(c->lane_main[i]);
    for (cudaStream_t st : c->lane_side[i])
      if (st) cudaStreamDestroy(st);
    for (auto& e : c->lane_ev[i])
      if (e) cudaEventDestroy(e);
    for (int r = 0; r < gpipe_ctx::kRing; ++r) {
      if (c->ev_bdone[i][r]) cudaEventDestroy(c->ev_bdone[i][r]);
      if (c->ev_bfree[i][r]) cudaEventDestroy(c->ev_bfree[i][r]);
    }
    if (c->ev_lane_end[i]) cudaEventDestroy(c->ev_lane_end[i]);
  }
  if (c->ev_origin) cudaEventDestroy(c->ev_origin);
  for (const auto* v : {&c->ev_hdone, &c->ev_fwd, &c->ev_sfree, &c->ev_hfree})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : c->lt_ev)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : c->kt_ev)
    if (e) cudaEventDestroy(e);
  delete c;
}

}  // extern "C"
