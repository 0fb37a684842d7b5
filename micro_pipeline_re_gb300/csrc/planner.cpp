// Host planner of the GPipe step.
//
// Partition: "GPipe technical review" (zzz0906.github.io), "GPipe algorithm:
// minimal interface" - consecutive layers are cut into K cells and balanced
// by minimising the variance of the per-cell estimated cost.  With the total
// fixed, variance = (1/K) sum S_k^2 - mean^2, so the exact integer objective
// sum S_k^2 is minimised by dynamic programming over suffixes.
//
// Clock model: "Pipeline flow" (phases 1-3) and "Bubble overhead analysis";
// with equal cells the bubble is (K-1)/(M+K-1).
//
// Issue orders: the GPipe order of "Pipeline flow", or the
// one-forward-one-backward order that the review's "Historical impact" section
// credits to PipeDream-2BW (forward and backward interleaved to cut the peak
// memory of accumulated activations); the PipeDream page's citing works
// describe it as starting backward passes earlier without changing the
// result.  Both orders differentiate each cell's micro-batches in ascending
// order, so the gradients accumulate in the same order.
//
// Workspace: "Preliminaries 5: re-materialisation" - only the cell-boundary
// activations of every micro-batch are kept (stash), plus the internals of
// the one cell being differentiated for one micro-batch, giving the review's
// O(N + (L/K)(N/M)) peak instead of O(N L).
#include "planner.h"

#include <algorithm>
#include <limits>

namespace gp {

using i128 = __int128;

bool partition_min_variance(const std::vector<int64_t>& costs, int K, std::vector<int32_t>& bounds) {
  const int L = static_cast<int>(costs.size());
  if (K < 1 || K > L) return false;
  std::vector<i128> pre(L + 1, 0);
  for (int i = 0; i < L; ++i) pre[i + 1] = pre[i] + costs[i];
  const i128 INF = (static_cast<i128>(1) << 126);
  // best[c][i]: minimum sum of squared cell sums splitting layers [i, L) into c cells
  std::vector<std::vector<i128>> best(K + 1, std::vector<i128>(L + 1, INF));
  best[0][L] = 0;
  for (int c = 1; c <= K; ++c) {
    for (int i = L - c; i >= 0; --i) {
      i128 b = INF;
      for (int j = i + 1; j <= L - (c - 1); ++j) {
        if (best[c - 1][j] >= INF) continue;
        const i128 s = pre[j] - pre[i];
        const i128 v = s * s + best[c - 1][j];
        if (v < b) b = v;
      }
      best[c][i] = b;
    }
  }
  bounds.assign(1, 0);
  int i = 0;
  for (int c = K; c >= 1; --c) {
    for (int j = i + 1; j <= L - (c - 1); ++j) {
      if (best[c - 1][j] >= INF) continue;
      const i128 s = pre[j] - pre[i];
      if (s * s + best[c - 1][j] == best[c][i]) {
        bounds.push_back(j);
        i = j;
        break;
      }
    }
  }
  return static_cast<int>(bounds.size()) == K + 1 && bounds.back() == L;
}

double simulate_gpipe(int K, int M, const double* t_f, const double* t_b, double* bubble) {
  std::vector<double> fe(static_cast<size_t>(M) * K, 0.0), be(static_cast<size_t>(M) * K, 0.0);
  auto F = [&](int m, int k) -> double& { return fe[static_cast<size_t>(m) * K + k]; };
  auto B = [&](int m, int k) -> double& { return be[static_cast<size_t>(m) * K + k]; };
  for (int m = 0; m < M; ++m)
    for (int k = 0; k < K; ++k) {
      double s = 0.0;
      if (m > 0) s = std::max(s, F(m - 1, k));
      if (k > 0) s = std::max(s, F(m, k - 1));
      F(m, k) = s + t_f[k];
    }
  for (int m = 0; m < M; ++m)
    for (int k = K - 1; k >= 0; --k) {
      double s = F(M - 1, k);
      if (m > 0) s = std::max(s, B(m - 1, k));
      if (k < K - 1) s = std::max(s, B(m, k + 1));
      B(m, k) = s + t_b[k];
    }
  double makespan = 0.0, busy = 0.0;
  for (int m = 0; m < M; ++m) makespan = std::max(makespan, B(m, 0));
  for (int k = 0; k < K; ++k) busy += M * (t_f[k] + t_b[k]);
  if (bubble) *bubble = makespan > 0 ? 1.0 - busy / (K * makespan) : 0.0;
  return makespan;
}

int stash_depth(int K, int M, int schedule) { return schedule == 1 ? std::min(M, K + 1) : M; }

namespace {
// Position of op (kind, k, m) in a K x M table per kind (the head uses k = 0).
inline size_t op_index(int kind, int k, int m, int K, int M) {
  return (static_cast<size_t>(kind) * (K + 1) + k) * M + m;
}
}  // namespace

bool issue_order(int K, int M, int schedule, int ring, std::vector<Op>& ops, int head_depth) {
  ops.clear();
  if (K < 1 || M < 1 || ring < 1) return false;
  if (schedule == 0) {
    // ticks: forward phase t = k + m; backward phase after it, t = M + K - 1 + (K - 1 - k) + m
    for (int m = 0; m < M; ++m) {
      for (int k = 0; k < K; ++k) ops.push_back(Op{OP_FWD, k, m, k + m});
      ops.push_back(Op{OP_HEAD, 0, m, K - 1 + m});
    }
    for (int m = 0; m < M; ++m)
      for (int k = K - 1; k >= 0; --k) ops.push_back(Op{OP_BWD, k, m, M + K - 1 + (K - 1 - k) + m});
    return true;
  }
  if (schedule != 1) return false;
  const int D = stash_depth(K, M, schedule);
  const int DK = head_depth > 0 ? std::min(head_depth, D) : D;
  // per-stage sequences: cells 0..K-1, then the head (stage K)
  std::vector<std::vector<Op>> seq(K + 1);
  for (int k = 0; k < K; ++k) {
    const int f0 = std::min(M, K + 1 - k);
    for (int m = 0; m < f0; ++m) seq[k].push_back(Op{OP_FWD, k, m, 0});
    for (int i = 0; i < M; ++i) {
      seq[k].push_back(Op{OP_BWD, k, i, 0});
      if (f0 + i < M) seq[k].push_back(Op{OP_FWD, k, f0 + i, 0});
    }
  }
  for (int m = 0; m < M; ++m) seq[K].push_back(Op{OP_HEAD, 0, m, 0});
  std::vector<int> round_of(static_cast<size_t>(3) * (K + 1) * M, -1);
  auto issued_before = [&](int kind, int k, int m, int r) {
    const int at = round_of[op_index(kind, k, m, K, M)];
    return at >= 0 && at < r;
  };
  auto ready = [&](const Op& o, int r) {
    if (o.kind == OP_FWD) {
      if (o.k > 0 && !issued_before(OP_FWD, o.k - 1, o.m, r)) return false;
      // the stash slot it writes (cell k's output; the embedding's for k = 0)
      // was released by the previous micro-batch in it
      if (o.m >= D) {
        const int pm = o.m - D;
        if (o.k + 1 < K && !issued_before(OP_BWD, o.k + 1, pm, r)) return false;
        if (o.k == 0 && !issued_before(OP_BWD, 0, pm, r)) return false;
      }
      // the last cell's output goes to the head's input ring
      if (o.k == K - 1 && o.m >= DK && !issued_before(OP_HEAD, 0, o.m - DK, r)) return false;
      return true;
    }
    if (o.kind == OP_HEAD) {
      if (!issued_before(OP_FWD, K - 1, o.m, r)) return false;
      return o.m < D || issued_before(OP_BWD, K - 1, o.m - D, r);  // its output-gradient slot
    }
    if (o.k == K - 1 ? !issued_before(OP_HEAD, 0, o.m, r) : !issued_before(OP_BWD, o.k + 1, o.m, r)) return false;
    return o.k == 0 || o.m < ring || issued_before(OP_BWD, o.k - 1, o.m - ring, r);  // its ring slot
  };
  std::vector<size_t> pos(K + 1, 0);
  const size_t total = static_cast<size_t>(2 * K + 1) * M;
  for (int r = 0; ops.size() < total; ++r) {
    std::vector<Op> batch;
    for (int s = 0; s <= K; ++s)
      if (pos[s] < seq[s].size() && ready(seq[s][pos[s]], r)) batch.push_back(seq[s][pos[s]]);
    if (batch.empty()) return false;
    for (Op o : batch) {
      o.tick = r;
      round_of[op_index(o.kind, o.k, o.m, K, M)] = r;
      ++pos[o.kind == OP_HEAD ? K : o.k];
      ops.push_back(o);
    }
  }
  return true;
}

double simulate_order(int K, int M, const std::vector<Op>& ops, const double* t_f, const double* t_b,
                      double* bubble) {
  std::vector<double> fin(static_cast<size_t>(3) * (K + 1) * M, 0.0), stage_free(K + 1, 0.0);
  double makespan = 0.0;
  for (const Op& o : ops) {
    const int s = o.kind == OP_HEAD ? K : o.k;
    double start = stage_free[s];
    double dur = 0.0;
    if (o.kind == OP_FWD) {
      if (o.k > 0) start = std::max(start, fin[op_index(OP_FWD, o.k - 1, o.m, K, M)]);
      dur = t_f[o.k];
    } else if (o.kind == OP_HEAD) {
      start = std::max(start, fin[op_index(OP_FWD, K - 1, o.m, K, M)]);
    } else {
      start = std::max(start, o.k == K - 1 ? fin[op_index(OP_HEAD, 0, o.m, K, M)]
                                           : fin[op_index(OP_BWD, o.k + 1, o.m, K, M)]);
      dur = t_b[o.k];
    }
    const double end = start + dur;
    fin[op_index(o.kind, o.k, o.m, K, M)] = end;
    stage_free[s] = end;
    makespan = std::max(makespan, end);
  }
  double busy = 0.0;
  for (int k = 0; k < K; ++k) busy += M * (t_f[k] + t_b[k]);
  if (bubble) *bubble = makespan > 0 ? 1.0 - busy / (K * makespan) : 0.0;
  return makespan;
}

ParamLayout make_param_layout(const Dims& dm, int L, const std::vector<int>& ffn) {
  ParamLayout p;
  const size_t d = dm.d;
  size_t o = 0;
  for (int l = 0; l < L; ++l) {
    const size_t f = ffn.empty() ? static_cast<size_t>(dm.ffn) : static_cast<size_t>(ffn[l]);
    LayerOff lo{};
    if (dm.kind == 0) {
      lo.ln1_g = o; o += d;
      lo.ln1_b = o; o += d;
      lo.w1 = o; o += f * d;
      lo.b1 = o; o += f;
      lo.w2 = o; o += d * f;
      lo.b2 = o; o += d;
    } else {
      lo.ln1_g = o; o += d;
      lo.ln1_b = o; o += d;
      lo.w_qkv = o; o += 3 * d * d;
      lo.b_qkv = o; o += 3 * d;
      lo.w_o = o; o += d * d;
      lo.b_o = o; o += d;
      lo.ln2_g = o; o += d;
      lo.ln2_b = o; o += d;
      lo.w1 = o; o += f * d;
      lo.b1 = o; o += f;
      lo.w2 = o; o += d * f;
      lo.b2 = o; o += d;
    }
    p.layers.push_back(lo);
  }
  if (dm.kind == 1) {
    p.lnf_g = o; o += d;
    p.lnf_b = o; o += d;
    p.emb = o; o += static_cast<size_t>(dm.vocab) * d;
  }
  p.total = o;
  return p;
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
}  // namespace

Workspace make_workspace(const Dims& dm, int L, int K, int M, int max_cell_layers, bool remat, bool remat_check,
                         bool pipelined, int inflight, int depth) {
  Workspace w;
  w.depth = depth > 0 && depth < M ? depth : M;
  const size_t es = dm.dtype == 0 ? 4 : 2;
  const size_t rs = 4;                          // the residual stream and its gradient: fp32
  const size_t cs = dm.dtype == 0 ? 0 : 2;      // bf16 copies of the gradient for the GEMMs
  const size_t T = static_cast<size_t>(dm.n) * (dm.kind == 1 ? dm.seq : 1);
  const size_t Tmb = T / M;
  const size_t d = dm.d, f = dm.ffn, H = dm.kind == 1 ? dm.heads : 0;
  // slot layout (per layer, per micro-batch of Tmb tokens)
  SlotLayout s{};
  size_t so = 0;
  auto stake = [&](size_t bytes) {
    size_t at = so;
    so += align256(bytes);
    return at;
  };
  s.u = stake(Tmb * d * es);
  if (dm.kind == 1) {
    s.qkv = stake(Tmb * 3 * d * es);
    s.o = stake(Tmb * d * es);
    s.h1 = stake(Tmb * d * rs);
    s.u2 = stake(Tmb * d * es);
  }
  s.z1 = stake(Tmb * f * es);
  s.g = stake(Tmb * f * es);
  s.mean1 = stake(Tmb * 4);
  s.rstd1 = stake(Tmb * 4);
  if (dm.kind == 1) {
    s.mean2 = stake(Tmb * 4);
    s.rstd2 = stake(Tmb * 4);
    s.lse = stake(Tmb * H * 4);
  }
  s.compare_bytes_last = so;
  s.y = stake(Tmb * d * rs);
  s.bytes = so;
  w.slot = s;
  w.slot_bytes = s.bytes;

  // lane layout
  LaneLayout ln{};
  size_t lo = 0;
  auto ltake = [&](size_t bytes) {
    size_t at = lo;
    lo += align256(bytes);
    return at;
  };
  ln.slots = ltake(remat ? static_cast<size_t>(max_cell_layers) * w.slot_bytes : 0);
  // a cell's gradient chain alternates g0 and g1 between its layers; the
  // first layer's input gradient goes out of the lane, so g1 is used only by
  // cells of three layers or more
  const size_t g1_rows = max_cell_layers >= 3 ? Tmb : 0;
  ln.g0 = ltake(Tmb * d * rs);
  ln.g1 = ltake(g1_rows * d * rs);
  ln.g0b = ltake(Tmb * d * cs);
  ln.g1b = ltake(g1_rows * d * cs);
  ln.gh32 = ltake(dm.kind == 1 ? Tmb * d * rs : 0);
  ln.gt = ltake(Tmb * d * es);
  for (int i = 0; i < 2; ++i) {
    ln.gf[i] = ltake(Tmb * f * es);
    if (dm.kind == 1) {
      ln.gh[i] = ltake(Tmb * d * es);
      ln.gq[i] = ltake(Tmb * 3 * d * es);
    }
  }
  const size_t parts = (Tmb + 7) / 8;
  w.scratch_bytes = Tmb * std::max<size_t>(H, 1) * 4;  // attention row sums rowsum(dO o O)
  ln.scratch = ltake(w.scratch_bytes);
  w.lnp_bytes = parts * 2 * d * 4;
  ln.lnp[0] = ltake(w.lnp_bytes);
  ln.lnp[1] = ltake(w.lnp_bytes);
  ln.bytes = lo;
  w.lane = ln;
  w.inflight = pipelined ? inflight : 1;
  w.nlanes = pipelined ? K * w.inflight : 1;

  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off += align256(bytes);
    return at;
  };
  w.stash_bytes = Tmb * d * rs;
  w.copy_bytes = Tmb * d * cs;
  // the last cell's output is read only by the head, right after the cell
  // forwarded it: a ring as deep as the head's lanes plus one (the cell can
  // write the next micro-batch while the head lanes read theirs)
  w.nheads = dm.kind == 1 && w.nlanes > 1 && M > 1 ? 2 : 1;  // a second head lane needs a second micro-batch
  w.head_depth = std::min(w.depth, w.nheads + 1);
  w.stash = take((static_cast<size_t>(K) * w.depth + w.head_depth) * w.stash_bytes);
  w.dx0 = take(dm.kind == 1 ? static_cast<size_t>(M) * w.stash_bytes : 0);
  // the gradient ring: as deep as the micro-batches in flight (at least 2, so
  // a cell can hand over m+1 while its neighbour still reads m), never deeper
  // than the micro-batches there are
  w.ring = std::min(std::max(w.inflight, 2), M);
  w.bgrad = take(static_cast<size_t>(K) * w.ring * w.stash_bytes);
  w.bgrad16 = take(static_cast<size_t>(K) * w.ring * w.copy_bytes);
  w.lanes = take(static_cast<size_t>(w.nlanes) * ln.bytes);
  w.nslots_noremat = remat ? 0 : static_cast<size_t>(L) * M;
  w.noremat_slots = take(w.nslots_noremat * w.slot_bytes);
  w.hdy = take(static_cast<size_t>(w.depth) * w.stash_bytes);
  w.hdy16 = take(static_cast<size_t>(w.depth) * w.copy_bytes);
  for (int h = 0; h < w.nheads && dm.kind == 1; ++h) {
    Workspace::Head& hb = w.head[h];
    hb.hf = take(Tmb * d * es);
    hb.meanf = take(Tmb * 4);
    hb.rstdf = take(Tmb * 4);
    hb.logits = take(Tmb * static_cast<size_t>(dm.vocab) * 4);
    hb.hgt = take(Tmb * d * es);
    hb.hlnp[0] = take(w.lnp_bytes);
    hb.hlnp[1] = take(w.lnp_bytes);
  }
  w.loss_rows = take(T * 4);
  w.act_bytes = off;
  w.misc = take(256);
  w.trace_count = 2 + static_cast<size_t>(K + 1) * M * 2;
  w.trace = take(w.trace_count * 8);
  if (remat && remat_check) {
    w.check_bytes = static_cast<size_t>(K) * max_cell_layers * w.slot_bytes;
    w.check = take(w.check_bytes);
  }
  w.total = off;
  return w;
}

MemoryModel review_memory_model(const Dims& dm, int L, int K, int M, int max_cell_layers, int depth, bool remat) {
  MemoryModel mm;
  const bool lm = dm.kind == 1;
  const size_t e = dm.dtype == 0 ? 4 : 2;
  const size_t T = static_cast<size_t>(dm.n) * (lm ? dm.seq : 1);
  const size_t Tmb = T / M;
  const size_t d = dm.d, f = dm.ffn, H = lm ? dm.heads : 0, V = lm ? dm.vocab : 0;
  const size_t D = depth > 0 && depth < M ? depth : M;
  const size_t r = 4, c = dm.dtype == 0 ? 0 : 2;  // residual stream (fp32) and bf16 gradient copies
  const size_t act = Tmb * d * r;                  // one boundary tensor of one micro-batch
  const size_t gcp = Tmb * d * (r + c);            // one residual gradient with its copy
  mm.boundary = static_cast<size_t>(K) * D * act + D * gcp + (lm ? static_cast<size_t>(M) * act : 0) + 2 * act +
                2 * static_cast<size_t>(K) * gcp;
  const size_t a = lm ? e * (6 * d + 2 * f) + 2 * d * r + 16 + 4 * H : e * (d + 2 * f) + d * r + 8;
  mm.cell = remat ? static_cast<size_t>(max_cell_layers) * Tmb * a : static_cast<size_t>(L) * M * Tmb * a;
  const size_t lnp = 2 * ((Tmb + 7) / 8) * 2 * d * 4;  // LayerNorm partial sums: a row of 2d per 8 tokens, x2
  mm.head = lm ? Tmb * (V * 4 + 2 * d * e + 8) + lnp : 0;
  mm.grads = 2 * gcp + (lm ? act : 0) + Tmb * d * e + 2 * Tmb * (f + (lm ? 4 * d : 0)) * e +
             Tmb * std::max<size_t>(H, 1) * 4 + lnp;
  mm.rows = T * 4;
  // every region of the arena starts on a 256-byte boundary (TMA and vector
  // access): at most 255 bytes of padding for each of the <= 13 regions of a
  // layer's internals and the <= 56 others
  mm.align = 256 * (13 * static_cast<size_t>(remat ? max_cell_layers : L * M) + 56);
  mm.total = mm.boundary + mm.cell + mm.head + mm.grads + mm.rows + mm.align;
  const size_t a_survey = e * ((lm ? 8 * d : 2 * d) + 2 * f) + 8;
  mm.survey = static_cast<size_t>(K) * T * d * e +
              (remat ? static_cast<size_t>(L) * Tmb * a_survey / static_cast<size_t>(K)
                     : static_cast<size_t>(L) * T * a_survey) +
              Tmb * V * 4 + 3 * Tmb * d * e;
  return mm;
}

}  // namespace gp
