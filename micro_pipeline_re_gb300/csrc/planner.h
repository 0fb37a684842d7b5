// Host planner: variance-minimising partition, GPipe clock model, parameter
// packing and the workspace (activation memory) layout.  Pure host code.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include <vector>

namespace gp {

// Contiguous K-way cut of costs[0..L) minimising sum_k S_k^2 (equivalently
// the variance of the cell sums S_k, whose total is fixed); every cell holds
// >= 1 layer; among optima the lexicographically smallest bounds.  Exact in
// 128-bit integers.  Returns false if K is out of range.
bool partition_min_variance(const std::vector<int64_t>& costs, int K, std::vector<int32_t>& bounds);

// Discrete-event GPipe clock: forwards of micro-batches 0..M-1 flow through
// cells 0..K-1, then backwards (micro-batches ascending, cells K-1..0); a
// cell starts an op when it finished its previous op and the neighbour handed
// it the data.  Returns makespan; bubble = 1 - sum busy / (K makespan).
double simulate_gpipe(int K, int M, const double* t_f, const double* t_b, double* bubble);

// One operation of a step's issue order: the forward of cell k (with the
// embedding first when k == 0), the head, or the backward (re-computation
// included) of cell k, for micro-batch m.  tick: the round of the list
// scheduler that issued it (ops of one tick can run at once).
enum OpKind { OP_FWD = 0, OP_HEAD = 1, OP_BWD = 2 };
struct Op {
  int kind, k, m, tick;
};

// Depth of the ring that holds each cell boundary (and the head's output
// gradient): M for the GPipe order (every micro-batch's stash lives until the
// backward), min(M, K + 1) for the one-forward-one-backward order.
int stash_depth(int K, int M, int schedule);

// The step's issue order.  schedule 0 (GPipe, the review's "Pipeline flow"):
// for m, for k: F(k, m), then H(m); then for m, for k = K-1..0: B(k, m).
// schedule 1 (one-forward-one-backward): cell k runs min(M, K + 1 - k)
// forwards, then alternates one backward and one forward (backwards in
// micro-batch order), then its remaining backwards; the head is a stage after
// the last cell.  The per-stage sequences are merged by a list scheduler that
// issues, round by round, every stage's next op whose producers were issued in
// earlier rounds and whose buffer slot (stash ring of depth stash_depth, the
// head's input ring of depth head_depth, input-gradient ring of depth ring)
// its previous user has released.  head_depth <= 0: stash_depth.  Returns
// false on a deadlock (cannot happen for ring >= 2, head_depth >= 1 and
// depth >= min(M, K + 1)).
bool issue_order(int K, int M, int schedule, int ring, std::vector<Op>& ops, int head_depth = 0);

// Clock of an issue order: each stage runs its ops in order; an op starts when
// its stage is free and its producers have finished (forward of cell k: t_f[k],
// backward: t_b[k], head: 0).  Same quantities as simulate_gpipe.
double simulate_order(int K, int M, const std::vector<Op>& ops, const double* t_f, const double* t_b,
                      double* bubble);

struct Dims {
  int kind, d, heads, ffn, seq, vocab, n, dtype;
  float lr, decay, eps;
};

// Element offsets of one layer's parameters in the flat packing.
struct LayerOff {
  size_t ln1_g, ln1_b, w_qkv, b_qkv, w_o, b_o, ln2_g, ln2_b, w1, b1, w2, b2;
};

struct ParamLayout {
  std::vector<LayerOff> layers;
  size_t lnf_g = 0, lnf_b = 0, emb = 0;
  size_t total = 0;
};
// ffn: per-layer FFN widths (empty: dm.ffn for every layer).
ParamLayout make_param_layout(const Dims& dm, int L, const std::vector<int>& ffn = {});

// Byte offsets of one layer's kept internals inside a slot.
struct SlotLayout {
  size_t u, qkv, o, h1, u2, z1, g, mean1, rstd1, mean2, rstd2, lse, y;
  size_t compare_bytes_last;  // bytes that are defined when the layer's output is not written (all but y)
  size_t bytes;
};

// Per-lane region (one lane per cell when the cells run as a pipeline of
// concurrent lanes; a single lane shared by all cells otherwise).
struct LaneLayout {
  size_t slots = 0;                             // re-materialised internals of one cell (Lc slots)
  size_t g0 = 0, g1 = 0, gt = 0;                // gradients in flight (g0/g1: the residual gradient, fp32)
  size_t g0b = 0, g1b = 0;                      // bf16 copies of g0/g1 (GEMM operands; bf16 models only)
  size_t gh32 = 0;                              // fp32 gradient of a layer's mid-residual h1 (Transformer)
  size_t gf[2] = {0, 0}, gh[2] = {0, 0}, gq[2] = {0, 0};  // weight-gradient operands, alternating by layer
  size_t scratch = 0;                           // attention row sums
  size_t lnp[2] = {0, 0};                       // LayerNorm-backward gamma/beta partials, alternating
  size_t bytes = 0;
};

// The residual stream (cell inputs, layer outputs, a layer's mid-residual h1)
// and the gradient flowing along it are kept in fp32 whatever the compute
// type: they add up every layer's contribution, the step's longest chains of
// additions.  Where a bf16 GEMM reads the gradient, a bf16 copy sits beside it.
struct Workspace {
  size_t stash = 0, stash_bytes = 0;        // K x depth cell inputs [Tmb, d] fp32, then head_depth head inputs
  size_t copy_bytes = 0;                    // one bf16 copy of a [Tmb, d] gradient (0: fp32 model, no copies)
  int depth = 1;                            // stash ring depth (micro-batch m in slot m mod depth)
  int head_depth = 1;                       // ring of the last cell's output (read only by the head)
  size_t dx0 = 0;                           // M x [Tmb, d]: gradient w.r.t. the embedding output (kind 1)
  size_t bgrad = 0;                         // K x ring x [Tmb, d]: gradient w.r.t. cell k's input
  size_t bgrad16 = 0;                       // its bf16 copies
  int ring = 2;                             // depth of that ring: max(2, in flight per cell), at most M
  size_t lanes = 0;                         // nlanes x lane
  int nlanes = 1;                           // K x inflight when the cells are pipelined, else 1
  int inflight = 1;                         // micro-batches a cell works on at once (its lanes)
  LaneLayout lane{};
  size_t slot_bytes = 0;
  SlotLayout slot{};
  size_t noremat_slots = 0, nslots_noremat = 0;  // L x M slots when re-materialisation is off
  struct Head {                             // one head lane's buffers (kind 1)
    size_t hf = 0, meanf = 0, rstdf = 0, logits = 0;
    size_t hgt = 0;                         // gradient temporary
    size_t hlnp[2] = {0, 0};                // LayerNorm-backward partials, alternating
  };
  Head head[2]{};
  int nheads = 1;                           // head lanes: 2 (alternate micro-batches) when pipelined and M > 1
  size_t lnp_bytes = 0;                     // ceil(Tmb / 8) x 2d fp32
  size_t hdy = 0;                           // depth x [Tmb, d]: gradient of the last cell's output per micro-batch
  size_t hdy16 = 0;                         // its bf16 copies
  size_t scratch_bytes = 0;
  size_t loss_rows = 0, misc = 0;            // misc: loss (float) at +0, remat counter (u64) at +8
  size_t trace = 0, trace_count = 0;         // phase timestamps (u64): start, end, then per (cell/head, m, phase)
  size_t check = 0, check_bytes = 0;         // re-materialisation check copies (debug)
  size_t act_bytes = 0;                      // activation bytes (everything but misc/check)
  size_t total = 0;
};

Workspace make_workspace(const Dims& dm, int L, int K, int M, int max_cell_layers, bool remat, bool remat_check,
                         bool pipelined, int inflight = 1, int depth = 0 /* 0: M */);

// The review's activation bound O(N + (L/K)(N/M)) ("Preliminaries 5:
// re-materialisation") written out in bytes from the model's shapes alone
// (nothing of the workspace layout enters it), for one device holding all K
// cells.  T tokens per step, Tmb = T/M, e activation element bytes, D the
// stash depth (M, or min(M, K+1) in the one-forward-one-backward order).
// The residual stream and its gradient take r = 4 bytes an element, with a
// bf16 copy (c = 2 bytes; 0 for the fp32 model) of every gradient a GEMM reads.
//   boundary  the O(N) term: every cell's input for D micro-batches (K D Tmb d
//             r), the head's output gradient for D micro-batches (D Tmb d (r +
//             c)) and, for the LM, the embedding's input gradient of all M
//             (M Tmb d r), the head's input for two micro-batches (2 Tmb d r)
//             and the gradient each cell receives from the next,
//             double-buffered (2 K Tmb d (r + c))
//   cell      the O((L/K)(N/M)) term: one cell (Lc layers) of kept internals
//             for one micro-batch, a bytes per token and layer (Transformer:
//             e (6d + 2 ffn) + 2d r + 16 + 4 heads, the layer's output and
//             mid-residual in fp32; FFN block: e (d + 2 ffn) + d r + 8);
//             without re-materialisation every layer of every micro-batch,
//             L M Tmb a, the O(N L) the review starts from
//   head      one micro-batch's fp32 logits and the final LayerNorm's output,
//             gradient and statistics (LM only)
//   grads     one layer's backward working set for one micro-batch: the
//             residual gradient in and out (2 Tmb d (r + c)) and the
//             mid-residual one (Tmb d r, Transformer), a GEMM output (Tmb d
//             e), the FFN-hidden, attention-output and QKV gradients
//             double-buffered (2 Tmb (ffn + 4d) e), attention row sums and
//             LayerNorm partial sums
//   rows      per-token losses (4 T)
//   align     256-byte alignment of the arena's regions
// survey: the same bound with the constants of the scoping survey's formula
// (K T d e + (L/K) Tmb ((8d + 2 ffn) e + 8) + Tmb V 4 + 3 Tmb d e), reported
// for comparison.
struct MemoryModel {
  size_t boundary = 0, cell = 0, head = 0, grads = 0, rows = 0, align = 0, total = 0, survey = 0;
};
MemoryModel review_memory_model(const Dims& dm, int L, int K, int M, int max_cell_layers, int depth, bool remat);

}  // namespace gp
