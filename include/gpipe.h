/*
 * gpipe.h - C ABI of libgpipe: one synchronous GPipe training step on one GPU.
 *
 * Method: "GPipe technical review" (zzz0906.github.io, a review of Huang et
 * al., "GPipe: Easy Scaling with Micro-Batch Pipeline Parallelism").
 *   - Interface ("GPipe algorithm: minimal interface"): the user gives K (cells),
 *     M (micro-batches) and a sequence of L layers, each with a forward, its
 *     parameters and an optional cost estimate c_i.  GPipe cuts the layers into
 *     K cells of consecutive layers, minimising the variance of the per-cell
 *     summed cost.
 *   - Step ("Pipeline flow", phases 1-3): the mini-batch of N samples is split
 *     into M micro-batches; forward keeps only each cell's input (the
 *     activations at cell boundaries); backward re-computes a cell's forward
 *     before differentiating it; per-micro-batch gradients are accumulated and
 *     applied once, after all M micro-batches.
 *   - Bubble ("Bubble overhead analysis"): (K-1)/(M+K-1).
 *   - Memory ("Preliminaries 5: re-materialisation"): peak activation memory
 *     O(N + (L/K)(N/M)) instead of O(N L).
 * Here all K cells run on one GPU: each cell owns one or more lanes of
 * concurrent CUDA streams ordered by events with exactly the pipeline's
 * dependencies (cell k works on micro-batch m while cell k+1 works on m-1;
 * with two lanes per cell, GPIPE_OPT_INFLIGHT, a cell also overlaps two of its
 * micro-batches), plus lanes for the head; or, with GPIPE_OPT_PIPELINE = 0,
 * the cells take turns on one lane.  Every parameter's gradient accumulates
 * on one stream in micro-batch order, so all schedules give identical bits.
 * The issue order is the review's GPipe order by default; GPIPE_OPT_SCHEDULE 1
 * interleaves each cell's forwards and backwards (one-forward-one-backward, the
 * order the review's "Historical impact" section credits to PipeDream-2BW for
 * its lower activation peak), which keeps min(M, K+1) micro-batches per cell
 * boundary in the stash instead of M.
 *
 * Conventions for every function:
 *   - Return value: 0 (GPIPE_OK) or a negative GPIPE_ERR_* code; the message of
 *     the last failure is available from gpipe_last_error(ctx).
 *   - Device pointers are CUDA device addresses owned by the caller; the
 *     library never allocates device memory for them, never frees them and
 *     keeps no pointer after the call returns (except inside a cached CUDA
 *     graph, which is re-captured whenever any pointer changes).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is stream-ordered; only functions with a host output that depends on
 *     device results (loss_out) synchronise the stream.
 *   - No function is thread-safe on the same context.
 */
#ifndef GPIPE_H
#define GPIPE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gpipe_ctx gpipe_ctx;  /* opaque, host-side, owned by the library */

enum {
  GPIPE_OK = 0,
  GPIPE_ERR_INVALID_ARG = -1,     /* bad shape/argument; nothing was launched          */
  GPIPE_ERR_NOT_PARTITIONED = -2, /* reserved: create always partitions                */
  GPIPE_ERR_CUDA = -3,            /* a CUDA runtime/driver call failed                 */
  GPIPE_ERR_DEVICE_TIMEOUT = -4,  /* a bounded device-side wait gave up (error flag)   */
  GPIPE_ERR_NONFINITE_LOSS = -5,  /* the step's loss is NaN or Inf                     */
  GPIPE_ERR_UNSUPPORTED = -6,     /* valid request this build does not implement       */
  GPIPE_ERR_IO = -7               /* a checkpoint file cannot be read or written, is
                                     corrupt, or belongs to another model            */
};

enum { GPIPE_KIND_FFN = 0, GPIPE_KIND_LM = 1 };
enum { GPIPE_DTYPE_F32 = 0, GPIPE_DTYPE_BF16 = 1 };

/* Layer dimensions shared by all L identical layers.
 *   kind 0: y = x + W2 GELU(W1 LN(x) + b1) + b2, MSE loss on fp32 targets.
 *   kind 1: pre-LN Transformer block (causal multi-head attention with head
 *           width d/heads = 64, GELU FFN), final LN, tied-embedding head,
 *           next-token cross-entropy over N(seq-1) targets.
 * dtype 0: everything fp32 (kind 0 only).  dtype 1: bf16 GEMM/attention
 * operands and activations with fp32 accumulation; fp32 master weights,
 * gradients and RMSProp state.
 * RMSProp: v = decay v + (1-decay) g^2;  w -= lr g / (sqrt(v) + eps).      */
typedef struct {
  int kind;
  int d, heads, ffn, seq, vocab; /* seq = 1 and vocab = 0 for kind 0          */
  int n;                         /* mini-batch N (sequences, or rows for kind 0) */
  int dtype;
  float lr, decay, eps;
} gpipe_dims;

/* Create a context for L layers cut into K cells and M micro-batches.
 * cost: L per-layer cost estimates c_i (>= 1), or NULL for the layer's forward
 * FLOPs per token: 2(4d^2 + 2d ffn) + 2d(seq+1) (kind 1), 4d ffn (kind 0).
 * Validates 1 <= K <= L, M >= 1, N % M == 0; kind 1: d % 64 == 0,
 * d/heads == 64, seq % 64 == 0, ffn % 64 == 0, vocab % 8 == 0; kind 0: d % 8 == 0,
 * ffn % 8 == 0; then partitions.
 * On failure *out is NULL and the return code says why; gpipe_last_error(NULL)
 * returns this thread's last message. */
int gpipe_create(gpipe_ctx** out, int L, int K, int M, const gpipe_dims* dims,
                 const int64_t* cost);

/* The same for layers of unequal FFN width (heterogeneous layers; the review's
 * "Limitations 3: load imbalance"): ffn is a host array of L int32 widths,
 * each validated like dims->ffn, or NULL for dims->ffn everywhere.  With ffn
 * given, dims->ffn is ignored.  Layer l's W1 is [ffn[l], d], b1 [ffn[l]] and W2
 * [d, ffn[l]] in the packing, and its default cost uses ffn[l], so the
 * partition balances the widths.  The workspace is sized for the widest. */
int gpipe_create_layers(gpipe_ctx** out, int L, int K, int M, const gpipe_dims* dims,
                        const int32_t* ffn, const int64_t* cost);

/* Re-partition an existing context on new per-layer costs (L host int64, each
 * >= 1), e.g. times measured with GPIPE_OPT_LAYER_TIMES: the same exact
 * variance-minimising cut as gpipe_create.  The workspace size may change
 * (the largest cell sizes it): query gpipe_sizes again before the next step.
 * The parameter packing does not change.  Host only, no CUDA call. */
int gpipe_repartition(gpipe_ctx* ctx, const int64_t* cost);

/* Cell bounds of the variance-minimising partition ("minimal interface"):
 * bounds_out[0] = 0 < bounds_out[1] < ... < bounds_out[K] = L; cell k holds
 * layers [bounds_out[k], bounds_out[k+1]).  Exact integer objective
 * (sum of squared cell costs); ties go to the lexicographically smallest
 * bounds.  bounds_out: host array of K+1 int32. */
int gpipe_partition(gpipe_ctx* ctx, int32_t* bounds_out);

/* Parameter count and workspace bytes the caller must allocate.
 * Parameter packing (same element offsets in every per-parameter buffer):
 *   per layer l = 0..L-1, kind 1: ln1_g[d] ln1_b[d] w_qkv[3d,d] b_qkv[3d]
 *     w_o[d,d] b_o[d] ln2_g[d] ln2_b[d] w1[ffn,d] b1[ffn] w2[d,ffn] b2[d];
 *   kind 0: ln_g[d] ln_b[d] w1[ffn,d] b1[ffn] w2[d,ffn] b2[d];
 *   then (kind 1) lnf_g[d] lnf_b[d] emb[vocab,d].
 * Matrices are [out, in] row-major (a projection computes x W^T).  w_qkv stacks
 * the query, key and value rows; head h owns rows h*64..h*64+63 of each.
 * Either output pointer may be NULL. */
int gpipe_sizes(const gpipe_ctx* ctx, size_t* param_elems, size_t* workspace_bytes);

/* Write the bf16 compute copy of the fp32 master weights (dtype 1; a no-op for
 * dtype 0).  Call once before the first step; every step's update rewrites it. */
int gpipe_init_params(gpipe_ctx* ctx, const float* params_fp32, void* params_bf16, void* stream);

/* One synchronous training step (forward of all M micro-batches through all K
 * cells keeping only cell inputs, backward with re-computation and fp32
 * gradient accumulation, then one RMSProp update of every parameter).
 *   params_fp32 [P] fp32 master weights (updated in place)
 *   params_bf16 [P] bf16 compute copy (dtype 1; rewritten by the update;
 *               ignored and may be NULL for dtype 0)
 *   grads_fp32  [P] fp32 gradient accumulator; must be all zero on entry; the
 *               update leaves it zero again (unless GPIPE_OPT_KEEP_GRADS)
 *   rms_v_fp32  [P] fp32 RMSProp state (zero before the first step)
 *   batch_in    kind 1: int32 token ids [N, seq]; kind 0: fp32 x [N, d]
 *   targets     kind 1: NULL (next-token targets come from batch_in);
 *               kind 0: fp32 targets [N, d]
 *   workspace   device buffer of gpipe_sizes' workspace_bytes, 256-B aligned;
 *               holds the boundary stash, each lane's re-computed cell
 *               internals and all scratch.  Its contents need no
 *               initialisation.
 *   loss_out    host float* or NULL.  When non-NULL the stream is synchronised,
 *               the device error flag is checked and the mean loss is written.
 * The step is captured into a CUDA graph on first use (per pointer set) and
 * replayed afterwards unless GPIPE_OPT_GRAPH is 0.  The library creates its own
 * streams and events (host-side objects) on the first call; the caller's
 * stream waits for all of them before the call's work is complete. */
int gpipe_step(gpipe_ctx* ctx, float* params_fp32, void* params_bf16, float* grads_fp32,
               float* rms_v_fp32, const void* batch_in, const void* targets,
               void* workspace, void* stream, float* loss_out);

/* (K-1)/(M+K-1), the review's bubble fraction for the context's K and M. */
double gpipe_bubble_fraction(const gpipe_ctx* ctx);

/* Discrete-event model of the pipeline clock on K devices for this context's
 * K, M and issue order (GPIPE_OPT_SCHEDULE): t_f[k], t_b[k] are per-cell
 * forward/backward times of one micro-batch (host arrays of K doubles, or NULL
 * for the partition's cell costs with t_b = 2 t_f); the head takes no time.
 * Outputs (any may be NULL): makespan, bubble fraction. */
int gpipe_schedule_model(const gpipe_ctx* ctx, const double* t_f, const double* t_b,
                         double* makespan, double* bubble);

/* The order in which gpipe_step issues its operations (host only, no CUDA
 * call; the review's "Pipeline flow" order, or the interleaved order of
 * GPIPE_OPT_SCHEDULE 1): (2K+1) M operations, written as int32 quadruples (kind, k, m, tick)
 * into ops_out (room for `count` of them; ops_out may be NULL when count is
 * 0).  kind 0 = forward of cell k for micro-batch m (the embedding first when
 * k = 0), 1 = the head of micro-batch m (k = 0), 2 = backward of cell k with
 * its re-computation.  tick = the round of the list scheduler that issued it.
 * Returns the number of operations, or a negative GPIPE_ERR_* code. */
int gpipe_issue_order(const gpipe_ctx* ctx, int32_t* ops_out, int count);

/* Activation memory of the step (bytes).  Source: the GPipe review's
 * "Preliminaries 5: re-materialisation" (only cell-boundary activations are
 * kept, so the peak falls from O(N L) to O(N + (L/K)(N/M))).
 *   peak_act_bytes    the workspace's activation region as laid out for the
 *                     current options: every byte of it is written by a step
 *                     (the high-water mark of the caller's arena);
 *   model_bound_bytes that bound written out in bytes from the model's shapes
 *                     alone (gpipe_memory_model's total), independent of the
 *                     layout: with all K cells on one device and one cell
 *                     differentiated at a time.  The single-lane executor
 *                     (GPIPE_OPT_PIPELINE 0) stays within it; the default
 *                     executor runs the K cells as concurrent lanes, each
 *                     with its own cell workspace, and exceeds it by about
 *                     (lanes - 1) cell workspaces (the price of running the
 *                     K cells at once, as K accelerators would).
 * Either output may be NULL. */
int gpipe_memory_report(const gpipe_ctx* ctx, size_t* peak_act_bytes, size_t* model_bound_bytes);

/* The terms of that bound, and the layout's total, in bytes (T tokens per
 * step, Tmb = T/M, e = GEMM operand element bytes, r = 4: the residual stream
 * and its gradient are kept in fp32, c = 2 (0 for the fp32 model): the bf16
 * copy of a gradient that a GEMM reads, D = stash depth: M in the GPipe
 * order, min(M, K+1) with GPIPE_OPT_SCHEDULE 1):
 *   [0] boundary  O(N): every cell's input for D micro-batches (K D Tmb d r),
 *                 the head's output gradient (D Tmb d (r + c)), for the LM the
 *                 embedding's input gradient (M Tmb d r), two head inputs
 *                 (2 Tmb d r), and the gradient each cell receives,
 *                 double-buffered (2 K Tmb d (r + c))
 *   [1] cell      O((L/K)(N/M)): one cell of Lc layers of internals for one
 *                 micro-batch, Lc Tmb a, a = e (6d + 2 ffn) + 2 d r + 16 + 4 heads
 *                 (FFN block: e (d + 2 ffn) + d r + 8); without
 *                 re-materialisation L M Tmb a
 *   [2] head      one micro-batch's fp32 logits, final-LN output, gradient
 *                 and statistics, and its LayerNorm partial sums:
 *                 Tmb (4 V + 2 d e + 8) + 2 ceil(Tmb/8) 2d 4 (LM only)
 *   [3] grads     one layer's backward working set for one micro-batch
 *   [4] rows      per-token losses, 4 T
 *   [5] align     256-byte alignment of the arena's regions, 256 (13 Lc + 56)
 *   [6] total     [0] + ... + [5]  (= model_bound_bytes)
 *   [7] survey    the scoping survey's concrete form of the same bound, all
 *                 activations of e bytes:
 *                 K T d e + (L/K) Tmb ((8d + 2 ffn) e + 8) + 4 Tmb V + 3 Tmb d e
 *   [8] layout    the workspace's activation region (= peak_act_bytes)
 * Writes min(count, GPIPE_MEMORY_TERMS) values; returns GPIPE_MEMORY_TERMS
 * or a negative GPIPE_ERR_* code. */
#define GPIPE_MEMORY_TERMS 9
int gpipe_memory_model(const gpipe_ctx* ctx, size_t* terms_out, int count);

/* Options (defaults in brackets). */
enum {
  GPIPE_OPT_KEEP_GRADS = 1,  /* [0] 1: the update does not zero the gradients       */
  GPIPE_OPT_GRAPH = 2,       /* [1] 0: launch kernels directly, no CUDA graph        */
  GPIPE_OPT_NO_REMAT = 3,    /* [0] 1: keep every layer's internals, no re-computing;
                                set before gpipe_sizes (changes the workspace)       */
  GPIPE_OPT_REMAT_CHECK = 4, /* [-1] m >= 0: keep micro-batch m's first-forward
                                internals of every cell and count the bytes that
                                differ from the re-computed ones
                                (gpipe_debug_counters); set before gpipe_sizes       */
  GPIPE_OPT_SKIP_UPDATE = 5, /* [0] 1: accumulate gradients but apply no update     */
  GPIPE_OPT_CONCURRENT = 6,  /* [1] run weight-gradient work on side streams of each
                                lane (ordered by events); 0: in program order on the
                                lane's stream, which applies to one lane per cell and
                                one head lane, i.e. GPIPE_OPT_PIPELINE = 0 (lanes that
                                share a cell or the head always share side streams).
                                Results are identical.                              */
  GPIPE_OPT_PIPELINE = 7,    /* [1] run the K cells as K concurrent lanes, each with its
                                own cell workspace: cell k works on micro-batch m while
                                cell k+1 works on m-1, as the review's K accelerators
                                do; 0: one lane, cells in turn (least memory).  Results
                                are identical.  Set before gpipe_sizes. */
  GPIPE_OPT_PDL = 8,         /* [0] 1: launch each kernel with programmatic dependent
                                launch (it waits for its predecessor on the GPU before
                                reading memory, so only the launch overlaps).  Off by
                                default: with concurrent lanes the early-launched
                                kernels hold SM resources other lanes need.          */
  GPIPE_OPT_TRACE = 9,       /* [0] 1: write the GPU clock (ns) when every cell (and
                                the head) finishes each micro-batch's forward and
                                backward; read with gpipe_trace                      */
  GPIPE_OPT_KERNEL_TIMES = 10, /* [0] e+1 (e <= 5): bracket every GEMM launch of the step whose
                                epilogue is e (GPIPE_EPI_* of gpipe_ops.h) with timing
                                events on the stream it is launched on (recorded as
                                event nodes of the step's graph); read with
                                gpipe_kernel_times                                   */
  GPIPE_OPT_SM_SHARE = 11,   /* [100] with lanes, a GEMM's grid is this percentage of
                                its fair share of the SMs (SMs / (cells busy at its
                                tick of the schedule + 1), doubled for GEMMs of at
                                most 4 x that many 128 x 128 tiles), 25..800; the tile
                                choice follows the grid, results stay identical    */
  GPIPE_OPT_INFLIGHT = 12,   /* [0] with lanes: micro-batches each cell works on at
                                once: 1..4, or 0 = 2 when a micro-batch's FFN GEMM
                                (tokens x d x ffn) is at most 2^30 multiply-adds,
                                else 1.  S > 1 gives each cell S lanes that take
                                its micro-batches in turn (S-1 more cell workspaces
                                per cell, and a gradient ring S deep between
                                neighbouring cells) and share the cell's side streams
                                (used whatever GPIPE_OPT_CONCURRENT says), so every
                                weight gradient still accumulates in micro-batch
                                order and results are identical.  Set before
                                gpipe_sizes.                                         */
  GPIPE_OPT_SIDE_SHARE = 13, /* [100] with lanes, GEMMs on the side streams (weight
                                gradients, off the critical path) get this percentage
                                of the SM share, 5..800: a smaller grid does the same
                                tiles with fewer CTAs, so less SM time; results stay
                                identical                                            */
  GPIPE_OPT_SIDE_STREAMS = 14, /* [2] side streams per lane, 1..4: the weight-gradient
                                work of W2, W1, W_o, W_qkv and the LayerNorm
                                reductions go to stream (group mod this); a group
                                always uses the same stream, so every gradient still
                                accumulates in micro-batch order and results are
                                identical                                            */
  GPIPE_OPT_SCHEDULE = 15,   /* [0] issue order of the step.  0: the review's GPipe
                                order (every micro-batch forward through all cells,
                                then every backward), each cell boundary stashed for
                                all M micro-batches.  1: one-forward-one-backward:
                                cell k runs min(M, K+1-k) forwards, then alternates
                                one backward and one forward, so a boundary holds at
                                most min(M, K+1) micro-batches (a ring of that depth,
                                also for the head's output gradient).  Each cell
                                still differentiates its micro-batches in ascending
                                order, so results are identical.  Set before
                                gpipe_sizes (it changes the workspace size).          */
  GPIPE_OPT_LOGIT_CLIP = 16, /* [0] value v > 0: logit clipping (the review's
                                "Training stability"): the cross-entropy sees each
                                logit clamped to [-c, c], c = v / 1000 rounded to
                                fp32, and its gradient is zero where |z| > c.  0: no
                                clipping.  0 <= v <= 1e9.  The FFN model (kind 0,
                                MSE loss) has no logits and ignores it.              */
  GPIPE_OPT_LAYER_TIMES = 17 /* [0] 1: bracket every layer's first forward and its
                                backward of micro-batch 0 with CUDA events (read by
                                gpipe_layer_times), to measure per-layer costs for
                                the partition.  The durations are the layer's own
                                work only when the step runs on one stream
                                (GPIPE_OPT_PIPELINE 0 and GPIPE_OPT_CONCURRENT 0);
                                otherwise they include waits for other lanes and
                                leave out side-stream work.                          */
};
int gpipe_set_option(gpipe_ctx* ctx, int option, int64_t value);

/* Per-layer durations (ms) of the last step taken with GPIPE_OPT_LAYER_TIMES:
 * fwd_ms[l] = layer l's first forward of micro-batch 0, bwd_ms[l] = its
 * backward of micro-batch 0 (re-computation excluded), for l < count (either
 * array may be NULL).  Waits for the step's events.  Returns L, 0 if no such
 * step was issued since the option was set, or a negative GPIPE_ERR_* code.
 * Measured costs, e.g. round(1e6 (fwd_ms + bwd_ms)), can be given to
 * gpipe_create as cost estimates (partitioning on measured times). */
int gpipe_layer_times(gpipe_ctx* ctx, float* fwd_ms, float* bwd_ms, int count);

/* Checkpoints of the training state between steps (host buffers, no CUDA
 * call).  The review's "Limitations 6" notes that GPipe itself has no fault
 * tolerance and that later systems recover through checkpoints.  The state is the
 * fp32 master weights and the RMSProp state, P floats each in the packing
 * order (the gradient buffer is zero after every update), plus a step count
 * chosen by the caller; with the bf16 copy re-derived by gpipe_init_params, a
 * run resumed from it takes exactly the steps an uninterrupted run would.
 * write: to path (via path.tmp, then renamed), with the model's shape
 *        fingerprint (kind, L, d, heads, seq, vocab, dtype, every layer's FFN
 *        width) and a checksum of the payload.
 * read:  checks magic, version, parameter count, shape fingerprint, length and
 *        checksum before it writes params_fp32 / rms_v_fp32 / step_out (any
 *        failure leaves them untouched and returns GPIPE_ERR_IO).          */
int gpipe_checkpoint_write(const gpipe_ctx* ctx, const char* path, const float* params_fp32,
                           const float* rms_v_fp32, uint64_t step);
int gpipe_checkpoint_read(const gpipe_ctx* ctx, const char* path, float* params_fp32,
                          float* rms_v_fp32, uint64_t* step_out);

/* Debug read-back after a step (synchronises `stream`):
 *   remat_mismatch_bytes: bytes of re-computed internals that differ from the
 *                         first forward (GPIPE_OPT_REMAT_CHECK), else 0;
 *   error_flag:           the device error flag (0 = none); reading clears it. */
int gpipe_debug_counters(gpipe_ctx* ctx, void* workspace, void* stream,
                         uint64_t* remat_mismatch_bytes, int* error_flag);

/* Per-target losses of the last step, copied to host (synchronises `stream`):
 * kind 1: rows [N*seq] (row n*seq+t is the loss of predicting token t+1 of
 * sequence n, 0 for t = seq-1), already divided by N(seq-1); kind 0: rows [N]
 * (sum over the row of (y-t)^2 / (N d)).  host_out holds `count` floats. */
int gpipe_loss_rows(gpipe_ctx* ctx, void* workspace, void* stream, float* host_out, size_t count);

/* Timestamps of the last step taken with GPIPE_OPT_TRACE (synchronises
 * `stream`): host_out[0] = step start, [1] = step end, then for c = 0..K (c = K is
 * the head) and m = 0..M-1: [2 + (c*M + m)*2] = end of c's forward of m (the head:
 * end of its loss and gradient for m), [2 + (c*M + m)*2 + 1] = end of cell c's
 * backward of m.  Nanoseconds of the GPU clock; count <= 2 + 2(K+1)M. */
int gpipe_trace(gpipe_ctx* ctx, void* workspace, void* stream, uint64_t* host_out, size_t count);

/* Durations of the GEMM launches that GPIPE_OPT_KERNEL_TIMES selected, in the
 * last step taken (waits for that step's events): ms_out[i] = event time of
 * launch i in issue order, flops_out[i] = its algorithmic work 2*M*N*K,
 * mnk_out[3i..3i+2] = its M, N, K.  Writes min(count, n) entries (any array may
 * be NULL) and returns n, the number of timed launches per step (0 when the
 * option is off), or a negative error. */
int gpipe_kernel_times(gpipe_ctx* ctx, float* ms_out, double* flops_out, int32_t* mnk_out, int count);

/* Number of kernels one step launches. */
int64_t gpipe_launches_per_step(const gpipe_ctx* ctx);

/* Message of the last failure on ctx, or, when ctx is NULL, of this thread's
 * last failed call of any entry point (gpipe_create and the gpipe_op_* calls
 * included).  Never NULL. */
const char* gpipe_last_error(const gpipe_ctx* ctx);

/* Destroy the context and its cached graph.  NULL-safe. */
void gpipe_destroy(gpipe_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* GPIPE_H */
