"""The step executor's ordering and memory bounds, checked on the CPU.

The library's own executor (gpipe.cpp) and planner are compiled with g++
against a stand-in CUDA runtime (tests/dryrun) that records, in host issue
order, every stream work item with the byte ranges it reads, writes or
accumulates into, and every event record and wait.  From that log:

* bounds: every range lies inside one of the buffers passed to gpipe_step
  (parameters, their bf16 copy, gradients, RMSProp state, batch, targets,
  workspace of gpipe_sizes bytes);
* races: any two accesses to overlapping bytes, one of them a write or an
  accumulation (two accumulations too: their order fixes the fp32 result;
  only integer atomic counts may meet unordered), are ordered by
  happens-before: stream order plus event edges (a wait orders after the work
  its event's last record followed).  Vector clocks over the streams decide
  the order.

This covers every issue order, in-flight count, side-stream count and lane
arrangement without a GPU; the GPU tests check the same schedules for
identical bits.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from synth import KIND_FFN, KIND_LM, WORKLOADS, Workload, param_count

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "micro_pipeline_re_gb300", "csrc")
SOURCES = [os.path.join(CSRC, "gpipe.cpp"), os.path.join(CSRC, "planner.cpp"),
           os.path.join(HERE, "dryrun", "dryrun.cpp")]
HEADERS = [os.path.join(HERE, "dryrun", "cuda_runtime.h"), os.path.join(CSRC, "kernels.h"),
           os.path.join(CSRC, "planner.h"), os.path.join(CSRC, "launch_util.cuh"),
           os.path.join(ROOT, "include", "gpipe.h")]
OUT = os.path.join(HERE, "dryrun", "_build", "libgpipe_dry.so")

OPT = dict(KEEP_GRADS=1, GRAPH=2, NO_REMAT=3, REMAT_CHECK=4, SKIP_UPDATE=5, CONCURRENT=6, PIPELINE=7, PDL=8,
           TRACE=9, KERNEL_TIMES=10, SM_SHARE=11, INFLIGHT=12, SIDE_SHARE=13, SIDE_STREAMS=14, SCHEDULE=15,
           LOGIT_CLIP=16, LAYER_TIMES=17)


def load_dry():
    """Build (when a source is newer) and load the dry-run library."""
    newest = max(os.path.getmtime(p) for p in SOURCES + HEADERS)
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < newest:
        os.makedirs(os.path.dirname(OUT), exist_ok=True)
        tmp = "%s.%d.tmp" % (OUT, os.getpid())   # concurrent test processes each build their own
        subprocess.run(["g++", "-std=c++17", "-O1", "-shared", "-fPIC", "-I", os.path.join(HERE, "dryrun"),
                        "-I", CSRC] + SOURCES + ["-Wl,--no-undefined", "-o", tmp], check=True)
        os.replace(tmp, OUT)
    lib = ctypes.CDLL(OUT)
    from micro_pipeline_re_gb300.binding import Dims
    c_int, c_vp, c_sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    lib.gpipe_create_layers.argtypes = [ctypes.POINTER(c_vp), c_int, c_int, c_int, ctypes.POINTER(Dims),
                                        ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)]
    lib.gpipe_set_option.argtypes = [c_vp, c_int, ctypes.c_int64]
    lib.gpipe_sizes.argtypes = [c_vp, ctypes.POINTER(c_sz), ctypes.POINTER(c_sz)]
    lib.gpipe_step.argtypes = [c_vp] * 9 + [ctypes.POINTER(ctypes.c_float)]
    lib.gpipe_destroy.argtypes = [c_vp]
    lib.gpipe_last_error.argtypes = [c_vp]
    lib.gpipe_last_error.restype = ctypes.c_char_p
    lib.dry_entry.argtypes = [c_int] + [ctypes.POINTER(c_int)] * 4 + [ctypes.c_char_p, c_int]
    lib.dry_access.argtypes = [c_int, c_int, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64),
                               ctypes.c_char_p]
    lib.Dims = Dims
    return lib


@pytest.fixture(scope="module")
def dry():
    return load_dry()


def _log(lib):
    entries = []
    t, s, e, n = (ctypes.c_int() for _ in range(4))
    name = ctypes.create_string_buffer(64)
    lo, hi = ctypes.c_uint64(), ctypes.c_uint64()
    mode = ctypes.create_string_buffer(2)
    for i in range(lib.dry_entries()):
        assert lib.dry_entry(i, t, s, e, n, name, 64) == 0
        acc = []
        for j in range(n.value):
            assert lib.dry_access(i, j, lo, hi, mode) == 0
            acc.append((lo.value, hi.value, mode.value.decode()))
        entries.append((t.value, s.value, e.value, name.value.decode(), acc))
    return entries


def run_step(lib, w, options=(), K=None, M=None):
    """Create a context, take one dry step; returns (log, buffers)."""
    K, M = K or w.K, M or w.M
    dims = lib.Dims(w.kind, w.d, w.heads, w.ffn, w.seq if w.kind == KIND_LM else 1, w.vocab, w.n,
                    0 if w.dtype == "f32" else 1, w.lr, w.decay, w.eps)
    h = ctypes.c_void_p()
    widths = (ctypes.c_int32 * w.L)(*w.ffn_layers) if w.ffn_layers else None
    rc = lib.gpipe_create_layers(ctypes.byref(h), w.L, K, M, ctypes.byref(dims), widths, None)
    assert rc == 0, lib.gpipe_last_error(None)
    try:
        for opt, val in options:
            assert lib.gpipe_set_option(h, OPT[opt], val) == 0, (opt, val)
        P, ws = ctypes.c_size_t(), ctypes.c_size_t()
        assert lib.gpipe_sizes(h, ctypes.byref(P), ctypes.byref(ws)) == 0
        assert P.value == param_count(w)
        sizes = {"p32": P.value * 4, "p16": P.value * 2, "g32": P.value * 4, "v32": P.value * 4,
                 "batch": w.n * (w.seq * 4 if w.kind == KIND_LM else w.d * 4),
                 "targets": w.n * w.d * 4 if w.kind == KIND_FFN else 0, "ws": ws.value}
        bufs, at = {}, 1 << 40
        for k, v in sizes.items():
            bufs[k] = (at, at + v)
            at += (v + (1 << 20)) & ~0xFFFF  # a gap after every buffer
        lib.dry_reset()
        ptr = lambda k: ctypes.c_void_p(bufs[k][0]) if sizes[k] else None
        rc = lib.gpipe_step(h, ptr("p32"), ptr("p16") if w.dtype == "bf16" else None, ptr("g32"), ptr("v32"),
                            ptr("batch"), ptr("targets"), ptr("ws"), None, None)
        assert rc == 0, lib.gpipe_last_error(h)
        return _log(lib), bufs
    finally:
        lib.gpipe_destroy(h)


def check_bounds(log, bufs):
    spans = sorted(v for v in bufs.values() if v[1] > v[0])
    for _, _, _, name, acc in log:
        for lo, hi, mode in acc:
            if hi == lo:
                continue
            assert any(a <= lo and hi <= b for a, b in spans), (name, hex(lo), hi - lo, mode)


def check_races(log):
    """Returns the number of work items; raises on an unordered conflict."""
    dense = {s: i for i, s in enumerate(sorted({e[1] for e in log}))}
    log = [(t, dense[s], e, n, a) for t, s, e, n, a in log]
    nstreams = len(dense)
    vc = np.zeros((nstreams, nstreams), dtype=np.int64)   # per stream: its vector clock
    ev = {}
    op_stream, op_vc, op_name = [], [], []
    lo_l, hi_l, md_l, cnt_l, op_l = [], [], [], [], []
    for typ, s, e, name, acc in log:
        if typ == 0:
            vc[s, s] += 1
            k = len(op_stream)
            op_stream.append(s)
            op_vc.append(vc[s].copy())
            op_name.append(name)
            for lo, hi, mode in acc:
                if hi > lo:
                    lo_l.append(lo), hi_l.append(hi), md_l.append(mode != "R"), cnt_l.append(mode == "I")
                    op_l.append(k)
        elif typ == 1:
            ev[e] = vc[s].copy()
        elif e in ev:
            np.maximum(vc[s], ev[e], out=vc[s])
    op_stream = np.array(op_stream)
    op_vc = np.array(op_vc)
    lo, hi = np.array(lo_l, dtype=np.uint64), np.array(hi_l, dtype=np.uint64)
    wr, cnt, op = np.array(md_l), np.array(cnt_l), np.array(op_l)
    own = op_vc[np.arange(len(op_stream)), op_stream]     # each op's own clock component
    for j in range(len(lo)):
        i = np.arange(j)
        cand = i[(op[i] != op[j]) & (lo[i] < hi[j]) & (lo[j] < hi[i]) & (wr[i] | wr[j]) & ~(cnt[i] & cnt[j])]
        if cand.size == 0:
            continue
        a = op[cand]
        ordered = own[a] <= op_vc[op[j], op_stream[a]]
        if not np.all(ordered):
            bad = a[~ordered][0]
            raise AssertionError(f"unordered conflict: {op_name[bad]} (stream {op_stream[bad]}) and "
                                 f"{op_name[op[j]]} (stream {op_stream[op[j]]}) on [{hex(int(lo[j]))}, +{int(hi[j] - lo[j])})")
    return len(op_stream)


def accumulation_order(log, bufs, w, M):
    """Per gradient tensor (byte range in the gradient buffer), the sequence of
    (kernel, micro-batch) that accumulate into it, in issue order (which is
    their happens-before order: check_races has shown they are ordered).  A
    kernel's micro-batch follows the data: the kernels that read a micro-batch's
    own inputs (its tokens or rows, its targets) carry its index, and any other
    kernel carries the largest index among the last writers of what it reads."""
    check_races(log)
    tmb = w.tokens // M
    b0, b1 = bufs["batch"]
    t0, t1 = bufs["targets"]
    g0, g1 = bufs["g32"]
    row_bytes = 4 if w.kind == KIND_LM else 4 * w.d
    wlo, whi, wtag = [], [], []
    order = {}
    for typ, s, e, name, acc in log:
        if typ != 0:
            continue
        tag = -1
        for lo, hi, mode in acc:
            if mode != "R" or hi <= lo:
                continue
            if b0 <= lo < b1:
                tag = max(tag, (lo - b0) // row_bytes // tmb)
            elif t0 <= lo < t1:
                tag = max(tag, (lo - t0) // (4 * w.d) // tmb)
            elif wlo:
                L_, H_ = np.array(wlo, dtype=np.uint64), np.array(whi, dtype=np.uint64)
                hit = np.nonzero((L_ < hi) & (lo < H_))[0]
                if hit.size:
                    tag = max(tag, wtag[hit[-1]])
        for lo, hi, mode in acc:
            if mode in "WA" and hi > lo:
                wlo.append(lo), whi.append(hi), wtag.append(tag)
                if mode == "A" and g0 <= lo and hi <= g1:
                    order.setdefault((lo - g0, hi - g0), []).append((name, tag))
    return order


SMALL = Workload("dry_lm", KIND_LM, L=4, K=2, M=4, d=128, heads=2, ffn=256, seq=64, vocab=512, n=8, dtype="bf16")
FFN = WORKLOADS["tiny_ffn"]

CASES = [
    ("lm", SMALL, []),
    ("lm_1f1b", SMALL, [("SCHEDULE", 1)]),
    ("lm_k4_m8_1f1b", SMALL.replace(K=4, M=8, n=16), [("SCHEDULE", 1)]),
    ("lm_k4_m8", SMALL.replace(K=4, M=8, n=16), []),
    ("lm_inflight2", SMALL.replace(K=4, M=8, n=16), [("INFLIGHT", 2)]),
    ("lm_inflight3_1f1b", SMALL.replace(K=4, M=8, n=16), [("INFLIGHT", 3), ("SCHEDULE", 1)]),
    ("lm_inflight4_sides4", SMALL.replace(K=4, M=8, n=16), [("INFLIGHT", 4), ("SIDE_STREAMS", 4)]),
    ("lm_inflight2_1f1b_sides1", SMALL.replace(K=4, M=8, n=16), [("INFLIGHT", 2), ("SCHEDULE", 1),
                                                                 ("SIDE_STREAMS", 1)]),
    ("lm_not_concurrent", SMALL.replace(K=4, M=8, n=16), [("CONCURRENT", 0), ("INFLIGHT", 1)]),
    ("lm_not_concurrent_inflight2", SMALL.replace(K=4, M=8, n=16), [("CONCURRENT", 0), ("INFLIGHT", 2)]),
    ("lm_one_lane", SMALL.replace(K=4, M=8, n=16), [("PIPELINE", 0)]),
    ("lm_one_lane_1f1b", SMALL.replace(K=4, M=8, n=16), [("PIPELINE", 0), ("SCHEDULE", 1)]),
    ("lm_one_stream", SMALL.replace(K=4, M=8, n=16), [("PIPELINE", 0), ("CONCURRENT", 0)]),
    ("lm_direct", SMALL.replace(K=4, M=8, n=16), [("GRAPH", 0), ("SCHEDULE", 1)]),
    ("lm_no_remat", SMALL.replace(K=4, M=8, n=16), [("NO_REMAT", 1), ("SCHEDULE", 1)]),
    ("lm_remat_check", SMALL.replace(K=4, M=8, n=16), [("REMAT_CHECK", 5), ("SCHEDULE", 1)]),
    ("lm_trace_times", SMALL.replace(K=4, M=8, n=16), [("TRACE", 1), ("KERNEL_TIMES", 4), ("LAYER_TIMES", 1)]),
    ("lm_k_eq_l", SMALL.replace(K=4, M=6, n=12), [("SCHEDULE", 1), ("INFLIGHT", 2)]),
    ("lm_k1", SMALL.replace(K=1, M=3, n=6), [("SCHEDULE", 1)]),
    ("lm_m1", SMALL.replace(M=1, n=2), [("SCHEDULE", 1)]),
    ("lm_m1_gpipe_inflight2", SMALL.replace(K=4, M=1, n=2), [("INFLIGHT", 2)]),
    ("lm_m2_inflight4", SMALL.replace(K=4, M=2, n=4), [("INFLIGHT", 4)]),
    ("lm_m3_inflight4_1f1b", SMALL.replace(K=4, M=3, n=6), [("INFLIGHT", 4), ("SCHEDULE", 1)]),
    ("ffn_m1", FFN.replace(M=1), []),
    ("lm_hetero", SMALL.replace(L=6, K=3, M=8, n=16, ffn_layers=(256, 64, 512, 128, 192, 320)),
     [("SCHEDULE", 1), ("INFLIGHT", 2)]),
    ("ffn", FFN, []),
    ("ffn_1f1b", FFN, [("SCHEDULE", 1)]),
    ("ffn_1f1b_inflight2", FFN.replace(M=8), [("SCHEDULE", 1), ("INFLIGHT", 2)]),
    ("ffn_not_concurrent", FFN, [("CONCURRENT", 0), ("SCHEDULE", 1)]),
]


@pytest.mark.parametrize("name,w,options", CASES, ids=[c[0] for c in CASES])
def test_executor_stays_in_bounds_and_orders_every_conflict(dry, name, w, options):
    log, bufs = run_step(dry, w, options)
    check_bounds(log, bufs)
    n = check_races(log)
    assert n > 10 * w.L


@pytest.mark.parametrize("sched", [0, 1])
def test_lm_small_full_size_orders_every_conflict(dry, sched):
    w = WORKLOADS["lm_small"]
    log, bufs = run_step(dry, w, [("SCHEDULE", sched)])
    check_bounds(log, bufs)
    assert check_races(log) > 3000


def test_checker_catches_a_missing_order(dry):
    """The checker itself: dropping from the log a cross-stream event wait
    issued after the first head (the first one whose loss matters) leaves a
    conflicting pair unordered, and the checker reports it; with every wait
    dropped it reports one too."""
    w = SMALL
    log, bufs = run_step(dry, w)
    check_races(log)
    # the first wait on a cell lane issued after the first cross_entropy
    ce = next(i for i, e in enumerate(log) if e[3] == "cross_entropy")
    rec_events = {e[2] for e in log[:ce + 60] if e[0] == 1}
    dropped = False
    for i in range(ce, len(log)):
        typ, s, e, name, _ = log[i]
        if typ == 2 and e in rec_events and s != log[ce][1]:
            trial = log[:i] + log[i + 1:]
            try:
                check_races(trial)
            except AssertionError:
                dropped = True
                break
    assert dropped
    with pytest.raises(AssertionError):
        check_races([e for e in log if e[0] != 2])


@pytest.mark.parametrize("w", [SMALL.replace(K=4, M=8, n=16), FFN.replace(M=8),
                               SMALL.replace(L=6, K=3, M=8, n=16, ffn_layers=(256, 64, 512, 128, 192, 320))],
                         ids=["lm", "ffn", "lm_hetero"])
def test_every_gradient_accumulates_in_micro_batch_order_in_every_schedule(dry, w):
    """The reason every schedule gives identical bits: for every parameter
    tensor the same kernels add into its fp32 gradient in the same order,
    micro-batch by micro-batch (0, 1, ..., M-1), whatever the issue order,
    lanes, side streams, graph or number of cells (K = 1 and K = L too)."""
    configs = [[], [("SCHEDULE", 1)], [("INFLIGHT", 2)], [("INFLIGHT", 3), ("SCHEDULE", 1)],
               [("INFLIGHT", 4), ("SIDE_STREAMS", 4)], [("PIPELINE", 0)], [("PIPELINE", 0), ("CONCURRENT", 0)],
               [("GRAPH", 0), ("SCHEDULE", 1), ("INFLIGHT", 2)], [("CONCURRENT", 0), ("SIDE_STREAMS", 1)]]
    ref = None
    cells = [(w.K, opts) for opts in configs] + [(1, []), (w.L, [("SCHEDULE", 1)]), (w.L, [("INFLIGHT", 2)])]
    for K, opts in cells:
        log, bufs = run_step(dry, w, opts, K=K)
        order = accumulation_order(log, bufs, w, w.M)
        for rng_, seq in order.items():
            ms = [m for name, m in seq if name != "embedding_bwd"]
            assert ms == sorted(ms) and ms[0] == 0 and ms[-1] == w.M - 1, (opts, rng_, seq)
        if ref is None:
            ref = order
            n_params = len(order)
        else:
            assert order == ref, opts
    assert n_params >= 4 * w.L


def touched_bytes(log, lo0, hi0):
    """Bytes of [lo0, hi0) that at least one work item of the log touches."""
    iv = sorted((max(lo, lo0), min(hi, hi0)) for _, _, _, _, acc in log for lo, hi, _ in acc if lo < hi0 and hi > lo0)
    total, cur_lo, cur_hi = 0, None, None
    for lo, hi in iv:
        if cur_hi is None or lo > cur_hi:
            if cur_hi is not None:
                total += cur_hi - cur_lo
            cur_lo, cur_hi = lo, hi
        else:
            cur_hi = max(cur_hi, hi)
    return total + (cur_hi - cur_lo if cur_hi is not None else 0)


@pytest.mark.parametrize("name", ["lm_small", "lm_wide"])
@pytest.mark.parametrize("sched", [0, 1])
def test_workspace_the_step_touches_matches_the_plan(dry, name, sched):
    """The activation memory the step actually uses (the union of the byte
    ranges its kernels touch in the workspace) against the planner's peak and
    the review's bound: used <= planned <= bound, and the plan holds no more
    than alignment and a few unused slot fields beyond what is used."""
    from micro_pipeline_re_gb300 import binding as b
    w = WORKLOADS[name]
    log, bufs = run_step(dry, w, [("SCHEDULE", sched)])
    check_bounds(log, bufs)
    g = b.GPipe.from_workload(w)
    g.set_option(b.OPT_SCHEDULE, sched)
    peak, bound = g.memory_report()
    used = touched_bytes(log, bufs["ws"][0], bufs["ws"][0] + peak)
    assert used <= peak
    assert used >= 0.97 * peak, used / peak
    # the single-lane executor: what it touches is within the review's bound
    log1, bufs1 = run_step(dry, w, [("SCHEDULE", sched), ("PIPELINE", 0)])
    check_bounds(log1, bufs1)
    g.set_option(b.OPT_PIPELINE, 0)
    peak1, bound1 = g.memory_report()
    used1 = touched_bytes(log1, bufs1["ws"][0], bufs1["ws"][0] + peak1)
    assert bound1 == bound and used1 <= peak1 <= bound
    assert used1 >= 0.97 * peak1, used1 / peak1


@pytest.mark.parametrize("name", ["lm_small", "lm_wide"])
@pytest.mark.parametrize("remat", [True, False])
def test_flop_accounting_matches_the_launched_gemms(dry, name, remat):
    """The benchmark's FLOP model (MFU counts 3 F_fwd T, HFU adds the
    re-computation) against the GEMMs the step actually launches: the sum of
    2 M N K over every GEMM equals the model's GEMM part (all but attention,
    2 d (seq+1) per token and layer in each of forward, backward x2 and
    re-computation)."""
    import bench
    w = WORKLOADS[name]
    opts = [] if remat else [("NO_REMAT", 1)]
    log, _ = run_step(dry, w, opts)
    launched = 0
    for typ, _, _, nm, _ in log:
        if typ == 0 and nm.startswith("gemm:"):
            M, N, K = (int(x) for x in nm.split(":")[1:])
            launched += 2 * M * N * K
    bounds = [k * (w.L // w.K) for k in range(w.K + 1)]
    attn_per_pass = 2 * w.d * (w.seq + 1) * w.L * w.tokens
    want = bench.model_flops(w) - 3 * attn_per_pass
    if remat:
        want += bench.recompute_flops(w, bounds) - attn_per_pass
    assert launched == pytest.approx(want, rel=1e-12)


def test_measured_activation_bytes_scale_as_the_review_bound_over_the_sweep_grid(dry):
    """The review's O(N + (L/K)(N/M)) with the bytes the step actually touches
    (dry run) over the micro-batch sweep grid: a (K+2) N + b L (N/M) + c K (N/M)
    + e H (N/M) (K lanes of one cell's internals and gradients, H head lanes
    of one micro-batch's logits: two when there are two micro-batches to
    alternate) fits every point within 10%, and every point is within its
    bound."""
    from micro_pipeline_re_gb300 import binding as b
    from synth import SWEEP_GRID
    w0 = WORKLOADS["lm_sweep"]
    rows, ys = [], []
    for K, M in SWEEP_GRID:
        w = w0.replace(K=K, M=M)
        log, bufs = run_step(dry, w)
        g = b.GPipe.from_workload(w)
        peak, bound = g.memory_report()
        used = touched_bytes(log, bufs["ws"][0], bufs["ws"][0] + peak)
        assert used <= peak
        T = w.tokens
        rows.append([(K + 2) * T, w.L * T / M, K * T / M, (2 if M > 1 else 1) * T / M])
        ys.append(used)
    A, y = np.array(rows, dtype=float), np.array(ys, dtype=float)
    coef, *_ = np.linalg.lstsq(A, y, rcond=None)
    resid = np.abs(A @ coef - y) / y
    assert resid.max() <= 0.10, resid
    assert np.all(coef > 0)


def critical_path(log):
    """Length, in work items, of the longest chain through stream order and
    event edges: the number of kernels that must run one after another."""
    last_on, ev, pending, best = {}, {}, {}, 0
    for typ, s, e, _, _ in log:
        if typ == 0:
            d = max(last_on.get(s, 0), pending.pop(s, 0)) + 1
            last_on[s] = d
            best = max(best, d)
        elif typ == 1:
            ev[e] = max(last_on.get(s, 0), pending.get(s, 0))
        elif e in ev:
            pending[s] = max(pending.get(s, 0), ev[e])
    return best


def test_lanes_shorten_the_critical_path(dry):
    """What the lanes buy on a latency-bound step (`lm_small`, ≈ 3500
    kernels): the chain of kernels that must run one after another is the
    whole step on one stream, shorter with side streams, far shorter with the
    cells as lanes, and shorter again with two micro-batches in flight per
    cell; the interleaved order lengthens it (a lane's forward waits behind its
    backward)."""
    w = WORKLOADS["lm_small"]
    cp = {}
    for key, opts in (("one_stream", [("PIPELINE", 0), ("CONCURRENT", 0)]), ("one_lane", [("PIPELINE", 0)]),
                      ("lanes", [("INFLIGHT", 1)]), ("lanes_s2", [("INFLIGHT", 2)]),
                      ("lanes_s2_1f1b", [("INFLIGHT", 2), ("SCHEDULE", 1)])):
        log, _ = run_step(dry, w, opts)
        cp[key] = critical_path(log)
        if key == "one_stream":
            assert cp[key] == sum(1 for e in log if e[0] == 0)
    assert cp["one_stream"] > cp["one_lane"] > 3 * cp["lanes"]
    assert cp["lanes_s2"] < cp["lanes"] and cp["lanes_s2"] < cp["lanes_s2_1f1b"]
