"""Throughput of one synchronous GPipe training step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line.  A step is one full pass of the hot path: forward of all
M micro-batches through all K cells (boundary stash), backward with
re-materialisation and fp32 gradient accumulation, one RMSProp update.
`value` is training tokens/s over the timed steps with every input resident
in HBM; `e2e` times the same through the C ABI from pinned host buffers
(tokens copied in, loss copied out, every step).  The step does not shard
(all cells on one GPU, no collectives): with N > 1 ranks each GPU runs an
independent replica ("replicas only") and `value` adds their tokens.

--impl reference times the CPU fp64 oracle (full-batch step, no micro-batches)
on this machine's host cores on a bounded sub-batch of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "training tokens/sec per synchronous step (1×GB300) and MFU vs BF16 peak"


def model_flops(w):
    """Model FLOPs of one step (forward + backward, no re-computation): 3 F_fwd T."""
    d, f, L, V, S = w.d, w.ffn, w.L, w.vocab, w.seq
    per_tok = 2 * (4 * d * d + 2 * d * f) * L + 2 * 2 * d * (S + 1) / 2 * L + 2 * d * V
    return 3.0 * per_tok * w.tokens


def recompute_flops(w, bounds):
    """FLOPs the re-materialisation adds: every cell's forward again, except
    the output projection of each cell's last layer (its result is the
    stashed cell output).  The head is not re-computed: it runs once per
    micro-batch, loss and gradient together."""
    d, f, S = w.d, w.ffn, w.seq
    layer = 2 * (4 * d * d + 2 * d * f) + 2 * 2 * d * (S + 1) / 2
    out_proj = 2 * d * f
    tot = 0.0
    for k in range(len(bounds) - 1):
        n = bounds[k + 1] - bounds[k]
        tot += n * layer - out_proj
    return tot * w.tokens


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"], bf16_sus=j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.out.flush()
        self.out.seek(0)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.out.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# Deeper workloads are sampled in depth: the oracle runs one sequence through
# a few of the (identical) layers, and its time for the full depth is
# extrapolated linearly in the layer count from two measured depths.
SAMPLE_DEPTHS = (4, 8)


class OracleSample:
    """A bounded sample of a workload for timing the fp64 oracle on the host.

    Up to 8 layers: the oracle's full step on a sub-batch of the workload
    (1, 2, 4, ... sequences, doubled while a step takes under budget_s / 3).
    Deeper: one sequence through SAMPLE_DEPTHS[0] and SAMPLE_DEPTHS[1] layers
    of the same shape; a full-depth step's time is the deeper sample's plus
    (L - its depth) times the measured time per layer (their difference over
    the difference in depth)."""

    def __init__(self, w, budget_s=15.0):
        from synth import make_inputs
        self.w = w
        self.deep = w.L > SAMPLE_DEPTHS[1]
        if self.deep:
            self.subs = [w.replace(n=1, M=1, K=1, L=l) for l in SAMPLE_DEPTHS]
            self.inps = [make_inputs(sw) for sw in self.subs]
            self.tokens = self.subs[0].tokens
            return
        n = 1
        while True:
            sub = w.replace(n=n, M=1, K=1)
            inp = make_inputs(sub)
            dt = self._one(sub, inp)
            if dt >= budget_s / 3 or n * 2 > w.n:
                break
            n *= 2
        self.subs, self.inps, self.tokens = [sub], [inp], sub.tokens

    @staticmethod
    def _one(sub, inp):
        from oracle import model as om
        t0 = time.perf_counter()
        om.step(sub, inp["params"], inp)
        return time.perf_counter() - t0

    def warm(self):
        """One step of every sample; returns the per-layer time (deep) or None."""
        ts = [self._one(sw, ip) for sw, ip in zip(self.subs, self.inps)]
        if self.deep:
            self.t_layer = max(ts[1] - ts[0], 0.0) / (SAMPLE_DEPTHS[1] - SAMPLE_DEPTHS[0])
        return ts

    def step(self):
        """Seconds of one full-depth oracle step (measured, or extrapolated in depth)."""
        t = self._one(self.subs[-1], self.inps[-1])
        if self.deep:
            return t + (self.w.L - SAMPLE_DEPTHS[1]) * self.t_layer
        return t

    def describe(self):
        sw = self.subs[-1]
        if self.deep:
            return (f"one sequence of {sw.seq} tokens of the {self.w.name} layers, fp64 full-batch step at "
                    f"{SAMPLE_DEPTHS[0]} and {SAMPLE_DEPTHS[1]} layers; the time of the full {self.w.L} layers "
                    f"extrapolated linearly in depth (identical layers)")
        return (f"full-batch fp64 step on a sub-batch of {sw.n} sequence(s) x {sw.seq} tokens of the "
                f"{self.w.name} layers (no micro-batching)")


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    smp = OracleSample(w, budget_s=6.0)
    for _ in range(max(args.warmup, 1)):
        smp.warm()
    dt = sum(smp.step() for _ in range(args.steps)) / args.steps
    toks = smp.tokens / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": toks, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg(w, args),
        "cpu_baseline": {"value": toks, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": smp.describe()},
        "e2e": {"value": toks, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cfg(w, args):
    return {"workload": w.name, "L": w.L, "K": w.K, "M": w.M, "d": w.d, "heads": w.heads, "ffn": w.ffn,
            "seq_len": w.seq, "vocab": w.vocab, "global_batch": w.n * max(args.gpus, 1),
            "parallelism": "replicas" if args.gpus > 1 else "single-gpu (all K cells on one GPU)",
            "l2": "working set larger than L2 (parameters, gradients and RMSProp state alone exceed 129 MB)",
            "schedule": getattr(args, "schedule", "gpipe"), **({"options": dict(parse_opts(args.opt))}
                                                             if getattr(args, "opt", None) else {})}


def parse_opts(opts):
    """--opt NAME=VALUE pairs (NAME: a GPIPE_OPT_* suffix, e.g. INFLIGHT=1)."""
    out = []
    for o in opts or []:
        name, _, val = o.partition("=")
        out.append((name.strip().upper(), int(val)))
    return out


def gp_opt(args, name, default):
    """The value given to library option NAME on the command line, else default."""
    for n, v in parse_opts(getattr(args, "opt", None)):
        if n == name:
            return v
    return default


def apply_options(b, gp, args):
    gp.set_option(b.OPT_SCHEDULE, SCHEDULES[args.schedule])
    for name, val in parse_opts(getattr(args, "opt", None)):
        gp.set_option(getattr(b, "OPT_" + name), val)


# issue orders of the step (GPIPE_OPT_SCHEDULE): the review's GPipe order, or
# one-forward-one-backward (same results, shorter stash)
SCHEDULES = {"gpipe": 0, "1f1b": 1}


def gemm_roofline(b, peaks, shape, epi, eager_launches=5, reps=100, b_mn=False):
    """Time one GEMM of the library alone: CUDA events around a CUDA graph of
    `reps` back-to-back launches on the launching stream (host launch cost is
    not in the number; operands stay in L2 where they fit).  epi 1: the FFN
    first projection (K-major operands, bias + GELU, two bf16 outputs); epi 3: a
    weight gradient (MN-major operands, fp32 TMA reduce-add, bias gradient)."""
    import torch
    M, N, K = shape
    bf = torch.bfloat16
    if epi == 0 and b_mn:
        A = torch.randn(M, K, device="cuda").to(bf)
        Bw = torch.randn(K, N, device="cuda").to(bf)
        Z = torch.empty(M, N, device="cuda", dtype=bf)
        args = (1, M, N, K, A.data_ptr(), K, 1, Bw.data_ptr(), N, 0, 0, Z.data_ptr(), N, None, None, 0,
                None, None, 0)
        name = f"input-gradient GEMM (W read MN-major, bf16 store) {M}x{N}x{K}"
    elif epi == 0:
        A = torch.randn(M, K, device="cuda").to(bf)
        Bw = torch.randn(N, K, device="cuda").to(bf)
        vec = torch.zeros(N, device="cuda")
        Z = torch.empty(M, N, device="cuda", dtype=bf)
        args = (1, M, N, K, A.data_ptr(), K, 1, Bw.data_ptr(), K, 1, 0, Z.data_ptr(), N, vec.data_ptr(), None, 0,
                None, None, 0)
        name = f"projection GEMM (bias, bf16 store) {M}x{N}x{K}"
    elif epi == 2:
        A = torch.randn(M, K, device="cuda").to(bf)
        Bw = torch.randn(K, N, device="cuda").to(bf)
        X = torch.randn(M, N, device="cuda").to(bf)
        C = torch.empty(M, N, device="cuda", dtype=bf)
        args = (1, M, N, K, A.data_ptr(), K, 1, Bw.data_ptr(), N, 0, 2, C.data_ptr(), N, None, None, 0,
                None, X.data_ptr(), N)
        name = f"GELU-backward GEMM (input gradient x GELU'(z)) {M}x{N}x{K}"
    elif epi == 4:
        A = torch.randn(M, K, device="cuda").to(bf)
        Bw = torch.randn(N, K, device="cuda").to(bf)
        C = torch.empty(M, N, device="cuda")
        args = (1, M, N, K, A.data_ptr(), K, 1, Bw.data_ptr(), K, 1, 4, C.data_ptr(), N, None, None, 0,
                None, None, 0)
        name = f"logits GEMM (fp32 store) {M}x{N}x{K}"
    elif epi == 5:
        A = torch.randn(M, K, device="cuda").to(bf)
        Bw = torch.randn(N, K, device="cuda").to(bf)
        vec = torch.zeros(N, device="cuda")
        R = torch.randn(M, N, device="cuda")
        C = torch.empty(M, N, device="cuda")
        args = (1, M, N, K, A.data_ptr(), K, 1, Bw.data_ptr(), K, 1, 5, C.data_ptr(), N, vec.data_ptr(),
                R.data_ptr(), N, None, None, 0)
        name = f"residual GEMM (bias + fp32 residual, fp32 store) {M}x{N}x{K}"
    elif epi == 3:
        A = torch.randn(K, M, device="cuda").to(bf)
        Bw = torch.randn(K, N, device="cuda").to(bf)
        C = torch.zeros(M, N, device="cuda")
        vec = torch.zeros(M, device="cuda")
        args = (1, M, N, K, A.data_ptr(), M, 0, Bw.data_ptr(), N, 0, 3, C.data_ptr(), N, vec.data_ptr(), None, 0,
                None, None, 0)
        name = f"weight-gradient GEMM (fp32 reduce-add + bias gradient) {M}x{N}x{K}"
    else:
        A = torch.randn(M, K, device="cuda").to(bf)
        Bw = torch.randn(N, K, device="cuda").to(bf)
        vec = torch.zeros(N, device="cuda")
        Z = torch.empty(M, N, device="cuda", dtype=bf)
        G = torch.empty(M, N, device="cuda", dtype=bf)
        args = (1, M, N, K, A.data_ptr(), K, 1, Bw.data_ptr(), K, 1, 1, Z.data_ptr(), N, vec.data_ptr(), None, 0,
                G.data_ptr(), None, 0)
        name = f"FFN first projection GEMM (bias + GELU) {M}x{N}x{K}"
    lib = b.lib()

    def launch():
        rc = lib.gpipe_op_gemm(*args, torch.cuda.current_stream().cuda_stream)
        assert rc == 0
    for _ in range(eager_launches):
        launch()
    torch.cuda.synchronize()
    if reps == 0:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            launch()
    g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    g.replay()
    e.record()
    torch.cuda.synchronize()
    dt = s.elapsed_time(e) / 1e3 / reps
    ach = 2.0 * M * N * K / dt / 1e12
    return {"kernel": name, "achieved": ach, "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": ach / peaks["bf16"],
            "peak_source": peaks["source"] + " (burst)", "avg_launch_us": dt * 1e6,
            "timing": f"CUDA events around a graph of {reps} back-to-back launches of this GEMM alone"}


def attention_roofline(b, peaks, nseq, seq, heads, reps=50):
    """Time the causal-attention forward and backward alone (CUDA events
    around a graph of `reps` back-to-back launches) at one micro-batch's shape.
    Algorithmic work per (sequence, head): forward 4 * 64 * seq(seq+1)/2 flops
    (S = QK^T and O = PV over the visible pairs), backward 2.5x that
    (S re-computed, dP, dV, dQ, dK)."""
    import torch
    D, R = heads * 64, nseq * seq
    qkv = (torch.randn(R, 3 * D, device="cuda") * 0.5).to(torch.bfloat16)
    dout = torch.randn(R, D, device="cuda").to(torch.bfloat16)
    o = torch.empty(R, D, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(R, heads, device="cuda")
    dvec = torch.empty(R, heads, device="cuda")
    dqkv = torch.empty(R, 3 * D, device="cuda", dtype=torch.bfloat16)
    lib = b.lib()
    out = {}
    pairs = nseq * heads * seq * (seq + 1) / 2
    for name, flops, fn in (
            ("forward", 4.0 * 64 * pairs, lambda st: lib.gpipe_op_attention_fwd(
                nseq, seq, heads, qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), st)),
            ("backward", 10.0 * 64 * pairs, lambda st: lib.gpipe_op_attention_bwd(
                nseq, seq, heads, qkv.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(), dvec.data_ptr(),
                dqkv.data_ptr(), st))):
        st = torch.cuda.current_stream().cuda_stream
        for _ in range(3):
            assert fn(st) == 0
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn(torch.cuda.current_stream().cuda_stream)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        dt = e0.elapsed_time(e1) / 1e3 / reps
        out[name] = {"us": dt * 1e6, "tflops": flops / dt / 1e12, "frac": flops / dt / 1e12 / peaks["bf16"]}
    return {"kernel": f"causal attention nseq={nseq} seq={seq} heads={heads}", **out,
            "peak": peaks["bf16"], "peak_source": peaks["source"] + " (burst)"}


def layernorm_roofline(b, peaks, rows, d, reps=50):
    """Time the LayerNorm forward and backward rows (fp32 in and out, as the
    step's residual stream) alone: CUDA events around a graph of `reps`
    launches that cycle through enough row blocks that every launch reads from
    HBM (the blocks together exceed L2).  Algorithmic bytes per launch:
    forward reads x and writes y (8 d B per row) and the row statistics (8 B);
    backward reads dy, x, the residual gradient and the statistics and writes
    dx (16 d B + 8 B per row) plus one partial row per 8 rows (two d-float
    halves)."""
    import torch
    lib = b.lib()
    nbuf = max(2, -(-(256 << 20) // (rows * d * 4 * 4)))  # > 256 MB across the buffers of one pass
    xs = [torch.randn(rows, d, device="cuda") for _ in range(nbuf)]
    dys = [torch.randn(rows, d, device="cuda") for _ in range(nbuf)]
    res = [torch.randn(rows, d, device="cuda") for _ in range(nbuf)]
    ys = [torch.empty(rows, d, device="cuda") for _ in range(nbuf)]
    g = torch.ones(d, device="cuda")
    bb = torch.zeros(d, device="cuda")
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    dg = torch.zeros(d, device="cuda")
    db = torch.zeros(d, device="cuda")
    scratch = torch.empty(lib.gpipe_op_scratch_bytes(rows, 2 * d) // 4 + 64, device="cuda")
    out = {}

    def fwd(i, st):
        return lib.gpipe_op_layernorm_fwd(0, rows, d, xs[i].data_ptr(), g.data_ptr(), bb.data_ptr(),
                                          ys[i].data_ptr(), mean.data_ptr(), rstd.data_ptr(), st)

    def bwd(i, st):
        return lib.gpipe_op_layernorm_bwd(0, rows, d, dys[i].data_ptr(), xs[i].data_ptr(), mean.data_ptr(),
                                          rstd.data_ptr(), g.data_ptr(), res[i].data_ptr(), ys[i].data_ptr(),
                                          dg.data_ptr(), db.data_ptr(), scratch.data_ptr(), st)
    for name, fn, nbytes in (("forward", fwd, rows * (8 * d + 8)),
                             ("backward", bwd, rows * (16 * d + 8) + (rows + 7) // 8 * 2 * d * 4)):
        for i in range(nbuf):
            assert fn(i, torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for r in range(reps):
                fn(r % nbuf, torch.cuda.current_stream().cuda_stream)
        gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gr.replay()
        e1.record()
        torch.cuda.synchronize()
        dt = e0.elapsed_time(e1) / 1e3 / reps
        out[name] = {"us": dt * 1e6, "gbs": nbytes / dt / 1e9, "frac": nbytes / dt / 1e9 / peaks["hbm"],
                     "bytes": nbytes}
    return {"kernel": f"LayerNorm fp32 rows={rows} d={d} (the backward includes its column-sum reduction)",
            **out, "peak": peaks["hbm"], "peak_source": peaks["source"],
            "timing": f"CUDA events around a graph of {reps} launches cycling over {nbuf} buffer sets"}


EPI_NAMES = {0: "bf16 store epilogue (bias)", 1: "bias + GELU epilogue", 2: "GELU-backward epilogue",
             3: "fp32 TMA reduce-add epilogue (weight gradient, bias gradient)", 4: "fp32 store epilogue",
             5: "fp32 residual epilogue (bias + fp32 residual, fp32 store)"}


# Per-launch DRAM traffic (read + write bytes) of the roofline classes'
# heaviest shapes, (epilogue, M, N, K) -> bytes, each from one ncu capture of
# that GEMM alone (`--probe-gemm`, cold L2) with the grid the one-stream pass
# gives it (the whole GPU): the memory-scaling workload's FFN input gradient
# (W read MN-major, single-tile 128 x 128 kernel) and FFN weight gradient
# (SM-pair kernel), and the small LM's shapes.  Inside the step the operands
# are often still in L2, so this bounds a launch's DRAM traffic from above.
ROOF_TRAFFIC = {(0, 2048, 1024, 8192): 50356480, (3, 8192, 1024, 2048): 71491584,
                (0, 1024, 1024, 8192): 33594368, (0, 512, 512, 2048): 4212224, (0, 512, 1536, 512): 2119168,
                (0, 512, 512, 512): 1066496, (0, 512, 512, 1536): 3163392,
                (3, 512, 2048, 512): 6832896, (3, 2048, 512, 512): 6839040, (3, 1536, 512, 512): 5264128,
                (3, 512, 512, 512): 2114304}


def live_roofline(b, gp, st, peaks, args):
    """Roofline of the step's dominant kernel, measured live on the step's own
    data: the step runs again with every launch on one stream (cells in turn,
    weight gradients inline: GPIPE_OPT_PIPELINE = GPIPE_OPT_CONCURRENT = 0, the
    same kernels and shapes, bit-identical results), once per GEMM epilogue
    class with CUDA events around each of that class's launches (event nodes in
    the step's graph, on the stream the kernel runs on).  With nothing running
    beside it, an event pair times one kernel.  The class with the largest
    total time is the dominant one; its achieved rate is its algorithmic flops
    (2 M N K per launch) over its launches' summed durations, against the
    sustained bf16 peak (the kernel runs inside a long step)."""
    import torch
    gp.set_option(b.OPT_PIPELINE, 0)
    gp.set_option(b.OPT_CONCURRENT, 0)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    st.step(want_loss=False)  # capture the one-stream graph
    torch.cuda.synchronize()
    ev0.record()
    st.step(want_loss=False)
    ev1.record()
    torch.cuda.synchronize()
    serial_ms = ev0.elapsed_time(ev1)
    classes = {}
    for epi in sorted(EPI_NAMES):
        gp.set_option(b.OPT_KERNEL_TIMES, epi + 1)
        st.step(want_loss=False)  # captures the step with the timing events and runs it
        ms, fl, mnk = gp.kernel_times(with_shapes=True)  # the launches of that step
        if ms.size:
            shapes = {}
            for t, f, s in zip(ms, fl, mnk):
                g = shapes.setdefault(tuple(int(x) for x in s), [0.0, 0.0, 0])
                g[0] += float(t)
                g[1] += float(f)
                g[2] += 1
            classes[epi] = (float(ms.sum()), float(fl.sum()), int(ms.size), shapes)
    gp.set_option(b.OPT_KERNEL_TIMES, 0)
    gp.set_option(b.OPT_PIPELINE, gp_opt(args, "PIPELINE", 1))
    gp.set_option(b.OPT_CONCURRENT, gp_opt(args, "CONCURRENT", 1))
    if not classes:
        return None
    epi, (tot_ms, tot_fl, n, shapes) = max(classes.items(), key=lambda kv: kv[1][0])
    shape, (sh_ms, sh_fl, sh_n) = max(shapes.items(), key=lambda kv: kv[1][0])
    ach = tot_fl / (tot_ms / 1e3) / 1e12
    sh_ach = sh_fl / (sh_ms / 1e3) / 1e12
    return {"bound": "tensor",
            "kernel": f"tcgen05 GEMM, {EPI_NAMES[epi]} ({n} launches per step, {len(shapes)} shapes)",
            "achieved": ach, "peak": peaks["bf16_sus"], "unit": "TFLOP/s", "frac": ach / peaks["bf16_sus"],
            "traffic": ROOF_TRAFFIC.get((epi,) + shape),
            "peak_source": peaks["source"] + " (sustained: the kernel runs inside a long step)",
            "algorithmic_flop_per_launch": tot_fl / n, "launches_per_step": n, "avg_launch_us": tot_ms / n * 1e3,
            "share_of_one_stream_step": tot_ms / serial_ms, "one_stream_step_ms": serial_ms,
            "timing": "CUDA events around every launch of the class in one step run on one stream (cells in turn, "
                      "weight gradients inline), on the stream the kernel runs on",
            "largest_shape": {"mnk": list(shape), "launches": sh_n, "achieved": sh_ach,
                              "frac": sh_ach / peaks["bf16_sus"], "avg_launch_us": sh_ms / sh_n * 1e3},
            "classes": {EPI_NAMES[e]: {"ms_per_step": c[0], "tflops": c[1] / (c[0] / 1e3) / 1e12, "launches": c[2]}
                        for e, c in classes.items()}}


def activation_memory(b, gp, st, w):
    """Activation memory of the step against the review's bound O(N + (L/K)(N/M)).

    model: the bound written out from the shapes (gpipe_memory_model); layout:
    the workspace's activation region; touched: measured on the device, the
    4 KiB pages of that region which one step writes (the region is filled
    with a sentinel first, so this is the arena's high-water mark as the GPU
    saw it); allocated_in_step: the drop in free device memory across the step
    (the library allocates nothing itself)."""
    import torch
    mm = gp.memory_model()
    layout = mm["layout"]
    st.ws.fill_(0xA5)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    st.step(want_loss=False)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    page = 4096
    sentinel = int.from_bytes(b"\xa5" * 4, "little", signed=True)
    words = st.ws[: layout - layout % page].view(torch.int32).view(-1, page // 4)
    touched = 0
    chunk = 1 << 18  # pages per pass (1 GiB)
    for i in range(0, words.shape[0], chunk):
        touched += int((words[i:i + chunk] != sentinel).any(dim=1).sum().item())
    touched *= page
    if layout % page:
        touched += int((st.ws[layout - layout % page: layout] != 0xA5).any().item()) * (layout % page)
    del words
    out = {"model_bytes": mm["total"], "survey_model_bytes": mm["survey"], "layout_bytes": layout,
           "touched_bytes": touched, "allocated_in_step_bytes": free0 - free1,
           "within_model": touched <= mm["total"],
           "terms": {k: mm[k] for k in ("boundary", "cell", "head", "grads", "rows", "align")}}
    return out


def max_over_ranks(value, dist, device):
    """Max of a per-rank float over the process group (the slowest replica sets
    the job's time); the value itself without a group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, t_step):
    """Whole-job tokens/s of N independent replicas timed by the slowest."""
    return tokens_per_rank * world / t_step


def run_ours(args, w):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from micro_pipeline_re_gb300._build import build as _build
    if rank == 0 or world == 1:
        _build()
    if dist:
        dist.barrier()
    from micro_pipeline_re_gb300 import binding as b
    from synth import make_inputs
    peaks = load_peaks()
    inp = make_inputs(w)
    gp = b.GPipe.from_workload(w)
    apply_options(b, gp, args)
    st = b.DeviceState(gp, w, inp)
    stream = st.stream
    for _ in range(args.warmup):
        st.step(want_loss=False)
    loss = st.step()  # checks the error flag and a finite loss
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        ev0.record()
        for _ in range(args.steps):
            st.step(want_loss=False)
        ev1.record()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t_step = ev0.elapsed_time(ev1) / 1e3 / args.steps
    clocks = clk.summary()
    t_step = max_over_ranks(t_step, dist, "cuda")
    tokens_all = w.tokens * world
    value = job_throughput(w.tokens, world, t_step)
    mf = model_flops(w)
    bounds = gp.partition()
    hf = mf + recompute_flops(w, bounds)
    launches = gp.launches_per_step()

    # end to end through the C ABI from pinned host memory (tokens in, loss out)
    host_tok = torch.from_numpy(inp["tokens"]).pin_memory()
    e2e_steps = max(3, args.steps // 2)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        st.batch.copy_(host_tok, non_blocking=True)
        st.step(want_loss=True)
    t_e2e = (time.perf_counter() - t0) / e2e_steps
    t_e2e = max_over_ranks(t_e2e, dist, "cuda")
    # roofline pass after the timed region (the event nodes and the one-stream
    # issue slow the step)
    roof = live_roofline(b, gp, st, peaks, args)
    mem = activation_memory(b, gp, st, w)
    mem["executor"] = "single lane (cells in turn)" if gp_opt(args, "PIPELINE", 1) == 0 else "concurrent lanes"
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            smp = OracleSample(w)
            smp.warm()
            dt = smp.step()
            cpu = {"value": smp.tokens / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                   "sample": smp.describe() + f" ({dt:.1f} s per step)"}
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (uniform random token ids, N(0,1/d) weights)",
            "config": cfg(w, args),
            "mfu": mf / t_step / (peaks["bf16_sus"] * 1e12) * 1.0,
            "hfu": hf / t_step / (peaks["bf16_sus"] * 1e12),
            "mfu_peak": f"{peaks['bf16_sus']} TFLOP/s bf16 sustained ({peaks['source']})",
            "loss": loss, "bubble_model": gp.bubble_fraction(), "activation_memory": mem,
            "e2e": {"value": tokens_all / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": int(host_tok.numel() * 4),
                    "d2h_bytes_per_step": 4},
            "gpu_launches": int(launches * args.steps), "launches_per_step": int(launches),
            "roofline": roof, "cpu_baseline": cpu, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_sweep(args):
    """The micro-batch sweep workload over its (K, M) grid: step throughput,
    activation memory (the bound from the shapes, the layout and the bytes the
    step writes, measured on the device) and the modelled bubble
    (K-1)/(M+K-1).  One JSON line per (K, M); not the throughput line."""
    import torch
    from micro_pipeline_re_gb300._build import build as _build
    _build()
    from micro_pipeline_re_gb300 import binding as b
    from synth import SWEEP_GRID, WORKLOADS, make_inputs
    peaks = load_peaks()
    w0 = WORKLOADS[args.workload if args.workload not in ("lm_small", "lm_deep") else "lm_sweep"]
    inp = make_inputs(w0)
    for K, M in SWEEP_GRID:
        w = w0.replace(K=K, M=M)
        gp = b.GPipe.from_workload(w)
        apply_options(b, gp, args)
        free0 = torch.cuda.mem_get_info()[0]
        st = b.DeviceState(gp, w, inp)
        free1 = torch.cuda.mem_get_info()[0]
        for _ in range(max(args.warmup, 2)):
            st.step(want_loss=False)
        loss = st.step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            st.step(want_loss=False)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / args.steps
        P, wsb = gp.sizes()
        mem = activation_memory(b, gp, st, w)
        print(json.dumps({"sweep": w.name, "K": K, "M": M, "ms_per_step": t * 1e3, "tokens_per_s": w.tokens / t,
                          "mfu": model_flops(w) / t / (peaks["bf16_sus"] * 1e12), "loss": loss,
                          "bubble_model": gp.bubble_fraction(), "activation_memory": mem, "workspace_bytes": wsb,
                          "device_bytes_taken_by_state": free0 - free1}), flush=True)
        del st
        gp.close()
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="lm_deep",
                    help="the memory-scaling workload (the largest that one GPU holds) by default")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--probe-gemm", action="store_true",
                    help="only run the roofline GEMM (5 eager launches, then a timed graph); for profilers")
    ap.add_argument("--shape", default=None, help="M,N,K for --probe-gemm (default: the workload's FFN1)")
    ap.add_argument("--sms", type=int, default=0,
                    help="--probe-gemm: the GEMM's SM share (its grid as the step would size it); 0: all SMs")
    ap.add_argument("--epi", type=int, default=1,
                    help="--probe-gemm epilogue: 0 bias + bf16 store, 1 bias+GELU, 2 GELU backward, 3 weight gradient, "
                         "4 fp32 store, 5 bias + fp32 residual")
    ap.add_argument("--reps", type=int, default=100)
    ap.add_argument("--b-mn", action="store_true",
                    help="--probe-gemm --epi 0: B read MN-major, as the step's input-gradient GEMMs read W")
    ap.add_argument("--schedule", default="gpipe", choices=sorted(SCHEDULES),
                    help="issue order: gpipe (all forwards, then all backwards) or 1f1b (interleaved, shorter stash)")
    ap.add_argument("--opt", action="append", default=[], metavar="NAME=VALUE",
                    help="a library option for the step, e.g. --opt INFLIGHT=1 --opt PIPELINE=0 (repeatable)")
    ap.add_argument("--sweep", action="store_true",
                    help="the micro-batch sweep workload over its (K, M) grid (one line per point)")
    ap.add_argument("--probe-attention", action="store_true",
                    help="only time the attention forward and backward at one micro-batch of the workload")
    ap.add_argument("--probe-layernorm", type=int, default=0, metavar="ROWS",
                    help="only time the LayerNorm forward and backward alone on ROWS rows of the workload's width")
    ap.add_argument("--layers", type=int, default=0,
                    help="run the workload with this many layers instead (memory measurements at reduced L)")
    args = ap.parse_args()
    from synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.layers:
        w = w.replace(L=args.layers, K=min(w.K, args.layers), name=f"{w.name}_L{args.layers}")
    if args.probe_gemm:
        import torch
        from micro_pipeline_re_gb300._build import build as _build
        _build()
        from micro_pipeline_re_gb300 import binding as b
        shape = tuple(int(x) for x in args.shape.split(",")) if args.shape else (w.tokens // w.M, w.ffn, w.d)
        if args.sms:
            assert b.lib().gpipe_op_gemm_set_sm_share(args.sms) == 0
        print(json.dumps(gemm_roofline(b, load_peaks(), shape, args.epi, reps=args.reps, b_mn=args.b_mn)), flush=True)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.probe_attention:
        from micro_pipeline_re_gb300._build import build as _build
        _build()
        from micro_pipeline_re_gb300 import binding as b
        print(json.dumps(attention_roofline(b, load_peaks(), w.tokens_per_micro_batch // w.seq, w.seq, w.heads)),
              flush=True)
        return
    if args.probe_layernorm:
        from micro_pipeline_re_gb300._build import build as _build
        _build()
        from micro_pipeline_re_gb300 import binding as b
        print(json.dumps(layernorm_roofline(b, load_peaks(), args.probe_layernorm, w.d)), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
