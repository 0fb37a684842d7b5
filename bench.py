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


def oracle_sample(w, budget_s=15.0):
    """Time the oracle's full step on a sub-batch sized to about budget_s."""
    from oracle import model as om
    from synth import make_inputs
    n = 1
    sub = w.replace(n=n, M=1, K=1)
    inp = make_inputs(sub)
    t0 = time.perf_counter()
    om.step(sub, inp["params"], inp)
    dt = time.perf_counter() - t0
    while dt < budget_s / 3 and n * 2 <= w.n:
        n *= 2
        sub = w.replace(n=n, M=1, K=1)
        inp = make_inputs(sub)
        t0 = time.perf_counter()
        om.step(sub, inp["params"], inp)
        dt = time.perf_counter() - t0
    return sub, inp, dt


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import model as om
    sub, inp, _ = oracle_sample(w, budget_s=6.0)
    for _ in range(args.warmup):
        om.step(sub, inp["params"], inp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        om.step(sub, inp["params"], inp)
    dt = (time.perf_counter() - t0) / args.steps
    toks = sub.tokens / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": toks, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg(w, args),
        "cpu_baseline": {"value": toks, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"full-batch fp64 step on a sub-batch of {sub.n} sequences x {sub.seq} tokens "
                                   f"of the {w.name} layers (no micro-batching)"},
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


def apply_options(b, gp, args):
    gp.set_option(b.OPT_SCHEDULE, SCHEDULES[args.schedule])
    for name, val in parse_opts(getattr(args, "opt", None)):
        gp.set_option(getattr(b, "OPT_" + name), val)


# issue orders of the step (GPIPE_OPT_SCHEDULE): the review's GPipe order, or
# one-forward-one-backward (same results, shorter stash)
SCHEDULES = {"gpipe": 0, "1f1b": 1}


def gemm_roofline(b, peaks, shape, epi, eager_launches=5, reps=100):
    """Time one GEMM of the library alone: CUDA events around a CUDA graph of
    `reps` back-to-back launches on the launching stream (host launch cost is
    not in the number; operands stay in L2 where they fit).  epi 1: the FFN
    first projection (K-major operands, bias + GELU, two bf16 outputs); epi 3: a
    weight gradient (MN-major operands, fp32 TMA reduce-add, bias gradient)."""
    import torch
    M, N, K = shape
    bf = torch.bfloat16
    if epi == 0:
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


# The kernel class the roofline reports: the GEMMs with the bf16 store
# epilogue (epilogue 0: the forward projections and the input gradients) take
# the largest share of kernel time in the step's launch list.
ROOF_EPI = 0
EPI_NAMES = {0: "bf16 store epilogue (bias / residual)", 1: "bias + GELU epilogue", 2: "GELU-backward epilogue",
             3: "fp32 TMA reduce-add epilogue (weight gradient, bias gradient)", 4: "fp32 store epilogue"}


# Per-launch DRAM traffic (read + write bytes) of GEMMs of the step's shapes,
# each from one ncu capture of that shape and epilogue alone (`--probe-gemm`,
# cold L2): (epilogue, M, N, K) -> bytes.  Inside the step the operands are
# often still in L2, so this is an upper bound of a launch's DRAM traffic.
ROOF_TRAFFIC = {(0, 1024, 1024, 8192): 33594368, (0, 512, 512, 2048): 4212224, (0, 512, 1536, 512): 2119168, (0, 512, 512, 512): 1066496,
                (0, 512, 512, 1536): 3163392,
                (3, 512, 2048, 512): 6832896, (3, 2048, 512, 512): 6839040, (3, 1536, 512, 512): 5264128,
                (3, 512, 512, 512): 2114304}


def live_roofline(kt, peaks, b):
    """Roofline of the dominant kernel: of the launches of the roofline class in
    one step (events bracket each launch on the stream it runs on, as event
    nodes of the step's graph, so durations include the concurrency of the real
    step), the GEMM shape with the largest total time."""
    ms, fl, mnk = kt
    if ms.size == 0:
        return None
    groups = {}
    for t, f, s in zip(ms, fl, mnk):
        g = groups.setdefault(tuple(int(x) for x in s), [0.0, 0.0, 0])
        g[0] += float(t)
        g[1] += float(f)
        g[2] += 1
    shape, (tot_ms, tot_fl, n) = max(groups.items(), key=lambda kv: kv[1][0])
    ach = tot_fl / (tot_ms / 1e3) / 1e12
    cls = float(fl.sum()) / (float(ms.sum()) / 1e3) / 1e12
    return {"bound": "tensor",
            "kernel": f"tcgen05 GEMM {shape[0]}x{shape[1]}x{shape[2]}, {EPI_NAMES[ROOF_EPI]}",
            "achieved": ach, "peak": peaks["bf16_sus"], "unit": "TFLOP/s", "frac": ach / peaks["bf16_sus"],
            "traffic": ROOF_TRAFFIC.get((ROOF_EPI,) + shape),
            "peak_source": peaks["source"] + " (sustained: the kernel runs inside a long step)",
            "algorithmic_flop_per_launch": tot_fl / n, "launches_per_step": n, "avg_launch_us": tot_ms / n * 1e3,
            "timing": "CUDA events around every launch of the class in one step (a pass after the timed region: "
                      "the same graph plus the event nodes), on the stream it runs on",
            "class": {"launches_per_step": int(ms.size), "achieved": cls, "frac": cls / peaks["bf16_sus"],
                      "shapes": len(groups)},
            "isolated": gemm_roofline(b, peaks, shape, ROOF_EPI)}


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
    # roofline pass: the same step again with timing events around every launch
    # of the roofline class (the event nodes slow the step, so not in the region above)
    gp.set_option(b.OPT_KERNEL_TIMES, ROOF_EPI + 1)
    for _ in range(2):
        st.step(want_loss=False)
    for _ in range(min(args.steps, 5)):
        st.step(want_loss=False)
    kt = gp.kernel_times(with_shapes=True)  # the launches of the last of these steps
    gp.set_option(b.OPT_KERNEL_TIMES, 0)
    roof = live_roofline(kt, peaks, b)
    peak_act, bound = gp.memory_report()
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            sub, _, dt = oracle_sample(w)
            cpu = {"value": sub.tokens / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                   "sample": f"one full-batch fp64 oracle step on {sub.n} sequence(s) x {sub.seq} tokens of the "
                             f"{w.name} layers ({dt:.1f} s)"}
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (uniform random token ids, N(0,1/d) weights)",
            "config": cfg(w, args),
            "mfu": mf / t_step / (peaks["bf16_sus"] * 1e12) * 1.0,
            "hfu": hf / t_step / (peaks["bf16_sus"] * 1e12),
            "mfu_peak": f"{peaks['bf16_sus']} TFLOP/s bf16 sustained ({peaks['source']})",
            "loss": loss, "bubble_model": gp.bubble_fraction(), "peak_activation_bytes": peak_act,
            "activation_bound_bytes": bound,
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
    peak activation bytes (the workspace's activation high-water mark, which
    is what is allocated) against the review's bound, and the modelled bubble
    (K-1)/(M+K-1).  One JSON line per (K, M); not the throughput line."""
    import torch
    from micro_pipeline_re_gb300._build import build as _build
    _build()
    from micro_pipeline_re_gb300 import binding as b
    from synth import SWEEP_GRID, WORKLOADS, make_inputs
    peaks = load_peaks()
    w0 = WORKLOADS[args.workload if args.workload != "lm_small" else "lm_sweep"]
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
        peak, bound = gp.memory_report()
        P, wsb = gp.sizes()
        print(json.dumps({"sweep": w.name, "K": K, "M": M, "ms_per_step": t * 1e3, "tokens_per_s": w.tokens / t,
                          "mfu": model_flops(w) / t / (peaks["bf16_sus"] * 1e12), "loss": loss,
                          "bubble_model": gp.bubble_fraction(), "peak_activation_bytes": peak,
                          "activation_bound_bytes": bound, "workspace_bytes": wsb,
                          "device_bytes_taken_by_state": free0 - free1}), flush=True)
        del st
        gp.close()
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="lm_small")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--probe-gemm", action="store_true",
                    help="only run the roofline GEMM (5 eager launches, then a timed graph); for profilers")
    ap.add_argument("--shape", default=None, help="M,N,K for --probe-gemm (default: the workload's FFN1)")
    ap.add_argument("--sms", type=int, default=0,
                    help="--probe-gemm: the GEMM's SM share (its grid as the step would size it); 0: all SMs")
    ap.add_argument("--epi", type=int, default=1,
                    help="--probe-gemm epilogue: 0 bias + bf16 store, 1 bias+GELU, 2 GELU backward, 3 weight gradient, "
                         "4 fp32 store")
    ap.add_argument("--reps", type=int, default=100)
    ap.add_argument("--schedule", default="gpipe", choices=sorted(SCHEDULES),
                    help="issue order: gpipe (all forwards, then all backwards) or 1f1b (interleaved, shorter stash)")
    ap.add_argument("--opt", action="append", default=[], metavar="NAME=VALUE",
                    help="a library option for the step, e.g. --opt INFLIGHT=1 --opt PIPELINE=0 (repeatable)")
    ap.add_argument("--sweep", action="store_true",
                    help="the micro-batch sweep workload over its (K, M) grid (one line per point)")
    args = ap.parse_args()
    from synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.probe_gemm:
        import torch
        from micro_pipeline_re_gb300._build import build as _build
        _build()
        from micro_pipeline_re_gb300 import binding as b
        shape = tuple(int(x) for x in args.shape.split(",")) if args.shape else (w.tokens // w.M, w.ffn, w.d)
        if args.sms:
            assert b.lib().gpipe_op_gemm_set_sm_share(args.sms) == 0
        print(json.dumps(gemm_roofline(b, load_peaks(), shape, args.epi, reps=args.reps)), flush=True)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
