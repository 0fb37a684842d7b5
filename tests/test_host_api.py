"""CPU-only tests of libgpipe's host side through the C ABI: exported symbols,
argument validation, the partitioner, the GPipe clock model and the
activation-memory plan.  No CUDA call is made here."""
import os
import re
from fractions import Fraction

import numpy as np
import pytest

from oracle import partition as op
from oracle import schedule as osch
from synth import KIND_FFN, KIND_LM, SWEEP_GRID, WORKLOADS, Workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def binding():
    from micro_pipeline_re_gb300 import _build
    _build.build()
    from micro_pipeline_re_gb300 import binding as b
    b.lib()
    return b


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(gpipe_\w+)\s*\(", txt))
    return names


def test_library_exports_every_declared_symbol(binding):
    declared = _declared_functions()
    assert len(declared) >= 20
    lib = binding.lib()
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(binding.exported_names())


@pytest.mark.parametrize("kwargs,code", [
    (dict(L=4, K=5, M=1), -1),          # K > L
    (dict(L=4, K=0, M=1), -1),          # K < 1
    (dict(L=4, K=2, M=3), -1),          # N % M != 0 (N = 32)
    (dict(L=4, K=2, M=0), -1),
])
def test_create_rejects_bad_shapes(binding, kwargs, code):
    w = WORKLOADS["tiny_ffn"]
    with pytest.raises(binding.GpipeError) as e:
        binding.GPipe(kwargs["L"], kwargs["K"], kwargs["M"], kind=0, d=w.d, heads=0, ffn=w.ffn, seq=1, vocab=0,
                      n=w.n, dtype=0)
    assert e.value.code == code


def test_create_rejects_bad_layer_dims(binding):
    with pytest.raises(binding.GpipeError) as e:   # head width must be 64
        binding.GPipe(2, 1, 1, kind=1, d=256, heads=8, ffn=512, seq=64, vocab=256, n=2, dtype=1)
    assert e.value.code == -1
    with pytest.raises(binding.GpipeError) as e:   # seq multiple of 64
        binding.GPipe(2, 1, 1, kind=1, d=128, heads=2, ffn=512, seq=100, vocab=256, n=2, dtype=1)
    assert e.value.code == -1
    with pytest.raises(binding.GpipeError) as e:   # the LM runs in bf16
        binding.GPipe(2, 1, 1, kind=1, d=128, heads=2, ffn=512, seq=64, vocab=256, n=2, dtype=0)
    assert e.value.code == -6
    with pytest.raises(binding.GpipeError) as e:   # bad optimizer constants
        binding.GPipe(2, 1, 1, kind=0, d=64, heads=0, ffn=64, seq=1, vocab=0, n=2, dtype=0, decay=1.0)
    assert e.value.code == -1


def test_partition_matches_brute_force(binding):
    rng = np.random.default_rng(11)
    for trial in range(60):
        L = int(rng.integers(1, 13))
        K = int(rng.integers(1, L + 1))
        costs = [int(c) for c in rng.integers(1, 40, size=L)]
        g = binding.GPipe(L, K, 1, kind=0, d=64, heads=0, ffn=64, seq=1, vocab=0, n=4, dtype=0, cost=costs)
        got = g.partition()
        want, _ = op.partition(costs, K)
        assert got == want, (costs, K, got, want)
        g.close()


def test_partition_huge_costs_exact(binding):
    """Costs near 1e15 (layer FLOPs of large models): squares need 128-bit."""
    costs = [10**15 + i for i in (5, 1, 3, 2, 9, 4, 7, 8)]
    g = binding.GPipe(8, 3, 1, kind=0, d=64, heads=0, ffn=64, seq=1, vocab=0, n=4, dtype=0, cost=costs)
    assert g.partition() == op.partition(costs, 3)[0]


def test_default_costs_split_identical_layers_evenly(binding):
    for name in ("lm_small", "lm_wide", "lm_deep"):
        w = WORKLOADS[name]
        g = binding.GPipe.from_workload(w)
        assert g.partition() == [k * (w.L // w.K) for k in range(w.K + 1)]


@pytest.mark.parametrize("K,M", [(1, 1), (2, 1), (4, 32), (8, 32), (4, 4), (3, 7)])
def test_bubble_fraction_and_clock_model(binding, K, M):
    g = binding.GPipe(8 * K, K, M, kind=0, d=64, heads=0, ffn=64, seq=1, vocab=0, n=M * 2, dtype=0)
    assert g.bubble_fraction() == pytest.approx(float(Fraction(K - 1, M + K - 1)), abs=1e-15)
    mk, bub = g.schedule_model([1.0] * K, [2.0] * K)
    sim = osch.simulate(K, M, 1, 2)
    assert mk == pytest.approx(float(sim["makespan"]), rel=1e-12)
    assert bub == pytest.approx(float(sim["bubble"]), abs=1e-12)


def test_clock_model_unequal_cells(binding):
    rng = np.random.default_rng(3)
    for _ in range(10):
        K, M = int(rng.integers(1, 6)), int(rng.integers(1, 9))
        tf = [float(x) for x in rng.integers(1, 9, size=K)]
        tb = [float(x) for x in rng.integers(1, 9, size=K)]
        g = binding.GPipe(K, K, M, kind=0, d=64, heads=0, ffn=64, seq=1, vocab=0, n=M, dtype=0)
        mk, bub = g.schedule_model(tf, tb)
        sim = osch.simulate(K, M, [int(x) for x in tf], [int(x) for x in tb])
        assert mk == pytest.approx(float(sim["makespan"]), rel=1e-12)
        assert bub == pytest.approx(float(sim["bubble"]), abs=1e-12)


def _report(binding, w, K, M, no_remat=False, pipelined=True, inflight=1):
    g = binding.GPipe.from_workload(w, K=K, M=M)
    g.set_option(binding.OPT_INFLIGHT, inflight)
    if no_remat:
        g.set_option(binding.OPT_NO_REMAT, 1)
    if not pipelined:
        g.set_option(binding.OPT_PIPELINE, 0)
    peak, bound = g.memory_report()
    P, ws = g.sizes()
    return peak, bound, ws


def _model_from_shapes(w, K, M, schedule, remat):
    """The review's bound O(N + (L/K)(N/M)) in bytes, evaluated here from the
    shapes as gpipe.h documents it (boundary, one cell, head, one layer's
    backward working set, per-token losses, region alignment; the residual
    stream and its gradient in fp32, a bf16 copy of each gradient a GEMM
    reads)."""
    lm = w.kind == 1
    e = 4 if w.dtype == "f32" else 2
    r, c = 4, (0 if w.dtype == "f32" else 2)
    T = w.tokens
    Tmb = T // M
    d, f, H, V = w.d, w.ffn, (w.heads if lm else 0), (w.vocab if lm else 0)
    D = min(M, K + 1) if schedule == 1 else M
    Lc = -(-w.L // K)
    act, gcp = Tmb * d * r, Tmb * d * (r + c)
    boundary = K * D * act + D * gcp + (M * act if lm else 0) + 2 * act + 2 * K * gcp
    a = e * (6 * d + 2 * f) + 2 * d * r + 16 + 4 * H if lm else e * (d + 2 * f) + d * r + 8
    cell = Lc * Tmb * a if remat else w.L * M * Tmb * a
    lnp = 2 * (-(-Tmb // 8)) * 2 * d * 4
    head = Tmb * (4 * V + 2 * d * e + 8) + lnp if lm else 0
    grads = 2 * gcp + (act if lm else 0) + Tmb * d * e + 2 * Tmb * (f + (4 * d if lm else 0)) * e + \
        Tmb * max(H, 1) * 4 + lnp
    align = 256 * (13 * (Lc if remat else w.L * M) + 56)
    return boundary + cell + head + grads + 4 * T + align


@pytest.mark.parametrize("schedule", [0, 1])
@pytest.mark.parametrize("remat", [True, False])
def test_single_lane_layout_within_the_review_bound(binding, schedule, remat):
    """The review's "Preliminaries 5": with re-materialisation only the
    boundary activations of every micro-batch and one cell's internals are
    kept.  The bound, written out from the shapes alone (not from the layout),
    is what gpipe_memory_report returns; the single-lane executor's arena fits
    in it for every workload, in both issue orders, with and without
    re-materialisation (then every layer's internals: the O(N L) it started
    from).  The concurrent-lane executor holds one cell workspace per lane on
    top: at least (lanes - 1) x one cell of internals more than the bound."""
    for name, w in WORKLOADS.items():
        g = binding.GPipe.from_workload(w)
        g.set_option(binding.OPT_SCHEDULE, schedule)
        g.set_option(binding.OPT_NO_REMAT, 0 if remat else 1)
        g.set_option(binding.OPT_PIPELINE, 0)
        peak, bound = g.memory_report()
        _, ws = g.sizes()
        mm = g.memory_model()
        assert bound == mm["total"] == _model_from_shapes(w, w.K, w.M, schedule, remat), name
        assert sum(mm[k] for k in ("boundary", "cell", "head", "grads", "rows", "align")) == bound
        assert peak == mm["layout"] and peak <= bound and ws >= peak, (name, peak, bound)
        if w.kind == 1:  # and nothing much of the bound goes unused (tiny_ffn is mostly alignment)
            assert peak >= 0.97 * bound, (name, peak / bound)
        if remat:
            g.set_option(binding.OPT_PIPELINE, 1)
            lanes_peak, lanes_bound = g.memory_report()
            assert lanes_bound == bound
            lanes = w.K * (2 if w.tokens_per_micro_batch * w.d * w.ffn <= 2 ** 30 else 1)
            assert lanes_peak - bound >= (lanes - 1) * mm["cell"], name


def test_two_in_flight_cost_one_more_cell_workspace_per_cell(binding):
    """Two micro-batches in flight per cell double the per-lane term of the
    activation memory (one more cell workspace per cell), nothing else."""
    w = WORKLOADS["lm_wide"]
    one, _, _ = _report(binding, w, w.K, w.M)
    two, _, _ = _report(binding, w, w.K, w.M, inflight=2)
    serial, _, _ = _report(binding, w, w.K, w.M, pipelined=False)
    # with lanes there are K lanes, a second head lane (one more head buffer
    # set) and one more slot in the head's input ring (three instead of two)
    Tmb = w.tokens // w.M
    head_set = Tmb * (2 * w.d * 2 + 8 + w.vocab * 4) + 2 * (-(-Tmb // 8)) * 2 * w.d * 4
    lane = (one - serial - head_set - Tmb * w.d * 4) / (w.K - 1)  # one lane's workspace
    assert lane > 0
    assert two - one == pytest.approx(w.K * lane, rel=1e-4)
    with pytest.raises(binding.GpipeError):
        binding.GPipe.from_workload(w).set_option(binding.OPT_INFLIGHT, 5)
    # by size (the default): two in flight for the small LM, one for the wide one
    small = WORKLOADS["lm_small"]
    auto_small, _, _ = _report(binding, small, small.K, small.M, inflight=0)
    two_small, _, _ = _report(binding, small, small.K, small.M, inflight=2)
    auto_wide, _, _ = _report(binding, w, w.K, w.M, inflight=0)
    assert auto_small == two_small and auto_wide == one
    # S in flight: S-1 more lane workspaces per cell, and the gradient ring S deep
    four, _, _ = _report(binding, w, w.K, w.M, inflight=4)
    ring_slot = w.tokens // w.M * w.d * 6  # fp32 gradient and its bf16 copy
    assert four - one == pytest.approx(3 * w.K * lane + 2 * w.K * ring_slot, rel=1e-4)


@pytest.mark.parametrize("pipelined", [False, True])
def test_memory_scales_as_review_bound_over_sweep_grid(binding, pipelined):
    """Peak activation bytes over the micro-batch sweep grid follow the
    review's O(N + (L/K)(N/M)) per accelerator: boundary tensors a (K+2) N,
    plus per lane (L/K)(N/M) kept internals and (N/M) gradient buffers.  One
    lane (cells in turn): a (K+2)N + b (L/K)(N/M) + c (N/M); K concurrent
    lanes: a (K+2)N + b L (N/M) + c K (N/M) + e H (N/M), with H head lanes
    (two when there are two micro-batches to alternate, each holding one
    micro-batch's logits)."""
    w = WORKLOADS["lm_sweep"]
    rows, ys = [], []
    for K, M in SWEEP_GRID:
        peak, bound, _ = _report(binding, w, K, M, pipelined=pipelined)
        assert peak <= bound or pipelined
        T = w.tokens
        lanes = K if pipelined else 1
        # the gradient ring between cells holds 2 K micro-batches: a K (N/M)
        # term (within O(N)), a lane's buffers with the lanes
        row = [(K + 2) * T, lanes * (w.L / K) * T / M, K * T / M]
        if not pipelined:
            row.append(T / M)
        if pipelined:
            row.append((2 if M > 1 else 1) * T / M)
        rows.append(row)
        ys.append(peak)
    A, y = np.array(rows, dtype=float), np.array(ys, dtype=float)
    coef, *_ = np.linalg.lstsq(A, y, rcond=None)
    resid = np.abs(A @ coef - y) / y
    assert resid.max() <= 0.10, resid
    assert np.all(coef > 0)


def test_pipelined_lanes_cost_memory_only_per_cell(binding):
    """K lanes hold K cells' internals at once (one per lane), so the extra
    memory over the one-lane schedule is (K-1) lanes' worth, not L layers x M."""
    w = WORKLOADS["lm_wide"]
    serial, _, _ = _report(binding, w, w.K, w.M, pipelined=False)
    piped, _, _ = _report(binding, w, w.K, w.M, pipelined=True)
    noremat, _, _ = _report(binding, w, w.K, w.M, no_remat=True, pipelined=False)
    assert serial < piped < noremat / 4


@pytest.mark.parametrize("name", ["lm_wide", "lm_deep"])
def test_rematerialisation_saves_memory(binding, name):
    """The memory-scaling comparison: peak activation bytes with and without
    re-materialisation, each within its bound; without it every layer keeps its
    internals for every micro-batch."""
    w = WORKLOADS[name]
    peak, bound, _ = _report(binding, w, w.K, w.M, pipelined=False)
    peak_nr, bound_nr, _ = _report(binding, w, w.K, w.M, no_remat=True, pipelined=False)
    assert peak <= bound and peak_nr <= bound_nr
    assert peak_nr > 10 * peak
    # the concurrent lanes cost cell workspaces, but far less than keeping everything
    lanes, _, _ = _report(binding, w, w.K, w.M)
    assert peak < lanes < peak_nr / 10


def test_last_error_without_context_reports_any_failed_call(binding):
    lib = binding.lib()
    rc = lib.gpipe_op_layernorm_fwd(1, 4, 12, None, None, None, None, None, None, None)   # d % 8 != 0
    assert rc == -1
    assert b"layernorm" in lib.gpipe_last_error(None)
    with pytest.raises(binding.GpipeError):
        binding.GPipe(4, 5, 1, kind=0, d=64, heads=0, ffn=64, seq=1, vocab=0, n=4, dtype=0)
    assert b"K <= L" in lib.gpipe_last_error(None)


def test_options_are_validated_and_kernel_times_start_empty(binding):
    from synth import WORKLOADS
    g = binding.GPipe.from_workload(WORKLOADS["lm_small"])
    with pytest.raises(binding.GpipeError) as e:
        g.set_option(999, 1)
    assert e.value.code == -1   # GPIPE_ERR_INVALID_ARG
    for bad in (-1, binding.EPI_RESID_F32 + 2):
        with pytest.raises(binding.GpipeError):
            g.set_option(binding.OPT_KERNEL_TIMES, bad)
    for bad in (24, 801):
        with pytest.raises(binding.GpipeError):
            g.set_option(binding.OPT_SM_SHARE, bad)
    g.set_option(binding.OPT_SM_SHARE, 200)
    for opt, bad in ((binding.OPT_SIDE_STREAMS, 0), (binding.OPT_SIDE_STREAMS, 5), (binding.OPT_SIDE_SHARE, 4)):
        with pytest.raises(binding.GpipeError):
            g.set_option(opt, bad)
    for opt, bad in ((binding.OPT_LOGIT_CLIP, -1), (binding.OPT_LOGIT_CLIP, 10**9 + 1), (binding.OPT_SCHEDULE, -1)):
        with pytest.raises(binding.GpipeError):
            g.set_option(opt, bad)
    g.set_option(binding.OPT_LOGIT_CLIP, 2500)
    g.set_option(binding.OPT_LOGIT_CLIP, 0)
    g.set_option(binding.OPT_KERNEL_TIMES, binding.EPI_BIAS_GELU + 1)
    ms, fl = g.kernel_times()   # no step taken yet: nothing timed, no CUDA call made
    assert ms.size == 0 and fl.size == 0
    g.set_option(binding.OPT_LAYER_TIMES, 1)
    fw, bw = g.layer_times()
    assert fw.size == 0 and bw.size == 0
    g.close()
    # the op API's SM share for gpipe_op_gemm: >= 0 (0 = the whole GPU)
    assert binding.lib().gpipe_op_gemm_set_sm_share(-1) == -1
    assert binding.lib().gpipe_op_gemm_set_sm_share(0) == 0


def _check_issue_order(ops, K, M, schedule, ring, lm=True):
    """Checks an issue order against the pipeline's dependencies (written out
    here from the review's "Pipeline flow": cell k forwards m after cell k-1,
    the head after the last cell, cell k differentiates m after cell k+1 (the
    last cell after the head)), the micro-batch order of each cell's
    backwards (the gradient accumulation order), and buffer reuse: a stash
    slot (depth D) or an input-gradient ring slot (depth R) is rewritten only
    after its previous reader was issued."""
    pos = {}
    for i, (kind, k, m, tick) in enumerate(ops):
        key = (kind, k, m)
        assert key not in pos, key
        pos[key] = i
    F = lambda k, m: pos[(0, k, m)]
    H = lambda m: pos[(1, 0, m)]
    B = lambda k, m: pos[(2, k, m)]
    assert len(pos) == (2 * K + 1) * M
    D = min(M, K + 1) if schedule == 1 else M
    for m in range(M):
        assert H(m) > F(K - 1, m) and B(K - 1, m) > H(m)
        if m:
            assert H(m) > H(m - 1)
        for k in range(K):
            assert B(k, m) > F(k, m)
            if k:
                assert F(k, m) > F(k - 1, m)
            if k < K - 1:
                assert B(k, m) > B(k + 1, m)
            if m:
                assert F(k, m) > F(k, m - 1) and B(k, m) > B(k, m - 1)
            if k and m >= ring:
                assert B(k, m) > B(k - 1, m - ring)
        if m >= D:
            # level 0 (embedding output) and level k+1 (cell k's output)
            if lm:
                assert F(0, m) > B(0, m - D)
            for k in range(K):
                reader = H(m - D) if k == K - 1 else B(k + 1, m - D)
                assert F(k, m) > reader
            assert H(m) > B(K - 1, m - D)
    # ticks: a producer is issued in an earlier tick than its consumer
    tick = {(kind, k, m): t for kind, k, m, t in ops}
    for m in range(M):
        for k in range(1, K):
            assert tick[(0, k, m)] > tick[(0, k - 1, m)]
            assert tick[(2, k - 1, m)] > tick[(2, k, m)]
    return D


@pytest.mark.parametrize("schedule", [0, 1])
@pytest.mark.parametrize("K,M,inflight", [(1, 1, 1), (1, 5, 2), (2, 1, 1), (3, 7, 1), (4, 16, 2), (4, 4, 1),
                                          (8, 32, 1), (8, 4, 4), (16, 64, 1), (5, 3, 3)])
def test_issue_order_respects_dependencies_and_buffer_reuse(binding, schedule, K, M, inflight):
    g = binding.GPipe(2 * K, K, M, kind=1, d=64, heads=1, ffn=64, seq=64, vocab=64, n=M, dtype=1)
    g.set_option(binding.OPT_INFLIGHT, inflight)
    g.set_option(binding.OPT_SCHEDULE, schedule)
    ops = g.issue_order()
    ring = max(2, inflight)
    _check_issue_order(ops, K, M, schedule, ring)
    if schedule == 0:
        # the review's figure: every forward (and head) before the first backward
        first_b = min(i for i, o in enumerate(ops) if o[0] == binding.OP_BWD)
        assert all(o[0] != binding.OP_BWD for o in ops[:first_b]) and first_b == (K + 1) * M
    else:
        # one-forward-one-backward: cell k runs min(M, K+1-k) forwards before its
        # first backward, then never more than that many ahead of its backwards
        for k in range(K):
            seq = [o[0] for o in ops if o[1] == k and o[0] != binding.OP_HEAD]
            assert seq.index(binding.OP_BWD) == min(M, K + 1 - k)
            ahead = 0
            for kind in seq:
                ahead += 1 if kind == binding.OP_FWD else -1
                assert 0 <= ahead <= min(M, K + 1 - k)


@pytest.mark.parametrize("K,M", [(1, 1), (2, 1), (4, 32), (8, 32), (4, 4), (3, 7), (16, 64)])
def test_one_f_one_b_clock_equals_gpipe_for_equal_cells(binding, K, M):
    """With equal cells the interleaved order finishes when the GPipe order
    does: the same bubble (K-1)/(M+K-1) (backward twice the forward here)."""
    g = binding.GPipe(K, K, M, kind=0, d=64, heads=0, ffn=64, seq=1, vocab=0, n=M, dtype=0)
    g.set_option(binding.OPT_SCHEDULE, 1)
    mk, bub = g.schedule_model([1.0] * K, [2.0] * K)
    sim = osch.simulate(K, M, 1, 2)
    assert mk == pytest.approx(float(sim["makespan"]), rel=1e-12)
    assert bub == pytest.approx(float(Fraction(K - 1, M + K - 1)), abs=1e-12)


def test_one_f_one_b_clock_model_unequal_cells(binding):
    """The library's clock of its one-forward-one-backward issue order against
    the oracle's independent simulation, on random unequal cells."""
    rng = np.random.default_rng(7)
    for _ in range(25):
        K, M = int(rng.integers(1, 7)), int(rng.integers(1, 12))
        tf = [float(x) for x in rng.integers(1, 9, size=K)]
        tb = [float(x) for x in rng.integers(1, 9, size=K)]
        g = binding.GPipe(K, K, M, kind=0, d=64, heads=0, ffn=64, seq=1, vocab=0, n=M, dtype=0)
        g.set_option(binding.OPT_SCHEDULE, 1)
        mk, bub = g.schedule_model(tf, tb)
        sim = osch.simulate_1f1b(K, M, [int(x) for x in tf], [int(x) for x in tb])
        assert mk == pytest.approx(float(sim["makespan"]), rel=1e-12), (K, M, tf, tb)
        assert bub == pytest.approx(float(sim["bubble"]), abs=1e-12)


@pytest.mark.parametrize("name", ["lm_small", "lm_wide", "lm_deep"])
def test_one_f_one_b_keeps_a_shorter_stash(binding, name):
    """The interleaved order holds min(M, K+1) micro-batches per cell boundary
    (and of the head's output gradient) instead of M: the workspace shrinks by
    exactly (K+2)(M - D) boundary tensors, and stays within its bound."""
    w = WORKLOADS[name]
    g = binding.GPipe.from_workload(w)
    peak0, bound0 = g.memory_report()
    ws0 = g.sizes()[1]
    g.set_option(binding.OPT_SCHEDULE, 1)
    peak1, bound1 = g.memory_report()
    ws1 = g.sizes()[1]
    D = min(w.M, w.K + 1)
    Tmb_d = w.tokens // w.M * w.d
    # K cell inputs (fp32) and the head's output gradient (fp32 and its bf16
    # copy) each hold D micro-batches instead of M
    assert peak0 - peak1 == (w.M - D) * Tmb_d * (4 * w.K + 6)
    assert ws0 - ws1 == peak0 - peak1
    assert bound0 - bound1 == peak0 - peak1
    g.set_option(binding.OPT_PIPELINE, 0)
    peak2, bound2 = g.memory_report()
    assert bound2 == bound1 and peak2 <= bound2
    with pytest.raises(binding.GpipeError):
        g.set_option(binding.OPT_SCHEDULE, 2)


def test_heterogeneous_ffn_widths_partition_and_packing(binding):
    """Layers of unequal FFN width (the review's "Limitations 3: load
    imbalance"): the default costs are each layer's forward FLOPs per token
    (the documented formula, evaluated here), the partition is the exact
    variance-minimising one for those costs, and the packing holds each layer's
    own W1/b1/W2."""
    from synth import KIND_LM, Workload, param_count
    widths = (256, 2048, 512, 1024, 64, 1536, 768, 128)
    w = Workload("hetero", KIND_LM, L=8, K=3, M=2, d=128, heads=2, ffn=64, seq=64, vocab=256, n=4, dtype="bf16",
                 ffn_layers=widths)
    g = binding.GPipe.from_workload(w)
    d, s = w.d, w.seq
    costs = [2 * (4 * d * d + 2 * d * f) + 2 * d * (s + 1) for f in widths]
    assert g.partition() == op.partition(costs, w.K)[0]
    assert g.sizes()[0] == param_count(w)
    g.set_option(binding.OPT_PIPELINE, 0)
    peak, bound = g.memory_report()
    assert peak <= bound
    g.set_option(binding.OPT_PIPELINE, 1)
    # the widest layer sizes the workspace: the same as all layers at 2048
    g_wide = binding.GPipe.from_workload(w.replace(ffn=2048, ffn_layers=()))
    assert g.sizes()[1] == g_wide.sizes()[1]
    # FFN model too, with explicit costs overriding the default
    wf = Workload("hetero_ffn", 0, L=4, K=2, M=2, d=64, heads=0, ffn=8, seq=1, vocab=0, n=4, dtype="f32",
                  ffn_layers=(64, 256, 8, 128))
    gf = binding.GPipe.from_workload(wf)
    assert gf.partition() == op.partition([4 * 64 * f for f in wf.ffn_layers], 2)[0]
    assert gf.sizes()[0] == param_count(wf)
    assert binding.GPipe.from_workload(wf, cost=[1, 1, 1, 1]).partition() == [0, 2, 4]
    for bad in ((256, 100, 512, 64, 64, 64, 64, 64), (256, 0, 512, 64, 64, 64, 64, 64)):
        with pytest.raises(binding.GpipeError):
            binding.GPipe.from_workload(w.replace(ffn_layers=bad))
    with pytest.raises(ValueError):
        param_count(w.replace(ffn_layers=(64, 64)))


def test_repartition_on_new_costs(binding):
    """Re-partitioning a context on measured (here: given) costs gives the same
    exact cut as creating it with them; the clock model follows the new cells;
    the packing stays, the workspace follows the largest cell."""
    rng = np.random.default_rng(13)
    w = WORKLOADS["lm_small"]
    g = binding.GPipe.from_workload(w)
    P0, ws0 = g.sizes()
    for _ in range(10):
        cost = [int(c) for c in rng.integers(1, 10**6, size=w.L)]
        g.repartition(cost)
        assert g.partition() == op.partition(cost, w.K)[0]
        fresh = binding.GPipe.from_workload(w, cost=cost)
        assert g.sizes() == fresh.sizes() and g.sizes()[0] == P0
        assert g.schedule_model() == fresh.schedule_model()
    g.repartition([1] * w.L)
    assert g.sizes() == (P0, ws0)
    with pytest.raises(binding.GpipeError):
        g.repartition([1] * (w.L - 1) + [0])
    assert g.partition() == [0, 2, 4, 6, 8]


def test_ops_reject_invalid_arguments_before_any_launch(binding):
    """Every per-kernel entry point checks its shapes and alignment on the host
    and returns GPIPE_ERR_INVALID_ARG with a message naming the operation,
    before any CUDA call (these run without a GPU).  16 stands for an aligned
    address and is never dereferenced; 8 for a misaligned one."""
    lib = binding.lib()
    A, U = 16, 8
    cases = [
        ("layernorm", lambda: lib.gpipe_op_layernorm_fwd(1, 4, 12, A, A, A, A, A, A, None)),
        ("layernorm_bwd", lambda: lib.gpipe_op_layernorm_bwd(1, 0, 64, A, A, A, A, A, None, A, A, A, A, None)),
        ("attention", lambda: lib.gpipe_op_attention_fwd(1, 100, 1, A, A, A, None)),
        ("attention", lambda: lib.gpipe_op_attention_bwd(1, 64, 0, A, A, A, A, A, A, None)),
        ("cross_entropy", lambda: lib.gpipe_op_cross_entropy(4, 10, 64, A, 0, 1.0, A, A, 1, None)),
        ("cross_entropy", lambda: lib.gpipe_op_cross_entropy(4, 16, 64, A, 0, 1.0, U, A, 1, None)),
        ("cross_entropy", lambda: lib.gpipe_op_cross_entropy_clip(4, 16, 64, A, 0, 1.0, -1.0, A, A, 1, None)),
        ("cross_entropy", lambda: lib.gpipe_op_cross_entropy_clip(4, 16, 64, A, 0, 1.0, float("nan"), A, A, 1,
                                                                  None)),
        ("mse", lambda: lib.gpipe_op_mse(0, 8, A, A, 1.0, A, A, None)),
        ("embedding_fwd", lambda: lib.gpipe_op_embedding_fwd(4, 16, 0, A, A, A, None)),
        ("embedding_fwd", lambda: lib.gpipe_op_embedding_fwd(4, 12, 10, A, A, A, None)),
        ("embedding_bwd", lambda: lib.gpipe_op_embedding_bwd(4, 16, 10, A, U, A, None)),
    ]
    for what, call in cases:
        assert call() == -1, what
        assert what.encode() in lib.gpipe_last_error(None), (what, lib.gpipe_last_error(None))
