"""Full synchronous GPipe step on the GPU (through gpipe_step) against the
CPU fp64 oracle's full-batch step, plus the properties the review states:
re-materialised activations equal the first forward, micro-batching does not
change the result, and steps are reproducible.

Tolerances: fp32 workload rel-L2 <= 1e-5 on loss, gradients and updated
weights; bf16 workloads rel-L2 <= 1e-3 on the loss and <= 2e-2 on gradients.
RMSProp's first step moves each weight by about lr/sqrt(1-decay) in the
direction of -sign(g), so where |g| is below the gradient's own error the
sign (and the step) is not determined by the oracle: updated weights are
compared where |g_oracle| exceeds a threshold, and elsewhere checked to be a
valid RMSProp step (|dw| <= lr/sqrt(1-decay)).
"""
import math

import numpy as np
import pytest

from oracle import model as om
from synth import KIND_LM, WORKLOADS, Workload, make_inputs
from tests.gpu_util import rel

pytestmark = pytest.mark.gpu

SMALL_LM = Workload("small_lm", KIND_LM, L=4, K=2, M=2, d=128, heads=2, ffn=256, seq=128, vocab=1000, n=4,
                    dtype="bf16")


@pytest.fixture(scope="module")
def b():
    import __graft_entry__ as ge
    ge.build()
    from micro_pipeline_re_gb300 import binding
    return binding


def _run(b, w, inp, steps=1, keep_grads=True, options=(), K=None, M=None, cost=None):
    import torch
    gp = b.GPipe.from_workload(w, K=K, M=M, cost=cost)
    if keep_grads:
        gp.set_option(b.OPT_KEEP_GRADS, 1)
    for o, v in options:
        gp.set_option(o, v)
    st = b.DeviceState(gp, w, inp)
    p0 = st.host(st.p32).copy()
    losses = []
    for _ in range(steps):
        if keep_grads and steps > 1:
            st.g32.zero_()
        losses.append(st.step())
    torch.cuda.synchronize()
    return gp, st, p0, losses


def _flat(w, d):
    from synth import param_specs
    return np.concatenate([np.asarray(d[n], dtype=np.float64).ravel() for n, _, _ in param_specs(w)])


def _check_update(w, p0, g_ref, p_ref, p_gpu, v_ref, v_gpu, tol_w, tol_v, thresh):
    dw_gpu = p_gpu - p0
    dw_ref = p_ref - p0
    mask = np.abs(g_ref) > thresh * np.sqrt(np.mean(g_ref ** 2))
    assert mask.mean() > 0.5
    assert rel(dw_gpu[mask], dw_ref[mask]) <= tol_w
    step_max = w.lr / math.sqrt(1 - w.decay)
    assert np.all(np.abs(dw_gpu) <= step_max * (1 + 1e-3))
    assert rel(p_gpu, p_ref) <= tol_w
    assert rel(v_gpu[mask], v_ref[mask]) <= tol_v


def test_tiny_ffn_fp32_step_matches_oracle(b):
    w = WORKLOADS["tiny_ffn"]
    inp = make_inputs(w)
    gp, st, p0, (loss,) = _run(b, w, inp)
    ref = om.step(w, inp["params"], inp)
    assert abs(loss - ref["loss"]) <= 1e-5 * abs(ref["loss"])
    g = st.host(st.g32)
    gref = _flat(w, ref["grads"])
    assert rel(g, gref) <= 1e-5
    for name, got in b.unpack(w, g).items():
        assert rel(got, ref["grads"][name]) <= 1e-5, name
    _check_update(w, p0, gref, _flat(w, ref["params"]), st.host(st.p32), _flat(w, ref["v"]), st.host(st.v32),
                  1e-5, 1e-5, 1e-3)


def test_tiny_ffn_two_steps(b):
    w = WORKLOADS["tiny_ffn"]
    inp = make_inputs(w)
    gp, st, p0, losses = _run(b, w, inp, steps=2, keep_grads=False)
    ref1 = om.step(w, inp["params"], inp)
    ref2 = om.step(w, ref1["params"], inp, v=ref1["v"])
    assert abs(losses[0] - ref1["loss"]) <= 1e-5 * abs(ref1["loss"])
    assert abs(losses[1] - ref2["loss"]) <= 1e-5 * abs(ref2["loss"])
    assert not np.any(st.host(st.g32))   # the update leaves the accumulator zeroed


def _lm_parity(b, w, inp, loss_tol=1e-3, grad_tol=2e-2, group_tol=5e-2, **kw):
    gp, st, p0, (loss,) = _run(b, w, inp, **kw)
    ref = om.step(w, inp["params"], inp)
    assert abs(loss - ref["loss"]) <= loss_tol * abs(ref["loss"]), (loss, ref["loss"])
    g = st.host(st.g32)
    gref = _flat(w, ref["grads"])
    assert rel(g, gref) <= grad_tol
    worst = max((rel(got, ref["grads"][name]), name) for name, got in b.unpack(w, g).items())
    assert worst[0] <= group_tol, worst
    _check_update(w, p0, gref, _flat(w, ref["params"]), st.host(st.p32), _flat(w, ref["v"]), st.host(st.v32),
                  2e-2, 5e-2, 0.1)
    return gp, st, ref


def test_small_lm_bf16_step_matches_oracle(b):
    w = SMALL_LM
    _lm_parity(b, w, make_inputs(w))


def test_small_lm_trainability_options_match_oracle(b):
    """The review's "Training stability" measures: FFN matrices initialised with
    variance 1/(d L) and logits clipped to [-1.5, 1.5] in the cross-entropy
    (about one logit in eight at this initialisation), in the one-forward-
    one-backward order; the oracle applies the same clip."""
    w = SMALL_LM.replace(ffn_init_depth_scaled=True, logit_clip_milli=1500)
    inp = make_inputs(w)
    ref_plain = om.forward_loss(w.replace(logit_clip_milli=0), inp["params"], inp)[0]
    _, _, ref = _lm_parity(b, w, inp, options=[(b.OPT_SCHEDULE, 1)])
    assert abs(ref["loss"] - ref_plain) > 1e-2 * abs(ref_plain)   # the clip is active


def test_heterogeneous_ffn_widths_match_oracle(b):
    """Layers of unequal FFN width (heterogeneous cells): LM in bf16 and the FFN
    model in fp32 against the oracle."""
    w = SMALL_LM.replace(ffn_layers=(256, 512, 128, 384), M=4, n=8)
    gp, _, _ = _lm_parity(b, w, make_inputs(w))
    assert gp.partition() == [0, 2, 4]
    wf = WORKLOADS["tiny_ffn"].replace(ffn_layers=(64, 256, 128, 192))
    inp = make_inputs(wf)
    _, st, p0, (loss,) = _run(b, wf, inp)
    ref = om.step(wf, inp["params"], inp)
    assert abs(loss - ref["loss"]) <= 1e-5 * abs(ref["loss"])
    for name, got in b.unpack(wf, st.host(st.g32)).items():
        assert rel(got, ref["grads"][name]) <= 1e-5, name


def test_partition_does_not_change_the_result(b):
    """Where the layers are cut changes where they run, not what they compute:
    partitions of the same heterogeneous model into 2 cells two ways, into one
    cell and into one cell per layer give identical bits."""
    w = SMALL_LM.replace(ffn_layers=(256, 512, 128, 384), M=4, n=8)
    inp = make_inputs(w)
    outs = []
    for cost, K in (([1, 1, 1, 1], None), ([1, 1, 1, 5], None), (None, None), (None, 1), (None, 4)):
        gp, st, _, (loss,) = _run(b, w, inp, cost=cost, K=K)
        outs.append((gp.partition(), loss, st.host(st.g32).copy(), st.host(st.p32).copy()))
    assert outs[0][0] == [0, 2, 4] and outs[1][0] == [0, 3, 4]
    assert outs[3][0] == [0, 4] and outs[4][0] == [0, 1, 2, 3, 4]
    for o in outs[1:]:
        assert o[1] == outs[0][1] and np.array_equal(o[2], outs[0][2]) and np.array_equal(o[3], outs[0][3])


def test_partition_on_measured_layer_times(b):
    """Per-layer costs measured on the GPU (events around each layer's forward
    and backward, one stream) see the wide layers as the expensive ones; the
    partition on those costs runs, with the same result."""
    w = Workload("hetero_wide", KIND_LM, L=8, K=2, M=2, d=1024, heads=16, ffn=256, seq=128, vocab=1000, n=16,
                 dtype="bf16", ffn_layers=(8192, 256, 256, 256, 8192, 256, 8192, 256))
    inp = make_inputs(w)
    gp, st, _, (loss,) = _run(b, w, inp, options=[(b.OPT_PIPELINE, 0), (b.OPT_CONCURRENT, 0),
                                                  (b.OPT_LAYER_TIMES, 1)])
    fwd, bwd = gp.layer_times()
    assert fwd.size == w.L and np.all(fwd > 0) and np.all(bwd > 0)
    t = fwd + bwd
    wide = np.array(w.ffn_layers) == 8192
    assert t[wide].min() > t[~wide].max(), t
    cost = [int(x) for x in np.rint(t * 1e6)]
    gm, st2, _, (loss2,) = _run(b, w, inp, cost=cost)
    from oracle import partition as opart
    assert gm.partition() == opart.partition(cost, w.K)[0]
    assert loss2 == loss and np.array_equal(st2.host(st2.g32), st.host(st.g32))


def test_checkpoint_resume_is_bit_identical(b):
    """Two steps straight, or one step, a checkpoint, a fresh context (in the
    other issue order) with buffers restored from it, and the second step:
    identical losses, weights and RMSProp state."""
    import os
    import torch
    w = SMALL_LM
    inp = make_inputs(w)
    _, st, _, losses = _run(b, w, inp, steps=2, keep_grads=False)
    p_ref, v_ref = st.host(st.p32).copy(), st.host(st.v32).copy()
    _, st1, _, (l1,) = _run(b, w, inp, steps=1, keep_grads=False)
    tmp = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_tmp")
    os.makedirs(tmp, exist_ok=True)
    path = os.path.join(tmp, "resume.ck")
    st1.save(path, 1)
    gp2 = b.GPipe.from_workload(w)
    gp2.set_option(b.OPT_SCHEDULE, 1)
    st2 = b.DeviceState(gp2, w, inp)
    assert st2.load(path) == 1
    l2 = st2.step()
    torch.cuda.synchronize()
    assert l1 == losses[0] and l2 == losses[1]
    assert np.array_equal(st2.host(st2.p32), p_ref) and np.array_equal(st2.host(st2.v32), v_ref)


def test_small_lm_uneven_partition(b):
    """Costs that force unequal cells (3 + 1 layers)."""
    w = SMALL_LM
    _lm_parity(b, w, make_inputs(w), cost=[1, 1, 1, 5])


def test_lm_small_full_size_matches_oracle(b):
    """The throughput workload (L=8, d=512, N=64, seq=128, K=4, M=16) at full size."""
    w = WORKLOADS["lm_small"]
    _lm_parity(b, w, make_inputs(w))


def test_lm_wide_layers_sub_batch(b):
    """The wide workload's layers (L=24, d=1024, ffn=8192, seq=256, K=8) on a
    sub-batch of N=2 sequences, M=2, which the fp64 oracle finishes in seconds."""
    w = WORKLOADS["lm_wide"].replace(n=2, M=2)
    _lm_parity(b, w, make_inputs(w))


def test_sweep_layers_single_micro_batch(b):
    """The sweep workload's layer (d=1024, ffn=8192, seq=256) with K=8 cells and
    the degenerate M=1 (no micro-batching), 16 layers on one sequence (the fp64
    oracle's time grows with layers x tokens)."""
    w = WORKLOADS["lm_sweep"].replace(L=16, n=1, M=1, K=8)
    _lm_parity(b, w, make_inputs(w))


def test_memory_scaling_layers_sub_batch(b):
    """The memory-scaling workload's layer at seq 512 with K=16 cells (one layer
    each) on one sequence, M=1."""
    w = WORKLOADS["lm_deep"].replace(L=16, n=1, M=1)
    _lm_parity(b, w, make_inputs(w))


@pytest.mark.parametrize("m_check", [0, 1])
def test_rematerialised_internals_bit_identical(b, m_check):
    w = SMALL_LM
    gp, st, _, _ = _run(b, w, make_inputs(w), options=[(b.OPT_REMAT_CHECK, m_check)])
    mism, err = gp.debug_counters(st.ws, st.stream)
    assert err == 0
    assert mism == 0


def test_steps_are_bit_reproducible_and_graph_equals_direct(b):
    w = SMALL_LM
    inp = make_inputs(w)
    outs = []
    for graph in (1, 1, 0):
        gp, st, _, (loss,) = _run(b, w, inp, options=[(b.OPT_GRAPH, graph)])
        outs.append((loss, st.g32.cpu().numpy().copy(), st.p32.cpu().numpy().copy()))
    for i, o in enumerate(outs[1:], 1):
        assert o[0] == outs[0][0], i
        assert np.array_equal(o[1], outs[0][1]), i
        assert np.array_equal(o[2], outs[0][2]), i


@pytest.mark.parametrize("wname", ["small_lm", "tiny_ffn", "lm_small"])
def test_schedules_are_bit_identical(b, wname):
    """Cells as concurrent lanes (the review's pipeline on one GPU), weight
    gradients on side streams and the one-forward-one-backward issue order
    (with its shorter stash ring) give exactly the one-stream, cells-in-turn
    GPipe result, with and without the CUDA graph."""
    w = SMALL_LM if wname == "small_lm" else WORKLOADS[wname]
    inp = make_inputs(w)
    outs = []
    for pipe, conc, graph, pdl, inflight, nside, sched in (
            (0, 0, 1, 0, 1, 1, 0), (1, 1, 1, 1, 1, 1, 0), (1, 0, 1, 1, 1, 1, 0), (0, 1, 1, 1, 1, 1, 0),
            (1, 1, 0, 1, 1, 1, 0), (1, 1, 1, 0, 1, 1, 0), (1, 1, 1, 0, 2, 1, 0), (1, 0, 0, 0, 2, 1, 0),
            (1, 1, 1, 0, 3, 1, 0), (1, 1, 1, 0, 4, 1, 0), (1, 1, 1, 0, 2, 4, 0), (1, 1, 1, 0, 1, 3, 0),
            (0, 1, 0, 0, 1, 2, 0), (1, 1, 1, 0, 1, 2, 1), (1, 1, 1, 0, 2, 2, 1), (1, 1, 0, 0, 2, 2, 1),
            (0, 1, 1, 0, 1, 2, 1), (1, 1, 1, 0, 4, 2, 1)):
        _, st, _, (loss,) = _run(b, w, inp, options=[(b.OPT_INFLIGHT, inflight), (b.OPT_PIPELINE, pipe),
                                                     (b.OPT_CONCURRENT, conc), (b.OPT_GRAPH, graph),
                                                     (b.OPT_PDL, pdl), (b.OPT_SIDE_STREAMS, nside),
                                                     (b.OPT_SCHEDULE, sched)])
        outs.append((loss, st.g32.cpu().numpy().copy(), st.p32.cpu().numpy().copy()))
    for i, o in enumerate(outs[1:], 1):
        assert o[0] == outs[0][0], i
        assert np.array_equal(o[1], outs[0][1]), i
        assert np.array_equal(o[2], outs[0][2]), i


def test_no_rematerialisation_mode_is_identical(b):
    w = SMALL_LM
    inp = make_inputs(w)
    _, st1, _, (l1,) = _run(b, w, inp)
    _, st2, _, (l2,) = _run(b, w, inp, options=[(b.OPT_NO_REMAT, 1)])
    assert l1 == l2
    assert np.array_equal(st1.g32.cpu().numpy(), st2.g32.cpu().numpy())


def test_micro_batch_count_does_not_change_result(b):
    """Synchronous accumulation equals the full-batch step for any M."""
    w = SMALL_LM
    inp = make_inputs(w)
    res = {}
    for M in (1, 2, 4):
        _, st, _, (loss,) = _run(b, w, inp, M=M)
        res[M] = (loss, st.host(st.g32))
    for M in (2, 4):
        assert abs(res[M][0] - res[1][0]) <= 1e-4 * abs(res[1][0])
        assert rel(res[M][1], res[1][1]) <= 1e-2


def test_per_sequence_losses_sampled(b):
    """Sampled per-sequence losses of a full-size step equal the oracle's
    forward on those sequences alone (sequences are independent)."""
    w = WORKLOADS["lm_small"]
    inp = make_inputs(w)
    gp, st, _, _ = _run(b, w, inp, options=[(b.OPT_SKIP_UPDATE, 1)])
    rows = gp.loss_rows(st.ws, w.n * w.seq, st.stream).reshape(w.n, w.seq)
    per_seq = rows.sum(axis=1) * w.n   # rows are divided by N (seq-1); per-sequence mean = sum * N
    for i in (0, 17, 63):
        sub = {"tokens": inp["tokens"][i:i + 1]}
        _, ex = om.forward_loss(w.replace(n=1), inp["params"], sub)
        assert abs(per_seq[i] - ex["per_seq_loss"][0]) <= 2e-3 * ex["per_seq_loss"][0]


def test_loss_near_log_vocab_and_update_from_zero_state(b):
    """Any size: at the init the loss is near ln V, and the first RMSProp step
    moves every weight with |g| >> eps by lr/sqrt(1-decay)."""
    w = WORKLOADS["lm_small"]
    gp, st, p0, (loss,) = _run(b, w, make_inputs(w))
    assert abs(loss - math.log(w.vocab)) < 1.5
    g = st.host(st.g32)
    dw = st.host(st.p32) - p0
    big = np.abs(g) > 1e-4
    expect = w.lr / math.sqrt(1 - w.decay)
    assert np.allclose(np.abs(dw[big]), expect, rtol=2e-3)
    assert np.all(np.sign(dw[big]) == -np.sign(g[big]))


@pytest.mark.parametrize("inflight,sched", [(1, 0), (2, 0), (4, 0), (1, 1), (2, 1)])
def test_trace_follows_the_pipeline_dependencies(b, inflight, sched):
    """With cells as concurrent lanes, GPU timestamps obey the review's pipeline:
    cell k finishes forwarding micro-batch m after cell k-1, the head after the
    last cell, the last cell's backward after the head, cell k-1's backward
    after cell k's, and every lane takes its micro-batches in order (with two
    in flight per cell, a cell's lanes take alternate micro-batches; so do the
    two head lanes).  In the one-forward-one-backward order a stash slot is
    rewritten only after its previous micro-batch's reader finished, and cell
    0 differentiates micro-batch 0 before it forwards the last one."""
    w = WORKLOADS["lm_small"]
    gp, st, _, _ = _run(b, w, make_inputs(w), options=[(b.OPT_INFLIGHT, inflight), (b.OPT_TRACE, 1),
                                                       (b.OPT_SCHEDULE, sched)])
    t0, t1, fwd, bwd = gp.trace(st.ws, st.stream)
    K, M = w.K, w.M
    assert t0 <= fwd.min() and max(fwd.max(), bwd[:K].max()) <= t1
    for m in range(M):
        for k in range(1, K + 1):
            assert fwd[k, m] >= fwd[k - 1, m]
        assert bwd[K - 1, m] >= fwd[K, m]
        for k in range(K - 1, 0, -1):
            assert bwd[k - 1, m] >= bwd[k, m]
    for r in range(inflight):
        assert np.all(np.diff(fwd[:K, r::inflight], axis=1) >= 0)
        assert np.all(np.diff(bwd[:K, r::inflight], axis=1) >= 0)
    for r in range(2):  # two head lanes take alternate micro-batches, each in order
        assert np.all(np.diff(fwd[K, r::2]) >= 0)
    if sched == 1:
        D = min(M, K + 1)
        assert D < M
        for m in range(D, M):
            assert fwd[0, m] >= bwd[0, m - D]          # the embedding's output slot
            for k in range(K - 1):
                assert fwd[k, m] >= bwd[k + 1, m - D]  # cell k's output slot
            assert fwd[K - 1, m] >= fwd[K, m - D]      # the head's input slot
            assert fwd[K, m] >= bwd[K - 1, m - D]      # the head's output-gradient slot
        assert bwd[0, 0] <= fwd[0, M - 1]


@pytest.mark.parametrize("graph", [1, 0])
def test_kernel_times_bracket_the_selected_gemms(b, graph):
    """GPIPE_OPT_KERNEL_TIMES times every FFN first-projection launch (forward
    and re-computation: 2 L M per step) on its own stream, inside the step's
    graph too, and changes no result."""
    w = SMALL_LM
    inp = make_inputs(w)
    opts = [(b.OPT_GRAPH, graph)]
    gp0, st0, _, _ = _run(b, w, inp, steps=2, options=opts)
    gp1, st1, _, _ = _run(b, w, inp, steps=2, options=opts + [(b.OPT_KERNEL_TIMES, b.EPI_BIAS_GELU + 1)])
    ms, fl, mnk = gp1.kernel_times(with_shapes=True)
    T = w.n * w.seq // w.M
    assert len(ms) == 2 * w.L * w.M
    assert np.all(mnk == np.array([T, w.ffn, w.d]))
    assert np.all(ms > 0) and np.all(ms < 100)
    assert np.all(fl == 2.0 * T * w.ffn * w.d)
    assert np.array_equal(st0.host(st0.p32), st1.host(st1.p32))
    assert gp0.kernel_times()[0].size == 0
