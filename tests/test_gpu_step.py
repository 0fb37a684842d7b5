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
from tests.gpu_util import elementwise_outliers, error_profile, local_scale, rel

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


# How the error is distributed, next to the rel-L2 norms (tests/gpu_util.py
# error_profile): in every group (one parameter of one layer) the worst row's
# rel-L2 (a corrupted row shows there), the worst 64 x 64 block's rel-L2 (a
# wrong tile shows there) and the largest element error against |ref| plus
# its row's rms (a wild value shows there).  bf16: activations are rounded to
# 8 significant bits at every store, through up to 96 layers, and the
# measured per-group rel-L2 is 0.3-2%; single elements of the deep stacks'
# attention projections reach their row's scale (their gradients go through
# the softmax's cancellations), but a row's or a block's rel-L2 averages that
# noise, so rows and blocks are held to 0.25 and elements to 3.  fp32: errors
# ~1e-6, bounds 1e-4 (elements 1e-3).
BF16_LIMITS = {"row": 0.25, "block": 0.25, "elem": 3.0}
FP32_LIMITS = {"row": 1e-4, "block": 1e-4, "elem": 1e-3}


def _offsets(w):
    from synth import param_specs
    out, o = {}, 0
    for name, shape, _ in param_specs(w):
        out[name] = (o, shape)
        o += int(np.prod(shape))
    return out


def _compare_step(w, st, p0, loss, ref_loss, ref_grads, loss_tol, grad_tol, group_tol, limits, upd_thresh,
                  flip_frac):
    """GPU step against the oracle's full-batch step, group by group (host
    memory stays at one group at a time): the loss; every gradient group by
    rel-L2 and by the distribution of its error (rows, 64 x 64 blocks,
    elements); the whole gradient by rel-L2; and the RMSProp update of every
    group: its arithmetic on the GPU's own gradient, and against the oracle's
    update where the gradient's sign is fixed (|g| > upd_thresh times its
    row's rms; at most flip_frac of those elements flipped by the gradient's
    own error).  Every group is measured before anything is
    asserted, so a failure reports the worst groups of every measure."""
    offs = _offsets(w)
    num = den = 0.0
    prof = {}
    upd_bad = []
    step_max = w.lr / math.sqrt(1 - w.decay)
    masked = 0
    for name, (o, shape) in offs.items():
        n = int(np.prod(shape))
        g = st.g32[o:o + n].double().cpu().numpy().reshape(shape)
        gr = np.asarray(ref_grads[name], dtype=np.float64)
        num += float(np.sum((g - gr) ** 2))
        den += float(np.sum(gr ** 2))
        prof[name] = error_profile(g, gr)
        # the update.  (1) The RMSProp arithmetic itself, on the GPU's own
        # gradient (v0 = 0): v = (1 - decay) g^2, w -= lr g / (sqrt(v) + eps),
        # within fp32 rounding everywhere, and no weight moved by more than
        # lr / sqrt(1 - decay).  (2) Against the oracle's update where the
        # gradient's sign is fixed (|g| > upd_thresh times its row's rms): the
        # same step, but for the few elements whose sign the gradient's own
        # error flips (its element bound allows errors near the row's rms).
        p_init = np.asarray(p0[name], dtype=np.float64)
        p_gpu = st.p32[o:o + n].double().cpu().numpy().reshape(shape)
        v_gpu = st.v32[o:o + n].double().cpu().numpy().reshape(shape)
        dw_gpu = p_gpu - p_init
        p_own, v_own = om.rmsprop({name: p_init}, {name: g}, {name: np.zeros(shape)}, w.lr, w.decay, w.eps)
        if not (np.allclose(v_gpu, v_own[name], rtol=1e-6, atol=0.0) and
                np.allclose(p_gpu, p_own[name], rtol=0.0, atol=1e-6 * (np.abs(p_init) + step_max))):
            upd_bad.append((name, "RMSProp arithmetic"))
        if not np.all(np.abs(dw_gpu) <= step_max * (1 + 1e-3)):
            upd_bad.append((name, "step beyond lr/sqrt(1-decay)"))
        p_ref, _ = om.rmsprop({name: p_init}, {name: gr}, {name: np.zeros(shape)}, w.lr, w.decay, w.eps)
        dw_ref = p_ref[name] - p_init
        mask = np.abs(gr) > upd_thresh * local_scale(gr)
        masked += int(mask.sum())
        if mask.any():
            flips = elementwise_outliers(dw_gpu[mask], dw_ref[mask], 1e-2, 0.0)
            if flips > max(2, flip_frac * mask.sum()):
                upd_bad.append((name, flips, int(mask.sum())))
    report = {k: sorted(((p[k], nm) for nm, p in prof.items()), reverse=True)[:4]
              for k in ("rel", "row", "block", "elem", "frac25")}
    assert abs(loss - ref_loss) <= loss_tol * abs(ref_loss), (loss, ref_loss)
    assert math.sqrt(num / den) <= grad_tol, (math.sqrt(num / den), report)
    assert report["rel"][0][0] <= group_tol, report
    for k, lim in limits.items():
        assert report[k][0][0] <= lim, (k, report)
    assert not upd_bad, upd_bad
    assert masked > 0.3 * sum(int(np.prod(s)) for _, s in offs.values())


def test_tiny_ffn_fp32_step_matches_oracle(b):
    w = WORKLOADS["tiny_ffn"]
    inp = make_inputs(w)
    gp, st, p0, (loss,) = _run(b, w, inp)
    ref = om.step(w, inp["params"], inp)
    _compare_step(w, st, inp["params"], loss, ref["loss"], ref["grads"], 1e-5, 1e-5, 1e-5, FP32_LIMITS, 1e-2, 0.0)


def test_tiny_ffn_two_steps(b):
    w = WORKLOADS["tiny_ffn"]
    inp = make_inputs(w)
    gp, st, p0, losses = _run(b, w, inp, steps=2, keep_grads=False)
    ref1 = om.step(w, inp["params"], inp)
    ref2 = om.step(w, ref1["params"], inp, v=ref1["v"])
    assert abs(losses[0] - ref1["loss"]) <= 1e-5 * abs(ref1["loss"])
    assert abs(losses[1] - ref2["loss"]) <= 1e-5 * abs(ref2["loss"])
    assert not np.any(st.host(st.g32))   # the update leaves the accumulator zeroed


def _lm_parity(b, w, inp, loss_tol=1e-3, grad_tol=2e-2, group_tol=5e-2, ref=None, **kw):
    """A bf16 LM step against the oracle: loss, every gradient group (rel-L2
    and element-wise), the whole gradient, and the update.  ref: the oracle's
    (loss, grads) if already computed for these inputs."""
    gp, st, _, (loss,) = _run(b, w, inp, **kw)
    if ref is None:
        ref_loss, ref_grads, _ = om.loss_and_grads(w, inp["params"], inp)
    else:
        ref_loss, ref_grads = ref
    _compare_step(w, st, inp["params"], loss, ref_loss, ref_grads, loss_tol, grad_tol, group_tol, BF16_LIMITS, 0.75, 1e-3)
    return gp, st, {"loss": ref_loss, "grads": ref_grads}


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


def test_lm_wide_all_layers_sub_batch(b):
    """The wide workload (L=24, d=1024, ffn=8192, seq=256, K=8) with all its
    layers on a sub-batch of N=4 sequences in M=4 micro-batches (the full
    batch of 128 sequences is 36 GiB of fp64 activations on the host)."""
    w = WORKLOADS["lm_wide"].replace(n=4, M=4)
    _lm_parity(b, w, make_inputs(w))


def test_sweep_all_layers_two_partitions(b):
    """The micro-batch-sweep workload's 48 layers (d=1024, ffn=8192, seq=256)
    on a sub-batch of N=2 sequences in M=2 micro-batches, cut into K=2 and
    K=8 cells: both match the one oracle step (the oracle has no K)."""
    w = WORKLOADS["lm_sweep"].replace(n=2, M=2)
    inp = make_inputs(w)
    ref = None
    for K in (2, 8):
        _, _, r = _lm_parity(b, w.replace(K=K), inp, ref=ref)
        ref = (r["loss"], r["grads"])


def test_memory_scaling_all_layers_sub_batch(b):
    """The memory-scaling workload's 96 layers (d=1024, ffn=8192, seq=512,
    K=16 cells of 6 layers) on a sub-batch of N=2 sequences in M=2
    micro-batches: gradients accumulate over micro-batches at the full depth."""
    w = WORKLOADS["lm_deep"].replace(n=2, M=2)
    _lm_parity(b, w, make_inputs(w))


def _golden_losses():
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "full_batch_losses.json")
    with open(path) as fh:
        return json.load(fh)


@pytest.mark.parametrize("name", ["lm_sweep", "lm_deep"])
def test_full_batch_loss_matches_oracle(b, name):
    """The full mini-batch (N=128 at L=48; N=256 at L=96, seq 512) in the
    workload's own configuration: its loss and every sequence's loss against
    the fp64 oracle's forward, stored by tests/golden/make_full_batch_losses.py
    (a script that calls only the oracle)."""
    w = WORKLOADS[name]
    gold = _golden_losses()[name]
    if "loss" not in gold:
        pytest.skip(f"the oracle's full-batch loss of {name} has {len(gold.get('parts', {}))} of its "
                    f"{w.n // gold['group']} sequence groups so far")
    assert (gold["L"], gold["n"], gold["seq"], gold["seed"]) == (w.L, w.n, w.seq, w.seed)
    inp = make_inputs(w)
    gp, st, _, (loss,) = _run(b, w, inp, keep_grads=False, options=[(b.OPT_SKIP_UPDATE, 1)])
    assert abs(loss - gold["loss"]) <= 1e-3 * abs(gold["loss"]), (loss, gold["loss"])
    rows = gp.loss_rows(st.ws, w.n * w.seq, st.stream).reshape(w.n, w.seq)
    per_seq = rows.astype(np.float64).sum(axis=1) * w.n   # rows are divided by N (seq - 1)
    ref = np.array(gold["per_seq_loss"])
    assert np.all(np.abs(per_seq - ref) <= 2e-3 * ref), np.max(np.abs(per_seq - ref) / ref)


def test_memory_scaling_micro_batch_count_does_not_change_the_full_batch_step(b):
    """The review's equivalence claim at the memory-scaling workload's full
    size (N=256, seq 512, 96 layers): M=64 and M=16 micro-batches give the same
    loss and gradients within the bf16 tolerance (one update equals the
    full-batch step for any M).  Compared on the device."""
    import torch
    w = WORKLOADS["lm_deep"]
    inp = make_inputs(w)
    gp, st, _, (l64,) = _run(b, w, inp)
    g64 = st.g32.clone()
    del st
    gp.close()
    torch.cuda.empty_cache()
    gp, st, _, (l16,) = _run(b, w, inp, M=16, options=[(b.OPT_PIPELINE, 0)])
    assert abs(l16 - l64) <= 1e-4 * abs(l64), (l16, l64)
    d = float(torch.linalg.vector_norm((st.g32 - g64).double()) / torch.linalg.vector_norm(g64.double()))
    assert d <= 1e-2, d
    offs = _offsets(w)
    for name in ("l0.w_qkv", "l47.w1", "l95.w2", "emb", "l95.ln2_g"):
        o, shape = offs[name]
        n = int(np.prod(shape))
        x, y = st.g32[o:o + n].double(), g64[o:o + n].double()
        assert float(torch.linalg.vector_norm(x - y) / torch.linalg.vector_norm(y)) <= 2e-2, name


REMAT_SHAPES = {
    "small_lm": SMALL_LM,
    # the wide layer (d=1024, ffn=8192, seq 256): 1024-token micro-batches take
    # the persistent 128 x 256 GEMM, the separate bias-gradient reduction of
    # the wide weight gradients and the seq-256 attention
    "wide_layer": WORKLOADS["lm_wide"].replace(L=4, K=2, n=8, M=2),
    # the memory-scaling layer (seq 512)
    "deep_layer": WORKLOADS["lm_deep"].replace(L=4, K=2, n=4, M=2),
}


@pytest.mark.parametrize("shape", sorted(REMAT_SHAPES))
@pytest.mark.parametrize("m_check", [0, 1])
def test_rematerialised_internals_bit_identical(b, shape, m_check):
    """Every internal the backward's re-computation produces (LayerNorm
    outputs and statistics, QKV, attention output and log-sum-exp, the FFN
    pre-activation and GELU output, layer outputs) equals the first forward's
    byte for byte, for every cell, at micro-batch m_check."""
    w = REMAT_SHAPES[shape]
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


@pytest.mark.parametrize("sched", [0, 1])
def test_single_lane_activation_memory_measured_within_the_review_bound(b, sched):
    """The review's "Preliminaries 5" bound O(N + (L/K)(N/M)), written out from
    the shapes (gpipe_memory_report), against what the GPU writes: the
    workspace is filled with a sentinel, one step of the single-lane executor
    (cells in turn, the review's one-accelerator setting) runs, and the 4 KiB
    pages of the activation region that changed are counted.  They stay within
    the bound, and the step allocates no device memory.  The concurrent-lane
    executor writes more: one cell workspace per lane."""
    import torch
    w = WORKLOADS["lm_wide"].replace(n=8, M=4, L=8, K=4)
    inp = make_inputs(w)

    def touched(pipeline):
        gp = b.GPipe.from_workload(w)
        gp.set_option(b.OPT_SCHEDULE, sched)
        gp.set_option(b.OPT_PIPELINE, pipeline)
        st = b.DeviceState(gp, w, inp)   # workspace sized for this executor
        layout, bound = gp.memory_report()
        st.step(want_loss=False)         # captures and instantiates the step's graph
        st.ws.fill_(0xA5)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        st.step(want_loss=False)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        page = 4096
        region = st.ws[: layout - layout % page].view(-1, page)
        pages = int((region != 0xA5).any(dim=1).sum().item())
        return pages * page + (layout % page), free0 - free1, layout, bound

    used, alloc, layout, bound = touched(0)
    assert alloc <= 0
    assert used <= bound, (used, bound)
    assert used >= 0.95 * layout
    used_lanes, _, lanes_layout, lanes_bound = touched(1)
    assert lanes_bound == bound and bound < used_lanes <= lanes_layout
