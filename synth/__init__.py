"""Seeded synthetic workloads shared by the oracle side and the GPU side.

This module holds only shapes, parameter names/order and random draws.  It
contains none of the method's arithmetic (no layer, loss, gradient, optimizer,
partition or schedule computation), so both the CPU oracle and the CUDA path
can take their inputs from here without sharing any computation.

Workloads follow the GPipe technical review (zzz0906.github.io), section
"Algorithm / minimal interface": a model is a sequence of L identical layers,
the user chooses K (cells) and M (micro-batches), and the mini-batch has N
samples.  The concrete shapes are the five synthetic workloads of this build
(tiny FFN check, small causal LM, wide LM, micro-batch sweep, memory scaling).

Random-draw recipe (fixed order, one generator per workload):
  rng = numpy.random.default_rng(seed)
  kind 0 (FFN blocks, MSE):  x ~ N(0,1) [N,d] fp32, then targets ~ N(0,1) [N,d]
  kind 1 (causal LM):        tokens ~ U{0..V-1} [N,seq] int32
  then every parameter in packing order: matrices ~ N(0, 1/d) (variance 1/d,
  d = model width), biases and LN shifts 0 (no draw), LN gains 1 (no draw).
  With ffn_init_depth_scaled, the FFN matrices W1 and W2 take variance
  1/(d L) instead (the same draws times 1/sqrt(L)).

Trainability options of the GPipe technical review's "Training stability"
section (off by default): ffn_init_depth_scaled (the feed-forward layers'
initialisation shrunk with the depth L) and logit_clip_milli (a logit
clipping threshold in thousandths, handed to the step, not applied here).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

KIND_FFN = 0   # residual pre-LN FFN block, no attention, MSE loss, no embedding/head
KIND_LM = 1    # pre-LN Transformer block, tied embedding, next-token cross-entropy


@dataclass(frozen=True)
class Workload:
    name: str
    kind: int
    L: int
    K: int
    M: int
    d: int
    heads: int
    ffn: int
    seq: int
    vocab: int
    n: int
    dtype: str            # "f32": fp32 throughout; "bf16": bf16 compute, fp32 master/grads/state
    lr: float = 1e-3
    decay: float = 0.9
    eps: float = 1e-8
    seed: int = 0
    ffn_init_depth_scaled: bool = False
    logit_clip_milli: int = 0
    ffn_layers: tuple = ()   # per-layer FFN widths (heterogeneous layers); empty: ffn everywhere

    @property
    def tokens(self) -> int:
        """Tokens (kind 1) or rows (kind 0) per mini-batch."""
        return self.n * (self.seq if self.kind == KIND_LM else 1)

    @property
    def tokens_per_micro_batch(self) -> int:
        return self.tokens // self.M

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads.  Index 0 is the tiny fp32 check that the oracle finishes
# in well under a second; index 1 is the small causal LM that the throughput
# line is quoted on; 2..4 are the larger shapes.
WORKLOADS = {
    "tiny_ffn": Workload("tiny_ffn", KIND_FFN, L=4, K=2, M=4, d=64, heads=0, ffn=256,
                         seq=1, vocab=0, n=32, dtype="f32"),
    "lm_small": Workload("lm_small", KIND_LM, L=8, K=4, M=16, d=512, heads=8, ffn=2048,
                         seq=128, vocab=32000, n=64, dtype="bf16"),
    "lm_wide": Workload("lm_wide", KIND_LM, L=24, K=8, M=32, d=1024, heads=16, ffn=8192,
                        seq=256, vocab=32000, n=128, dtype="bf16"),
    "lm_sweep": Workload("lm_sweep", KIND_LM, L=48, K=8, M=32, d=1024, heads=16, ffn=8192,
                         seq=256, vocab=32000, n=128, dtype="bf16"),
    "lm_deep": Workload("lm_deep", KIND_LM, L=96, K=16, M=64, d=1024, heads=16, ffn=8192,
                        seq=512, vocab=32000, n=256, dtype="bf16"),
}

# (K, M) grid of the micro-batch sweep workload.
SWEEP_GRID = [(k, m) for k in (2, 4, 8) for m in (1, 4, 32)]


def layer_ffn(w: Workload):
    """FFN width of every layer."""
    if w.ffn_layers:
        if len(w.ffn_layers) != w.L:
            raise ValueError("ffn_layers needs one width per layer")
        return [int(f) for f in w.ffn_layers]
    return [w.ffn] * w.L


def param_specs(w: Workload):
    """Parameters in flat packing order: list of (name, shape, init).

    init is "normal" (N(0, 1/d)), "ones" or "zeros".  Weight matrices are stored
    [out_features, in_features] row-major, so a projection computes x @ W^T.
    The fused QKV matrix stacks the query, key and value rows in that order,
    each block d rows with heads contiguous (head h owns rows h*dh..(h+1)*dh-1).
    """
    d = w.d
    specs = []
    for l, f in enumerate(layer_ffn(w)):
        p = f"l{l}."
        if w.kind == KIND_FFN:
            specs += [(p + "ln_g", (d,), "ones"), (p + "ln_b", (d,), "zeros"),
                      (p + "w1", (f, d), "normal"), (p + "b1", (f,), "zeros"),
                      (p + "w2", (d, f), "normal"), (p + "b2", (d,), "zeros")]
        else:
            specs += [(p + "ln1_g", (d,), "ones"), (p + "ln1_b", (d,), "zeros"),
                      (p + "w_qkv", (3 * d, d), "normal"), (p + "b_qkv", (3 * d,), "zeros"),
                      (p + "w_o", (d, d), "normal"), (p + "b_o", (d,), "zeros"),
                      (p + "ln2_g", (d,), "ones"), (p + "ln2_b", (d,), "zeros"),
                      (p + "w1", (f, d), "normal"), (p + "b1", (f,), "zeros"),
                      (p + "w2", (d, f), "normal"), (p + "b2", (d,), "zeros")]
    if w.kind == KIND_LM:
        specs += [("lnf_g", (d,), "ones"), ("lnf_b", (d,), "zeros"),
                  ("emb", (w.vocab, d), "normal")]
    return specs


def param_count(w: Workload) -> int:
    return int(sum(np.prod(s) for _, s, _ in param_specs(w)))


def make_inputs(w: Workload, params: bool = True):
    """Draw the batch (and parameters) of workload ``w``.

    Returns dict with "x" and "targets" (kind 0, fp32 [N,d]) or "tokens"
    (kind 1, int32 [N,seq]), and "params": {name: fp32 array} in packing order.
    """
    rng = np.random.default_rng(w.seed)
    out = {}
    if w.kind == KIND_FFN:
        out["x"] = rng.standard_normal((w.n, w.d), dtype=np.float32)
        out["targets"] = rng.standard_normal((w.n, w.d), dtype=np.float32)
    else:
        out["tokens"] = rng.integers(0, w.vocab, size=(w.n, w.seq), dtype=np.int32)
    if params:
        scale = np.float32(1.0 / np.sqrt(w.d))
        ffn_scale = np.float32(1.0 / np.sqrt(w.d * w.L)) if w.ffn_init_depth_scaled else scale
        ps = {}
        for name, shape, init in param_specs(w):
            if init == "normal":
                is_ffn = name.endswith(".w1") or name.endswith(".w2")
                ps[name] = rng.standard_normal(shape, dtype=np.float32) * (ffn_scale if is_ffn else scale)
            elif init == "ones":
                ps[name] = np.ones(shape, dtype=np.float32)
            else:
                ps[name] = np.zeros(shape, dtype=np.float32)
        out["params"] = ps
    return out


def random_costs(rng: np.random.Generator, L: int, lo: int = 1, hi: int = 100):
    """Integer per-layer cost estimates for partition tests."""
    return [int(c) for c in rng.integers(lo, hi + 1, size=L)]
