"""Writes full_batch_losses.json: the fp64 oracle's loss of the full mini-batch
for the micro-batch-sweep workload (L=48, N=128, seq=256) and the
memory-scaling workload (L=96, N=256, seq=512), at their seeded inputs.

Calls only the oracle (oracle.model.forward_loss) and the seeded input
recipe.  Sequences are independent in the forward pass (LayerNorm and causal
attention act within a sequence; the review's "Batch Normalization" section
makes the same point for LayerNorm), so the full-batch loss is the sum over
disjoint groups of sequences of each group's loss normalised by the full
batch's N (seq - 1) targets; the oracle's own tests pin that identity.  The
groups only bound the host memory of one forward (one layer's activations of
a group live at a time); every per-sequence loss is the oracle's own.

The groups can be computed in separate runs (on different machines) and
merged: each run stores its groups under "parts"; once every group of a
workload is present the loss (summed in group order) and the per-sequence
losses are written.

    python tests/golden/make_full_batch_losses.py WORKLOAD [FIRST LAST] [--out FILE]
    python tests/golden/make_full_batch_losses.py --merge FILE ...
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import model as om  # noqa: E402
from synth import WORKLOADS, make_inputs  # noqa: E402

OUT = os.path.join(HERE, "full_batch_losses.json")
GROUP = {"lm_sweep": 16, "lm_deep": 8}   # sequences per forward


def _load(path):
    return json.load(open(path)) if os.path.exists(path) else {}


def _finalize(data):
    for name, entry in data.items():
        w = WORKLOADS[name]
        g = GROUP[name]
        parts = entry.get("parts", {})
        if len(parts) == w.n // g and "loss" not in entry:
            order = sorted(parts, key=int)
            entry["loss"] = float(sum(parts[i]["loss_part"] for i in order))
            entry["per_seq_loss"] = [x for i in order for x in parts[i]["per_seq_loss"]]
    return data


def compute(name, first, last, out):
    w = WORKLOADS[name]
    g = GROUP[name]
    inp = make_inputs(w)
    params = {k: np.asarray(v, dtype=np.float64) for k, v in inp.pop("params").items()}  # once, not per group
    count = w.n * (w.seq - 1)
    for gi in range(first, min(last, w.n // g)):
        data = _load(out)
        entry = data.setdefault(name, {"L": w.L, "n": w.n, "seq": w.seq, "d": w.d, "ffn": w.ffn,
                                       "vocab": w.vocab, "seed": w.seed, "group": g,
                                       "how": "oracle.model.forward_loss (fp64) over groups of sequences, "
                                              "count = N (seq - 1)", "parts": {}})
        if str(gi) in entry["parts"]:
            continue
        t0 = time.time()
        sub = {"tokens": inp["tokens"][gi * g:(gi + 1) * g]}
        loss, ex = om.forward_loss(w.replace(n=g), params, sub, count=count)
        entry["parts"][str(gi)] = {"loss_part": float(loss), "per_seq_loss": [float(x) for x in ex["per_seq_loss"]],
                                   "seconds": round(time.time() - t0, 1)}
        _finalize(data)
        with open(out + ".tmp", "w") as fh:
            json.dump(data, fh, indent=1)
        os.replace(out + ".tmp", out)
        print(f"{name}: group {gi} ({time.time() - t0:.0f} s)", flush=True)


def merge(paths, out):
    data = _load(out)
    for p in paths:
        for name, entry in _load(p).items():
            tgt = data.setdefault(name, {k: v for k, v in entry.items() if k not in ("parts", "loss", "per_seq_loss")})
            tgt.setdefault("parts", {}).update(entry.get("parts", {}))
    _finalize(data)
    with open(out, "w") as fh:
        json.dump(data, fh, indent=1)


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("workload", nargs="?")
    ap.add_argument("first", nargs="?", type=int, default=0)
    ap.add_argument("last", nargs="?", type=int, default=1 << 30)
    ap.add_argument("--out", default=OUT)
    ap.add_argument("--merge", nargs="*")
    a = ap.parse_args()
    if a.merge:
        merge(a.merge, a.out)
    else:
        compute(a.workload, a.first, a.last, a.out)
