"""The depth-scaled FFN initialisation of the input recipe (the GPipe technical
review's "Training stability": the feed-forward layers' initialisation shrunk
with the depth L), read as variance 1/(d L) for W1 and W2 instead of 1/d."""
import numpy as np

from synth import WORKLOADS, make_inputs


def test_ffn_init_depth_scaled_shrinks_only_the_ffn_matrices():
    w = WORKLOADS["lm_small"].replace(L=4, vocab=1000)
    plain = make_inputs(w)
    scaled = make_inputs(w.replace(ffn_init_depth_scaled=True))
    assert np.array_equal(plain["tokens"], scaled["tokens"])
    s = 1.0 / np.sqrt(w.L)
    for name, a in plain["params"].items():
        b = scaled["params"][name]
        if name.endswith(".w1") or name.endswith(".w2"):
            # the same draws, times 1/sqrt(L) (up to the fp32 scale factors' rounding)
            assert np.allclose(b, a * s, rtol=2e-7, atol=0), name
            assert abs(np.var(b) * w.d * w.L - 1.0) < 0.02, name
        else:
            assert np.array_equal(a, b), name
