"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (a dropped term, a wrong sign,
scale, index or mask, a transposed operand, a misread recurrence), on the CPU,
through monkeypatching, and checks that at least the named pin then fails.
The oracle itself is never modified on disk.
"""
import numpy as np
import pytest
from scipy.special import erf

import tests.test_oracle_model as tm
import tests.test_oracle_partition_schedule as tps
from oracle import model as om
from oracle import partition as opart
from oracle import schedule as osch


# ---------------------------------------------------------------- mutants
def ln_no_eps(x, g, b):
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var)
    xhat = (x - mu) * rstd
    return xhat * g + b, (xhat, rstd)


def ln_bwd_dropped_term(dy, cache, g):
    xhat, rstd = cache
    d = xhat.shape[-1]
    dxhat = dy * g
    dx = rstd * (dxhat - dxhat.mean(axis=-1, keepdims=True))
    return dx, (dy * xhat).reshape(-1, d).sum(axis=0), dy.reshape(-1, d).sum(axis=0)


def gelu_tanh(z):
    return 0.5 * z * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (z + 0.044715 * z ** 3)))


def gelu_grad_wrong_sign(z):
    return 0.5 * (1.0 + erf(z / np.sqrt(2.0))) - z / np.sqrt(2.0 * np.pi) * np.exp(-0.5 * z * z)


def attention_scale_1_over_d(q, k, v):
    dh = q.shape[-1]
    s = (q @ np.swapaxes(k, -1, -2)) / dh
    S = s.shape[-1]
    s = np.where(np.triu(np.ones((S, S), dtype=bool), k=1), -np.inf, s)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ v, p


def attention_mask_one_late(q, k, v):
    """Query i also sees key i+1."""
    dh = q.shape[-1]
    s = (q @ np.swapaxes(k, -1, -2)) / np.sqrt(dh)
    S = s.shape[-1]
    s = np.where(np.triu(np.ones((S, S), dtype=bool), k=2), -np.inf, s)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ v, p


def attention_bwd_dk_untransposed(do, q, k, v, p):
    scale = 1.0 / np.sqrt(q.shape[-1])
    dv = np.swapaxes(p, -1, -2) @ do
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (dp * p).sum(axis=-1, keepdims=True))
    return (ds @ k) * scale, (ds @ q) * scale, dv


def ce_target_not_shifted(z, tokens, count, clip=0.0):
    return _orig_ce(z, np.concatenate([tokens[:, :1], tokens[:, :-1]], axis=1), count, clip)


def ce_clip_without_mask(z, tokens, count, clip=0.0):
    if clip > 0:
        return _orig_ce(np.clip(z, -clip, clip), tokens, count, 0.0)
    return _orig_ce(z, tokens, count, 0.0)


def rmsprop_eps_inside(params, grads, v, lr, decay, eps):
    new_p, new_v = {}, {}
    for name, w0 in params.items():
        g = grads[name]
        vv = decay * np.asarray(v[name], dtype=np.float64) + (1.0 - decay) * g * g
        new_v[name] = vv
        new_p[name] = np.asarray(w0, dtype=np.float64) - lr * g / np.sqrt(vv + eps)
    return new_p, new_v


def rmsprop_decay_swapped(params, grads, v, lr, decay, eps):
    return _orig_rmsprop(params, grads, v, lr, 1.0 - decay, eps)


def partition_min_largest_cell(costs, K):
    """Minimises the largest cell instead of the variance."""
    from itertools import combinations
    L = len(costs)
    best, best_b = None, None
    for cuts in combinations(range(1, L), K - 1):
        b = [0, *cuts, L]
        v = max(opart.cell_sums(costs, b))
        if best is None or v < best:
            best, best_b = v, b
    return best_b, best


def one_f_one_b_warmup_without_head(K, M, k):
    """The warm-up as if the last cell were the last stage (min(M, K-k)
    forwards), forgetting the head."""
    warm = min(M, K - k)
    seq = [("F", m) for m in range(warm)]
    for m in range(M):
        seq.append(("B", m))
        if warm + m < M:
            seq.append(("F", warm + m))
    return seq


_orig_ce = om.next_token_ce
_orig_rmsprop = om.rmsprop


def block_backward_no_residual(kind, p, pre, x, cache, dy, grads):
    dx = _orig_block_backward(kind, p, pre, x, cache, dy, grads)
    return dx - dy   # drops the identity path of the outer residual


_orig_block_backward = om.block_backward


def simulate_backward_without_forward_barrier(K, M, t_f, t_b):
    """The GPipe clock with backward of (m, K-1) starting right after its own
    forward, not after the cell's last forward."""
    from fractions import Fraction
    tf = [Fraction(t_f)] * K if not hasattr(t_f, "__len__") else [Fraction(x) for x in t_f]
    tb = [Fraction(t_b)] * K if not hasattr(t_b, "__len__") else [Fraction(x) for x in t_b]
    f = [[Fraction(0)] * K for _ in range(M)]
    for m in range(M):
        for k in range(K):
            s = max(f[m - 1][k] if m else 0, f[m][k - 1] if k else 0)
            f[m][k] = s + tf[k]
    b = [[Fraction(0)] * K for _ in range(M)]
    for m in range(M):
        for k in reversed(range(K)):
            s = max(f[m][k], b[m - 1][k] if m else 0, b[m][k + 1] if k < K - 1 else 0)
            b[m][k] = s + tb[k]
    mk = max(b[m][0] for m in range(M))
    busy = [M * (tf[k] + tb[k]) for k in range(K)]
    return dict(makespan=mk, busy=busy, bubble=1 - Fraction(sum(busy)) / (K * mk))


# ---------------------------------------------------------------- cases
CASES = [
    ("layer_norm without eps", om, "layer_norm", ln_no_eps, tm.test_layer_norm_closed_form),
    ("LayerNorm backward drops its projection term", om, "layer_norm_backward", ln_bwd_dropped_term,
     lambda: tm.test_independent_autograd_library(tm.TINY_LM)),
    ("GELU by the tanh approximation", om, "gelu", gelu_tanh, tm.test_gelu_textbook_values),
    ("GELU derivative with a wrong sign", om, "gelu_grad", gelu_grad_wrong_sign,
     lambda: tm.test_independent_autograd_library(tm.TINY_FFN)),
    ("attention scaled by 1/dh", om, "causal_attention", attention_scale_1_over_d,
     tm.test_attention_causal_special_cases),
    ("attention mask one token late", om, "causal_attention", attention_mask_one_late,
     tm.test_attention_future_tokens_do_not_leak),
    ("attention backward with dK untransposed", om, "causal_attention_backward", attention_bwd_dk_untransposed,
     lambda: tm.test_independent_autograd_library(tm.TINY_LM)),
    ("block backward drops the residual path", om, "block_backward", block_backward_no_residual,
     lambda: tm.test_independent_autograd_library(tm.TINY_LM)),
    ("cross-entropy targets not shifted", om, "next_token_ce", ce_target_not_shifted,
     tm.test_cross_entropy_special_cases),
    ("clipped logits pass gradient", om, "next_token_ce", ce_clip_without_mask,
     tm.test_clipped_cross_entropy_closed_forms),
    ("RMSProp eps inside the square root", om, "rmsprop", rmsprop_eps_inside, tm.test_rmsprop_first_step_closed_form),
    ("RMSProp decay and (1-decay) swapped", om, "rmsprop", rmsprop_decay_swapped,
     tm.test_rmsprop_first_step_closed_form),
    ("partition minimises the largest cell", opart, "partition", partition_min_largest_cell,
     tps.test_partition_hand_worked_cases),
    ("one-forward-one-backward warm-up too short", osch, "one_f_one_b_sequence", one_f_one_b_warmup_without_head,
     tps.test_one_f_one_b_clock_hand_worked),
    ("GPipe clock without the all-forwards barrier", osch, "simulate", simulate_backward_without_forward_barrier,
     tps.test_simulation_unequal_cells_hand_worked),
]


@pytest.mark.parametrize("what,module,name,mutant,pin", CASES, ids=[c[0] for c in CASES])
def test_a_planted_mistake_fails_its_pin(monkeypatch, what, module, name, mutant, pin):
    pin()                                   # the pin passes on the oracle as written
    monkeypatch.setattr(module, name, mutant)
    with pytest.raises(Exception):
        pin()
