"""Helpers shared by the GPU tests: device tensors, bf16 rounding, error norms."""
import numpy as np


def torch():
    import torch as t
    return t


def rel(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# Tensors made by dev() stay alive until the end of the test (conftest clears
# this list), so a pointer taken inline from a temporary stays valid while the
# kernel that was given it runs.
KEEP = []


def dev(x, dtype=None):
    """numpy -> cuda tensor (float arrays become fp32, or bf16 with dtype='bf16')."""
    t = torch()
    x = np.ascontiguousarray(x)
    if x.dtype.kind == "f":
        tt = t.from_numpy(x.astype(np.float32)).cuda()
        if dtype == "bf16":
            tt = tt.to(t.bfloat16)
    else:
        tt = t.from_numpy(x).cuda()
    KEEP.append(tt)
    return tt


def host(t_):
    return t_.detach().float().cpu().numpy().astype(np.float64)


def bf16_round(x):
    """Round-to-nearest-even to bf16, returned as float64 (via torch's CPU cast)."""
    t = torch()
    return t.from_numpy(np.asarray(x, dtype=np.float32)).to(t.bfloat16).float().numpy().astype(np.float64)


def stream():
    return torch().cuda.current_stream().cuda_stream


def sync():
    torch().cuda.synchronize()


def local_scale(ref):
    """Per-element scale of a reference array: the rms of its row for a matrix
    (a weight gradient's row is one output unit), of the whole for a vector."""
    r = np.asarray(ref, dtype=np.float64)
    if r.ndim >= 2:
        r2 = r.reshape(r.shape[0], -1)
        return np.broadcast_to(np.sqrt(np.mean(r2 * r2, axis=1, keepdims=True)), r2.shape).reshape(r.shape)
    return np.full(r.shape, np.sqrt(np.mean(r * r)) if r.size else 0.0)


def elementwise_outliers(got, ref, a, b):
    """Count of elements with |got - ref| > a |ref| + b scale (scale: local_scale(ref))."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    return int(np.count_nonzero(np.abs(g - r) > a * np.abs(r) + b * local_scale(r)))


def assert_elementwise(got, ref, a, b, max_frac, what=""):
    """Every element within a |ref| + b scale of the reference, but for at most
    max(2, max_frac * size) outliers (a rel-L2 norm alone would let a few
    corrupted rows or a wrong ragged tile through)."""
    n = int(np.size(ref))
    out = elementwise_outliers(got, ref, a, b)
    allowed = max(2, int(max_frac * n))
    assert out <= allowed, f"{what}: {out} of {n} elements outside {a}|ref| + {b} rms(row) (allowed {allowed})"
