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
