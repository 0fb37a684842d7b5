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
    (a weight gradient's row is one output unit), of the whole for a vector;
    never below 1% of the whole array's rms (a row whose exact value is 0,
    such as the first query's dQ, which cancels exactly, is then judged
    against the array's scale, not against 0)."""
    r = np.asarray(ref, dtype=np.float64)
    whole = np.sqrt(np.mean(r * r)) if r.size else 0.0
    if r.ndim >= 2:
        r2 = r.reshape(r.shape[0], -1)
        row = np.maximum(np.sqrt(np.mean(r2 * r2, axis=1, keepdims=True)), 1e-2 * whole)
        return np.broadcast_to(row, r2.shape).reshape(r.shape)
    return np.full(r.shape, whole)


def elementwise_outliers(got, ref, a, b):
    """Count of elements with |got - ref| > a |ref| + b scale (scale: local_scale(ref))."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    return int(np.count_nonzero(np.abs(g - r) > a * np.abs(r) + b * local_scale(r)))


def assert_elementwise(got, ref, a, b, max_frac, what=""):
    """Every element within a |ref| + b scale of the reference, but for at most
    max(2, max_frac * size) outliers (none when max_frac is 0); a rel-L2 norm
    alone would let a few corrupted rows or a wrong ragged tile through."""
    n = int(np.size(ref))
    out = elementwise_outliers(got, ref, a, b)
    allowed = max(2, int(max_frac * n)) if max_frac > 0 else 0
    assert out <= allowed, f"{what}: {out} of {n} elements outside {a}|ref| + {b} rms(row) (allowed {allowed})"


def error_profile(got, ref, block=64):
    """How the error of got against ref is distributed, scale by scale:
    rel       the whole array's rel-L2;
    row       the worst row's rel-L2 (rows of a matrix, 64-element blocks of a
              vector), each row's norm floored at a quarter of the array's
              typical row norm, so a row whose exact value is near 0 is judged
              against the array's scale;
    block     the worst 64 x 64 block's rel-L2 (the granularity of a GEMM
              tile's corner), floored likewise;
    elem      the largest |got - ref| / (|ref| + local_scale(ref));
    frac25    the fraction of elements with |got - ref| > 0.25 (|ref| + local_scale).
    A corrupted row shows in `row`, a wrong tile in `block`, a wild value in
    `elem`, while statistical rounding noise spreads over all of them."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    e = g - r
    out = {"rel": float(np.linalg.norm(e) / max(np.linalg.norm(r), 1e-300))}
    whole_rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0

    def worst_rel(pieces):
        w = 0.0
        for rp, ep in pieces:
            fl = 0.25 * whole_rms * np.sqrt(rp.size)
            w = max(w, float(np.sqrt(np.sum(ep * ep)) / max(np.sqrt(np.sum(rp * rp)), fl, 1e-300)))
        return w

    if r.ndim >= 2:
        r2, e2 = r.reshape(r.shape[0], -1), e.reshape(r.shape[0], -1)
        rows = [(r2[i], e2[i]) for i in range(r2.shape[0])]
        blocks = [(r2[i:i + block, j:j + block], e2[i:i + block, j:j + block])
                  for i in range(0, r2.shape[0], block) for j in range(0, r2.shape[1], block)]
    else:
        rows = blocks = [(r[i:i + block], e[i:i + block]) for i in range(0, r.size, block)]
    out["row"] = worst_rel(rows)
    out["block"] = worst_rel(blocks)
    sc = np.abs(r) + local_scale(r)
    q = np.abs(e) / np.maximum(sc, 1e-300)
    out["elem"] = float(np.max(q)) if q.size else 0.0
    out["frac25"] = float(np.mean(q > 0.25)) if q.size else 0.0
    return out
