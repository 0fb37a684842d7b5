"""ctypes binding of libgpipe (include/gpipe.h, include/gpipe_ops.h).

Argument marshalling only: every step of the training step runs in the
library's CUDA kernels.  PyTorch is used by ``DeviceState`` for device memory
and the current stream; nothing here computes any part of the method.  If the
shared library is missing this module raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import (POINTER, Structure, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_uint64,
                    c_void_p)

import numpy as np

from ._build import LIB

OK = 0
ERR = {-1: "INVALID_ARG", -2: "NOT_PARTITIONED", -3: "CUDA", -4: "DEVICE_TIMEOUT", -5: "NONFINITE_LOSS",
       -6: "UNSUPPORTED", -7: "IO"}

OPT_KEEP_GRADS, OPT_GRAPH, OPT_NO_REMAT, OPT_REMAT_CHECK, OPT_SKIP_UPDATE, OPT_CONCURRENT, OPT_PIPELINE, OPT_PDL = \
    1, 2, 3, 4, 5, 6, 7, 8
OPT_TRACE = 9
OPT_KERNEL_TIMES = 10
OPT_SM_SHARE = 11
OPT_INFLIGHT = 12
OPT_SIDE_SHARE = 13
OPT_SIDE_STREAMS = 14
OPT_SCHEDULE = 15
OPT_LOGIT_CLIP = 16
OPT_LAYER_TIMES = 17
SCHEDULE_GPIPE, SCHEDULE_1F1B = 0, 1
OP_FWD, OP_HEAD, OP_BWD = 0, 1, 2
EPI_STORE, EPI_BIAS_GELU, EPI_GELU_BWD, EPI_ACC_F32, EPI_STORE_F32, EPI_RESID_F32 = 0, 1, 2, 3, 4, 5


class GpipeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERR.get(code, code)}: {msg}")
        self.code = code


class Dims(Structure):
    _fields_ = [("kind", c_int), ("d", c_int), ("heads", c_int), ("ffn", c_int), ("seq", c_int),
                ("vocab", c_int), ("n", c_int), ("dtype", c_int), ("lr", c_float), ("decay", c_float),
                ("eps", c_float)]


_lib = None

# name: (restype, argtypes)
_SIGS = {
    "gpipe_create": (c_int, [POINTER(c_void_p), c_int, c_int, c_int, POINTER(Dims), POINTER(c_int64)]),
    "gpipe_create_layers": (c_int, [POINTER(c_void_p), c_int, c_int, c_int, POINTER(Dims), POINTER(c_int32),
                                    POINTER(c_int64)]),
    "gpipe_partition": (c_int, [c_void_p, POINTER(c_int32)]),
    "gpipe_repartition": (c_int, [c_void_p, POINTER(c_int64)]),
    "gpipe_checkpoint_write": (c_int, [c_void_p, ctypes.c_char_p, c_void_p, c_void_p, c_uint64]),
    "gpipe_checkpoint_read": (c_int, [c_void_p, ctypes.c_char_p, c_void_p, c_void_p, POINTER(c_uint64)]),
    "gpipe_sizes": (c_int, [c_void_p, POINTER(c_size_t), POINTER(c_size_t)]),
    "gpipe_init_params": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "gpipe_step": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                           c_void_p, POINTER(c_float)]),
    "gpipe_bubble_fraction": (c_double, [c_void_p]),
    "gpipe_schedule_model": (c_int, [c_void_p, POINTER(c_double), POINTER(c_double), POINTER(c_double),
                                     POINTER(c_double)]),
    "gpipe_memory_report": (c_int, [c_void_p, POINTER(c_size_t), POINTER(c_size_t)]),
    "gpipe_memory_model": (c_int, [c_void_p, POINTER(c_size_t), c_int]),
    "gpipe_issue_order": (c_int, [c_void_p, POINTER(c_int32), c_int]),
    "gpipe_layer_times": (c_int, [c_void_p, POINTER(c_float), POINTER(c_float), c_int]),
    "gpipe_set_option": (c_int, [c_void_p, c_int, c_int64]),
    "gpipe_debug_counters": (c_int, [c_void_p, c_void_p, c_void_p, POINTER(c_uint64), POINTER(c_int)]),
    "gpipe_loss_rows": (c_int, [c_void_p, c_void_p, c_void_p, POINTER(c_float), c_size_t]),
    "gpipe_launches_per_step": (c_int64, [c_void_p]),
    "gpipe_trace": (c_int, [c_void_p, c_void_p, c_void_p, POINTER(c_uint64), c_size_t]),
    "gpipe_kernel_times": (c_int, [c_void_p, POINTER(ctypes.c_float), POINTER(ctypes.c_double),
                                   POINTER(ctypes.c_int32), c_int]),
    "gpipe_last_error": (ctypes.c_char_p, [c_void_p]),
    "gpipe_destroy": (None, [c_void_p]),
    "gpipe_op_gemm": (c_int, [c_int, c_int, c_int, c_int, c_void_p, c_int64, c_int, c_void_p, c_int64, c_int, c_int,
                              c_void_p, c_int64, c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_int64,
                              c_void_p]),
    "gpipe_op_scratch_bytes": (c_size_t, [c_int, c_int]),
    "gpipe_op_layernorm_fwd": (c_int, [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p]),
    "gpipe_op_layernorm_bwd": (c_int, [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_layernorm_bwd_noalloc": (c_int, [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_colsum": (c_int, [c_int, c_int, c_int, c_void_p, c_int64, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_attention_fwd": (c_int, [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_attention_bwd": (c_int, [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p]),
    "gpipe_op_cross_entropy_clip": (c_int, [c_int, c_int, c_int, c_void_p, c_int, c_float, c_float, c_void_p, c_void_p,
                                            c_int, c_void_p]),
    "gpipe_op_cross_entropy": (c_int, [c_int, c_int, c_int, c_void_p, c_int, c_float, c_void_p, c_void_p, c_int,
                                       c_void_p]),
    "gpipe_op_mse": (c_int, [c_int, c_int, c_void_p, c_void_p, c_float, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_embedding_fwd": (c_int, [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_embedding_bwd": (c_int, [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_rmsprop": (c_int, [c_size_t, c_void_p, c_void_p, c_void_p, c_void_p, c_float, c_float, c_float,
                                 c_int, c_void_p]),
    "gpipe_op_cast_bf16": (c_int, [c_size_t, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_gelu": (c_int, [c_size_t, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gpipe_op_gemm_set_sm_share": (c_int, [c_int]),
    "gpipe_op_wait_probe": (c_int, [c_void_p]),
    "gpipe_op_device_error": (c_int, [POINTER(c_int), c_int, c_void_p]),
}


def exported_names():
    """The C symbols this binding expects (the declarations of include/*.h)."""
    return sorted(_SIGS)


def lib():
    """Load libgpipe.so (built in-tree by ``build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built: run __graft_entry__.build() (there is no fallback)")
        L = ctypes.CDLL(LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc, ctx=None):
    if rc != OK:
        msg = lib().gpipe_last_error(ctx)
        raise GpipeError(rc, msg.decode() if msg else "")


def _ptr(x):
    """Device pointer of a torch tensor (or an int / None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def current_stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


class GPipe:
    """Owns one gpipe_ctx (host state only).  Names mirror the C ABI."""

    def __init__(self, L, K, M, *, kind, d, heads, ffn, seq, vocab, n, dtype, lr=1e-3, decay=0.9, eps=1e-8,
                 cost=None, ffn_layers=None):
        self.dims = Dims(kind, d, heads, ffn, seq, vocab, n, dtype, lr, decay, eps)
        self.L, self.K, self.M = L, K, M
        h = c_void_p()
        carr = None
        if cost is not None:
            carr = (c_int64 * L)(*[int(c) for c in cost])
        farr = (c_int32 * L)(*[int(f) for f in ffn_layers]) if ffn_layers else None
        rc = lib().gpipe_create_layers(ctypes.byref(h), L, K, M, ctypes.byref(self.dims), farr, carr)
        if rc != OK:
            raise GpipeError(rc, lib().gpipe_last_error(None).decode())
        self.h = h

    @classmethod
    def from_workload(cls, w, cost=None, K=None, M=None):
        g = cls(w.L, K or w.K, M or w.M, kind=w.kind, d=w.d, heads=w.heads, ffn=w.ffn,
                seq=w.seq if w.kind == 1 else 1, vocab=w.vocab, n=w.n, dtype=0 if w.dtype == "f32" else 1,
                lr=w.lr, decay=w.decay, eps=w.eps, cost=cost, ffn_layers=tuple(getattr(w, "ffn_layers", ())))
        if getattr(w, "logit_clip_milli", 0):
            g.set_option(OPT_LOGIT_CLIP, w.logit_clip_milli)
        return g

    def close(self):
        if getattr(self, "h", None):
            lib().gpipe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- C ABI ---------------------------------------------------------------
    def partition(self):
        out = (c_int32 * (self.K + 1))()
        _check(lib().gpipe_partition(self.h, out), self.h)
        return list(out)

    def checkpoint_write(self, path, params, rms_v, step):
        """Write host float32 arrays (P each, packing order) and a step count."""
        p = np.ascontiguousarray(params, dtype=np.float32)
        v = np.ascontiguousarray(rms_v, dtype=np.float32)
        _check(lib().gpipe_checkpoint_write(self.h, os.fsencode(path), p.ctypes.data, v.ctypes.data, int(step)),
               self.h)

    def checkpoint_read(self, path):
        """(params, rms_v, step) from a checkpoint of this model (host arrays)."""
        P, _ = self.sizes()
        p = np.empty(P, dtype=np.float32)
        v = np.empty(P, dtype=np.float32)
        step = c_uint64()
        _check(lib().gpipe_checkpoint_read(self.h, os.fsencode(path), p.ctypes.data, v.ctypes.data,
                                           ctypes.byref(step)), self.h)
        return p, v, step.value

    def repartition(self, cost):
        arr = (c_int64 * self.L)(*[int(c) for c in cost])
        _check(lib().gpipe_repartition(self.h, arr), self.h)

    def sizes(self):
        p, w = c_size_t(), c_size_t()
        _check(lib().gpipe_sizes(self.h, ctypes.byref(p), ctypes.byref(w)), self.h)
        return p.value, w.value

    def init_params(self, p32, p16, stream=None):
        _check(lib().gpipe_init_params(self.h, _ptr(p32), _ptr(p16), stream), self.h)

    def step(self, p32, p16, g32, v32, batch, targets, workspace, stream=None, want_loss=True):
        loss = c_float()
        rc = lib().gpipe_step(self.h, _ptr(p32), _ptr(p16), _ptr(g32), _ptr(v32), _ptr(batch), _ptr(targets),
                              _ptr(workspace), stream, ctypes.byref(loss) if want_loss else None)
        _check(rc, self.h)
        return loss.value if want_loss else None

    def bubble_fraction(self):
        return lib().gpipe_bubble_fraction(self.h)

    def schedule_model(self, t_f=None, t_b=None):
        mk, bb = c_double(), c_double()
        tf = (c_double * self.K)(*t_f) if t_f is not None else None
        tb = (c_double * self.K)(*t_b) if t_b is not None else None
        _check(lib().gpipe_schedule_model(self.h, tf, tb, ctypes.byref(mk), ctypes.byref(bb)), self.h)
        return mk.value, bb.value

    def issue_order(self):
        """The step's issue order as a list of (kind, k, m, tick)."""
        n = lib().gpipe_issue_order(self.h, None, 0)
        _check(min(n, 0), self.h)
        buf = (c_int32 * (4 * n))()
        _check(min(lib().gpipe_issue_order(self.h, buf, n), 0), self.h)
        return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]

    def layer_times(self):
        """(forward ms, backward ms) per layer of the last step taken with
        OPT_LAYER_TIMES (empty arrays if none)."""
        fw = (c_float * self.L)()
        bw = (c_float * self.L)()
        n = lib().gpipe_layer_times(self.h, fw, bw, self.L)
        _check(min(n, 0), self.h)
        return np.array(fw[:n], dtype=np.float64), np.array(bw[:n], dtype=np.float64)

    def memory_report(self):
        a, b = c_size_t(), c_size_t()
        _check(lib().gpipe_memory_report(self.h, ctypes.byref(a), ctypes.byref(b)), self.h)
        return a.value, b.value

    MEMORY_TERMS = ("boundary", "cell", "head", "grads", "rows", "align", "total", "survey", "layout")

    def memory_model(self):
        """The review's activation bound term by term (gpipe_memory_model), in bytes."""
        buf = (c_size_t * len(self.MEMORY_TERMS))()
        n = lib().gpipe_memory_model(self.h, buf, len(buf))
        _check(min(n, 0), self.h)
        return dict(zip(self.MEMORY_TERMS, (int(x) for x in buf[:n])))

    def set_option(self, opt, value):
        _check(lib().gpipe_set_option(self.h, opt, int(value)), self.h)

    def debug_counters(self, workspace, stream=None):
        n, e = c_uint64(), c_int()
        _check(lib().gpipe_debug_counters(self.h, _ptr(workspace), stream, ctypes.byref(n), ctypes.byref(e)), self.h)
        return n.value, e.value

    def loss_rows(self, workspace, count, stream=None):
        out = (c_float * count)()
        _check(lib().gpipe_loss_rows(self.h, _ptr(workspace), stream, out, count), self.h)
        return np.frombuffer(out, dtype=np.float32).copy()

    def kernel_times(self, with_shapes=False):
        """(ms, flops[, mnk]) arrays of the GEMM launches selected by
        OPT_KERNEL_TIMES in the last step (waits for its events)."""
        n = lib().gpipe_kernel_times(self.h, None, None, None, 0)
        if n < 0:
            _check(n, self.h)
        ms = (ctypes.c_float * max(n, 1))()
        fl = (ctypes.c_double * max(n, 1))()
        mnk = (ctypes.c_int32 * max(3 * n, 1))()
        r = lib().gpipe_kernel_times(self.h, ms, fl, mnk, n)
        if r < 0:
            _check(r, self.h)
        out = (np.frombuffer(ms, dtype=np.float32)[:n].copy(), np.frombuffer(fl, dtype=np.float64)[:n].copy())
        if with_shapes:
            out += (np.frombuffer(mnk, dtype=np.int32)[:3 * n].reshape(n, 3).copy(),)
        return out

    def trace(self, workspace, stream=None):
        """(start, end, fwd[c][m], bwd[c][m]) in ns; c = 0..K (K: the head)."""
        n = 2 + 2 * (self.K + 1) * self.M
        out = (c_uint64 * n)()
        _check(lib().gpipe_trace(self.h, _ptr(workspace), stream, out, n), self.h)
        a = np.frombuffer(out, dtype=np.uint64).astype(np.int64)
        per = a[2:].reshape(self.K + 1, self.M, 2)
        return int(a[0]), int(a[1]), per[:, :, 0], per[:, :, 1]

    def launches_per_step(self):
        return lib().gpipe_launches_per_step(self.h)


def pack_params(w, params):
    """Flat fp32 array of the named parameters in the library's packing order."""
    from synth import param_specs
    return np.concatenate([np.asarray(params[name], dtype=np.float32).ravel() for name, _, _ in param_specs(w)])


def unpack(w, flat):
    """Named views of a flat per-parameter array (inverse of pack_params)."""
    from synth import param_specs
    out, o = {}, 0
    for name, shape, _ in param_specs(w):
        n = int(np.prod(shape))
        out[name] = flat[o:o + n].reshape(shape)
        o += n
    return out


class DeviceState:
    """Device buffers of one training run, allocated with torch on cuda.

    params_fp32 / params_bf16 / grads / rms_v (flat, packing order), the batch
    (tokens or x), targets, and the workspace of gpipe_sizes.
    """

    def __init__(self, gp: GPipe, w, inputs, device="cuda"):
        import torch
        self.torch = torch
        self.gp, self.w = gp, w
        P, ws = gp.sizes()
        flat = pack_params(w, inputs["params"])
        assert flat.size == P, (flat.size, P)
        self.P = P
        self.p32 = torch.from_numpy(flat).to(device)
        self.p16 = torch.empty(P, dtype=torch.bfloat16, device=device) if w.dtype == "bf16" else None
        self.g32 = torch.zeros(P, dtype=torch.float32, device=device)
        self.v32 = torch.zeros(P, dtype=torch.float32, device=device)
        if w.kind == 1:
            self.batch = torch.from_numpy(np.ascontiguousarray(inputs["tokens"], dtype=np.int32)).to(device)
            self.targets = None
        else:
            self.batch = torch.from_numpy(np.ascontiguousarray(inputs["x"], dtype=np.float32)).to(device)
            self.targets = torch.from_numpy(np.ascontiguousarray(inputs["targets"], dtype=np.float32)).to(device)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=device)
        self.stream = current_stream()
        gp.init_params(self.p32, self.p16, self.stream)

    def step(self, want_loss=True):
        return self.gp.step(self.p32, self.p16, self.g32, self.v32, self.batch, self.targets, self.ws,
                            self.stream, want_loss=want_loss)

    def host(self, t):
        return t.detach().float().cpu().numpy() if t is not None else None

    def save(self, path, step):
        """Checkpoint the state between steps (weights and RMSProp state)."""
        self.torch.cuda.synchronize()
        self.gp.checkpoint_write(path, self.host(self.p32), self.host(self.v32), step)

    def load(self, path):
        """Restore a checkpoint of this model: weights, RMSProp state and the
        bf16 copy; the gradient buffer is zeroed.  Returns the step count."""
        p, v, step = self.gp.checkpoint_read(path)
        self.p32.copy_(self.torch.from_numpy(p))
        self.v32.copy_(self.torch.from_numpy(v))
        self.g32.zero_()
        self.torch.cuda.synchronize()   # the copies ran on torch's current stream, the cast runs on ours
        self.gp.init_params(self.p32, self.p16, self.stream)
        return step
