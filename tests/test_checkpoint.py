"""Checkpoint files of the training state (host side): round trip, and every
way a file can be wrong is refused without touching the caller's buffers."""
import os

import numpy as np
import pytest

from synth import KIND_LM, WORKLOADS, Workload

TMP = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_tmp")


@pytest.fixture(scope="module")
def binding():
    from micro_pipeline_re_gb300 import binding
    from micro_pipeline_re_gb300._build import build
    build()
    os.makedirs(TMP, exist_ok=True)
    return binding


def _state(g, seed):
    P, _ = g.sizes()
    rng = np.random.default_rng(seed)
    return rng.standard_normal(P).astype(np.float32), np.abs(rng.standard_normal(P)).astype(np.float32)


def test_round_trip_and_format(binding):
    g = binding.GPipe.from_workload(WORKLOADS["tiny_ffn"])
    p, v = _state(g, 1)
    path = os.path.join(TMP, "tiny.ck")
    g.checkpoint_write(path, p, v, 12345678901)
    assert os.path.getsize(path) == 72 + 8 * p.size
    p2, v2, step = g.checkpoint_read(path)
    assert step == 12345678901 and np.array_equal(p2, p) and np.array_equal(v2, v)
    # a second context of the same model reads it too
    p3, v3, _ = binding.GPipe.from_workload(WORKLOADS["tiny_ffn"], K=4, M=2).checkpoint_read(path)
    assert np.array_equal(p3, p) and np.array_equal(v3, v)
    assert not os.path.exists(path + ".tmp")


def _expect_io_error(g, path, what):
    """Reading fails with GPIPE_ERR_IO naming the problem, and leaves the
    caller's buffers as they were."""
    import ctypes
    from micro_pipeline_re_gb300 import binding
    with pytest.raises(binding.GpipeError) as e:
        g.checkpoint_read(path)
    assert e.value.code == -7 and what in str(e.value), str(e.value)
    P, _ = g.sizes()
    p = np.full(P, 3.0, dtype=np.float32)
    v = np.full(P, 4.0, dtype=np.float32)
    step = ctypes.c_uint64(99)
    rc = binding.lib().gpipe_checkpoint_read(g.h, os.fsencode(path), p.ctypes.data, v.ctypes.data, ctypes.byref(step))
    assert rc == -7 and np.all(p == 3.0) and np.all(v == 4.0) and step.value == 99


def test_damaged_or_foreign_files_are_refused(binding):
    w = Workload("ck_lm", KIND_LM, L=2, K=2, M=1, d=64, heads=1, ffn=128, seq=64, vocab=64, n=1, dtype="bf16",
                 ffn_layers=(128, 256))
    g = binding.GPipe.from_workload(w)
    p, v = _state(g, 2)
    path = os.path.join(TMP, "lm.ck")
    g.checkpoint_write(path, p, v, 7)
    blob = open(path, "rb").read()
    bad = os.path.join(TMP, "bad.ck")

    def with_bytes(data):
        with open(bad, "wb") as f:
            f.write(data)
        return bad

    flipped = bytearray(blob)
    flipped[100] ^= 1
    _expect_io_error(g, with_bytes(bytes(flipped)), "checksum")
    _expect_io_error(g, with_bytes(blob[:-4]), "length")
    _expect_io_error(g, with_bytes(blob + b"\0"), "length")
    _expect_io_error(g, with_bytes(b"NOTACKPT" + blob[8:]), "not a checkpoint")
    _expect_io_error(g, os.path.join(TMP, "missing.ck"), "cannot open")
    # same parameter count, layers of the other widths: another model
    other = binding.GPipe.from_workload(w.replace(ffn_layers=(256, 128)))
    assert other.sizes()[0] == g.sizes()[0]
    _expect_io_error(other, path, "different model")
    _expect_io_error(binding.GPipe.from_workload(w.replace(vocab=128)), path, "different model")
    # the good file still reads
    p2, v2, step = g.checkpoint_read(path)
    assert step == 7 and np.array_equal(p2, p) and np.array_equal(v2, v)


def test_interrupted_write_leaves_the_previous_checkpoint(binding):
    """A write that died before its rename leaves a truncated path.tmp behind:
    the previous checkpoint at path still reads back whole, and the next write
    replaces both."""
    g = binding.GPipe.from_workload(WORKLOADS["tiny_ffn"])
    p, v = _state(g, 3)
    path = os.path.join(TMP, "interrupted.ck")
    g.checkpoint_write(path, p, v, 5)
    with open(path + ".tmp", "wb") as f:
        f.write(open(path, "rb").read()[:1000])
    p2, v2, step = g.checkpoint_read(path)
    assert step == 5 and np.array_equal(p2, p) and np.array_equal(v2, v)
    q, u = _state(g, 4)
    g.checkpoint_write(path, q, u, 6)
    q2, u2, step = g.checkpoint_read(path)
    assert step == 6 and np.array_equal(q2, q) and np.array_equal(u2, u)
    assert not os.path.exists(path + ".tmp")
