"""The LayerNorm backward entry point that needs no caller scratch.

Some callers cannot allocate device memory when they call into the library
(a plugin whose host framework owns all device memory through its own pool, a
latency-critical path that must not enter the CUDA allocator).  For them
gpipe_op_layernorm_bwd_noalloc keeps its reduction scratch in a fixed array
inside the library.  This test calls it through the C ABI twice in a row, with
different shapes, and checks each result against the regular entry point
(which takes caller scratch): both run the same kernels in the same order on
the same inputs, so dx, dgamma and dbeta must agree bit for bit, in bf16 and in
fp32, and at exactly the largest size the fixed array holds; it also checks
that a size beyond the fixed array is refused.

The file name makes pytest collect it last.
"""
import numpy as np
import pytest

from tests.gpu_util import bf16_round, dev, host, rel, stream, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as ge
    ge.build()
    from micro_pipeline_re_gb300 import binding
    return binding.lib()


def _inputs(rows, d, seed):
    rng = np.random.default_rng(seed)
    x = bf16_round(rng.standard_normal((rows, d)) * 2 + 0.5)
    dy = bf16_round(rng.standard_normal((rows, d)))
    dres = bf16_round(rng.standard_normal((rows, d)))
    g = (1 + 0.3 * rng.standard_normal(d)).astype(np.float32)
    b = (0.2 * rng.standard_normal(d)).astype(np.float32)
    acc_g = rng.standard_normal(d).astype(np.float32)
    acc_b = rng.standard_normal(d).astype(np.float32)
    return x, dy, dres, g, b, acc_g, acc_b


def _run(lib, rows, d, seed, noalloc, dtype=1):
    import torch
    x, dy, dres, g, b, acc_g, acc_b = _inputs(rows, d, seed)
    act = "bf16" if dtype == 1 else None
    dx_in, ddy, ddres, dg, db = dev(x, act), dev(dy, act), dev(dres, act), dev(g), dev(b)
    y = torch.empty_like(dx_in)
    mean = torch.empty(rows, dtype=torch.float32, device="cuda")
    rstd = torch.empty(rows, dtype=torch.float32, device="cuda")
    assert lib.gpipe_op_layernorm_fwd(dtype, rows, d, dx_in.data_ptr(), dg.data_ptr(), db.data_ptr(), y.data_ptr(),
                                      mean.data_ptr(), rstd.data_ptr(), stream()) == 0
    dxo = torch.empty_like(dx_in)
    ag, ab = dev(acc_g), dev(acc_b)
    if noalloc:
        rc = lib.gpipe_op_layernorm_bwd_noalloc(dtype, rows, d, ddy.data_ptr(), dx_in.data_ptr(), mean.data_ptr(),
                                                rstd.data_ptr(), dg.data_ptr(), ddres.data_ptr(), dxo.data_ptr(),
                                                ag.data_ptr(), ab.data_ptr(), stream())
    else:
        scratch = torch.empty(lib.gpipe_op_scratch_bytes(rows, 2 * d) // 4 + 64, dtype=torch.float32, device="cuda")
        rc = lib.gpipe_op_layernorm_bwd(dtype, rows, d, ddy.data_ptr(), dx_in.data_ptr(), mean.data_ptr(),
                                        rstd.data_ptr(), dg.data_ptr(), ddres.data_ptr(), dxo.data_ptr(),
                                        ag.data_ptr(), ab.data_ptr(), scratch.data_ptr(), stream())
    assert rc == 0, lib.gpipe_last_error(None)
    sync()
    return host(dxo), host(ag), host(ab)


@pytest.mark.parametrize("dtype", [1, 0])
def test_noalloc_matches_regular_entry_point_twice(lib, dtype):
    # two calls in a row with different shapes; the second also shows that
    # what the first left in the shared array does not leak into its result
    for rows, d, seed in [(1000, 1024, 1), (203, 512, 2)]:
        ref = _run(lib, rows, d, seed, noalloc=False, dtype=dtype)
        got = _run(lib, rows, d, seed, noalloc=True, dtype=dtype)
        for a, r in zip(got, ref):
            assert np.array_equal(a, r)
        assert np.all(np.isfinite(got[0])) and rel(got[1], ref[1]) == 0.0


def test_noalloc_at_the_size_limit(lib):
    # ceil(4096 / 8) * 2 * 1024 = 2^20 floats: exactly the fixed array
    ref = _run(lib, 4096, 1024, 3, noalloc=False)
    got = _run(lib, 4096, 1024, 3, noalloc=True)
    for a, r in zip(got, ref):
        assert np.array_equal(a, r)


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    # ceil(rows/8) * 2d floats must fit in 2^20: rows = 8192 at d = 1024 needs 2^21
    rc = lib.gpipe_op_layernorm_bwd_noalloc(1, 8192, 1024, 16, 16, 16, 16, 16, None, 16, 16, 16, None)
    assert rc == -1
    assert b"more than the fixed" in lib.gpipe_last_error(None)
