"""Kernel-level parity through the gpipe_op_* C entry points.

Every expected value is computed on the CPU in fp64 from the same seeded
inputs (rounded to bf16 where the kernel reads bf16), with the oracle's layer
functions where one exists.  Shapes span several tiles and leave ragged tails.
"""
import numpy as np
import pytest

from oracle import model as om
from tests.gpu_util import assert_elementwise, bf16_round, dev, host, rel, stream, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    import __graft_entry__ as ge
    ge.build()
    from micro_pipeline_re_gb300 import binding
    return binding


def _gemm_ref(A, B, ak, bk):
    """sum_k A(m,k) B(n,k) with the op's layout conventions (A, B as stored)."""
    Am = A if ak else A.T
    Bm = B if bk else B.T
    return Am @ Bm.T


# (M, N, K): several tiles with ragged tails in every dimension
# (the last one has enough 128-wide tiles to take the 128-column variant;
# the others take the 64-column one)
# (1704^2 has enough 128-wide tiles for the 128-column variant or, for the
# 128-wide epilogues, the persistent kernel; the others take the 64-column one;
# the two long-K shapes split K across a cluster; 2056 x 2568 takes the
# persistent kernel for every epilogue, ragged in M, N and K; 1000 x 1280 x
# 2056 has fewer 128-wide tiles than SMs but a long K, so it takes the
# 128-column single-tile kernel)
SHAPES = [(384, 640, 512), (200, 136, 200), (128, 128, 64), (1000, 96, 72), (1704, 1704, 200),
          (200, 256, 16384), (256, 136, 4096), (2056, 2568, 264), (1000, 1280, 2056)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("ak,bk,epi", [
    (1, 1, 0), (1, 1, 1), (1, 1, 3), (1, 1, 4),
    (1, 0, 0), (1, 0, 2), (1, 0, 3),
    (0, 0, 0), (0, 0, 3),
])
def test_gemm_tensor_core(b, shape, ak, bk, epi):
    _check_gemm(b, shape, ak, bk, epi)


# (M, N, K) that the persistent path runs on 256 x 256 tiles over SM pairs
# (256-row MMAs across two CTAs; K >= 1024) at a 16-SM share: one that tiles
# exactly and one ragged in every dimension (a pair's second CTA past the last
# row, its half of B past the last column, a partial last k-block).
PAIR_SHAPES = [(2048, 2048, 1024), (1000, 1288, 1064)]


@pytest.mark.parametrize("shape", PAIR_SHAPES)
@pytest.mark.parametrize("ak,bk,epi", [
    (1, 1, 0), (1, 1, 1), (1, 1, 3), (1, 1, 4),
    (1, 0, 0), (1, 0, 2), (1, 0, 3),
    (0, 0, 0), (0, 0, 3),
])
def test_gemm_sm_pair_tiles(b, shape, ak, bk, epi):
    assert b.lib().gpipe_op_gemm_set_sm_share(16) == 0
    try:
        _check_gemm(b, shape, ak, bk, epi)
    finally:
        assert b.lib().gpipe_op_gemm_set_sm_share(0) == 0


def _check_gemm(b, shape, ak, bk, epi):
    M, N, K = shape
    rng = np.random.default_rng(M * 7 + N * 3 + K + 10 * ak + 20 * bk + epi)
    A = bf16_round(rng.standard_normal((M, K) if ak else (K, M)))
    B = bf16_round(rng.standard_normal((N, K) if bk else (K, N)))
    acc = _gemm_ref(A, B, ak, bk)
    t = __import__("torch")
    dA, dB = dev(A, "bf16"), dev(B, "bf16")
    lda, ldb = A.shape[1], B.shape[1]
    bias = rng.standard_normal(N).astype(np.float32)
    resid = bf16_round(rng.standard_normal((M, N)))
    aux = bf16_round(rng.standard_normal((M, N)))
    if epi in (3, 4):
        C0 = rng.standard_normal((M, N)).astype(np.float32) if epi == 3 else np.zeros((M, N), np.float32)
        dC = dev(C0)
        db0 = rng.standard_normal(M).astype(np.float32)
        ddb = dev(db0) if epi == 3 else None   # fused bias gradient: += sum_k A(m,k)
        rc = b.lib().gpipe_op_gemm(1, M, N, K, dA.data_ptr(), lda, ak, dB.data_ptr(), ldb, bk, epi, dC.data_ptr(), N,
                                   ddb.data_ptr() if epi == 3 else None, None, 0, None, None, 0, stream())
        assert rc == 0, b.lib().gpipe_last_error(None)
        sync()
        want = acc + (C0 if epi == 3 else 0)
        # fp32 accumulation over K terms: relative error grows like sqrt(K) 2^-24
        tol = 1e-5 * max(1.0, (K / 1024) ** 0.5)
        assert rel(host(dC), want) <= tol
        if epi == 3:
            assert rel(host(ddb), db0 + (A if ak else A.T).sum(axis=1)) <= tol
        return
    dC = t.empty((M, N), dtype=t.bfloat16, device="cuda")
    dC2 = t.empty((M, N), dtype=t.bfloat16, device="cuda")
    dbias, dres, daux = dev(bias), dev(resid, "bf16"), dev(aux, "bf16")
    use_bias = epi in (0, 1)
    use_res = epi == 0 and ak == 1 and bk == 1
    rc = b.lib().gpipe_op_gemm(1, M, N, K, dA.data_ptr(), lda, ak, dB.data_ptr(), ldb, bk, epi, dC.data_ptr(), N,
                               dbias.data_ptr() if use_bias else None, dres.data_ptr() if use_res else None, N,
                               dC2.data_ptr() if epi == 1 else None, daux.data_ptr() if epi == 2 else None, N,
                               stream())
    assert rc == 0, b.lib().gpipe_last_error(None)
    sync()
    if epi == 0:
        want = acc + (bias if use_bias else 0) + (resid if use_res else 0)
        assert rel(host(dC), want) <= 6e-3
    elif epi == 1:
        z = acc + bias
        assert rel(host(dC), z) <= 6e-3
        assert rel(host(dC2), om.gelu(z)) <= 6e-3
    else:
        assert rel(host(dC), acc * om.gelu_grad(aux)) <= 6e-3


@pytest.mark.parametrize("shape", [(384, 640, 512), (200, 136, 200), (1000, 96, 72), (2056, 2568, 264),
                                   (2048, 1024, 8192)])
def test_gemm_fp32_residual_epilogue(b, shape):
    """The residual adds that keep the residual stream in fp32: C (fp32) =
    (A B^T + bias) + R (fp32), against fp64, through the single-tile and the
    persistent kernels (ragged tiles; the memory-scaling workload's output
    projection shape), and with the same bits whatever the SM share (so
    whichever kernel the share picks)."""
    t = __import__("torch")
    M, N, K = shape
    rng = np.random.default_rng(M + N + K)
    A = bf16_round(rng.standard_normal((M, K)))
    B = bf16_round(rng.standard_normal((N, K)) / np.sqrt(K))
    bias = rng.standard_normal(N).astype(np.float32)
    R = (rng.standard_normal((M, N)) * 4).astype(np.float32)
    dA, dB, dbias, dR = dev(A, "bf16"), dev(B, "bf16"), dev(bias), dev(R)
    outs = []
    lib = b.lib()
    for sms in (0, 16):
        assert lib.gpipe_op_gemm_set_sm_share(sms) == 0
        dC = t.empty((M, N), dtype=t.float32, device="cuda")
        rc = lib.gpipe_op_gemm(1, M, N, K, dA.data_ptr(), K, 1, dB.data_ptr(), K, 1, b.EPI_RESID_F32, dC.data_ptr(),
                               N, dbias.data_ptr(), dR.data_ptr(), N, None, None, 0, stream())
        assert rc == 0, lib.gpipe_last_error(None)
        sync()
        outs.append(host(dC))
    assert lib.gpipe_op_gemm_set_sm_share(0) == 0
    want = A @ B.T + bias + R
    # fp32 accumulation of bf16 products: relative to the product's scale
    tol = 1e-5 * max(1.0, (K / 1024) ** 0.5)
    assert np.max(np.abs(outs[0] - want)) <= tol * (np.sqrt(K) * np.abs(B).max() * 4 + 8)
    assert rel(outs[0], want) <= 1e-5
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("ak,bk,epi", [(1, 1, 0), (1, 1, 1), (1, 0, 2), (0, 0, 3), (0, 1, 0), (1, 1, 5)])
def test_gemm_fp32_ffma(b, ak, bk, epi):
    M, N, K = 136, 200, 72
    rng = np.random.default_rng(5 + epi)
    A = rng.standard_normal((M, K) if ak else (K, M)).astype(np.float32)
    B = rng.standard_normal((N, K) if bk else (K, N)).astype(np.float32)
    acc = _gemm_ref(A.astype(np.float64), B.astype(np.float64), ak, bk)
    bias = rng.standard_normal(N).astype(np.float32)
    resid = rng.standard_normal((M, N)).astype(np.float32)
    aux = rng.standard_normal((M, N)).astype(np.float32)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    dC, dC2 = dev(C0), dev(np.zeros((M, N), np.float32))
    keep = [dev(A), dev(B), dev(bias), dev(resid), dev(aux)]  # hold device buffers until the kernel ran
    db0 = rng.standard_normal(M).astype(np.float32)
    ddb = dev(db0)
    rc = b.lib().gpipe_op_gemm(0, M, N, K, keep[0].data_ptr(), A.shape[1], ak, keep[1].data_ptr(), B.shape[1], bk,
                               epi, dC.data_ptr(), N,
                               keep[2].data_ptr() if epi in (0, 1, 5) else (ddb.data_ptr() if epi == 3 else None),
                               keep[3].data_ptr() if epi in (0, 5) else None, N, dC2.data_ptr() if epi == 1 else None,
                               keep[4].data_ptr() if epi == 2 else None, N, stream())
    assert rc == 0
    sync()
    if epi in (0, 5):
        assert rel(host(dC), acc + bias + resid) <= 1e-6
    elif epi == 1:
        assert rel(host(dC), acc + bias) <= 1e-6
        assert rel(host(dC2), om.gelu(acc + bias)) <= 1e-6
    elif epi == 2:
        assert rel(host(dC), acc * om.gelu_grad(aux)) <= 1e-6
    else:
        assert rel(host(dC), C0 + acc) <= 1e-6
        assert rel(host(ddb), db0 + (A if ak else A.T).astype(np.float64).sum(axis=1)) <= 1e-6


def test_gemm_rejects_misaligned_leading_dimension(b):
    t = __import__("torch")
    A = t.zeros((64, 72), dtype=t.bfloat16, device="cuda")
    C = t.zeros((64, 64), dtype=t.bfloat16, device="cuda")
    rc = b.lib().gpipe_op_gemm(1, 64, 64, 70, A.data_ptr(), 70, 1, A.data_ptr(), 70, 1, 0, C.data_ptr(), 64,
                               None, None, 0, None, None, 0, stream())
    assert rc == -1


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("rows,d", [(203, 64), (77, 512), (130, 1024)])
def test_layernorm_fwd_bwd(b, dtype, rows, d):
    t = __import__("torch")
    rng = np.random.default_rng(rows + d + dtype)
    x = rng.standard_normal((rows, d)) * 2 + 0.5
    dy = rng.standard_normal((rows, d))
    dres = rng.standard_normal((rows, d))
    g = (1 + 0.3 * rng.standard_normal(d)).astype(np.float32)
    bb = (0.2 * rng.standard_normal(d)).astype(np.float32)
    if dtype == 1:
        x, dy, dres = bf16_round(x), bf16_round(dy), bf16_round(dres)
    tdt = "bf16" if dtype else None
    dx_in = dev(x, tdt)
    y = t.empty_like(dx_in)
    mean = t.empty(rows, dtype=t.float32, device="cuda")
    rstd = t.empty(rows, dtype=t.float32, device="cuda")
    lib = b.lib()
    assert lib.gpipe_op_layernorm_fwd(dtype, rows, d, dx_in.data_ptr(), dev(g).data_ptr(), dev(bb).data_ptr(),
                                      y.data_ptr(), mean.data_ptr(), rstd.data_ptr(), stream()) == 0
    ref, cache = om.layer_norm(x, g.astype(np.float64), bb.astype(np.float64))
    sync()
    tol = 1e-6 if dtype == 0 else 6e-3
    assert rel(host(y), ref) <= tol
    assert rel(host(mean), x.mean(axis=1)) <= 1e-6
    assert rel(host(rstd), cache[1][:, 0]) <= 1e-5
    dg0 = rng.standard_normal(d).astype(np.float32)
    db0 = rng.standard_normal(d).astype(np.float32)
    ddg, ddb = dev(dg0), dev(db0)
    dxo = t.empty_like(dx_in)
    scratch = t.empty(lib.gpipe_op_scratch_bytes(rows, 2 * d) // 4 + 64, dtype=t.float32, device="cuda")
    assert lib.gpipe_op_layernorm_bwd(dtype, rows, d, dev(dy, tdt).data_ptr(), dx_in.data_ptr(), mean.data_ptr(),
                                      rstd.data_ptr(), dev(g).data_ptr(), dev(dres, tdt).data_ptr(), dxo.data_ptr(),
                                      ddg.data_ptr(), ddb.data_ptr(), scratch.data_ptr(), stream()) == 0
    sync()
    rdx, rdg, rdb = om.layer_norm_backward(dy, cache, g.astype(np.float64))
    assert rel(host(dxo), rdx + dres) <= (1e-5 if dtype == 0 else 8e-3)
    assert rel(host(ddg), dg0 + rdg) <= 1e-5
    assert rel(host(ddb), db0 + rdb) <= 1e-5


@pytest.mark.parametrize("dtype", [0, 1])
def test_colsum(b, dtype):
    t = __import__("torch")
    rows, cols, ld = 333, 3 * 1024, 3 * 1024 + 64
    rng = np.random.default_rng(9)
    y = rng.standard_normal((rows, ld))
    if dtype:
        y = bf16_round(y)
    out0 = rng.standard_normal(cols).astype(np.float32)
    dout = dev(out0)
    scratch = t.empty(b.lib().gpipe_op_scratch_bytes(rows, cols) // 4 + 64, dtype=t.float32, device="cuda")
    assert b.lib().gpipe_op_colsum(dtype, rows, cols, dev(y, "bf16" if dtype else None).data_ptr(), ld,
                                   dout.data_ptr(), scratch.data_ptr(), stream()) == 0
    sync()
    assert rel(host(dout), out0 + y[:, :cols].sum(axis=0)) <= 1e-6


def _attn_inputs(nseq, seq, heads, seed):
    rng = np.random.default_rng(seed)
    D = heads * 64
    qkv = bf16_round(rng.standard_normal((nseq * seq, 3 * D)))
    dout = bf16_round(rng.standard_normal((nseq * seq, D)))
    return qkv, dout


def _split(qkv, nseq, seq, heads):
    D = heads * 64
    parts = []
    for i in range(3):
        t = qkv[:, i * D:(i + 1) * D].reshape(nseq, seq, heads, 64).transpose(0, 2, 1, 3)
        parts.append(t)
    return parts


@pytest.mark.parametrize("nseq,seq,heads", [(2, 128, 2), (1, 192, 3), (3, 64, 1), (2, 512, 1), (1, 320, 2),
                                             (4, 512, 16)])
def test_attention_fwd_bwd(b, nseq, seq, heads):
    """Causal attention forward and backward against the oracle's, by rel-L2
    and element by element (the output within 5% of its value plus 5% of its
    row's rms, the gradients within 10%, a few outliers allowed), over ragged sequence lengths (64 past a
    multiple of 128) and the memory-scaling workload's micro-batch shape."""
    t = __import__("torch")
    qkv, dout = _attn_inputs(nseq, seq, heads, nseq * seq + heads)
    D = heads * 64
    R = nseq * seq
    dqkv_in = dev(qkv, "bf16")
    o = t.empty((R, D), dtype=t.bfloat16, device="cuda")
    lse = t.empty((R, heads), dtype=t.float32, device="cuda")
    lib = b.lib()
    assert lib.gpipe_op_attention_fwd(nseq, seq, heads, dqkv_in.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      stream()) == 0
    q, k, v = _split(qkv, nseq, seq, heads)
    ref_o, p = om.causal_attention(q, k, v)
    sync()
    go = host(o).reshape(nseq, seq, heads, 64).transpose(0, 2, 1, 3)
    assert rel(go, ref_o) <= 1e-2
    assert_elementwise(go.reshape(-1, 64), ref_o.reshape(-1, 64), 0.05, 0.05, 1e-4, "attention output")
    s = (q @ np.swapaxes(k, -1, -2)) / 8.0
    s = np.where(np.triu(np.ones((seq, seq), bool), 1), -np.inf, s)
    m = s.max(axis=-1, keepdims=True)
    ref_lse = (m + np.log(np.exp(s - m).sum(axis=-1, keepdims=True)))[..., 0]  # [n, h, s]
    assert np.max(np.abs(host(lse).reshape(nseq, seq, heads).transpose(0, 2, 1) - ref_lse)) <= 1e-3
    # backward from the kernel's own forward output (what the step does)
    dvec = t.empty((R, heads), dtype=t.float32, device="cuda")
    dqkv = t.empty((R, 3 * D), dtype=t.bfloat16, device="cuda")
    assert lib.gpipe_op_attention_bwd(nseq, seq, heads, dqkv_in.data_ptr(), o.data_ptr(),
                                      dev(dout, "bf16").data_ptr(), lse.data_ptr(), dvec.data_ptr(),
                                      dqkv.data_ptr(), stream()) == 0
    do = dout.reshape(nseq, seq, heads, 64).transpose(0, 2, 1, 3)
    rq, rk, rv = om.causal_attention_backward(do, q, k, v, p)
    sync()
    gq, gk, gv = _split(host(dqkv), nseq, seq, heads)
    for got, want, name in ((gq, rq, "dQ"), (gk, rk, "dK"), (gv, rv, "dV")):
        assert rel(got, want) <= 2e-2, name
        assert_elementwise(got.reshape(-1, 64), want.reshape(-1, 64), 0.1, 0.1, 1e-3, name)
    # D = rowsum(dO o O) of the kernel's own (bf16) output
    od = host(o).reshape(nseq, seq, heads, 64) * dout.reshape(nseq, seq, heads, 64)
    assert rel(host(dvec), od.sum(axis=-1).reshape(R, heads)) <= 1e-5


def test_attention_bwd_deterministic(b):
    t = __import__("torch")
    nseq, seq, heads = 2, 256, 2
    qkv, dout = _attn_inputs(nseq, seq, heads, 4)
    D, R = heads * 64, nseq * seq
    lib = b.lib()
    x = dev(qkv, "bf16")
    o = t.empty((R, D), dtype=t.bfloat16, device="cuda")
    lse = t.empty((R, heads), dtype=t.float32, device="cuda")
    lib.gpipe_op_attention_fwd(nseq, seq, heads, x.data_ptr(), o.data_ptr(), lse.data_ptr(), stream())
    outs = []
    for _ in range(2):
        dvec = t.empty((R, heads), dtype=t.float32, device="cuda")
        dq = t.empty((R, 3 * D), dtype=t.bfloat16, device="cuda")
        lib.gpipe_op_attention_bwd(nseq, seq, heads, x.data_ptr(), o.data_ptr(), dev(dout, "bf16").data_ptr(),
                                   lse.data_ptr(), dvec.data_ptr(), dq.data_ptr(), stream())
        outs.append(dq.view(t.int16).cpu().numpy())
    sync()
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("rows,vocab,seq,row0", [(130, 1000, 64, 0), (64, 32000, 64, 64), (37, 4096, 16, 5)])
def test_cross_entropy(b, rows, vocab, seq, row0):
    t = __import__("torch")
    rng = np.random.default_rng(rows + vocab)
    n_tok = row0 + rows + seq
    n_tok += (-n_tok) % seq
    tokens = rng.integers(0, vocab, size=n_tok).astype(np.int32)
    z = (rng.standard_normal((rows, vocab)) * 3).astype(np.float32)
    inv = 1.0 / 1234.0
    dz_buf = dev(z)
    loss = t.empty(rows, dtype=t.float32, device="cuda")
    assert b.lib().gpipe_op_cross_entropy(rows, vocab, seq, dev(tokens).data_ptr(), row0, inv, dz_buf.data_ptr(),
                                          loss.data_ptr(), 1, stream()) == 0
    sync()
    # expected from the oracle's cross-entropy, one row at a time
    want_loss = np.zeros(rows)
    want_dz = np.zeros((rows, vocab))
    for r in range(rows):
        gidx = row0 + r
        if gidx % seq == seq - 1:
            continue
        zz = z[r].astype(np.float64)[None, None, :].repeat(2, axis=1)
        tok = np.array([[0, tokens[gidx + 1]]])
        l, dz, per = om.next_token_ce(zz, tok, 1.0)
        want_loss[r] = per[0, 0] * inv
        want_dz[r] = dz[0, 0] * inv
    assert rel(host(loss), want_loss) <= 1e-5
    got_dz = dz_buf.view(t.bfloat16).view(rows, 2 * vocab)[:, :vocab].float().cpu().numpy()
    assert rel(got_dz, want_dz) <= 8e-3


@pytest.mark.parametrize("rows,vocab,seq,row0", [(130, 1000, 64, 0), (64, 32000, 64, 64)])
def test_cross_entropy_logit_clipping(b, rows, vocab, seq, row0):
    """Clipped cross-entropy against the oracle's clipped loss on the same fp32
    logits: the pass/zero decision is taken on identical values, so the
    zero pattern of dz matches exactly; clip 0 is the unclipped op, bit for
    bit; a negative clip is rejected."""
    t = __import__("torch")
    rng = np.random.default_rng(rows + vocab + 1)
    n_tok = row0 + rows + seq
    n_tok += (-n_tok) % seq
    tokens = rng.integers(0, vocab, size=n_tok).astype(np.int32)
    z = (rng.standard_normal((rows, vocab)) * 3).astype(np.float32)
    inv = 1.0 / 1234.0
    clip_milli = 3000
    c = float(np.float32(clip_milli / 1000.0))
    outs = {}
    for cc in (c, 0.0):
        dz_buf = dev(z)
        loss = t.empty(rows, dtype=t.float32, device="cuda")
        assert b.lib().gpipe_op_cross_entropy_clip(rows, vocab, seq, dev(tokens).data_ptr(), row0, inv, cc,
                                                   dz_buf.data_ptr(), loss.data_ptr(), 1, stream()) == 0
        sync()
        outs[cc] = (host(loss), dz_buf.view(t.bfloat16).view(rows, 2 * vocab)[:, :vocab].float().cpu().numpy())
    dz_plain = dev(z)
    loss_plain = t.empty(rows, dtype=t.float32, device="cuda")
    assert b.lib().gpipe_op_cross_entropy(rows, vocab, seq, dev(tokens).data_ptr(), row0, inv, dz_plain.data_ptr(),
                                          loss_plain.data_ptr(), 1, stream()) == 0
    sync()
    assert np.array_equal(outs[0.0][0], host(loss_plain))
    assert np.array_equal(outs[0.0][1], dz_plain.view(t.bfloat16).view(rows, 2 * vocab)[:, :vocab].float().cpu().numpy())
    want_loss = np.zeros(rows)
    want_dz = np.zeros((rows, vocab))
    for r in range(rows):
        gidx = row0 + r
        if gidx % seq == seq - 1:
            continue
        zz = z[r].astype(np.float64)[None, None, :].repeat(2, axis=1)
        tok = np.array([[0, tokens[gidx + 1]]])
        _, dz, per = om.next_token_ce(zz, tok, 1.0, clip=c)
        want_loss[r] = per[0, 0] * inv
        want_dz[r] = dz[0, 0] * inv
    got_loss, got_dz = outs[c]
    assert rel(got_loss, want_loss) <= 1e-5
    assert rel(got_dz, want_dz) <= 8e-3
    assert np.array_equal(got_dz == 0, want_dz == 0)
    assert 0.2 < np.mean(np.abs(z) > c) < 0.5
    assert b.lib().gpipe_op_cross_entropy_clip(rows, vocab, seq, dev(tokens).data_ptr(), row0, inv, -1.0,
                                               dev(z).data_ptr(), t.empty(rows, device="cuda").data_ptr(), 1,
                                               stream()) != 0


def test_mse(b):
    t = __import__("torch")
    rng = np.random.default_rng(3)
    y = rng.standard_normal((50, 64)).astype(np.float32)
    tt = rng.standard_normal((50, 64)).astype(np.float32)
    loss = t.empty(50, dtype=t.float32, device="cuda")
    dy = t.empty((50, 64), dtype=t.float32, device="cuda")
    inv = 1.0 / (50 * 64)
    assert b.lib().gpipe_op_mse(50, 64, dev(y).data_ptr(), dev(tt).data_ptr(), inv, loss.data_ptr(), dy.data_ptr(),
                                stream()) == 0
    sync()
    _, gref = om.mse_loss(y.astype(np.float64), tt.astype(np.float64), 50 * 64)
    assert rel(host(loss), ((y.astype(np.float64) - tt) ** 2).sum(axis=1) * inv) <= 1e-6
    assert rel(host(dy), gref) <= 1e-6


def test_embedding_fwd_bwd(b):
    t = __import__("torch")
    rng = np.random.default_rng(8)
    V, d, rows = 1000, 256, 777
    tokens = rng.integers(0, V, size=rows).astype(np.int32)
    tokens[:50] = 7  # many repeats of one row
    E = bf16_round(rng.standard_normal((V, d)))
    x = t.empty((rows, d), dtype=t.bfloat16, device="cuda")
    dtok = dev(tokens)
    assert b.lib().gpipe_op_embedding_fwd(rows, d, V, dtok.data_ptr(), dev(E, "bf16").data_ptr(), x.data_ptr(),
                                          stream()) == 0
    sync()
    assert np.array_equal(host(x), E[tokens])
    dx = bf16_round(rng.standard_normal((rows, d)))
    dE0 = rng.standard_normal((V, d)).astype(np.float32)
    ddE = dev(dE0)
    assert b.lib().gpipe_op_embedding_bwd(rows, d, V, dtok.data_ptr(), dev(dx, "bf16").data_ptr(), ddE.data_ptr(),
                                          stream()) == 0
    sync()
    want = dE0.astype(np.float64)
    np.add.at(want, tokens, dx)
    assert rel(host(ddE), want) <= 1e-6


def test_rmsprop_and_bf16_copy(b):
    t = __import__("torch")
    rng = np.random.default_rng(12)
    n = 100003  # ragged tail after the 4-wide vector body
    w = rng.standard_normal(n).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    g[::97] = 0.0
    v = (np.abs(rng.standard_normal(n)) * 1e-4).astype(np.float32)
    dw, dg, dv = dev(w), dev(g), dev(v)
    wb = t.empty(n, dtype=t.bfloat16, device="cuda")
    assert b.lib().gpipe_op_rmsprop(n, dw.data_ptr(), dg.data_ptr(), dv.data_ptr(), wb.data_ptr(), 1e-3, 0.9, 1e-8,
                                    1, stream()) == 0
    sync()
    new_p, new_v = om.rmsprop({"a": w}, {"a": g.astype(np.float64)}, {"a": v}, 1e-3, 0.9, 1e-8)
    # fp32 master: within one fp32 ulp of w plus the fp32 rounding of the
    # update term itself (about 2^-24 relative, taken with margin as 1e-6)
    ulp = np.spacing(np.abs(new_p["a"]).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(host(dw) - new_p["a"]) <= ulp + 1e-6 * np.abs(new_p["a"] - w))
    assert rel(host(dv), new_v["a"]) <= 1e-6
    assert not np.any(host(dg))
    # bf16 copy is the round-to-nearest-even of the updated fp32 master
    assert np.array_equal(wb.float().cpu().numpy(), bf16_round(host(dw)).astype(np.float32))


def test_cast_bf16(b):
    t = __import__("torch")
    x = np.random.default_rng(1).standard_normal(4099).astype(np.float32)
    out = t.empty(4099, dtype=t.bfloat16, device="cuda")
    assert b.lib().gpipe_op_cast_bf16(4099, dev(x).data_ptr(), out.data_ptr(), stream()) == 0
    sync()
    assert np.array_equal(out.float().cpu().numpy(), bf16_round(x).astype(np.float32))


def test_gelu_arithmetic_within_its_error_bound(b):
    """The epilogues' GELU and GELU' (erf by Abramowitz & Stegun 7.1.26, whose
    |error| <= 1.5e-7) against the exact-erf definitions in fp64: Phi is off by
    at most 0.75e-7 from the formula plus ~2e-7 from evaluating it in fp32, so
    |GELU error| <= 3e-7 |z| (+ rounding of the result) and |GELU' error| <=
    4e-7 (+ rounding).  CUDA's erff is itself ~2 ulp (~2.4e-7 near 1)."""
    from scipy.special import erf
    t = __import__("torch")
    rng = np.random.default_rng(11)
    z = np.concatenate([np.linspace(-12, 12, 200001), rng.standard_normal(100000) * 3]).astype(np.float32)
    zd = dev(z)
    y = t.empty_like(zd)
    dy = t.empty_like(zd)
    assert b.lib().gpipe_op_gelu(z.size, zd.data_ptr(), y.data_ptr(), dy.data_ptr(), stream()) == 0
    sync()
    z64 = z.astype(np.float64)
    cdf = 0.5 * (1 + erf(z64 / np.sqrt(2)))
    ref = z64 * cdf
    dref = cdf + z64 * np.exp(-0.5 * z64 * z64) / np.sqrt(2 * np.pi)
    err = np.abs(host(y) - ref)
    derr = np.abs(host(dy) - dref)
    assert np.all(err <= 3e-7 * np.abs(z64) + 2e-7 * np.abs(ref)), err.max()
    assert np.all(derr <= 4e-7 + 2e-7 * np.abs(dref)), derr.max()
    # the sign of the tiny negative tail is kept (no cancellation in 1 + erf)
    neg = z64 < -3
    assert np.all(host(y)[neg] <= 0)


@pytest.mark.parametrize("ak,bk,epi,shape", [(1, 1, 1, (1024, 2048, 512)), (1, 1, 0, (512, 1536, 512)),
                                             (1, 0, 2, (512, 2048, 512)), (0, 0, 3, (2048, 512, 512)),
                                             (0, 0, 3, (1152, 1088, 256)), (1, 1, 5, (2048, 1024, 1024)),
                                             (1, 1, 5, (1000, 1000, 264)), (1, 0, 0, (1024, 1280, 2048))])
def test_gemm_bits_do_not_depend_on_sm_share(b, ak, bk, epi, shape):
    """The step sizes each GEMM's grid by its share of the SMs, which changes
    the kernel (one tile per CTA, 64/128 wide, or persistent 128/256 wide) but
    must not change a bit of the result."""
    t = __import__("torch")
    M, N, K = shape
    rng = np.random.default_rng(M + N + K + epi)
    A = dev(bf16_round(rng.standard_normal((M, K) if ak else (K, M))), "bf16")
    B = dev(bf16_round(rng.standard_normal((N, K) if bk else (K, N)) / np.sqrt(K)), "bf16")
    bias = dev(rng.standard_normal(N if epi != 3 else M).astype(np.float32))
    aux = dev(bf16_round(rng.standard_normal((M, N))), "bf16") if epi == 2 else None
    resid = dev(rng.standard_normal((M, N)).astype(np.float32)) if epi == 5 else None
    outs = []
    for share in (0, 16, 40, 7):
        assert b.lib().gpipe_op_gemm_set_sm_share(share) == 0
        C = t.zeros((M, N), device="cuda", dtype=t.float32 if epi in (3, 5) else t.bfloat16)
        C2 = t.zeros((M, N), device="cuda", dtype=t.bfloat16) if epi == 1 else None
        db = bias.clone() if epi == 3 else bias
        rc = b.lib().gpipe_op_gemm(1, M, N, K, A.data_ptr(), K if ak else M, ak, B.data_ptr(), K if bk else N, bk,
                                   epi, C.data_ptr(), N, db.data_ptr(),
                                   resid.data_ptr() if resid is not None else None, N if resid is not None else 0,
                                   C2.data_ptr() if C2 is not None else None,
                                   aux.data_ptr() if aux is not None else None, N if aux is not None else 0,
                                   stream())
        assert rc == 0, b.lib().gpipe_last_error(None)
        sync()
        outs.append([C.cpu(), C2.cpu() if C2 is not None else None, db.cpu() if epi == 3 else None])
    assert b.lib().gpipe_op_gemm_set_sm_share(0) == 0
    for o in outs[1:]:
        for x, y in zip(o, outs[0]):
            assert (x is None and y is None) or t.equal(x, y)


def _device_error(b, clear=1):
    import ctypes
    f = ctypes.c_int(-1)
    assert b.lib().gpipe_op_device_error(ctypes.byref(f), clear, stream()) == 0
    return f.value


def test_bounded_wait_gives_up_and_reports_without_a_fault(b):
    """Failure detection without a GPU fault: a kernel's bounded wait on an
    mbarrier that nothing completes gives up after the limit (2 s), sets the
    device error word (code 6) and returns; the context keeps working."""
    import time
    t = __import__("torch")
    _device_error(b)  # start clean
    t0 = time.perf_counter()
    assert b.lib().gpipe_op_wait_probe(stream()) == 0
    assert _device_error(b) == 6
    assert 1.5 < time.perf_counter() - t0 < 60
    # the same context still computes: a GEMM afterwards is right and flags nothing
    rng = np.random.default_rng(3)
    A = bf16_round(rng.standard_normal((256, 128)))
    B = bf16_round(rng.standard_normal((192, 128)))
    C = t.zeros((256, 192), dtype=t.bfloat16, device="cuda")
    assert b.lib().gpipe_op_gemm(1, 256, 192, 128, dev(A, "bf16").data_ptr(), 128, 1, dev(B, "bf16").data_ptr(), 128,
                                 1, 0, C.data_ptr(), 192, None, None, 0, None, None, 0, stream()) == 0
    sync()
    assert rel(host(C), A @ B.T) <= 1e-2
    assert _device_error(b) == 0


def test_invalid_token_is_flagged_not_read(b):
    """A next-token target outside [0, vocab) is skipped (no out-of-range read)
    and reported through the device error word (code 5)."""
    t = __import__("torch")
    rows, vocab, seq = 64, 1000, 64
    rng = np.random.default_rng(5)
    tokens = rng.integers(0, vocab, size=rows).astype(np.int32)
    tokens[10] = vocab + 3
    z = dev((rng.standard_normal((rows, vocab)) * 3).astype(np.float32))
    loss = t.empty(rows, dtype=t.float32, device="cuda")
    _device_error(b)
    assert b.lib().gpipe_op_cross_entropy(rows, vocab, seq, dev(tokens).data_ptr(), 0, 1.0, z.data_ptr(),
                                          loss.data_ptr(), 1, stream()) == 0
    sync()
    assert _device_error(b) == 5
    got = host(loss)
    assert np.all(np.isfinite(got)) and got[9] == 0.0  # row 9's target was token 10
