"""GPU parity of fp8_gemm_mx_pow2, the block-scaled FP8 GEMM for power-of-2 scales whose
scales the tensor cores apply (microscaling MMA with UE8M0 scale factors), against the FP64
oracle, for Fprop / Dgrad / Wgrad.

Operands are quantized by the oracle with power-of-2 scales on both sides; the bound per
element is the method's: |gpu - ref| <= 2^-7 |ref| + 1e-6 sum_k |a_k b_k|.  The software
promotion path (fp8_gemm_blockscaled) computes the same sum and is compared within the same
bound (the FP32 roundings differ in order, so the outputs need not be equal bit for bit).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_gemm_close, bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mpq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_quant_b300 as m
    return m


def _bf16(shape, std, seed, outliers=0.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * std
    if outliers:
        cols = torch.randperm(shape[1], generator=g)[: max(1, int(outliers * shape[1]))]
        x[:, cols] *= 50
    return x.to(torch.bfloat16)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _host(C):
    return C.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(300, 512, 1024), (256, 256, 128), (1, 256, 256), (77, 384, 640),
                                   (513, 768, 4096), (129, 128, 8192)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_mx_fprop_oracle_operands(mpq, M, N, K, out):
    a = _bf16((M, K), 1.0, M * 7 + K, outliers=0.01)
    w = _bf16((N, K), 0.02, N * 13 + K)
    qa, sa = oracle.quant_tile_1x128(bf16_bits(a), pow2=True)
    qb, _, sb = oracle.quant_block_128x128(bf16_bits(w), pow2=True)
    od = mpq.OUT_FP32 if out == "fp32" else mpq.OUT_BF16
    dqa, dsa, dqb, dsb = _dev(qa), _dev(sa), _dev(qb), _dev(sb)
    C = mpq.fp8_gemm_mx_pow2(mpq.FPROP, dqa, dsa, dqb, dsb, out_dtype=od)
    ref, absref = oracle.gemm_ref(oracle.FPROP, qa, sa, qb, sb)
    assert_gemm_close(_host(C), ref, absref, f"mx fprop {M}x{N}x{K} {out}")
    # the software promotion path on the same operands: the same sum within the same bound
    Cs = mpq.fp8_gemm_blockscaled(mpq.FPROP, dqa, dsa, dqb, dsb, out_dtype=od)
    assert_gemm_close(_host(Cs), ref, absref, f"software path {M}x{N}x{K} {out}")
    assert mpq.mpq_check_device_status() == (0, 0)


def test_mx_small_integers_exact(mpq):
    """Small-integer codes with power-of-2 scales per row, column and 128-K slice: every
    scaled product and partial sum is exactly representable, so the FP32 output must equal
    the exact sum."""
    g = np.random.default_rng(11)
    vals = np.array([-4, -3, -2, -1, 0, 1, 2, 3, 4], np.float32)
    M, N, K = 260, 512, 1024
    ai = g.choice(vals, size=(M, K)); bi = g.choice(vals, size=(N, K))
    enc = lambda v: torch.tensor(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    qa, qb = enc(ai), enc(bi)
    sa = (2.0 ** g.integers(-1, 2, size=(K // 128, M))).astype(np.float32)
    sb = (2.0 ** g.integers(-1, 2, size=(K // 128, N))).astype(np.float32)     # Wgrad layout [K/128][N]
    C = mpq.fp8_gemm_mx_pow2(mpq.WGRAD, _dev(qa), _dev(sa), _dev(qb), _dev(sb), out_dtype=mpq.OUT_FP32)
    exact = np.zeros((M, N))
    for kb in range(K // 128):
        sl = slice(kb * 128, kb * 128 + 128)
        exact += (ai[:, sl].astype(np.float64) @ bi[:, sl].astype(np.float64).T) * sa[kb][:, None] * sb[kb][None, :]
    np.testing.assert_array_equal(_host(C), exact)


@pytest.mark.parametrize("T,Nout,Kin", [(256, 512, 384), (200, 256, 256)])
def test_mx_dgrad(mpq, T, Nout, Kin):
    """dX = dY W_lin with dY (1x128) and the weight blocks both on power-of-2 scales; B is
    the transposed weight codes with the block scales seen as [K/128][N/128]."""
    g = torch.Generator().manual_seed(T)
    dy = workloads.student_t3((T, Nout), 1e-3, g, "cpu")
    w = _bf16((Nout, Kin), 0.02, Kin)
    qa, sa = oracle.quant_tile_1x128(bf16_bits(dy), pow2=True)
    _, qbT, sw = oracle.quant_block_128x128(bf16_bits(w), pow2=True, transposed=True)
    C = mpq.fp8_gemm_mx_pow2(mpq.DGRAD, _dev(qa), _dev(sa), _dev(qbT), _dev(sw), out_dtype=mpq.OUT_FP32)
    ref, absref = oracle.gemm_ref(oracle.DGRAD, qa, sa, qbT, sw)
    assert_gemm_close(_host(C), ref, absref, "mx dgrad")


@pytest.mark.parametrize("T,Kin,Nout", [(512, 384, 256), (256, 128, 512), (1024, 256, 384)])
def test_mx_wgrad(mpq, T, Kin, Nout):
    """dW = X^T dY with both operands quantized 128x1 along tokens, power-of-2 scales."""
    g = torch.Generator().manual_seed(T + Kin)
    x = _bf16((T, Kin), 1.0, T)
    dy = workloads.student_t3((T, Nout), 1e-3, g, "cpu")
    qxT, sxT = oracle.quant_tile_128x1(bf16_bits(x), pow2=True)
    qdT, sdT = oracle.quant_tile_128x1(bf16_bits(dy), pow2=True)
    C = mpq.fp8_gemm_mx_pow2(mpq.WGRAD, _dev(qxT), _dev(sxT), _dev(qdT), _dev(sdT), out_dtype=mpq.OUT_FP32)
    ref, absref = oracle.gemm_ref(oracle.WGRAD, qxT, sxT, qdT, sdT)
    assert_gemm_close(_host(C), ref, absref, "mx wgrad")


@pytest.mark.parametrize("op,M", [("fprop", 2560), ("wgrad", 2560), ("fprop", 2600), ("dgrad", 2560)])
def test_mx_stream_k(mpq, op, M):
    """Stream-K forced on M x 2048 outputs with K = 1280 (2560 rows: 80 pair tiles over 74
    SM pairs, so nearly every tile is split between two units, and the runs start and end
    inside groups of four slices; 2600 rows add a ragged last row of tiles).  Every output is
    within FP32 rounding of the data-parallel schedule's (head + tail instead of one
    accumulation: a dropped, doubled or misplaced partial would not be); two runs agree bit
    for bit; sampled outputs meet the oracle bound."""
    N, K = 2048, 1280
    g = torch.Generator().manual_seed(31)
    if op == "fprop":
        a = _bf16((M, K), 1.0, 32, outliers=0.01)
        w = _bf16((N, K), 0.02, 33)
        qa, sa = oracle.quant_tile_1x128(bf16_bits(a), pow2=True)
        qb, _, sb = oracle.quant_block_128x128(bf16_bits(w), pow2=True)
        o, mop = oracle.FPROP, mpq.FPROP
    elif op == "dgrad":   # dX [M, N] = dY [M, K] W_lin [K, N]: B = W_lin^T codes, [K/128][N/128] scales
        dy = workloads.student_t3((M, K), 1e-3, g, "cpu")
        w = _bf16((K, N), 0.02, 34)
        qa, sa = oracle.quant_tile_1x128(bf16_bits(dy), pow2=True)
        _, qb, sb = oracle.quant_block_128x128(bf16_bits(w), pow2=True, transposed=True)
        o, mop = oracle.DGRAD, mpq.DGRAD
    else:
        x = _bf16((K, M), 1.0, 35)                           # tokens x input features
        dy = workloads.student_t3((K, N), 1e-3, g, "cpu")    # tokens x output features
        qa, sa = oracle.quant_tile_128x1(bf16_bits(x), pow2=True)
        qb, sb = oracle.quant_tile_128x1(bf16_bits(dy), pow2=True)
        o, mop = oracle.WGRAD, mpq.WGRAD
    args = (mop, _dev(qa), _dev(sa), _dev(qb), _dev(sb))
    try:
        mpq.mpq_set_gemm_stream_k(0)
        dp = mpq.fp8_gemm_mx_pow2(*args, out_dtype=mpq.OUT_FP32)
        mpq.mpq_set_gemm_stream_k(2)
        sk1 = mpq.fp8_gemm_mx_pow2(*args, out_dtype=mpq.OUT_FP32)
        sk2 = mpq.fp8_gemm_mx_pow2(*args, out_dtype=mpq.OUT_FP32)
        torch.cuda.synchronize()
        st, where = mpq.mpq_check_device_status()
        assert st == 0, (st, where)
    finally:
        mpq.mpq_set_gemm_stream_k(1)
    assert torch.equal(sk1, sk2)
    d = dp.double()
    assert float((sk1.double() - d).abs().max()) <= 1e-5 * float(d.abs().max())
    rng = np.random.default_rng(36)
    ms = np.unique(np.concatenate([rng.integers(0, M, 40), [0, 255, 256, M - 1]])).astype(np.int64)
    ns = np.unique(np.concatenate([rng.integers(0, N, 40), [0, 255, 256, N - 1]])).astype(np.int64)
    mm, nn = np.meshgrid(ms, ns, indexing="ij")
    ref, absref = oracle.gemm_ref_at(o, qa, sa, qb, sb, mm.ravel(), nn.ravel())
    got = sk1.cpu().numpy().astype(np.float64)[mm.ravel(), nn.ravel()]
    assert_gemm_close(got, ref, absref, f"microscaling stream-K {op}")


def test_mx_full_size_fprop_sampled(mpq):
    """The dense Fprop shape (4096 x 18432 x 7168) quantized on the GPU with power-of-2
    scales on both operands: codes and scales checked against the oracle on sampled rows,
    outputs on sampled elements (every tile-boundary row and column among them)."""
    d = workloads.dense_fprop(device="cuda")
    A, W = d["A"], d["W"]
    qa, sa, _, _ = mpq.fp8_quant_tile_1x128(A, pow2=True)
    qb, _, sb = mpq.fp8_quant_block_128x128(W, pow2=True)
    C = mpq.fp8_gemm_mx_pow2(mpq.FPROP, qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert mpq.mpq_check_device_status() == (0, 0)
    rng = np.random.default_rng(5)
    M, N = C.shape
    rows = np.unique(np.concatenate([rng.integers(0, M, 24), [0, 255, 256, M - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, N, 24), [0, 255, 256, N - 1]]))
    oqa, osa = oracle.quant_tile_1x128(bf16_bits(A[torch.from_numpy(rows).cuda()]), pow2=True)
    assert np.array_equal(qa[torch.from_numpy(rows).cuda()].cpu().numpy(), oqa)
    assert np.array_equal(sa[:, torch.from_numpy(rows).cuda()].cpu().numpy(), osa)
    qb_h, sb_h = qb.cpu().numpy(), sb.cpu().numpy()
    ms, ns = np.meshgrid(np.arange(len(rows)), cols, indexing="ij")
    ref, absref = oracle.gemm_ref_at(oracle.FPROP, oqa, osa, qb_h, sb_h, ms.ravel(), ns.ravel())
    got = C.float()[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy().ravel()
    assert_gemm_close(got.astype(np.float64), ref, absref, "mx full-size fprop")


def test_mx_rejects_scales_that_are_not_powers_of_two(mpq):
    """A scale that is not a power of 2 is reported through the status word (the output of
    that call is not valid); the next call with valid scales is exact again."""
    M, N, K = 256, 256, 256
    a = _bf16((M, K), 1.0, 1)
    w = _bf16((N, K), 0.02, 2)
    qa, sa = oracle.quant_tile_1x128(bf16_bits(a), pow2=True)
    qb, _, sb = oracle.quant_block_128x128(bf16_bits(w), pow2=True)
    bad = sa.copy()
    bad[1, 17] *= 1.5
    mpq.fp8_gemm_mx_pow2(mpq.FPROP, _dev(qa), _dev(bad), _dev(qb), _dev(sb), out_dtype=mpq.OUT_FP32)
    st, where = mpq.mpq_check_device_status()
    assert st == 9 and where != 0
    C = mpq.fp8_gemm_mx_pow2(mpq.FPROP, _dev(qa), _dev(sa), _dev(qb), _dev(sb), out_dtype=mpq.OUT_FP32)
    ref, absref = oracle.gemm_ref(oracle.FPROP, qa, sa, qb, sb)
    assert_gemm_close(_host(C), ref, absref, "after a rejected call")
    assert mpq.mpq_check_device_status() == (0, 0)


def test_mx_validation_before_launch(mpq):
    q = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    s = torch.ones((2, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(mpq.MPQError) as ei:   # N not a multiple of 128
        mpq.fp8_gemm_mx_pow2(mpq.WGRAD, q, s, q[:200], s[:, :200])
    assert ei.value.status == 2
    with pytest.raises(mpq.MPQError) as ei:
        mpq.fp8_gemm_mx_pow2(7, q, s, q, s)
    assert ei.value.status == 4
