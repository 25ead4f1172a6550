"""GPU parity of the block-scaled FP8 GEMM (Fprop / Dgrad / Wgrad) against the FP64 oracle.

Operand codes and scales are produced by the oracle's quantizers from seeded BF16 inputs
and copied to the device, so the GEMM kernel is checked on its own; the end-to-end tests
quantize on the GPU and compare with the oracle run end to end on the same BF16 inputs.
Bound per element: |gpu - ref| <= 2^-7 |ref| + 1e-6 sum_k |a_k b_k|.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_gemm_close, bf16_bits, np_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mpq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_quant_b300 as m
    return m


@pytest.fixture(params=[True, False], ids=["sm_pair", "single_sm"])
def tiles(request, mpq):
    """Run the test with 256x256 tiles on SM pairs and with 128x256 tiles on single SMs."""
    mpq.mpq_set_gemm_cta_pair(2 if request.param else 0)
    yield request.param
    mpq.mpq_set_gemm_cta_pair(1)


def _bf16(shape, std, seed, outliers=0.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * std
    if outliers:
        cols = torch.randperm(shape[1], generator=g)[: max(1, int(outliers * shape[1]))]
        x[:, cols] *= 50
    return x.to(torch.bfloat16)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _out_host(C):
    return C.float().cpu().numpy().astype(np.float64)


# --------------------------------------------------------------------- Fprop

@pytest.mark.parametrize("M,N,K", [(300, 512, 1024), (128, 256, 128), (1, 256, 256), (77, 384, 640),
                                   (129, 128, 8192)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_fprop_oracle_operands(mpq, tiles, M, N, K, out):
    a = _bf16((M, K), 1.0, M * 7 + K, outliers=0.01)
    w = _bf16((N, K), 0.02, N * 13 + K)
    qa, sa = oracle.quant_tile_1x128(bf16_bits(a))
    qb, _, sb = oracle.quant_block_128x128(bf16_bits(w))
    od = mpq.OUT_FP32 if out == "fp32" else mpq.OUT_BF16
    C = mpq.fp8_gemm_blockscaled(mpq.FPROP, _dev(qa), _dev(sa), _dev(qb), _dev(sb), out_dtype=od)
    ref, absref = oracle.gemm_ref(oracle.FPROP, qa, sa, qb, sb)
    assert_gemm_close(_out_host(C), ref, absref, f"fprop {M}x{N}x{K} {out}")


def test_fprop_small_integers_exact(mpq, tiles):
    """Codes of small integers with unit scales: every partial and sum is an exact
    integer below 2^24, so the FP32 output must equal the integer matmul exactly."""
    g = np.random.default_rng(3)
    vals = np.array([-4, -3, -2, -1, 0, 1, 2, 3, 4], np.float32)
    M, N, K = 200, 256, 2048
    ai = g.choice(vals, size=(M, K)); bi = g.choice(vals, size=(N, K))
    enc = lambda v: torch.tensor(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    qa, qb = enc(ai), enc(bi)
    sa = np.ones((K // 128, M), np.float32); sb = np.ones((N // 128, K // 128), np.float32)
    C = mpq.fp8_gemm_blockscaled(mpq.FPROP, _dev(qa), _dev(sa), _dev(qb), _dev(sb), out_dtype=mpq.OUT_FP32)
    exact = (ai.astype(np.int64) @ bi.astype(np.int64).T).astype(np.float64)
    np.testing.assert_array_equal(_out_host(C), exact)


def test_fprop_tiny_config_end_to_end(mpq):
    """256x512 activations (1% outlier columns x50) and 256x512 weight: GPU quantize +
    GEMM against the oracle run from the same BF16 inputs."""
    d = workloads.tiny_fprop()
    A, W = d["A"].cuda(), d["W"].cuda()
    qa, sa, _, _ = mpq.fp8_quant_tile_1x128(A)
    qb, _, sb = mpq.fp8_quant_block_128x128(W)
    C = mpq.fp8_gemm_blockscaled(mpq.FPROP, qa, sa, qb, sb)
    oqa, osa = oracle.quant_tile_1x128(bf16_bits(d["A"]))
    oqb, _, osb = oracle.quant_block_128x128(bf16_bits(d["W"]))
    ref, absref = oracle.gemm_ref(oracle.FPROP, oqa, osa, oqb, osb)
    assert_gemm_close(_out_host(C), ref, absref, "tiny fprop")


# --------------------------------------------------------------------- Dgrad

@pytest.mark.parametrize("T,Nout,Kin", [(256, 512, 384), (200, 256, 256)])
def test_dgrad_pow2(mpq, tiles, T, Nout, Kin):
    """dX[T, Kin] = dY[T, Nout] . W_lin[Nout, Kin]: A = dY (1x128, power-of-2 scales),
    B = transposed weight codes [Kin, Nout] with the weight's block scales."""
    g = torch.Generator().manual_seed(T)
    dy = workloads.student_t3((T, Nout), 1e-3, g, "cpu")
    w = _bf16((Nout, Kin), 0.02, Kin)
    qa, sa = oracle.quant_tile_1x128(bf16_bits(dy), pow2=True)
    _, qbT, sw = oracle.quant_block_128x128(bf16_bits(w), transposed=True)
    C = mpq.fp8_gemm_blockscaled(mpq.DGRAD, _dev(qa), _dev(sa), _dev(qbT), _dev(sw), out_dtype=mpq.OUT_FP32)
    ref, absref = oracle.gemm_ref(oracle.DGRAD, qa, sa, qbT, sw)
    assert_gemm_close(_out_host(C), ref, absref, "dgrad")


# --------------------------------------------------------------------- Wgrad

@pytest.mark.parametrize("T,Kin,Nout", [(512, 384, 256), (256, 128, 512)])
def test_wgrad(mpq, tiles, T, Kin, Nout):
    """dW[Kin, Nout] = X^T dY: both operands quantized in 128x1 tiles along tokens."""
    g = torch.Generator().manual_seed(T + Kin)
    x = _bf16((T, Kin), 1.0, T)
    dy = workloads.student_t3((T, Nout), 1e-3, g, "cpu")
    qaT, saT = oracle.quant_tile_128x1(bf16_bits(x))
    qbT, sbT = oracle.quant_tile_128x1(bf16_bits(dy), pow2=True)
    C = mpq.fp8_gemm_blockscaled(mpq.WGRAD, _dev(qaT), _dev(saT), _dev(qbT), _dev(sbT), out_dtype=mpq.OUT_FP32)
    ref, absref = oracle.gemm_ref(oracle.WGRAD, qaT, saT, qbT, sbT)
    assert_gemm_close(_out_host(C), ref, absref, "wgrad")


@pytest.mark.parametrize("op", ["fprop", "wgrad"])
def test_pair_and_single_tiles_agree_bit_for_bit(mpq, op):
    """2-SM pair tiles (M = 256 MMAs over two SMs) and single-SM tiles (M = 128) give the
    same FP32 results, bit for bit."""
    g = torch.Generator().manual_seed(17)
    if op == "fprop":
        a = _bf16((300, 640), 1.0, 5)
        w = _bf16((384, 640), 0.02, 6)
        qa, sa = oracle.quant_tile_1x128(bf16_bits(a))
        qb, _, sb = oracle.quant_block_128x128(bf16_bits(w))
        args = (mpq.FPROP, _dev(qa), _dev(sa), _dev(qb), _dev(sb))
    else:
        x = _bf16((512, 384), 1.0, 7)
        dy = workloads.student_t3((512, 256), 1e-3, g, "cpu")
        qaT, saT = oracle.quant_tile_128x1(bf16_bits(x))
        qbT, sbT = oracle.quant_tile_128x1(bf16_bits(dy), pow2=True)
        args = (mpq.WGRAD, _dev(qaT), _dev(saT), _dev(qbT), _dev(sbT))
    outs = []
    mpq.mpq_set_gemm_stream_k(0)
    for mode in (2, 0):
        mpq.mpq_set_gemm_cta_pair(mode)
        outs.append(mpq.fp8_gemm_blockscaled(*args, out_dtype=mpq.OUT_FP32))
    mpq.mpq_set_gemm_cta_pair(1)
    mpq.mpq_set_gemm_stream_k(1)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


# ------------------------------------------------------------------- stream-K

@pytest.mark.parametrize("op,M", [("fprop", 2560), ("wgrad", 2560), ("fprop", 2600)])
def test_stream_k(mpq, tiles, op, M):
    """Stream-K forced on M x 2048 outputs with K = 1280 (M = 2560: 80 pair tiles over 74 SM
    pairs, 160 single-SM tiles over 148 SMs, so nearly every tile is shared by two units;
    M = 2600 adds a ragged last row of tiles).  Sampled
    outputs meet the oracle bound; every output is within FP32 rounding of the data-parallel
    schedule's (a dropped or misplaced partial would not be); two runs agree bit for bit."""
    N, K = 2048, 1280                  # M = 2600: the last row tiles are ragged
    if op == "fprop":
        a = _bf16((M, K), 1.0, 21, outliers=0.01)
        w = _bf16((N, K), 0.02, 22)
        qa, sa = oracle.quant_tile_1x128(bf16_bits(a))
        qb, _, sb = oracle.quant_block_128x128(bf16_bits(w))
        o = oracle.FPROP
        args = (mpq.FPROP, _dev(qa), _dev(sa), _dev(qb), _dev(sb))
    else:
        g = torch.Generator().manual_seed(23)
        x = _bf16((K, M), 1.0, 24)                           # tokens x input features
        dy = workloads.student_t3((K, N), 1e-3, g, "cpu")    # tokens x output features
        qa, sa = oracle.quant_tile_128x1(bf16_bits(x))
        qb, sb = oracle.quant_tile_128x1(bf16_bits(dy), pow2=True)
        o = oracle.WGRAD
        args = (mpq.WGRAD, _dev(qa), _dev(sa), _dev(qb), _dev(sb))
    try:
        mpq.mpq_set_gemm_stream_k(0)
        dp = mpq.fp8_gemm_blockscaled(*args, out_dtype=mpq.OUT_FP32)
        mpq.mpq_set_gemm_stream_k(2)
        sk1 = mpq.fp8_gemm_blockscaled(*args, out_dtype=mpq.OUT_FP32)
        sk2 = mpq.fp8_gemm_blockscaled(*args, out_dtype=mpq.OUT_FP32)
        torch.cuda.synchronize()
        st, where = mpq.mpq_check_device_status()
        assert st == 0, (st, where)
    finally:
        mpq.mpq_set_gemm_stream_k(1)
    assert torch.equal(sk1, sk2)
    # every output: the two schedules sum the same slices in two orders (FP32 roundings only)
    d = dp.double()
    assert float((sk1.double() - d).abs().max()) <= 1e-5 * float(d.abs().max())
    rng = np.random.default_rng(25)
    ms = np.unique(np.concatenate([rng.integers(0, M, 40), [0, 255, 256, M - 1]])).astype(np.int64)
    ns = np.unique(np.concatenate([rng.integers(0, N, 40), [0, 255, 256, N - 1]])).astype(np.int64)
    mm, nn = np.meshgrid(ms, ns, indexing="ij")
    ref, absref = oracle.gemm_ref_at(o, qa, sa, qb, sb, mm.ravel(), nn.ravel())
    got = sk1.cpu().numpy().astype(np.float64)[mm.ravel(), nn.ravel()]
    assert_gemm_close(got, ref, absref, f"stream-K {op}")


# ------------------------------------------------------------ full-size samples

def _sample_pairs(M, N, ncols_blocks, rng, rows=48):
    ms = np.unique(np.concatenate([rng.integers(0, M, rows), [0, 127, 128, M - 1]]))
    nblocks = np.unique(np.concatenate([rng.integers(0, N // 128, ncols_blocks), [0, N // 128 - 1]]))
    return ms, nblocks


def test_dense_fprop_full_size_sampled(mpq):
    """4096 x 7168 . 7168 x 18432 on the GPU; the oracle recomputes sampled rows (incl.
    tile boundaries) for sampled 128-column blocks from the same BF16 inputs."""
    d = workloads.dense_fprop(device="cuda")
    A, W = d["A"], d["W"]
    qa, sa, _, _ = mpq.fp8_quant_tile_1x128(A)
    qb, _, sb = mpq.fp8_quant_block_128x128(W)
    C = mpq.fp8_gemm_blockscaled(mpq.FPROP, qa, sa, qb, sb)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    M, N = A.shape[0], W.shape[0]
    ms, nbs = _sample_pairs(M, N, 4, rng)
    oqa, osa = oracle.quant_tile_1x128(bf16_bits(A[torch.from_numpy(ms).cuda()]))
    for nb in nbs:
        oqb, _, osb = oracle.quant_block_128x128(bf16_bits(W[nb * 128:(nb + 1) * 128]))
        ref, absref = oracle.gemm_ref(oracle.FPROP, oqa, osa, oqb, osb)
        got = _out_host(C[torch.from_numpy(ms).cuda(), nb * 128:(nb + 1) * 128])
        assert_gemm_close(got, ref, absref, f"dense fprop block {nb}")


def test_backward_pair_full_size_sampled(mpq):
    """dY 8192 x 2048 (pow2), X 8192 x 7168, W_lin 2048 x 7168: Dgrad (K = 2048) and
    Wgrad (K = 8192 tokens) on the GPU, sampled outputs against the oracle."""
    d = workloads.backward_pair(device="cuda")
    dY, X, W = d["dY"], d["X"], d["W"]
    qdy, sdy, qdyT, sdyT = mpq.fp8_quant_tile_1x128(dY, pow2=True, transposed=True)
    _, _, qxT, sxT = mpq.fp8_quant_tile_1x128(X, rows_out=False, transposed=True)
    _, qwT, sw = mpq.fp8_quant_block_128x128(W, transposed=True)
    dX = mpq.fp8_gemm_blockscaled(mpq.DGRAD, qdy, sdy, qwT, sw, out_dtype=mpq.OUT_FP32)
    dW = mpq.fp8_gemm_blockscaled(mpq.WGRAD, qxT, sxT, qdyT, sdyT, out_dtype=mpq.OUT_FP32)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    # Dgrad: sampled token rows, two column blocks of dX
    ms = np.unique(np.concatenate([rng.integers(0, dY.shape[0], 32), [0, dY.shape[0] - 1]]))
    oq, os_ = oracle.quant_tile_1x128(bf16_bits(dY[torch.from_numpy(ms).cuda()]), pow2=True)
    _, oqwT, osw = oracle.quant_block_128x128(bf16_bits(W), transposed=True)
    for kb in (0, W.shape[1] // 128 - 1):
        cols = slice(kb * 128, (kb + 1) * 128)
        ref, absref = oracle.gemm_ref(oracle.DGRAD, oq, os_, np.ascontiguousarray(oqwT[cols]),
                                      np.ascontiguousarray(osw[:, kb:kb + 1]))
        got = _out_host(dX[torch.from_numpy(ms).cuda(), cols])
        assert_gemm_close(got, ref, absref, f"dgrad cols {kb}")
    # Wgrad: sampled rows of dW (input features) x all 2048 output columns
    feat = np.unique(np.concatenate([rng.integers(0, X.shape[1], 24), [0, X.shape[1] - 1]]))
    xs = X[:, torch.from_numpy(feat).cuda()].contiguous()
    # 128x1 groups of the sampled columns only need those columns
    oqxT, osxT = oracle.quant_tile_128x1(bf16_bits(xs))
    oqdT, osdT = oracle.quant_tile_128x1(bf16_bits(dY), pow2=True)
    ref, absref = oracle.gemm_ref(oracle.WGRAD, oqxT, osxT, oqdT, osdT)
    got = _out_host(dW[torch.from_numpy(feat).cuda()])
    assert_gemm_close(got, ref, absref, "wgrad sampled rows")


# --------------------------------------------------------------- validation

def test_gemm_validation(mpq):
    A = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    sA = torch.ones((2, 128), device="cuda")
    B = torch.zeros((200, 256), dtype=torch.uint8, device="cuda")  # N % 128 != 0
    sB = torch.ones((2, 2), device="cuda")
    with pytest.raises(mpq.MPQError) as e:
        mpq.fp8_gemm_blockscaled(mpq.FPROP, A, sA, B, sB)
    assert e.value.status == 2
    with pytest.raises(mpq.MPQError) as e:
        mpq.fp8_gemm_blockscaled(7, A, sA, A, sB)
    assert e.value.status == 4


def test_bounded_wait_reports_timeout_and_context_survives(mpq):
    """A device wait that nothing completes gives up after its limit, records a timeout
    in the status word, and later launches still run correctly."""
    assert mpq.mpq_check_device_status()[0] == 0
    mpq.mpq_selftest_wait_timeout(2_000_000)  # 2 ms
    st, where = mpq.mpq_check_device_status()
    assert st == 6 and where == 0x7F01
    assert mpq.mpq_check_device_status()[0] == 0  # cleared on read
    test_fprop_small_integers_exact(mpq, True)
