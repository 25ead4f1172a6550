"""GPU parity of fp8_grouped_gemm_swiglu_quant: the MoE up projection with SwiGLU and the
1x128 quantization of its result in the GEMM's epilogue.

Checked against (a) the two-step path on the GPU -- fp8_grouped_gemm_blockscaled with BF16
output, then fp8_swiglu_quant_1x128 -- bit for bit (codes, scales and the BF16 SwiGLU input);
(b) the oracle: the BF16 SwiGLU input within the GEMM bound of the FP64 grouped GEMM, and the
codes and scales bit-exact against the oracle's SwiGLU quantizer run on that same BF16 input.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._util import assert_gemm_close, bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mpq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_quant_b300 as m
    return m


@pytest.fixture(params=[0, 2], ids=["single_sm", "sm_pair"])
def tiles(request, mpq):
    mpq.mpq_set_gemm_cta_pair(request.param)
    yield request.param
    mpq.mpq_set_gemm_cta_pair(1)


def _problem(counts, lead, trail, W, K, seed, gate_scale=2.0):
    """Expert rows (BF16 ~ N(0,1)), per-expert gate+up weights [2W, K] quantized by the
    oracle in 128x128 blocks.  The gate weights are scaled up so that silu sees arguments
    spread over both signs and several units."""
    G = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]) + lead
    M = int(off[-1]) + trail
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((M, K), generator=g).to(torch.bfloat16)
    qs, ss = [], []
    for _ in range(G):
        w = torch.randn((2 * W, K), generator=g) * 0.02
        w[:W] *= gate_scale
        q, _, s = oracle.quant_block_128x128(bf16_bits(w.to(torch.bfloat16)))
        qs.append(q); ss.append(s)
    return off, x, np.stack(qs), np.stack(ss)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


CASES = [([3, 0, 130, 1, 200], 2, 5, 256, 384),
         ([256, 40, 0, 257, 17], 0, 0, 384, 1024),
         ([600, 300, 1], 0, 3, 128, 512)]


@pytest.mark.parametrize("pow2", [True, False])
@pytest.mark.parametrize("counts,lead,trail,W,K", CASES)
def test_swiglu_epilogue_equals_two_steps_and_oracle(mpq, tiles, counts, lead, trail, W, K, pow2):
    off, x_cpu, qb, sb = _problem(counts, lead, trail, W, K, 900 + W + K)
    M = x_cpu.shape[0]
    offs = _dev(off.astype(np.int64))
    qx, sx = oracle.quant_tile_1x128(bf16_bits(x_cpu))
    dqx, dsx, dqb, dsb = _dev(qx), _dev(sx), _dev(qb), _dev(sb)
    H = torch.full((M, 2 * W), -3.0, dtype=torch.bfloat16, device="cuda")
    q = torch.full((M, W), 0x55, dtype=torch.uint8, device="cuda")
    s = torch.full((W // 128, M), -7.0, dtype=torch.float32, device="cuda")
    mpq.fp8_grouped_gemm_swiglu_quant(offs, dqx, dsx, dqb, dsb, pow2=pow2, H=H, q=q, s=s)
    # the two-step path: grouped GEMM (BF16 out) on the same tiling, then SwiGLU + quantization
    C = torch.full((M, 2 * W), -3.0, dtype=torch.bfloat16, device="cuda")
    mpq.fp8_grouped_gemm_blockscaled(offs, dqx, dsx, dqb, dsb, C=C, tiles="rows")
    rows = slice(int(off[0]), int(off[-1]))
    q2, s2 = mpq.fp8_swiglu_quant_1x128(C[rows].contiguous(), pow2=pow2)
    torch.cuda.synchronize()
    assert torch.equal(H, C), "BF16 SwiGLU input differs from the grouped GEMM's output"
    assert torch.equal(q[rows], q2), "codes differ from GEMM + SwiGLU quantizer"
    assert torch.equal(s[:, rows], s2), "scales differ from GEMM + SwiGLU quantizer"
    # rows outside every expert untouched
    assert torch.all(q[: rows.start] == 0x55) and torch.all(q[rows.stop:] == 0x55)
    assert torch.all(s[:, : rows.start] == -7.0) and torch.all(s[:, rows.stop:] == -7.0)
    # the oracle: H against the FP64 grouped GEMM, codes/scales against its SwiGLU quantizer
    ref, absref = oracle.grouped_gemm_ref(off, qx, sx, qb, sb)
    Hh = H.float().cpu().numpy().astype(np.float64)
    assert_gemm_close(Hh[rows], ref[rows], absref[rows], "SwiGLU input")
    oq, os_ = oracle.swiglu_quant_1x128(bf16_bits(H[rows].cpu()), pow2=pow2)
    assert np.array_equal(q[rows].cpu().numpy(), oq)
    assert np.array_equal(s[:, rows].cpu().numpy(), os_)
    assert mpq.mpq_check_device_status() == (0, 0)


def test_swiglu_epilogue_many_tiles_per_cta(mpq, tiles):
    """About 16,000 rows over 8 experts, W = 512 (4 output tiles per m-tile): 500 single-SM
    tiles on 148 SMs, 250 pair tiles on 74 pairs, so every CTA hands over three or four tiles
    in turn through the same shared-memory area.  Bit-exact against GEMM + SwiGLU quantizer;
    sampled rows bit-exact against the oracle's SwiGLU quantizer on the GPU's BF16 input."""
    counts = [2100, 1900, 2050, 1999, 2001, 1950, 2048, 1950]
    off, x_cpu, qb, sb = _problem(counts, 0, 0, 512, 256, 4242)
    M = x_cpu.shape[0]
    offs = _dev(off.astype(np.int64))
    qx, sx = oracle.quant_tile_1x128(bf16_bits(x_cpu))
    dqx, dsx, dqb, dsb = _dev(qx), _dev(sx), _dev(qb), _dev(sb)
    q, s, H = mpq.fp8_grouped_gemm_swiglu_quant(offs, dqx, dsx, dqb, dsb, pow2=True, H=True)
    C = torch.empty((M, 1024), dtype=torch.bfloat16, device="cuda")
    mpq.fp8_grouped_gemm_blockscaled(offs, dqx, dsx, dqb, dsb, C=C, tiles="rows")
    q2, s2 = mpq.fp8_swiglu_quant_1x128(C, pow2=True)
    torch.cuda.synchronize()
    assert mpq.mpq_check_device_status() == (0, 0)
    assert torch.equal(H, C) and torch.equal(q, q2) and torch.equal(s, s2)
    rows = np.unique(np.random.default_rng(7).integers(0, M, 64))
    sel = torch.from_numpy(rows).cuda()
    oq, os_ = oracle.swiglu_quant_1x128(bf16_bits(H[sel].cpu()), pow2=True)
    assert np.array_equal(q[sel].cpu().numpy(), oq)
    assert np.array_equal(s[:, sel].cpu().numpy(), os_)


def test_swiglu_epilogue_without_cached_input(mpq):
    """H = None: only the codes and scales are written (the same values)."""
    off, x_cpu, qb, sb = _problem([70, 200], 0, 0, 256, 256, 31)
    offs = _dev(off.astype(np.int64))
    qx, sx = oracle.quant_tile_1x128(bf16_bits(x_cpu))
    args = (offs, _dev(qx), _dev(sx), _dev(qb), _dev(sb))
    qa, sa, Ha = mpq.fp8_grouped_gemm_swiglu_quant(*args, H=True)
    qn, sn, Hn = mpq.fp8_grouped_gemm_swiglu_quant(*args)
    torch.cuda.synchronize()
    assert Hn is None and torch.equal(qa, qn) and torch.equal(sa, sn)


@pytest.mark.parametrize("pow2", [True, False])
def test_swiglu_epilogue_with_fused_activation_quantization(mpq, pow2):
    """BF16 token rows quantized inside the launch (decode): equal to quantizing first."""
    off, x_cpu, qb, sb = _problem([1, 17, 0, 256, 90], 1, 2, 256, 512, 77)
    M = x_cpu.shape[0]
    offs = _dev(off.astype(np.int64))
    x = x_cpu.cuda()
    dqb, dsb = _dev(qb), _dev(sb)
    qf, sf, Hf = mpq.fp8_grouped_gemm_swiglu_quant(offs, x, None, dqb, dsb, pow2=pow2, fuse_quant=True, H=True)
    mpq.mpq_set_gemm_cta_pair(0)
    try:
        qx, sx, _, _ = mpq.fp8_quant_tile_1x128(x)
        q2, s2, H2 = mpq.fp8_grouped_gemm_swiglu_quant(offs, qx, sx, dqb, dsb, pow2=pow2, H=True)
    finally:
        mpq.mpq_set_gemm_cta_pair(1)
    torch.cuda.synchronize()
    rows = slice(int(off[0]), int(off[-1]))
    assert torch.equal(Hf[rows], H2[rows]) and torch.equal(qf[rows], q2[rows]) and torch.equal(sf[:, rows], s2[:, rows])
    assert mpq.mpq_check_device_status() == (0, 0)


def test_swiglu_epilogue_validation(mpq):
    off, x_cpu, qb, sb = _problem([10], 0, 0, 128, 128, 5)
    offs = _dev(off.astype(np.int64))
    qx, sx = oracle.quant_tile_1x128(bf16_bits(x_cpu))
    with pytest.raises(ValueError):          # odd number of weight rows
        mpq.fp8_grouped_gemm_swiglu_quant(offs, _dev(qx), _dev(sx), _dev(qb[:, :129].copy()),
                                          _dev(np.ones((1, 2, 1), np.float32)))
    M = qx.shape[0]
    with pytest.raises(mpq.MPQError) as ei:  # W not a multiple of 128
        mpq.fp8_grouped_gemm_swiglu_quant(offs, _dev(qx), _dev(sx), _dev(qb[:, :192].copy()),
                                          _dev(np.ones((1, 2, 1), np.float32)),
                                          s=torch.empty((1, M), dtype=torch.float32, device="cuda"))
    assert ei.value.status == 2
