"""GPU test of fp8_grouped_gemm_fused_quant_noalloc, the allocation-free form of the fused
grouped GEMM (its scratch is a fixed area in the library's device code).

Collected last on purpose: it must pass on its own and after every other test."""
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


def _problem(counts, lead, trail, N, K, seed):
    G = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]) + lead
    M = int(off[-1]) + trail
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((M, K), generator=g) * 1.5).to(torch.bfloat16)
    qs, ss = [], []
    for _ in range(G):
        w = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16)
        q, _, s = oracle.quant_block_128x128(bf16_bits(w))
        qs.append(q); ss.append(s)
    return off, x, np.stack(qs), np.stack(ss)


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("counts,lead,trail,N,K", [
    ([3, 0, 130, 1, 200], 2, 5, 256, 384),
    ([256, 40, 0, 257, 17], 0, 0, 384, 1024),
])
def test_noalloc_matches_fused_entry_point(mpq, counts, lead, trail, N, K, pow2):
    off, x_cpu, qb, sb = _problem(counts, lead, trail, N, K, 4242 + len(counts))
    M = x_cpu.shape[0]
    offs = torch.from_numpy(off.astype(np.int64)).cuda()
    x, qbd, sbd = x_cpu.cuda(), torch.from_numpy(qb).cuda(), torch.from_numpy(sb).cuda()
    # the entry point with a workspace (same launch, same tiling): the results must agree
    # bit for bit, as the header promises
    fused = torch.full((M, N), -5.0, dtype=torch.float32, device="cuda")
    mpq.fp8_grouped_gemm_blockscaled(offs, x, None, qbd, sbd, out_dtype=mpq.OUT_FP32, C=fused, fuse_quant=True,
                                     pow2=pow2)
    # the oracle: 1x128 quantization of the BF16 rows, then the FP64 grouped GEMM
    ref, absref = oracle.grouped_gemm_ref(off, *oracle.quant_tile_1x128(bf16_bits(x_cpu), pow2=pow2), qb, sb)
    rows = np.zeros(M, bool)
    rows[int(off[0]):int(off[-1])] = True
    assert_gemm_close(fused.cpu().numpy()[rows], ref[rows], absref[rows], "fused entry point")
    for call in range(2):   # two calls in a row reuse the same scratch area
        C = torch.full((M, N), -5.0, dtype=torch.float32, device="cuda")
        mpq.fp8_grouped_gemm_fused_quant_noalloc(offs, x, qbd, sbd, C, out_dtype=mpq.OUT_FP32, pow2=pow2)
        torch.cuda.synchronize()
        assert torch.equal(C, fused), f"no-alloc call {call} differs from the fused entry point"
        got = C.cpu().numpy().astype(np.float64)
        assert_gemm_close(got[rows], ref[rows], absref[rows], f"no-alloc call {call}")
        assert np.all(got[~rows] == -5.0), "rows outside every expert were written"
    assert mpq.mpq_check_device_status() == (0, 0)


def test_noalloc_allocates_nothing_and_rejects_oversize(mpq):
    off, x_cpu, qb, sb = _problem([100, 60, 3], 0, 0, 256, 512, 77)
    M, N = x_cpu.shape[0], 256
    offs = torch.from_numpy(off.astype(np.int64)).cuda()
    x, qbd, sbd = x_cpu.cuda(), torch.from_numpy(qb).cuda(), torch.from_numpy(sb).cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mpq.fp8_grouped_gemm_fused_quant_noalloc(offs, x, qbd, sbd, C)   # first call: scratch lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        mpq.fp8_grouped_gemm_fused_quant_noalloc(offs, x, qbd, sbd, C)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "device memory changed across calls"
    # a problem whose scratch need exceeds the fixed area is rejected before any launch
    K_big = 7168
    M_big = mpq.NOALLOC_SCRATCH_BYTES // K_big + 1
    xb = torch.zeros((M_big, K_big), dtype=torch.bfloat16, device="cuda")
    wb = torch.zeros((1, 128, K_big), dtype=torch.uint8, device="cuda")
    sw = torch.ones((1, 1, K_big // 128), dtype=torch.float32, device="cuda")
    ob = torch.tensor([0, M_big], dtype=torch.int64, device="cuda")
    Cb = torch.empty((M_big, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mpq.MPQError) as ei:
        mpq.fp8_grouped_gemm_fused_quant_noalloc(ob, xb, wb, sw, Cb)
    assert ei.value.status == 7
