"""GEMM error against the unquantized product versus K (the accuracy the 128-element FP32
promotion is for): with the partial sums promoted every 128 elements, the error relative
to the FP64 product of the BF16 inputs comes from the FP8 quantization of the operands
only, so it must not grow with K.  Reference: plain PyTorch FP64 matmul on the CPU."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mpq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_quant_b300 as m
    return m


def _rel_err(mpq, k):
    d = workloads.dense_fprop(device="cuda", m=256, k=k, n=256)
    a, w = d["A"], d["W"]
    qa, sa, _, _ = mpq.fp8_quant_tile_1x128(a)
    qw, _, sw = mpq.fp8_quant_block_128x128(w)
    c = mpq.fp8_gemm_blockscaled(mpq.FPROP, qa, sa, qw, sw, out_dtype=mpq.OUT_FP32)
    ref = a.double().cpu() @ w.double().cpu().T
    return float((c.double().cpu() - ref).norm() / ref.norm())


def test_error_flat_in_k(mpq):
    errs = {k: _rel_err(mpq, k) for k in (512, 2048, 8192, 16384)}
    # E4M3 has 3 mantissa bits: per-element relative error up to 2^-4, about 2-3% in norm
    assert all(e < 0.05 for e in errs.values()), errs
    assert errs[16384] < 1.25 * errs[512], errs
