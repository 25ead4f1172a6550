"""Host-side argument checks of the Python binding (no GPU): a wrong dtype of the expert
offsets or of a caller-given output is reported before anything reaches the library, so
the C side never reads an int32 offsets array as int64 or writes FP32 rows into a BF16
buffer."""
import pytest
import torch


@pytest.fixture(scope="module")
def mpq():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import mixed_precision_quant_b300 as m
    return m


def _noalloc_args(G=2, N=256, K=256, M=64):
    off = torch.tensor([0, 30, M], dtype=torch.int64)
    X = torch.zeros((M, K), dtype=torch.bfloat16)
    B = torch.zeros((G, N, K), dtype=torch.uint8)
    sB = torch.ones((G, N // 128, K // 128), dtype=torch.float32)
    C = torch.zeros((M, N), dtype=torch.bfloat16)
    return off, X, B, sB, C


def test_noalloc_rejects_int32_offsets(mpq):
    off, X, B, sB, C = _noalloc_args()
    with pytest.raises(TypeError, match="offsets"):
        mpq.fp8_grouped_gemm_fused_quant_noalloc(off.to(torch.int32), X, B, sB, C)


def test_noalloc_rejects_output_dtype_mismatch(mpq):
    off, X, B, sB, C = _noalloc_args()
    with pytest.raises(TypeError, match="C: out_dtype asks for torch.float32"):
        mpq.fp8_grouped_gemm_fused_quant_noalloc(off, X, B, sB, C, out_dtype=mpq.OUT_FP32)
    with pytest.raises(TypeError, match="C: out_dtype asks for torch.bfloat16"):
        mpq.fp8_grouped_gemm_fused_quant_noalloc(off, X, B, sB, C.float(), out_dtype=mpq.OUT_BF16)


def test_noalloc_rejects_wrong_output_shape_and_host_tensors(mpq):
    off, X, B, sB, C = _noalloc_args()
    with pytest.raises(ValueError, match="C: expected shape"):
        mpq.fp8_grouped_gemm_fused_quant_noalloc(off, X, B, sB, C[:, :128])
    # right dtypes and shapes, but host memory: refused before any call into the library
    with pytest.raises(TypeError, match="CUDA"):
        mpq.fp8_grouped_gemm_fused_quant_noalloc(off, X, B, sB, C)


def test_grouped_rejects_int32_offsets(mpq):
    off, X, B, sB, C = _noalloc_args()
    A = torch.zeros(X.shape, dtype=torch.uint8)
    sA = torch.ones((X.shape[1] // 128, X.shape[0]), dtype=torch.float32)
    with pytest.raises(TypeError, match="offsets"):
        mpq.fp8_grouped_gemm_blockscaled(off.to(torch.int32), A, sA, B, sB)
    with pytest.raises(TypeError, match="offsets"):
        mpq.fp8_grouped_gemm_blockscaled(off.to(torch.int32), X, None, B, sB, fuse_quant=True)


def test_output_check_names_dtype_shape_and_device(mpq):
    C = torch.zeros((4, 256), dtype=torch.float32)
    with pytest.raises(TypeError, match="bfloat16"):
        mpq._check_output(C, mpq.OUT_BF16, 4, 256, torch.device("cpu"))
    with pytest.raises(ValueError, match="shape"):
        mpq._check_output(C, mpq.OUT_FP32, 8, 256, torch.device("cpu"))
    with pytest.raises(ValueError, match="out_dtype"):
        mpq._check_output(C, 7, 4, 256, torch.device("cpu"))
