"""GPU parity of the SwiGLU + 1x128 quantization (the down projection's FP8 input) against
the CPU oracle: codes and scales bit-exact, the binary32 SwiGLU (own exponential) followed
operation by operation on both sides.  Inputs are seeded CPU tensors or workload tensors."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import bf16_bits, np_f32, np_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mpq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_quant_b300 as m
    return m


def _check(mpq, hcat_cpu, pow2):
    q, s = mpq.fp8_swiglu_quant_1x128(hcat_cpu.cuda(), pow2=pow2)
    oq, os_ = oracle.swiglu_quant_1x128(bf16_bits(hcat_cpu), pow2=pow2)
    np.testing.assert_array_equal(np_u8(q), oq)
    np.testing.assert_array_equal(np_f32(s).view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("pow2", [True, False])
def test_swiglu_quant_random(mpq, pow2):
    """Gate ~ 3 N(0,1), up ~ N(0,1) times per-row magnitudes 2^+-7; rows span several
    batches of the grid-stride loop and a ragged tail."""
    g = torch.Generator().manual_seed(60)
    rows, w = 333, 640
    gate = torch.randn((rows, w), generator=g) * 3
    up = torch.randn((rows, w), generator=g) * torch.exp(torch.empty((rows, 1)).uniform_(-5, 5, generator=g))
    _check(mpq, torch.cat([gate, up], 1).to(torch.bfloat16), pow2)


@pytest.mark.parametrize("pow2", [True, False])
def test_swiglu_quant_every_gate_value(mpq, pow2):
    """Every finite BF16 gate value (e^-g from underflow to overflow, signed zeros,
    subnormals) against up values of several magnitudes, all below 1/2 so that every
    product stays finite (the contract)."""
    bits = np.arange(0x10000, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.isfinite(vals)]
    w = 1024
    n = (vals.size + w - 1) // w * w
    gate = np.resize(vals, n).reshape(-1, w)
    rng = np.random.default_rng(61)
    up = (np.clip(rng.standard_normal(gate.shape), -4, 4)
          * 2.0 ** rng.integers(-30, -3, (gate.shape[0], 1))).astype(np.float32)
    hc = np.concatenate([(gate.view(np.uint32) >> 16).astype(np.uint16),
                         (up.view(np.uint32) >> 16).astype(np.uint16)], 1)
    _check(mpq, torch.from_numpy(hc.view(np.int16)).view(torch.bfloat16), pow2)


def test_swiglu_quant_strided_and_empty(mpq):
    g = torch.Generator().manual_seed(62)
    hc = (torch.randn((130, 2 * 256 + 64), generator=g) * 2).to(torch.bfloat16).cuda()
    view = hc[:, :512]                                   # ldh = 576
    q = torch.full((130, 272), 0x5A, dtype=torch.uint8, device="cuda")
    s = torch.full((2, 140), -1.0, dtype=torch.float32, device="cuda")
    mpq.fp8_swiglu_quant_1x128(view, q=q[:, :256], s=s[:, :130])
    oq, os_ = oracle.swiglu_quant_1x128(bf16_bits(view.cpu()), pow2=True)
    np.testing.assert_array_equal(np_u8(q[:, :256]), oq)
    np.testing.assert_array_equal(np_f32(s[:, :130]), os_)
    assert np.all(np_u8(q[:, 256:]) == 0x5A) and np.all(np_f32(s[:, 130:]) == -1.0)
    q0, s0 = mpq.fp8_swiglu_quant_1x128(hc[:0, :512])
    assert q0.shape == (0, 256) and s0.shape == (2, 0)


def test_swiglu_quant_full_size_prefill_sampled(mpq):
    """The MoE prefill's up-projection output shape (131072 x 2*2048): every group of 300
    sampled rows (plus the first and last) checked against the oracle."""
    rows, w = 131072, 2048
    gen = torch.Generator(device="cuda").manual_seed(63)
    hc = (torch.randn((rows, 2 * w), generator=gen, device="cuda") * 2).to(torch.bfloat16)
    q, s = mpq.fp8_swiglu_quant_1x128(hc)
    idx = torch.randperm(rows, generator=torch.Generator().manual_seed(64))[:300]
    idx = torch.cat([idx, torch.tensor([0, rows - 1])]).unique().cuda()
    oq, os_ = oracle.swiglu_quant_1x128(bf16_bits(hc[idx].cpu()), pow2=True)
    np.testing.assert_array_equal(np_u8(q[idx]), oq)
    np.testing.assert_array_equal(np_f32(s[:, idx]), os_)


def test_swiglu_quant_validation(mpq):
    hc = torch.zeros((4, 200), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((4, 128), dtype=torch.uint8, device="cuda")
    s = torch.empty((1, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(mpq.MPQError) as e:
        mpq.fp8_swiglu_quant_1x128(hc, q=q, s=s)              # width 100: not a multiple of 128
    assert e.value.status == 2
