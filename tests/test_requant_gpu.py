"""GPU parity of the re-quantization of cached FP8 codes into 128x1 groups (page 2, last
paragraph: the FP8 matrix is read out, dequantized, transposed and re-quantized into 128x1
tiles) against the CPU oracle: codes and scales bit-exact.  Every input is made on the CPU
(seeded) or by the oracle's own quantizer, never by the CUDA path."""
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


def _check(mpq, q, s, pow2):
    qT, sT = mpq.fp8_requant_tile_128x1(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), pow2=pow2)
    oqT, osT = oracle.requant_tile_128x1(q, s, pow2=pow2)
    np.testing.assert_array_equal(np_u8(qT), oqT)
    np.testing.assert_array_equal(np_f32(sT).view(np.uint32), osT.view(np.uint32))


def _bf16(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("pow2_in", [False, True])
@pytest.mark.parametrize("pow2_out", [False, True])
def test_requant_of_quantized_activations(mpq, pow2_in, pow2_out):
    """384 x 640 activations with outlier channels and row magnitudes over 2^+-8, quantized
    1x128 by the oracle, then re-quantized (several tiles in both directions)."""
    rng = np.random.default_rng(40)
    x = (rng.standard_normal((384, 640)) * np.exp(rng.uniform(-6, 6, (384, 1)))
         * rng.choice([1.0, 1.0, 1.0, 60.0], size=(1, 640))).astype(np.float32)
    q, s = oracle.quant_tile_1x128(_bf16(x), pow2=pow2_in)
    _check(mpq, q, s, pow2_out)


def _adversarial(rows=256, cols=512, seed=41):
    """Random finite codes under random 24-bit scales spanning the binary32 range, plus
    groups that are all +0 / all -0, single nonzero elements, the max at every row of a
    group, ties of +-max, and input scales near 2^-149 where the output scale floor
    applies."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 0x7F, size=(rows, cols)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=(rows, cols)) * 0x80).astype(np.uint8)
    exps = rng.integers(-140, 100, size=(cols // 128, rows))
    mant = rng.integers(0, 1 << 23, size=(cols // 128, rows)).astype(np.uint32)
    s = (((exps + 127).clip(1, 254).astype(np.uint32) << 23) | mant).view(np.float32)
    codes[:128, 0] = 0                      # all +0 column group
    codes[:128, 1] = 0x80                   # all -0
    codes[:128, 2] = 0; codes[77, 2] = 0xB5  # one nonzero element
    for r in range(128):                    # the max at every row position
        codes[128:, 3 + (r % 60)] &= 0x7F
    codes[128 + np.arange(128), 3 + (np.arange(128) % 60)] = 0x7E
    codes[130, 70] = 0x7E; codes[200, 70] = 0xFE   # +-max ties
    s[1, :] = np.float32(2.0 ** -149)       # column block 1: tiny input scales
    s[2, 5] = np.float32(3.0 * 2.0 ** -149)
    s[3, :64] = np.float32(2.0 ** -100) * np.float32(1.0 + 2.0 ** -23)
    return codes, s


@pytest.mark.parametrize("pow2_out", [False, True])
def test_requant_adversarial(mpq, pow2_out):
    q, s = _adversarial()
    _check(mpq, q, s, pow2_out)


def test_requant_every_code_under_many_scales(mpq):
    """All 254 finite codes in every column group, rotated so each code meets each row
    position, under 512 input scales (one per column block and row) with random
    significands over 2^-126 .. 2^119 (448 s stays finite, as it does for any scale the
    1x128 quantizer writes)."""
    rng = np.random.default_rng(42)
    rows, cols = 512, 1024
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    idx = (np.arange(rows)[:, None] + 7 * np.arange(cols)[None, :]) % finite.size
    q = finite[idx]
    exps = rng.integers(-126, 119, size=(cols // 128, rows))
    mant = rng.integers(0, 1 << 23, size=(cols // 128, rows)).astype(np.uint32)
    s = (((exps + 127).astype(np.uint32) << 23) | mant).view(np.float32)
    for pow2 in (False, True):
        _check(mpq, q, s, pow2)


def test_requant_strided(mpq):
    rng = np.random.default_rng(43)
    x = rng.standard_normal((256, 384)).astype(np.float32)
    q, s = oracle.quant_tile_1x128(_bf16(x))
    qb = torch.zeros((256, 512), dtype=torch.uint8, device="cuda")
    sb = torch.zeros((3, 260), dtype=torch.float32, device="cuda")
    qb[:, :384] = torch.from_numpy(q).cuda()
    sb[:, :256] = torch.from_numpy(s).cuda()
    qTb = torch.full((384, 272), 0x5A, dtype=torch.uint8, device="cuda")
    sTb = torch.full((2, 400), -1.0, dtype=torch.float32, device="cuda")
    mpq.fp8_requant_tile_128x1(qb[:, :384], sb[:, :256], qT=qTb[:, :256], sT=sTb[:, :384])
    oqT, osT = oracle.requant_tile_128x1(q, s)
    np.testing.assert_array_equal(np_u8(qTb[:, :256]), oqT)
    np.testing.assert_array_equal(np_f32(sTb[:, :384]), osT)
    assert np.all(np_u8(qTb[:, 256:]) == 0x5A) and np.all(np_f32(sTb[:, 384:]) == -1.0)   # untouched


def test_requant_full_size_backward_activation(mpq):
    """X 8192 x 7168 of the backward workload (the Wgrad operand), quantized 1x128 by the
    oracle, re-quantized on the GPU in the benchmark's launch configuration; every code
    and scale checked."""
    x = workloads.backward_pair(device="cpu", n=128)["X"]
    q, s = oracle.quant_tile_1x128(bf16_bits(x))
    _check(mpq, q, s, False)


def test_requant_validation_errors(mpq):
    q = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2, 128), dtype=torch.float32, device="cuda")
    qT = torch.empty((256, 112), dtype=torch.uint8, device="cuda")
    sT = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(mpq.MPQError) as e:
        mpq.fp8_requant_tile_128x1(q[:100], s[:, :100], qT=qT[:, :100], sT=sT)   # rows % 128
    assert e.value.status == 2
    sbig = torch.zeros((2, 130), dtype=torch.float32, device="cuda")
    with pytest.raises(mpq.MPQError) as e:
        mpq.fp8_requant_tile_128x1(q, sbig[:, 1:129])        # scales not 16-byte aligned
    assert e.value.status == 3
    qT, sT = mpq.fp8_requant_tile_128x1(q[:0], s[:, :0])     # zero rows: nothing to do
    assert qT.shape == (256, 0) and sT.shape == (0, 256)
