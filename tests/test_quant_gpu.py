"""GPU parity of the quantizers against the CPU oracle: FP8 codes and scales bit-exact."""
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


def _rows_parity(mpq, x_cpu, pow2):
    x = x_cpu.cuda()
    q, s, _, _ = mpq.fp8_quant_tile_1x128(x, pow2=pow2)
    oq, os_ = oracle.quant_tile_1x128(bf16_bits(x_cpu), pow2=pow2)
    np.testing.assert_array_equal(np_u8(q), oq)
    np.testing.assert_array_equal(np_f32(s).view(np.uint32), os_.view(np.uint32))


def _adversarial(rows=200, cols=512, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, cols), generator=g)
    x[0] = 0                                    # all-zero groups
    x[1] = 0; x[1, 77] = -3.0                   # one nonzero element
    for r in range(2, 34):                      # amax at every lane position of a 32-lane row
        x[r, (r * 4) % 128] *= 1000.0
    x[34, :] = 7.0; x[34, 5] = -7.0             # +-amax ties
    x[35] = torch.randn(cols, generator=g) * 1e-38   # subnormal-range inputs (tiny scales)
    x[36] = torch.randn(cols, generator=g) * 1e-30
    x[37] = -0.0
    x[38, :] = 448.0 * 2.0 ** torch.randint(-10, 10, (cols,), generator=g).float()  # binade boundaries
    x[39] = torch.randn(cols, generator=g) * (3e38 / 8)  # large but finite
    # values whose quotient lands on / next to an E4M3 rounding boundary
    lo = torch.tensor(oracle.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8)))
    hi = torch.tensor(oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8)))
    mids = ((lo + hi) / 2).float()
    for r in range(40, 48):
        v = mids[torch.randint(0, mids.numel(), (cols,), generator=g)]
        v[0] = 448.0
        x[r] = v * 2.0 ** (r - 44)
    return x.to(torch.bfloat16)


def _sweep_rows():
    """Every finite BF16 value x, each under many group scales: row = [amax, 127 values with
    |x| <= amax].  The max-abs values span the binary32 range, with significands 1, 1.75
    (the power-of-2 exponent step), just above 1.75 and all ones, and bracket 448 * 2^-80,
    below which the kernels switch from the multiply-and-correct path to IEEE division."""
    bits = np.arange(0x10000, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = np.sort(vals[np.isfinite(vals)].astype(np.float32))
    amaxes = []
    for e in list(range(-133, 127, 9)) + [-72, -71, -70, -69, -8, 0, 8]:
        for sig in (1.0, 1.75, 1.7578125, 1.9921875):
            a = np.float32(np.ldexp(sig, e))
            if np.isfinite(a) and a > 0:
                amaxes.append(a)
    rows = []
    for a in amaxes:
        v = vals[np.abs(vals) <= a]
        v = np.concatenate([v, np.zeros((-len(v)) % 127, np.float32)]).reshape(-1, 127)
        rows.append(np.concatenate([np.full((len(v), 1), a, np.float32), v], axis=1))
    x = torch.from_numpy(np.concatenate(rows)).to(torch.bfloat16)
    # the amax entries are BF16-exact; shuffle each row so the amax is not always in column 0
    g = torch.Generator().manual_seed(11)
    perm = torch.argsort(torch.rand(x.shape, generator=g), dim=1)
    return torch.gather(x, 1, perm)


@pytest.mark.parametrize("pow2", [False, True])
def test_tile_rows_every_bf16_value(mpq, pow2):
    _rows_parity(mpq, _sweep_rows(), pow2)


@pytest.mark.parametrize("pow2", [False, True])
def test_tile_rows_tiny_config(mpq, pow2):
    _rows_parity(mpq, workloads.tiny_fprop()["A"], pow2)


@pytest.mark.parametrize("pow2", [False, True])
def test_tile_rows_adversarial(mpq, pow2):
    _rows_parity(mpq, _adversarial(), pow2)


@pytest.mark.parametrize("rows", [1, 31, 33, 257])
def test_tile_rows_ragged(mpq, rows):
    g = torch.Generator().manual_seed(rows)
    x = (torch.randn((rows, 384), generator=g) * 5).to(torch.bfloat16)
    _rows_parity(mpq, x, False)


def test_tile_rows_strided(mpq):
    g = torch.Generator().manual_seed(5)
    big = (torch.randn((64, 640), generator=g)).to(torch.bfloat16).cuda()
    x = big[:, 128:512]  # ldx = 640, 16-byte aligned start
    q = torch.empty((64, 416), dtype=torch.uint8, device="cuda")[:, :384]
    s = torch.empty((3, 80), dtype=torch.float32, device="cuda")[:, :64]
    mpq.fp8_quant_tile_1x128(x, q=q, s=s)
    oq, os_ = oracle.quant_tile_1x128(bf16_bits(x.cpu()))
    np.testing.assert_array_equal(np_u8(q), oq)
    np.testing.assert_array_equal(np_f32(s), os_)


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("rows_out", [True, False])
def test_dual_quantizer(mpq, pow2, rows_out):
    x_cpu = torch.cat([_adversarial(128, 384, 1), (torch.randn((256, 384)) * 1e-3).to(torch.bfloat16)])
    x = x_cpu.cuda()
    q, s, qT, sT = mpq.fp8_quant_tile_1x128(x, pow2=pow2, rows_out=rows_out, transposed=True)
    bits = bf16_bits(x_cpu)
    if rows_out:
        oq, os_ = oracle.quant_tile_1x128(bits, pow2=pow2)
        np.testing.assert_array_equal(np_u8(q), oq)
        np.testing.assert_array_equal(np_f32(s), os_)
    oqT, osT = oracle.quant_tile_128x1(bits, pow2=pow2)
    np.testing.assert_array_equal(np_u8(qT), oqT)
    np.testing.assert_array_equal(np_f32(sT).view(np.uint32), osT.view(np.uint32))


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("transposed", [False, True])
def test_block_quantizer(mpq, pow2, transposed):
    g = torch.Generator().manual_seed(11)
    w_cpu = (torch.randn((384, 256), generator=g) * 0.02).to(torch.bfloat16)
    w_cpu[:128, :128] = 0
    w_cpu[128:256, 128:] *= 1e-35
    w = w_cpu.cuda()
    q, qT, s = mpq.fp8_quant_block_128x128(w, pow2=pow2, transposed=transposed)
    oq, oqT, os_ = oracle.quant_block_128x128(bf16_bits(w_cpu), pow2=pow2, transposed=transposed)
    np.testing.assert_array_equal(np_u8(q), oq)
    np.testing.assert_array_equal(np_f32(s).view(np.uint32), os_.view(np.uint32))
    if transposed:
        np.testing.assert_array_equal(np_u8(qT), oqT)


def test_full_size_dense_activation_sampled_rows(mpq):
    """4096 x 7168 activations with outlier channels: every row-group of 256 sampled rows."""
    d = workloads.dense_fprop(device="cuda", n=128)
    x = d["A"]
    q, s, _, _ = mpq.fp8_quant_tile_1x128(x)
    rows = torch.randperm(x.shape[0], generator=torch.Generator().manual_seed(0))[:256].sort().values
    rows = torch.cat([rows, torch.tensor([0, x.shape[0] - 1])]).unique()
    xs = x[rows.cuda()].cpu()
    oq, os_ = oracle.quant_tile_1x128(bf16_bits(xs))
    np.testing.assert_array_equal(np_u8(q[rows.cuda()]), oq)
    np.testing.assert_array_equal(np_f32(s[:, rows.cuda()]), os_)


def test_full_size_backward_dual_sampled(mpq):
    """8192 x 2048 dY (Student-t, pow2) through the fused dual quantizer: sampled row and
    column groups checked against the oracle."""
    d = workloads.backward_pair(device="cuda", k=128)
    dy = d["dY"]
    q, s, qT, sT = mpq.fp8_quant_tile_1x128(dy, pow2=True, transposed=True)
    # row groups on 128 sampled rows
    rows = torch.randperm(dy.shape[0], generator=torch.Generator().manual_seed(1))[:128].sort().values.cuda()
    oq, os_ = oracle.quant_tile_1x128(bf16_bits(dy[rows].cpu()), pow2=True)
    np.testing.assert_array_equal(np_u8(q[rows]), oq)
    np.testing.assert_array_equal(np_f32(s[:, rows]), os_)
    # column groups on two 128-row blocks x all columns
    for rb in (0, dy.shape[0] // 128 - 1):
        blk = dy[rb * 128:(rb + 1) * 128].cpu()
        oqT, osT = oracle.quant_tile_128x1(bf16_bits(blk), pow2=True)
        np.testing.assert_array_equal(np_u8(qT[:, rb * 128:(rb + 1) * 128]), oqT)
        np.testing.assert_array_equal(np_f32(sT[rb:rb + 1]), osT)


def test_full_size_weight_blocks_sampled(mpq):
    """18432 x 7168 weight: two block rows checked in full (codes, transposed codes, scales)."""
    d = workloads.dense_fprop(device="cuda", m=128)
    w = d["W"]
    q, qT, s = mpq.fp8_quant_block_128x128(w, transposed=True)
    for bi in (0, w.shape[0] // 128 - 1):
        blk = w[bi * 128:(bi + 1) * 128].cpu()
        oq, oqT, os_ = oracle.quant_block_128x128(bf16_bits(blk), transposed=True)
        np.testing.assert_array_equal(np_u8(q[bi * 128:(bi + 1) * 128]), oq)
        np.testing.assert_array_equal(np_u8(qT[:, bi * 128:(bi + 1) * 128]), oqT)
        np.testing.assert_array_equal(np_f32(s[bi:bi + 1]), os_)


def test_quantizer_validation_errors(mpq):
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mpq.MPQError) as e:
        mpq.fp8_quant_tile_1x128(x)
    assert e.value.status in (1, 2)  # cols % 128 != 0 (its empty scale array is also NULL)
    x = torch.zeros((100, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mpq.MPQError):
        mpq.fp8_quant_tile_1x128(x, transposed=True)  # rows % 128 != 0
    with pytest.raises(mpq.MPQError):
        mpq.fp8_quant_block_128x128(x)
