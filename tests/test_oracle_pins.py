"""Pins for the CPU oracle: each test ties it to something other than itself.

* the E4M3 codec against PyTorch's independent float8_e4m3fn conversion (a library
  routine the oracle does not use), plus round-trip / tie / saturation enumeration;
* hand-derived worked examples under tests/golden/;
* quantizers on inputs built by construction (codes and power-of-2 scales chosen
  first, the BF16 input made from them), so the expected output is known without
  evaluating the oracle's formula;
* closed forms of the scale rule and the error bound of round-to-nearest;
* the GEMM against a numpy matmul of dense dyadic matrices whose factorisation into
  (codes, scales) the test builds itself, and against exact integer matmul.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_decode(codes):
    t = torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_encode(vals):
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def f32_bits_to_bf16_bits(h):
    assert h & 0xFFFF == 0
    return (h >> 16) & 0xFFFF


def bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """BF16 bits of float32 values that are exactly representable in BF16."""
    b = np.asarray(x_f32, np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


# ------------------------------------------------------------------ codec

def test_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch_decode(codes)
    nan_ours, nan_ref = np.isnan(ours), np.isnan(ref)
    assert np.array_equal(nan_ours, nan_ref)
    assert set(np.nonzero(nan_ours)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan_ours], ref[~nan_ref])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9
    # signed zero
    assert math.copysign(1.0, ours[0x80]) == -1.0


def _probe_values():
    rng = np.random.default_rng(7)
    finite = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (finite[:-1] + finite[1:]) / 2.0  # exact in float32
    base = np.concatenate([finite, mids]).astype(np.float32)
    ulp_up = np.nextafter(base, np.float32(np.inf))
    ulp_dn = np.nextafter(base, np.float32(0))
    rnd = np.concatenate([
        rng.standard_normal(20000) * s for s in (1e-3, 1e-1, 1, 10, 100)
    ]).astype(np.float32)
    rnd = rnd[np.abs(rnd) <= 464]
    tiny = np.array([1e-30, 1e-42, 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11], np.float32)
    v = np.concatenate([base, ulp_up, ulp_dn, rnd, tiny]).astype(np.float32)
    v = np.concatenate([v, -v])
    return v[np.abs(v) <= 464]


def test_encode_matches_torch_in_range():
    v = _probe_values()
    assert np.array_equal(oracle.e4m3_encode(v), torch_encode(v))


def test_encode_saturates():
    big = np.array([448.0, 449.0, 464.0, 465.0, 1000.0, 3.0e38, np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)


def test_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = torch_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_midpoints_go_to_even_code():
    codes = np.arange(0, 0x7E, dtype=np.uint8)
    lo = torch_decode(codes)
    hi = torch_decode(codes + 1)
    mids = ((lo + hi) / 2).astype(np.float32)
    expect = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(mids), expect)
    assert np.array_equal(oracle.e4m3_encode(-mids), expect | 0x80)


# ---------------------------------------------------------- golden files

def _read_tile_golden():
    groups = {}
    cur = None
    with open(os.path.join(GOLDEN, "tile_1x128_worked.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "group":
                cur = tok[1]
                groups[cur] = {"amax": float(tok[2]), "scale": int(tok[3], 16), "elems": []}
            else:
                groups[cur]["elems"].append((int(tok[0]), int(tok[1], 16), int(tok[2], 16)))
    return groups


def test_golden_worked_tiles():
    groups = _read_tile_golden()
    assert set(groups) == {"A", "B", "C"}
    x = np.zeros((len(groups), 128), np.uint16)
    expect = np.zeros((len(groups), 128), np.uint8)
    for r, name in enumerate(sorted(groups)):
        for i, xbits, code in groups[name]["elems"]:
            x[r, i] = f32_bits_to_bf16_bits(xbits)
            expect[r, i] = code
    q, s = oracle.quant_tile_1x128(x)
    for r, name in enumerate(sorted(groups)):
        assert s[0, r].view(np.uint32) == groups[name]["scale"], name
    assert np.array_equal(q, expect)


def test_golden_gemm_one_slice():
    A = np.zeros((2, 128), np.uint8)
    B = np.zeros((2, 128), np.uint8)
    C = np.zeros((2, 2))
    with open(os.path.join(GOLDEN, "gemm_k128_worked.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            t = line.split()
            if t[0] == "A":
                A[int(t[1]), int(t[2])] = int(t[3], 16)
            elif t[0] == "B":
                B[int(t[1]), int(t[2])] = int(t[3], 16)
            elif t[0] == "SA":
                sa = np.array([[float(t[1]), float(t[2])]], np.float32)
            elif t[0] == "SB":
                sb = np.array([[float(t[1])]], np.float32)
            elif t[0] == "C":
                C[int(t[1]), int(t[2])] = float(t[3])
    ref, absref = oracle.gemm_ref(oracle.FPROP, A, sa, B, sb)
    assert np.array_equal(ref, C)
    assert absref[0, 0] == 2.5 and absref[1, 0] == 0.375


# ------------------------------------------------------------ scale rule

def test_scale_closed_forms():
    assert oracle.group_scale(896.0) == np.float32(2.0)
    assert oracle.group_scale(448.0) == np.float32(1.0)
    assert oracle.group_scale(0.0) == np.float32(1.0)
    assert oracle.group_scale(0.0, pow2=True) == np.float32(1.0)
    assert oracle.group_scale(448.0, pow2=True) == np.float32(1.0)
    assert oracle.group_scale(449.0, pow2=True) == np.float32(2.0)
    assert oracle.group_scale(224.0, pow2=True) == np.float32(0.5)
    assert oracle.group_scale(224.5, pow2=True) == np.float32(1.0)
    # smallest BF16 subnormal: 2^-133 <= 448 * 2^e  <=>  e >= -141.8...  -> e = -141
    assert oracle.group_scale(2.0 ** -133, pow2=True) == np.float32(2.0 ** -141)


def test_pow2_scale_is_smallest_covering_power():
    rng = np.random.default_rng(3)
    amax = np.float32(np.exp(rng.uniform(-60, 60, 400))).astype(np.float32)
    for a in amax:
        s = float(oracle.group_scale(a, pow2=True))
        e = math.frexp(s)[1] - 1
        assert s == 2.0 ** e
        assert float(a) <= 448.0 * 2.0 ** e
        assert float(a) > 448.0 * 2.0 ** (e - 1)


def test_amax_element_maps_to_448():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, (64, 1)))).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    for pow2 in (False, True):
        q, s = oracle.quant_tile_1x128(xb, pow2=pow2)
        xf = (xb.astype(np.uint32) << 16).view(np.float32).reshape(64, 2, 128)
        qq = q.reshape(64, 2, 128)
        idx = np.abs(xf).argmax(axis=2)
        top = np.take_along_axis(qq, idx[..., None], axis=2)[..., 0] & 0x7F
        if not pow2:
            assert np.all(top == 0x7E)
        else:
            # the largest magnitude lands in (224, 448]: codes 0x76 .. 0x7E
            assert np.all((top >= 0x76) & (top <= 0x7E))


# --------------------------------------------------- quantizers by construction

def _constructed(rows, cols, grid_r, grid_c, rng, pow2_exps):
    """Build a BF16 matrix from chosen codes and power-of-2 group scales.

    Groups are grid_r x grid_c; in each group one element gets code 0x7E (448) so the
    group's amax is exactly 448 * scale; the rest get random finite codes.  Returns
    (x bf16 bits, codes, scales[gr, gc])."""
    codes = rng.integers(0, 0x7F, size=(rows, cols)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=(rows, cols)) * 0x80).astype(np.uint8)
    gr, gc = rows // grid_r, cols // grid_c
    exps = rng.choice(pow2_exps, size=(gr, gc))
    for i in range(gr):
        for j in range(gc):
            r = i * grid_r + rng.integers(grid_r)
            c = j * grid_c + rng.integers(grid_c)
            codes[r, c] = 0x7E | (codes[r, c] & 0x80)
    vals = torch_decode(codes)
    sc = np.repeat(np.repeat(2.0 ** exps, grid_r, 0), grid_c, 1)
    x = (vals * sc).astype(np.float32)
    return bf16_bits(x), codes, (2.0 ** exps).astype(np.float32)


@pytest.mark.parametrize("pow2", [False, True])
def test_tile_1x128_by_construction(pow2):
    rng = np.random.default_rng(21)
    xb, codes, sc = _constructed(40, 384, 1, 128, rng, np.arange(-20, 21))
    q, s = oracle.quant_tile_1x128(xb, pow2=pow2)
    assert np.array_equal(q, codes)
    assert np.array_equal(s, sc.T)


@pytest.mark.parametrize("pow2", [False, True])
def test_tile_128x1_by_construction(pow2):
    rng = np.random.default_rng(22)
    xb, codes, sc = _constructed(256, 48, 128, 1, rng, np.arange(-20, 21))
    qT, sT = oracle.quant_tile_128x1(xb, pow2=pow2)
    assert np.array_equal(qT, codes.T)
    assert np.array_equal(sT, sc)


@pytest.mark.parametrize("pow2", [False, True])
def test_block_by_construction(pow2):
    rng = np.random.default_rng(23)
    xb, codes, sc = _constructed(256, 384, 128, 128, rng, np.arange(-20, 21))
    q, qT, s = oracle.quant_block_128x128(xb, pow2=pow2, transposed=True)
    assert np.array_equal(q, codes)
    assert np.array_equal(qT, codes.T)
    assert np.array_equal(s, sc)


def test_zero_groups():
    x = np.zeros((3, 256), np.uint16)
    x[1, :] = 0x8000  # -0.0
    q, s = oracle.quant_tile_1x128(x)
    assert np.all(s == 1.0)
    assert np.all(q[0] == 0) and np.all(q[1] == 0x80) and np.all(q[2] == 0)


def test_transposed_equals_row_quantizer_on_transpose():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((256, 384)) * rng.choice([1, 1, 50], size=(1, 384))).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    for pow2 in (False, True):
        qT, sT = oracle.quant_tile_128x1(xb, pow2=pow2)
        q2, s2 = oracle.quant_tile_1x128(np.ascontiguousarray(xb.T), pow2=pow2)
        assert np.array_equal(qT, q2) and np.array_equal(sT, s2)


def test_quantization_error_bound():
    """Round-to-nearest: |dec(q) s - x| <= 2^-4 |x| where x/s is in the E4M3 normal
    range (3 mantissa bits), and <= 2^-10 s below it (subnormal step 2^-9)."""
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((128, 512)) * np.exp(rng.uniform(-10, 10, (128, 1)))).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for pow2 in (False, True):
        q, s = oracle.quant_tile_1x128(xb, pow2=pow2)
        srow = np.repeat(s.T.astype(np.float64), 128, axis=1)
        deq = torch_decode(q) * srow
        err = np.abs(deq - xf)
        y = np.abs(xf) / srow
        normal = y >= 2.0 ** -6
        slack = 1 + 2.0 ** -20  # the binary32 quotient's own rounding
        assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xf[normal]) * slack)
        assert np.all(err[~normal] <= 2.0 ** -10 * srow[~normal] * slack)


# ------------------------------------------------------------------ GEMM

def _factor(dense, group_rows, group_cols, rng, exps=(-3, -2, -1, 0, 1, 2)):
    """Factor a dense dyadic matrix into E4M3 codes and power-of-2 group scales chosen
    by the test: codes = encode(dense / scale) exactly (values stay representable)."""
    R, C = dense.shape
    gr, gc = R // group_rows, C // group_cols
    e = rng.choice(exps, size=(gr, gc))
    sc = np.repeat(np.repeat(2.0 ** e, group_rows, 0), group_cols, 1)
    codes = torch_encode((dense / sc).astype(np.float32))
    assert np.array_equal(torch_decode(codes) * sc, dense)
    return codes, (2.0 ** e).astype(np.float32)


def _dyadic(rng, shape):
    # small integers times a per-element power of two: exact through every step
    return (rng.integers(-6, 7, size=shape) * 2.0 ** rng.integers(-2, 3, size=shape)).astype(np.float64)


@pytest.mark.parametrize("op", ["fprop", "dgrad", "wgrad"])
def test_gemm_matches_dense_dyadic_matmul(op):
    rng = np.random.default_rng({"fprop": 1, "dgrad": 2, "wgrad": 3}[op])
    M, N, K = 48, 256, 384
    Ad = _dyadic(rng, (M, K))
    Bd = _dyadic(rng, (N, K))
    qa, sa = _factor(Ad, 1, 128, rng)            # 1x128 tiles: sa[m, kb]
    sa_layout = np.ascontiguousarray(sa.T)       # [K/128, M]
    if op == "fprop":
        qb, sb = _factor(Bd, 128, 128, rng)      # blocks [N/128, K/128]
        code, sb_layout = oracle.FPROP, sb
    elif op == "dgrad":
        qb, sb = _factor(Bd, 128, 128, rng)
        code, sb_layout = oracle.DGRAD, np.ascontiguousarray(sb.T)  # [K/128, N/128]
    else:
        qb, sb = _factor(Bd, 1, 128, rng)        # per-row tiles sb[n, kb]
        code, sb_layout = oracle.WGRAD, np.ascontiguousarray(sb.T)  # [K/128, N]
    ref, absref = oracle.gemm_ref(code, qa, sa_layout, qb, sb_layout)
    expect = Ad @ Bd.T
    assert np.array_equal(ref, expect)
    assert np.array_equal(absref, np.abs(Ad) @ np.abs(Bd).T)


def test_gemm_small_integers_exact():
    rng = np.random.default_rng(4)
    vals = np.array([-4, -3, -2, -1, 0, 1, 2, 3, 4], np.float32)
    M, N, K = 33, 128, 1024
    ai = rng.choice(vals, size=(M, K)); bi = rng.choice(vals, size=(N, K))
    qa, qb = torch_encode(ai), torch_encode(bi)
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones((1, K // 128), np.float32)
    ref, _ = oracle.gemm_ref(oracle.FPROP, qa, sa, qb, sb)
    assert np.array_equal(ref, (ai.astype(np.int64) @ bi.astype(np.int64).T).astype(np.float64))


def test_gemm_ref_at_matches_full():
    rng = np.random.default_rng(6)
    qa = rng.integers(0, 0x7F, size=(20, 256)).astype(np.uint8)
    qb = rng.integers(0, 0x7F, size=(128, 256)).astype(np.uint8)
    sa = rng.uniform(0.1, 2, size=(2, 20)).astype(np.float32)
    sb = rng.uniform(0.1, 2, size=(1, 2)).astype(np.float32)
    full, fabs_ = oracle.gemm_ref(oracle.FPROP, qa, sa, qb, sb)
    ms = rng.integers(0, 20, 50); ns = rng.integers(0, 128, 50)
    at, aabs = oracle.gemm_ref_at(oracle.FPROP, qa, sa, qb, sb, ms, ns)
    assert np.array_equal(at, full[ms, ns]) and np.array_equal(aabs, fabs_[ms, ns])


def test_grouped_matches_per_expert_dense():
    rng = np.random.default_rng(8)
    G, N, K = 5, 128, 256
    counts = np.array([3, 0, 130, 1, 0])
    off = np.concatenate([[0], np.cumsum(counts)])
    M = int(off[-1]) + 4  # 4 trailing rows belong to no expert
    Ad = _dyadic(rng, (M, K))
    qa, sa = _factor(Ad, 1, 128, rng)
    Bd = [_dyadic(rng, (N, K)) for _ in range(G)]
    fac = [_factor(b, 128, 128, rng) for b in Bd]
    qb = np.stack([f[0] for f in fac]); sb = np.stack([f[1] for f in fac])
    ref, _ = oracle.grouped_gemm_ref(off, qa, np.ascontiguousarray(sa.T), qb, sb)
    expect = np.zeros((M, N))
    for g in range(G):
        expect[off[g]:off[g + 1]] = Ad[off[g]:off[g + 1]] @ Bd[g].T
    assert np.array_equal(ref, expect)


# ------------------------------------------- re-quantization of cached FP8 into 128x1

def test_scale_floor():
    """A positive max-abs never gives a zero scale: below 448 * 2^-149 (power of 2) or
    224 * 2^-149 (amax / 448 rounding to 0) the scale is 2^-149, the smallest positive
    binary32; just above, the ordinary rule applies."""
    tiny = np.float32(2.0 ** -149)
    for pow2 in (False, True):
        assert oracle.group_scale(tiny, pow2) == tiny
        assert oracle.group_scale(np.float32(224 * 2.0 ** -149), pow2) == tiny
        assert oracle.group_scale(np.float32(448 * 2.0 ** -149), pow2) == tiny
    # 449 * 2^-149 needs 2^-148 as a power of 2; amax / 448 rounds to 2^-149
    assert oracle.group_scale(np.float32(449 * 2.0 ** -149), True) == np.float32(2.0 ** -148)
    assert oracle.group_scale(np.float32(449 * 2.0 ** -149), False) == tiny
    # BF16's smallest subnormal is far above the floor
    assert oracle.group_scale(np.float32(2.0 ** -133), True) == np.float32(2.0 ** -141)


def _requant_constructed(rows, cols, rng):
    """Choose the re-quantization's answer first: output codes Qo [rows, cols] with
    magnitudes in [4, 64] plus one +-448 per 128x1 column group, and power-of-2 output
    scales So[rows/128, cols] in 2^-6 .. 1, so xhat = dec(Qo) So is exact.  Then factor
    xhat into a 1x128 input: scales s[cols/128, rows] = 2^k (k = 0, 1, 2) and codes
    q = encode(xhat / s), exact because xhat / s stays in the E4M3 normal range."""
    mags = rng.integers(0x48, 0x70, size=(rows, cols)).astype(np.uint8)   # 4 .. 60
    signs = (rng.integers(0, 2, size=(rows, cols)) * 0x80).astype(np.uint8)
    qo = mags | signs
    for rb in range(rows // 128):
        for c in range(cols):
            t = rb * 128 + rng.integers(128)
            qo[t, c] = 0x7E | (qo[t, c] & 0x80)
    so = (2.0 ** rng.integers(-6, 1, size=(rows // 128, cols))).astype(np.float32)
    xhat = torch_decode(qo) * np.repeat(so, 128, axis=0)
    s_in = (2.0 ** rng.integers(0, 3, size=(cols // 128, rows))).astype(np.float32)
    s_full = np.repeat(s_in.T, 128, axis=1)                                # [rows, cols]
    q = torch_encode((xhat / s_full).astype(np.float32))
    assert np.array_equal(torch_decode(q) * s_full, xhat)                 # exact factorisation
    return q, s_in, qo, so


@pytest.mark.parametrize("pow2", [False, True])
def test_requant_by_construction(pow2):
    rng = np.random.default_rng(31)
    q, s, qo, so = _requant_constructed(256, 384, rng)
    qT, sT = oracle.requant_tile_128x1(q, s, pow2=pow2)
    assert np.array_equal(qT, qo.T)
    assert np.array_equal(sT, so)


def test_requant_equals_128x1_quantizer_of_dequantized_values():
    """With power-of-2 input scales, dec(q) * s is exact and fits BF16 (four significant
    bits), so re-quantizing equals the 128x1 quantizer applied to the dequantized matrix."""
    rng = np.random.default_rng(32)
    x = (rng.standard_normal((384, 256)) * np.exp(rng.uniform(-6, 6, (384, 1)))
         * rng.choice([1.0, 1.0, 40.0], size=(1, 256))).astype(np.float32)
    q, s = oracle.quant_tile_1x128((x.view(np.uint32) >> 16).astype(np.uint16), pow2=True)
    xhat = (torch_decode(q) * np.repeat(s.T, 128, axis=1)).astype(np.float32)
    xb = bf16_bits(xhat)
    assert np.array_equal(((xb.astype(np.uint32) << 16).view(np.float32)), xhat)
    for pow2 in (False, True):
        qT, sT = oracle.requant_tile_128x1(q, s, pow2=pow2)
        q2, s2 = oracle.quant_tile_128x1(xb, pow2=pow2)
        assert np.array_equal(qT, q2) and np.array_equal(sT, s2)


def test_requant_zero_and_signed_zero_groups():
    q = np.zeros((128, 256), np.uint8)
    q[:, 128:] = 0x80                                      # -0
    s = np.full((2, 128), 3.0, np.float32)
    qT, sT = oracle.requant_tile_128x1(q, s)
    assert np.all(sT == 1.0)
    assert np.all(qT[:128] == 0) and np.all(qT[128:] == 0x80)



def _read_requant_golden():
    """tests/golden/requant_128x1_worked.txt: a hand-worked tile whose binary32 rounding of
    dec(q) * s decides one code (column 0) and one scale (column 1)."""
    q = np.zeros((128, 128), np.uint8)
    s = np.ones((1, 128), np.float32)
    expect = {}
    with open(os.path.join(GOLDEN, "requant_128x1_worked.txt")) as f:
        for line in f:
            tok = line.split("#", 1)[0].split()
            if not tok:
                continue
            if tok[0] == "scale_in":
                s[0, int(tok[1])] = np.array([int(tok[2], 16)], np.uint32).view(np.float32)[0]
            elif tok[0] == "code_in":
                q[int(tok[1]), int(tok[2])] = int(tok[3], 16)
            elif tok[0] == "expect":
                rule = expect.setdefault(tok[1], {"scale": {}, "code": {}})
                if tok[2] == "scale":
                    rule["scale"][int(tok[3])] = int(tok[4], 16)
                else:
                    rule["code"][(int(tok[3]), int(tok[4]))] = int(tok[5], 16)
    return q, s, expect


@pytest.mark.parametrize("rule", ["amax", "pow2"])
def test_golden_requant_binary32_dequantization(rule):
    """The dequantized value is one binary32 product: with exact (or FP64) products the
    code of column 0, row 1 would be 0x39 and the amax-rule scale of column 1 would be
    0x3F92492C."""
    q, s, expect = _read_requant_golden()
    qT, sT = oracle.requant_tile_128x1(q, s, pow2=(rule == "pow2"))
    want_s = np.ones(128, np.float32).view(np.uint32)
    for c, bits in expect[rule]["scale"].items():
        want_s[c] = bits
    assert np.array_equal(sT[0].view(np.uint32), want_s)
    want_q = np.zeros((128, 128), np.uint8)
    for (c, t), code in expect[rule]["code"].items():
        want_q[c, t] = code
    assert np.array_equal(qT, want_q)



# ------------------------------------------------------ SwiGLU + quantization

def _ulp32(v):
    """Spacing of binary32 numbers at |v| (2^-149 in the subnormal range)."""
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 23)


def test_exp_within_two_ulp_of_the_true_exponential():
    rng = np.random.default_rng(50)
    x = np.concatenate([rng.uniform(-103.0, 88.7, 200000), rng.uniform(-1, 1, 20000),
                        np.linspace(-0.4, 0.4, 4001)]).astype(np.float32)
    got = oracle.exp_f32(x).astype(np.float64)
    true = np.exp(x.astype(np.float64))
    assert np.all(np.abs(got - true) <= 2 * _ulp32(true))
    assert oracle.exp_f32(np.float32(0.0)) == 1.0
    assert oracle.exp_f32(np.float32(-104.5)) == 0.0 and oracle.exp_f32(np.float32(-1e30)) == 0.0
    assert np.isinf(oracle.exp_f32(np.float32(89.0))) and np.isinf(oracle.exp_f32(np.float32(3e38)))


def test_silu_close_to_the_true_function():
    rng = np.random.default_rng(51)
    # below about -88.7, e^-g overflows binary32 and the formula gives -0 (checked below)
    g = np.concatenate([rng.standard_normal(100000) * 4, rng.uniform(-88, 90, 20000)]).astype(np.float32)
    got = oracle.silu_f32(g).astype(np.float64)
    gd = g.astype(np.float64)
    true = gd / (1.0 + np.exp(-gd))
    assert np.all(np.abs(got - true) <= 4 * _ulp32(true) + 2.0 ** -149)
    # large positive g: e^-g is below half an ulp of 1, so silu(g) == g exactly
    big = np.float32([17.0, 100.0, 3e38])
    assert np.array_equal(oracle.silu_f32(big), big)
    # large negative g: e^-g overflows, silu(g) == -0
    neg = oracle.silu_f32(np.float32([-90.0, -3e38]))
    assert np.all(neg == 0) and np.all(np.signbit(neg))


def _bf16_trunc(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("pow2", [False, True])
def test_swiglu_quant_reduces_to_the_tile_quantizer(pow2):
    """With gate >= 17 silu is the identity, and with up = +-2^k the product is exact and a
    BF16 value: the SwiGLU quantizer must equal the 1x128 quantizer of gate * up."""
    rng = np.random.default_rng(52)
    rows, w = 64, 384
    gate = rng.uniform(17, 3000, (rows, w)).astype(np.float32)
    gate = ((_bf16_trunc(gate).astype(np.uint32) << 16).view(np.float32))
    up = (rng.choice([-1.0, 1.0], (rows, w)) * 2.0 ** rng.integers(-20, 10, (rows, w))).astype(np.float32)
    hcat = np.concatenate([_bf16_trunc(gate), _bf16_trunc(up)], axis=1)
    q, s = oracle.swiglu_quant_1x128(hcat, pow2=pow2)
    prod = (gate * up).astype(np.float32)
    q2, s2 = oracle.quant_tile_1x128(bf16_bits(prod), pow2=pow2)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_swiglu_quant_zero_groups_and_signs():
    """gate = 0 or up = 0, or a very negative gate, give +-0 products: zero groups, scale 1,
    codes carrying the product's sign."""
    rows, w = 4, 128
    gate = np.zeros((rows, w), np.float32)
    up = np.ones((rows, w), np.float32)
    gate[1] = -200.0                     # silu = -0, times +1 -> -0
    up[2] = -1.0                         # +0 * -1 -> -0
    gate[3] = 5.0; up[3] = 0.0           # silu(5) * +0 -> +0
    hcat = np.concatenate([_bf16_trunc(gate), _bf16_trunc(up)], axis=1)
    q, s = oracle.swiglu_quant_1x128(hcat, pow2=True)
    assert np.all(s == 1.0)
    assert np.all(q[0] == 0) and np.all(q[1] == 0x80) and np.all(q[2] == 0x80) and np.all(q[3] == 0)


@pytest.mark.parametrize("pow2", [False, True])
def test_swiglu_quant_error_bound(pow2):
    """Against silu(gate) * up in float64: the 1x128 quantization error bound (2^-4 relative
    in the E4M3 normal range, 2^-10 s below it) plus the binary32 SwiGLU's own few ulps."""
    rng = np.random.default_rng(53)
    rows, w = 128, 512
    gate = (rng.standard_normal((rows, w)) * 3).astype(np.float32)
    up = (rng.standard_normal((rows, w)) * np.exp(rng.uniform(-5, 5, (rows, 1)))).astype(np.float32)
    hcat = np.concatenate([_bf16_trunc(gate), _bf16_trunc(up)], axis=1)
    g = (hcat[:, :w].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    u = (hcat[:, w:].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x = g / (1.0 + np.exp(-g)) * u
    q, s = oracle.swiglu_quant_1x128(hcat, pow2=pow2)
    srow = np.repeat(s.T.astype(np.float64), 128, axis=1)
    err = np.abs(torch_decode(q) * srow - x)
    y = np.abs(x) / srow
    normal = y >= 2.0 ** -6
    slack = 1 + 2.0 ** -18
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) * slack + 8 * _ulp32(x[normal]))
    assert np.all(err[~normal] <= 2.0 ** -10 * srow[~normal] * slack + 8 * _ulp32(x[~normal]))


def _read_swiglu_golden():
    groups = {}
    cur = None
    with open(os.path.join(GOLDEN, "swiglu_1x128_worked.txt")) as f:
        for line in f:
            tok = line.split("#", 1)[0].split()
            if not tok:
                continue
            if tok[0] == "group":
                cur = tok[1]
                groups[cur] = {"scale": int(tok[2], 16), "elems": []}
            else:
                groups[cur]["elems"].append(tuple(int(t, 0) for t in tok))
    return groups


def test_golden_swiglu_binary32_sequence():
    """silu(g) * u is a sequence of binary32 operations, each rounded once: computing it in
    FP64 and rounding once would give the scales 0x3D65B6DA and 0x3B80D919 instead."""
    groups = _read_swiglu_golden()
    assert set(groups) == {"P", "Q"}
    names = sorted(groups)
    h = np.zeros((len(names), 256), np.uint16)
    want_q = np.zeros((len(names), 128), np.uint8)
    for r, name in enumerate(names):
        for i, gate, up, code in groups[name]["elems"]:
            h[r, i], h[r, 128 + i] = gate, up
            want_q[r, i] = code
    q, sc = oracle.swiglu_quant_1x128(h, pow2=False)
    assert np.array_equal(q, want_q)
    for r, name in enumerate(names):
        assert sc[0, r].view(np.uint32) == groups[name]["scale"], name
