"""Pins for the limited-precision accumulator of the accuracy study (bench._acc_limited).

The study models the observation that FP8 GEMM accumulation on the pages' GPUs keeps only
about 14 bits (page 3, blog.cameseeing.com freeboard 1171527, first paragraph, its last
sentence).  The pages do not say how the bits are lost.  Our reading: for each chunk of 32
products the running sum and the products are aligned to the largest exponent among them,
every term is truncated toward zero to a multiple of 2^(e - bits), and the truncated terms
are added exactly.  These tests tie the emulation to values derived by hand and to properties that
follow from that reading, not to a second copy of its formula:

* wide windows reduce it to the exact sum (checked with rational arithmetic);
* hand-worked truncations: one product, small products swallowed by a large running sum,
  truncation toward zero for negative terms, the running sum truncated at a chunk boundary;
* non-negative products: the result never exceeds the exact sum and falls short of it by less
  than one window unit per truncated term;
* the error shrinks as the window grows, on random E4M3-code products.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import bench


def _run(a, b, bits, chunk=32):
    ca = torch.tensor(np.asarray(a, np.float64)).reshape(1, -1)
    cb = torch.tensor(np.asarray(b, np.float64)).reshape(1, -1)
    return float(bench._acc_limited(ca, cb, bits, chunk)[0, 0])


def _exact(a, b):
    return sum(Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a, b))


def test_wide_window_is_exact():
    """A 60-bit window holds every term of these small dyadic products: exact sum."""
    rng = np.random.default_rng(11)
    a = rng.integers(-448, 449, 96) * 2.0 ** rng.integers(-6, 3, 96)
    b = rng.integers(-448, 449, 96) * 2.0 ** rng.integers(-6, 3, 96)
    assert Fraction(_run(a, b, 60)) == _exact(a, b)


def test_single_product_truncates_toward_zero():
    """-1.75 with a 2-bit window: |p| < 2^1, unit 2^(1-2) = 0.5, -3.5 units -> -3 -> -1.5
    (round to nearest would give -2)."""
    assert _run([-1.75], [1.0], 2) == -1.5
    assert _run([1.75], [1.0], 2) == 1.5
    # 1.75 < 2^1 needs 3 bits: a 3-bit window keeps it
    assert _run([1.75], [1.0], 3) == 1.75


def test_small_terms_swallowed_by_large_sum():
    """32 products of 1 give 32 exactly; then 32 products of 2^-20 meet a running sum of
    32 < 2^6, unit 2^(6-14) = 2^-8, so each truncates to 0 and the sum stays 32 (the exact
    sum is 32 + 2^-15)."""
    a = [1.0] * 32 + [2.0 ** -20] * 32
    b = [1.0] * 64
    assert _run(a, b, 14) == 32.0
    assert _exact(a, b) == 32 + Fraction(1, 2 ** 15)


def test_running_sum_truncated_at_chunk_boundary():
    """Chunk 1: 1 + 2^-10 (exact in a 14-bit window, max 1 < 2^1, unit 2^-13).  Chunk 2:
    one product of 8, max 8 < 2^4, unit 2^-10: the running sum 1 + 2^-10 stays, then the
    product 2^-12 in the same chunk truncates to 0 -> 9 + 2^-10.  A chunk of 2 puts the
    two small terms in separate chunks."""
    a = [1.0, 2.0 ** -10, 8.0, 2.0 ** -12]
    b = [1.0, 1.0, 1.0, 1.0]
    assert _run(a, b, 14, chunk=2) == 9.0 + 2.0 ** -10
    # one chunk of four: max 8 < 2^4, unit 2^-10 for every term: 2^-12 is lost, 2^-10 kept
    assert _run(a, b, 14, chunk=4) == 9.0 + 2.0 ** -10
    # a 12-bit window: unit 2^-8 in the second chunk drops the carried 2^-10 too
    assert _run(a, b, 12, chunk=2) == 9.0


@pytest.mark.parametrize("bits", [8, 11, 14])
def test_nonnegative_products_one_sided_bound(bits):
    """With non-negative products every truncation removes a value in [0, unit): the result
    is at most the exact sum, and short of it by less than (terms + 1) units per chunk,
    a unit being 2^(e - bits) with the chunk's magnitude below 2^e <= 2 * magnitude."""
    rng = np.random.default_rng(bits)
    a = rng.integers(0, 449, 256) * 2.0 ** rng.integers(-8, 1, 256)
    b = rng.integers(0, 449, 256) * 2.0 ** rng.integers(-8, 1, 256)
    got = Fraction(_run(a, b, bits))
    exact = _exact(a, b)
    assert got <= exact
    bound = Fraction(0)
    partial = Fraction(0)
    for k0 in range(0, 256, 32):
        prods = [Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a[k0:k0 + 32], b[k0:k0 + 32])]
        partial += sum(prods)
        mag = max(max(prods), partial)     # the running sum only grows with non-negative terms
        bound += 33 * 2 * mag / 2 ** bits
    assert exact - got < bound


def test_error_shrinks_with_window():
    """On products of random E4M3 codes the error against the exact sum does not grow as the
    window widens, and vanishes at 53 bits."""
    rng = np.random.default_rng(7)
    codes = torch.tensor(rng.integers(0, 256, (4, 512)), dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64)
    vals = torch.where(torch.isnan(vals), torch.zeros_like(vals), vals)
    ca, cb = vals[:2], vals[2:]
    exact = torch.tensor([[float(_exact(ca[i].numpy(), cb[j].numpy())) for j in range(2)] for i in range(2)],
                         dtype=torch.float64)
    errs = [float((bench._acc_limited(ca, cb, bits) - exact).abs().max()) for bits in (6, 10, 14, 20, 53)]
    assert all(errs[i + 1] <= errs[i] for i in range(len(errs) - 1)), errs
    assert errs[-1] == 0.0
    assert errs[0] > 0.0
