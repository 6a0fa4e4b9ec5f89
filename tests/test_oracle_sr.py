"""Pins for the oracle's stochastic-rounding accumulate.

"Zero 2 #593" (llm.c), review of llmc/cuda_utils.cuh: vector_add sums dst and
src in fp32 and rounds back to bf16 stochastically so that the accumulation
is correct in expectation; review of llmc/zero.cuh: zeroing src belongs in the
same kernel.  Pins:
  * the hash's finalizer against MurmurHash3_x86_32's published vectors;
  * exact unbiasedness: averaging SR(x, r) over all 65536 values of r gives
    x exactly (rational arithmetic), for 20 values across the range;
  * empirical unbiasedness over 10^6 seeds at a fixed index, within
    5 standard errors, and a chi-squared check of the 16 random bits;
  * values already representable in bf16 are unchanged; src ends zero;
  * eight accumulation steps stay unbiased against the exact sum.
"""
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest

from exact import frac_of_bf16_bits

GOLDEN = Path(__file__).parent / "golden" / "murmur3_x86_32.txt"


def _murmur3_x86_32(orc, key: bytes, seed: int) -> int:
    """MurmurHash3_x86_32 body and tail (the published algorithm), finalized
    by the oracle's fmix32."""
    c1, c2 = 0xCC9E2D51, 0x1B873593
    M = 0xFFFFFFFF
    rotl = lambda x, r: ((x << r) | (x >> (32 - r))) & M
    h = seed & M
    nblocks = len(key) // 4
    for i in range(nblocks):
        k = int.from_bytes(key[4 * i:4 * i + 4], "little")
        k = (k * c1) & M
        k = rotl(k, 15)
        k = (k * c2) & M
        h ^= k
        h = rotl(h, 13)
        h = (h * 5 + 0xE6546B64) & M
    tail = key[4 * nblocks:]
    if tail:
        k = int.from_bytes(tail, "little")
        k = (k * c1) & M
        k = rotl(k, 15)
        k = (k * c2) & M
        h ^= k
    h ^= len(key)
    return orc.fmix32(h)


def test_fmix32_against_published_vectors(orc):
    n = 0
    for line in GOLDEN.read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        key_hex, seed_hex, want_hex = line.split()
        key = b"" if key_hex == "-" else bytes.fromhex(key_hex)
        assert _murmur3_x86_32(orc, key, int(seed_hex, 16)) == int(want_hex, 16), line
        n += 1
    assert n == 10


def _f32(bits: int) -> float:
    return float(np.array([bits], dtype=np.uint32).view(np.float32)[0])


X_BITS = [0x3F800000, 0x3F800001, 0x3F80FFFF, 0x3F808000, 0xBF812345, 0x40490FDB,
          0xC0490FDB, 0x00000001, 0x8000FFFF, 0x007FFFFF, 0x00800000, 0x3A83126F,
          0xBA83126F, 0x4B7FFFFF, 0x3F7FFFFF, 0xBF7F8001, 0x38D1B717, 0x2F800000,
          0x7F000001, 0xFF01ABCD]


@pytest.mark.parametrize("bits", X_BITS)
def test_sr_is_exactly_unbiased_over_all_r(orc, bits):
    x = _f32(bits)
    total = Fraction(0)
    counts = {}
    for r in range(65536):
        h = orc.sr_round(x, r)
        counts[h] = counts.get(h, 0) + 1
    for h, cnt in counts.items():
        total += cnt * frac_of_bf16_bits(h)
    assert total / 65536 == Fraction(x)
    assert len(counts) <= 2                      # only the two neighbours


def test_sr_rounds_by_the_carry(orc):
    """The carry form: bf16 = (bits(x) + r) >> 16, so x rounds its magnitude up
    exactly when its low 16 bits plus r reach 2^16.  x = 1 + 2^-8 has the
    encoding 0x3F808000, low half 0x8000: r = 0x8000 carries (0x3F81, up) and
    r = 0x7FFF does not (0x3F80, down).  The other unbiased form, "up when the
    low half exceeds r", gives the opposite at both.  Negative values round
    their magnitude the same way; infinity passes through."""
    x = float(np.float32(1 + 2.0 ** -8))
    assert orc.sr_round(x, 0x8000) == 0x3F81
    assert orc.sr_round(x, 0x7FFF) == 0x3F80
    assert orc.sr_round(-x, 0x8000) == 0xBF81
    assert orc.sr_round(-x, 0x7FFF) == 0xBF80
    assert orc.sr_round(float("inf"), 0xFFFF) == 0x7F80


def test_sr_empirical_mean_over_seeds(orc):
    x = _f32(0x3F80_5A3C)                        # p = 0x5A3C / 65536
    lo, hi = frac_of_bf16_bits(0x3F80), frac_of_bf16_bits(0x3F81)
    ulp = float(hi - lo)
    p = 0x5A3C / 65536
    trials = 1_000_000
    ups = 0
    for seed in range(trials):
        r = orc.sr_bits(seed, 0, 12345)
        h = orc.sr_round(x, r)
        assert h in (0x3F80, 0x3F81)
        ups += h == 0x3F81
    mean = float(lo) + ulp * ups / trials
    assert abs(mean - x) <= 5 * ulp * (p * (1 - p) / trials) ** 0.5


def test_sr_bits_uniform(orc):
    n = 1 << 20
    bits = np.fromiter((orc.sr_bits(7, 3, i) for i in range(n)), dtype=np.uint32, count=n)
    assert bits.max() < 65536
    hist = np.bincount(bits, minlength=65536).astype(np.float64)
    expect = n / 65536
    chi2 = ((hist - expect) ** 2 / expect).sum()
    dof = 65535
    assert abs(chi2 - dof) < 6 * (2 * dof) ** 0.5
    # the low bit of the element index alone does not decide the low bit
    assert 0.45 < (bits[::2] & 1).mean() < 0.55


def test_sr_accumulate_semantics(orc):
    rng = np.random.default_rng(0)
    n = 4096
    dst = (rng.standard_normal(n).astype(np.float32)).view(np.uint32) >> 16
    dst = dst.astype(np.uint16)
    src = ((rng.standard_normal(n) * 1e-2).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    d0, s0 = dst.copy(), src.copy()
    orc.sr_accumulate_bf16(dst, src, seed=5, step=2)
    assert not src.any()
    for i in range(0, n, 97):
        x = np.float32(frac_of_bf16_bits(int(d0[i])) + frac_of_bf16_bits(int(s0[i])))
        assert dst[i] == orc.sr_round(float(x), orc.sr_bits(5, 2, i))
    # deterministic for the same (seed, step); a different step changes bits
    a, b = d0.copy(), s0.copy()
    orc.sr_accumulate_bf16(a, b, seed=5, step=2)
    assert np.array_equal(a, dst)
    a, b = d0.copy(), s0.copy()
    orc.sr_accumulate_bf16(a, b, seed=5, step=3)
    assert not np.array_equal(a, dst)
    # sums representable in bf16 pass through for any random bits
    same = d0.copy()
    zero = np.zeros(n, np.uint16)
    orc.sr_accumulate_bf16(same, zero, seed=1, step=0)
    assert np.array_equal(same, d0)


def test_eight_step_accumulation_is_unbiased(orc):
    """dst starts at 0 and receives 8 bf16 micro-gradients; over many elements
    the mean error against the exact fp64 sum is zero within its standard
    error, while round-to-nearest accumulation of the same data is biased
    when increments are small against the accumulator."""
    rng = np.random.default_rng(1)
    n = 1 << 17
    base = np.float32(1.0)
    dst = np.full(n, 0x3F80, np.uint16)                     # accumulator 1.0
    truth = np.full(n, 1.0)
    for t in range(8):
        inc = (np.abs(rng.standard_normal(n)) * 1e-3).astype(np.float32)
        src = (inc.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16
        truth += (src.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        orc.sr_accumulate_bf16(dst, src, seed=5, step=t)
    got = (dst.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = got - truth
    assert abs(err.mean()) < 5 * err.std() / n ** 0.5 + 1e-12
    # increments ~1e-3 are below half a bf16 step at 1.0 (2^-8): nearest
    # rounding would never move the accumulator
    assert float(base) + 8e-3 * 0.5 < got.mean()
