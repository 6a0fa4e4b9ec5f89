"""Pins for the oracle's bf16 conversions against torch's CPU conversions.

Rounding to bf16 is round-to-nearest-even at bit 16; torch's CPU float32 ->
bfloat16 cast is that library routine, so the oracle is compared with it over
every bf16 upper half and the low halves where rounding decides (0, 1, just
below / at / above the tie, all ones)."""
import numpy as np
import torch


def _f32_from_bits(u):
    return np.asarray(u, dtype=np.uint32).view(np.float32)


def test_widening_is_exact_for_every_pattern(orc):
    h = np.arange(65536, dtype=np.uint32)
    ref = torch.from_numpy(h.astype(np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([orc.bf16_to_f32(int(v)) for v in h], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_rne_matches_torch_on_every_upper_half(orc):
    upper = np.arange(65536, dtype=np.uint32)
    exp_all_ones = (upper & 0x7F80) == 0x7F80
    upper = upper[~exp_all_ones]          # inf / nan handled below
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    bits = (upper[:, None] << 16 | lows[None, :]).ravel()
    x = _f32_from_bits(bits)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_round(x)
    assert np.array_equal(got, ref)


def test_rne_specials(orc):
    inf = np.float32(np.inf)
    assert orc.f32_to_bf16(float(inf)) == 0x7F80
    assert orc.f32_to_bf16(float(-inf)) == 0xFF80
    # a NaN whose payload lies only in the low half must stay NaN
    for bits in (0x7F800001, 0x7FC00000, 0xFF800001, 0x7FFFFFFF):
        h = orc.f32_to_bf16(float(_f32_from_bits([bits])[0]))
        assert (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0
    # ties go to even: 1 + 2^-8 lies halfway between two bf16 values
    assert orc.f32_to_bf16(1.0 + 2.0**-8) == 0x3F80           # down to even 1.0
    assert orc.f32_to_bf16(1.0 + 3 * 2.0**-8) == 0x3F82       # up to even
    # largest finite fp32 rounds up into infinity
    assert orc.f32_to_bf16(float(np.finfo(np.float32).max)) == 0x7F80
    # signed zero is kept
    assert orc.f32_to_bf16(-0.0) == 0x8000
