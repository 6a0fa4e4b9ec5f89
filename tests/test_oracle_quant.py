"""Pins for the oracle's symmetric absmax block quantization (int4 and int8).

Block quantization with one scale per block is what ZeROPlusPlus.md §1.2
describes for both qwZ (int8 weights) and qgZ (int4 gradients).  The pins:
  * exhaustive pairs over a 256-value bf16 grid (B=2): codes and scale equal
    the stated chain of single-rounded operations evaluated in exact rational
    arithmetic, and every code is the exact nearest integer of c*qmax/m
    within 2^-20 (only near-ties may differ from the exact rounding);
  * round-half-even at exact ties, read off blocks where inv is exactly 1;
  * the round-trip bound |c - d| <= scale * (0.5 + 2^-18) on seeded blocks;
  * zero and subnormal blocks give scale 0 and all-zero codes;
  * the wire layout of the int4 codes (nibble order, two's complement).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from exact import EMIN, frac_of_bf16_bits, q_model, unpack_int4
from weight_communication_gb300 import workloads as wl


def _grid_bf16() -> np.ndarray:
    """256 bf16 patterns: zeros, subnormals, the normal boundary, exact
    half-step values, extremes and a seeded spread of exponents."""
    special = [0x0000, 0x0001, 0x0002, 0x0040, 0x007F, 0x0080, 0x0081, 0x00FF,
               0x3F80, 0x40E0, 0x4060, 0x4020, 0x3F00, 0x3FC0, 0x4090, 0x40B0,
               0x40D0, 0x4010, 0x3F40, 0x3E80, 0x7F7F, 0x7F00, 0x0100, 0x3C00,
               0x4000, 0x40C0, 0x4040, 0x4080, 0x40A0, 0x3FA0, 0x3FE0, 0x4050]
    rng = np.random.default_rng(20240530)
    rest = []
    while len(special) + len(rest) < 128:
        exp = int(rng.integers(0x60, 0x90))           # 2^-31 .. 2^16
        v = (exp << 7) | int(rng.integers(0, 128))
        if v not in special and v not in rest:
            rest.append(v)
    pos = np.array(special + rest, dtype=np.uint16)
    return np.concatenate([pos, pos | 0x8000]).astype(np.uint16)


@pytest.mark.parametrize("qmax", [7, 127])
def test_exhaustive_pairs_against_exact_arithmetic(orc, qmax):
    grid = _grid_bf16()
    a, b = np.meshgrid(grid, grid, indexing="ij")
    pairs = np.stack([a.ravel(), b.ravel()], axis=1)           # 65536 blocks of 2
    x = pairs.astype(np.uint32) << 16
    xf = x.view(np.float32).reshape(-1, 2)
    if qmax == 7:
        codes, scales = orc.ef_quant_int4(pairs.ravel().copy(), None, pairs.size, 1, 1,
                                          2, 1.0, 0.0)
        q = unpack_int4(codes).reshape(-1, 2)
    else:
        codes, scales = orc.qwz_quant_int8(pairs.ravel().copy(), 2)
        q = codes.reshape(-1, 2)
    fr = {int(h): frac_of_bf16_bits(int(h)) for h in grid}
    tie_band = Fraction(1, 2**20)
    for i in range(pairs.shape[0]):
        c = [fr[int(pairs[i, 0])], fr[int(pairs[i, 1])]]
        qm, sm = q_model(c, qmax)
        assert [int(q[i, 0]), int(q[i, 1])] == qm, (i, xf[i], q[i], qm)
        assert Fraction(float(scales[i])) == sm
        m = max(abs(v) for v in c)
        if m >= qmax * Fraction(2) ** EMIN:
            for j in range(2):
                exact = c[j] * qmax / m
                err = abs(exact - int(q[i, j]))
                assert err <= Fraction(1, 2) + tie_band
                assert abs(int(q[i, j])) <= qmax


def test_ties_round_half_even(orc):
    # absmax 7 makes scale = inv = 1 exactly, so the code is rint(c).
    vals = np.array([7.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5, -1.5, 4.5, 5.5,
                     6.5, -6.5, 0.25, 0.75, 1.25], dtype=np.float32)
    q, s = orc.quant_block(vals, 7)
    assert s == 1.0
    assert q.tolist() == [7, 2, 4, -2, -4, 0, 2, 0, -2, 4, 6, 6, -6, 0, 1, 1]
    # int8: absmax 127 gives scale = inv = 1
    vals8 = np.array([127.0, 2.5, -2.5, 126.5, -126.5, 0.5], dtype=np.float32)
    q8, s8 = orc.quant_block(vals8, 127)
    assert s8 == 1.0
    assert q8.tolist() == [127, 2, -2, 126, -126, 0]


def test_scale_is_absmax_over_qmax(orc):
    vals = np.array([0.5, -14.0, 3.0, 0.0], dtype=np.float32)
    q, s = orc.quant_block(vals, 7)
    assert s == 2.0                       # 14 / 7
    assert q.tolist() == [0, -7, 2, 0]    # 0.5/2 -> 0, 3/2 -> 2 (tie to even)
    q8, s8 = orc.quant_block(np.array([-254.0, 1.0, 3.0], dtype=np.float32), 127)
    assert s8 == 2.0 and q8.tolist() == [-127, 0, 2]


@pytest.mark.parametrize("B", [2, 32, 256, 512])
def test_zero_and_subnormal_blocks(orc, B):
    sub = np.full(B, np.float32(1e-40))
    sub[::2] *= -1
    for block in (np.zeros(B, np.float32), -np.zeros(B, np.float32), sub):
        q, s = orc.quant_block(block, 7)
        assert s == 0.0 and not q.any()
    # blocks whose scale would be subnormal are zero blocks too: at
    # m = 2^-126 the reciprocal 7/m would overflow to infinity
    tiny = np.float32(np.finfo(np.float32).tiny)
    for qmax in (7, 127):
        block = np.zeros(B, np.float32)
        block[0] = tiny
        q, s = orc.quant_block(block, qmax)
        assert s == 0.0 and not q.any()
        edge = np.float32(qmax) * tiny                      # exact
        block[0] = edge
        block[1] = -edge / 2
        q, s = orc.quant_block(block, qmax)
        assert s == tiny and q[0] == qmax and q[1] == -(qmax // 2 + (qmax // 2) % 2)
        block[0] = np.nextafter(edge, np.float32(0))
        q, s = orc.quant_block(block, qmax)
        assert s == 0.0 and not q.any()


@pytest.mark.parametrize("B,qmax", [(256, 7), (512, 7), (2048, 127)])
def test_round_trip_bound(orc, B, qmax):
    g = wl.draw_bf16(64 * B, 1e-3, seed=77, outlier_frac=1e-2, outlier_mult=100.0)
    gu = wl.as_u16(g)
    c = g.float().numpy()
    if qmax == 7:
        codes, scales = orc.ef_quant_int4(gu.copy(), None, gu.size, 1, 1, B, 1.0, 0.0)
        q = unpack_int4(codes).astype(np.float64)
    else:
        codes, scales = orc.qwz_quant_int8(gu.copy(), B)
        q = codes.astype(np.float64)
    sc = np.repeat(scales.astype(np.float64), B)
    d = (q * sc).astype(np.float32).astype(np.float64)
    bound = sc * (0.5 + 2.0**-18)
    assert np.all(np.abs(c - d) <= bound)
    assert np.all(np.abs(q) <= qmax)
    # every block reaches its absmax code
    assert np.all(np.abs(q.reshape(-1, B)).max(axis=1) == qmax)


def test_int4_wire_layout_hand_example(orc):
    # absmax 7 -> scale 1; codes are the values themselves.
    vals = np.array([1, -1, 7, -7, 0, 3, -4, 2], dtype=np.float32)
    g = torch.from_numpy(vals).to(torch.bfloat16)
    codes, scales = orc.ef_quant_int4(wl.as_u16(g).copy(), None, 8, 1, 1, 8, 1.0, 0.0)
    # byte k = low nibble: element 2k, high nibble: element 2k+1 (two's complement)
    assert codes.tolist() == [0xF1, 0x97, 0x30, 0x2C]
    assert scales.tolist() == [1.0]
    # the oracle's own reader agrees with the layout
    assert [orc.get_nibble(codes, i) for i in range(8)] == vals.astype(int).tolist()
