"""Pins for the oracle's qgZ path: error-feedback quantization, send order,
flat and hierarchical dequant-reduce.

Passages: "Merge LoCo with Zero++" (DeepSpeed PR #6730), Overview (error
feedback on 4-bit gradients); ZeROPlusPlus.md §1.2 (block int4, all-to-all
replacing reduce-scatter, full-precision reduce, intra- then inter-node).

What pins what:
  * hand-worked exact cases fix the error update (which term gets beta, the
    sign of c - d, where s enters) and the send order;
  * the telescoping identity sum_t d_t = sum_t g_t + e_0 - e_T (pure error
    feedback) ties codes, scales and error buffer together over several steps;
  * the LoCo recurrence bound ties the moving average to the quantization
    error;
  * the reduced shards approximate the exact sum of the ranks' gradient
    slices within the quantization error -- a wrong chunk, rank or
    permutation gives an O(|g|) error;
  * with one group the hierarchical first hop is the requantized flat reduce.
"""
import numpy as np
import pytest
import torch

from exact import unpack_int4
from weight_communication_gb300 import workloads as wl


def _bf16_bits(vals):
    return wl.as_u16(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)).copy()


def _deq(codes, scales, B):
    """fp64 dequantized values in code order (q * scale is exact in fp64)."""
    return unpack_int4(codes).astype(np.float64) * np.repeat(scales.astype(np.float64), B)


# --------------------------------------------------------------------------
# send order
# --------------------------------------------------------------------------

def test_send_position_tables(orc):
    # G = 1: identity
    assert [orc.send_position(k, 8, 1) for k in range(8)] == list(range(8))
    # R = 4 in 2 groups of 2: destination local rank 0 gets slices 0 and 2,
    # local rank 1 gets slices 1 and 3
    assert [orc.send_position(k, 4, 2) for k in range(4)] == [0, 2, 1, 3]
    # R = 8 in 2 groups of 4: slice g'*4 + l sits at position 2*l + g'
    assert [orc.send_position(k, 8, 2) for k in range(8)] == [0, 2, 4, 6, 1, 3, 5, 7]
    # R = 16 in 2 groups of 8 (the hierarchical workload)
    assert [orc.send_position(k, 16, 2) for k in range(16)] == \
        [0, 2, 4, 6, 8, 10, 12, 14, 1, 3, 5, 7, 9, 11, 13, 15]


@pytest.mark.parametrize("R,G", [(1, 1), (6, 3), (12, 4), (16, 2), (16, 16), (32, 4)])
def test_send_position_is_a_permutation(orc, R, G):
    pos = sorted(orc.send_position(k, R, G) for k in range(R))
    assert pos == list(range(R))


def test_codes_land_at_send_positions(orc):
    # R = 4, G = 2, one block per slice; slice k holds the constant k + 1, so
    # the block at chunk position p has absmax (slice + 1) and scale (slice+1)/7.
    B = 8
    R, G, N = 4, 2, 4 * 8
    g = _bf16_bits(np.repeat(np.arange(1, 5, dtype=np.float32), B))
    g = np.tile(g, R)
    codes, scales = orc.ef_quant_int4(g, None, N, R, G, B, 1.0, 0.0)
    per_rank = scales.reshape(R, 4)
    expect = np.array([1, 3, 2, 4], dtype=np.float32) / np.float32(7)
    for r in range(R):
        assert np.array_equal(per_rank[r], expect)
    assert np.all(unpack_int4(codes) == 7)


# --------------------------------------------------------------------------
# error update, worked exactly
# --------------------------------------------------------------------------

def test_error_update_worked_example(orc):
    # B = 2 blocks, every quantity a short dyadic rational so each operation
    # is exact:  c = g + s*e,  scale = m/7,  q = rint(c/scale),
    # e' = beta*e + (1-beta)*(c - q*scale).
    # s = 2, beta = 0.25:
    #   block 0: g = (7, 1), e = (0, 0.375) -> c = (7, 1.75), scale 1,
    #            q = (7, 2), c - d = (0, -0.25), e' = (0, 0.09375 - 0.1875)
    #   block 1: g = (-3, 0.5), e = (-0.5, 0.25) -> c = (-4, 1), scale 4/7,
    #            q = (-7, rint(1.75) = 2), d = (-4, 8/7 rounded)
    g = _bf16_bits([7.0, 1.0, -3.0, 0.5])
    e = np.array([0.0, 0.375, -0.5, 0.25], dtype=np.float32)
    codes, scales = orc.ef_quant_int4(g, e, 4, 1, 1, 2, 2.0, 0.25)
    q = unpack_int4(codes)
    assert q.tolist() == [7, 2, -7, 2]
    s1 = np.float32(4) / np.float32(7)
    assert scales.tolist() == [1.0, float(s1)]
    assert e[0] == 0.0
    assert e[1] == np.float32(-0.09375)
    assert e[2] == np.float32(0.25 * -0.5)            # c - d = 0 exactly
    d3 = np.float32(2) * s1
    assert e[3] == np.float32(np.float32(0.25 * 0.25) + np.float32(0.75) * np.float32(np.float32(1.0) - d3))


def test_plain_error_feedback_keeps_residual(orc):
    # s = 1, beta = 0: e' = c - d exactly when c - d is representable.
    g = _bf16_bits([7.0, 2.25, -1.0, 0.0])
    e = np.zeros(4, dtype=np.float32)
    codes, scales = orc.ef_quant_int4(g, e, 4, 1, 1, 4, 1.0, 0.0)
    assert unpack_int4(codes).tolist() == [7, 2, -1, 0]
    assert e.tolist() == [0.0, 0.25, 0.0, 0.0]
    # next step with zero gradient sends the stored residual
    g0 = _bf16_bits([0.0, 0.0, 0.0, 0.0])
    codes, scales = orc.ef_quant_int4(g0, e, 4, 1, 1, 4, 1.0, 0.0)
    assert scales[0] == np.float32(0.25) / np.float32(7)
    assert unpack_int4(codes).tolist() == [0, 7, 0, 0]


def test_error_update_rounds_as_stated(orc):
    """e' = fl(fl(beta*e) + fl(fl(1 - beta) * fl(c - d))): (1 - beta) is formed
    once and multiplies the residual.  Worked by hand, beta = 0.75, s = 1, B = 2:
      g = (2, 28), e = (-1 + 2^-23, 0)  ->  c = (1 + 2^-23, 28), exact;
      m = 28, scale = 4, inv = 0.25; c*inv = (0.25 + 2^-25, 7), q = (0, 7);
      residual r = 1 + 2^-23 and (1 - beta)*r = 0.25 + 2^-25, exact;
      beta*e = -0.75 + 1.5*2^-24 lies halfway between floats 2^-24 apart, and
      ties to even give -0.75 + 2^-23;
      e'_0 = -0.75 + 2^-23 + 0.25 + 2^-25 = -0.5 + 5*2^-25, exact.
    The algebraically equal r - beta*r rounds beta*r = 0.75 + 1.5*2^-24 to
    0.75 + 2^-23, leaves 0.25, and would give e'_0 = -0.5 + 2^-23."""
    g = _bf16_bits([2.0, 28.0])
    e = np.array([-1.0 + 2.0 ** -23, 0.0], dtype=np.float32)
    codes, scales = orc.ef_quant_int4(g, e, 2, 1, 1, 2, 1.0, 0.75)
    assert unpack_int4(codes).tolist() == [0, 7]
    assert scales.tolist() == [4.0]
    assert e[0] == np.float32(-0.5 + 5 * 2.0 ** -25)
    assert e[1] == 0.0


def test_compensation_rounds_the_product_first(orc):
    """c = fl(g + fl(s*e)).  With s = 3, e = 1 + 2^-23 and g = -3:
    s*e = 3 + 1.5*2^-22 lies halfway between floats 2^-22 apart, ties to even
    give 3 + 2^-21, and c = 2^-21 exactly (a fused multiply-add would give
    1.5*2^-22).  The block's maximum is then 2^-21, its scale fl(2^-21 / 7),
    and c quantizes to the code 7."""
    g = _bf16_bits([-3.0, 0.0])
    e = np.array([1.0 + 2.0 ** -23, 0.0], dtype=np.float32)
    codes, scales = orc.ef_quant_int4(g, e, 2, 1, 1, 2, 3.0, 0.0)
    assert unpack_int4(codes).tolist() == [7, 0]
    assert scales[0] == np.float32(2.0 ** -21) / np.float32(7)
    assert scales[0] != np.float32(1.5 * 2.0 ** -22) / np.float32(7)


def test_code_rounds_the_product_before_rint(orc):
    """q = rint(fl(c*inv)): the product is rounded to fp32 first.  Block
    (c0, m) = (1.5 + 5*2^-23, 7 + 3*2^-20), made exact as c = 0 + 1*e:
      inv = fl(7/m) = 1 - 7*2^-24 (7/m = 1 - 6.86*2^-24 + ...);
      c0*inv = 1.5 - 2^-25 - 35*2^-47 exactly, within half an ulp (2^-24) of
      1.5, so fl(c0*inv) = 1.5 and rint ties it to the even 2; rounding the
      exact product straight to an integer would give 1;
      m*inv = 7 - 2^-24 - ..., fl = 7, q = 7; scale = fl(m/7) = 1 + 3*2^-23."""
    c = np.array([1.5 + 5 * 2.0 ** -23, 7 + 3 * 2.0 ** -20], np.float32)
    g = _bf16_bits([0.0, 0.0])
    e = c.copy()
    codes, scales = orc.ef_quant_int4(g, e, 2, 1, 1, 2, 1.0, 0.0)
    assert unpack_int4(codes).tolist() == [2, 7]
    assert scales[0] == np.float32(1 + 3 * 2.0 ** -23)


def test_error_scale_zero_and_null_buffer_quantize_g_alone(orc):
    w = wl.QGZ_TINY.scaled(8192)
    g = wl.as_u16(wl.qgz_gradients(w, 0)).ravel().copy()
    c0, s0 = orc.ef_quant_int4(g, None, w.N, w.R, 1, w.B, 1.0, 0.0)
    zero_ef = np.zeros(g.size, np.float32)
    c1, s1 = orc.ef_quant_int4(g, zero_ef, w.N, w.R, 1, w.B, 1.0, 0.5)
    rng = np.random.default_rng(3)
    rand_ef = rng.standard_normal(g.size).astype(np.float32)
    c2, s2 = orc.ef_quant_int4(g, rand_ef, w.N, w.R, 1, w.B, 0.0, 0.5)
    for c, s in ((c1, s1), (c2, s2)):
        assert np.array_equal(c, c0) and np.array_equal(s, s0)


# --------------------------------------------------------------------------
# multi-step identities
# --------------------------------------------------------------------------

def test_telescoping_pure_error_feedback(orc):
    """sum_t d_t = sum_t g_t + e_0 - e_T elementwise (s = 1, beta = 0), to
    1e-5 relative, over the 3 steps of the 4-rank, 1M-element workload."""
    w = wl.QGZ_TINY
    assert (w.err_scale, w.err_beta) == (1.0, 0.0)
    e = np.zeros(w.R * w.N, np.float32)
    sum_d = np.zeros(w.R * w.N)
    sum_g = np.zeros(w.R * w.N)
    mag = np.zeros(w.R * w.N)
    for t in range(w.steps):
        gt = wl.qgz_gradients(w, t)
        gu = wl.as_u16(gt).ravel().copy()
        codes, scales = orc.ef_quant_int4(gu, e, w.N, w.R, w.G, w.B, 1.0, 0.0)
        d = _deq(codes, scales, w.B)               # G = 1: send order = gradient order
        gf = gt.float().numpy().ravel().astype(np.float64)
        sum_d += d
        sum_g += gf
        mag += np.abs(gf) + np.abs(e)
    lhs = sum_d
    rhs = sum_g - e.astype(np.float64)
    assert np.all(np.abs(lhs - rhs) <= 1e-5 * mag + 1e-30)
    # the identity is not vacuous: the residual carried is of quantization size
    assert np.abs(e).max() > 1e-6


@pytest.mark.parametrize("beta", [0.5, 0.25, 0.75])
def test_loco_recurrence_bound(orc, beta):
    """|e_t| <= beta |e_{t-1}| + (1 - beta) scale_t (1/2 + 2^-18), up to one
    rounding per operation; a swapped beta or a wrong sign breaks it."""
    w = wl.QGZ_SINGLE_HOP.scaled(1 << 16)
    e = np.zeros(w.R * w.N, np.float32)
    for t in range(4):
        gu = wl.as_u16(wl.qgz_gradients(w, t)).ravel().copy()
        e_prev = e.astype(np.float64).copy()
        codes, scales = orc.ef_quant_int4(gu, e, w.N, w.R, w.G, w.B, 1.0, beta)
        sc = np.repeat(scales.astype(np.float64), w.B)
        bound = beta * np.abs(e_prev) + (1 - beta) * sc * (0.5 + 2.0**-18)
        assert np.all(np.abs(e) <= bound * (1 + 2.0**-21))
        if t > 0:
            # with the moving average the old error survives: a swapped beta
            # (old error weighted 1 - beta) misses this tighter two-sided check
            c = wl.qgz_gradients(w, t).float().numpy().ravel().astype(np.float64) + e_prev
            d = _deq(codes, scales, w.B)
            pred = beta * e_prev + (1 - beta) * (c - d)
            assert np.all(np.abs(e - pred) <= 4 * 2.0**-24 * (np.abs(e_prev) + np.abs(c)) + 1e-38)


# --------------------------------------------------------------------------
# reductions
# --------------------------------------------------------------------------

def test_reduce_of_one_rank_is_dequantization(orc):
    w = wl.QGZ_TINY.scaled(4096)
    gu = wl.as_u16(wl.qgz_gradients(w, 0))[0].copy()
    codes, scales = orc.ef_quant_int4(gu, None, w.N, 1, 1, w.B, 1.0, 0.0)
    out = orc.dequant_reduce(codes, scales, w.N, 1, 1, w.B)
    d = _deq(codes, scales, w.B).astype(np.float32)
    assert np.array_equal(out.view(np.uint32), d.view(np.uint32))


@pytest.mark.parametrize("G,out_bf16", [(1, False), (2, True)])
def test_destination_ranges_tile_the_destination(orc, G, out_bf16):
    """Every output is its own sum, so the outputs [i0, i1) of a destination
    are exactly that part of the destination's result, for any split -- the
    all-cores CPU baseline relies on this."""
    R, N, B = 4, 4 * 6 * 64, 64
    g = wl.as_u16(wl.draw_bf16(R * N, 1e-3, 7)).copy()
    codes, scales = orc.ef_quant_int4(g, None, N, R, G, B, 1.0, 0.0)
    if G > 1:
        codes, scales = orc.dequant_reduce_requant(codes, scales, N, R, G, B)
    S = N // R
    for k in range(R):
        whole = orc.dequant_reduce_dest(codes, scales, N, R, G, B, k, 0.5, out_bf16)
        for cuts in ([0, S], [0, 64, S], [0, 0, 128, 320, S]):
            parts = [orc.dequant_reduce_dest_range(codes, scales, N, R, G, B, k, a, b, 0.5, out_bf16)
                     for a, b in zip(cuts[:-1], cuts[1:])]
            got = np.concatenate(parts)
            assert got.dtype == whole.dtype and np.array_equal(got.view(np.uint8), whole.view(np.uint8))
    with pytest.raises(ValueError):
        orc.dequant_reduce_dest_range(codes, scales, N, R, G, B, 0, 10, 5)


def test_identical_ranks_sum_to_r_times_d(orc):
    R, N, B = 8, 8 * 512, 256
    one = wl.as_u16(wl.draw_bf16(N, 1e-3, 11)).copy()
    g = np.tile(one, R)
    codes, scales = orc.ef_quant_int4(g, None, N, R, 1, B, 1.0, 0.0)
    out = orc.dequant_reduce(codes, scales, N, R, 1, B).astype(np.float64)
    d = _deq(codes[: N // 2], scales[: N // B], B)        # rank 0, in send order
    # R = 8: d + d + ... is exact at every power of two and rounds in between
    assert np.all(np.abs(out - R * d) <= R * 2.0**-24 * np.abs(R * d))
    avg = orc.dequant_reduce(codes, scales, N, R, 1, B, out_scale=1.0 / R).astype(np.float64)
    assert np.all(np.abs(avg - d) <= R * 2.0**-24 * np.abs(d))


@pytest.mark.parametrize("R,B", [(4, 256), (8, 256), (3, 64), (8, 512)])
def test_flat_reduce_approximates_sum_of_slices(orc, R, B):
    N = R * B * 5
    w = wl.QgzWorkload(9, "t", R, N, 1, B, 1.0, 0.0, 1, 1e-3, 1e-3, 100.0, False)
    gt = wl.qgz_gradients(w, 0)
    gu = wl.as_u16(gt).ravel().copy()
    codes, scales = orc.ef_quant_int4(gu, None, N, R, 1, B, 1.0, 0.0)
    out = orc.dequant_reduce(codes, scales, N, R, 1, B).astype(np.float64)
    gsum = gt.double().sum(0).numpy()                      # exact enough in fp64
    sc = scales.reshape(R, N // B).astype(np.float64)
    err_bound = np.repeat(sc.sum(0), B) * (0.5 + 2.0**-18) + R * 2.0**-23 * gt.double().abs().sum(0).numpy()
    assert np.all(np.abs(out - gsum) <= err_bound)
    wrong = np.roll(out.reshape(R, -1), 1, axis=0).ravel()
    assert np.any(np.abs(wrong - gsum) > err_bound)
    # destination k alone equals slice k of the full call
    S = N // R
    for k in range(R):
        one = orc.dequant_reduce_dest(codes, scales, N, R, 1, B, k)
        assert np.array_equal(one, out[k * S:(k + 1) * S].astype(np.float32))
    # bf16 output is the round-to-nearest of the fp32 one
    ob = orc.dequant_reduce(codes, scales, N, R, 1, B, out_bf16=True)
    assert np.array_equal(ob, orc.bf16_round(out.astype(np.float32)))


@pytest.mark.parametrize("R,G,B", [(8, 2, 32), (16, 2, 512), (12, 3, 64), (8, 4, 128)])
def test_hierarchical_reduce_approximates_sum(orc, R, G, B):
    """Concatenated final shards (rank order) approximate sum_r g_r within the
    first quantization (sum of the ranks' scales / 2), the requantization
    (its scale / 2) and the bf16 rounding; a wrong permutation anywhere gives
    an error of the size of the gradients."""
    L = R // G
    N = R * B * 3
    S = N // R
    w = wl.QgzWorkload(9, "t", R, N, G, B, 1.0, 0.0, 1, 1e-3, 1e-3, 100.0, True)
    gt = wl.qgz_gradients(w, 0)
    gu = wl.as_u16(gt).ravel().copy()
    codes, scales = orc.ef_quant_int4(gu, None, N, R, G, B, 1.0, 0.0)
    c1, s1 = orc.dequant_reduce_requant(codes, scales, N, R, G, B)
    out = orc.dequant_reduce(c1, s1, N, R, G, B, out_bf16=True)
    outf = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    gsum = gt.double().sum(0).numpy()
    # bound per element: hop-1 quantization of every rank, hop-1 requant of
    # every group's partial sum, bf16 rounding of the result
    sc = scales.reshape(R, N // B).astype(np.float64)
    # first-quantization scales in gradient order: rank r's slice k lies at
    # send position p(k), blocks of slice k are [p*S/B, (p+1)*S/B)
    sc_grad = np.zeros((R, N // B))
    for k in range(R):
        p = orc.send_position(k, R, G)
        sc_grad[:, k * S // B:(k + 1) * S // B] = sc[:, p * S // B:(p + 1) * S // B]
    q1 = np.repeat(sc_grad.sum(0), B) * (0.5 + 2.0**-18)
    # requant scales: slice k = g*L + l is sub-slice g of unit (g', l), for every g'
    s1u = s1.reshape(R, G, S // B).astype(np.float64)
    q2 = np.zeros(N)
    for k in range(R):
        g, l = divmod(k, L)
        for gq in range(G):
            q2[k * S:(k + 1) * S] += np.repeat(s1u[gq * L + l, g], B) * (0.5 + 2.0**-18)
    rnd = np.abs(gsum) * 2.0**-8 + 8 * R * 2.0**-24 * gt.double().abs().sum(0).numpy()
    bound = q1 + q2 + rnd + 1e-30
    assert np.all(np.abs(outf - gsum) <= bound)
    # the bound is tight enough to reject a result with its shards permuted
    wrong = np.roll(outf.reshape(R, S), 1, axis=0).ravel()
    assert np.any(np.abs(wrong - gsum) > bound)
    # hop 1 on its own: unit (g, l) sub-slice g' approximates the sum, over
    # the L ranks of group g only, of slice g'*L + l
    gg = gt.double().numpy()
    for g in range(G):
        for l in range(L):
            u = g * L + l
            dq = _deq(c1[u * G * S // 2:(u + 1) * G * S // 2],
                      s1[u * G * S // B:(u + 1) * G * S // B], B)
            for gq in range(G):
                k = gq * L + l
                part = gg[g * L:(g + 1) * L, k * S:(k + 1) * S]
                b1 = np.repeat(sc_grad[g * L:(g + 1) * L, k * S // B:(k + 1) * S // B].sum(0), B)
                b2 = np.repeat(s1u[u, gq], B)
                lim = (b1 + b2) * (0.5 + 2.0**-18) + 8 * L * 2.0**-24 * np.abs(part).sum(0) + 1e-30
                err = np.abs(dq[gq * S:(gq + 1) * S] - part.sum(0))
                assert np.all(err <= lim), (g, l, gq)
    # per-unit and per-destination forms agree with the whole-buffer calls
    for g in range(G):
        for l in range(L):
            u = g * L + l
            cu, su = orc.dequant_reduce_requant_unit(codes, scales, N, R, G, B, g, l)
            assert np.array_equal(cu, c1[u * G * S // 2:(u + 1) * G * S // 2])
            assert np.array_equal(su, s1[u * G * S // B:(u + 1) * G * S // B])
    for k in range(R):
        ok = orc.dequant_reduce_dest(c1, s1, N, R, G, B, k, out_bf16=True)
        assert np.array_equal(ok, out[k * S:(k + 1) * S])


def test_one_group_first_hop_is_requantized_flat_reduce(orc):
    R, B = 8, 256
    N = R * B * 4
    w = wl.QgzWorkload(9, "t", R, N, 1, B, 1.0, 0.0, 1, 1e-3, 1e-3, 100.0, False)
    gu = wl.as_u16(wl.qgz_gradients(w, 0)).ravel().copy()
    codes, scales = orc.ef_quant_int4(gu, None, N, R, 1, B, 1.0, 0.0)
    flat = orc.dequant_reduce(codes, scales, N, R, 1, B)
    c1, s1 = orc.dequant_reduce_requant(codes, scales, N, R, 1, B)
    for b in range(N // B):
        q, s = orc.quant_block(flat[b * B:(b + 1) * B], 7)
        assert s == s1[b]
        assert np.array_equal(q, unpack_int4(c1[b * B // 2:(b + 1) * B // 2]))


def test_requantization_is_idempotent(orc):
    rng = np.random.default_rng(5)
    for _ in range(200):
        x = (rng.standard_normal(256) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        q, s = orc.quant_block(x, 7)
        d = (q.astype(np.float32) * np.float32(s)).astype(np.float32)
        q2, s2 = orc.quant_block(d, 7)
        assert np.array_equal(q, q2)
        assert abs(s2 - s) <= 2 * np.spacing(np.float32(s))


# --------------------------------------------------------------------------
# summation order, worked by hand
# --------------------------------------------------------------------------
# Three terms 1, 2^-24, 2^-24 added in source order: 1 + 2^-24 is a tie
# between 1 and 1 + 2^-23 and rounds to the even 1, twice, so the sum is 1.
# In the opposite order the two small terms first make 2^-23 and the sum is
# 1 + 2^-23.  Every code is 1 (byte 0x11) and the block scales carry the
# terms, so each dequantized value is exactly its scale.

ONE, TINY = np.float32(1.0), np.float32(2.0**-24)


def test_order_example_is_not_vacuous():
    assert np.float32(np.float32(ONE + TINY) + TINY) == ONE
    assert np.float32(ONE + np.float32(TINY + TINY)) == np.float32(1 + 2.0**-23)


def test_flat_reduce_adds_ranks_in_order(orc):
    R, B = 3, 32
    N = R * B                                   # S = B: one block per chunk
    codes = np.full(R * N // 2, 0x11, np.uint8)
    scales = np.ones(R * N // B, np.float32)    # rank r, chunk k: block r*(N/B) + k
    scales[[0, 3, 6]] = [ONE, TINY, TINY]       # chunk 0 of ranks 0, 1, 2
    out = orc.dequant_reduce(codes, scales, N, R, 1, B)
    assert np.all(out[:B] == ONE)
    assert np.all(out[B:] == np.float32(3.0))


def test_second_hop_adds_groups_in_order(orc):
    R, G, B = 3, 3, 32                          # one rank per group
    N = R * B
    codes = np.full(G * N // 2, 0x11, np.uint8)
    scales = np.ones(G * N // B, np.float32)    # unit gq, sub-slice g: block gq*G + g
    scales[[0, 3, 6]] = [ONE, TINY, TINY]       # sub-slice 0 from groups 0, 1, 2
    out = orc.dequant_reduce(codes, scales, N, R, G, B)
    assert np.all(out[:B] == ONE)
    assert np.all(out[B:] == np.float32(3.0))


def test_first_hop_adds_local_ranks_in_order(orc):
    R, G, B = 3, 1, 32                          # three local ranks, one group
    N = R * B
    codes = np.full(R * N // 2, 0x11, np.uint8)
    scales = np.ones(R * N // B, np.float32)
    scales[[0, 3, 6]] = [ONE, TINY, TINY]       # chunk 0 of local ranks 0, 1, 2
    oc, os_ = orc.dequant_reduce_requant(codes, scales, N, R, G, B)
    # unit 0's partial sums are all exactly 1: scale fl(1/7), every code 7
    assert os_[0] == ONE / np.float32(7)
    assert os_[0] != np.float32(1 + 2.0**-23) / np.float32(7)
    assert np.all(oc[:B // 2] == 0x77)


@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_reduce_sums_start_at_positive_zero(orc, G, out_bf16):
    """Every reduce sum starts at +0 (IEEE: +0 + -0 = +0 when rounding to
    nearest).  Codes of -7 with scales of +0, and codes of +1 with scales of
    -0, give products of -0 from every source. Their sums, flat or over the
    second hop's groups, must be +0, whose encoding is all zero bits, not -0."""
    R, B = 4, 32
    N = R * B * 2
    nsrc = R if G == 1 else G
    codes = np.full(nsrc * N // 2, 0x99, np.uint8)   # nibble 9: the code -7
    scales = np.zeros(nsrc * N // B, np.float32)      # +0
    codes[: N // 4] = 0x11                            # the code +1 ...
    scales[: N // (4 * B)] = np.float32(-0.0)         # ... with scale -0
    assert np.signbit(np.float32(-7) * scales[-1]) and np.signbit(np.float32(1) * scales[0])
    out = orc.dequant_reduce(codes, scales, N, R, G, B, 1.0, out_bf16)
    assert not out.view(np.uint16 if out_bf16 else np.uint32).any(), "a sum came out as -0"


def test_output_scale_applies_before_bf16_rounding(orc):
    """out = bf16_rn(fl(sum * out_scale)), flat and second hop: codes 7 at
    scale 1 sum to 7 per source; with out_scale 0.5 one source gives 3.5
    (bf16 0x4060) and two give 7 (0x40E0), never the unscaled 7 and 14."""
    one = orc.dequant_reduce(np.full(1, 0x77, np.uint8), np.ones(1, np.float32), 2, 1, 1, 2,
                             0.5, True)
    assert one.tolist() == [0x4060, 0x4060]
    two = orc.dequant_reduce(np.full(4, 0x77, np.uint8), np.ones(4, np.float32), 4, 2, 2, 2,
                             0.5, True)
    assert two.tolist() == [0x40E0] * 4

