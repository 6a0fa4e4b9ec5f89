"""Pins for the oracle's extensions beyond the basic path:

  * error feedback on the first hop's requantization ("Merge LoCo with
    Zero++", review thread: `inter_ef_buf`, the error buffer of the
    inter-node message) -- a hand-worked exact case, zero error = plain hop,
    the telescoping identity over steps with plain error feedback, and the
    LoCo recurrence bound;
  * a bf16 error buffer (the memory LoCo costs, "Merge LoCo with Zero++",
    Overview) -- one step equals the fp32-buffer step with only the stored
    error rounded to bf16 by torch's conversion; over several steps the
    telescoping identity holds up to the bf16 storage rounding;
  * an int8 error buffer (a quarter of the fp32 buffer's memory) -- a
    hand-worked two-step example, one step equal to the fp32-buffer step with
    the stored error quantized by the pinned int8 block rule (in gradient
    order, also with groups), and the telescoping identity up to the int8
    storage error;
  * qwZ quantization with the bf16 replica written alongside
    (ZeROPlusPlus.md §1.2) -- equal to quantize then dequantize.
"""
import numpy as np
import pytest
import torch

from exact import unpack_int4
from weight_communication_gb300 import workloads as wl


def _deq(codes, scales, B):
    return unpack_int4(codes).astype(np.float64) * np.repeat(scales.astype(np.float64), B)


def _bf16(vals):
    return wl.as_u16(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)).copy()


# --------------------------------------------------------------------------
# first-hop error feedback
# --------------------------------------------------------------------------

def test_first_hop_error_feedback_worked_example(orc):
    # R = 2 ranks, one group (L = 2), B = S = 2, N = 4.  Unit (0, 0) adds
    # chunk 0 of both ranks: rank 0 codes (7, 1), rank 1 codes (0, 2), scale 1
    # -> partial sums p = (7, 3).  With e1 = (0, 0.25), s = 2, beta = 0.25:
    # c = (7, 3.5), absmax 7 -> scale 1, q = (7, rint(3.5) = 4), d = (7, 4),
    # c - d = (0, -0.5), e1' = (0, 0.25*0.25 + 0.75*(-0.5)) = (0, -0.3125).
    codes = np.array([0x17, 0x00, 0x20, 0x00], np.uint8)
    scales = np.ones(4, np.float32)
    e1 = np.array([0.0, 0.25], np.float32)
    oc, os_ = orc.dequant_reduce_requant_unit_ef(codes, scales, 4, 2, 1, 2, 0, 0, e1, 2.0, 0.25)
    assert unpack_int4(oc).tolist() == [7, 4]
    assert os_.tolist() == [1.0]
    assert e1.tolist() == [0.0, -0.3125]
    # without the error buffer: p = (7, 3) quantizes to (7, 3)
    oc0, _ = orc.dequant_reduce_requant_unit(codes, scales, 4, 2, 1, 2, 0, 0)
    assert unpack_int4(oc0).tolist() == [7, 3]


def _hop0(orc, w, t):
    g = wl.as_u16(wl.qgz_gradients(w, t)).ravel().copy()
    return orc.ef_quant_int4(g, None, w.N, w.R, w.G, w.B, 1.0, 0.0)


def _partial_sums(codes, scales, w, magnitude=False):
    """fp64 sums (or sums of magnitudes), over the L ranks of each group, of
    the chunks every unit receives, in the unit-major [R][G][S] layout of the
    first hop's output."""
    R, N, G, L, S, B = w.R, w.N, w.G, w.L, w.S, w.B
    d = _deq(codes, scales, B).reshape(R, N)
    if magnitude:
        d = np.abs(d)
    p = np.zeros((R, G, S))
    for g in range(G):
        for l in range(L):
            for gq in range(G):
                ch = (l * G + gq) * S
                p[g * L + l, gq] = d[g * L:(g + 1) * L, ch:ch + S].sum(0)
    return p.ravel()


def test_first_hop_error_feedback_zero_buffer_is_plain(orc):
    w = wl.QgzWorkload(9, "t", 8, 8 * 256 * 3, 2, 256, 1.0, 0.5, 1, 1e-3, 1e-3, 100.0, True)
    codes, scales = _hop0(orc, w, 0)
    plain_c, plain_s = orc.dequant_reduce_requant(codes, scales, w.N, w.R, w.G, w.B)
    e1 = np.zeros(w.G * w.N, np.float32)
    c1, s1 = orc.dequant_reduce_requant_ef(codes, scales, w.N, w.R, w.G, w.B, e1, 1.0, 0.5)
    assert np.array_equal(c1, plain_c) and np.array_equal(s1, plain_s)
    c2, s2 = orc.dequant_reduce_requant_ef(codes, scales, w.N, w.R, w.G, w.B, None, 1.0, 0.5)
    assert np.array_equal(c2, plain_c) and np.array_equal(s2, plain_s)
    # the unit form matches the whole-buffer form
    e_a = np.zeros(w.G * w.N, np.float32)
    ca, sa = orc.dequant_reduce_requant_ef(codes, scales, w.N, w.R, w.G, w.B, e_a, 1.0, 0.5)
    unit = w.G * w.S
    for u in range(w.R):
        g, l = divmod(u, w.L)
        eu = np.zeros(unit, np.float32)
        cu, su = orc.dequant_reduce_requant_unit_ef(codes, scales, w.N, w.R, w.G, w.B, g, l,
                                                    eu, 1.0, 0.5)
        assert np.array_equal(cu, ca[u * unit // 2:(u + 1) * unit // 2])
        assert np.array_equal(eu, e_a[u * unit:(u + 1) * unit])


def test_first_hop_telescoping(orc):
    """Plain error feedback on the requantization (s = 1, beta = 0): the
    requantized values sent over T steps add up to the partial sums received
    plus e1_0 - e1_T."""
    w = wl.QgzWorkload(9, "t", 8, 8 * 512 * 2, 2, 512, 1.0, 0.0, 1, 1e-3, 1e-3, 100.0, True)
    e1 = np.zeros(w.G * w.N, np.float32)
    sum_d = np.zeros(w.G * w.N)
    sum_p = np.zeros(w.G * w.N)
    mag = np.zeros(w.G * w.N)
    for t in range(4):
        codes, scales = _hop0(orc, w, t)
        p = _partial_sums(codes, scales, w)
        c1, s1 = orc.dequant_reduce_requant_ef(codes, scales, w.N, w.R, w.G, w.B, e1, 1.0, 0.0)
        sum_d += _deq(c1, s1, w.B)
        sum_p += p
        mag += np.abs(p) + np.abs(e1)
    assert np.all(np.abs(sum_d - (sum_p - e1)) <= 1e-5 * mag + 1e-30)
    assert np.abs(e1).max() > 0


@pytest.mark.parametrize("s,beta", [(1.0, 0.5), (0.7, 0.3)])
def test_first_hop_error_feedback_is_the_ranks_error_feedback_chain(orc, s, beta):
    """On partial sums that are exactly bf16 values, a unit's first hop with
    error feedback computes what the ranks' EF-quant computes on a gradient
    equal to those sums: the same compensation, block quantization and error
    update, rounded in the same order (pinned by hand-worked cases of its own).
    Codes in [-7, 7] at power-of-two scales 2^-12 .. 2^-8 make every sum of
    the two local ranks exact and bf16-representable.  The errors are full
    24-bit fp32 values, and s = 0.7, beta = 0.3 are not dyadic, so any other
    rounding order shows in many elements."""
    R, G, B, k = 4, 2, 64, 8
    L = R // G
    N = R * B * k
    S = N // R
    rng = np.random.default_rng(int(s * 10) + 7)
    q = rng.integers(-7, 8, size=R * N)
    codes = np.zeros(R * N // 2, np.uint8)
    codes[:] = (q[0::2] & 15) | ((q[1::2] & 15) << 4)
    scales = (2.0 ** -rng.integers(8, 13, size=R * N // B)).astype(np.float32)
    d = q.astype(np.float64) * np.repeat(scales.astype(np.float64), B)
    for g in range(G):
        for l in range(L):
            # partial sums of unit (g, l): sub-slice gq adds chunk l*G + gq of
            # the group's ranks, in local-rank order
            p = np.concatenate([sum(d[(g * L + lq) * N + (l * G + gq) * S:
                                      (g * L + lq) * N + (l * G + gq + 1) * S] for lq in range(L))
                                for gq in range(G)])
            p_bf16 = _bf16(p.tolist())
            assert np.array_equal(torch.from_numpy(p_bf16.view(np.int16)).view(torch.bfloat16)
                                  .float().numpy().astype(np.float64), p)
            e_start = (rng.standard_normal(G * S) * 1e-3).astype(np.float32)
            e_hop = e_start.copy()
            c1, s1 = orc.dequant_reduce_requant_unit_ef(codes, scales, N, R, G, B, g, l, e_hop,
                                                        s, beta)
            e_ref = e_start.copy()
            c0, s0 = orc.ef_quant_int4(p_bf16, e_ref, G * S, 1, 1, B, s, beta)
            assert np.array_equal(c1, c0) and np.array_equal(s1, s0), (g, l)
            assert np.array_equal(e_hop.view(np.uint32), e_ref.view(np.uint32)), (g, l)


@pytest.mark.parametrize("beta", [0.25, 0.5])
def test_first_hop_loco_bound(orc, beta):
    w = wl.QgzWorkload(9, "t", 8, 8 * 256 * 2, 2, 256, 1.0, beta, 1, 1e-3, 1e-3, 100.0, True)
    e1 = np.zeros(w.G * w.N, np.float32)
    for t in range(3):
        codes, scales = _hop0(orc, w, t)
        prev = e1.astype(np.float64).copy()
        p = _partial_sums(codes, scales, w)
        pm = _partial_sums(codes, scales, w, magnitude=True)
        c1, s1 = orc.dequant_reduce_requant_ef(codes, scales, w.N, w.R, w.G, w.B, e1, 1.0, beta)
        sc = np.repeat(s1.astype(np.float64), w.B)
        bound = beta * np.abs(prev) + (1 - beta) * sc * (0.5 + 2.0**-18)
        assert np.all(np.abs(e1) <= bound * (1 + 2.0**-20) + 1e-38)
        # two-sided: which term beta multiplies; the fp32 partial sum rounds
        # against the magnitude of its L terms
        pred = beta * prev + (1 - beta) * (p + prev - _deq(c1, s1, w.B))
        assert np.all(np.abs(e1 - pred) <= 8 * 2.0**-24 * (w.L * pm + np.abs(prev)) + 1e-38)


# --------------------------------------------------------------------------
# bf16 error buffer
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n_blocks,params", [
    (4, ((1.0, 0.5), (1.0, 0.0), (0.5, 0.25))),
    # s and beta that are not dyadic: another rounding order of the chain
    # changes the fp32 error by an ulp in many elements, and over 2 M elements
    # some of those changes cross a bf16 rounding boundary
    (128, ((0.7, 0.3),)),
])
def test_bf16_error_buffer_one_step_equals_rounded_fp32(orc, n_blocks, params):
    w = wl.QGZ_SINGLE_HOP.scaled(8 * 256 * n_blocks)
    g = wl.as_u16(wl.qgz_gradients(w, 0)).ravel().copy()
    rng = np.random.default_rng(4)
    e_start = torch.from_numpy((rng.standard_normal(w.R * w.N) * 1e-4).astype(np.float32)) \
        .to(torch.bfloat16)
    e16 = wl.as_u16(e_start).copy()
    e32 = e_start.float().numpy().copy()
    for s, beta in params:
        a16, a32 = e16.copy(), e32.copy()
        c16, s16 = orc.ef_quant_int4_bf16ef(g, a16, w.N, w.R, w.G, w.B, s, beta)
        c32, s32 = orc.ef_quant_int4(g, a32, w.N, w.R, w.G, w.B, s, beta)
        assert np.array_equal(c16, c32) and np.array_equal(s16, s32)
        want = wl.as_u16(torch.from_numpy(a32).to(torch.bfloat16))
        assert np.array_equal(a16, want)


def test_bf16_error_buffer_worked_example(orc):
    # the fp32 worked example's first three errors are bf16-representable
    g = _bf16([7.0, 1.0, -3.0, 0.5])
    e16 = _bf16([0.0, 0.375, -0.5, 0.25])
    codes, scales = orc.ef_quant_int4_bf16ef(g, e16, 4, 1, 1, 2, 2.0, 0.25)
    assert unpack_int4(codes).tolist() == [7, 2, -7, 2]
    back = (e16.astype(np.uint32) << 16).view(np.float32)
    assert back[:3].tolist() == [0.0, -0.09375, -0.125]


def test_bf16_error_buffer_telescoping_up_to_storage_rounding(orc):
    w = wl.QGZ_TINY.scaled(4 * 256 * 64)
    e16 = np.zeros(w.R * w.N, np.uint16)
    sum_d = np.zeros(w.R * w.N)
    sum_g = np.zeros(w.R * w.N)
    slack = np.zeros(w.R * w.N)
    for t in range(4):
        gt = wl.qgz_gradients(w, t)
        g = wl.as_u16(gt).ravel().copy()
        codes, scales = orc.ef_quant_int4_bf16ef(g, e16, w.N, w.R, w.G, w.B, 1.0, 0.0)
        e_now = (e16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        sum_d += _deq(codes, scales, w.B)
        sum_g += gt.double().numpy().ravel()
        slack += np.abs(e_now) * 2.0**-8 + 1e-5 * (np.abs(gt.double().numpy().ravel()) + np.abs(e_now))
    e_T = (e16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.abs(sum_d - (sum_g - e_T)) <= slack + 1e-30)


# --------------------------------------------------------------------------
# int8 error buffer
# --------------------------------------------------------------------------

def _int8_error(e8, e8s, B):
    """fp64 view of an int8 error buffer: code * scale (exact in fp64)."""
    return e8.astype(np.float64) * np.repeat(e8s.astype(np.float64), B)


def test_int8_error_buffer_worked_example(orc):
    # B = 32, s = 1, beta = 0.5, one block: g = 7, 3.25, -1.5, 0, ...
    B = 32
    g = _bf16([7.0, 3.25, -1.5] + [0.0] * (B - 3))
    e8 = np.zeros(B, np.int8)
    e8s = np.zeros(1, np.float32)
    # step 1 from a zero buffer: m = 7, scale = inv = 1, codes rint(g) with
    # -1.5 -> -2 (ties to even); c - d = 0, 0.25, 0.5, so the new error is
    # 0, 0.125, 0.25; stored with m' = 0.25: inv = 127/0.25 = 508 exactly,
    # codes rint(0, 63.5, 127) = 0, 64 (tie to even), 127
    codes, scales = orc.ef_quant_int4_int8ef(g, e8, e8s, B, 1, 1, B, 1.0, 0.5)
    assert unpack_int4(codes)[:4].tolist() == [7, 3, -2, 0] and scales[0] == 1.0
    assert e8[:4].tolist() == [0, 64, 127, 0] and not e8[4:].any()
    assert e8s[0] == np.float32(0.25) / np.float32(127)
    # step 2, same g: the error reads back as about 0, 0.126, 0.25, so
    # c = 7, 3.376, -1.25 and the codes are 7, 3, -1; the new error
    # 0.5 e + 0.5 (c - d) is about 0, 0.251 and 0.5 * 0.25 + 0.5 * -0.25 = 0
    # (to within the rounding of 127 * fl(0.25/127), some 1e-8), stored
    # against its own maximum 0.251: codes 0, 127, 0
    codes, scales = orc.ef_quant_int4_int8ef(g, e8, e8s, B, 1, 1, B, 1.0, 0.5)
    assert unpack_int4(codes)[:4].tolist() == [7, 3, -1, 0]
    assert e8[:4].tolist() == [0, 127, 0, 0]
    assert 0.25 < e8s[0] * 127 < 0.252


@pytest.mark.parametrize("G,n_blocks,params", [
    (1, 3, ((1.0, 0.5), (0.5, 0.25))),
    (2, 3, ((1.0, 0.5), (0.5, 0.25))),
    # not dyadic: over 2 M elements some ulp changes of the fp32 error from
    # another rounding order cross an int8 rounding boundary
    (1, 128, ((0.7, 0.3),)),
])
def test_int8_error_buffer_one_step_equals_quantized_fp32(orc, G, n_blocks, params):
    """From the same stored error, one step gives the fp32-buffer step's codes
    and scales, and stores exactly the int8 block quantization (the pinned
    qwZ rule) of the fp32 step's new error, block by block in gradient order."""
    R, B = 8, 256
    w = wl.QgzWorkload(9, "t", R, R * B * n_blocks, G, B, 1.0, 0.5, 1, 1e-3, 1e-3, 100.0, False)
    g = wl.as_u16(wl.qgz_gradients(w, 0)).ravel().copy()
    rng = np.random.default_rng(G)
    e8 = rng.integers(-127, 128, size=R * w.N).astype(np.int8)
    e8s = (rng.random(R * w.N // B) * 1e-6).astype(np.float32)
    e32 = (e8.astype(np.float32) * np.repeat(e8s, B)).astype(np.float32)   # code * scale, one rounding
    for s, beta in params:
        a8, a8s, a32 = e8.copy(), e8s.copy(), e32.copy()
        c8, s8 = orc.ef_quant_int4_int8ef(g, a8, a8s, w.N, R, G, B, s, beta)
        c32, s32 = orc.ef_quant_int4(g, a32, w.N, R, G, B, s, beta)
        assert np.array_equal(c8, c32) and np.array_equal(s8, s32)
        for b in range(R * w.N // B):
            q, sc = orc.quant_block(a32[b * B:(b + 1) * B], 127)
            assert np.array_equal(a8[b * B:(b + 1) * B], q) and a8s[b] == sc, b


def test_int8_error_buffer_telescoping_up_to_storage_error(orc):
    """Plain error feedback (s = 1, beta = 0): the dequantized values sum to
    the gradients minus the last stored error, up to the int8 storage error
    (at most half a storage step per element and step)."""
    w = wl.QGZ_TINY.scaled(4 * 256 * 64)
    B = w.B
    e8 = np.zeros(w.R * w.N, np.int8)
    e8s = np.zeros(w.R * w.N // B, np.float32)
    sum_d = np.zeros(w.R * w.N)
    sum_g = np.zeros(w.R * w.N)
    slack = np.zeros(w.R * w.N)
    for t in range(4):
        gt = wl.qgz_gradients(w, t)
        g = wl.as_u16(gt).ravel().copy()
        e_before = _int8_error(e8, e8s, B)
        codes, scales = orc.ef_quant_int4_int8ef(g, e8, e8s, w.N, w.R, w.G, B, 1.0, 0.0)
        sum_d += _deq(codes, scales, B)
        sum_g += gt.double().numpy().ravel()
        slack += (np.repeat(e8s.astype(np.float64), B) * (0.5 + 2.0**-18)
                  + 1e-5 * (np.abs(gt.double().numpy().ravel()) + np.abs(e_before)))
    e_T = _int8_error(e8, e8s, B)
    assert np.all(np.abs(sum_d - (sum_g - e_T)) <= slack + 1e-30)
    assert np.any(e8 != 0)


# --------------------------------------------------------------------------
# qwZ with the bf16 replica
# --------------------------------------------------------------------------

def test_qwz_replica_is_quantize_then_dequantize(orc):
    w = wl.as_u16(wl.draw_bf16(2048 * 6, 0.02, 8)).copy()
    codes, scales, rep = orc.qwz_quant_replica_int8(w, 2048)
    c2, s2 = orc.qwz_quant_int8(w, 2048)
    assert np.array_equal(codes, c2) and np.array_equal(scales, s2)
    assert np.array_equal(rep, orc.qwz_dequant_int8(c2, s2, 2048))
