"""GPU parity of the qgZ kernels (through the C ABI) against the CPU oracle.

Inputs are seeded bf16 gradients (normal with sparse outliers, as the
Llama-2 layer workloads) plus hand-made edge blocks; both sides get the same
bytes.  Sizes span many warp tiles with ragged tails, every supported block
size, flat and grouped send orders, with and without error feedback, and the
multi-step error-feedback recurrence.  Full-size runs of the three qgZ
workloads are in test_parity_fullsize.py.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (assert_bf16_parity, assert_bits_equal, assert_f32_parity, deq_magnitude,
                      dev, to_dev, to_host)
from weight_communication_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

ORC = oracle.get()


def edge_gradients(R: int, N: int, B: int, seed: int) -> np.ndarray:
    """[R*N] bf16 bits: seeded values with outliers, with some blocks replaced
    by edge cases -- all zero, signed zeros, subnormal, at the zero-block
    threshold 7*2^-126 and just below it, exact rounding ties, huge values."""
    g = wl.as_u16(wl.draw_bf16(R * N, 1e-3, seed, outlier_frac=1e-3, outlier_mult=100.0)).copy()
    nb = R * N // B
    rng = np.random.default_rng(seed)
    tiny = np.float32(np.finfo(np.float32).tiny)
    specials = [
        np.zeros(B, np.float32),
        np.where(np.arange(B) % 2 == 0, np.float32(0.0), np.float32(-0.0)),
        np.float32(1e-39) * rng.standard_normal(B).astype(np.float32),       # subnormal
        np.concatenate([[np.float32(7) * tiny], rng.uniform(-1, 1, B - 1).astype(np.float32) * tiny]),
        np.concatenate([[np.float32(6) * tiny], np.zeros(B - 1, np.float32)]),
        np.concatenate([[np.float32(7.0)], (np.arange(B - 1) % 15 - 7 + 0.5).astype(np.float32)]),
        np.concatenate([[np.float32(-7.0)], (np.arange(B - 1) % 13 - 6.5).astype(np.float32)]),
        rng.standard_normal(B).astype(np.float32) * np.float32(1e30),
    ]
    picks = rng.choice(nb, size=min(nb, 3 * len(specials)), replace=False)
    for j, b in enumerate(picks):
        blk = torch.from_numpy(specials[j % len(specials)].astype(np.float32)).to(torch.bfloat16)
        g[b * B:(b + 1) * B] = wl.as_u16(blk)
    return g


def gpu_ef_quant(g_u16, ef, N, R, G, B, s, beta, dev):
    gd = to_dev(g_u16, dev)
    efd = to_dev(ef, dev) if ef is not None else None
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    binding.ef_quant_int4(gd, efd, codes, scales, N, R, G, B, s, beta)
    torch.cuda.synchronize()
    return to_host(codes), to_host(scales), (to_host(efd) if efd is not None else None)


CASES = [
    # R, N, G, B, s, beta, with_ef
    (4, 4 * 256 * 37, 1, 256, 1.0, 0.0, True),
    (8, 8 * 256 * 11, 1, 256, 1.0, 0.5, True),
    (3, 3 * 512 * 7, 1, 512, 1.0, 0.5, True),
    (16, 16 * 512 * 3, 2, 512, 1.0, 0.5, True),
    (6, 6 * 1024 * 2, 3, 1024, 0.75, 0.25, True),
    (8, 8 * 128 * 9, 4, 128, 2.0, 0.5, True),
    (4, 4 * 64 * 13, 2, 64, 1.0, 0.5, True),       # 2 blocks per warp tile, ragged tail
    (2, 2 * 32 * 7, 1, 32, 1.0, 0.0, True),        # 4 blocks per warp tile, ragged tail
    (1, 32, 1, 32, 1.0, 0.5, True),                # a single block, partial warp tile
    (5, 5 * 256 * 3, 5, 256, 1.0, 0.0, False),
    (12, 12 * 64 * 5, 4, 64, 1.0, 0.0, False),
]


@pytest.mark.parametrize("R,N,G,B,s,beta,with_ef", CASES)
def test_ef_quant_int4_parity(dev, R, N, G, B, s, beta, with_ef):
    g = edge_gradients(R, N, B, seed=R * 1000 + B)
    rng = np.random.default_rng(B)
    ef0 = (rng.standard_normal(R * N) * 1e-4).astype(np.float32) if with_ef else None
    gc, gs, ge = gpu_ef_quant(g, ef0, N, R, G, B, s, beta, dev)
    ef_cpu = ef0.copy() if with_ef else None
    cc, cs = ORC.ef_quant_int4(g, ef_cpu, N, R, G, B, s, beta)
    assert_bits_equal(gc, cc, "codes")
    assert_bits_equal(gs, cs, "scales")
    if with_ef:
        gf = (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ref = np.abs(gf) + abs(s) * np.abs(ef0) + np.abs(ef_cpu)
        assert_f32_parity(ge, ef_cpu, ref, "error feedback")


def test_error_feedback_recurrence_tiny_workload(dev):
    """Three steps of the 4-rank, 1M-element workload with plain error
    feedback: each side carries its own error buffer from step to step."""
    w = wl.QGZ_TINY
    ef_cpu = np.zeros(w.R * w.N, np.float32)
    efd = torch.zeros(w.R * w.N, dtype=torch.float32, device=dev)
    codes = torch.empty(w.R * w.N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(w.R * w.N // w.B, dtype=torch.float32, device=dev)
    out = torch.empty(w.N, dtype=torch.float32, device=dev)
    for t in range(w.steps):
        gd = wl.qgz_gradients(w, t, device=dev)
        g = to_host(gd).ravel()
        binding.ef_quant_int4(gd.view(-1), efd, codes, scales, w.N, w.R, w.G, w.B,
                              w.err_scale, w.err_beta)
        binding.dequant_reduce(codes, scales, out, w.N, w.R, 1, w.B)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4(g, ef_cpu, w.N, w.R, w.G, w.B, w.err_scale, w.err_beta)
        co = ORC.dequant_reduce(cc, cs, w.N, w.R, 1, w.B)
        assert_bits_equal(to_host(codes), cc, f"codes step {t}")
        assert_bits_equal(to_host(scales), cs, f"scales step {t}")
        assert_f32_parity(to_host(efd), ef_cpu, np.abs(ef_cpu) + 1e-3, f"ef step {t}")
        ref = deq_magnitude(cc, cs, w.B).reshape(w.R, w.N).sum(0)
        assert_f32_parity(to_host(out), co, ref, f"reduced step {t}")


REDUCE_CASES = [
    # R, N, B, out_bf16, out_scale
    (4, 4 * 256 * 19, 256, False, 1.0),
    (8, 8 * 256 * 5, 256, False, 0.125),
    (8, 8 * 256 * 5, 256, True, 1.0),
    (1, 256 * 9, 256, False, 1.0),
    (3, 3 * 32 * 11, 32, False, 1.0),
    (11, 11 * 64 * 3, 64, True, 1.0 / 11),
    (20, 20 * 128 * 2, 128, False, 1.0),          # more sources than one load batch
    (16, 16 * 1024, 1024, False, 1.0),
    (1024, 1024 * 32, 32, False, 1.0),            # a thousand sources in the loop kernel
]


@pytest.mark.parametrize("R,N,B,out_bf16,out_scale", REDUCE_CASES)
def test_flat_dequant_reduce_parity(dev, R, N, B, out_bf16, out_scale):
    g = edge_gradients(R, N, B, seed=7 * R + B)
    cc, cs = ORC.ef_quant_int4(g, None, N, R, 1, B, 1.0, 0.0)
    out = torch.empty(N, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    binding.dequant_reduce(to_dev(cc, dev), to_dev(cs, dev), out, N, R, 1, B, out_scale)
    torch.cuda.synchronize()
    want = ORC.dequant_reduce(cc, cs, N, R, 1, B, out_scale, out_bf16)
    if out_bf16:
        assert_bf16_parity(to_host(out), want, "bf16 shards")
    else:
        ref = deq_magnitude(cc, cs, B).reshape(R, N).sum(0) * abs(out_scale)
        assert_f32_parity(to_host(out), want, ref, "fp32 shards")


HIER_CASES = [
    # R, G, B, shards of S = B * k
    (16, 2, 512, 3),
    (8, 4, 128, 5),
    (12, 3, 64, 7),
    (8, 2, 32, 9),
    (8, 1, 256, 4),        # one group: first hop requantizes the flat reduce
    (4, 4, 1024, 1),       # one rank per group: first hop is a requantization
    (32, 2, 512, 1),       # 16 ranks per group
    (4, 2, 256, 3),        # 2 ranks per group
    (16, 2, 1024, 1),      # 8 ranks per group, 1024-blocks
    (6, 2, 512, 2),        # 3 ranks per group: general kernel at B = 512
    (64, 32, 32, 1),       # 32 groups: the second hop's source loop (more than 16)
    (96, 3, 64, 1),        # 32 ranks per group: the general first hop in batches of 8
]


@pytest.mark.parametrize("R,G,B,k", HIER_CASES)
def test_hierarchical_parity(dev, R, G, B, k):
    N = R * B * k
    g = edge_gradients(R, N, B, seed=31 * R + G)
    ef0 = np.zeros(R * N, np.float32)
    # quantization with error feedback on the first hop
    gc, gs, ge = gpu_ef_quant(g, ef0.copy(), N, R, G, B, 1.0, 0.5, dev)
    ef_cpu = ef0.copy()
    cc, cs = ORC.ef_quant_int4(g, ef_cpu, N, R, G, B, 1.0, 0.5)
    assert_bits_equal(gc, cc, "codes")
    assert_bits_equal(gs, cs, "scales")
    # hop 1 from the oracle's codes
    c1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    binding.dequant_reduce_requant(to_dev(cc, dev), to_dev(cs, dev), c1, s1, N, R, G, B)
    torch.cuda.synchronize()
    oc1, os1 = ORC.dequant_reduce_requant(cc, cs, N, R, G, B)
    assert_bits_equal(to_host(c1), oc1, "hop-1 codes")
    assert_bits_equal(to_host(s1), os1, "hop-1 scales")
    # hop 2 from the oracle's hop-1 output
    if G > 1:
        out = torch.empty(N, dtype=torch.bfloat16, device=dev)
        binding.dequant_reduce(to_dev(oc1, dev), to_dev(os1, dev), out, N, R, G, B)
        torch.cuda.synchronize()
        want = ORC.dequant_reduce(oc1, os1, N, R, G, B, 1.0, True)
        assert_bf16_parity(to_host(out), want, "hop-2 shards")
        outf = torch.empty(N, dtype=torch.float32, device=dev)
        binding.dequant_reduce(to_dev(oc1, dev), to_dev(os1, dev), outf, N, R, G, B, 0.5)
        torch.cuda.synchronize()
        wantf = ORC.dequant_reduce(oc1, os1, N, R, G, B, 0.5, False)
        assert_bits_equal(to_host(outf), wantf, "hop-2 fp32 shards")


def test_zero_size_calls_launch_nothing(dev):
    sentinel = torch.full((64,), 7, dtype=torch.uint8, device=dev)
    binding.ef_quant_int4(torch.empty(0, dtype=torch.bfloat16, device=dev), None,
                          torch.empty(0, dtype=torch.uint8, device=dev),
                          torch.empty(0, dtype=torch.float32, device=dev), 0, 4, 1, 256)
    torch.cuda.synchronize()
    assert bool((sentinel == 7).all())


def test_outputs_stay_inside_their_buffers(dev):
    """Guard regions around every output stay untouched (ragged sizes)."""
    R, G, B = 6, 3, 64
    N = R * B * 5
    g = edge_gradients(R, N, B, seed=99)
    pad = 4096
    gd = to_dev(g, dev)
    efd = torch.zeros(R * N + 2 * pad, dtype=torch.float32, device=dev).fill_(13.0)
    efd[pad:pad + R * N] = 0.0
    codes = torch.full((R * N // 2 + 2 * pad,), 0xA5, dtype=torch.uint8, device=dev)
    scales = torch.full((R * N // B + 2 * pad,), -5.0, dtype=torch.float32, device=dev)
    binding.ef_quant_int4(gd, efd[pad:pad + R * N], codes[pad:pad + R * N // 2],
                          scales[pad:pad + R * N // B], N, R, G, B, 1.0, 0.5)
    c1 = torch.full((G * N // 2 + 2 * pad,), 0x5A, dtype=torch.uint8, device=dev)
    s1 = torch.full((G * N // B + 2 * pad,), -9.0, dtype=torch.float32, device=dev)
    binding.dequant_reduce_requant(codes[pad:pad + R * N // 2], scales[pad:pad + R * N // B],
                                   c1[pad:pad + G * N // 2], s1[pad:pad + G * N // B], N, R, G, B)
    out = torch.full((N + 2 * pad,), -1.0, dtype=torch.float32, device=dev)
    binding.dequant_reduce(c1[pad:pad + G * N // 2], s1[pad:pad + G * N // B],
                           out[pad:pad + N], N, R, G, B)
    torch.cuda.synchronize()
    for t, fill, n in ((efd, 13.0, R * N), (codes, 0xA5, R * N // 2), (scales, -5.0, R * N // B),
                       (c1, 0x5A, G * N // 2), (s1, -9.0, G * N // B), (out, -1.0, N)):
        assert bool((t[:pad] == fill).all()) and bool((t[pad + n:] == fill).all())


FUSED_CASES = [
    # R, N, B, with_ef, write_codes, out_bf16
    (8, 8 * 256 * 13, 256, True, True, False),
    (8, 8 * 256 * 13, 256, True, False, True),
    (4, 4 * 512 * 5, 512, True, True, True),
    (3, 3 * 128 * 7, 128, False, True, False),
    (1, 1024, 1024, True, True, False),
    (16, 16 * 256 * 2, 256, False, False, False),
]


@pytest.mark.parametrize("R,N,B,with_ef,write_codes,out_bf16", FUSED_CASES)
def test_fused_step_parity(dev, R, N, B, with_ef, write_codes, out_bf16):
    """One-kernel flat step against the oracle's two-stage definition, over
    two chained steps (the error buffer carries over)."""
    s, beta = 1.0, 0.5
    ef_cpu = np.zeros(R * N, np.float32) if with_ef else None
    efd = torch.zeros(R * N, dtype=torch.float32, device=dev) if with_ef else None
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev) if write_codes else None
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev) if write_codes else None
    out = torch.empty(N, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    for t in range(2):
        g = edge_gradients(R, N, B, seed=77 * t + R)
        binding.qgz_step_fused(to_dev(g, dev), efd, codes, scales, out, N, R, B, s, beta, 0.5)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4(g, ef_cpu, N, R, 1, B, s, beta)
        want = ORC.dequant_reduce(cc, cs, N, R, 1, B, 0.5, out_bf16)
        if write_codes:
            assert_bits_equal(to_host(codes), cc, f"codes step {t}")
            assert_bits_equal(to_host(scales), cs, f"scales step {t}")
        if with_ef:
            assert_bits_equal(to_host(efd), ef_cpu, f"error feedback step {t}")
        if out_bf16:
            assert_bf16_parity(to_host(out), want, f"bf16 shards step {t}")
        else:
            ref = deq_magnitude(cc, cs, B).reshape(R, N).sum(0) * 0.5
            assert_f32_parity(to_host(out), want, ref, f"fp32 shards step {t}")


def direct_codes_scales(R: int, N: int, B: int, seed: int):
    """Codes drawn uniformly from [-7, 7] and scales just above 2^-126 (the
    smallest non-zero block scale), as the exchange would deliver them: the
    dequantized terms are all normal, but their sums cancel into the
    subnormal range often enough to exercise gradual underflow in every
    fp32 add of the reduce."""
    rng = np.random.default_rng(seed)
    q = rng.integers(-7, 8, size=R * N).astype(np.int64) & 0xF
    codes = (q[0::2] | (q[1::2] << 4)).astype(np.uint8)
    tiny = np.float32(np.finfo(np.float32).tiny)
    k = rng.integers(0, 64, size=R * N // B).astype(np.float32)
    scales = (tiny * (np.float32(1) + k * np.float32(2.0 ** -23))).astype(np.float32)
    return codes, scales


@pytest.mark.parametrize("R,G,B", [(8, 1, 256), (16, 2, 512), (8, 2, 256), (6, 3, 64)])
def test_subnormal_sums_parity(dev, R, G, B):
    N = R * B * 6
    cc, cs = direct_codes_scales(R, N, B, seed=R * G + B)
    cd, sd = to_dev(cc, dev), to_dev(cs, dev)
    if G == 1:
        out = torch.empty(N, dtype=torch.float32, device=dev)
        binding.dequant_reduce(cd, sd, out, N, R, 1, B)
        torch.cuda.synchronize()
        want = ORC.dequant_reduce(cc, cs, N, R, 1, B)
        sub = (want != 0) & (np.abs(want) < np.finfo(np.float32).tiny)
        assert sub.sum() > 0, "the case must produce subnormal sums"
        assert_bits_equal(to_host(out), want, "flat sums")
    # first hop, plain and with error feedback started from subnormal errors
    c1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    binding.dequant_reduce_requant(cd, sd, c1, s1, N, R, G, B)
    torch.cuda.synchronize()
    oc1, os1 = ORC.dequant_reduce_requant(cc, cs, N, R, G, B)
    assert_bits_equal(to_host(c1), oc1, "hop-1 codes")
    assert_bits_equal(to_host(s1), os1, "hop-1 scales")
    rng = np.random.default_rng(B)
    e1 = (rng.standard_normal(G * N) * 1e-39).astype(np.float32)
    e1d = to_dev(e1, dev)
    binding.dequant_reduce_requant_ef(cd, sd, c1, s1, e1d, N, R, G, B, 1.0, 0.5)
    torch.cuda.synchronize()
    oc1e, os1e = ORC.dequant_reduce_requant_ef(cc, cs, N, R, G, B, e1, 1.0, 0.5)
    assert_bits_equal(to_host(c1), oc1e, "hop-1 codes with error feedback")
    assert_bits_equal(to_host(s1), os1e, "hop-1 scales with error feedback")
    assert_bits_equal(to_host(e1d), e1, "hop-1 error buffer")
    if G > 1:
        # second hop straight from drawn codes, so that its sums underflow too
        outf = torch.empty(N, dtype=torch.float32, device=dev)
        c2, s2 = direct_codes_scales(1, G * N, B, seed=B + 1)
        binding.dequant_reduce(to_dev(c2, dev), to_dev(s2, dev), outf, N, R, G, B)
        torch.cuda.synchronize()
        assert_bits_equal(to_host(outf), ORC.dequant_reduce(c2, s2, N, R, G, B), "hop-2 sums")


SIGNED_ZERO_SCALES = np.array([0.0, -0.0, 2.0 ** -149, -(2.0 ** -149), 3 * 2.0 ** -149, -1.5,
                               2.0 ** -127, 1.0, -(2.0 ** -126), 1e30], np.float32)


@pytest.mark.parametrize("R,G,B", [(1, 1, 256), (2, 1, 64), (8, 1, 256), (5, 1, 32),
                                   (16, 2, 512), (8, 2, 256), (4, 4, 128)])
def test_zero_and_negative_scales_parity(dev, R, G, B):
    """Every reduce sum starts at +0 and adds fl(q * scale) in source order.
    Scales of +-0 with nonzero codes make products of -0, which +0 turns into
    +0, and negative and subnormal scales down to 2^-149 make tiny nonzero
    products.  The quantizer never writes such scales, but the reduce's
    definition covers them, and the kernels' first-term shortcut must match
    it for every one of them.  (|q * scale| stays below 8e30: no infinities.)"""
    N = R * B * 4
    rng = np.random.default_rng(R * 97 + B)
    codes = rng.integers(0, 256, size=R * N // 2, dtype=np.uint8)
    scales = rng.choice(SIGNED_ZERO_SCALES, size=R * N // B).astype(np.float32)
    # the first block of every source buffer (what shard 0 reads first, flat
    # or second hop) gets a zero scale of alternating sign: all-zero sums
    scales[np.arange(R) * (N // B)] = np.where(np.arange(R) % 2 == 0, np.float32(0.0),
                                               np.float32(-0.0))
    cd, sd = to_dev(codes, dev), to_dev(scales, dev)
    # the reduce reads R source buffers (flat) or G (second hop) of N codes each
    nsrc = R if G == 1 else G
    c2, s2 = codes[:nsrc * N // 2], scales[:nsrc * N // B]
    for out_bf16 in (False, True):
        out = torch.empty(N, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
        binding.dequant_reduce(to_dev(c2, dev), to_dev(s2, dev), out, N, R, G, B)
        torch.cuda.synchronize()
        want = ORC.dequant_reduce(c2, s2, N, R, G, B, 1.0, out_bf16)
        assert_bits_equal(to_host(out), want, f"sums, {'bf16' if out_bf16 else 'fp32'}")
        if not out_bf16:
            assert np.all(want[:B].view(np.uint32) == 0), "shard 0's first block must be +0"
    c1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    binding.dequant_reduce_requant(cd, sd, c1, s1, N, R, G, B)
    torch.cuda.synchronize()
    oc1, os1 = ORC.dequant_reduce_requant(codes, scales, N, R, G, B)
    assert_bits_equal(to_host(c1), oc1, "first-hop codes")
    assert_bits_equal(to_host(s1), os1, "first-hop scales")
