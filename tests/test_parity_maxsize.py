"""Parity at the largest sizes the ABI accepts, where 32-bit indexing ends.

qgZ with R*N = 2^32 - 1024 (R = 2), the fused first hop with R*N = 2^32 - 8192
(4 ranks in 2 groups), qwZ with n = 2^32 - 2048 and SR with
n = 2^32 - 1 (its scalar tail included).  The oracle cannot run these sizes
whole, so sampled blocks at the start and the very end of every rank,
slice and shard are recomputed on the CPU as small problems of their own.
For qgZ, one block is one error-feedback quantization problem, and one
shard block is a reduce of the sources' blocks.  The comparison is bit for
bit.  About 40 GB of device memory at the peak."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bits_equal, dev, to_host  # noqa: F401
from weight_communication_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

ORC = oracle.get()


def test_qgz_at_the_largest_size(dev):
    R, B, s, beta = 2, 256, 1.0, 0.5
    N = (1 << 31) - 512               # R*N = 2^32 - 1024; B divides N/R
    S = N // R
    g = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
    for r in range(R):
        wl.draw_bf16(N, 1e-3, 7100 + r, dev, out=g[r])
    gf = g.view(-1)
    ef = torch.zeros(R * N, dtype=torch.float32, device=dev)
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    out = torch.empty(N, dtype=torch.float32, device=dev)
    binding.ef_quant_int4(gf, ef, codes, scales, N, R, 1, B, s, beta)
    binding.dequant_reduce(codes, scales, out, N, R, 1, B)
    torch.cuda.synchronize()
    last_block = N // B - 1
    for r in range(R):
        for b in (0, S // B - 1, S // B, last_block):       # first/last block of each slice
            x0 = r * N + b * B
            e_cpu = np.zeros(B, np.float32)
            cc, cs = ORC.ef_quant_int4(to_host(gf[x0:x0 + B]).copy(), e_cpu, B, 1, 1, B, s, beta)
            assert_bits_equal(to_host(codes[x0 // 2:(x0 + B) // 2]), cc, f"codes r={r} b={b}")
            assert_bits_equal(to_host(scales[x0 // B:x0 // B + 1]), cs, f"scale r={r} b={b}")
            assert_bits_equal(to_host(ef[x0:x0 + B]), e_cpu, f"error r={r} b={b}")
    for k in range(R):
        for j in (0, S // B - 1):
            # R ranks of R blocks each, whose chunk 0 is block (r, k*S/B + j)
            mc = np.zeros(R * R * B // 2, np.uint8)
            ms = np.ones(R * R, np.float32)
            for r in range(R):
                src = r * N + k * S + j * B
                mc[r * R * B // 2:(r * R * B + B) // 2] = to_host(codes[src // 2:(src + B) // 2])
                ms[r * R] = to_host(scales[src // B:src // B + 1])[0]
            want = ORC.dequant_reduce(mc, ms, R * B, R, 1, B)[:B]
            o0 = k * S + j * B
            assert_bits_equal(to_host(out[o0:o0 + B]), want, f"shard {k} block {j}")
    del g, ef, codes, scales, out
    torch.cuda.empty_cache()


def test_qwz_at_the_largest_size(dev):
    B = 2048
    n = (1 << 32) - B
    w = wl.draw_bf16(n, 0.02, 7200, dev)
    codes = torch.empty(n, dtype=torch.int8, device=dev)
    scales = torch.empty(n // B, dtype=torch.float32, device=dev)
    back = torch.empty(n, dtype=torch.bfloat16, device=dev)
    binding.qwz_quant_int8(w, codes, scales, B)
    binding.qwz_dequant_int8(codes, scales, back, B)
    torch.cuda.synchronize()
    for b in (0, n // B // 2, n // B - 1):
        x0 = b * B
        oc, os_ = ORC.qwz_quant_int8(to_host(w[x0:x0 + B]).copy(), B)
        assert_bits_equal(to_host(codes[x0:x0 + B]), oc, f"codes block {b}")
        assert_bits_equal(to_host(scales[b:b + 1]), os_, f"scale block {b}")
        assert_bits_equal(to_host(back[x0:x0 + B]), ORC.qwz_dequant_int8(oc, os_, B),
                          f"dequantized block {b}")
    del w, codes, scales, back
    torch.cuda.empty_cache()


def test_sr_at_the_largest_size(dev):
    n = (1 << 32) - 1                 # odd: the last 7 elements take the scalar tail
    seed, step = 5, 3
    dst = wl.draw_bf16(n, 1.0, 7300, dev)
    src = wl.draw_bf16(n, 1e-2, 7301, dev)
    picks = np.r_[0:16, n // 2:n // 2 + 16, n - 24:n]
    d0 = to_host(dst[torch.as_tensor(picks, device=dev)]).copy()
    s0 = to_host(src[torch.as_tensor(picks, device=dev)]).copy()
    binding.sr_accumulate_bf16(dst, src, seed, step)
    torch.cuda.synchronize()
    got = to_host(dst[torch.as_tensor(picks, device=dev)])
    assert not to_host(src[torch.as_tensor(picks, device=dev)]).any()
    for j, i in enumerate(picks):
        x = np.float32(ORC.bf16_to_f32(int(d0[j]))) + np.float32(ORC.bf16_to_f32(int(s0[j])))
        want = ORC.sr_round(float(x), ORC.sr_bits(seed, step, int(i)))
        assert int(got[j]) == want, (int(i), int(got[j]), want)
    del dst, src
    torch.cuda.empty_cache()


def test_small_blocks_at_the_largest_size(dev):
    """B = 32 takes the kernels' other paths: the tiled EF-quant, the general
    first hop, qwZ with 8 blocks per warp tile.  Their grid sizes round up
    from sizes within a tile of 2^32 (a 32-bit rounding would wrap there)."""
    B = 32
    # EF-quant (no error buffer) and the one-rank reduce, R*N = 2^32 - 32
    N = (1 << 32) - B
    g = wl.draw_bf16(N, 1e-3, 7400, dev)
    codes = torch.empty(N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(N // B, dtype=torch.float32, device=dev)
    binding.ef_quant_int4(g, None, codes, scales, N, 1, 1, B, 1.0, 0.0)
    torch.cuda.synchronize()
    out = torch.empty(N, dtype=torch.float32, device=dev)
    binding.dequant_reduce(codes, scales, out, N, 1, 1, B)
    torch.cuda.synchronize()
    for b in (0, N // B // 2, N // B - 1):
        x0 = b * B
        cc, cs = ORC.ef_quant_int4(to_host(g[x0:x0 + B]).copy(), None, B, 1, 1, B, 1.0, 0.0)
        assert_bits_equal(to_host(codes[x0 // 2:(x0 + B) // 2]), cc, f"codes block {b}")
        assert_bits_equal(to_host(scales[b:b + 1]), cs, f"scale block {b}")
        assert_bits_equal(to_host(out[x0:x0 + B]), ORC.dequant_reduce(cc, cs, B, 1, 1, B),
                          f"reduced block {b}")
    del g, codes, scales, out
    torch.cuda.empty_cache()

    # first hop, general kernel: R = G = 2 (one rank per group), G*N = 2^32 - 128
    # (B divides the shard N/R)
    R = G = 2
    N = (1 << 31) - 2 * B
    S = N // R
    g = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
    for r in range(R):
        wl.draw_bf16(N, 1e-3, 7500 + r, dev, out=g[r])
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    binding.ef_quant_int4(g.view(-1), None, codes, scales, N, R, G, B, 1.0, 0.0)
    c1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    binding.dequant_reduce_requant(codes, scales, c1, s1, N, R, G, B)
    torch.cuda.synchronize()
    # unit u (= rank u) sub-slice gq block j requantizes the one source block
    # at rank u, chunk gq, block j
    for u in range(R):
        for gq in range(G):
            for j in (0, S // B - 1):
                src = u * N + gq * S + j * B
                dst = (u * G + gq) * S + j * B
                mc = to_host(codes[src // 2:(src + B) // 2]).copy()
                ms = to_host(scales[src // B:src // B + 1]).copy()
                oc, os_ = ORC.dequant_reduce_requant(mc, ms, B, 1, 1, B)
                assert_bits_equal(to_host(c1[dst // 2:(dst + B) // 2]), oc, f"hop 1 u={u} gq={gq} j={j}")
                assert_bits_equal(to_host(s1[dst // B:dst // B + 1]), os_, f"hop 1 scale u={u} gq={gq} j={j}")
    del g, codes, scales, c1, s1
    torch.cuda.empty_cache()

    # qwZ with 32-weight blocks, n = 2^32 - 32
    n = (1 << 32) - B
    w = wl.draw_bf16(n, 0.02, 7600, dev)
    qc = torch.empty(n, dtype=torch.int8, device=dev)
    qs = torch.empty(n // B, dtype=torch.float32, device=dev)
    back = torch.empty(n, dtype=torch.bfloat16, device=dev)
    binding.qwz_quant_int8(w, qc, qs, B)
    binding.qwz_dequant_int8(qc, qs, back, B)
    torch.cuda.synchronize()
    for b in (0, n // B - 1):
        x0 = b * B
        oc, os_ = ORC.qwz_quant_int8(to_host(w[x0:x0 + B]).copy(), B)
        assert_bits_equal(to_host(qc[x0:x0 + B]), oc, f"qwZ codes block {b}")
        assert_bits_equal(to_host(back[x0:x0 + B]), ORC.qwz_dequant_int8(oc, os_, B),
                          f"qwZ dequantized block {b}")
    del w, qc, qs, back
    torch.cuda.empty_cache()


def _random_codes(n_bytes: int, seed: int, dev) -> torch.Tensor:
    """n_bytes random code bytes on the device (every nibble, -8 included)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    return torch.randint(0, 256, (n_bytes,), dtype=torch.uint8, device=dev, generator=gen)


def _random_scales(n: int, seed: int, dev) -> torch.Tensor:
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    return (torch.randn(n, device=dev, generator=gen) * 1e-3).to(torch.float32)


def test_packed_kernels_at_the_largest_size(dev):
    """The packed and product-table kernels where 32-bit indexing ends: the
    packed flat reduce (4 sources, B = 256), the first hop's table path
    (16 ranks in 2 groups, B = 512) and the int8 error buffer's kernel
    (three blocks per warp, B = 256), each with R*N just under 2^32.
    Sampled blocks at the start and the end of shards and units are
    recomputed by the oracle as small problems of their own."""
    # packed flat reduce, R = 4, R*N = 2^32 - 4096
    R, B = 4, 256
    N = (1 << 30) - 1024
    S = N // R
    codes = _random_codes(R * N // 2, 7700, dev)
    scales = _random_scales(R * N // B, 7701, dev)
    out = torch.empty(N, dtype=torch.float32, device=dev)
    binding.dequant_reduce(codes, scales, out, N, R, 1, B)
    torch.cuda.synchronize()
    for k in (0, R - 1):
        for j in (0, S // B - 1):
            mc = np.zeros(R * R * B // 2, np.uint8)
            ms = np.ones(R * R, np.float32)
            for r in range(R):
                src = r * N + k * S + j * B
                mc[r * R * B // 2:(r * R * B + B) // 2] = to_host(codes[src // 2:(src + B) // 2])
                ms[r * R] = to_host(scales[src // B:src // B + 1])[0]
            want = ORC.dequant_reduce(mc, ms, R * B, R, 1, B)[:B]
            o0 = k * S + j * B
            assert_bits_equal(to_host(out[o0:o0 + B]), want, f"packed reduce shard {k} block {j}")
    del codes, scales, out
    torch.cuda.empty_cache()

    # first hop through product tables: R = 16, G = 2, L = 8, R*N = 2^32 - 131072
    R, G, B = 16, 2, 512
    L = R // G
    N = (1 << 28) - 8192
    S = N // R
    codes = _random_codes(R * N // 2, 7702, dev)
    scales = _random_scales(R * N // B, 7703, dev)
    c1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    binding.dequant_reduce_requant(codes, scales, c1, s1, N, R, G, B)
    torch.cuda.synchronize()
    for u in (0, R - 1):
        grp, l = divmod(u, L)
        for gq in (0, G - 1):
            for j in (0, S // B - 1):
                # one group of L ranks whose chunk 0 is the unit's source block
                mc = np.zeros(L * L * B // 2, np.uint8)
                ms = np.ones(L * L, np.float32)
                for lq in range(L):
                    src = (grp * L + lq) * N + (l * G + gq) * S + j * B
                    mc[lq * L * B // 2:(lq * L * B + B) // 2] = to_host(codes[src // 2:(src + B) // 2])
                    ms[lq * L] = to_host(scales[src // B:src // B + 1])[0]
                oc, os_ = ORC.dequant_reduce_requant(mc, ms, L * B, L, 1, B)
                dst = (u * G + gq) * S + j * B
                assert_bits_equal(to_host(c1[dst // 2:(dst + B) // 2]), oc[:B // 2],
                                  f"table hop 1 u={u} gq={gq} j={j}")
                assert_bits_equal(to_host(s1[dst // B:dst // B + 1]), os_[:1],
                                  f"table hop 1 scale u={u} gq={gq} j={j}")
    del codes, scales, c1, s1
    torch.cuda.empty_cache()

    # int8 error buffer, R = 4, R*N = 2^32 - 4096, stored errors random
    R, B, s, beta = 4, 256, 1.0, 0.5
    N = (1 << 30) - 1024
    S = N // R
    g = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
    for r in range(R):
        wl.draw_bf16(N, 1e-3, 7800 + r, dev, out=g[r])
    gf = g.view(-1)
    e8 = _random_codes(R * N, 7810, dev).view(torch.int8)
    es = (_random_scales(R * N // B, 7811, dev).abs() * 1e-2).contiguous()
    e8_0 = {}
    es_0 = {}
    picks = [(r, b) for r in (0, R - 1) for b in (0, S // B - 1, N // B - 1)]
    for r, b in picks:
        x0 = r * N + b * B
        e8_0[(r, b)] = to_host(e8[x0:x0 + B]).copy()
        es_0[(r, b)] = to_host(es[x0 // B:x0 // B + 1]).copy()
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    binding.ef_quant_int4_int8ef(gf, e8, es, codes, scales, N, R, 1, B, s, beta)
    torch.cuda.synchronize()
    for r, b in picks:
        x0 = r * N + b * B
        e8c, esc = e8_0[(r, b)].copy(), es_0[(r, b)].copy()
        cc, cs = ORC.ef_quant_int4_int8ef(to_host(gf[x0:x0 + B]).copy(), e8c, esc, B, 1, 1, B, s, beta)
        assert_bits_equal(to_host(codes[x0 // 2:(x0 + B) // 2]), cc, f"int8-EF codes r={r} b={b}")
        assert_bits_equal(to_host(scales[x0 // B:x0 // B + 1]), cs, f"int8-EF scale r={r} b={b}")
        assert_bits_equal(to_host(e8[x0:x0 + B]), e8c, f"int8 error r={r} b={b}")
        assert_bits_equal(to_host(es[x0 // B:x0 // B + 1]), esc, f"int8 error scale r={r} b={b}")
    del g, e8, es, codes, scales
    torch.cuda.empty_cache()


def test_fused_first_hop_at_the_largest_size(dev):
    """wc_qgz_first_hop_fused with R*N = 2^32 - 8192 (4 ranks in 2 groups,
    B = 512).  Each sampled first-hop output block is one small problem: the
    L ranks' error-feedback quantization of the blocks they send to the unit,
    then a first hop of L sources with one block each.  About 27 GB of device
    memory."""
    R, G, B, s, beta = 4, 2, 512, 1.0, 0.5
    L = R // G
    N = (1 << 30) - R * B             # R*N = 2^32 - 8192; B divides N/R
    S = N // R
    g = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
    for r in range(R):
        wl.draw_bf16(N, 1e-3, 7300 + r, dev, out=g[r])
    gf = g.view(-1)
    ef = torch.zeros(R * N, dtype=torch.float32, device=dev)
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    oc = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    os_ = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    binding.qgz_first_hop_fused(gf, ef, codes, scales, oc, os_, N, R, G, B, s, beta)
    torch.cuda.synchronize()
    for u in (0, R - 1):
        grp, l = divmod(u, L)
        for gq in (0, G - 1):
            for j in (0, S // B - 1):
                mc = np.zeros(L * L * B // 2, np.uint8)
                ms = np.ones(L * L, np.float32)
                for lq in range(L):
                    r = grp * L + lq
                    x0 = r * N + (gq * L + l) * S + j * B      # gradient order
                    p0 = r * N + (l * G + gq) * S + j * B      # send position
                    e_cpu = np.zeros(B, np.float32)
                    cc, cs = ORC.ef_quant_int4(to_host(gf[x0:x0 + B]).copy(), e_cpu, B, 1, 1, B,
                                               s, beta)
                    where = f"rank {r} sub-slice {gq} block {j}"
                    assert_bits_equal(to_host(codes[p0 // 2:(p0 + B) // 2]), cc, "codes " + where)
                    assert_bits_equal(to_host(scales[p0 // B:p0 // B + 1]), cs, "scale " + where)
                    assert_bits_equal(to_host(ef[x0:x0 + B]), e_cpu, "error " + where)
                    mc[lq * L * B // 2:(lq * L * B + B) // 2] = cc
                    ms[lq * L] = cs[0]
                wc_, ws_ = ORC.dequant_reduce_requant(mc, ms, L * B, L, 1, B)
                o0 = (u * G + gq) * S + j * B
                where = f"unit {u} sub-slice {gq} block {j}"
                assert_bits_equal(to_host(oc[o0 // 2:(o0 + B) // 2]), wc_[:B // 2], "codes " + where)
                assert_bits_equal(to_host(os_[o0 // B:o0 // B + 1]), ws_[:1], "scale " + where)
    del g, ef, codes, scales, oc, os_
    torch.cuda.empty_cache()
