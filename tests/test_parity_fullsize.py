"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (QgzReducer and the same bindings), against the CPU oracle.

  * qgZ single hop (R=8, N=50,593,792, B=256, LoCo s=1, beta=0.5): two chained
    steps, every output compared.
  * qgZ hierarchical (R=16 in 2 groups of 8, N=202,375,168, B=512): codes and
    scales of every rank, the error buffers of two ranks, first-hop outputs
    of two units and final bf16 shards of two ranks (the oracle computes the
    sampled units and ranks one by one from its own codes).
  * qwZ (875,036,672 weights, B=2048): three sampled ranges of blocks.
  * SR accumulate (124,475,904 elements, 8 micro-steps): every element.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (assert_bf16_parity, assert_bits_equal, assert_f32_parity, deq_magnitude,
                      dev, to_host)
from weight_communication_gb300 import binding, workloads as wl
from weight_communication_gb300.qgz import QgzReducer

pytestmark = pytest.mark.gpu

ORC = oracle.get()


def test_single_hop_full_size(dev):
    w = wl.QGZ_SINGLE_HOP
    red = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, device=dev)
    ef_cpu = np.zeros(w.R * w.N, np.float32)
    gd = torch.empty((w.R, w.N), dtype=torch.bfloat16, device=dev)
    for t in range(2):
        wl.qgz_gradients(w, t, device=dev, out=gd)
        red.step(gd)
        torch.cuda.synchronize()
        g = to_host(gd).ravel()
        ef_prev = ef_cpu.copy()
        cc, cs = ORC.ef_quant_int4(g, ef_cpu, w.N, w.R, w.G, w.B, w.err_scale, w.err_beta)
        assert_bits_equal(to_host(red.codes), cc, f"codes step {t}")
        assert_bits_equal(to_host(red.scales), cs, f"scales step {t}")
        gf = (g.astype(np.uint32) << 16).view(np.float32)
        ref = np.abs(gf) + np.abs(ef_prev) + np.abs(ef_cpu)
        assert_f32_parity(to_host(red.ef), ef_cpu, ref, f"error feedback step {t}")
        del gf, ref, ef_prev
        co = ORC.dequant_reduce(cc, cs, w.N, w.R, 1, w.B)
        ref = deq_magnitude(cc, cs, w.B).reshape(w.R, w.N).sum(0)
        assert_f32_parity(to_host(red.out), co, ref, f"reduced shards step {t}")


def test_hierarchical_full_size(dev):
    w = wl.QGZ_HIERARCHICAL
    R, N, G, B, L, S = w.R, w.N, w.G, w.B, w.L, w.S
    red = QgzReducer(N, R, G, B, w.err_scale, w.err_beta, out_dtype=torch.bfloat16, device=dev)
    gd = wl.qgz_gradients(w, 0, device=dev)
    red.step(gd)
    torch.cuda.synchronize()
    oc = np.zeros(R * N // 2, np.uint8)
    os_ = np.zeros(R * N // B, np.float32)
    gpu_codes = to_host(red.codes)
    gpu_scales = to_host(red.scales)
    for r in range(R):
        g_r = to_host(gd[r])
        ef_r = np.zeros(N, np.float32)
        c_r, s_r = ORC.ef_quant_int4_rank(g_r, ef_r, N, R, G, B, w.err_scale, w.err_beta)
        oc[r * N // 2:(r + 1) * N // 2] = c_r
        os_[r * N // B:(r + 1) * N // B] = s_r
        assert_bits_equal(gpu_codes[r * N // 2:(r + 1) * N // 2], c_r, f"codes rank {r}")
        assert_bits_equal(gpu_scales[r * N // B:(r + 1) * N // B], s_r, f"scales rank {r}")
        if r in (0, R - 1):
            gf = (g_r.astype(np.uint32) << 16).view(np.float32)
            assert_f32_parity(to_host(red.ef[r * N:(r + 1) * N]), ef_r,
                              np.abs(gf) + np.abs(ef_r), f"error feedback rank {r}")
    del gpu_codes, gpu_scales
    # first hop: units (g, l) for the sampled l, both groups; the oracle's
    # hop-1 buffer holds only those units, which is all that hop 2 reads for
    # destinations g*L + l
    l = 5
    gpu_c1 = to_host(red.codes1)
    gpu_s1 = to_host(red.scales1)
    oc1 = np.zeros(G * N // 2, np.uint8)
    os1 = np.zeros(G * N // B, np.float32)
    unit_c, unit_s = G * S // 2, G * S // B
    for g in range(G):
        u = g * L + l
        cu, su = ORC.dequant_reduce_requant_unit(oc, os_, N, R, G, B, g, l)
        assert_bits_equal(gpu_c1[u * unit_c:(u + 1) * unit_c], cu, f"hop-1 codes unit {u}")
        assert_bits_equal(gpu_s1[u * unit_s:(u + 1) * unit_s], su, f"hop-1 scales unit {u}")
        oc1[u * unit_c:(u + 1) * unit_c] = cu
        os1[u * unit_s:(u + 1) * unit_s] = su
    gpu_out = to_host(red.out)
    for g in range(G):
        k = g * L + l
        want = ORC.dequant_reduce_dest(oc1, os1, N, R, G, B, k, 1.0, True)
        assert_bf16_parity(gpu_out[k * S:(k + 1) * S], want, f"final shard {k}")


def test_qwz_full_size(dev):
    w = wl.QWZ_WEIGHTS
    wd = wl.qwz_weights(w, device=dev)
    codes = torch.empty(w.n, dtype=torch.int8, device=dev)
    scales = torch.empty(w.n // w.B, dtype=torch.float32, device=dev)
    back = torch.empty(w.n, dtype=torch.bfloat16, device=dev)
    binding.qwz_quant_int8(wd, codes, scales, w.B)
    binding.qwz_dequant_int8(codes, scales, back, w.B)
    torch.cuda.synchronize()
    span = 2048 * 2048
    for start in (0, (w.n // 2) // w.B * w.B, w.n - span):
        sl = slice(start, start + span)
        wu = to_host(wd[sl])
        oc, os_ = ORC.qwz_quant_int8(wu, w.B)
        assert_bits_equal(to_host(codes[sl]), oc, f"codes at {start}")
        assert_bits_equal(to_host(scales[start // w.B:(start + span) // w.B]), os_, f"scales at {start}")
        assert_bits_equal(to_host(back[sl]), ORC.qwz_dequant_int8(oc, os_, w.B), f"bf16 at {start}")


def test_sr_accumulate_full_size(dev):
    w = wl.SR_ACCUMULATE
    dst = torch.zeros(w.n, dtype=torch.bfloat16, device=dev)
    src = torch.empty(w.n, dtype=torch.bfloat16, device=dev)
    dst_cpu = np.zeros(w.n, np.uint16)
    truth = np.zeros(w.n, np.float64)
    for t in range(w.micro_steps):
        wl.sr_micro_gradient(w, t, device=dev, out=src)
        src_cpu = to_host(src)
        truth += (src_cpu.astype(np.uint32) << 16).view(np.float32)
        binding.sr_accumulate_bf16(dst, src, w.seed, t)
        torch.cuda.synchronize()
        ORC.sr_accumulate_bf16(dst_cpu, src_cpu, w.seed, t)
        assert_bits_equal(to_host(dst), dst_cpu, f"dst micro-step {t}")
        assert bool((src == 0).all()), f"src not zeroed at micro-step {t}"
    # no bias against the exact sum: mean error within 5 standard errors
    got = (dst_cpu.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = got - truth
    assert abs(err.mean()) <= 5 * err.std() / np.sqrt(w.n)
