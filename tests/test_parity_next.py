"""GPU parity (through the C ABI) of the entry points beyond the basic path,
against the CPU oracle:

  * wc_ef_quant_int4_bf16ef and wc_ef_quant_int4_int8ef -- EF-quant with a
    bf16 or an int8 error buffer, over chained steps, every block size and
    grouped send orders, and at full size;
  * wc_qwz_quant_replica_int8 -- qwZ quantization writing the bf16 replica.

The fused flat step's parity is in test_parity_qgz.py.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bits_equal, dev, to_dev, to_host
from test_parity_qgz import edge_gradients
from test_parity_secondary import weights_with_edges
from weight_communication_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

ORC = oracle.get()

BF16EF_CASES = [
    # R, N, G, B, s, beta
    (8, 8 * 256 * 9, 1, 256, 1.0, 0.5),
    (4, 4 * 256 * 5, 1, 256, 1.0, 0.0),
    (16, 16 * 512 * 2, 2, 512, 1.0, 0.5),
    (6, 6 * 64 * 11, 3, 64, 0.75, 0.25),
    (2, 2 * 32 * 9, 1, 32, 2.0, 0.5),
    (3, 3 * 1024, 1, 1024, 1.0, 0.5),
]


@pytest.mark.parametrize("R,N,G,B,s,beta", BF16EF_CASES)
def test_bf16_error_buffer_parity(dev, R, N, G, B, s, beta):
    rng = np.random.default_rng(N + B)
    e0 = wl.as_u16(torch.from_numpy((rng.standard_normal(R * N) * 1e-4).astype(np.float32))
                   .to(torch.bfloat16)).copy()
    e_cpu = e0.copy()
    e_dev = to_dev(e0, dev)
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    for t in range(3):
        g = edge_gradients(R, N, B, seed=13 * t + R + B)
        binding.ef_quant_int4_bf16ef(to_dev(g, dev), e_dev, codes, scales, N, R, G, B, s, beta)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4_bf16ef(g, e_cpu, N, R, G, B, s, beta)
        assert_bits_equal(to_host(codes), cc, f"codes step {t}")
        assert_bits_equal(to_host(scales), cs, f"scales step {t}")
        assert_bits_equal(to_host(e_dev), e_cpu, f"bf16 error step {t}")


def test_bf16_error_buffer_full_size(dev):
    """Single-hop workload size, two chained steps, every output."""
    w = wl.QGZ_SINGLE_HOP
    e_dev = torch.zeros(w.R * w.N, dtype=torch.bfloat16, device=dev)
    e_cpu = np.zeros(w.R * w.N, np.uint16)
    codes = torch.empty(w.R * w.N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(w.R * w.N // w.B, dtype=torch.float32, device=dev)
    gd = torch.empty((w.R, w.N), dtype=torch.bfloat16, device=dev)
    for t in range(2):
        wl.qgz_gradients(w, t, device=dev, out=gd)
        binding.ef_quant_int4_bf16ef(gd.view(-1), e_dev, codes, scales, w.N, w.R, 1, w.B,
                                     w.err_scale, w.err_beta)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4_bf16ef(to_host(gd).ravel(), e_cpu, w.N, w.R, 1, w.B,
                                          w.err_scale, w.err_beta)
        assert_bits_equal(to_host(codes), cc, f"codes step {t}")
        assert_bits_equal(to_host(scales), cs, f"scales step {t}")
        assert_bits_equal(to_host(e_dev), e_cpu, f"bf16 error step {t}")


@pytest.mark.parametrize("R,N,G,B,s,beta", BF16EF_CASES)
def test_int8_error_buffer_parity(dev, R, N, G, B, s, beta):
    """int8 error buffer over three chained steps, from random stored codes and
    scales: codes, scales, stored error codes and error scales bit for bit."""
    rng = np.random.default_rng(N + 3 * B)
    e8_0 = rng.integers(-127, 128, size=R * N).astype(np.int8)
    es_0 = (rng.random(R * N // B) * 1e-5).astype(np.float32)
    es_0[::7] = 0.0                                   # some zero blocks in the buffer
    e8_cpu, es_cpu = e8_0.copy(), es_0.copy()
    e8_dev, es_dev = to_dev(e8_0, dev), to_dev(es_0, dev)
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    for t in range(3):
        g = edge_gradients(R, N, B, seed=17 * t + R + B)
        binding.ef_quant_int4_int8ef(to_dev(g, dev), e8_dev, es_dev, codes, scales, N, R, G, B,
                                     s, beta)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4_int8ef(g, e8_cpu, es_cpu, N, R, G, B, s, beta)
        assert_bits_equal(to_host(codes), cc, f"codes step {t}")
        assert_bits_equal(to_host(scales), cs, f"scales step {t}")
        assert_bits_equal(to_host(e8_dev), e8_cpu, f"int8 error codes step {t}")
        assert_bits_equal(to_host(es_dev), es_cpu, f"int8 error scales step {t}")


def test_int8_error_buffer_full_size(dev):
    """Single-hop workload size, two chained steps from a zero buffer, every
    output."""
    w = wl.QGZ_SINGLE_HOP
    e8_dev = torch.zeros(w.R * w.N, dtype=torch.int8, device=dev)
    es_dev = torch.zeros(w.R * w.N // w.B, dtype=torch.float32, device=dev)
    e8_cpu = np.zeros(w.R * w.N, np.int8)
    es_cpu = np.zeros(w.R * w.N // w.B, np.float32)
    codes = torch.empty(w.R * w.N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(w.R * w.N // w.B, dtype=torch.float32, device=dev)
    gd = torch.empty((w.R, w.N), dtype=torch.bfloat16, device=dev)
    for t in range(2):
        wl.qgz_gradients(w, t, device=dev, out=gd)
        binding.ef_quant_int4_int8ef(gd.view(-1), e8_dev, es_dev, codes, scales, w.N, w.R, 1, w.B,
                                     w.err_scale, w.err_beta)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4_int8ef(to_host(gd).ravel(), e8_cpu, es_cpu, w.N, w.R, 1, w.B,
                                          w.err_scale, w.err_beta)
        assert_bits_equal(to_host(codes), cc, f"codes step {t}")
        assert_bits_equal(to_host(scales), cs, f"scales step {t}")
        assert_bits_equal(to_host(e8_dev), e8_cpu, f"int8 error codes step {t}")
        assert_bits_equal(to_host(es_dev), es_cpu, f"int8 error scales step {t}")


HOP1_EF_CASES = [
    # R, G, B, k (shard = k blocks), s, beta
    (16, 2, 512, 3, 1.0, 0.5),      # the hierarchical workload's shape
    (8, 2, 256, 4, 1.0, 0.0),
    (8, 4, 128, 5, 2.0, 0.25),      # general kernel
    (12, 3, 64, 7, 1.0, 0.5),       # general kernel, blocks shorter than the warp tile
    (32, 2, 512, 1, 1.0, 0.5),      # 16 ranks per group
    (16, 2, 1024, 1, 0.5, 0.75),
]


@pytest.mark.parametrize("R,G,B,k,s,beta", HOP1_EF_CASES)
def test_first_hop_error_feedback_parity(dev, R, G, B, k, s, beta):
    """Three chained steps; each side carries its own first-hop error."""
    N = R * B * k
    e1_cpu = np.zeros(G * N, np.float32)
    e1_dev = torch.zeros(G * N, dtype=torch.float32, device=dev)
    c1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    for t in range(3):
        g = edge_gradients(R, N, B, seed=101 * t + R + G)
        cc, cs = ORC.ef_quant_int4(g, None, N, R, G, B, 1.0, 0.0)
        binding.dequant_reduce_requant_ef(to_dev(cc, dev), to_dev(cs, dev), c1, s1, e1_dev, N, R,
                                          G, B, s, beta)
        torch.cuda.synchronize()
        oc, os_ = ORC.dequant_reduce_requant_ef(cc, cs, N, R, G, B, e1_cpu, s, beta)
        assert_bits_equal(to_host(c1), oc, f"hop-1 codes step {t}")
        assert_bits_equal(to_host(s1), os_, f"hop-1 scales step {t}")
        assert_bits_equal(to_host(e1_dev), e1_cpu, f"hop-1 error step {t}")


@pytest.mark.parametrize("n,B", [(2048 * 21, 2048), (256 * 33, 256), (32 * 13, 32), (4096 * 2, 4096)])
def test_qwz_replica_parity(dev, n, B):
    w = weights_with_edges(n, B, seed=3 * n + B)
    codes = torch.empty(n, dtype=torch.int8, device=dev)
    scales = torch.empty(n // B, dtype=torch.float32, device=dev)
    rep = torch.empty(n, dtype=torch.bfloat16, device=dev)
    binding.qwz_quant_replica_int8(to_dev(w, dev), codes, scales, rep, B)
    torch.cuda.synchronize()
    oc, os_, orep = ORC.qwz_quant_replica_int8(w, B)
    assert_bits_equal(to_host(codes), oc, "codes")
    assert_bits_equal(to_host(scales), os_, "scales")
    assert_bits_equal(to_host(rep), orep, "replica")


def test_host_pipeline_matches_serial_steps(dev):
    """Pipelined host-to-host steps give the same shards and error buffer as
    the same steps run one after another on one stream."""
    from weight_communication_gb300.qgz import HostPipeline, QgzReducer
    for w in (wl.QGZ_SINGLE_HOP.scaled(8 * 256 * 64), wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 8)):
        out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
        a = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype, device=dev,
                       hop1_ef=w.G > 1)
        b = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype, device=dev,
                       hop1_ef=w.G > 1)
        steps = 5
        g_host = [wl.qgz_gradients(w, t).pin_memory() for t in range(steps)]
        out_host = [torch.empty(w.N, dtype=out_dtype).pin_memory() for _ in range(steps)]
        HostPipeline(a).run(g_host, out_host)
        torch.cuda.synchronize()
        for t in range(steps):
            want = b.step(g_host[t].to(dev).view(-1)).cpu()
            assert torch.equal(out_host[t].view(torch.int16) if out_dtype == torch.bfloat16
                               else out_host[t].view(torch.int32),
                               want.view(torch.int16) if out_dtype == torch.bfloat16
                               else want.view(torch.int32)), (w.name, t)
        assert torch.equal(a.ef.view(torch.int32), b.ef.view(torch.int32))
        if w.G > 1:
            assert torch.equal(a.ef1.view(torch.int32), b.ef1.view(torch.int32))


def test_reducer_with_first_hop_error_feedback_matches_oracle(dev):
    """QgzReducer's hierarchical step with error feedback on both hops,
    two chained steps, against the oracle's composition."""
    from weight_communication_gb300.qgz import QgzReducer
    w = wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 6)
    red = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=torch.bfloat16,
                     device=dev, hop1_ef=True)
    e = np.zeros(w.R * w.N, np.float32)
    e1 = np.zeros(w.G * w.N, np.float32)
    for t in range(2):
        g = wl.qgz_gradients(w, t, device=dev)
        out = red.step(g)
        torch.cuda.synchronize()
        gu = to_host(g).ravel()
        cc, cs = ORC.ef_quant_int4(gu, e, w.N, w.R, w.G, w.B, w.err_scale, w.err_beta)
        c1, s1 = ORC.dequant_reduce_requant_ef(cc, cs, w.N, w.R, w.G, w.B, e1, w.err_scale, w.err_beta)
        want = ORC.dequant_reduce(c1, s1, w.N, w.R, w.G, w.B, 1.0, True)
        assert_bits_equal(to_host(out), want, f"shards step {t}")
        assert_bits_equal(to_host(red.ef1), e1, f"first-hop error step {t}")


EF_BITS = {torch.float32: torch.int32, torch.bfloat16: torch.int16, torch.int8: torch.int8}


def _same_state(a, b, what):
    """The reducers' error buffers (with the int8 buffer's scales and the
    first-hop errors) are equal bit for bit."""
    assert torch.equal(a.ef.view(EF_BITS[a.ef.dtype]), b.ef.view(EF_BITS[b.ef.dtype])), what
    if a.ef_scales is not None:
        assert torch.equal(a.ef_scales.view(torch.int32), b.ef_scales.view(torch.int32)), what
    if a.ef1 is not None:
        assert torch.equal(a.ef1.view(torch.int32), b.ef1.view(torch.int32)), what


@pytest.mark.parametrize("ef_dtype", [torch.float32, torch.bfloat16, torch.int8])
def test_device_pipeline_matches_serial_steps(dev, ef_dtype):
    """Steps with the reduce on a second stream give the same shards, error
    buffers and (hierarchical) first-hop errors as serial steps."""
    from weight_communication_gb300.qgz import DevicePipeline, QgzReducer
    for w in (wl.QGZ_SINGLE_HOP.scaled(8 * 256 * 64), wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 8)):
        out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
        a = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype, device=dev,
                       ef_dtype=ef_dtype, hop1_ef=w.G > 1)
        b = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype, device=dev,
                       ef_dtype=ef_dtype, hop1_ef=w.G > 1)
        pipe = DevicePipeline(a)
        grads = [wl.qgz_gradients(w, t, device=dev) for t in range(5)]
        outs = []
        for t in range(5):
            pipe.step(grads[t])
            snap = torch.empty_like(a.out)
            with torch.cuda.stream(pipe.reduce_stream):  # after step t's reduce
                snap.copy_(a.out)
            outs.append(snap)
        torch.cuda.synchronize()
        for t in range(5):
            want = b.step(grads[t])
            assert torch.equal(outs[t].view(torch.int16 if out_dtype == torch.bfloat16 else torch.int32),
                               want.view(torch.int16 if out_dtype == torch.bfloat16 else torch.int32)), t
        _same_state(a, b, w.name)


@pytest.mark.parametrize("ef_dtype", [torch.float32, torch.bfloat16, torch.int8])
def test_graphed_step_matches_eager_steps(dev, ef_dtype):
    """A step captured in a CUDA graph and replayed gives, step after step,
    the same shards, error buffers and first-hop errors as eager steps."""
    from weight_communication_gb300.qgz import GraphedStep, QgzReducer
    for w in (wl.QGZ_SINGLE_HOP.scaled(8 * 256 * 16), wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 4)):
        out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
        a = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype, device=dev,
                       ef_dtype=ef_dtype, hop1_ef=w.G > 1)
        b = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype, device=dev,
                       ef_dtype=ef_dtype, hop1_ef=w.G > 1)
        graphed = GraphedStep(a)
        assert not a.ef.any(), "capturing must not run the step"
        view = torch.int16 if out_dtype == torch.bfloat16 else torch.int32
        for t in range(3):
            g = wl.qgz_gradients(w, t, device=dev)
            graphed.g.copy_(g.view(-1))
            got = graphed.replay().clone()
            want = b.step(g)
            torch.cuda.synchronize()
            assert torch.equal(got.view(view), want.view(view)), (w.name, t)
            _same_state(a, b, (w.name, t))
