"""Parity of wc_qgz_first_hop_fused -- every rank's EF-quant fused with the
first (intra-group) hop -- against the oracle's composition of the two steps
(orc_ef_quant_int4 with G groups, then orc_dequant_reduce_requant, or
orc_dequant_reduce_requant_ef with the first hop's own error buffer), bit for
bit, over chained steps: the first hop's codes and scales, the error buffers,
and, when written, the ranks' send buffers.  Also QgzReducer(fused=True),
alone, in HostPipeline and in a replayed CUDA graph, guard regions around
every output, and a zero-size call.

"ZeROPlusPlus.md", §1.2 ZeRO++ (qgZ: intra-node reduce first, kernel fusion);
"Merge LoCo with Zero++", Overview (error feedback before quantization)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bits_equal, dev, to_dev, to_host
from test_parity_qgz import edge_gradients
from weight_communication_gb300 import binding

pytestmark = pytest.mark.gpu

ORC = oracle.get()

CASES = [
    # R, G, B, k (blocks per shard), error feedback, write the send buffers
    (16, 2, 512, 3, True, True),
    (16, 2, 512, 2, True, False),
    (8, 4, 128, 5, True, True),
    (8, 2, 256, 3, False, True),
    (8, 2, 256, 1, False, False),
    (6, 3, 1024, 1, True, True),
    (8, 1, 256, 4, True, True),       # one group: requantized flat reduce
    (4, 4, 256, 2, True, True),       # one rank per group
    (32, 2, 128, 1, True, True),      # 16 ranks per group
    (12, 3, 128, 7, True, True),
]


@pytest.mark.parametrize("R,G,B,k,with_ef,write_codes", CASES)
def test_first_hop_fused_parity(dev, R, G, B, k, with_ef, write_codes):
    N = R * B * k
    s, beta = 1.0, 0.5
    ef_cpu = np.zeros(R * N, np.float32) if with_ef else None
    ef_dev = to_dev(np.zeros(R * N, np.float32), dev) if with_ef else None
    codes = torch.full((R * N // 2,), 0xAB, dtype=torch.uint8, device=dev) if write_codes else None
    scales = torch.full((R * N // B,), -1.0, dtype=torch.float32, device=dev) if write_codes else None
    oc = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    os_ = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    for t in range(3):
        g = edge_gradients(R, N, B, seed=41 * t + 7 * R + B + k)
        binding.qgz_first_hop_fused(to_dev(g, dev), ef_dev, codes, scales, oc, os_, N, R, G, B,
                                    s, beta)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4(g, ef_cpu, N, R, G, B, s, beta)
        oc1, os1 = ORC.dequant_reduce_requant(cc, cs, N, R, G, B)
        assert_bits_equal(to_host(oc), oc1, f"first-hop codes step {t}")
        assert_bits_equal(to_host(os_), os1, f"first-hop scales step {t}")
        if with_ef:
            assert_bits_equal(to_host(ef_dev), ef_cpu, f"error buffer step {t}")
        if write_codes:
            assert_bits_equal(to_host(codes), cc, f"send codes step {t}")
            assert_bits_equal(to_host(scales), cs, f"send scales step {t}")


EF1_CASES = [
    # R, G, B, k, s, beta (the ranks' and the first hop's error feedback)
    (16, 2, 512, 3, 1.0, 0.5),
    (8, 4, 128, 5, 1.0, 0.5),
    (6, 3, 256, 2, 0.75, 0.25),
    (8, 1, 256, 3, 2.0, 0.9),
    (12, 3, 1024, 1, 1.0, 0.0),
]


@pytest.mark.parametrize("R,G,B,k,s,beta", EF1_CASES)
def test_first_hop_fused_with_its_error_buffer(dev, R, G, B, k, s, beta):
    """With ef1 the fused first stage equals orc_ef_quant_int4 followed by
    orc_dequant_reduce_requant_ef, over three chained steps: the first hop's
    codes, scales and error buffer, the ranks' error buffer and send buffers."""
    N = R * B * k
    ef_cpu = np.zeros(R * N, np.float32)
    e1_cpu = np.zeros(G * N, np.float32)
    ef_dev = to_dev(ef_cpu.copy(), dev)
    e1_dev = to_dev(e1_cpu.copy(), dev)
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    oc = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    os_ = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    for t in range(3):
        g = edge_gradients(R, N, B, seed=53 * t + 5 * R + B + k)
        binding.qgz_first_hop_fused(to_dev(g, dev), ef_dev, codes, scales, oc, os_, N, R, G, B,
                                    s, beta, ef1=e1_dev)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4(g, ef_cpu, N, R, G, B, s, beta)
        oc1, os1 = ORC.dequant_reduce_requant_ef(cc, cs, N, R, G, B, e1_cpu, s, beta)
        assert_bits_equal(to_host(oc), oc1, f"first-hop codes step {t}")
        assert_bits_equal(to_host(os_), os1, f"first-hop scales step {t}")
        assert_bits_equal(to_host(e1_dev), e1_cpu, f"first-hop error step {t}")
        assert_bits_equal(to_host(ef_dev), ef_cpu, f"error buffer step {t}")
        assert_bits_equal(to_host(codes), cc, f"send codes step {t}")
        assert_bits_equal(to_host(scales), cs, f"send scales step {t}")


def test_first_hop_fused_then_second_hop(dev):
    """The fused first stage followed by the second hop gives the oracle's
    two-hop shards (the hierarchical workload's shape at a small size)."""
    R, G, B = 16, 2, 512
    N = R * B * 4
    g = edge_gradients(R, N, B, seed=1234)
    ef_cpu = np.zeros(R * N, np.float32)
    ef_dev = to_dev(ef_cpu.copy(), dev)
    oc = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    os_ = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    out = torch.empty(N, dtype=torch.bfloat16, device=dev)
    binding.qgz_first_hop_fused(to_dev(g, dev), ef_dev, None, None, oc, os_, N, R, G, B, 1.0, 0.5)
    binding.dequant_reduce(oc, os_, out, N, R, G, B)
    torch.cuda.synchronize()
    cc, cs = ORC.ef_quant_int4(g, ef_cpu, N, R, G, B, 1.0, 0.5)
    oc1, os1 = ORC.dequant_reduce_requant(cc, cs, N, R, G, B)
    want = ORC.dequant_reduce(oc1, os1, N, R, G, B, 1.0, True)
    assert_bits_equal(to_host(out), want, "two-hop shards")
    assert_bits_equal(to_host(ef_dev), ef_cpu, "error buffer")


def _oracle_step(w, g, ef, e1=None):
    """The oracle's step: quantization of every rank, then the flat reduce or
    the two hops (the first with its error buffer e1, if given); returns
    (shards, send codes, send scales, first-hop codes, first-hop scales)."""
    cc, cs = ORC.ef_quant_int4(g, ef, w.N, w.R, w.G, w.B, w.err_scale, w.err_beta)
    if w.G > 1:
        c1, s1 = ORC.dequant_reduce_requant_ef(cc, cs, w.N, w.R, w.G, w.B, e1, w.err_scale,
                                               w.err_beta)
        return ORC.dequant_reduce(c1, s1, w.N, w.R, w.G, w.B, 1.0, w.out_bf16), cc, cs, c1, s1
    return ORC.dequant_reduce(cc, cs, w.N, w.R, 1, w.B, 1.0, w.out_bf16), cc, cs, None, None


@pytest.mark.parametrize("which", ["single_hop", "hierarchical", "hierarchical_hop1_ef"])
def test_fused_reducer_matches_oracle(dev, which):
    """QgzReducer(fused=True): three chained steps against the oracle --
    shards, error buffers, send buffers and (hierarchical) the first hop's
    output -- in one launch (flat) or two (hierarchical)."""
    from weight_communication_gb300 import workloads as wl
    from weight_communication_gb300.qgz import QgzReducer
    w = (wl.QGZ_SINGLE_HOP.scaled(8 * 256 * 24) if which == "single_hop"
         else wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 5))
    hop1_ef = which == "hierarchical_hop1_ef"
    out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
    red = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype,
                     device=dev, fused=True, hop1_ef=hop1_ef)
    assert red.launches_per_step == (2 if w.G > 1 else 1)
    ef = np.zeros(w.R * w.N, np.float32)
    e1 = np.zeros(w.G * w.N, np.float32) if hop1_ef else None
    for t in range(3):
        g = wl.qgz_gradients(w, t, device=dev)
        out = red.step(g)
        torch.cuda.synchronize()
        want, cc, cs, c1, s1 = _oracle_step(w, to_host(g).ravel(), ef, e1)
        if hop1_ef:
            assert_bits_equal(to_host(red.ef1), e1, f"first-hop error step {t}")
        assert_bits_equal(to_host(out), want, f"{which} shards step {t}")
        assert_bits_equal(to_host(red.ef), ef, f"{which} error buffer step {t}")
        assert_bits_equal(to_host(red.codes), cc, f"{which} send codes step {t}")
        assert_bits_equal(to_host(red.scales), cs, f"{which} send scales step {t}")
        if w.G > 1:
            assert_bits_equal(to_host(red.codes1), c1, f"first-hop codes step {t}")
            assert_bits_equal(to_host(red.scales1), s1, f"first-hop scales step {t}")


def test_fused_reducer_in_host_pipeline_and_graph(dev):
    """A fused reducer in HostPipeline and in a replayed CUDA graph gives, step
    after step, the shards and error buffers (the first hop's included) of
    unfused serial steps."""
    from weight_communication_gb300 import workloads as wl
    from weight_communication_gb300.qgz import GraphedStep, HostPipeline, QgzReducer
    for w in (wl.QGZ_SINGLE_HOP.scaled(8 * 256 * 16), wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 4)):
        out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
        view = torch.int16 if out_dtype == torch.bfloat16 else torch.int32

        def make(fused):
            return QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype,
                              device=dev, fused=fused, hop1_ef=w.G > 1)
        piped, graphed_red, serial = make(True), make(True), make(False)
        steps = 4
        g_host = [wl.qgz_gradients(w, t).pin_memory() for t in range(steps)]
        out_host = [torch.empty(w.N, dtype=out_dtype).pin_memory() for _ in range(steps)]
        HostPipeline(piped).run(g_host, out_host)
        graphed = GraphedStep(graphed_red)
        for t in range(steps):
            graphed.g.copy_(g_host[t].view(-1).to(dev))
            got = graphed.replay().clone()
            want = serial.step(g_host[t].to(dev).view(-1))
            torch.cuda.synchronize()
            assert torch.equal(got.view(view), want.view(view)), (w.name, "graph", t)
            assert torch.equal(out_host[t].view(view), want.cpu().view(view)), (w.name, "host", t)
        for red in (piped, graphed_red):
            assert torch.equal(red.ef.view(torch.int32), serial.ef.view(torch.int32)), w.name
            if w.G > 1:
                assert torch.equal(red.ef1.view(torch.int32), serial.ef1.view(torch.int32))


def test_fused_first_hop_stays_inside_its_buffers(dev):
    """Guard regions around every output of the fused first stage stay
    untouched, and a zero-size call writes nothing."""
    R, G, B = 6, 3, 128
    N = R * B * 5
    pad = 4096
    g = edge_gradients(R, N, B, seed=98)
    efd = torch.full((R * N + 2 * pad,), 13.0, dtype=torch.float32, device=dev)
    efd[pad:pad + R * N] = 0.0
    codes = torch.full((R * N // 2 + 2 * pad,), 0xA5, dtype=torch.uint8, device=dev)
    scales = torch.full((R * N // B + 2 * pad,), -5.0, dtype=torch.float32, device=dev)
    c1 = torch.full((G * N // 2 + 2 * pad,), 0x5A, dtype=torch.uint8, device=dev)
    s1 = torch.full((G * N // B + 2 * pad,), -9.0, dtype=torch.float32, device=dev)
    binding.qgz_first_hop_fused(to_dev(g, dev), efd[pad:pad + R * N], codes[pad:pad + R * N // 2],
                                scales[pad:pad + R * N // B], c1[pad:pad + G * N // 2],
                                s1[pad:pad + G * N // B], N, R, G, B, 1.0, 0.5)
    torch.cuda.synchronize()
    for t, fill, n in ((efd, 13.0, R * N), (codes, 0xA5, R * N // 2), (scales, -5.0, R * N // B),
                       (c1, 0x5A, G * N // 2), (s1, -9.0, G * N // B)):
        assert bool((t[:pad] == fill).all()) and bool((t[pad + n:] == fill).all())
    ef_cpu = np.zeros(R * N, np.float32)
    cc, cs = ORC.ef_quant_int4(g, ef_cpu, N, R, G, B, 1.0, 0.5)
    oc1, os1 = ORC.dequant_reduce_requant(cc, cs, N, R, G, B)
    assert_bits_equal(to_host(c1[pad:pad + G * N // 2]), oc1, "first-hop codes")
    assert_bits_equal(to_host(s1[pad:pad + G * N // B]), os1, "first-hop scales")
    empty_u8 = torch.empty(0, dtype=torch.uint8, device=dev)
    empty_f = torch.empty(0, dtype=torch.float32, device=dev)
    binding.qgz_first_hop_fused(torch.empty(0, dtype=torch.bfloat16, device=dev), None, None, None,
                                empty_u8, empty_f, 0, 4, 2, 256)
    torch.cuda.synchronize()
    assert bool((c1[:pad] == 0x5A).all())
