"""Parity of wc_qgz_first_hop_fused -- every rank's EF-quant fused with the
first (intra-group) hop -- against the oracle's composition of the two steps
(orc_ef_quant_int4 with G groups, then orc_dequant_reduce_requant), bit for
bit, over chained steps: the first hop's codes and scales, the error buffer,
and, when written, the ranks' send buffers.

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
