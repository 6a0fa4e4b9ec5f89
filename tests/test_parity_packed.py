"""Parity of the kernels that run in packed fp32x2 arithmetic or read their
products from per-block tables, against the oracle, bit for bit:

  * the flat reduce and the second hop for every source count the packed
    reduce kernel takes (3 to 8) at B = 256, 512 and 1024, fp32 and bf16 out,
    with and without an output scale, from random codes (every nibble,
    including -8, which the quantizer never writes) and scales that include
    +-0, negative and subnormal values;
  * the first hop's table path for every group size L it takes (1, 2, 4, 8,
    16) at B = 256, 512 and 1024, from the same kind of codes and scales;
  * the int8 error buffer's packed kernel (two blocks per warp at B = 128 and
    256) over chained steps, with odd block counts per slice (the last warp
    of a slice then has one block) and grouped send orders.

"ZeROPlusPlus.md", §1.2 ZeRO++ (qgZ: full-precision reduce, intra-group
first); "Merge LoCo with Zero++", Overview (error feedback, its buffer)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bits_equal, dev, to_dev, to_host
from test_parity_qgz import edge_gradients
from weight_communication_gb300 import binding

pytestmark = pytest.mark.gpu

ORC = oracle.get()

SCALES = np.array([0.0, -0.0, 2.0 ** -149, -(2.0 ** -140), 1.5e-38, -2.5, 1e-3, 7.1e-5,
                   -3.3e-4, 1.0, 6e29], np.float32)


def random_codes_scales(nsrc: int, N: int, B: int, seed: int):
    """nsrc source buffers of N codes: uniform random bytes (every nibble) and
    scales drawn from SCALES or a normal spread (|q * scale| < 5e30)."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=nsrc * N // 2, dtype=np.uint8)
    scales = np.where(rng.random(nsrc * N // B) < 0.5,
                      rng.choice(SCALES, size=nsrc * N // B),
                      (rng.standard_normal(nsrc * N // B) * 1e-3)).astype(np.float32)
    return codes, scales


PAIR_CASES = [(n, B) for n in range(3, 9) for B in (256, 512, 1024)]


@pytest.mark.parametrize("n,B", PAIR_CASES)
def test_flat_reduce_packed_parity(dev, n, B):
    R = n
    k = 3 if B < 1024 else 1          # an odd number of blocks per shard
    N = R * B * k
    codes, scales = random_codes_scales(R, N, B, seed=13 * n + B)
    cd, sd = to_dev(codes, dev), to_dev(scales, dev)
    for out_bf16, out_scale in ((False, 1.0), (True, 1.0), (False, 0.25), (True, 3.0)):
        out = torch.empty(N, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
        binding.dequant_reduce(cd, sd, out, N, R, 1, B, out_scale)
        torch.cuda.synchronize()
        want = ORC.dequant_reduce(codes, scales, N, R, 1, B, out_scale, out_bf16)
        assert_bits_equal(to_host(out), want, f"flat, {n} sources, bf16={out_bf16}, x{out_scale}")


@pytest.mark.parametrize("G,L,B", [(3, 2, 256), (4, 1, 512), (5, 2, 1024), (6, 1, 256),
                                   (7, 2, 512), (8, 2, 256), (8, 1, 1024)])
def test_second_hop_packed_parity(dev, G, L, B):
    R = G * L
    N = R * B * 2
    codes, scales = random_codes_scales(G, N, B, seed=G * 101 + B)   # G first-hop buffers
    cd, sd = to_dev(codes, dev), to_dev(scales, dev)
    for out_bf16, out_scale in ((True, 1.0), (False, 1.0), (True, 0.5)):
        out = torch.empty(N, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
        binding.dequant_reduce(cd, sd, out, N, R, G, B, out_scale)
        torch.cuda.synchronize()
        want = ORC.dequant_reduce(codes, scales, N, R, G, B, out_scale, out_bf16)
        assert_bits_equal(to_host(out), want, f"second hop, G={G}, bf16={out_bf16}")


@pytest.mark.parametrize("L,B", [(L, B) for L in (1, 2, 4, 8, 16) for B in (256, 512, 1024)])
def test_first_hop_table_path_parity(dev, L, B):
    G = 2
    R = G * L
    N = R * B * 3
    codes, scales = random_codes_scales(R, N, B, seed=L * 1009 + B)
    c1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    binding.dequant_reduce_requant(to_dev(codes, dev), to_dev(scales, dev), c1, s1, N, R, G, B)
    torch.cuda.synchronize()
    oc, os_ = ORC.dequant_reduce_requant(codes, scales, N, R, G, B)
    assert_bits_equal(to_host(c1), oc, f"first-hop codes, L={L}, B={B}")
    assert_bits_equal(to_host(s1), os_, f"first-hop scales, L={L}, B={B}")


@pytest.mark.parametrize("R,G,B,k,s,beta", [(4, 1, 128, 1, 1.0, 0.5), (4, 2, 128, 3, 0.75, 0.25),
                                             (6, 3, 256, 5, 1.0, 0.0), (8, 2, 256, 7, 2.0, 0.9),
                                             (2, 1, 512, 3, 1.0, 0.5), (3, 1, 1024, 1, 1.0, 0.5)])
def test_int8_error_buffer_packed_parity(dev, R, G, B, k, s, beta):
    """Shards of k blocks: with k odd, the last warp of every slice has only
    its first block (two blocks per warp at B = 128 and 256)."""
    N = R * B * k
    rng = np.random.default_rng(R * 7 + B + k)
    e8_cpu = rng.integers(-127, 128, size=R * N).astype(np.int8)
    es_cpu = (rng.random(R * N // B) * 1e-4).astype(np.float32)
    es_cpu[::5] = 0.0
    e8_dev, es_dev = to_dev(e8_cpu, dev), to_dev(es_cpu, dev)
    codes = torch.full((R * N // 2,), 0xAB, dtype=torch.uint8, device=dev)
    scales = torch.full((R * N // B,), -1.0, dtype=torch.float32, device=dev)
    for t in range(3):
        g = edge_gradients(R, N, B, seed=29 * t + R * B + k)
        binding.ef_quant_int4_int8ef(to_dev(g, dev), e8_dev, es_dev, codes, scales, N, R, G, B,
                                     s, beta)
        torch.cuda.synchronize()
        cc, cs = ORC.ef_quant_int4_int8ef(g, e8_cpu, es_cpu, N, R, G, B, s, beta)
        assert_bits_equal(to_host(codes), cc, f"codes step {t}")
        assert_bits_equal(to_host(scales), cs, f"scales step {t}")
        assert_bits_equal(to_host(e8_dev), e8_cpu, f"int8 error codes step {t}")
        assert_bits_equal(to_host(es_dev), es_cpu, f"int8 error scales step {t}")
