"""Parity of the fused kernels with the low-precision error buffers -- the
flat step (wc_qgz_step_fused_bf16ef / _int8ef) and the hierarchical first
stage (wc_qgz_first_hop_fused_bf16ef / _int8ef, with and without the first
hop's own error buffer) -- against the oracle's composition of the same
quantization (orc_ef_quant_int4_bf16ef / _int8ef) with the reduce
(orc_dequant_reduce) or the first hop (orc_dequant_reduce_requant[_ef]),
bit for bit over chained steps: shards or first-hop codes and scales, the
error buffers (bf16 values; int8 codes and block scales), the send buffers.
The stored errors start random, not zero.

"Merge LoCo with Zero++", Overview (error feedback, the buffer's memory);
"ZeROPlusPlus.md", §1.2 ZeRO++ (qgZ, intra-node first, kernel fusion)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bits_equal, dev, to_dev, to_host
from test_parity_qgz import edge_gradients
from weight_communication_gb300 import binding

pytestmark = pytest.mark.gpu

ORC = oracle.get()


def initial_error(kind: str, R: int, N: int, B: int, seed: int):
    """A random stored error buffer: bf16 bit patterns of N(0, 1e-4) values
    with some zeros, or int8 codes in [-127, 127] with block scales (some 0)."""
    rng = np.random.default_rng(seed)
    if kind == "bf16":
        v = (rng.standard_normal(R * N) * 1e-4).astype(np.float32)
        v[rng.random(R * N) < 0.05] = 0.0
        return ORC.bf16_round(v), None
    e8 = rng.integers(-127, 128, size=R * N).astype(np.int8)
    es = (rng.random(R * N // B) * 1e-6).astype(np.float32)
    es[::7] = 0.0
    return e8, es


def oracle_quant(kind, g, e, es, N, R, G, B, s, beta):
    if kind == "bf16":
        return ORC.ef_quant_int4_bf16ef(g, e, N, R, G, B, s, beta)
    return ORC.ef_quant_int4_int8ef(g, e, es, N, R, G, B, s, beta)


def device_error(kind, e, es, dev):
    if kind == "bf16":
        return torch.from_numpy(e.view(np.int16).copy()).to(dev).view(torch.bfloat16), None
    return to_dev(e, dev), to_dev(es, dev)


def host_error(t: torch.Tensor) -> np.ndarray:
    return to_host(t.view(torch.int16) if t.dtype == torch.bfloat16 else t)


FLAT_CASES = [
    # kind, R, B, k (blocks per shard), write codes, bf16 shards, s, beta
    ("bf16", 8, 256, 3, True, False, 1.0, 0.5),
    ("bf16", 4, 512, 2, False, True, 0.75, 0.25),
    ("bf16", 3, 128, 5, True, True, 1.0, 0.0),
    ("bf16", 1, 1024, 2, True, False, 2.0, 0.9),
    ("int8", 8, 256, 3, True, False, 1.0, 0.5),
    ("int8", 4, 512, 2, False, True, 0.75, 0.25),
    ("int8", 6, 128, 5, True, True, 1.0, 0.0),
    ("int8", 2, 1024, 1, True, False, 2.0, 0.9),
]


@pytest.mark.parametrize("kind,R,B,k,write_codes,out_bf16,s,beta", FLAT_CASES)
def test_fused_step_low_precision_error(dev, kind, R, B, k, write_codes, out_bf16, s, beta):
    N = R * B * k
    e, es = initial_error(kind, R, N, B, seed=R * 31 + B + k)
    ed, esd = device_error(kind, e, es, dev)
    codes = torch.full((R * N // 2,), 0xAB, dtype=torch.uint8, device=dev) if write_codes else None
    scales = torch.full((R * N // B,), -1.0, dtype=torch.float32, device=dev) if write_codes else None
    out = torch.empty(N, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    for t in range(3):
        g = edge_gradients(R, N, B, seed=61 * t + 3 * R + B + k)
        binding.qgz_step_fused(to_dev(g, dev), ed, codes, scales, out, N, R, B, s, beta, 0.5,
                               ef_scales=esd)
        torch.cuda.synchronize()
        cc, cs = oracle_quant(kind, g, e, es, N, R, 1, B, s, beta)
        want = ORC.dequant_reduce(cc, cs, N, R, 1, B, 0.5, out_bf16)
        assert_bits_equal(to_host(out), want, f"{kind} shards step {t}")
        assert_bits_equal(host_error(ed), e.view(np.int16) if kind == "bf16" else e,
                          f"{kind} error buffer step {t}")
        if kind == "int8":
            assert_bits_equal(to_host(esd), es, f"int8 error scales step {t}")
        if write_codes:
            assert_bits_equal(to_host(codes), cc, f"send codes step {t}")
            assert_bits_equal(to_host(scales), cs, f"send scales step {t}")


HIER_CASES = [
    # kind, R, G, B, k, write codes, first-hop error buffer, s, beta
    ("bf16", 16, 2, 512, 2, True, False, 1.0, 0.5),
    ("bf16", 8, 4, 128, 3, False, True, 1.0, 0.5),
    ("bf16", 6, 3, 256, 2, True, True, 0.75, 0.25),
    ("int8", 16, 2, 512, 2, True, False, 1.0, 0.5),
    ("int8", 8, 4, 128, 3, False, True, 1.0, 0.5),
    ("int8", 6, 3, 256, 2, True, True, 2.0, 0.9),
    ("int8", 4, 4, 1024, 1, True, True, 1.0, 0.0),
]


@pytest.mark.parametrize("kind,R,G,B,k,write_codes,with_ef1,s,beta", HIER_CASES)
def test_fused_first_hop_low_precision_error(dev, kind, R, G, B, k, write_codes, with_ef1, s,
                                             beta):
    N = R * B * k
    e, es = initial_error(kind, R, N, B, seed=R * 37 + G + B + k)
    ed, esd = device_error(kind, e, es, dev)
    e1 = np.zeros(G * N, np.float32) if with_ef1 else None
    e1d = to_dev(e1.copy(), dev) if with_ef1 else None
    codes = torch.full((R * N // 2,), 0xAB, dtype=torch.uint8, device=dev) if write_codes else None
    scales = torch.full((R * N // B,), -1.0, dtype=torch.float32, device=dev) if write_codes else None
    oc = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
    os_ = torch.empty(G * N // B, dtype=torch.float32, device=dev)
    for t in range(3):
        g = edge_gradients(R, N, B, seed=67 * t + 5 * R + G + B)
        binding.qgz_first_hop_fused(to_dev(g, dev), ed, codes, scales, oc, os_, N, R, G, B, s,
                                    beta, ef1=e1d, ef_scales=esd)
        torch.cuda.synchronize()
        cc, cs = oracle_quant(kind, g, e, es, N, R, G, B, s, beta)
        oc1, os1 = ORC.dequant_reduce_requant_ef(cc, cs, N, R, G, B, e1, s, beta)
        assert_bits_equal(to_host(oc), oc1, f"{kind} first-hop codes step {t}")
        assert_bits_equal(to_host(os_), os1, f"{kind} first-hop scales step {t}")
        assert_bits_equal(host_error(ed), e.view(np.int16) if kind == "bf16" else e,
                          f"{kind} error buffer step {t}")
        if kind == "int8":
            assert_bits_equal(to_host(esd), es, f"int8 error scales step {t}")
        if with_ef1:
            assert_bits_equal(to_host(e1d), e1, f"first-hop error step {t}")
        if write_codes:
            assert_bits_equal(to_host(codes), cc, f"send codes step {t}")
            assert_bits_equal(to_host(scales), cs, f"send scales step {t}")


@pytest.mark.parametrize("ef_dtype", [torch.bfloat16, torch.int8])
@pytest.mark.parametrize("which", ["single_hop", "hierarchical"])
def test_fused_reducer_low_precision_error_matches_unfused(dev, which, ef_dtype):
    """QgzReducer(fused=True) with a bf16 or int8 error buffer gives, step
    after step, the shards and error buffers of the unfused reducer (whose
    kernels the other parity suites pin to the oracle)."""
    from weight_communication_gb300 import workloads as wl
    from weight_communication_gb300.qgz import QgzReducer
    w = (wl.QGZ_SINGLE_HOP.scaled(8 * 256 * 12) if which == "single_hop"
         else wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 3))
    out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
    view = torch.int16 if out_dtype == torch.bfloat16 else torch.int32

    def make(fused):
        return QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype,
                          device=dev, ef_dtype=ef_dtype, hop1_ef=w.G > 1, fused=fused)
    a, b = make(True), make(False)
    assert a.launches_per_step == (2 if w.G > 1 else 1)
    for t in range(3):
        g = wl.qgz_gradients(w, t, device=dev)
        got = a.step(g).clone()
        want = b.step(g)
        torch.cuda.synchronize()
        assert torch.equal(got.view(view), want.view(view)), (which, t)
    ev = torch.int16 if ef_dtype == torch.bfloat16 else torch.int8
    assert torch.equal(a.ef.view(ev), b.ef.view(ev))
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales.view(torch.int32),
                                                         b.scales.view(torch.int32))
    if ef_dtype == torch.int8:
        assert torch.equal(a.ef_scales.view(torch.int32), b.ef_scales.view(torch.int32))
    if w.G > 1:
        assert torch.equal(a.ef1.view(torch.int32), b.ef1.view(torch.int32))
