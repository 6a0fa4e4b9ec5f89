"""Seeded sweep of random qgZ geometries, each run as whole chained steps on
the GPU and through the oracle, compared bit for bit.

The fixed parity cases in test_parity_qgz.py and test_parity_next.py each pick
one kernel variant.  Here each case draws a rank count R, a group count G
dividing R, a block size B (a power of two in [32, 1024]) and a shard length
of k blocks. It also draws an error buffer (none, fp32, bf16 or int8),
first-hop error feedback, the output type, the output scale and LoCo's s and
beta. It then runs three chained steps through QgzReducer, so every
combination of the kernels' fixed and general forms meets the others.  The
flat cases also run the fused single-kernel step, and draws with B >= 128
(every error buffer form) run through the fused reducer.  The send buffers, the
first-hop buffers, the error buffers and the shards must all equal the
oracle's composition of the same steps ("ZeRO++", qgZ; "Merge LoCo with
Zero++", Overview)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bits_equal, dev, to_dev, to_host
from weight_communication_gb300 import binding, workloads as wl
from weight_communication_gb300.qgz import QgzReducer

pytestmark = pytest.mark.gpu

ORC = oracle.get()

RANKS = [1, 2, 3, 4, 5, 6, 8, 12, 16, 24, 32, 48]
EF_DTYPES = [None, torch.float32, torch.bfloat16, torch.int8]
MAX_ELEMENTS = 1 << 21          # R*N per case, so the oracle stays well under a second


def draw_geometry(seed: int) -> dict:
    rng = np.random.default_rng(1_000_003 * seed + 17)
    R = int(rng.choice(RANKS))
    divisors = [d for d in range(1, R + 1) if R % d == 0]
    G = int(rng.choice(divisors))
    while True:
        B = 32 << int(rng.integers(0, 6))
        k = int(rng.integers(1, 8))
        if R * R * B * k <= MAX_ELEMENTS:
            break
    return dict(R=R, G=G, B=B, N=R * B * k,
                ef=EF_DTYPES[int(rng.integers(0, 4))],
                hop1_ef=bool(G > 1 and rng.integers(0, 2)),
                out_bf16=bool(rng.integers(0, 2)),
                out_scale=float(rng.choice([1.0, 0.5, 1.0 / R, 3.0])),
                s=float(rng.choice([1.0, 0.5, 2.0])),
                beta=float(rng.choice([0.0, 0.25, 0.5, 0.9])),
                sigma=float(rng.choice([1e-4, 1e-2, 1.0])),
                zero_blocks=bool(rng.integers(0, 2)))


def gradients(geo: dict, seed: int, step: int) -> np.ndarray:
    """[R*N] bf16 bits: normal values with sparse outliers, and in some cases
    a few whole blocks set to zero (the zero-block rule)."""
    R, N, B = geo["R"], geo["N"], geo["B"]
    g = wl.as_u16(wl.draw_bf16(R * N, geo["sigma"], 7919 * seed + step,
                               outlier_frac=1e-3, outlier_mult=50.0)).copy()
    if geo["zero_blocks"]:
        rng = np.random.default_rng(31 * seed + step)
        nb = R * N // B
        for b in rng.choice(nb, size=min(nb, 3), replace=False):
            g[b * B:(b + 1) * B] = 0
    return g


class OracleSteps:
    """The oracle's composition of one reducer's steps, with its own copies
    of the error buffers."""

    def __init__(self, geo: dict):
        self.geo = geo
        R, N, G, B = geo["R"], geo["N"], geo["G"], geo["B"]
        ef = geo["ef"]
        self.e = (np.zeros(R * N, np.float32) if ef is torch.float32 else
                  np.zeros(R * N, np.uint16) if ef is torch.bfloat16 else
                  np.zeros(R * N, np.int8) if ef is torch.int8 else None)
        self.es = np.zeros(R * N // B, np.float32) if ef is torch.int8 else None
        self.e1 = np.zeros(G * N, np.float32) if geo["hop1_ef"] else None

    def step(self, g: np.ndarray):
        geo = self.geo
        R, N, G, B, s, beta = geo["R"], geo["N"], geo["G"], geo["B"], geo["s"], geo["beta"]
        if geo["ef"] is torch.bfloat16:
            cc, cs = ORC.ef_quant_int4_bf16ef(g, self.e, N, R, G, B, s, beta)
        elif geo["ef"] is torch.int8:
            cc, cs = ORC.ef_quant_int4_int8ef(g, self.e, self.es, N, R, G, B, s, beta)
        else:
            cc, cs = ORC.ef_quant_int4(g, self.e, N, R, G, B, s, beta)
        c1 = s1 = None
        if G > 1:
            if self.e1 is not None:
                c1, s1 = ORC.dequant_reduce_requant_ef(cc, cs, N, R, G, B, self.e1, s, beta)
            else:
                c1, s1 = ORC.dequant_reduce_requant(cc, cs, N, R, G, B)
            out = ORC.dequant_reduce(c1, s1, N, R, G, B, geo["out_scale"], geo["out_bf16"])
        else:
            out = ORC.dequant_reduce(cc, cs, N, R, 1, B, geo["out_scale"], geo["out_bf16"])
        return cc, cs, c1, s1, out


SEEDS = list(range(160))


def _describe(seed: int) -> str:
    g = draw_geometry(seed)
    ef = {None: "noef", torch.float32: "f32ef", torch.bfloat16: "bf16ef", torch.int8: "i8ef"}[g["ef"]]
    return (f"s{seed}-R{g['R']}G{g['G']}B{g['B']}k{g['N'] // (g['R'] * g['B'])}-{ef}"
            f"{'-h1ef' if g['hop1_ef'] else ''}{'-bf16' if g['out_bf16'] else ''}")


@pytest.mark.parametrize("seed", SEEDS, ids=[_describe(s) for s in SEEDS])
def test_random_geometry_chained_steps(dev, seed):
    _chained_steps(dev, seed, fused=False)


def _reducer_fusable(geo: dict) -> bool:
    """QgzReducer(fused=True) takes B >= 128 and every error buffer form,
    flat or hierarchical, with or without the first hop's error buffer."""
    return geo["B"] >= 128


REDUCER_FUSED_SEEDS = ([s for s in range(2000) if _reducer_fusable(draw_geometry(s))
                        and draw_geometry(s)["G"] > 1][:32]
                       + [s for s in range(2000) if _reducer_fusable(draw_geometry(s))
                          and draw_geometry(s)["G"] == 1][:12])


@pytest.mark.parametrize("seed", REDUCER_FUSED_SEEDS,
                         ids=[_describe(s) for s in REDUCER_FUSED_SEEDS])
def test_random_geometry_fused_reducer(dev, seed):
    """The same chained steps through QgzReducer(fused=True): the flat step
    as one kernel, or the hierarchical first stage (with the first hop's
    error buffer when drawn) as one kernel, then the second hop."""
    _chained_steps(dev, seed, fused=True)


def _chained_steps(dev, seed, fused):
    geo = draw_geometry(seed)
    R, N, G, B = geo["R"], geo["N"], geo["G"], geo["B"]
    red = QgzReducer(N, R, G, B, geo["s"], geo["beta"], use_ef=geo["ef"] is not None,
                     out_dtype=torch.bfloat16 if geo["out_bf16"] else torch.float32,
                     out_scale=geo["out_scale"], device=dev,
                     ef_dtype=geo["ef"] or torch.float32, hop1_ef=geo["hop1_ef"], fused=fused)
    orc = OracleSteps(geo)
    for t in range(3):
        g = gradients(geo, seed, t)
        out = red.step(to_dev(g, dev).view(R, N))
        torch.cuda.synchronize()
        cc, cs, c1, s1, want = orc.step(g)
        assert_bits_equal(to_host(red.codes), cc, f"send codes, step {t}")
        assert_bits_equal(to_host(red.scales), cs, f"send scales, step {t}")
        if G > 1:
            assert_bits_equal(to_host(red.codes1), c1, f"first-hop codes, step {t}")
            assert_bits_equal(to_host(red.scales1), s1, f"first-hop scales, step {t}")
        assert_bits_equal(to_host(out), want, f"shards, step {t}")
        if orc.e is not None:
            assert_bits_equal(to_host(red.ef), orc.e, f"error buffer, step {t}")
        if orc.es is not None:
            assert_bits_equal(to_host(red.ef_scales), orc.es, f"error scales, step {t}")
        if orc.e1 is not None:
            assert_bits_equal(to_host(red.ef1), orc.e1, f"first-hop error, step {t}")


def _fusable(geo: dict) -> bool:
    """The fused step takes flat geometries, B >= 128, fp32 error or none."""
    return geo["G"] == 1 and geo["B"] >= 128 and geo["ef"] in (None, torch.float32)


FUSED_SEEDS = [s for s in range(1000) if _fusable(draw_geometry(s))][:32]


@pytest.mark.parametrize("seed", FUSED_SEEDS, ids=[_describe(s) for s in FUSED_SEEDS])
def test_random_geometry_fused_step(dev, seed):
    """The flat draws with an fp32 error buffer or none, through the fused
    single-kernel step; it writes the send buffers too."""
    geo = draw_geometry(seed)
    R, N, B = geo["R"], geo["N"], geo["B"]
    orc = OracleSteps(geo)
    ef = torch.zeros(R * N, dtype=torch.float32, device=dev) if geo["ef"] is not None else None
    codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
    out = torch.empty(N, dtype=torch.bfloat16 if geo["out_bf16"] else torch.float32, device=dev)
    for t in range(3):
        g = gradients(geo, seed, t)
        binding.qgz_step_fused(to_dev(g, dev), ef, codes, scales, out, N, R, B,
                               geo["s"], geo["beta"], geo["out_scale"])
        torch.cuda.synchronize()
        cc, cs, _, _, want = orc.step(g)
        assert_bits_equal(to_host(codes), cc, f"send codes, step {t}")
        assert_bits_equal(to_host(scales), cs, f"send scales, step {t}")
        assert_bits_equal(to_host(out), want, f"shards, step {t}")
        if ef is not None:
            assert_bits_equal(to_host(ef), orc.e, f"error buffer, step {t}")


QWZ_SEEDS = list(range(40))


def draw_qwz(seed: int) -> dict:
    rng = np.random.default_rng(7_000_003 * seed + 5)
    B = 32 << int(rng.integers(0, 8))
    blocks = (int(rng.integers(1, 41)) if rng.integers(0, 2)
              else int(rng.integers(1, max(2, (1 << 20) // B))))
    return dict(B=B, n=B * blocks,
                sigma=float(rng.choice([1e-6, 1e-3, 0.02, 3.0])),
                replica=bool(rng.integers(0, 2)), zero_blocks=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("seed", QWZ_SEEDS,
                         ids=[f"s{s}-B{draw_qwz(s)['B']}-n{draw_qwz(s)['n']}" for s in QWZ_SEEDS])
def test_random_qwz(dev, seed):
    """qwZ int8 block quantization (with or without the bf16 replica) and its
    dequantization for a random block size in [32, 4096] and block count
    ("ZeRO++", qwZ)."""
    q = draw_qwz(seed)
    n, B = q["n"], q["B"]
    w = wl.as_u16(wl.draw_bf16(n, q["sigma"], 104729 * seed + 1, outlier_frac=1e-3,
                               outlier_mult=30.0)).copy()
    if q["zero_blocks"]:
        for b in np.random.default_rng(seed).choice(n // B, size=min(n // B, 2), replace=False):
            w[b * B:(b + 1) * B] = 0
    codes = torch.empty(n, dtype=torch.int8, device=dev)
    scales = torch.empty(n // B, dtype=torch.float32, device=dev)
    back = torch.empty(n, dtype=torch.bfloat16, device=dev)
    if q["replica"]:
        rep = torch.empty(n, dtype=torch.bfloat16, device=dev)
        binding.qwz_quant_replica_int8(to_dev(w, dev), codes, scales, rep, B)
        oc, os_, orep = ORC.qwz_quant_replica_int8(w, B)
    else:
        binding.qwz_quant_int8(to_dev(w, dev), codes, scales, B)
        oc, os_ = ORC.qwz_quant_int8(w, B)
    binding.qwz_dequant_int8(codes, scales, back, B)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(codes), oc, "int8 codes")
    assert_bits_equal(to_host(scales), os_, "scales")
    if q["replica"]:
        assert_bits_equal(to_host(rep), orep, "bf16 replica")
    assert_bits_equal(to_host(back), ORC.qwz_dequant_int8(oc, os_, B), "dequantized bf16")


SR_SEEDS = list(range(40))


def draw_sr(seed: int) -> dict:
    rng = np.random.default_rng(9_000_011 * seed + 3)
    n = int(rng.integers(1, 64)) if rng.integers(0, 4) == 0 else int(rng.integers(1, 1 << 19))
    return dict(n=n, offset=int(rng.integers(0, 8)) * 8,
                seed=int(rng.integers(0, 1 << 32)), step0=int(rng.integers(0, 1 << 32)),
                ratio=float(rng.choice([1.0, 1e-2, 1e-4, 1e-8])))


@pytest.mark.parametrize("seed", SR_SEEDS,
                         ids=[f"s{s}-n{draw_sr(s)['n']}" for s in SR_SEEDS])
def test_random_sr_accumulate(dev, seed):
    """bf16 stochastic-rounding accumulate of a random length, starting at a
    random 16-byte-aligned offset into its buffers, with random seed and step
    counters and a random source-to-destination magnitude ratio, over three
    micro-steps ("Stochastic rounding", vector_add)."""
    p = draw_sr(seed)
    n, off = p["n"], p["offset"]
    rng = np.random.default_rng(seed)

    def bf16(x):
        return wl.as_u16(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)).copy()

    dst = bf16(rng.standard_normal(n))
    dbuf = torch.zeros(n + off, dtype=torch.bfloat16, device=dev)
    sbuf = torch.zeros(n + off, dtype=torch.bfloat16, device=dev)
    dbuf[off:].copy_(to_dev(dst, dev))
    for t in range(3):
        step = (p["step0"] + t) & 0xFFFFFFFF
        src = bf16(rng.standard_normal(n) * p["ratio"])
        sbuf[off:].copy_(to_dev(src, dev))
        binding.sr_accumulate_bf16(dbuf[off:], sbuf[off:], seed=p["seed"], step=step)
        torch.cuda.synchronize()
        ORC.sr_accumulate_bf16(dst, src, seed=p["seed"], step=step)
        assert_bits_equal(to_host(dbuf[off:]), dst, f"dst, micro-step {t}")
        assert not to_host(sbuf).any(), f"source not zeroed, micro-step {t}"
        assert not to_host(dbuf[:off]).any(), "write before the destination"
