"""GPU parity of qwZ int8 quantize/dequantize and of the SR accumulate
(through the C ABI) against the CPU oracle: bit-exact codes, scales, bf16
outputs and zeroed sources, over ragged sizes, every block size and edge
values; full-size runs of the qwZ and SR workloads are in
test_parity_fullsize.py."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bits_equal, dev, to_dev, to_host
from weight_communication_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

ORC = oracle.get()


def weights_with_edges(n: int, B: int, seed: int) -> np.ndarray:
    w = wl.as_u16(wl.draw_bf16(n, 0.02, seed, outlier_frac=1e-3, outlier_mult=30.0)).copy()
    nb = n // B
    rng = np.random.default_rng(seed)
    tiny = np.float32(np.finfo(np.float32).tiny)
    specials = [np.zeros(B, np.float32),
                np.float32(1e-39) * rng.standard_normal(B).astype(np.float32),
                np.concatenate([[np.float32(127) * tiny], np.zeros(B - 1, np.float32)]),
                np.concatenate([[np.float32(126) * tiny], np.zeros(B - 1, np.float32)]),
                np.concatenate([[np.float32(127.0)],
                                (np.arange(B - 1) % 255 - 127 + 0.5).astype(np.float32)])]
    for j, b in enumerate(rng.choice(nb, size=min(nb, len(specials)), replace=False)):
        blk = torch.from_numpy(specials[j]).to(torch.bfloat16)
        w[b * B:(b + 1) * B] = wl.as_u16(blk)
    return w


@pytest.mark.parametrize("n,B", [(2048 * 37, 2048), (4096 * 3, 4096), (256 * 101, 256),
                                 (32 * 77, 32), (64 * 5, 64), (128 * 3, 128), (512 * 9, 512),
                                 (1024, 1024)])
def test_qwz_parity(dev, n, B):
    w = weights_with_edges(n, B, seed=n + B)
    wd = to_dev(w, dev)
    codes = torch.empty(n, dtype=torch.int8, device=dev)
    scales = torch.empty(n // B, dtype=torch.float32, device=dev)
    back = torch.empty(n, dtype=torch.bfloat16, device=dev)
    binding.qwz_quant_int8(wd, codes, scales, B)
    binding.qwz_dequant_int8(codes, scales, back, B)
    torch.cuda.synchronize()
    oc, os_ = ORC.qwz_quant_int8(w, B)
    assert_bits_equal(to_host(codes), oc, "int8 codes")
    assert_bits_equal(to_host(scales), os_, "scales")
    assert_bits_equal(to_host(back), ORC.qwz_dequant_int8(oc, os_, B), "dequantized bf16")


@pytest.mark.parametrize("n", [8, 7, 1, 1000, 4096 * 33 + 5, 1 << 20])
def test_sr_accumulate_parity(dev, n):
    rng = np.random.default_rng(n)
    dst = wl.as_u16(torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(torch.bfloat16)).copy()
    src = wl.as_u16(torch.from_numpy((rng.standard_normal(n) * 1e-2).astype(np.float32))
                    .to(torch.bfloat16)).copy()
    # edge values: zeros, signed zeros, values that cancel, subnormals, large
    k = min(n, 6)
    dst[:k] = np.array([0x0000, 0x8000, 0x3F80, 0x0001, 0x7F00, 0xC2F6], np.uint16)[:k]
    src[:k] = np.array([0x8000, 0x8000, 0xBF80, 0x0001, 0x7E80, 0x3C00], np.uint16)[:k]
    dd, sd = to_dev(dst, dev), to_dev(src, dev)
    for step in range(3):
        binding.sr_accumulate_bf16(dd, sd, seed=5, step=step)
        torch.cuda.synchronize()
        ORC.sr_accumulate_bf16(dst, src, seed=5, step=step)
        assert_bits_equal(to_host(dd), dst, f"dst step {step}")
        assert_bits_equal(to_host(sd), src, f"src step {step}")
        assert not src.any()
        # refill the source for the next step
        src = wl.as_u16(torch.from_numpy((rng.standard_normal(n) * 1e-2).astype(np.float32))
                        .to(torch.bfloat16)).copy()
        sd = to_dev(src, dev)


def test_sr_accumulate_unaligned_tail_stays_inside(dev):
    n = 4096 + 3
    pad = 64
    dst = torch.full((n + 2 * pad,), 1.5, dtype=torch.bfloat16, device=dev)
    src = torch.full((n + 2 * pad,), 0.25, dtype=torch.bfloat16, device=dev)
    binding.sr_accumulate_bf16(dst[pad:pad + n], src[pad:pad + n], seed=1, step=0)
    torch.cuda.synchronize()
    assert bool((dst[:pad] == 1.5).all()) and bool((dst[pad + n:] == 1.5).all())
    assert bool((src[:pad] == 0.25).all()) and bool((src[pad + n:] == 0.25).all())
    assert bool((src[pad:pad + n] == 0).all())
    assert bool((dst[pad:pad + n] == 1.75).all())    # 1.75 is exact in bf16
