"""Pins for the oracle's qwZ int8 block weight quantization, and the wire
volume figures of ZeROPlusPlus.md (abstract and §1.2).

qwZ (ZeROPlusPlus.md §1.2, first item): weights go fp16 -> int8 with
block-based quantization, halving the forward all-gather.  Pins:
  * round trip |w - w'| <= scale (1/2 + 2^-18) + half a bf16 step of w';
  * dequantization is the bf16 rounding of code * scale (torch's conversion);
  * zero blocks; a block reaching +-127;
  * the page's volume arithmetic from the sizes the oracle produces.
"""
from pathlib import Path

import numpy as np
import pytest
import torch

from weight_communication_gb300 import workloads as wl

GOLDEN = Path(__file__).parent / "golden" / "zeropp_volume.txt"


def _bf16_to_f64(h):
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("B", [2048, 256, 64])
def test_qwz_round_trip(orc, B):
    w = wl.draw_bf16(B * 40, 0.02, seed=41, outlier_frac=1e-3, outlier_mult=30.0)
    wu = wl.as_u16(w).copy()
    codes, scales = orc.qwz_quant_int8(wu, B)
    back = orc.qwz_dequant_int8(codes, scales, B)
    wf = w.double().numpy()
    bf = _bf16_to_f64(back)
    sc = np.repeat(scales.astype(np.float64), B)
    half_ulp = np.abs(bf) * 2.0**-8
    assert np.all(np.abs(wf - bf) <= sc * (0.5 + 2.0**-18) + half_ulp)
    assert np.all(np.abs(codes.reshape(-1, B)).max(axis=1) == 127)
    # dequantization = torch's bf16 rounding of the fp32 product
    prod = torch.from_numpy(codes.astype(np.float32) * np.repeat(scales, B))
    ref = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(back, ref)


def test_qwz_zero_block_and_exact_block(orc):
    B = 16
    w = np.zeros(2 * B, np.float32)
    w[B:] = np.arange(B, dtype=np.float32) * 8 - 60      # absmax 60 -> scale 60/127
    w[B] = -127.0                                         # absmax 127 -> scale 1
    wu = wl.as_u16(torch.from_numpy(w).to(torch.bfloat16)).copy()
    codes, scales = orc.qwz_quant_int8(wu, B)
    assert scales[0] == 0.0 and not codes[:B].any()
    assert scales[1] == 1.0
    assert codes[B:].tolist() == [-127] + [int(v) for v in w[B + 1:]]
    back = orc.qwz_dequant_int8(codes, scales, B)
    assert np.array_equal(back[B:], wu[B:])                # exact round trip


def test_wire_volume_matches_the_page(orc):
    want = {}
    for line in GOLDEN.read_text().splitlines():
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            want[k] = float(v)
    n = 1 << 16                                            # parameters (M)
    fp16_bytes = 2 * n
    wu = wl.as_u16(wl.draw_bf16(n, 0.02, 1)).copy()
    q8, s8 = orc.qwz_quant_int8(wu, 2048)
    c4, s4 = orc.ef_quant_int4(wu, None, n, 1, 1, 256, 1.0, 0.0)
    # codes alone, in units of M fp16 elements
    assert q8.nbytes / fp16_bytes == want["zeropp_fwd_weights"]
    assert c4.nbytes / fp16_bytes == want["zeropp_gradients"]
    zeropp = (q8.nbytes + 0 + c4.nbytes) / fp16_bytes
    assert zeropp == want["zeropp_total"] == want["zeropp_fwd_weights"] + \
        want["zeropp_bwd_weights"] + want["zeropp_gradients"]
    assert want["zero_total"] / zeropp == 4.0
    # with the per-block fp32 scales the gradient message is 0.2578 M at B=256
    assert (c4.nbytes + s4.nbytes) / fp16_bytes == pytest.approx(0.25 + 4 / (2 * 256))
    assert (q8.nbytes + s8.nbytes) / fp16_bytes == pytest.approx(0.5 + 4 / (2 * 2048))
