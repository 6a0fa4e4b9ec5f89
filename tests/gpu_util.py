"""Helpers for the GPU parity tests: device fixture, host<->device moves of
bf16 bit patterns, and the comparison rules.

Comparison rules (GPU against the CPU oracle on identical inputs):
  * integer codes, scales, bf16 stochastic-rounding outputs and zeroed
    sources: bit-exact;
  * fp32 error buffers and fp32 reduced sums: |gpu - cpu| <= 1e-6 * ref,
    ref being the magnitude sum of the terms (so near-zero sums cannot blow
    the relative error up); both sides run the same operations in the same
    order, so the tests also require bit equality;
  * bf16 reduced outputs: within 1 bf16 ulp (bit equality also required).
"""
import numpy as np
import pytest
import torch

from weight_communication_gb300 import build, workloads as wl


def ensure_built():
    srcs = build.sources()
    if not build.LIB.exists() or build.LIB.stat().st_mtime < max(p.stat().st_mtime for p in srcs):
        build.build()


@pytest.fixture(scope="session")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    return torch.device("cuda:0")


def to_dev(a: np.ndarray, dev) -> torch.Tensor:
    """Host numpy array -> device tensor with the same bytes (uint16 -> bf16)."""
    if a.dtype == np.uint16:
        return wl.from_u16(a, dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return wl.as_u16(t)
    return t.detach().cpu().numpy()


def assert_bits_equal(gpu: np.ndarray, cpu: np.ndarray, what: str):
    g = np.ascontiguousarray(gpu).view(np.uint8)
    c = np.ascontiguousarray(cpu).view(np.uint8)
    assert g.shape == c.shape, (what, g.shape, c.shape)
    if not np.array_equal(g, c):
        bad = np.flatnonzero(g != c)
        raise AssertionError(f"{what}: {bad.size} differing bytes, first at byte {bad[0]}")


def assert_f32_parity(gpu: np.ndarray, cpu: np.ndarray, ref: np.ndarray, what: str):
    """The fp32 bar (1e-6 of the magnitude reference), then bit equality."""
    gpu = gpu.astype(np.float64)
    cpu64 = cpu.astype(np.float64)
    err = np.abs(gpu - cpu64)
    lim = 1e-6 * np.abs(ref).astype(np.float64) + 1e-45
    assert np.all(err <= lim), f"{what}: max err {err.max()} exceeds 1e-6 of the reference"
    assert_bits_equal(gpu.astype(np.float32), cpu, what)


def assert_bf16_parity(gpu_u16: np.ndarray, cpu_u16: np.ndarray, what: str):
    """Within one bf16 ulp (as ordered integers), then bit equality."""
    def ordered(h):
        h = h.astype(np.int32)
        return np.where(h & 0x8000, -(h & 0x7FFF), h)
    d = np.abs(ordered(gpu_u16) - ordered(cpu_u16))
    assert d.max(initial=0) <= 1, f"{what}: {int((d > 1).sum())} values differ by more than 1 ulp"
    assert_bits_equal(gpu_u16, cpu_u16, what)


def deq_magnitude(codes: np.ndarray, scales: np.ndarray, B: int) -> np.ndarray:
    """|q| * scale per position (fp64), used to build magnitude references."""
    lo = (codes & 0x0F).astype(np.int16)
    hi = (codes >> 4).astype(np.int16)
    q = np.empty(codes.size * 2, np.int16)
    q[0::2], q[1::2] = lo, hi
    q[q >= 8] -= 16
    return np.abs(q).astype(np.float64) * np.repeat(scales.astype(np.float64), B)
