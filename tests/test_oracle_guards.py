"""The oracle's C entry points refuse block sizes their per-block scratch
cannot hold.

Every function that quantizes one block at a time keeps the block on the
stack in arrays of orc_max_block() values, so it checks B itself, before
anything is written, instead of trusting its caller.  These tests call the
raw C symbols through ctypes (bypassing the Python wrapper's own checks) with
B = 16384 and B = 0 and expect the refusal status, with every output buffer
left as it was.  A guard only: no arithmetic is involved.
"""
import ctypes

import numpy as np
import pytest

import oracle

BIG = 2 * oracle.MAX_BLOCK  # 16384


def _p(a):
    return a.ctypes.data


@pytest.fixture(scope="module")
def lib(orc):
    return orc._lib


def test_max_block_exported(lib):
    assert lib.orc_max_block() == oracle.MAX_BLOCK == 8192


@pytest.mark.parametrize("B", [BIG, 0, -2])
def test_qgz_entry_points_refuse_block_size(lib, B):
    R, G = 2, 1
    N = 2 * BIG
    g = np.full(R * N, 0x3F80, np.uint16)               # 1.0 everywhere
    ef = np.full(R * N, 0.25, np.float32)
    e16 = np.full(R * N, 0x3E80, np.uint16)
    e8 = np.full(R * N, 3, np.int8)
    e8s = np.full(R * N // BIG, 0.5, np.float32)
    codes = np.full(R * N // 2, 0xAB, np.uint8)
    scales = np.full(R * N // BIG + 8, 7.0, np.float32)
    e1 = np.full(R * N, 0.125, np.float32)
    before = [a.copy() for a in (ef, e16, e8, e8s, codes, scales, e1)]
    calls = [
        ("orc_ef_quant_int4", lambda: lib.orc_ef_quant_int4(_p(g), _p(ef), _p(codes), _p(scales), N, R, G, B, 1.0, 0.5)),
        ("orc_ef_quant_int4_rank", lambda: lib.orc_ef_quant_int4_rank(_p(g), _p(ef), _p(codes), _p(scales), N, R, G, B, 1.0, 0.5)),
        ("orc_ef_quant_int4_bf16ef", lambda: lib.orc_ef_quant_int4_bf16ef(_p(g), _p(e16), _p(codes), _p(scales), N, R, G, B, 1.0, 0.5)),
        ("orc_ef_quant_int4_rank_bf16ef", lambda: lib.orc_ef_quant_int4_rank_bf16ef(_p(g), _p(e16), _p(codes), _p(scales), N, R, G, B, 1.0, 0.5)),
        ("orc_ef_quant_int4_int8ef", lambda: lib.orc_ef_quant_int4_int8ef(_p(g), _p(e8), _p(e8s), _p(codes), _p(scales), N, R, G, B, 1.0, 0.5)),
        ("orc_ef_quant_int4_rank_int8ef", lambda: lib.orc_ef_quant_int4_rank_int8ef(_p(g), _p(e8), _p(e8s), _p(codes), _p(scales), N, R, G, B, 1.0, 0.5)),
        ("orc_dequant_reduce_requant", lambda: lib.orc_dequant_reduce_requant(_p(codes), _p(scales), N, R, G, B, _p(codes), _p(scales))),
        ("orc_dequant_reduce_requant_ef", lambda: lib.orc_dequant_reduce_requant_ef(_p(codes), _p(scales), N, R, G, B, _p(codes), _p(scales), _p(e1), 1.0, 0.5)),
        ("orc_dequant_reduce_requant_unit", lambda: lib.orc_dequant_reduce_requant_unit(_p(codes), _p(scales), N, R, G, B, 0, 0, _p(codes), _p(scales))),
        ("orc_dequant_reduce_requant_unit_ef", lambda: lib.orc_dequant_reduce_requant_unit_ef(_p(codes), _p(scales), N, R, G, B, 0, 0, _p(codes), _p(scales), _p(e1), 1.0, 0.5)),
    ]
    for name, call in calls:
        assert call() == oracle.EBLOCK, name
        for a, b in zip((ef, e16, e8, e8s, codes, scales, e1), before):
            assert np.array_equal(a, b), f"{name} wrote before refusing"


@pytest.mark.parametrize("B", [BIG, 0])
def test_qwz_entry_points_refuse_block_size(lib, B):
    n = 2 * BIG
    w = np.full(n, 0x3F80, np.uint16)
    codes = np.full(n, 5, np.int8)
    scales = np.full(8, 3.0, np.float32)
    rep = np.full(n, 0x1234, np.uint16)
    assert lib.orc_qwz_quant_int8(_p(w), _p(codes), _p(scales), n, B) == oracle.EBLOCK
    assert lib.orc_qwz_quant_replica_int8(_p(w), _p(codes), _p(scales), _p(rep), n, B) == oracle.EBLOCK
    assert (codes == 5).all() and (scales == 3.0).all() and (rep == 0x1234).all()


def test_largest_block_is_accepted(lib):
    """B = orc_max_block() itself is within the scratch: it runs and returns 0."""
    B = oracle.MAX_BLOCK
    n = 2 * B
    w = np.full(n, 0x3F80, np.uint16)
    codes = np.zeros(n, np.int8)
    scales = np.zeros(n // B, np.float32)
    assert lib.orc_qwz_quant_int8(_p(w), _p(codes), _p(scales), n, B) == 0
    assert (codes == 127).all() and np.array_equal(scales, np.full(2, np.float32(1.0) / np.float32(127.0)))


def test_wrapper_raises_on_refusal(orc):
    """The Python wrapper turns a refusal into an exception (its own range
    check is bypassed here by calling the status check directly)."""
    with pytest.raises(ValueError, match="refused"):
        oracle._status(oracle.EBLOCK, "orc_qwz_quant_int8")
    assert ctypes.sizeof(ctypes.c_int) == 4
