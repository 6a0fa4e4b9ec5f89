"""CPU oracle for the quantized-gradient hot path (ctypes over oracle.c).

TEST INFRASTRUCTURE ONLY.  The product (the CUDA library and its binding)
never imports this package; only the tests, the smoke check and the
benchmark's CPU-baseline leg do.  It shares no code with the GPU path: the C
source here is the whole definition, and its Python side only moves numpy
arrays in and out.

Sources (see oracle.c for the step-by-step statement):
  * "Merge LoCo with Zero++" (DeepSpeed PR #6730), Overview and review thread:
    error feedback on 4-bit gradients, one error buffer per parameter, two
    LoCo parameters.
  * "ZeROPlusPlus.md", §1.2 ZeRO++: qgZ (block int4, all-to-all, full-precision
    reduce, intra- then inter-node) and qwZ (block int8 weights).
  * "Zero 2 #593" (llm.c), review of vector_add: fp32 sum with stochastic
    rounding to bf16, source zeroing fused in.

Every function is pinned by tests/test_oracle_*.py; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import subprocess
import sys
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "oracle.c"
BUILD_DIR = _HERE / "_build"
LIB_PATH = BUILD_DIR / "liboracle.so"

# -ffp-contract=off matters: gcc on aarch64 fuses a*b+c by default.
CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
          "-fno-strict-aliasing", "-fPIC", "-shared", "-Wall", "-Wextra",
          "-fvisibility=hidden"]


def build(source: Path = SOURCE, out: Path = LIB_PATH, extra: list[str] | None = None) -> Path:
    """Compile oracle.c (or a given variant of it) into a shared library."""
    out = Path(out)
    out.parent.mkdir(parents=True, exist_ok=True)
    cmd = ["gcc", *CFLAGS, *(extra or []), str(source), "-o", str(out), "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale(lib: Path, src: Path) -> bool:
    return not lib.exists() or lib.stat().st_mtime < src.stat().st_mtime


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_F = ctypes.c_float
_U32 = ctypes.c_uint32
_U16 = ctypes.c_uint16

_SIGS = {
    "orc_max_block": (_I, []),
    "orc_bf16_to_f32": (ctypes.c_float, [_U16]),
    "orc_f32_to_bf16_rne": (_U16, [_F]),
    "orc_quant_block": (None, [_P, _I, _I, _P, _P]),
    "orc_dequant": (ctypes.c_float, [_I, _F]),
    "orc_get_nibble": (_I, [_P, _I64]),
    "orc_send_position": (_I64, [_I64, _I, _I]),
    "orc_ef_quant_int4_rank": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _F, _F]),
    "orc_ef_quant_int4": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _F, _F]),
    "orc_dequant_reduce_dest": (None, [_P, _P, _I64, _I, _I, _I, _I, _F, _P, _I]),
    "orc_dequant_reduce_dest_range": (None, [_P, _P, _I64, _I, _I, _I, _I, _I64, _I64, _F, _P, _I]),
    "orc_dequant_reduce": (None, [_P, _P, _I64, _I, _I, _I, _F, _P, _I]),
    "orc_dequant_reduce_requant_unit": (_I, [_P, _P, _I64, _I, _I, _I, _I, _I, _P, _P]),
    "orc_dequant_reduce_requant": (_I, [_P, _P, _I64, _I, _I, _I, _P, _P]),
    "orc_dequant_reduce_requant_unit_ef": (_I, [_P, _P, _I64, _I, _I, _I, _I, _I, _P, _P, _P, _F, _F]),
    "orc_dequant_reduce_requant_ef": (_I, [_P, _P, _I64, _I, _I, _I, _P, _P, _P, _F, _F]),
    "orc_ef_quant_int4_rank_bf16ef": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _F, _F]),
    "orc_ef_quant_int4_bf16ef": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _F, _F]),
    "orc_ef_quant_int4_rank_int8ef": (_I, [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _F, _F]),
    "orc_ef_quant_int4_int8ef": (_I, [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _F, _F]),
    "orc_qwz_quant_replica_int8": (_I, [_P, _P, _P, _P, _I64, _I]),
    "orc_qwz_quant_int8": (_I, [_P, _P, _P, _I64, _I]),
    "orc_qwz_dequant_int8": (None, [_P, _P, _P, _I64, _I]),
    "orc_fmix32": (_U32, [_U32]),
    "orc_mix32": (_U32, [_U32]),
    "orc_sr_bits": (_U32, [_U32, _U32, _U32]),
    "orc_sr_round": (_U16, [_F, _U32]),
    "orc_sr_accumulate_bf16": (None, [_P, _P, _I64, _U32, _U32]),
}

MAX_BLOCK = 8192  # the oracle's per-block scratch holds this many values
EBLOCK = -1       # status of a C call refused for a block size outside [1, MAX_BLOCK]


def _status(rc: int, name: str) -> None:
    """The C functions with per-block scratch check B themselves and return a
    nonzero status, having written nothing, when it is out of range."""
    if rc != 0:
        raise ValueError(f"{name} refused the call (status {rc}): block size outside "
                         f"[1, {MAX_BLOCK}]")


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _check_qgz(N: int, R: int, G: int, B: int) -> tuple[int, int, int]:
    if R < 1 or G < 1 or R % G:
        raise ValueError(f"need R >= 1, G >= 1 and G | R (R={R}, G={G})")
    if N <= 0 or N % R:
        raise ValueError(f"R must divide N (N={N}, R={R})")
    S = N // R
    if B < 2 or B % 2 or B > MAX_BLOCK or S % B:
        raise ValueError(f"B must be even, <= {MAX_BLOCK} and divide S={S} (B={B})")
    return S, R // G, S // B


class Oracle:
    """numpy-facing wrapper around one build of oracle.c.

    Arrays: bf16 tensors travel as uint16 bit patterns; codes as uint8 (int4
    packed) or int8; everything else as float32.  Functions that the C code
    updates in place (error buffers, SR dst/src) are updated in place here.
    """

    def __init__(self, lib_path: Path | str | None = None):
        if lib_path is None:
            if _stale(LIB_PATH, SOURCE):
                build()
            lib_path = LIB_PATH
        self.lib_path = Path(lib_path)
        self._lib = ctypes.CDLL(str(self.lib_path))
        for name, (res, args) in _SIGS.items():
            fn = getattr(self._lib, name)
            fn.restype = res
            fn.argtypes = args

    # -- scalar helpers -------------------------------------------------
    def bf16_to_f32(self, h: int) -> float:
        return self._lib.orc_bf16_to_f32(h)

    def f32_to_bf16(self, x: float) -> int:
        return self._lib.orc_f32_to_bf16_rne(x)

    def fmix32(self, h: int) -> int:
        return self._lib.orc_fmix32(h)

    def mix32(self, z: int) -> int:
        return self._lib.orc_mix32(z)

    def sr_bits(self, seed: int, step: int, i: int) -> int:
        return self._lib.orc_sr_bits(seed, step, i)

    def sr_round(self, x: float, r: int) -> int:
        return self._lib.orc_sr_round(x, r)

    def send_position(self, slice_: int, R: int, G: int) -> int:
        return self._lib.orc_send_position(slice_, R, G)

    def get_nibble(self, codes: np.ndarray, pos: int) -> int:
        return self._lib.orc_get_nibble(_ptr(codes), pos)

    # -- vector helpers -------------------------------------------------
    def bf16_round(self, x: np.ndarray) -> np.ndarray:
        """float32 array -> bf16 bit patterns (uint16), element by element."""
        x = np.ascontiguousarray(x, dtype=np.float32).ravel()
        f = self._lib.orc_f32_to_bf16_rne
        return np.array([f(float(v)) for v in x], dtype=np.uint16)

    def quant_block(self, x: np.ndarray, qmax: int) -> tuple[np.ndarray, float]:
        x = np.ascontiguousarray(x, dtype=np.float32)
        q = np.empty(x.size, dtype=np.int8)
        s = np.zeros(1, dtype=np.float32)
        self._lib.orc_quant_block(_ptr(x), x.size, qmax, _ptr(q), _ptr(s))
        return q, float(s[0])

    def unpack_int4(self, codes: np.ndarray, n: int) -> np.ndarray:
        """Signed int4 codes of the first n positions, element by element."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        return np.array([self.get_nibble(codes, i) for i in range(n)], dtype=np.int8)

    # -- qgZ --------------------------------------------------------------
    def ef_quant_int4(self, g: np.ndarray, ef: np.ndarray | None, N: int, R: int,
                      G: int, B: int, s: float, beta: float):
        """All ranks.  g: uint16 [R*N]; ef: float32 [R*N] updated in place.
        Returns (codes uint8 [R*N/2], scales float32 [R*N/B])."""
        _check_qgz(N, R, G, B)
        assert g.dtype == np.uint16 and g.size == R * N
        if ef is not None:
            assert ef.dtype == np.float32 and ef.size == R * N
        codes = np.zeros(R * N // 2, dtype=np.uint8)
        scales = np.zeros(R * N // B, dtype=np.float32)
        _status(self._lib.orc_ef_quant_int4(_ptr(g), _ptr(ef), _ptr(codes), _ptr(scales),
                                    N, R, G, B, s, beta), "orc_ef_quant_int4")
        return codes, scales

    def ef_quant_int4_rank(self, g_r: np.ndarray, ef_r: np.ndarray | None, N: int,
                           R: int, G: int, B: int, s: float, beta: float):
        """One rank (its N elements).  Returns (codes [N/2], scales [N/B])."""
        _check_qgz(N, R, G, B)
        assert g_r.dtype == np.uint16 and g_r.size == N
        codes = np.zeros(N // 2, dtype=np.uint8)
        scales = np.zeros(N // B, dtype=np.float32)
        _status(self._lib.orc_ef_quant_int4_rank(_ptr(g_r), _ptr(ef_r), _ptr(codes),
                                         _ptr(scales), N, R, G, B, s, beta), "orc_ef_quant_int4_rank")
        return codes, scales

    def dequant_reduce(self, codes, scales, N, R, G, B, out_scale=1.0, out_bf16=False):
        """Every destination; returns [R*S] float32 or uint16 (bf16 bits)."""
        _check_qgz(N, R, G, B)
        out = np.zeros(N, dtype=np.uint16 if out_bf16 else np.float32)
        self._lib.orc_dequant_reduce(_ptr(codes), _ptr(scales), N, R, G, B,
                                     out_scale, _ptr(out), int(out_bf16))
        return out

    def dequant_reduce_dest(self, codes, scales, N, R, G, B, k, out_scale=1.0,
                            out_bf16=False):
        """Destination k only; returns [S]."""
        S, _, _ = _check_qgz(N, R, G, B)
        out = np.zeros(S, dtype=np.uint16 if out_bf16 else np.float32)
        self._lib.orc_dequant_reduce_dest(_ptr(codes), _ptr(scales), N, R, G, B, k,
                                          out_scale, _ptr(out), int(out_bf16))
        return out

    def dequant_reduce_dest_range(self, codes, scales, N, R, G, B, k, i0, i1, out_scale=1.0,
                                  out_bf16=False):
        """Outputs [i0, i1) of destination k; returns [i1 - i0]."""
        S, _, _ = _check_qgz(N, R, G, B)
        if not 0 <= i0 <= i1 <= S:
            raise ValueError(f"need 0 <= i0 <= i1 <= S={S} (i0={i0}, i1={i1})")
        out = np.zeros(i1 - i0, dtype=np.uint16 if out_bf16 else np.float32)
        self._lib.orc_dequant_reduce_dest_range(_ptr(codes), _ptr(scales), N, R, G, B, k, i0, i1,
                                                out_scale, _ptr(out), int(out_bf16))
        return out

    def dequant_reduce_requant(self, codes, scales, N, R, G, B):
        """Hop 1, every unit.  Returns (codes [R*G*S/2], scales [R*G*S/B])."""
        S, _, _ = _check_qgz(N, R, G, B)
        oc = np.zeros(R * G * S // 2, dtype=np.uint8)
        os_ = np.zeros(R * G * S // B, dtype=np.float32)
        _status(self._lib.orc_dequant_reduce_requant(_ptr(codes), _ptr(scales), N, R, G, B,
                                             _ptr(oc), _ptr(os_)), "orc_dequant_reduce_requant")
        return oc, os_

    def dequant_reduce_requant_unit(self, codes, scales, N, R, G, B, g, l):
        """Hop 1, unit (g, l).  Returns (codes [G*S/2], scales [G*S/B])."""
        S, _, _ = _check_qgz(N, R, G, B)
        oc = np.zeros(G * S // 2, dtype=np.uint8)
        os_ = np.zeros(G * S // B, dtype=np.float32)
        _status(self._lib.orc_dequant_reduce_requant_unit(_ptr(codes), _ptr(scales), N, R, G,
                                                  B, g, l, _ptr(oc), _ptr(os_)), "orc_dequant_reduce_requant_unit")
        return oc, os_

    def dequant_reduce_requant_ef(self, codes, scales, N, R, G, B, e1, s, beta):
        """Hop 1 with error feedback on the requantization; e1 float32
        [R*G*S] (unit order) updated in place, or None."""
        S, _, _ = _check_qgz(N, R, G, B)
        if e1 is not None:
            assert e1.dtype == np.float32 and e1.size == R * G * S
        oc = np.zeros(R * G * S // 2, dtype=np.uint8)
        os_ = np.zeros(R * G * S // B, dtype=np.float32)
        _status(self._lib.orc_dequant_reduce_requant_ef(_ptr(codes), _ptr(scales), N, R, G, B,
                                                _ptr(oc), _ptr(os_), _ptr(e1), s, beta), "orc_dequant_reduce_requant_ef")
        return oc, os_

    def dequant_reduce_requant_unit_ef(self, codes, scales, N, R, G, B, g, l, e1u, s, beta):
        """Hop 1 with error feedback, unit (g, l); e1u float32 [G*S] in place."""
        S, _, _ = _check_qgz(N, R, G, B)
        oc = np.zeros(G * S // 2, dtype=np.uint8)
        os_ = np.zeros(G * S // B, dtype=np.float32)
        _status(self._lib.orc_dequant_reduce_requant_unit_ef(_ptr(codes), _ptr(scales), N, R, G, B,
                                                     g, l, _ptr(oc), _ptr(os_), _ptr(e1u),
                                                     s, beta), "orc_dequant_reduce_requant_unit_ef")
        return oc, os_

    def ef_quant_int4_bf16ef(self, g: np.ndarray, e16: np.ndarray, N: int, R: int, G: int,
                             B: int, s: float, beta: float):
        """All ranks with a bf16 error buffer (uint16 [R*N], in place)."""
        _check_qgz(N, R, G, B)
        assert g.dtype == np.uint16 and g.size == R * N
        assert e16.dtype == np.uint16 and e16.size == R * N
        codes = np.zeros(R * N // 2, dtype=np.uint8)
        scales = np.zeros(R * N // B, dtype=np.float32)
        _status(self._lib.orc_ef_quant_int4_bf16ef(_ptr(g), _ptr(e16), _ptr(codes), _ptr(scales),
                                           N, R, G, B, s, beta), "orc_ef_quant_int4_bf16ef")
        return codes, scales

    def ef_quant_int4_rank_bf16ef(self, g_r, e16_r, N, R, G, B, s, beta):
        _check_qgz(N, R, G, B)
        codes = np.zeros(N // 2, dtype=np.uint8)
        scales = np.zeros(N // B, dtype=np.float32)
        _status(self._lib.orc_ef_quant_int4_rank_bf16ef(_ptr(g_r), _ptr(e16_r), _ptr(codes),
                                                _ptr(scales), N, R, G, B, s, beta), "orc_ef_quant_int4_rank_bf16ef")
        return codes, scales

    def ef_quant_int4_int8ef(self, g: np.ndarray, e8: np.ndarray, e8s: np.ndarray, N: int,
                             R: int, G: int, B: int, s: float, beta: float):
        """All ranks with an int8 error buffer: e8 int8 [R*N] codes and e8s
        float32 [R*N/B] scales (gradient order), both in place."""
        _check_qgz(N, R, G, B)
        assert g.dtype == np.uint16 and g.size == R * N
        assert e8.dtype == np.int8 and e8.size == R * N
        assert e8s.dtype == np.float32 and e8s.size == R * N // B
        codes = np.zeros(R * N // 2, dtype=np.uint8)
        scales = np.zeros(R * N // B, dtype=np.float32)
        _status(self._lib.orc_ef_quant_int4_int8ef(_ptr(g), _ptr(e8), _ptr(e8s), _ptr(codes),
                                           _ptr(scales), N, R, G, B, s, beta), "orc_ef_quant_int4_int8ef")
        return codes, scales

    # -- qwZ --------------------------------------------------------------
    def qwz_quant_int8(self, w: np.ndarray, B: int):
        n = w.size
        if B < 1 or B > MAX_BLOCK or n % B:
            raise ValueError(f"B must divide n and be <= {MAX_BLOCK}")
        assert w.dtype == np.uint16
        codes = np.zeros(n, dtype=np.int8)
        scales = np.zeros(n // B, dtype=np.float32)
        _status(self._lib.orc_qwz_quant_int8(_ptr(w), _ptr(codes), _ptr(scales), n, B), "orc_qwz_quant_int8")
        return codes, scales

    def qwz_dequant_int8(self, codes: np.ndarray, scales: np.ndarray, B: int):
        n = codes.size
        out = np.zeros(n, dtype=np.uint16)
        self._lib.orc_qwz_dequant_int8(_ptr(codes), _ptr(scales), _ptr(out), n, B)
        return out

    def qwz_quant_replica_int8(self, w: np.ndarray, B: int):
        """(codes, scales, bf16 replica) of the weights."""
        n = w.size
        if B < 1 or B > MAX_BLOCK or n % B:
            raise ValueError(f"B must divide n and be <= {MAX_BLOCK}")
        codes = np.zeros(n, dtype=np.int8)
        scales = np.zeros(n // B, dtype=np.float32)
        rep = np.zeros(n, dtype=np.uint16)
        _status(self._lib.orc_qwz_quant_replica_int8(_ptr(w), _ptr(codes), _ptr(scales), _ptr(rep), n, B), "orc_qwz_quant_replica_int8")
        return codes, scales, rep

    # -- SR accumulate ------------------------------------------------------
    def sr_accumulate_bf16(self, dst: np.ndarray, src: np.ndarray, seed: int, step: int):
        """In place: dst <- SR(dst + src), src <- 0 (uint16 bf16 bits)."""
        assert dst.dtype == np.uint16 and src.dtype == np.uint16 and dst.size == src.size
        if dst.size >= 2**32:
            raise ValueError("element index must fit in 32 bits")
        self._lib.orc_sr_accumulate_bf16(_ptr(dst), _ptr(src), dst.size, seed, step)


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from oracle.c (compiled on first use if missing)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


if __name__ == "__main__":  # python -m oracle  -> (re)build
    print(build())
    sys.exit(0)
