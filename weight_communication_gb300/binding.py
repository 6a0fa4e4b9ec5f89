"""ctypes binding of libwc.so (include/wc.h): argument marshalling only.

Every function takes torch CUDA tensors, checks dtype, device, contiguity and
sizes, and calls the entry point of the same name on the tensors' current
stream.  All arithmetic happens in the CUDA kernels; there is no CPU or
PyTorch fallback -- if the library is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import os
from pathlib import Path

import torch

from . import build as _build

WC_OK, WC_EINVAL, WC_EALIGN, WC_ERANGE, WC_ECUDA = 0, -1, -2, -3, -4
WC_F32, WC_BF16 = 0, 1

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_F = ctypes.c_float
_U32 = ctypes.c_uint32

# name -> argtypes (all return int except the two informational calls)
SIGNATURES = {
    "wc_ef_quant_int4": [_P, _P, _P, _P, _I64, _I, _I, _I, _F, _F, _P],
    "wc_dequant_reduce": [_P, _P, _I64, _I, _I, _I, _F, _P, _I, _P],
    "wc_dequant_reduce_requant": [_P, _P, _I64, _I, _I, _I, _P, _P, _P],
    "wc_dequant_reduce_requant_ef": [_P, _P, _I64, _I, _I, _I, _P, _P, _P, _F, _F, _P],
    "wc_qgz_step_fused": [_P, _P, _P, _P, _I64, _I, _I, _F, _F, _F, _P, _I, _P],
    "wc_qgz_step_fused_bf16ef": [_P, _P, _P, _P, _I64, _I, _I, _F, _F, _F, _P, _I, _P],
    "wc_qgz_step_fused_int8ef": [_P, _P, _P, _P, _P, _I64, _I, _I, _F, _F, _F, _P, _I, _P],
    "wc_qgz_first_hop_fused": [_P, _P, _P, _P, _I64, _I, _I, _I, _F, _F, _P, _P, _P, _P],
    "wc_qgz_first_hop_fused_bf16ef": [_P, _P, _P, _P, _I64, _I, _I, _I, _F, _F, _P, _P, _P, _P],
    "wc_qgz_first_hop_fused_int8ef": [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _F, _F, _P, _P, _P,
                                      _P],
    "wc_ef_quant_int4_bf16ef": [_P, _P, _P, _P, _I64, _I, _I, _I, _F, _F, _P],
    "wc_ef_quant_int4_int8ef": [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _F, _F, _P],
    "wc_qwz_quant_int8": [_P, _P, _P, _I64, _I, _P],
    "wc_qwz_quant_replica_int8": [_P, _P, _P, _P, _I64, _I, _P],
    "wc_qwz_dequant_int8": [_P, _P, _P, _I64, _I, _P],
    "wc_sr_accumulate_bf16": [_P, _P, _I64, _U32, _U32, _P],
    "wc_checked_violations": [_I],
    "wc_last_error": [],
    "wc_version": [],
}


class WcError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


_lib: ctypes.CDLL | None = None


def library_path() -> Path:
    """The in-tree libwc.so, or the file named by the WC_LIBRARY environment
    variable (for instance the bounds-checked build)."""
    env = os.environ.get("WC_LIBRARY")
    return Path(env) if env else _build.LIB


def load(path: str | Path | None = None) -> ctypes.CDLL:
    """Load libwc.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else library_path()
    if not p.exists():
        raise RuntimeError(f"CUDA library {p} is missing: build it with "
                           "`python -m weight_communication_gb300.build`")
    lib = ctypes.CDLL(str(p))
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "wc_last_error" else ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def last_error() -> str:
    return load().wc_last_error().decode()


def version() -> int:
    return load().wc_version()


WC_CHECK_RESET, WC_CHECK_PROBE = 1, 2


def checked_violations(reset: bool = False, probe: bool = False) -> int:
    """wc_checked_violations: accesses a checked build skipped (synchronize
    first); probe adds one deliberate violation per kernel file first.
    Raises WcError on an ordinary build."""
    lib = load()
    rc = lib.wc_checked_violations((WC_CHECK_RESET if reset else 0) |
                                   (WC_CHECK_PROBE if probe else 0))
    if rc < 0:
        raise WcError("wc_checked_violations", rc, lib.wc_last_error().decode())
    return rc


def _call(device: torch.device, name: str, *args) -> None:
    """Calls the entry point with the tensors' GPU as the current device (the
    kernels launch on the current device)."""
    lib = load()
    with torch.cuda.device(device):
        rc = getattr(lib, name)(*args)
    if rc != WC_OK:
        raise WcError(name, rc, lib.wc_last_error().decode())


def _stream(t: torch.Tensor, stream: torch.cuda.Stream | None):
    """The launch stream: `stream`, which must belong to the tensors' GPU, or
    that GPU's current stream."""
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)
    if stream.device != t.device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {t.device}")
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor | None, name: str, dtype: torch.dtype, numel: int, device=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    return ctypes.c_void_p(t.data_ptr())


def ef_quant_int4(g: torch.Tensor, ef: torch.Tensor | None, codes: torch.Tensor,
                  scales: torch.Tensor, N: int, R: int, G: int, B: int,
                  err_scale: float = 1.0, err_beta: float = 0.0, stream=None) -> None:
    """wc_ef_quant_int4: g bf16 [R*N], ef fp32 [R*N] (in place) or None,
    codes uint8 [R*N/2], scales fp32 [R*N/B] -- all written in send order."""
    d = g.device
    _call(d, "wc_ef_quant_int4", _dev(g, "g", torch.bfloat16, R * N, d),
          _dev(ef, "ef", torch.float32, R * N, d), _dev(codes, "codes", torch.uint8, R * N // 2, d),
          _dev(scales, "scales", torch.float32, R * N // B, d), N, R, G, B, err_scale, err_beta,
          _stream(g, stream))


def dequant_reduce(codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, N: int,
                   R: int, G: int, B: int, out_scale: float = 1.0, stream=None) -> None:
    """wc_dequant_reduce: out fp32 or bf16 [R*S] = [N] in destination order.
    G == 1: codes/scales are the ranks' send buffers ([R*N/2], [R*N/B]);
    G > 1: they are the first hop's outputs ([G*N/2], [G*N/B])."""
    d = codes.device
    span = N * (G if G > 1 else R)
    if out.dtype == torch.float32:
        od = WC_F32
    elif out.dtype == torch.bfloat16:
        od = WC_BF16
    else:
        raise TypeError("out must be float32 or bfloat16")
    _call(d, "wc_dequant_reduce", _dev(codes, "codes", torch.uint8, span // 2, d),
          _dev(scales, "scales", torch.float32, span // B, d), N, R, G, B, out_scale,
          _dev(out, "out", out.dtype, N, d), od, _stream(codes, stream))


def dequant_reduce_requant(codes: torch.Tensor, scales: torch.Tensor, out_codes: torch.Tensor,
                           out_scales: torch.Tensor, N: int, R: int, G: int, B: int,
                           stream=None) -> None:
    """wc_dequant_reduce_requant: first hop; out_codes uint8 [G*N/2],
    out_scales fp32 [G*N/B] (unit u = g*L + l holds G*S values)."""
    d = codes.device
    _call(d, "wc_dequant_reduce_requant", _dev(codes, "codes", torch.uint8, R * N // 2, d),
          _dev(scales, "scales", torch.float32, R * N // B, d), N, R, G, B,
          _dev(out_codes, "out_codes", torch.uint8, G * N // 2, d),
          _dev(out_scales, "out_scales", torch.float32, G * N // B, d), _stream(codes, stream))


def dequant_reduce_requant_ef(codes: torch.Tensor, scales: torch.Tensor, out_codes: torch.Tensor,
                              out_scales: torch.Tensor, ef1: torch.Tensor, N: int, R: int, G: int,
                              B: int, err_scale: float = 1.0, err_beta: float = 0.0,
                              stream=None) -> None:
    """wc_dequant_reduce_requant_ef: first hop with error feedback on the
    requantization; ef1 fp32 [G*N] updated in place."""
    d = codes.device
    _call(d, "wc_dequant_reduce_requant_ef", _dev(codes, "codes", torch.uint8, R * N // 2, d),
          _dev(scales, "scales", torch.float32, R * N // B, d), N, R, G, B,
          _dev(out_codes, "out_codes", torch.uint8, G * N // 2, d),
          _dev(out_scales, "out_scales", torch.float32, G * N // B, d),
          _dev(ef1, "ef1", torch.float32, G * N, d), err_scale, err_beta, _stream(codes, stream))


def _fused_error(ef: torch.Tensor | None, ef_scales: torch.Tensor | None, n: int, B: int, d):
    """The fused entry point's suffix and error-buffer pointers for ef's
    dtype: fp32 (or None), bf16, or int8 with its block scales."""
    if ef is None or ef.dtype == torch.float32:
        if ef_scales is not None:
            raise ValueError("ef_scales goes with an int8 error buffer only")
        return "", [_dev(ef, "ef", torch.float32, n, d)]
    if ef.dtype == torch.bfloat16:
        if ef_scales is not None:
            raise ValueError("ef_scales goes with an int8 error buffer only")
        return "_bf16ef", [_dev(ef, "ef", torch.bfloat16, n, d)]
    if ef.dtype == torch.int8:
        if ef_scales is None:
            raise ValueError("an int8 error buffer needs ef_scales")
        return "_int8ef", [_dev(ef, "ef", torch.int8, n, d),
                           _dev(ef_scales, "ef_scales", torch.float32, n // B, d)]
    raise TypeError(f"ef must be float32, bfloat16 or int8, got {ef.dtype}")


def qgz_step_fused(g: torch.Tensor, ef: torch.Tensor | None, codes: torch.Tensor | None,
                   scales: torch.Tensor | None, out: torch.Tensor, N: int, R: int, B: int,
                   err_scale: float = 1.0, err_beta: float = 0.0, out_scale: float = 1.0,
                   stream=None, ef_scales: torch.Tensor | None = None) -> None:
    """wc_qgz_step_fused (fp32 or no error buffer), _bf16ef (bf16 ef) or
    _int8ef (int8 ef with fp32 ef_scales [R*N/B]): flat EF-quant +
    dequant-reduce in one kernel.  codes/scales (the send buffers) may both be
    None to skip writing them."""
    d = g.device
    if out.dtype == torch.float32:
        od = WC_F32
    elif out.dtype == torch.bfloat16:
        od = WC_BF16
    else:
        raise TypeError("out must be float32 or bfloat16")
    suffix, err = _fused_error(ef, ef_scales, R * N, B, d)
    _call(d, "wc_qgz_step_fused" + suffix, _dev(g, "g", torch.bfloat16, R * N, d), *err,
          _dev(codes, "codes", torch.uint8, R * N // 2, d),
          _dev(scales, "scales", torch.float32, R * N // B, d), N, R, B, err_scale, err_beta,
          out_scale, _dev(out, "out", out.dtype, N, d), od, _stream(g, stream))


def qgz_first_hop_fused(g: torch.Tensor, ef: torch.Tensor | None, codes: torch.Tensor | None,
                        scales: torch.Tensor | None, out_codes: torch.Tensor,
                        out_scales: torch.Tensor, N: int, R: int, G: int, B: int,
                        err_scale: float = 1.0, err_beta: float = 0.0, stream=None,
                        ef1: torch.Tensor | None = None,
                        ef_scales: torch.Tensor | None = None) -> None:
    """wc_qgz_first_hop_fused (fp32 or no error buffer), _bf16ef or _int8ef
    (by ef's dtype, as qgz_step_fused): every rank's EF-quant and the first
    hop in one kernel.  codes/scales (the send buffers) may both be None to
    skip writing them; out_codes/out_scales receive the first hop's output;
    ef1 (fp32 [G*N], or None) is the first hop's own error buffer."""
    d = g.device
    suffix, err = _fused_error(ef, ef_scales, R * N, B, d)
    _call(d, "wc_qgz_first_hop_fused" + suffix, _dev(g, "g", torch.bfloat16, R * N, d), *err,
          _dev(codes, "codes", torch.uint8, R * N // 2, d),
          _dev(scales, "scales", torch.float32, R * N // B, d), N, R, G, B, err_scale, err_beta,
          _dev(out_codes, "out_codes", torch.uint8, G * N // 2, d),
          _dev(out_scales, "out_scales", torch.float32, G * N // B, d),
          _dev(ef1, "ef1", torch.float32, G * N, d), _stream(g, stream))


def qwz_quant_int8(w: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, B: int,
                   stream=None) -> None:
    n = w.numel()
    d = w.device
    _call(d, "wc_qwz_quant_int8", _dev(w, "w", torch.bfloat16, n, d),
          _dev(codes, "codes", torch.int8, n, d), _dev(scales, "scales", torch.float32, n // B, d),
          n, B, _stream(w, stream))


def ef_quant_int4_bf16ef(g: torch.Tensor, ef16: torch.Tensor, codes: torch.Tensor,
                         scales: torch.Tensor, N: int, R: int, G: int, B: int,
                         err_scale: float = 1.0, err_beta: float = 0.0, stream=None) -> None:
    """wc_ef_quant_int4_bf16ef: as ef_quant_int4 with a bf16 error buffer."""
    d = g.device
    _call(d, "wc_ef_quant_int4_bf16ef", _dev(g, "g", torch.bfloat16, R * N, d),
          _dev(ef16, "ef16", torch.bfloat16, R * N, d),
          _dev(codes, "codes", torch.uint8, R * N // 2, d),
          _dev(scales, "scales", torch.float32, R * N // B, d), N, R, G, B, err_scale, err_beta,
          _stream(g, stream))


def ef_quant_int4_int8ef(g: torch.Tensor, ef8: torch.Tensor, ef8_scales: torch.Tensor,
                         codes: torch.Tensor, scales: torch.Tensor, N: int, R: int, G: int, B: int,
                         err_scale: float = 1.0, err_beta: float = 0.0, stream=None) -> None:
    """wc_ef_quant_int4_int8ef: as ef_quant_int4 with an int8 error buffer
    (ef8 int8 [R*N] codes, ef8_scales fp32 [R*N/B], both in place)."""
    d = g.device
    _call(d, "wc_ef_quant_int4_int8ef", _dev(g, "g", torch.bfloat16, R * N, d),
          _dev(ef8, "ef8", torch.int8, R * N, d),
          _dev(ef8_scales, "ef8_scales", torch.float32, R * N // B, d),
          _dev(codes, "codes", torch.uint8, R * N // 2, d),
          _dev(scales, "scales", torch.float32, R * N // B, d), N, R, G, B, err_scale, err_beta,
          _stream(g, stream))


def qwz_quant_replica_int8(w: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                           replica: torch.Tensor, B: int, stream=None) -> None:
    """wc_qwz_quant_replica_int8: codes, scales and the bf16 replica in one pass."""
    n = w.numel()
    d = w.device
    _call(d, "wc_qwz_quant_replica_int8", _dev(w, "w", torch.bfloat16, n, d),
          _dev(codes, "codes", torch.int8, n, d), _dev(scales, "scales", torch.float32, n // B, d),
          _dev(replica, "replica", torch.bfloat16, n, d), n, B, _stream(w, stream))


def qwz_dequant_int8(codes: torch.Tensor, scales: torch.Tensor, w_out: torch.Tensor, B: int,
                     stream=None) -> None:
    n = codes.numel()
    d = codes.device
    _call(d, "wc_qwz_dequant_int8", _dev(codes, "codes", torch.int8, n, d),
          _dev(scales, "scales", torch.float32, n // B, d),
          _dev(w_out, "w_out", torch.bfloat16, n, d), n, B, _stream(codes, stream))


def sr_accumulate_bf16(dst: torch.Tensor, src: torch.Tensor, seed: int, step: int,
                       stream=None) -> None:
    """dst <- SR_bf16(dst + src) in place; src <- 0."""
    n = dst.numel()
    d = dst.device
    _call(d, "wc_sr_accumulate_bf16", _dev(dst, "dst", torch.bfloat16, n, d),
          _dev(src, "src", torch.bfloat16, n, d), n, seed & 0xFFFFFFFF, step & 0xFFFFFFFF,
          _stream(dst, stream))
