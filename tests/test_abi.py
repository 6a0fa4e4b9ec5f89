"""The C-ABI library on the CPU: it loads, exports every entry point that
include/wc.h declares, and rejects bad arguments with the documented status
codes before touching the GPU (these calls launch nothing)."""
import ctypes
import re
from pathlib import Path

import pytest

from weight_communication_gb300 import binding, build

ROOT = Path(__file__).resolve().parent.parent
HEADERS = sorted((ROOT / "include").glob("*.h"))


def _declared():
    names = []
    for h in HEADERS:
        text = h.read_text()
        names += re.findall(r"^WC_API\s+[\w\s\*]+?\b(wc_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    csrc = ROOT / "weight_communication_gb300" / "csrc"
    srcs = build.sources() + HEADERS + sorted(csrc.glob("*.cuh")) + sorted(csrc.glob("*.h"))
    if not build.LIB.exists() or build.LIB.stat().st_mtime < max(p.stat().st_mtime for p in srcs):
        build.build()
    return binding.load()


def test_header_declares_the_hot_path(lib):
    names = _declared()
    for fn in ("wc_ef_quant_int4", "wc_dequant_reduce", "wc_dequant_reduce_requant",
               "wc_qwz_quant_int8", "wc_qwz_dequant_int8", "wc_sr_accumulate_bf16",
               "wc_last_error", "wc_version"):
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert names
    raw = ctypes.CDLL(str(build.LIB))
    for n in names:
        assert hasattr(raw, n), n
        assert n in binding.SIGNATURES, f"{n} has no binding"


def test_version(lib):
    assert lib.wc_version() == 10000


FAKE = 0x10000          # 16-byte aligned, never dereferenced: calls fail first
MIS = 0x10004


def _ef(lib, g=FAKE, ef=FAKE, codes=FAKE, scales=FAKE, N=1024, R=4, G=1, B=256):
    return lib.wc_ef_quant_int4(g, ef, codes, scales, N, R, G, B, 1.0, 0.0, None)


def test_ef_quant_argument_errors(lib):
    assert _ef(lib, R=0) == binding.WC_EINVAL
    assert _ef(lib, G=3) == binding.WC_EINVAL                     # G does not divide R
    assert _ef(lib, B=200) == binding.WC_EINVAL                   # not a power of two
    assert _ef(lib, B=16) == binding.WC_EINVAL                    # too small
    assert _ef(lib, B=2048) == binding.WC_EINVAL                  # too large for int4
    assert _ef(lib, N=1000) == binding.WC_EINVAL                  # R does not divide N... S%B
    assert _ef(lib, N=1026) == binding.WC_EINVAL
    assert _ef(lib, N=-4) == binding.WC_EINVAL
    assert _ef(lib, g=None) == binding.WC_EINVAL
    assert "g is NULL" in binding.last_error()
    assert _ef(lib, codes=MIS) == binding.WC_EALIGN
    assert _ef(lib, ef=MIS) == binding.WC_EALIGN
    assert _ef(lib, N=1 << 31, R=2, B=1024) == binding.WC_ERANGE
    assert _ef(lib, N=1 << 32, R=1, B=1024) == binding.WC_ERANGE
    # zero elements: a valid call that launches nothing
    assert _ef(lib, N=0, g=None, codes=None, scales=None) == binding.WC_OK


def test_reduce_argument_errors(lib):
    f = lib.wc_dequant_reduce
    assert f(FAKE, FAKE, 1024, 4, 1, 256, 1.0, FAKE, 7, None) == binding.WC_EINVAL
    assert f(FAKE, FAKE, 1024, 4, 1, 256, 1.0, MIS, 0, None) == binding.WC_EALIGN
    assert f(FAKE, None, 1024, 4, 1, 256, 1.0, FAKE, 0, None) == binding.WC_EINVAL
    assert f(FAKE, FAKE, 1024, 4, 3, 256, 1.0, FAKE, 0, None) == binding.WC_EINVAL
    assert f(None, None, 0, 4, 1, 256, 1.0, None, 0, None) == binding.WC_OK
    h = lib.wc_dequant_reduce_requant
    assert h(FAKE, FAKE, 1024, 4, 2, 100, FAKE, FAKE, None) == binding.WC_EINVAL
    assert h(FAKE, FAKE, 1024, 4, 2, 128, FAKE, MIS, None) == binding.WC_EALIGN
    assert h(FAKE, FAKE, (1 << 31) - 1024 * 1024, 1, 4, 1024, FAKE, FAKE, None) in \
        (binding.WC_EINVAL, binding.WC_ERANGE)


def test_qwz_and_sr_argument_errors(lib):
    q = lib.wc_qwz_quant_int8
    assert q(FAKE, FAKE, FAKE, 4096, 3000, None) == binding.WC_EINVAL
    assert q(FAKE, FAKE, FAKE, 4096, 8192, None) == binding.WC_EINVAL
    assert q(FAKE, FAKE, FAKE, 4000, 2048, None) == binding.WC_EINVAL
    assert q(MIS, FAKE, FAKE, 4096, 2048, None) == binding.WC_EALIGN
    assert q(FAKE, FAKE, FAKE, 1 << 32, 2048, None) == binding.WC_ERANGE
    d = lib.wc_qwz_dequant_int8
    assert d(FAKE, FAKE, None, 4096, 2048, None) == binding.WC_EINVAL
    s = lib.wc_sr_accumulate_bf16
    assert s(FAKE, FAKE + 64, 100, 1, 0, None) == binding.WC_EINVAL      # overlap
    assert "overlap" in binding.last_error()
    assert s(FAKE, MIS + 4096, 100, 1, 0, None) == binding.WC_EALIGN
    assert s(FAKE, FAKE + 4096, -1, 1, 0, None) == binding.WC_EINVAL
    assert s(FAKE, FAKE + 4096, 1 << 32, 1, 0, None) == binding.WC_ERANGE
    assert s(None, None, 0, 1, 0, None) == binding.WC_OK


def test_binding_rejects_cpu_tensors(lib):
    import torch
    g = torch.zeros(1024, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.ef_quant_int4(g, None, torch.zeros(512, dtype=torch.uint8),
                              torch.zeros(4), 256, 4, 1, 256)


def test_binding_rejects_a_stream_of_another_gpu():
    """A stream must belong to the tensors' GPU: a launch on another GPU's
    stream would fail in the driver, so the binding refuses it first."""
    import types
    import torch
    t = torch.empty(0, device="meta")
    other = types.SimpleNamespace(device=torch.device("cuda", 1), cuda_stream=0)
    with pytest.raises(ValueError, match="stream is on cuda:1"):
        binding._stream(t, other)
    same = types.SimpleNamespace(device=t.device, cuda_stream=1234)
    assert binding._stream(t, same).value == 1234


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        binding.load(tmp_path / "libwc.so")


def test_fused_step_argument_errors(lib):
    f = lib.wc_qgz_step_fused
    ok = (FAKE, FAKE, FAKE, FAKE, 8192, 8, 256, 1.0, 0.5, 1.0, FAKE, 0, None)
    def call(**kw):
        a = list(ok)
        names = ["g", "ef", "codes", "scales", "N", "R", "B", "s", "beta", "os", "out", "dt", "st"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)
    assert call(B=64) == binding.WC_EINVAL                 # below 128
    assert call(codes=None) == binding.WC_EINVAL           # codes without scales
    assert call(dt=3) == binding.WC_EINVAL
    assert call(out=MIS) == binding.WC_EALIGN
    assert call(ef=MIS) == binding.WC_EALIGN
    assert call(g=None) == binding.WC_EINVAL
    assert call(N=0, g=None, out=None) == binding.WC_OK


def test_fused_low_precision_error_buffer_argument_errors(lib):
    """The bf16 and int8 error-buffer forms of both fused entry points: the
    buffer (and the int8 scales) are required and 16-byte aligned.  Every
    call here fails its checks before any launch."""
    def caller(f, ok, names):
        def call(**kw):
            a = list(ok)
            for k, v in kw.items():
                a[names.index(k)] = v
            return f(*a)
        return call
    step16 = caller(lib.wc_qgz_step_fused_bf16ef,
                    (FAKE, FAKE, FAKE, FAKE, 8192, 8, 256, 1.0, 0.5, 1.0, FAKE, 0, None),
                    ["g", "ef", "codes", "scales", "N", "R", "B", "s", "beta", "os", "out", "dt",
                     "st"])
    step8 = caller(lib.wc_qgz_step_fused_int8ef,
                   (FAKE, FAKE, FAKE, FAKE, FAKE, 8192, 8, 256, 1.0, 0.5, 1.0, FAKE, 0, None),
                   ["g", "ef", "es", "codes", "scales", "N", "R", "B", "s", "beta", "os", "out",
                    "dt", "st"])
    hop16 = caller(lib.wc_qgz_first_hop_fused_bf16ef,
                   (FAKE, FAKE, FAKE, FAKE, 16 * 512, 8, 2, 256, 1.0, 0.5, FAKE, FAKE, None, None),
                   ["g", "ef", "codes", "scales", "N", "R", "G", "B", "s", "beta", "oc", "os",
                    "ef1", "st"])
    hop8 = caller(lib.wc_qgz_first_hop_fused_int8ef,
                  (FAKE, FAKE, FAKE, FAKE, FAKE, 16 * 512, 8, 2, 256, 1.0, 0.5, FAKE, FAKE, None,
                   None),
                  ["g", "ef", "es", "codes", "scales", "N", "R", "G", "B", "s", "beta", "oc",
                   "os", "ef1", "st"])
    for call in (step16, step8, hop16, hop8):
        assert call(ef=None) == binding.WC_EINVAL          # the buffer is required
        assert call(ef=MIS) == binding.WC_EALIGN
        assert call(B=64) == binding.WC_EINVAL
        assert call(codes=None) == binding.WC_EINVAL       # codes without scales
        assert call(g=None) == binding.WC_EINVAL
    for call in (step8, hop8):
        assert call(es=None) == binding.WC_EINVAL          # int8 needs its block scales
        assert call(es=MIS) == binding.WC_EALIGN
    for call in (step16, step8):
        assert call(dt=3) == binding.WC_EINVAL
        assert call(N=0, g=None, ef=None, out=None) == binding.WC_OK
    for call in (hop16, hop8):
        assert call(ef1=MIS) == binding.WC_EALIGN
        assert call(N=0, g=None, ef=None, oc=None, os=None) == binding.WC_OK


def test_fused_first_hop_argument_errors(lib):
    f = lib.wc_qgz_first_hop_fused
    ok = (FAKE, FAKE, FAKE, FAKE, 16 * 512, 8, 2, 256, 1.0, 0.5, FAKE, FAKE, None, None)
    names = ["g", "ef", "codes", "scales", "N", "R", "G", "B", "s", "beta", "oc", "os", "ef1",
             "st"]
    def call(**kw):
        a = list(ok)
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)
    assert call(B=64) == binding.WC_EINVAL                 # below 128
    assert call(G=3) == binding.WC_EINVAL                  # G must divide R
    assert call(scales=None) == binding.WC_EINVAL          # scales without codes
    assert call(oc=None) == binding.WC_EINVAL
    assert call(os=MIS) == binding.WC_EALIGN
    assert call(ef=MIS) == binding.WC_EALIGN
    assert call(codes=MIS) == binding.WC_EALIGN
    assert call(ef1=MIS) == binding.WC_EALIGN
    assert call(g=None) == binding.WC_EINVAL
    assert call(N=1 << 31, R=2, G=2, B=512) == binding.WC_ERANGE  # G*N reaches 2^32
    assert call(N=0, g=None, oc=None, os=None) == binding.WC_OK


def test_bf16ef_and_replica_argument_errors(lib):
    f = lib.wc_ef_quant_int4_bf16ef
    assert f(FAKE, None, FAKE, FAKE, 1024, 4, 1, 256, 1.0, 0.5, None) == binding.WC_EINVAL
    assert f(FAKE, MIS, FAKE, FAKE, 1024, 4, 1, 256, 1.0, 0.5, None) == binding.WC_EALIGN
    assert f(FAKE, FAKE, FAKE, FAKE, 1024, 4, 1, 100, 1.0, 0.5, None) == binding.WC_EINVAL
    assert f(None, None, None, None, 0, 4, 1, 256, 1.0, 0.5, None) == binding.WC_OK
    h = lib.wc_dequant_reduce_requant_ef
    assert h(FAKE, FAKE, 8192, 8, 2, 256, FAKE, FAKE, None, 1.0, 0.5, None) == binding.WC_EINVAL
    assert h(FAKE, FAKE, 8192, 8, 2, 256, FAKE, FAKE, MIS, 1.0, 0.5, None) == binding.WC_EALIGN
    assert h(FAKE, FAKE, 8192, 8, 3, 256, FAKE, FAKE, FAKE, 1.0, 0.5, None) == binding.WC_EINVAL
    q = lib.wc_qwz_quant_replica_int8
    assert q(FAKE, FAKE, FAKE, None, 4096, 2048, None) == binding.WC_EINVAL
    assert q(FAKE, FAKE, FAKE, MIS, 4096, 2048, None) == binding.WC_EALIGN
    assert q(FAKE, FAKE, FAKE, FAKE, 4000, 2048, None) == binding.WC_EINVAL


def test_checked_violations_needs_a_checked_build(lib):
    """The ordinary library has no bounds checks: the debugging call says so
    (and rejects unknown flags) without touching the GPU."""
    assert lib.wc_checked_violations(0) == binding.WC_EINVAL
    assert b"without checks" in lib.wc_last_error()
    assert lib.wc_checked_violations(4) == binding.WC_EINVAL
    assert b"unknown flags" in lib.wc_last_error()


def test_checked_build_exports_the_same_symbols():
    """The bounds-checked library (WC_CHECKED=1) builds from the same sources
    and exports every declared entry point."""
    lib_path = build.build(checked=True)
    raw = ctypes.CDLL(str(lib_path))
    for n in _declared():
        assert hasattr(raw, n), n
