"""GB300-native quantized gradient communication kernels.

ZeRO++ quantized gradient reduction (qgZ) with LoCo error feedback, qwZ int8
weight quantization and ZeRO-2 stochastic-rounding accumulation, as sm_103a
CUDA kernels behind the C ABI of include/wc.h.  `binding` is the Python face
of that ABI; `workloads` draws the seeded synthetic inputs; `qgz` composes the
calls into whole reduce steps.
"""
from . import workloads  # noqa: F401  (no CUDA needed to import)

__all__ = ["binding", "workloads", "qgz"]


def __getattr__(name):
    # The binding and the composed steps load libwc.so lazily, so importing
    # the package works on a machine without the library or a GPU.
    if name in ("binding", "qgz"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
