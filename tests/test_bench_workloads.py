"""The default bench line's summary of the other configurations
(`workloads`): every entry carries per-kernel times, algorithmic bytes and
fractions, and a parity verdict from a sample through the CUDA path against
the oracle.  Run here on small
stand-ins of the workloads (same R, G, B and parameters, fewer elements)."""
import argparse
import dataclasses

import pytest

pytestmark = pytest.mark.gpu


def test_other_workloads_summary(monkeypatch):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    from weight_communication_gb300 import binding, workloads as wl
    binding.load()
    monkeypatch.setattr(wl, "QGZ_HIERARCHICAL", wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 128))
    monkeypatch.setattr(wl, "QGZ_SINGLE_HOP", wl.QGZ_SINGLE_HOP.scaled(8 * 256 * 256))
    monkeypatch.setattr(wl, "QWZ_WEIGHTS", dataclasses.replace(wl.QWZ_WEIGHTS, n=2048 * 1024))
    monkeypatch.setattr(wl, "SR_ACCUMULATE", dataclasses.replace(wl.SR_ACCUMULATE, n=(1 << 22) + 24))
    args = argparse.Namespace(steps=4, warmup=3, batches=2, clocks=False, no_e2e=True,
                              no_overlap=True, no_cpu_baseline=False)
    dev = torch.device("cuda", 0)
    out = bench.other_workloads(args, dev, None, 1, 0)
    assert set(out) == {"qgz_hierarchical", "qgz_hier_ef", "qgz_hier_fused", "qgz_hier_ef_fused",
                        "qgz_bf16ef", "qgz_int8ef", "qgz_fused", "qgz_bf16ef_fused",
                        "qgz_int8ef_fused", "qwz", "sr"}
    want_kernels = {
        "qgz_hierarchical": {"ef_quant_int4", "dequant_reduce_requant", "dequant_reduce"},
        "qgz_hier_ef": {"ef_quant_int4", "dequant_reduce_requant", "dequant_reduce"},
        "qgz_hier_fused": {"qgz_first_hop_fused", "dequant_reduce"},
        "qgz_hier_ef_fused": {"qgz_first_hop_fused", "dequant_reduce"},
        "qgz_bf16ef": {"ef_quant_int4", "dequant_reduce"},
        "qgz_int8ef": {"ef_quant_int4", "dequant_reduce"},
        "qgz_fused": {"qgz_step_fused"},
        "qgz_bf16ef_fused": {"qgz_step_fused"},
        "qgz_int8ef_fused": {"qgz_step_fused"},
        "qwz": {"qwz_quant_int8", "qwz_dequant_int8", "qwz_quant_replica_int8"},
        "sr": {"sr_accumulate"},
    }
    for name, e in out.items():
        assert e["steps"] == 4 and e["ms_per_step"] > 0, name
        assert set(e["kernels"]) == want_kernels[name], name
        for k in e["kernels"].values():
            assert k["ms"] > 0 and k["algorithmic_bytes"] > 0 and k["frac"] > 0
            assert set(k["ms_percentiles"]) == {"median", "p10", "p90"}
    for name, e in out.items():
        assert e["parity"]["verdict"] == "bit-exact", (name, e["parity"])
