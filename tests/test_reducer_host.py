"""Host-side checks of QgzReducer's options (no GPU): the fused step's
preconditions and the launch count it reports, and the binding's choice of
fused entry point by the error buffer's dtype."""
import pytest
import torch

from weight_communication_gb300.qgz import DevicePipeline, QgzReducer


def test_fused_step_preconditions():
    kw = dict(N=8 * 256, R=8, G=1, B=256, device="cpu")
    for ef_dtype in (torch.bfloat16, torch.int8):
        assert QgzReducer(**kw, ef_dtype=ef_dtype, fused=True).launches_per_step == 1
    with pytest.raises(ValueError, match="B >= 128"):
        QgzReducer(N=8 * 64, R=8, G=1, B=64, device="cpu", fused=True)
    red = QgzReducer(N=16 * 512, R=16, G=2, B=512, device="cpu", hop1_ef=True, fused=True)
    assert red.ef1 is not None and red.launches_per_step == 2
    assert QgzReducer(**kw, fused=True).launches_per_step == 1
    assert QgzReducer(**kw, use_ef=False, fused=True).launches_per_step == 1
    assert QgzReducer(N=16 * 512, R=16, G=2, B=512, device="cpu", fused=True).launches_per_step == 2
    assert QgzReducer(**kw).launches_per_step == 2
    assert QgzReducer(N=16 * 512, R=16, G=2, B=512, device="cpu").launches_per_step == 3


def test_device_pipeline_refuses_a_fused_reducer():
    red = QgzReducer(N=8 * 256, R=8, G=1, B=256, device="cpu", fused=True)
    with pytest.raises(ValueError, match="no separate reduce"):
        DevicePipeline(red)


def test_fused_binding_picks_the_entry_point_by_error_dtype():
    from weight_communication_gb300 import binding
    assert binding._fused_error(None, None, 1024, 256, None)[0] == ""
    with pytest.raises(ValueError, match="needs ef_scales"):
        binding._fused_error(torch.zeros(1024, dtype=torch.int8), None, 1024, 256, None)
    with pytest.raises(ValueError, match="int8 error buffer only"):
        binding._fused_error(None, torch.zeros(4), 1024, 256, None)
    with pytest.raises(TypeError, match="float32, bfloat16 or int8"):
        binding._fused_error(torch.zeros(1024, dtype=torch.float16), None, 1024, 256, None)
