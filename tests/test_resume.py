"""Checkpoint and resume: the error buffers (with the int8 buffer's scales)
are the only state a qgZ step carries from one step to the next (LoCo's
extra memory, "Merge LoCo with Zero++", Overview).  Saving them after step k,
loading them into a fresh reducer and continuing must reproduce an
uninterrupted run bit for bit."""
import pytest
import torch

from gpu_util import dev
from weight_communication_gb300 import workloads as wl
from weight_communication_gb300.qgz import QgzReducer

pytestmark = pytest.mark.gpu


def _reducer(w, dev, ef_dtype):
    return QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta,
                      out_dtype=torch.bfloat16 if w.out_bf16 else torch.float32, device=dev,
                      ef_dtype=ef_dtype, hop1_ef=w.G > 1)


@pytest.mark.parametrize("name,ef_dtype", [("single_hop", torch.float32),
                                           ("single_hop", torch.bfloat16),
                                           ("single_hop", torch.int8),
                                           ("hierarchical", torch.float32)])
def test_resume_from_saved_error_buffers(dev, tmp_path, name, ef_dtype):
    w = (wl.QGZ_SINGLE_HOP.scaled(8 * 256 * 32) if name == "single_hop"
         else wl.QGZ_HIERARCHICAL.scaled(16 * 512 * 4))
    steps, k = 6, 3
    grads = [wl.qgz_gradients(w, t, device=dev) for t in range(steps)]

    whole = _reducer(w, dev, ef_dtype)
    ref = [whole.step(g).clone() for g in grads]

    first = _reducer(w, dev, ef_dtype)
    for g in grads[:k]:
        first.step(g)
    ckpt = tmp_path / "qgz_state.pt"
    torch.save({"ef": first.ef.cpu(),
                "ef_scales": None if first.ef_scales is None else first.ef_scales.cpu(),
                "ef1": None if first.ef1 is None else first.ef1.cpu()}, ckpt)
    del first

    state = torch.load(ckpt)
    resumed = _reducer(w, dev, ef_dtype)
    resumed.ef.copy_(state["ef"])
    if state["ef_scales"] is not None:
        resumed.ef_scales.copy_(state["ef_scales"])
    if state["ef1"] is not None:
        resumed.ef1.copy_(state["ef1"])
    for t in range(k, steps):
        out = resumed.step(grads[t])
        assert torch.equal(out.view(torch.int16 if w.out_bf16 else torch.int32),
                           ref[t].view(torch.int16 if w.out_bf16 else torch.int32)), t
    bits = {torch.float32: torch.int32, torch.bfloat16: torch.int16, torch.int8: torch.int8}[ef_dtype]
    assert torch.equal(resumed.ef.view(bits), whole.ef.view(bits))
    if whole.ef_scales is not None:
        assert torch.equal(resumed.ef_scales.view(torch.int32), whole.ef_scales.view(torch.int32))
    if whole.ef1 is not None:
        assert torch.equal(resumed.ef1.view(torch.int32), whole.ef1.view(torch.int32))
