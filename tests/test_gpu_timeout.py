"""The failure path of the cooperative layer kernels: a bounded device wait
that runs out is reported, the layer's output is left unwritten, and the next
call on the same workspace computes the layer again.

The fault is injected without faulting the GPU: qmoe_set_fault_injection
shortens every bounded wait to a few milliseconds and makes one CTA skip its
grid-barrier arrivals, so the other CTAs' waits expire and every CTA returns.
The model is the CudaError of "ferrox-cuda 0.14.0 — src/gpu.rs": report the
failure, never compute something else.
"""
import numpy as np
import pytest

from moe_ffn_gb300 import synth
from tests.parity import check_moe

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 5], ids=["fused_1tok", "batched_5tok"])
def test_grid_barrier_timeout_reported_then_recovers(qm, orc, T):
    import torch
    shp = dict(synth.MOE_DECODE, n_tokens=T)
    K = shp["top_k"]
    inp = synth.moe_inputs(23 + T, **shp)
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], K, T, shp["gate"],
                     shp["up"], shp["down"])
    dev = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
           for k in ("router", "gate", "up", "down", "x")}
    ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device="cuda")

    def call():
        res = torch.from_numpy(inp["residual"].copy()).cuda()
        idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, K), device="cuda")
        qm.moe_ffn(dev["router"], dev["gate"], dev["up"], dev["down"], s, dev["x"], res, idx, w,
                   ws)
        torch.cuda.synchronize()
        return res.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()

    assert qm.device_status() == qm.OK
    qm.set_fault_injection(5_000_000, 3)  # 5 ms waits; CTA 3 never arrives
    try:
        out, idx, _ = call()
        assert qm.device_status() == qm.ERR_TIMEOUT
        assert "grid barrier" in qm.last_error()
    finally:
        qm.set_fault_injection(0, -1)
    # nothing of the layer was written: the residual and the routes are as given
    assert np.array_equal(out, inp["residual"].reshape(out.shape))
    assert np.all(idx == -1)
    # the same workspace serves the next call, which computes the layer
    out, idx, w = call()
    assert qm.device_status() == qm.OK
    ref = orc.moe_ffn(shp["hidden"], shp["expert_dim"], shp["num_experts"], K, shp["gate"],
                      shp["up"], shp["down"], inp["router"], inp["gate"], inp["up"], inp["down"],
                      inp["x"], inp["residual"])
    assert check_moe(out, idx, w, ref) == 0


def test_fault_injection_refuses_bad_cta(qm):
    with pytest.raises(qm.QmoeError) as ei:
        qm.set_fault_injection(0, -2)
    assert ei.value.status == qm.ERR_INVALID_ARGUMENT
