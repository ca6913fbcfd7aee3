"""The allocation-free MoE entry point (moe_ffn_noalloc) against moe_ffn.

moe_ffn_noalloc serves callers that cannot allocate device memory (a host
framework that owns all device memory, a serving loop that forbids
allocation once running): it takes no workspace and uses the library's
built-in scratch array instead.  This test calls it through the C ABI twice
in a row and checks each result against moe_ffn with a caller workspace on
the same inputs, within the tolerance the parity tests use.  It lives in a
file of its own, collected last.
"""
import numpy as np
import pytest

from moe_ffn_gb300 import synth
from tests.parity import check_close

pytestmark = pytest.mark.gpu


def _run(qm, inp, shp, noalloc):
    import torch
    T, K = shp["n_tokens"], shp["top_k"]
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], K, T, shp["gate"],
                     shp["up"], shp["down"])
    dev = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
           for k in ("router", "gate", "up", "down", "x")}
    res = torch.from_numpy(inp["residual"].copy()).cuda()
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), device="cuda")
    if noalloc:
        qm.moe_ffn_noalloc(dev["router"], dev["gate"], dev["up"], dev["down"], s, dev["x"], res,
                           idx, w)
    else:
        ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device="cuda")
        qm.moe_ffn(dev["router"], dev["gate"], dev["up"], dev["down"], s, dev["x"], res, idx, w,
                   ws)
    torch.cuda.synchronize()
    return res.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("shp", [
    dict(synth.MOE_DECODE),                                                 # one decode token
    dict(hidden=512, expert_dim=256, num_experts=16, top_k=4, n_tokens=3,
         gate=synth.Q4_K, up=synth.Q4_K, down=synth.Q6_K),                  # a few tokens
    dict(synth.MOE_DECODE, n_tokens=35),  # the stated limit: the tensor-core path's buffers
], ids=["decode_1tok", "decode_3tok", "decode_35tok"])
def test_noalloc_matches_workspace_entry_point(qm, orc, shp):
    inp = synth.moe_inputs(5, **shp)
    ref_out, ref_idx, ref_w = _run(qm, inp, shp, noalloc=False)
    oracle = orc.moe_ffn(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"],
                         shp["gate"], shp["up"], shp["down"], inp["router"], inp["gate"],
                         inp["up"], inp["down"], inp["x"], inp["residual"])
    for call in range(2):  # two calls in a row share the built-in scratch
        out, idx, w = _run(qm, inp, shp, noalloc=True)
        # the tensor-core path (32 tokens and more) adds the k experts' down
        # products with atomics: their order, not the routing, may differ
        assert np.array_equal(idx, ref_idx), call
        check_close(w, ref_w, 1e-6 * np.abs(ref_w) + 1e-7, f"noalloc weights, call {call}")
        check_close(out, ref_out, oracle["tol"], f"noalloc residual, call {call}")
    assert qm.device_status() == qm.OK


def test_noalloc_refuses_shapes_beyond_its_scratch(qm):
    import torch
    shp = dict(synth.MOE_DECODE, n_tokens=64)  # needs about 1.9 MB of scratch
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"], 64,
                     shp["gate"], shp["up"], shp["down"])
    assert qm.moe_ffn_workspace_size(s) > qm.NOALLOC_SCRATCH_BYTES
    z = torch.zeros(16, device="cuda")
    with pytest.raises(qm.QmoeError) as ei:
        qm.moe_ffn_noalloc(z, z, z, z, s, z, z)
    assert ei.value.status == qm.ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)
