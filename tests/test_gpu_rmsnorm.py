"""GPU parity of the entry points with ffn_norm in front (ffn_swiglu_rmsnorm,
moe_ffn_rmsnorm) against the oracle composed the same way: the oracle's
RMSNorm of the residual, rounded to f32, as the input of the oracle FFN/MoE.
Covers the fused per-layer kernel (decode, dense FFN), several tokens, and the
tensor-core path for many tokens."""
import numpy as np
import pytest

from moe_ffn_gb300 import synth
from tests.parity import check_close, check_moe
from tests.test_gpu_parity import _dev

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _normed(orc, residual, w):
    return orc.rmsnorm(residual, w, EPS).astype(np.float32)


@pytest.mark.parametrize("H,F,gq,dq", [(256, 512, synth.Q4_K, synth.Q6_K),
                                       (768, 256, synth.Q5_K, synth.Q8_0),
                                       (4096, 14336, synth.Q4_K, synth.Q6_K)])
def test_ffn_swiglu_rmsnorm(qm, orc, H, F, gq, dq):
    import torch
    inp = synth.ffn_inputs(3 * H + F, hidden=H, inter=F, gate=gq, up=gq, down=dq)
    nw = synth.norm_weight(synth.rng(11), H)
    res = _dev(inp["residual"])
    ws = torch.empty(qm.ffn_swiglu_rmsnorm_workspace_size(H, F), dtype=torch.uint8,
                     device="cuda")
    qm.ffn_swiglu_rmsnorm(_dev(inp["gate"]), _dev(inp["up"]), _dev(inp["down"]), gq, gq, dq, H,
                          F, _dev(nw), EPS, res, ws)
    torch.cuda.synchronize()
    assert qm.device_status() == qm.OK
    xn = _normed(orc, inp["residual"], nw)
    ref, tol = orc.ffn_swiglu(gq, gq, dq, H, F, inp["gate"], inp["up"], inp["down"], xn,
                              inp["residual"])
    check_close(res.cpu().numpy(), ref, tol, f"ffn_rmsnorm {H}x{F}")


MOE_NORM = [
    dict(hidden=2048, expert_dim=768, num_experts=128, top_k=8, n_tokens=1),   # decode shape
    dict(hidden=512, expert_dim=512, num_experts=16, top_k=4, n_tokens=3),     # a few tokens
    dict(hidden=2048, expert_dim=768, num_experts=128, top_k=8, n_tokens=16),  # batched decode
    dict(hidden=256, expert_dim=256, num_experts=8, top_k=2, n_tokens=64),     # tensor cores
]


@pytest.mark.parametrize("shp", MOE_NORM, ids=lambda s: "H{hidden}E{num_experts}T{n_tokens}".format(**s))
def test_moe_ffn_rmsnorm(qm, orc, shp):
    import torch
    shp = dict(shp, gate=synth.Q4_K, up=synth.Q4_K, down=synth.Q6_K)
    inp = synth.moe_inputs(17 + shp["n_tokens"], **shp)
    nw = synth.norm_weight(synth.rng(12), shp["hidden"])
    T, K = shp["n_tokens"], shp["top_k"]
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], K, T, shp["gate"],
                     shp["up"], shp["down"])
    res = _dev(inp["residual"])
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), device="cuda")
    ws = torch.empty(qm.moe_ffn_rmsnorm_workspace_size(s), dtype=torch.uint8, device="cuda")
    qm.moe_ffn_rmsnorm(_dev(inp["router"]), _dev(inp["gate"]), _dev(inp["up"]), _dev(inp["down"]),
                       s, _dev(nw), EPS, res, idx, w, ws)
    torch.cuda.synchronize()
    assert qm.device_status() == qm.OK
    xn = _normed(orc, inp["residual"], nw)
    ref = orc.moe_ffn(shp["hidden"], shp["expert_dim"], shp["num_experts"], K, shp["gate"],
                      shp["up"], shp["down"], inp["router"], inp["gate"], inp["up"], inp["down"],
                      xn, inp["residual"])
    assert check_moe(res.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), ref) <= max(1, T // 20)


def test_rmsnorm_layer_equals_norm_then_layer(qm, orc):
    """The fused norm and the plain entry point fed the same normed input
    agree to within the GEMV tolerance (same routing, same experts)."""
    import torch
    shp = dict(hidden=1024, expert_dim=512, num_experts=32, top_k=4, n_tokens=1,
               gate=synth.Q8_0, up=synth.Q8_0, down=synth.Q5_K)
    inp = synth.moe_inputs(5, **shp)
    nw = synth.norm_weight(synth.rng(13), shp["hidden"])
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], 4, 1, shp["gate"],
                     shp["up"], shp["down"])
    dev = {k: _dev(inp[k]) for k in ("router", "gate", "up", "down")}
    r1 = _dev(inp["residual"])
    ws = torch.zeros(qm.moe_ffn_rmsnorm_workspace_size(s), dtype=torch.uint8, device="cuda")
    qm.moe_ffn_rmsnorm(dev["router"], dev["gate"], dev["up"], dev["down"], s, _dev(nw), EPS, r1,
                       None, None, ws)
    xn = _normed(orc, inp["residual"], nw)
    r2 = _dev(inp["residual"])
    qm.moe_ffn(dev["router"], dev["gate"], dev["up"], dev["down"], s, _dev(xn), r2, None, None,
               ws)
    torch.cuda.synchronize()
    ref = orc.moe_ffn(shp["hidden"], shp["expert_dim"], shp["num_experts"], 4, shp["gate"],
                      shp["up"], shp["down"], inp["router"], inp["gate"], inp["up"], inp["down"],
                      xn, inp["residual"])
    check_close(r1.cpu().numpy(), r2.cpu().numpy().astype(np.float64), 2 * ref["tol"],
                "fused norm vs norm then layer")
