"""GPU parity of the batched decode MoE path: 2..31 tokens per moe_ffn call,
where each routed expert's weights are read once for all the tokens routed
to it (one cooperative launch per group of up to 16 tokens).  Every token of
every case is checked against the oracle: routing exactly (wherever the
logits are unambiguous), weights and residuals within the composite bound."""
import numpy as np
import pytest

from moe_ffn_gb300 import synth
from tests.parity import check_moe
from tests.test_gpu_parity import QNAME, _dev, gpu_moe, oracle_moe

pytestmark = pytest.mark.gpu

BATCH_SHAPES = [
    # the decode layer at several batch sizes (one, two and three launches)
    dict(synth.MOE_DECODE, n_tokens=2),
    dict(synth.MOE_DECODE, n_tokens=13),
    dict(synth.MOE_DECODE, n_tokens=16),
    dict(synth.MOE_DECODE, n_tokens=31),
    # every token routed to every expert: each expert has all T pairs
    dict(hidden=512, expert_dim=256, num_experts=8, top_k=8, n_tokens=16),
    # one expert, top-1: a single expert with every token
    dict(hidden=256, expert_dim=512, num_experts=1, top_k=1, n_tokens=7),
    # wide k and many experts; F > H
    dict(hidden=256, expert_dim=1024, num_experts=256, top_k=16, n_tokens=5),
    dict(hidden=1024, expert_dim=256, num_experts=40, top_k=3, n_tokens=9),
]


def _id(s):
    return "H{hidden}F{expert_dim}E{num_experts}k{top_k}T{n_tokens}".format(**s)


@pytest.mark.parametrize("shp", BATCH_SHAPES, ids=_id)
def test_batch_moe_all_tokens(qm, orc, shp):
    shp = dict(dict(gate=synth.Q4_K, up=synth.Q4_K, down=synth.Q6_K), **shp)
    inp = synth.moe_inputs(500 + shp["n_tokens"] + shp["num_experts"], **shp)
    out, idx, w = gpu_moe(qm, inp, shp)
    ref = oracle_moe(orc, inp, shp)
    assert check_moe(out, idx, w, ref) <= 1
    assert qm.device_status() == qm.OK


FMT_PAIRS = [(g, d) for g in (synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q5_K, synth.Q6_K)
             for d in (synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q5_K, synth.Q6_K)]


@pytest.mark.parametrize("fmts", FMT_PAIRS, ids=lambda f: f"{QNAME[f[0]]}-{QNAME[f[1]]}")
def test_batch_moe_formats(qm, orc, fmts):
    """Every pair of gate/up and down formats through the batched kernel."""
    shp = dict(hidden=512, expert_dim=768, num_experts=12, top_k=4, n_tokens=6,
               gate=fmts[0], up=fmts[0], down=fmts[1])
    inp = synth.moe_inputs(600 + 7 * fmts[0] + fmts[1], **shp)
    out, idx, w = gpu_moe(qm, inp, shp)
    ref = oracle_moe(orc, inp, shp)
    assert check_moe(out, idx, w, ref) <= 1


def test_batch_matches_token_by_token(qm):
    """The batched call and the same tokens passed one call at a time route
    identically and agree to float rounding (the down products reach the
    residual in a different order)."""
    import torch
    shp = dict(synth.MOE_DECODE, n_tokens=8)
    inp = synth.moe_inputs(77, **shp)
    out_b, idx_b, w_b = gpu_moe(qm, inp, shp)
    one = dict(shp, n_tokens=1)
    s = qm.moe_shape(one["hidden"], one["expert_dim"], one["num_experts"], one["top_k"], 1,
                     one["gate"], one["up"], one["down"])
    ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device="cuda")
    R, G, U, D = (_dev(inp[k]) for k in ("router", "gate", "up", "down"))
    outs, idxs = [], []
    for t in range(shp["n_tokens"]):
        res = _dev(inp["residual"][t:t + 1])
        idx = torch.full((1, one["top_k"]), -1, dtype=torch.int32, device="cuda")
        qm.moe_ffn(R, G, U, D, s, _dev(inp["x"][t:t + 1]), res, idx, None, ws)
        outs.append(res.cpu().numpy()[0])
        idxs.append(idx.cpu().numpy()[0])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx_b, np.stack(idxs))
    np.testing.assert_allclose(out_b, np.stack(outs), rtol=0, atol=2e-5 * np.abs(out_b).max())
