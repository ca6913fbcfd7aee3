"""Pins of the oracle's dense SwiGLU FFN and MoE FFN (op order of moe_layer on
"aprender-serve 0.70.2 — forward_qwen3_moe_resident.rs"; SwiGLU of
SILU_MUL_KERNEL_SRC on "ferrox-cuda 0.14.0 — src/gpu.rs").

Pins: a brute-force composition from library primitives on tiny shapes
(numpy matmul on decoded matrices — the decoders are pinned in
test_oracle_pins — scipy softmax, numpy stable argsort), invariants (one
expert of weight 1 is the dense FFN; permuting experts changes nothing; a
zero down projection leaves the residual), and the routing-fault analogue:
the parity checker must reject a forward that routed a token wrongly.
"""
import numpy as np
import pytest
from scipy.special import expit, softmax

from moe_ffn_gb300 import synth
from tests import blocks as B
from tests.parity import ParityError, check_moe

SMALL = dict(hidden=256, expert_dim=256, num_experts=6, top_k=2, n_tokens=3,
             gate=synth.Q4_K, up=synth.Q4_K, down=synth.Q6_K)


def _run(orc, shp, inp, **kw):
    return orc.moe_ffn(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"],
                       shp["gate"], shp["up"], shp["down"], inp["router"], inp["gate"],
                       inp["up"], inp["down"], inp["x"], inp["residual"], **kw)


def test_moe_brute_force_numpy(orc):
    shp = SMALL
    inp = synth.moe_inputs(11, **shp)
    H, F, E, K = shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"]
    G = [orc.dequant(shp["gate"], inp["gate"][e], F, H).astype(np.float64) for e in range(E)]
    U = [orc.dequant(shp["up"], inp["up"][e], F, H).astype(np.float64) for e in range(E)]
    D = [orc.dequant(shp["down"], inp["down"][e], H, F).astype(np.float64) for e in range(E)]
    ref = _run(orc, shp, inp)
    for t in range(shp["n_tokens"]):
        x = inp["x"][t].astype(np.float64)
        p = softmax(inp["router"].astype(np.float64) @ x)
        sel = np.argsort(-p, kind="stable")[:K]
        w = p[sel] / p[sel].sum()
        out = inp["residual"][t].astype(np.float64).copy()
        for s, e in enumerate(sel):
            g, u = G[e] @ x, U[e] @ x
            out += D[e] @ (w[s] * (g * expit(g) * u))
        assert list(ref["idx"][t]) == list(sel)
        assert np.allclose(ref["w"][t], w, rtol=1e-12)
        assert np.allclose(ref["out"][t], out, rtol=1e-10, atol=1e-9)


def test_moe_without_renormalisation_brute_force(orc):
    """renormalize=False: the same composition with w = the selected softmax
    probabilities (no division by their sum)."""
    shp = dict(SMALL, top_k=3)
    inp = synth.moe_inputs(13, **shp)
    H, F, E, K = shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"]
    G = [orc.dequant(shp["gate"], inp["gate"][e], F, H).astype(np.float64) for e in range(E)]
    U = [orc.dequant(shp["up"], inp["up"][e], F, H).astype(np.float64) for e in range(E)]
    D = [orc.dequant(shp["down"], inp["down"][e], H, F).astype(np.float64) for e in range(E)]
    ref = _run(orc, shp, inp, renormalize=False)
    for t in range(shp["n_tokens"]):
        x = inp["x"][t].astype(np.float64)
        p = softmax(inp["router"].astype(np.float64) @ x)
        sel = np.argsort(-p, kind="stable")[:K]
        out = inp["residual"][t].astype(np.float64).copy()
        for e in sel:
            g, u = G[e] @ x, U[e] @ x
            out += D[e] @ (p[e] * (g * expit(g) * u))
        assert list(ref["idx"][t]) == list(sel)
        assert np.allclose(ref["w"][t], p[sel], rtol=1e-12)
        assert ref["w"][t].sum() < 1.0
        assert np.allclose(ref["out"][t], out, rtol=1e-10, atol=1e-9)


def test_one_expert_is_dense_ffn(orc):
    shp = dict(SMALL, num_experts=1, top_k=1, n_tokens=1)
    inp = synth.moe_inputs(12, **shp)
    ref = _run(orc, shp, inp)
    out, tol = orc.ffn_swiglu(shp["gate"], shp["up"], shp["down"], shp["hidden"],
                              shp["expert_dim"], inp["gate"][0], inp["up"][0], inp["down"][0],
                              inp["x"][0], inp["residual"][0])
    assert ref["w"][0, 0] == 1.0
    assert np.array_equal(ref["out"][0], out)
    assert np.allclose(ref["tol"][0], tol, rtol=1e-12)


def test_expert_permutation_invariance(orc):
    shp = SMALL
    inp = synth.moe_inputs(13, **shp)
    perm = np.array([3, 0, 5, 1, 4, 2])
    inp2 = dict(inp, router=inp["router"][perm], gate=inp["gate"][perm], up=inp["up"][perm],
                down=inp["down"][perm])
    a, b = _run(orc, shp, inp), _run(orc, shp, inp2)
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(perm[b["idx"]], a["idx"])


def test_zero_down_leaves_residual(orc):
    shp = SMALL
    inp = synth.moe_inputs(14, **shp)
    down = inp["down"].copy().reshape(-1, 210)
    down[:, 208:210] = 0  # Q6_K d = +0: every weight is 0
    inp["down"] = down.reshape(inp["down"].shape)
    ref = _run(orc, shp, inp)
    assert np.array_equal(ref["out"], inp["residual"].astype(np.float64))


def test_ffn_zero_x_leaves_residual(orc):
    inp = synth.ffn_inputs(15, hidden=256, inter=512, gate=synth.Q4_K, up=synth.Q4_K,
                           down=synth.Q6_K)
    out, _ = orc.ffn_swiglu(synth.Q4_K, synth.Q4_K, synth.Q6_K, 256, 512, inp["gate"],
                            inp["up"], inp["down"], np.zeros(256, np.float32), inp["residual"])
    assert np.array_equal(out, inp["residual"].astype(np.float64))


def test_tolerance_covers_perturbed_gemv_outputs(orc):
    """The propagated tolerance bounds the change of the output when every
    gate/up GEMV output moves by its own allowed error (checked by brute
    force on a tiny FFN: g -> g + dg, u -> u + du with worst-case signs)."""
    H, F = 256, 256
    inp = synth.ffn_inputs(16, hidden=H, inter=F, gate=synth.Q4_K, up=synth.Q4_K,
                           down=synth.Q6_K)
    out, tol = orc.ffn_swiglu(synth.Q4_K, synth.Q4_K, synth.Q6_K, H, F, inp["gate"], inp["up"],
                              inp["down"], inp["x"], inp["residual"])
    Gm = orc.dequant(synth.Q4_K, inp["gate"], F, H).astype(np.float64)
    Um = orc.dequant(synth.Q4_K, inp["up"], F, H).astype(np.float64)
    Dm = orc.dequant(synth.Q6_K, inp["down"], H, F).astype(np.float64)
    x = inp["x"].astype(np.float64)
    g, u = Gm @ x, Um @ x
    dg = 1e-3 * (np.abs(Gm) @ np.abs(x)) + 1e-6
    du = 1e-3 * (np.abs(Um) @ np.abs(x)) + 1e-6
    rng = np.random.default_rng(0)
    for _ in range(20):
        sg, su = rng.choice([-1.0, 1.0], F), rng.choice([-1.0, 1.0], F)
        g2, u2 = g + sg * dg, u + su * du
        a2 = g2 * expit(g2) * u2
        moved = inp["residual"].astype(np.float64) + Dm @ a2
        assert np.all(np.abs(moved - out) <= tol)


def test_checker_rejects_wrong_route(orc):
    """Routing-fault analogue: a forward in which one token took a different
    expert (planted in the oracle's inputs) fails the parity check."""
    shp = dict(SMALL, n_tokens=2)
    inp = synth.moe_inputs(17, **shp)
    ref = _run(orc, shp, inp)
    t = 0
    chosen = ref["idx"][t]
    other = next(e for e in range(shp["num_experts"]) if e not in chosen)
    # swap the router rows of the rank-0 expert and an unselected one
    r2 = inp["router"].copy()
    r2[[chosen[0], other]] = r2[[other, chosen[0]]]
    bad = _run(orc, shp, dict(inp, router=r2))
    assert not np.array_equal(bad["idx"][t], ref["idx"][t])
    with pytest.raises(ParityError):
        check_moe(bad["out"], bad["idx"], bad["w"], ref)
    # the same route with a wrong residual also fails
    out = ref["out"].copy()
    out[1, 5] += 10 * ref["tol"][1, 5]
    with pytest.raises(ParityError):
        check_moe(out, ref["idx"], ref["w"], ref)
    # and the oracle's own result passes
    assert check_moe(ref["out"], ref["idx"], ref["w"], ref) == 0


def test_moe_rejects_bad_shape(orc):
    shp = dict(SMALL, top_k=7)
    inp = synth.moe_inputs(18, **dict(SMALL))
    with pytest.raises(ValueError):
        _run(orc, shp, inp)
