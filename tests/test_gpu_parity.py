"""GPU parity: the CUDA library (called through the C ABI) against the CPU
oracle on the same seeded inputs — element by element at sizes that span
several tiles and a ragged tail, and at the workloads' full sizes."""
import numpy as np
import pytest

from moe_ffn_gb300 import synth
from tests.parity import AMBIGUITY, check_close, check_gemv, check_moe, route_is_valid

pytestmark = pytest.mark.gpu

QTS = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q5_K, synth.Q6_K]
QNAME = {1: "Q8_0", 2: "Q4_0", 3: "Q4_K", 4: "Q5_K", 5: "Q6_K", 0: "F32"}


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_qmv(qm, qt, W, rows, cols, x):
    import torch
    Wd, xd = _dev(W), _dev(x)
    y = torch.full((rows,), float("nan"), device="cuda")
    qm.qmv(qt, Wd, rows, cols, xd, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("qt", QTS, ids=lambda q: QNAME[q])
@pytest.mark.parametrize("rows,cols", [(1, 256), (7, 256), (37, 768), (300, 1024),
                                       (153, 4096), (64, 14336), (9, 32768)])
def test_qmv_small(qm, orc, qt, rows, cols):
    g = synth.rng(1000 + qt * 7 + rows)
    W = synth.quant_matrix(g, qt, rows, cols, nan_row=rows // 2 if rows > 2 else None)
    x = synth.normal(g, cols)
    y = gpu_qmv(qm, qt, W, rows, cols, x)
    ref, sabs = orc.matvec(qt, W, rows, cols, x, with_sabs=True)
    check_gemv(y, ref, sabs, f"qmv {QNAME[qt]} {rows}x{cols}")


def test_qmv_f32(qm, orc):
    g = synth.rng(5)
    rows, cols = 129, 2048
    R = synth.normal(g, (rows, cols), 0.02)
    x = synth.normal(g, cols)
    y = gpu_qmv(qm, synth.F32, R, rows, cols, x)
    ref, sabs = orc.matvec(orc.F32, R.view(np.uint8), rows, cols, x, with_sabs=True)
    check_gemv(y, ref, sabs, "qmv F32")


def test_qmv_single_q4_0_workload(qm, orc):
    """256 x 1024 Q4_0, d ~ U(1e-3, 1e-2), uniform nibbles, x ~ N(0,1), seed 0."""
    w = synth.GEMV_SMALL
    g = synth.rng(0)
    W = synth.quant_matrix(g, w["qtype"], w["rows"], w["cols"])
    x = synth.normal(g, w["cols"])
    y = gpu_qmv(qm, w["qtype"], W, w["rows"], w["cols"], x)
    ref, sabs = orc.matvec(w["qtype"], W, w["rows"], w["cols"], x, with_sabs=True)
    check_gemv(y, ref, sabs, "Q4_0 256x1024")


@pytest.mark.parametrize("qt", QTS, ids=lambda q: QNAME[q])
def test_qmv_sweep_workload(qm, orc, qt):
    """4096 x 4096 per format, NaN f16 scale in block 0 of row 1."""
    w = synth.GEMV_SWEEP
    g = synth.rng(qt)
    W = synth.quant_matrix(g, qt, w["rows"], w["cols"], nan_row=w["nan_row"])
    x = synth.normal(g, w["cols"])
    y = gpu_qmv(qm, qt, W, w["rows"], w["cols"], x)
    ref, sabs = orc.matvec(qt, W, w["rows"], w["cols"], x, with_sabs=True)
    assert np.isnan(ref[1]) and np.isnan(y[1])
    check_gemv(y, ref, sabs, f"sweep {QNAME[qt]}")


@pytest.mark.parametrize("qt", QTS, ids=lambda q: QNAME[q])
def test_qmv_wide_range_x(qm, orc, qt):
    """Blocks whose activations span six decades (one value 1e3, the rest
    ~1e-3, random signs): the products take every bit of each f32 x, so the
    small values are not lost beside the large one."""
    g = synth.rng(900 + qt)
    rows, cols = 300, 2048
    W = synth.quant_matrix(g, qt, rows, cols)
    x = (synth.normal(g, cols) * 1e-3).astype(np.float32)
    x[g.integers(0, 32, cols // 32) + np.arange(0, cols, 32)] = 1e3 * np.sign(g.standard_normal(cols // 32))
    y = gpu_qmv(qm, qt, W, rows, cols, x)
    ref, sabs = orc.matvec(qt, W, rows, cols, x, with_sabs=True)
    assert check_gemv(y, ref, sabs, f"wide-range x {QNAME[qt]}") < 0.05


@pytest.mark.parametrize("qt", [synth.Q4_0, synth.Q8_0], ids=lambda q: QNAME[q])
def test_qmv_outlier_on_zero_weight_column(qm, orc, qt):
    """x[0] = 1e3 inside an N(0,1) block, on a column whose weight is zero in
    every row (Q4_0 nibble 8, Q8_0 quant 0); the other blocks ~1e-3.  The
    bound 1e-3 * sum |w x| then holds no term of the outlier, so an
    activation rounded relative to its block's largest value would miss it;
    with f32 activations every row meets it with a wide margin."""
    g = synth.rng(4242 + qt)
    rows, cols = 256, 2048
    W = synth.quant_matrix(g, qt, rows, cols)
    if qt == synth.Q4_0:
        W[:, 2] = (W[:, 2] & 0xF0) | 0x08  # block 0, element 0: low nibble of byte 2
    else:
        W[:, 2] = 0                        # block 0, element 0: int8 quant at byte 2
    x = (synth.normal(g, cols) * 1e-3).astype(np.float32)
    x[:32] = synth.normal(g, 32)
    x[0] = 1e3
    y = gpu_qmv(qm, qt, W, rows, cols, x)
    ref, sabs = orc.matvec(qt, W, rows, cols, x, with_sabs=True)
    assert np.all(orc.dequant(qt, W, rows, cols)[:, 0] == 0)
    assert check_gemv(y, ref, sabs, f"outlier on a zero column {QNAME[qt]}") < 0.05


@pytest.mark.parametrize("qt", QTS, ids=lambda q: QNAME[q])
def test_qmv_activation_range(qm, orc, qt):
    """Activations from 1e-30 to 1e30 in one vector (blocks of very different
    magnitude, and values 2^40 apart inside one block): each product keeps
    its full precision.  Values of 2^106 and more are outside the range and
    reported as UNSUPPORTED by the device status."""
    g = synth.rng(77 + qt)
    rows, cols = 64, 2048
    W = synth.quant_matrix(g, qt, rows, cols)
    x = synth.normal(g, cols)
    x *= (10.0 ** g.integers(-30, 31, cols // 32)).repeat(32).astype(np.float32)
    x[5::32] *= 2.0 ** -40
    y = gpu_qmv(qm, qt, W, rows, cols, x)
    assert qm.device_status() == qm.OK
    ref, sabs = orc.matvec(qt, W, rows, cols, x, with_sabs=True)
    assert check_gemv(y, ref, sabs, f"activation range {QNAME[qt]}") < 0.05
    x[100] = 2.0 ** 107
    gpu_qmv(qm, qt, W, rows, cols, x)
    assert qm.device_status() == qm.ERR_UNSUPPORTED
    assert "2^106" in qm.last_error()
    assert qm.device_status() == qm.OK


@pytest.mark.parametrize("qt", QTS, ids=lambda q: QNAME[q])
def test_qmv_nan_x_reaches_every_row(qm, orc, qt):
    """A NaN activation makes every output NaN (each row multiplies it), as in
    the oracle."""
    g = synth.rng(950 + qt)
    rows, cols = 64, 1024
    W = synth.quant_matrix(g, qt, rows, cols)
    x = synth.normal(g, cols)
    x[517] = np.nan
    y = gpu_qmv(qm, qt, W, rows, cols, x)
    ref = orc.matvec(qt, W, rows, cols, x)
    assert np.all(np.isnan(ref)) and np.all(np.isnan(y))


def test_qmv_repeatable_and_in_stream_order(qm, orc):
    """Back-to-back calls on one stream with a dependent x: y2 = W (y1[:cols])."""
    import torch
    g = synth.rng(77)
    rows = cols = 1024
    W = synth.quant_matrix(g, synth.Q4_K, rows, cols)
    x = synth.normal(g, cols)
    Wd, xd = _dev(W), _dev(x)
    y1 = torch.empty(rows, device="cuda")
    y2 = torch.empty(rows, device="cuda")
    for _ in range(3):
        qm.qmv(synth.Q4_K, Wd, rows, cols, xd, y1)
        qm.qmv(synth.Q4_K, Wd, rows, cols, y1, y2)
    torch.cuda.synchronize()
    r1, s1 = orc.matvec(synth.Q4_K, W, rows, cols, x, with_sabs=True)
    r2, s2 = orc.matvec(synth.Q4_K, W, rows, cols, y1.cpu().numpy(), with_sabs=True)
    check_gemv(y2.cpu().numpy(), r2, s2, "chained")
    check_gemv(y1.cpu().numpy(), r1, s1, "first of the chain")
    assert qm.device_status() == qm.OK


# ------------------------------------------------------------- dense FFN
def gpu_ffn(qm, inp, H, F, gq, uq, dq):
    import torch
    res = _dev(inp["residual"])
    ws = torch.empty(qm.ffn_swiglu_workspace_size(H, F), dtype=torch.uint8, device="cuda")
    qm.ffn_swiglu(_dev(inp["gate"]), _dev(inp["up"]), _dev(inp["down"]), gq, uq, dq, H, F,
                  _dev(inp["x"]), res, ws)
    torch.cuda.synchronize()
    return res.cpu().numpy()


@pytest.mark.parametrize("H,F,gq,dq", [(256, 512, synth.Q4_K, synth.Q6_K),
                                       (512, 768, synth.Q8_0, synth.Q4_0),
                                       (768, 256, synth.Q5_K, synth.Q8_0),
                                       (1024, 2048, synth.Q4_0, synth.Q5_K)])
def test_ffn_small(qm, orc, H, F, gq, dq):
    inp = synth.ffn_inputs(H + F, hidden=H, inter=F, gate=gq, up=gq, down=dq)
    got = gpu_ffn(qm, inp, H, F, gq, gq, dq)
    ref, tol = orc.ffn_swiglu(gq, gq, dq, H, F, inp["gate"], inp["up"], inp["down"], inp["x"],
                              inp["residual"])
    check_close(got, ref, tol, f"ffn {H}x{F}")


def test_ffn_dense_workload(qm, orc):
    """hidden 4096, intermediate 14336, gate/up Q4_K, down Q6_K."""
    w = synth.DENSE_FFN
    inp = synth.ffn_inputs(0, **w)
    got = gpu_ffn(qm, inp, w["hidden"], w["inter"], w["gate"], w["up"], w["down"])
    ref, tol = orc.ffn_swiglu(w["gate"], w["up"], w["down"], w["hidden"], w["inter"],
                              inp["gate"], inp["up"], inp["down"], inp["x"], inp["residual"])
    check_close(got, ref, tol, "dense ffn")


# ------------------------------------------------------------------ MoE
def gpu_moe(qm, inp, shp):
    import torch
    T, K = shp["n_tokens"], shp["top_k"]
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], K, T,
                     shp["gate"], shp["up"], shp["down"], shp.get("renormalize", True))
    res = _dev(inp["residual"])
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), device="cuda")
    ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device="cuda")
    qm.moe_ffn(_dev(inp["router"]), _dev(inp["gate"]), _dev(inp["up"]), _dev(inp["down"]), s,
               _dev(inp["x"]), res, idx, w, ws)
    torch.cuda.synchronize()
    return res.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def oracle_moe(orc, inp, shp, tokens=None):
    return orc.moe_ffn(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"],
                       shp["gate"], shp["up"], shp["down"], inp["router"], inp["gate"],
                       inp["up"], inp["down"], inp["x"], inp["residual"], tokens=tokens,
                       renormalize=shp.get("renormalize", True))


MOE_SMALL = [
    dict(hidden=256, expert_dim=256, num_experts=6, top_k=2, n_tokens=3),
    dict(hidden=512, expert_dim=512, num_experts=1, top_k=1, n_tokens=1),
    dict(hidden=256, expert_dim=768, num_experts=4, top_k=4, n_tokens=2),
    dict(hidden=1024, expert_dim=256, num_experts=40, top_k=16, n_tokens=1),
    dict(hidden=768, expert_dim=512, num_experts=256, top_k=3, n_tokens=2),
]


@pytest.mark.parametrize("shp", MOE_SMALL, ids=lambda s: "E{num_experts}k{top_k}T{n_tokens}".format(**s))
@pytest.mark.parametrize("fmts", [(synth.Q4_K, synth.Q6_K), (synth.Q8_0, synth.Q4_0),
                                  (synth.Q5_K, synth.Q4_K)], ids=lambda f: f"{QNAME[f[0]]}-{QNAME[f[1]]}")
def test_moe_small(qm, orc, shp, fmts):
    shp = dict(shp, gate=fmts[0], up=fmts[0], down=fmts[1])
    inp = synth.moe_inputs(31 + shp["num_experts"], **shp)
    out, idx, w = gpu_moe(qm, inp, shp)
    ref = oracle_moe(orc, inp, shp)
    assert check_moe(out, idx, w, ref) <= 1


def test_moe_decode_workload(qm, orc):
    """Qwen3-30B-A3B-shaped: hidden 2048, 128 experts, top-8, expert_dim 768."""
    shp = synth.MOE_DECODE
    inp = synth.moe_inputs(0, **shp)
    out, idx, w = gpu_moe(qm, inp, shp)
    ref = oracle_moe(orc, inp, shp)
    assert check_moe(out, idx, w, ref) == 0


@pytest.mark.parametrize("T", [1, 3])
def test_moe_input_is_residual(qm, orc, T):
    """x and residual the same buffer: every token reads its input before any
    product is added to it (the clusters of the single-token kernel do not
    wait for each other, so such a call takes the other kernels)."""
    import torch
    shp = dict(synth.MOE_DECODE, n_tokens=T)
    inp = synth.moe_inputs(44 + T, **shp)
    inp = dict(inp, x=inp["residual"].copy())
    K = shp["top_k"]
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], K, T, shp["gate"],
                     shp["up"], shp["down"])
    res = _dev(inp["residual"])
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), device="cuda")
    ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device="cuda")
    qm.moe_ffn(_dev(inp["router"]), _dev(inp["gate"]), _dev(inp["up"]), _dev(inp["down"]), s,
               res, res, idx, w, ws)
    torch.cuda.synchronize()
    assert qm.device_status() == qm.OK
    ref = oracle_moe(orc, inp, shp)
    assert check_moe(res.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), ref) == 0


def test_moe_prefill_workload_sampled(qm, orc):
    """OLMoE-shaped, 512 tokens: every token's routing checked exactly;
    residuals of 12 sampled tokens checked against the oracle."""
    shp = synth.MOE_PREFILL
    inp = synth.moe_inputs(0, **shp)
    out, idx, w = gpu_moe(qm, inp, shp)
    toks = np.array([0, 1, 2, 63, 64, 127, 200, 255, 256, 384, 510, 511])
    ref = oracle_moe(orc, inp, shp, tokens=toks)
    assert check_moe(out[toks], idx[toks], w[toks], ref) <= 2
    # routing of all tokens: exact top-k wherever the oracle's logits are
    # unambiguous, a valid top-k elsewhere
    K = shp["top_k"]
    R64, X64 = inp["router"].astype(np.float64), inp["x"].astype(np.float64)
    logits = X64 @ R64.T
    scales = (np.abs(X64) @ np.abs(R64).T).max(axis=1)
    mismatched = 0
    for t in range(shp["n_tokens"]):
        ri, _ = orc.route(logits[t], K)
        srt = np.sort(logits[t])[::-1][: K + 1]
        if np.min(-np.diff(srt)) > AMBIGUITY * scales[t]:
            assert list(idx[t]) == list(ri), t
        else:
            assert route_is_valid(idx[t], logits[t], scales[t], K), t
            mismatched += list(idx[t]) != list(ri)
    assert mismatched <= 5


# ------------------------------------------ routing without renormalisation
NO_RENORM = [
    dict(synth.MOE_DECODE),                                                # fused, 1 token
    dict(synth.MOE_DECODE, n_tokens=5),                                    # batched
    dict(hidden=256, expert_dim=256, num_experts=8, top_k=2, n_tokens=64,
         gate=synth.Q4_K, up=synth.Q4_K, down=synth.Q6_K),                 # tensor cores
    dict(hidden=512, expert_dim=256, num_experts=256, top_k=16, n_tokens=1,
         gate=synth.Q5_K, up=synth.Q5_K, down=synth.Q8_0),                 # E = 256, k = 16
]


@pytest.mark.parametrize("shp", NO_RENORM, ids=lambda s: "E{num_experts}k{top_k}T{n_tokens}".format(**s))
def test_moe_no_renorm(qm, orc, shp):
    """route_flags = QMOE_ROUTE_NO_RENORM: weights are the softmax
    probabilities of the selected experts; they sum to less than one."""
    shp = dict(shp, renormalize=False)
    inp = synth.moe_inputs(41 + shp["n_tokens"], **shp)
    out, idx, w = gpu_moe(qm, inp, shp)
    ref = oracle_moe(orc, inp, shp)
    assert check_moe(out, idx, w, ref) <= 1
    assert np.all(w.sum(axis=1) < 1.0)
    assert qm.device_status() == qm.OK


# ----------------------------------------------- many tokens (tensor cores)
MOE_PREFILL_SMALL = [
    dict(hidden=256, expert_dim=256, num_experts=8, top_k=2, n_tokens=64),
    dict(hidden=512, expert_dim=512, num_experts=16, top_k=4, n_tokens=40),
    dict(hidden=256, expert_dim=256, num_experts=2, top_k=1, n_tokens=300),   # >128 per expert
    dict(hidden=768, expert_dim=256, num_experts=64, top_k=8, n_tokens=32),   # smallest T
    dict(hidden=256, expert_dim=768, num_experts=33, top_k=3, n_tokens=97),
]


@pytest.mark.parametrize("shp", MOE_PREFILL_SMALL,
                         ids=lambda s: "H{hidden}F{expert_dim}E{num_experts}k{top_k}T{n_tokens}".format(**s))
def test_moe_many_tokens_all_checked(qm, orc, shp):
    """Grouped tensor-core path (Q4_K gate/up, Q6_K down): every token."""
    shp = dict(shp, gate=synth.Q4_K, up=synth.Q4_K, down=synth.Q6_K)
    inp = synth.moe_inputs(71 + shp["n_tokens"], **shp)
    out, idx, w = gpu_moe(qm, inp, shp)
    ref = oracle_moe(orc, inp, shp)
    assert check_moe(out, idx, w, ref) <= max(2, shp["n_tokens"] // 20)
    assert qm.device_status() == qm.OK


def test_moe_many_tokens_f16_range_reported(qm):
    """A Q4_K gate weight beyond f16 range (d = 60000, scales 63, quants 15)
    cannot be a tensor-core operand: the many-token path reports it as
    UNSUPPORTED through the device status, and the status is cleared after."""
    shp = dict(hidden=256, expert_dim=256, num_experts=4, top_k=2, n_tokens=64,
               gate=synth.Q4_K, up=synth.Q4_K, down=synth.Q6_K)
    inp = synth.moe_inputs(9, **shp)
    gate = inp["gate"].reshape(shp["num_experts"], shp["expert_dim"], -1).copy()
    blocks = gate.reshape(shp["num_experts"], shp["expert_dim"], -1, 144)
    blocks[:, 0, :, 0:2] = np.frombuffer(np.float16(60000.0).tobytes(), np.uint8)
    blocks[:, 0, :, 4:] = 0xFF
    inp["gate"] = gate.reshape(inp["gate"].shape)
    gpu_moe(qm, inp, shp)
    assert qm.device_status() == qm.ERR_UNSUPPORTED
    assert "f16 range" in qm.last_error()
    assert qm.device_status() == qm.OK


# ------------------------------------------------- non-finite activations
NON_FINITE = [
    dict(synth.MOE_DECODE),                                                # fused, 1 token
    dict(synth.MOE_DECODE, n_tokens=5),                                    # batched
    dict(hidden=512, expert_dim=256, num_experts=16, top_k=4, n_tokens=64,
         gate=synth.Q4_K, up=synth.Q4_K, down=synth.Q6_K),                 # tensor cores
]


@pytest.mark.parametrize("bad", ["nan", "inf"])
@pytest.mark.parametrize("shp", NON_FINITE, ids=lambda s: "T{n_tokens}".format(**s))
def test_moe_non_finite_activation(qm, orc, shp, bad):
    """One activation of one token is NaN or +Inf.  That token's logits are
    then NaN or +-Inf, its softmax is NaN throughout, and its route is experts
    0..k-1 with NaN weights (the order the oracle's stable sort leaves NaN
    probabilities in); its residual becomes NaN.  Every slot names an expert
    in range, and the other tokens are routed and computed as usual."""
    inp = synth.moe_inputs(61 + shp["n_tokens"], **shp)
    T, K = shp["n_tokens"], shp["top_k"]
    tb = T // 2
    inp["x"] = inp["x"].copy()
    inp["x"].reshape(T, -1)[tb, 100] = np.nan if bad == "nan" else np.inf
    out, idx, w = gpu_moe(qm, inp, shp)
    assert qm.device_status() == qm.OK
    ref = oracle_moe(orc, inp, shp)
    assert list(ref["idx"][tb]) == list(range(K)) and np.all(np.isnan(ref["w"][tb]))
    assert idx[tb].tolist() == list(range(K))
    assert np.all(np.isnan(w[tb])) and np.all(np.isnan(out.reshape(T, -1)[tb]))
    assert check_moe(out, idx, w, ref) <= max(1, T // 20)


# ------------------------------------- Q8_0 / Q4_0 widths of 32-element blocks
@pytest.mark.parametrize("qt", [synth.Q8_0, synth.Q4_0], ids=lambda q: QNAME[q])
@pytest.mark.parametrize("rows,cols", [(5, 96), (37, 896), (300, 4128), (64, 32), (17, 288),
                                       (153, 4064), (9, 32736)])
def test_qmv_widths_of_32(qm, orc, qt, rows, cols):
    """cols a multiple of 32 but not of 256 (block_bytes_per_row on
    "ferrox-core 0.16.0 — weight_matrix.rs" needs only whole 32-element
    blocks): the last 256-element group of each row is partial, and rows of
    an odd number of blocks sit at 2-byte-aligned offsets."""
    g = synth.rng(2000 + qt * 11 + cols)
    W = synth.quant_matrix(g, qt, rows, cols, nan_row=rows // 2 if rows > 2 else None)
    x = synth.normal(g, cols)
    y = gpu_qmv(qm, qt, W, rows, cols, x)
    ref, sabs = orc.matvec(qt, W, rows, cols, x, with_sabs=True)
    check_gemv(y, ref, sabs, f"qmv {QNAME[qt]} {rows}x{cols}")
    assert qm.device_status() == qm.OK


# ------------------------------------------------------ lm_head-sized GEMVs
@pytest.mark.parametrize("qt", [synth.F32, synth.Q6_K, synth.Q8_0], ids=lambda q: QNAME[q])
def test_qmv_lm_head_size(qm, orc, qt):
    """vocab 151,936 x hidden 2048 (a Qwen3-sized output projection): every
    row checked.  The pages keep the F32 router and the lm_head GEMV on the
    host ("ferrox-core 0.16.0 — weight_matrix.rs", apply_gpu); here they run
    on the device through the same entry point."""
    g = synth.rng(151936 + qt)
    rows, cols = 151936, 2048
    if qt == synth.F32:
        W = synth.normal(g, (rows, cols), 0.02)
        Wb = W.view(np.uint8)
    else:
        W = Wb = synth.quant_matrix(g, qt, rows, cols, nan_row=7)
    x = synth.normal(g, cols)
    y = gpu_qmv(qm, qt, W, rows, cols, x)
    ref, sabs = orc.matvec(orc.F32 if qt == synth.F32 else qt, Wb, rows, cols, x, with_sabs=True)
    check_gemv(y, ref, sabs, f"lm_head {QNAME[qt]}")
