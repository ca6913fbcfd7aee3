"""The C-ABI library on CPU: it builds, loads, exports every function the
header declares, and its host-side argument checks refuse bad calls before
any CUDA work (no compute call is made without a GPU)."""
import ctypes
import re

import pytest

import moe_ffn_gb300 as qm


@pytest.fixture(scope="module")
def lib():
    qm.build()
    return qm.lib()


def header_functions():
    text = open(qm.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined"})


def test_header_symbols_exported(lib):
    names = header_functions()
    assert {"qmv", "ffn_swiglu", "moe_ffn", "moe_ffn_workspace_size",
            "ffn_swiglu_workspace_size", "qmoe_device_status", "qmoe_last_error",
            "qmoe_row_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in qm.SIGNATURES, n


def test_row_bytes(lib):
    assert qm.row_bytes(qm.Q4_K, 4096) == 2304
    assert qm.row_bytes(qm.Q6_K, 768) == 630
    assert qm.row_bytes(qm.Q8_0, 4096) == 4352
    assert qm.row_bytes(qm.Q4_0, 1024) == 576
    assert qm.row_bytes(qm.Q5_K, 4096) == 2816
    assert qm.row_bytes(qm.F32, 7) == 28
    assert qm.row_bytes(qm.Q4_K, 300) == -1
    assert qm.row_bytes(99, 256) == -1


def test_workspace_sizes_cover_batched_launches(lib):
    """2..31 tokens run in batched launches of up to 16 tokens, whose
    activations are [tokens][k][F] f32: the workspace grows with T up to 16
    tokens' worth and covers the logits of every token."""
    H, F, E, K = 2048, 768, 128, 8
    prev = 0
    for T in (1, 2, 3, 8, 16, 17, 31):
        s = qm.moe_shape(H, F, E, K, T, qm.Q4_K, qm.Q4_K, qm.Q6_K)
        need = qm.moe_ffn_workspace_size(s)
        assert need >= 256 + T * E * 4 + min(T, 16) * K * F * 4
        assert need % 256 == 0 and need >= prev
        prev = need


def test_workspace_sizes(lib):
    s = qm.moe_shape(2048, 768, 128, 8, 1, qm.Q4_K, qm.Q4_K, qm.Q6_K)
    assert qm.moe_ffn_workspace_size(s) >= 128 * 4 + 8 * 768 * 4
    assert qm.moe_ffn_workspace_size(s) % 256 == 0
    assert qm.ffn_swiglu_workspace_size(4096, 14336) >= 14336 * 4
    assert qm.moe_ffn_workspace_size(qm.moe_shape(0, 0, 0, 0, 0, 0, 0, 0)) == 0


FAKE = 1 << 20  # a 16-byte-aligned non-null address, never dereferenced


@pytest.mark.parametrize("args,status", [
    ((qm.Q4_K, None, 4, 256, FAKE, FAKE), qm.ERR_INVALID_ARGUMENT),
    ((qm.Q4_K, FAKE, 0, 256, FAKE, FAKE), qm.ERR_INVALID_ARGUMENT),
    ((qm.Q4_K, FAKE, 4, 100, FAKE, FAKE), qm.ERR_INVALID_ARGUMENT),
    ((qm.Q4_K, FAKE, 4, 96, FAKE, FAKE), qm.ERR_INVALID_ARGUMENT),
    ((qm.F32, FAKE, 4, 6, FAKE, FAKE), qm.ERR_UNSUPPORTED),
    ((qm.Q4_K, FAKE + 4, 4, 256, FAKE, FAKE), qm.ERR_INVALID_ARGUMENT),
    ((17, FAKE, 4, 256, FAKE, FAKE), qm.ERR_UNSUPPORTED),
    ((qm.Q4_K, FAKE, 4, 1 << 20, FAKE, FAKE), qm.ERR_UNSUPPORTED),
])
def test_qmv_refuses_before_cuda(lib, args, status):
    qt, W, rows, cols, x, y = args
    st = lib.qmv(qt, W, rows, cols, x, y, None)
    assert st == status
    assert qm.last_error()


def test_moe_refusals(lib):
    def call(shape, ws_bytes=1 << 20, ptr=FAKE):
        return lib.moe_ffn(ptr, ptr, ptr, ptr, ctypes.byref(shape), ptr, ptr, None, None, ptr,
                           ws_bytes, None)
    ok = dict(hidden=2048, expert_dim=768, num_experts=128, top_k=8, n_tokens=1,
              gate_qtype=qm.Q4_K, up_qtype=qm.Q4_K, down_qtype=qm.Q6_K)

    def shape(**kw):
        d = dict(ok, **kw)
        return qm.moe_shape(**{k: d[k] for k in ok})
    assert call(shape(top_k=129)) == qm.ERR_INVALID_ARGUMENT        # k > E
    assert call(shape(num_experts=0)) == qm.ERR_INVALID_ARGUMENT
    assert call(shape(num_experts=300, top_k=8)) == qm.ERR_UNSUPPORTED
    assert call(shape(top_k=17, num_experts=64)) == qm.ERR_UNSUPPORTED
    assert call(shape(up_qtype=qm.Q5_K)) == qm.ERR_UNSUPPORTED      # mixed gate/up
    assert call(shape(down_qtype=qm.F32)) == qm.ERR_UNSUPPORTED
    assert call(shape(hidden=2048 + 32)) == qm.ERR_INVALID_ARGUMENT  # not whole Q4_K blocks
    assert call(shape(), ws_bytes=16) == qm.ERR_INVALID_ARGUMENT
    assert call(shape(), ptr=None) == qm.ERR_INVALID_ARGUMENT
    assert "top_k" in qm.last_error() or "null" in qm.last_error()
    bad = shape()
    bad.route_flags = 2  # not a known flag
    assert call(bad) == qm.ERR_INVALID_ARGUMENT
    assert "route_flags" in qm.last_error()


def test_ffn_refusals(lib):
    f = lib.ffn_swiglu
    assert f(FAKE, FAKE, FAKE, qm.Q4_K, qm.Q8_0, qm.Q6_K, 4096, 14336, FAKE, FAKE, FAKE,
             1 << 20, None) == qm.ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, qm.Q4_K, qm.Q4_K, qm.Q6_K, 4096, 14336, FAKE, FAKE, FAKE,
             16, None) == qm.ERR_INVALID_ARGUMENT
    assert f(None, FAKE, FAKE, qm.Q4_K, qm.Q4_K, qm.Q6_K, 4096, 14336, FAKE, FAKE, FAKE,
             1 << 20, None) == qm.ERR_INVALID_ARGUMENT


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(qm, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(qm, "_libh", None)
    with pytest.raises(qm.QmoeError):
        qm.lib()


def test_rmsnorm_workspace_sizes(lib):
    s = qm.moe_shape(2048, 768, 128, 8, 3, qm.Q4_K, qm.Q4_K, qm.Q6_K)
    assert qm.moe_ffn_rmsnorm_workspace_size(s) == qm.moe_ffn_workspace_size(s) + 3 * 2048 * 4
    assert qm.ffn_swiglu_rmsnorm_workspace_size(4096, 14336) >= \
        qm.ffn_swiglu_workspace_size(4096, 14336) + 4096 * 4
    assert qm.moe_ffn_rmsnorm_workspace_size(qm.moe_shape(0, 0, 0, 0, 0, 0, 0, 0)) == 0


def test_rmsnorm_refusals(lib):
    s = qm.moe_shape(2048, 768, 128, 8, 1, qm.Q4_K, qm.Q4_K, qm.Q6_K)
    big = 1 << 24

    def moe(norm=FAKE, eps=1e-6, res=FAKE, ws_bytes=big):
        return lib.moe_ffn_rmsnorm(FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), norm, eps, res, None,
                                   None, FAKE, ws_bytes, None)
    assert moe(norm=None) == qm.ERR_INVALID_ARGUMENT
    assert moe(eps=-1.0) == qm.ERR_INVALID_ARGUMENT
    assert moe(eps=float("nan")) == qm.ERR_INVALID_ARGUMENT
    assert moe(eps=float("inf")) == qm.ERR_INVALID_ARGUMENT
    assert moe(res=FAKE + 4) == qm.ERR_INVALID_ARGUMENT   # the norm reads the residual as float4
    assert moe(ws_bytes=qm.moe_ffn_workspace_size(s)) == qm.ERR_INVALID_ARGUMENT  # no room for xn
    assert "moe_ffn_rmsnorm" in qm.last_error()

    def ffn(norm=FAKE, eps=1e-6, ws_bytes=big):
        return lib.ffn_swiglu_rmsnorm(FAKE, FAKE, FAKE, qm.Q4_K, qm.Q4_K, qm.Q6_K, 4096, 14336,
                                      norm, eps, FAKE, FAKE, ws_bytes, None)
    assert ffn(norm=None) == qm.ERR_INVALID_ARGUMENT
    assert ffn(eps=-0.5) == qm.ERR_INVALID_ARGUMENT
    assert ffn(ws_bytes=qm.ffn_swiglu_workspace_size(4096, 14336)) == qm.ERR_INVALID_ARGUMENT
    assert "ffn_swiglu_rmsnorm" in qm.last_error()


def test_noalloc_scratch_constant_matches_header():
    """The binding's NOALLOC_SCRATCH_BYTES is the header's macro."""
    text = open(qm.HEADER).read()
    m = re.search(r"#define\s+QMOE_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "QMOE_NOALLOC_SCRATCH_BYTES not found in the header"
    assert int(m.group(1)) << int(m.group(2)) == qm.NOALLOC_SCRATCH_BYTES


def test_exec_mode_refuses_unknown(lib):
    assert lib.qmoe_set_exec_mode(7) == qm.ERR_INVALID_ARGUMENT
    assert "mode" in qm.last_error()
    assert lib.qmoe_set_exec_mode(qm.EXEC_DEFAULT) == qm.OK
