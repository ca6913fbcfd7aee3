"""CPU oracle for GGUF block-quantized GEMV and the decode-time MoE FFN.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only code allowed to import it; the
CUDA library never calls it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation, built with
gcc -O2 and no fast-math).  This module only compiles it, loads it with
ctypes and marshals numpy arrays.  Every function cites, in ``oracle.c``, the
page section it follows.

Pins: every function here is pinned by ``tests/test_oracle_*.py`` to values
fixed by the pages or by mathematics (hand-built blocks, exhaustive f16 and
scale/min checks, one-hot extraction, closed forms, library special cases,
brute force on tiny cases).  None is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Format codes (the oracle's own numbering; mirrors the enum in oracle.c).
F32, Q8_0, Q4_0, Q4_K, Q5_K, Q6_K = 0, 1, 2, 3, 4, 5
NAMES = {F32: "F32", Q8_0: "Q8_0", Q4_0: "Q4_0", Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K"}
BLOCK_ELEMS = {F32: 1, Q8_0: 32, Q4_0: 32, Q4_K: 256, Q5_K: 256, Q6_K: 256}
BLOCK_BYTES = {F32: 4, Q8_0: 34, Q4_0: 18, Q4_K: 144, Q5_K: 176, Q6_K: 210}


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.orc_f16_to_f32.restype = ctypes.c_float
            lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_k_scale_min.restype = None
            lib.orc_k_scale_min.argtypes = [ctypes.c_int, P, P, P]
            lib.orc_decode_block.restype = ctypes.c_int
            lib.orc_decode_block.argtypes = [ctypes.c_int, P, P]
            lib.orc_dequant_row.restype = ctypes.c_int
            lib.orc_dequant_row.argtypes = [ctypes.c_int, P, i64, P]
            lib.orc_matvec.restype = ctypes.c_int
            lib.orc_matvec.argtypes = [ctypes.c_int, P, i64, i64, P, P, P]
            lib.orc_matvec_fused.restype = ctypes.c_int
            lib.orc_matvec_fused.argtypes = [ctypes.c_int, P, i64, i64, P, P]
            lib.orc_route.restype = ctypes.c_int
            lib.orc_route.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
            lib.orc_moe_ffn.restype = ctypes.c_int
            lib.orc_moe_ffn.argtypes = [P, i64, P, P, P, P, P, P, P, P, P, P, P, P, P]
            lib.orc_ffn_swiglu.restype = ctypes.c_int
            lib.orc_ffn_swiglu.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, i64,
                                           P, P, P, P, P, P, P]
            lib.orc_row_bytes.restype = i64
            lib.orc_row_bytes.argtypes = [ctypes.c_int, i64]
            lib.orc_rmsnorm.restype = ctypes.c_int
            lib.orc_rmsnorm.argtypes = [P, P, i64, ctypes.c_double, P]
            _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _u8(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint8).reshape(-1)


def row_bytes(qt: int, cols: int) -> int:
    return int(_load().orc_row_bytes(qt, cols))


def f16_to_f32(bits: int) -> float:
    return float(_load().orc_f16_to_f32(int(bits) & 0xFFFF))


def k_scale_min(j: int, scales12) -> tuple[int, int]:
    s = np.ascontiguousarray(np.asarray(scales12, dtype=np.uint8))
    assert s.size == 12
    sc = np.zeros(1, np.uint8)
    m = np.zeros(1, np.uint8)
    _load().orc_k_scale_min(j, _ptr(s), _ptr(sc), _ptr(m))
    return int(sc[0]), int(m[0])


def decode_block(qt: int, block) -> np.ndarray:
    b = _u8(np.asarray(block, dtype=np.uint8))
    assert b.size == BLOCK_BYTES[qt]
    out = np.zeros(BLOCK_ELEMS[qt], np.float32)
    assert _load().orc_decode_block(qt, _ptr(b), _ptr(out)) == 0
    return out


def dequant(qt: int, W, rows: int, cols: int) -> np.ndarray:
    """Decode a [rows][row_bytes] matrix to f32 [rows][cols]."""
    w = _u8(W)
    rb = row_bytes(qt, cols)
    assert rb > 0 and w.size >= rows * rb
    out = np.zeros((rows, cols), np.float32)
    lib = _load()
    for r in range(rows):
        rowv = w[r * rb:(r + 1) * rb]
        assert lib.orc_dequant_row(qt, _ptr(rowv), cols, _ptr(out[r])) == 0
    return out


def matvec(qt: int, W, rows: int, cols: int, x, with_sabs: bool = False):
    """y = W x in double (decode-then-dot); optionally S_r = sum_j |w_rj x_j|."""
    w = _u8(W)
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == cols
    y = np.zeros(rows, np.float64)
    s = np.zeros(rows, np.float64) if with_sabs else None
    assert _load().orc_matvec(qt, _ptr(w), rows, cols, _ptr(x), _ptr(y), _ptr(s)) == 0
    return (y, s) if with_sabs else y


def matvec_fused(qt: int, W, rows: int, cols: int, x) -> np.ndarray:
    w = _u8(W)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.zeros(rows, np.float64)
    assert _load().orc_matvec_fused(qt, _ptr(w), rows, cols, _ptr(x), _ptr(y)) == 0
    return y


def route(logits, k: int, renormalize: bool = True):
    """(idx, w): the k routed experts in rank order and their weights,
    renormalised over the k (default) or the softmax probabilities over all
    experts (renormalize=False)."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    E = lg.size
    idx = np.zeros(k, np.int32)
    w = np.zeros(k, np.float64)
    rc = _load().orc_route(_ptr(lg), E, k, int(bool(renormalize)), _ptr(idx), _ptr(w))
    if rc != 0:
        raise ValueError(f"orc_route rejected E={E} k={k}")
    return idx, w


class _Shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("expert_dim", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("gate_qt", ctypes.c_int32), ("up_qt", ctypes.c_int32),
                ("down_qt", ctypes.c_int32), ("no_renorm", ctypes.c_int32)]


def moe_ffn(hidden, expert_dim, num_experts, top_k, gate_qt, up_qt, down_qt,
            router, gate, up, down, x, residual, tokens=None, renormalize=True):
    """MoE FFN per token.  x, residual: [T][hidden].  ``tokens`` (optional)
    restricts the computation to those token rows (sampled checks).
    ``renormalize`` selects the routing weights (see route).

    Returns dict(out [T'][hidden] f64, tol, idx [T'][k], w [T'][k], gap [T'],
    logits [T'][E], lscale [T'] = max_e sum_j |R_ej x_j|)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, hidden)
    residual = np.ascontiguousarray(residual, dtype=np.float32).reshape(-1, hidden)
    if tokens is not None:
        tokens = np.asarray(tokens, dtype=np.int64)
        x = np.ascontiguousarray(x[tokens])
        residual = np.ascontiguousarray(residual[tokens])
    T = x.shape[0]
    sh = _Shape(hidden, expert_dim, num_experts, top_k, gate_qt, up_qt, down_qt,
                0 if renormalize else 1)
    router = np.ascontiguousarray(router, dtype=np.float32)
    out = np.zeros((T, hidden), np.float64)
    tol = np.zeros((T, hidden), np.float64)
    idx = np.zeros((T, top_k), np.int32)
    w = np.zeros((T, top_k), np.float64)
    gap = np.zeros(T, np.float64)
    logits = np.zeros((T, num_experts), np.float64)
    lscale = np.zeros(T, np.float64)
    rc = _load().orc_moe_ffn(ctypes.byref(sh), T, _ptr(router), _ptr(_u8(gate)), _ptr(_u8(up)),
                             _ptr(_u8(down)), _ptr(x), _ptr(residual), _ptr(out), _ptr(tol),
                             _ptr(idx), _ptr(w), _ptr(gap), _ptr(logits), _ptr(lscale))
    if rc != 0:
        raise ValueError(f"orc_moe_ffn rejected the shape (rc={rc})")
    return dict(out=out, tol=tol, idx=idx, w=w, gap=gap, logits=logits, lscale=lscale)


def ffn_swiglu(gate_qt, up_qt, down_qt, hidden, inter, gate, up, down, x, residual):
    """Dense SwiGLU FFN added to the residual; returns (out f64 [hidden], tol)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    residual = np.ascontiguousarray(residual, dtype=np.float32)
    out = np.zeros(hidden, np.float64)
    tol = np.zeros(hidden, np.float64)
    rc = _load().orc_ffn_swiglu(gate_qt, up_qt, down_qt, hidden, inter, _ptr(_u8(gate)),
                                _ptr(_u8(up)), _ptr(_u8(down)), _ptr(x), _ptr(residual),
                                _ptr(out), _ptr(tol))
    if rc != 0:
        raise ValueError("orc_ffn_swiglu rejected the shape")
    return out, tol


def rmsnorm(h, w, eps: float) -> np.ndarray:
    """ffn_norm: h * w / sqrt(mean(h^2) + eps) per row of h ([T][n] or [n]),
    in double (orc_rmsnorm)."""
    h = np.ascontiguousarray(h, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    n = w.shape[0]
    rows = h.reshape(-1, n)
    out = np.zeros(rows.shape, np.float64)
    for t in range(rows.shape[0]):
        r = np.ascontiguousarray(rows[t])
        o = np.zeros(n, np.float64)
        if _load().orc_rmsnorm(_ptr(r), _ptr(w), n, float(eps), _ptr(o)) != 0:
            raise ValueError("orc_rmsnorm rejected the arguments")
        out[t] = o
    return out.reshape(h.shape)
