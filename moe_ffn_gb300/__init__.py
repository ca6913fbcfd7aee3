"""moe_ffn_gb300 — Python binding of libqmoe.so, the GB300 (sm_103a) GGUF
block-quantized GEMV and decode-time MoE FFN library.

This module only marshals arguments: every step of every call runs in the
library's CUDA kernels.  PyTorch supplies device memory (``tensor.data_ptr()``)
and streams (``torch.cuda.current_stream().cuda_stream``).  There is no CPU
fallback: if the compiled library is missing, loading it raises.

Function names follow the C ABI declared in ``include/qmoe.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
LIB_PATH = os.path.join(_HERE, "libqmoe.so")
HEADER = os.path.join(_ROOT, "include", "qmoe.h")

# qmoe_qtype
F32, Q8_0, Q4_0, Q4_K, Q5_K, Q6_K = 0, 1, 2, 3, 4, 5
QTYPES = {"F32": F32, "Q8_0": Q8_0, "Q4_0": Q4_0, "Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K}
BLOCK_ELEMS = {F32: 1, Q8_0: 32, Q4_0: 32, Q4_K: 256, Q5_K: 256, Q6_K: 256}
BLOCK_BYTES = {F32: 4, Q8_0: 34, Q4_0: 18, Q4_K: 144, Q5_K: 176, Q6_K: 210}

# qmoe_status
OK, ERR_INVALID_ARGUMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
STATUS_NAMES = {0: "OK", 1: "INVALID_ARGUMENT", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT"}

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-ftz=false",
              "-std=c++17", "-Xcompiler", "-fPIC"]
# Translation units of libqmoe.so, compiled in parallel and linked together.
UNITS = ("qmoe.cu", "batch.cu")


class QmoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


def _sources():
    return sorted(os.path.join(_CSRC, f) for f in os.listdir(_CSRC)
                  if f.endswith((".cu", ".cuh")))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libqmoe.so in-tree for sm_103a with nvcc."""
    srcs = _sources() + [HEADER]
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(s) for s in srcs)):
        return LIB_PATH
    nvcc = os.environ.get("NVCC", "nvcc")
    if not os.path.exists(nvcc) and os.path.exists("/usr/local/cuda/bin/nvcc"):
        nvcc = "/usr/local/cuda/bin/nvcc"
    tag = f".{os.getpid()}.tmp"
    objs = [os.path.join(_HERE, u.replace(".cu", f".{os.getpid()}.o")) for u in UNITS]
    procs = []
    for u, o in zip(UNITS, objs):
        cmd = [nvcc, *NVCC_FLAGS, "-c", "-o", o, os.path.join(_CSRC, u)]
        if verbose:
            print(" ".join(cmd))
        procs.append(subprocess.Popen(cmd))
    codes = [p.wait() for p in procs]
    try:
        for u, c in zip(UNITS, codes):
            if c:
                raise subprocess.CalledProcessError(c, f"nvcc {u}")
        tmp = LIB_PATH + tag
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd))
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB_PATH


class _Shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("expert_dim", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("n_tokens", ctypes.c_int32), ("gate_qtype", ctypes.c_int32),
                ("up_qtype", ctypes.c_int32), ("down_qtype", ctypes.c_int32),
                ("route_flags", ctypes.c_int32)]


_lock = threading.Lock()
_libh = None

# Exported symbols and their ctypes signatures (mirrors include/qmoe.h).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
SIGNATURES = {
    "qmv": (ctypes.c_int, [ctypes.c_int, _P, _I64, _I64, _P, _P, _P]),
    "ffn_swiglu_workspace_size": (ctypes.c_size_t, [_I64, _I64]),
    "ffn_swiglu": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64, _I64,
                                  _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_ffn_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(_Shape)]),
    "moe_ffn": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(_Shape), _P, _P, _P, _P, _P,
                               ctypes.c_size_t, _P]),
    "moe_ffn_noalloc": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(_Shape), _P, _P, _P, _P,
                                        _P]),
    "ffn_swiglu_rmsnorm_workspace_size": (ctypes.c_size_t, [_I64, _I64]),
    "ffn_swiglu_rmsnorm": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          _I64, _I64, _P, ctypes.c_float, _P, _P, ctypes.c_size_t,
                                          _P]),
    "moe_ffn_rmsnorm_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(_Shape)]),
    "moe_ffn_rmsnorm": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(_Shape), _P, ctypes.c_float,
                                       _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "qmoe_device_status": (ctypes.c_int, [_P]),
    "qmoe_set_exec_mode": (ctypes.c_int, [ctypes.c_int]),
    "qmoe_set_fault_injection": (ctypes.c_int, [ctypes.c_uint64, ctypes.c_int]),
    "qmoe_last_error": (ctypes.c_char_p, []),
    "qmoe_row_bytes": (_I64, [ctypes.c_int, _I64]),
}


def lib():
    """The loaded library; raises if it has not been built."""
    global _libh
    with _lock:
        if _libh is None:
            if not os.path.exists(LIB_PATH):
                raise QmoeError(ERR_CUDA, f"{LIB_PATH} is missing: run moe_ffn_gb300.build()")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _libh = h
    return _libh


def last_error() -> str:
    return lib().qmoe_last_error().decode()


def _check(status: int):
    if status != OK:
        raise QmoeError(status, last_error())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def row_bytes(qtype: int, cols: int) -> int:
    return int(lib().qmoe_row_bytes(qtype, cols))


def qmv(qtype: int, W, rows: int, cols: int, x, y, stream=None) -> None:
    """y = W x (see include/qmoe.h)."""
    _check(lib().qmv(qtype, _ptr(W), rows, cols, _ptr(x), _ptr(y), _stream(stream)))


def ffn_swiglu_workspace_size(hidden: int, inter: int) -> int:
    return int(lib().ffn_swiglu_workspace_size(hidden, inter))


def ffn_swiglu(gate, up, down, gate_qtype, up_qtype, down_qtype, hidden, inter, x, residual,
               ws, ws_bytes=None, stream=None) -> None:
    """residual += down(silu(gate x) * (up x)) (see include/qmoe.h)."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().ffn_swiglu(_ptr(gate), _ptr(up), _ptr(down), gate_qtype, up_qtype, down_qtype,
                            hidden, inter, _ptr(x), _ptr(residual), _ptr(ws), ws_bytes,
                            _stream(stream)))


# shape.route_flags: routing weights are the softmax probabilities, not renormalised
ROUTE_NO_RENORM = 1


def moe_shape(hidden, expert_dim, num_experts, top_k, n_tokens, gate_qtype, up_qtype,
              down_qtype, renormalize: bool = True) -> _Shape:
    return _Shape(hidden, expert_dim, num_experts, top_k, n_tokens, gate_qtype, up_qtype,
                  down_qtype, 0 if renormalize else ROUTE_NO_RENORM)


def moe_ffn_workspace_size(shape: _Shape) -> int:
    return int(lib().moe_ffn_workspace_size(ctypes.byref(shape)))


def moe_ffn(router_W, gate_stack, up_stack, down_stack, shape: _Shape, x, residual,
            topk_idx=None, topk_w=None, ws=None, ws_bytes=None, stream=None) -> None:
    """One MoE FFN layer for shape.n_tokens tokens (see include/qmoe.h)."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().moe_ffn(_ptr(router_W), _ptr(gate_stack), _ptr(up_stack), _ptr(down_stack),
                         ctypes.byref(shape), _ptr(x), _ptr(residual), _ptr(topk_idx),
                         _ptr(topk_w), _ptr(ws), ws_bytes, _stream(stream)))


def ffn_swiglu_rmsnorm_workspace_size(hidden: int, inter: int) -> int:
    return int(lib().ffn_swiglu_rmsnorm_workspace_size(hidden, inter))


def ffn_swiglu_rmsnorm(gate, up, down, gate_qtype, up_qtype, down_qtype, hidden, inter, norm_w,
                       eps, residual, ws, ws_bytes=None, stream=None) -> None:
    """residual += FFN(rmsnorm(residual)) (see include/qmoe.h)."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().ffn_swiglu_rmsnorm(_ptr(gate), _ptr(up), _ptr(down), gate_qtype, up_qtype,
                                    down_qtype, hidden, inter, _ptr(norm_w), float(eps),
                                    _ptr(residual), _ptr(ws), ws_bytes, _stream(stream)))


def moe_ffn_rmsnorm_workspace_size(shape: _Shape) -> int:
    return int(lib().moe_ffn_rmsnorm_workspace_size(ctypes.byref(shape)))


def moe_ffn_rmsnorm(router_W, gate_stack, up_stack, down_stack, shape: _Shape, norm_w, eps,
                    residual, topk_idx=None, topk_w=None, ws=None, ws_bytes=None,
                    stream=None) -> None:
    """residual_t += MoE(rmsnorm(residual_t)) for every token (see include/qmoe.h)."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().moe_ffn_rmsnorm(_ptr(router_W), _ptr(gate_stack), _ptr(up_stack),
                                 _ptr(down_stack), ctypes.byref(shape), _ptr(norm_w), float(eps),
                                 _ptr(residual), _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws_bytes,
                                 _stream(stream)))


NOALLOC_SCRATCH_BYTES = 1 << 20


def moe_ffn_noalloc(router_W, gate_stack, up_stack, down_stack, shape: _Shape, x, residual,
                    topk_idx=None, topk_w=None, stream=None) -> None:
    """moe_ffn without a workspace argument: for callers that cannot allocate
    device memory.  Scratch is the library's built-in array
    (NOALLOC_SCRATCH_BYTES); calls share it, so calls that overlap on the
    GPU race (see include/qmoe.h)."""
    _check(lib().moe_ffn_noalloc(_ptr(router_W), _ptr(gate_stack), _ptr(up_stack),
                                 _ptr(down_stack), ctypes.byref(shape), _ptr(x), _ptr(residual),
                                 _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


# qmoe_set_exec_mode
EXEC_DEFAULT, EXEC_SEPARATE, EXEC_UNBATCHED = 0, 1, 2


def set_exec_mode(mode: int) -> None:
    """Diagnostics and tests: which equivalent kernel forms later calls launch
    (EXEC_DEFAULT, EXEC_SEPARATE or EXEC_UNBATCHED; see include/qmoe.h)."""
    _check(lib().qmoe_set_exec_mode(mode))


def set_fault_injection(wait_limit_ns: int = 0, skip_arrive_cta: int = -1) -> None:
    """Failure-path tests only: shorten every bounded device wait and make one
    CTA of the cooperative kernels skip its grid-barrier arrivals; (0, -1)
    restores normal operation (see include/qmoe.h)."""
    _check(lib().qmoe_set_fault_injection(wait_limit_ns, skip_arrive_cta))


def device_status(stream=None) -> int:
    """Synchronise the stream and read/clear the device error word."""
    return int(lib().qmoe_device_status(_stream(stream)))
