"""Seeded synthetic inputs for the GEMV / MoE FFN workloads.

Shared by the tests (for both the CUDA path and the CPU oracle) and by
``bench.py``.  This module holds none of the method's arithmetic: it writes
random bytes into the fixed byte positions of each block layout and encodes
random scales as IEEE half floats (numpy's float16 encoder).  Every array is
drawn from ``numpy.random.Generator(PCG64(seed))``.

Distributions (the workload statements):
  * Q8_0: d ~ U(1e-3, 1e-2) as f16, 32 uniform int8 quants.
  * Q4_0: d ~ U(1e-3, 1e-2) as f16, 16 uniform bytes of nibbles.
  * Q4_K / Q5_K: d, dmin ~ U(1e-4, 1e-2) as f16; the 12 scale bytes uniform,
    which makes every packed 6-bit scale and min uniform on 0..63; quants
    (and the Q5_K high-bit plane) uniform bytes.
  * Q6_K: ql, qh uniform bytes; the 16 int8 scales uniform on -128..127;
    d ~ U(1e-4, 1e-2) as f16.
  * F32 router ~ N(0, 0.02); x, residual ~ N(0, 1).
  * Optional NaN row: the f16 scale d of block 0 of the given row is set to
    0x7E00 (a quiet NaN).
"""
from __future__ import annotations

import numpy as np

F32, Q8_0, Q4_0, Q4_K, Q5_K, Q6_K = 0, 1, 2, 3, 4, 5
BLOCK_ELEMS = {F32: 1, Q8_0: 32, Q4_0: 32, Q4_K: 256, Q5_K: 256, Q6_K: 256}
BLOCK_BYTES = {F32: 4, Q8_0: 34, Q4_0: 18, Q4_K: 144, Q5_K: 176, Q6_K: 210}
# byte offset of the f16 scale d inside a block
D_OFFSET = {Q8_0: 0, Q4_0: 0, Q4_K: 0, Q5_K: 0, Q6_K: 208}
NAN_F16 = 0x7E00


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _f16_bytes(vals: np.ndarray) -> np.ndarray:
    """Little-endian bytes of values rounded to IEEE half: shape (..., 2)."""
    h = vals.astype("<f2")
    return h.view(np.uint8).reshape(*vals.shape, 2)


def quant_matrix(g: np.random.Generator, qt: int, rows: int, cols: int,
                 nan_row: int | None = None) -> np.ndarray:
    """[rows][row_bytes] uint8 of random blocks of format qt."""
    be, bb = BLOCK_ELEMS[qt], BLOCK_BYTES[qt]
    assert cols % be == 0
    nb = cols // be
    blk = g.integers(0, 256, size=(rows, nb, bb), dtype=np.uint8)
    if qt in (Q8_0, Q4_0):
        blk[:, :, 0:2] = _f16_bytes(g.uniform(1e-3, 1e-2, size=(rows, nb)))
    elif qt in (Q4_K, Q5_K):
        blk[:, :, 0:2] = _f16_bytes(g.uniform(1e-4, 1e-2, size=(rows, nb)))
        blk[:, :, 2:4] = _f16_bytes(g.uniform(1e-4, 1e-2, size=(rows, nb)))
    elif qt == Q6_K:
        blk[:, :, 208:210] = _f16_bytes(g.uniform(1e-4, 1e-2, size=(rows, nb)))
    else:
        raise ValueError(f"qtype {qt} is not a block format")
    if nan_row is not None:
        o = D_OFFSET[qt]
        blk[nan_row, 0, o] = NAN_F16 & 0xFF
        blk[nan_row, 0, o + 1] = NAN_F16 >> 8
    return blk.reshape(rows, nb * bb)


def expert_stack(g: np.random.Generator, qt: int, n_experts: int, rows: int,
                 cols: int) -> np.ndarray:
    """[E][rows][row_bytes] — one allocation of n_experts [rows][cols] matrices."""
    m = quant_matrix(g, qt, n_experts * rows, cols)
    return m.reshape(n_experts, rows, -1)


def norm_weight(g: np.random.Generator, n: int) -> np.ndarray:
    """An ffn_norm weight vector: 1 + N(0, 0.1^2) per element, f32."""
    return (1.0 + 0.1 * g.standard_normal(n)).astype(np.float32)


def normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(size=shape) * std).astype(np.float32)


# ---------------------------------------------------------------- workloads
# Sizes of the five workloads; the value distributions are those of the
# generators above.
GEMV_SMALL = dict(qtype=Q4_0, rows=256, cols=1024)                       # single Q4_0 matvec
GEMV_SWEEP = dict(qtypes=(Q8_0, Q4_0, Q4_K, Q5_K, Q6_K), rows=4096, cols=4096, nan_row=1)
DENSE_FFN = dict(hidden=4096, inter=14336, gate=Q4_K, up=Q4_K, down=Q6_K)
MOE_DECODE = dict(hidden=2048, expert_dim=768, num_experts=128, top_k=8, n_tokens=1,
                  gate=Q4_K, up=Q4_K, down=Q6_K)
MOE_PREFILL = dict(hidden=2048, expert_dim=1024, num_experts=64, top_k=8, n_tokens=512,
                   gate=Q4_K, up=Q4_K, down=Q6_K)


def moe_inputs(seed: int, hidden, expert_dim, num_experts, top_k, n_tokens, gate, up, down,
               **_):
    """Router, stacks, x and residual of one MoE layer."""
    g = rng(seed)
    return dict(
        router=normal(g, (num_experts, hidden), 0.02),
        gate=expert_stack(g, gate, num_experts, expert_dim, hidden),
        up=expert_stack(g, up, num_experts, expert_dim, hidden),
        down=expert_stack(g, down, num_experts, hidden, expert_dim),
        x=normal(g, (n_tokens, hidden)),
        residual=normal(g, (n_tokens, hidden)),
    )


def ffn_inputs(seed: int, hidden, inter, gate, up, down, **_):
    g = rng(seed)
    return dict(
        gate=quant_matrix(g, gate, inter, hidden),
        up=quant_matrix(g, up, inter, hidden),
        down=quant_matrix(g, down, hidden, inter),
        x=normal(g, hidden),
        residual=normal(g, hidden),
    )
