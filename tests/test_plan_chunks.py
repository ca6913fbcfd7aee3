"""The streaming engine's chunk planner (plan_chunks in
moe_ffn_gb300/csrc/stream.cuh), compiled for the host: for every format,
mode, row shape and stage budget it accepts, its chunks cover every
(k-segment, group) of a row exactly once in order, each chunk's bytes fit the
stage it lands in (with the slack the consumers' loads need), per-row slots
keep the bank spacing the decoders rely on, and QMV chunks of several groups
keep a group on the same consumer warp in every chunk."""
import ctypes
import itertools
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
FORMATS = {"Q8_0": 1, "Q4_0": 2, "Q4_K": 3, "Q5_K": 4, "Q6_K": 5}
MODES = {"QMV": 0, "GATEUP": 1, "DOWN": 2}
# formats read with 128-bit loads, whose rows may sit at their global stride
RUNS_OK = {"Q8_0": False, "Q4_0": False, "Q4_K": True, "Q5_K": True, "Q6_K": True}
# per-row slot stride wanted modulo 128 (None: any odd multiple of 16)
SLOT_REM128 = {"Q8_0": None, "Q4_0": None, "Q4_K": None, "Q5_K": None, "Q6_K": 32}
FIELDS = ("ok", "runs", "n_sbc", "chunk_ks", "chunk_sb", "n_chunk", "piece_stride",
          "slot_stride", "stage_bytes", "seg_bytes", "sbb", "rows", "wk")


@pytest.fixture(scope="module")
def pc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tempfile.mkdtemp(prefix="plan_chunks_")
    so = os.path.join(d, "libplan_chunks.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-o", so,
                    os.path.join(HERE, "host", "plan_chunks.cu")], check=True)
    lib = ctypes.CDLL(so)
    lib.plan_chunks_host.restype = ctypes.c_int
    lib.plan_chunks_host.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p]
    return lib


def plan(pc, fmt, mode, nb_seg, n_kseg, tail, budget, rows):
    out = (ctypes.c_int64 * len(FIELDS))()
    assert pc.plan_chunks_host(FORMATS[fmt], MODES[mode], nb_seg, n_kseg, tail, budget, rows,
                               ctypes.cast(out, ctypes.c_void_p)) == 0
    return dict(zip(FIELDS, (int(v) for v in out)))


def chunks(p, nb_seg, n_kseg):
    """The (k-segment, group) pairs of every chunk, as the engine's chunk
    descriptor numbers them."""
    out = []
    for c in range(p["n_chunk"]):
        if p["n_sbc"] == 1:
            ks0 = c * p["chunk_ks"]
            kss = range(ks0, min(ks0 + p["chunk_ks"], n_kseg))
            bs = range(nb_seg)
        else:
            kss = [c // p["n_sbc"]]
            b0 = (c % p["n_sbc"]) * p["chunk_sb"]
            bs = range(b0, min(b0 + p["chunk_sb"], nb_seg))
        out.append([(k, b) for k in kss for b in bs])
    return out


def cases():
    for fmt, mode in itertools.product(FORMATS, MODES):
        for nb_seg, n_kseg in [(1, 1), (3, 1), (8, 1), (16, 1), (56, 1), (128, 1), (3, 8),
                               (4, 8), (3, 16), (8, 2)]:
            if mode != "DOWN" and n_kseg > 1:
                continue
            for tail in ([0, 3] if fmt in ("Q8_0", "Q4_0") else [0]):
                for budget in (4096, 20480, 49152, 98304):
                    for rows in ([0, 27, 5] if mode == "QMV" else [0]):
                        yield fmt, mode, nb_seg, n_kseg, tail, budget, rows


@pytest.mark.parametrize("fmt", list(FORMATS))
def test_plans_cover_and_fit(pc, fmt):
    n = 0
    for f, mode, nb_seg, n_kseg, tail, budget, rows in cases():
        if f != fmt:
            continue
        p = plan(pc, f, mode, nb_seg, n_kseg, tail, budget, rows)
        r = p["rows"]
        sbb = p["sbb"]
        what = (f, mode, nb_seg, n_kseg, tail, budget, rows, p)
        if not p["ok"]:
            # refused only when not even one group per row fits the budget
            assert budget < r * (sbb + 31), what
            continue
        n += 1
        seg = nb_seg * sbb - ((8 - tail) * (sbb // 8) if tail else 0)
        assert p["seg_bytes"] == seg, what
        # every (k-segment, group) exactly once, in order
        flat = [kb for ch in chunks(p, nb_seg, n_kseg) for kb in ch]
        assert flat == [(k, b) for k in range(n_kseg) for b in range(nb_seg)], what
        assert all(len(ch) > 0 for ch in chunks(p, nb_seg, n_kseg)), what
        if p["runs"]:
            # whole rows at their global stride, one piece per k-segment
            assert p["n_sbc"] == 1 and p["chunk_sb"] == nb_seg, what
            assert RUNS_OK[f] or seg < 2048, what
            assert p["slot_stride"] == seg, what
            assert p["piece_stride"] >= -(-r * seg // 16) * 16 + 144, what
            assert p["stage_bytes"] == p["chunk_ks"] * p["piece_stride"], what
            assert p["stage_bytes"] <= budget, what
        else:
            # per-row slots: each holds its chunk's groups at any 16-byte phase
            nbp_max = nb_seg if p["n_sbc"] == 1 else p["chunk_sb"]
            assert p["piece_stride"] >= nbp_max * sbb + 15, what
            assert p["piece_stride"] % 16 == 0, what
            assert p["slot_stride"] >= p["chunk_ks"] * p["piece_stride"], what
            assert p["stage_bytes"] == r * p["slot_stride"], what
            rem = SLOT_REM128[f]
            if rem is not None:
                assert p["slot_stride"] % 128 == rem, what
            else:
                assert p["slot_stride"] % 32 == 16, what
            if p["n_sbc"] > 1 and p["chunk_sb"] >= p["wk"]:
                # a group stays on warp (group mod WK) in every chunk
                assert p["chunk_sb"] % p["wk"] == 0, what
    assert n > 0


def test_one_tile_qmv_4096_plans(pc):
    """The sweep's 4096-wide GEMVs, 27 rows per CTA: one chunk within about
    half an SM's shared memory beside the x table (93 KB) for every format but
    Q8_0, whose 4352-byte rows take one chunk only within the opt-in maximum
    (about 207 KB beside the x table)."""
    for f in FORMATS:
        half = plan(pc, f, "QMV", 16, 1, 0, 93 * 1024, 27)
        full = plan(pc, f, "QMV", 16, 1, 0, 207 * 1024, 27)
        assert full["ok"] and full["n_chunk"] == 1, (f, full)
        assert half["ok"]
        assert (half["n_chunk"] == 1) == (f != "Q8_0"), (f, half)
