"""The decoders' lane maps (moe_ffn_gb300/csrc/formats.cuh), compiled for the
host: every lane's 64 elements of a 256-element group form a permutation of
the group, the x-table slot map is its inverse on granules of four, and the
field positions the x table scales for (pos) follow the pattern the table
build assumes: {0, 8, 16, 0} by i % 4, or {0, 8, 16, 0, 4, 12, 20, 0} by i % 8
for the formats that split bytes into low and high nibbles (POS8)."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
FORMATS = {"Q8_0": 1, "Q4_0": 2, "Q4_K": 3, "Q5_K": 4, "Q6_K": 5}


@pytest.fixture(scope="module")
def fm():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tempfile.mkdtemp(prefix="format_maps_")
    so = os.path.join(d, "libformat_maps.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-o", so,
                    os.path.join(HERE, "host", "format_maps.cu")], check=True)
    lib = ctypes.CDLL(so)
    lib.fmt_maps.restype = ctypes.c_int
    lib.fmt_maps.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 4
    return lib


def get(fm, code):
    elem = np.zeros(256, np.int32)
    xslot = np.zeros(64, np.int32)
    pos = np.zeros(256, np.int32)
    pos8 = np.zeros(1, np.int32)
    assert fm.fmt_maps(code, elem.ctypes.data, xslot.ctypes.data, pos.ctypes.data,
                       pos8.ctypes.data) == 0
    return elem.reshape(4, 64), xslot, pos.reshape(4, 64), bool(pos8[0])


@pytest.mark.parametrize("name", list(FORMATS))
def test_lane_order_is_a_permutation(fm, name):
    elem, _, _, _ = get(fm, FORMATS[name])
    assert sorted(elem.ravel().tolist()) == list(range(256))


@pytest.mark.parametrize("name", list(FORMATS))
def test_xslot_inverts_the_lane_order(fm, name):
    elem, xslot, _, _ = get(fm, FORMATS[name])
    assert sorted(xslot.tolist()) == list(range(64))
    for e4 in range(64):
        s = xslot[e4]
        q, i4 = s & 3, s >> 2
        assert [elem[q, 4 * i4 + j] for j in range(4)] == [4 * e4 + j for j in range(4)]


@pytest.mark.parametrize("name", list(FORMATS))
def test_positions_follow_the_table_pattern(fm, name):
    _, _, pos, pos8 = get(fm, FORMATS[name])
    lo, hi = [0, 8, 16, 0], [4, 12, 20, 0]
    for q in range(4):
        for i in range(64):
            want = (hi if pos8 and (i & 4) else lo)[i & 3]
            assert pos[q, i] == want, (q, i)
    # fields fit below bit 24 (linear bit pattern -> value map)
    assert pos.max() <= 20
