"""The on-device routing rule, compiled for the host (tests/host/route_host.cpp
includes the kernels' own moe_ffn_gb300/csrc/route.cuh), against the oracle's
route on finite, tied and non-finite logits.

The rule ("softmax, top-k, renormalize" of "aprender-serve 0.70.2 —
forward_qwen3_moe_resident.rs", moe_layer): experts ranked on a total order
(NaN > +Inf > finite > -Inf, -0 as +0, ties to the lower index), so the ranks
are always a permutation and every slot is written; when the top logit is not
finite every softmax probability is NaN and the route is experts 0..k-1 with
NaN weights — the order the oracle's stable sort leaves NaN probabilities in.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def rt():
    d = tempfile.mkdtemp(prefix="route_host_")
    so = os.path.join(d, "libroute_host.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-o", so,
                    os.path.join(HERE, "host", "route_host.cpp")], check=True)
    lib = ctypes.CDLL(so)
    P = ctypes.c_void_p
    lib.route_host.restype = ctypes.c_int
    lib.route_host.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P]
    lib.route_key_host.restype = ctypes.c_uint32
    lib.route_key_host.argtypes = [ctypes.c_float]
    lib.route_key_value_host.restype = ctypes.c_float
    lib.route_key_value_host.argtypes = [ctypes.c_uint32]
    return lib


def host_route(rt, logits, k, renorm=True):
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    E = lg.size
    idx = np.zeros(k, np.int32)
    w = np.zeros(k, np.float32)
    ranks = np.zeros(E, np.int32)
    rc = rt.route_host(lg.ctypes.data, E, k, 1 if renorm else 0, idx.ctypes.data, w.ctypes.data,
                       ranks.ctypes.data)
    assert rc == 0, "a clamp fired"
    return idx, w, ranks


SPECIAL = [np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1e-45, -1e-45]


def test_key_order_is_total(rt):
    vals = np.array(SPECIAL + list(np.linspace(-5, 5, 11)), dtype=np.float32)
    keys = np.array([rt.route_key_host(float(v)) for v in vals], dtype=np.uint64)
    assert np.all(keys != 0)  # 0 marks a taken expert in the batched kernel
    for a, ka in zip(vals, keys):
        for b, kb in zip(vals, keys):
            if np.isnan(a) or np.isnan(b):
                if np.isnan(a) and np.isnan(b):
                    assert ka == kb
                else:
                    assert (ka > kb) == bool(np.isnan(a))  # NaN ranks above everything
            else:
                assert (ka > kb) == bool(a > b) and (ka == kb) == bool(a == b), (a, b)


def test_key_value_round_trip(rt):
    for v in SPECIAL + [2.5, -7.25, 1e30]:
        back = rt.route_key_value_host(rt.route_key_host(v))
        if np.isnan(v):
            assert np.isnan(back)
        else:
            assert back == np.float32(v)  # -0 comes back as +0, which compares equal


@pytest.mark.parametrize("seed", range(40))
def test_ranks_are_a_permutation_whatever_the_logits(rt, seed):
    g = np.random.default_rng(seed)
    E = int(g.integers(1, 257))
    k = int(g.integers(1, min(E, 16) + 1))
    lg = g.standard_normal(E).astype(np.float32)
    sel = g.random(E) < 0.5  # about half the experts get NaN, +-Inf, +-0, ties, extremes
    lg[sel] = g.choice(np.array(SPECIAL + [0.5, 0.5, 2.0], np.float32), size=int(sel.sum()))
    idx, w, ranks = host_route(rt, lg, k)
    assert sorted(ranks.tolist()) == list(range(E))
    assert len(set(idx.tolist())) == k and np.all((idx >= 0) & (idx < E))


def _oracle_route(orc, lg, k, renorm=True):
    return orc.route(np.asarray(lg, np.float64), k, renormalize=renorm)


@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("case", [
    "finite", "ties", "neg_inf_some", "signed_zero"])
def test_finite_top_matches_oracle(rt, orc, case, renorm):
    g = np.random.default_rng(len(case) * 31 + (7 if renorm else 3))
    E, k = 64, 8
    lg = g.standard_normal(E).astype(np.float32)
    if case == "ties":
        lg = np.round(lg * 2).astype(np.float32) / 2  # many equal logits
    elif case == "neg_inf_some":
        lg[g.choice(E, 60, replace=False)] = -np.inf  # k reaches into the -Inf experts
    elif case == "signed_zero":
        lg[:] = 0.0
        lg[::2] = -0.0
        lg[5] = 1.0
    idx, w, _ = host_route(rt, lg, k, renorm)
    ri, rw = _oracle_route(orc, lg, k, renorm)
    assert idx.tolist() == list(ri)
    np.testing.assert_allclose(w, rw, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("case", ["nan_one", "nan_all", "pos_inf", "pos_inf_and_nan",
                                  "neg_inf_all"])
def test_non_finite_top_is_index_order_nan_weights(rt, orc, case, renorm):
    g = np.random.default_rng(7)
    E, k = 48, 5
    lg = g.standard_normal(E).astype(np.float32)
    if case == "nan_one":
        lg[17] = np.nan
    elif case == "nan_all":
        lg[:] = np.nan
    elif case == "pos_inf":
        lg[30] = np.inf
    elif case == "pos_inf_and_nan":
        lg[3], lg[40] = np.inf, np.nan
    elif case == "neg_inf_all":
        lg[:] = -np.inf
    idx, w, _ = host_route(rt, lg, k, renorm)
    ri, rw = _oracle_route(orc, lg, k, renorm)
    assert list(ri) == list(range(k)) and np.all(np.isnan(rw))  # the oracle's reading
    assert idx.tolist() == list(range(k))
    assert np.all(np.isnan(w))
