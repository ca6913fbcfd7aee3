"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Each test states what it pins.  None compares the oracle with a retyped copy
of its own formula: expected values are exact closed forms of hand-built
blocks (small integers, powers of two), one-hot probes of element positions,
exhaustive enumerations, invariants, or special cases that reduce to a
library routine (numpy / scipy).
"""
import itertools
import math

import numpy as np
import pytest

from tests import blocks as B

# --------------------------------------------------------------- f16 decode
def test_f16_exhaustive(orc):
    """All 65,536 half bit patterns decode as numpy's IEEE half -> single
    conversion (NaN class equality, signed zeros, subnormals)."""
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view("<f2").astype(np.float32)
    got = np.array([orc.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


# ------------------------------------------------------- 6-bit scale / min
def test_k_scale_min_exhaustive(orc):
    """For every pair j and every (sc, m) in 0..63 x 0..63, unpacking the
    packed bytes returns (sc, m); the other pairs stay intact."""
    rng = np.random.default_rng(1)
    for j in range(8):
        for sc in range(64):
            for m in range(64):
                scs = list(rng.integers(0, 64, 8))
                ms = list(rng.integers(0, 64, 8))
                scs[j], ms[j] = sc, m
                s = np.frombuffer(B.pack_k_scales(scs, ms), dtype=np.uint8)
                assert orc.k_scale_min(j, s) == (sc, m)
                if sc == 0 and m in (0, 63):
                    for jj in range(8):
                        assert orc.k_scale_min(jj, s) == (scs[jj], ms[jj])


def test_k_scale_min_bit_positions(orc):
    """The unpacking reads the bit positions of ferrox_q4_k_scale_min: for
    j < 4 the low 6 bits of bytes j and j+4; for j >= 4 the low / high
    nibble of byte j+4 joined with the top two bits of bytes j-4 / j."""
    for j in range(8):
        s = np.zeros(12, np.uint8)
        if j < 4:
            s[j], s[j + 4] = 0x3F, 0x15
            assert orc.k_scale_min(j, s) == (63, 21)
            s[j], s[j + 4] = 0xC0, 0xC0  # top bits belong to pair j+4
            assert orc.k_scale_min(j, s) == (0, 0)
        else:
            s[j + 4] = 0xA5            # sc low nibble 5, m low nibble 10
            s[j - 4] = 0x80            # sc high bits 10b
            s[j] = 0x40                # m high bits 01b
            assert orc.k_scale_min(j, s) == (5 | (2 << 4), 10 | (1 << 4))


# ------------------------------------------------------------------- Q4_0
def test_q4_0_all_eights_decode_to_zero(orc):
    blk = B.q4_0(B.f16_bits(0.01), [8] * 32)
    assert np.all(orc.decode_block(orc.Q4_0, np.frombuffer(blk, np.uint8)) == 0.0)


def test_q4_0_byte_0x91(orc):
    """d = 1, byte i = 0x91: element i = 1-8 = -7, element i+16 = 9-8 = +1."""
    for i in range(16):
        nib = [8] * 32
        nib[i], nib[i + 16] = 1, 9
        out = orc.decode_block(orc.Q4_0, np.frombuffer(B.q4_0(B.f16_bits(1.0), nib), np.uint8))
        want = np.zeros(32, np.float32)
        want[i], want[i + 16] = -7.0, 1.0
        assert np.array_equal(out, want)
        raw = bytearray(B.q4_0(B.f16_bits(1.0), [8] * 32))
        raw[2 + i] = 0x91
        assert np.array_equal(orc.decode_block(orc.Q4_0, np.frombuffer(bytes(raw), np.uint8)), want)


def test_q4_0_scale_exact(orc):
    """value = (nibble - 8) * d exactly for d = 2^-3 and every nibble."""
    nib = list(range(16)) + list(range(15, -1, -1))
    out = orc.decode_block(orc.Q4_0, np.frombuffer(B.q4_0(B.f16_bits(0.125), nib), np.uint8))
    assert np.array_equal(out, (np.array(nib, np.float32) - 8) * np.float32(0.125))


# ------------------------------------------------------------------- Q8_0
def test_q8_0_integers_and_signs(orc):
    q = [(-128 + 9 * i) % 256 - 128 if i % 2 else (5 * i) % 128 - 64 for i in range(32)]
    q[0], q[1] = -128, 127
    out = orc.decode_block(orc.Q8_0, np.frombuffer(B.q8_0(B.f16_bits(1.0), q), np.uint8))
    assert np.array_equal(out, np.array(q, np.float32))
    out4 = orc.decode_block(orc.Q8_0, np.frombuffer(B.q8_0(B.f16_bits(4.0), q), np.uint8))
    assert np.array_equal(out4, 4 * np.array(q, np.float32))


def test_q8_0_matvec_reduces_to_integer_matmul(orc):
    """d = 1: the GEMV of a Q8_0 matrix is the integer matrix times x
    (numpy's matmul in float64)."""
    rng = np.random.default_rng(2)
    rows, cols = 7, 96
    Q = rng.integers(-128, 128, size=(rows, cols))
    W = b"".join(B.q8_0(B.f16_bits(1.0), Q[r, 32 * k:32 * k + 32])
                 for r in range(rows) for k in range(cols // 32))
    x = rng.standard_normal(cols).astype(np.float32)
    y = orc.matvec(orc.Q8_0, np.frombuffer(W, np.uint8), rows, cols, x)
    assert np.allclose(y, Q.astype(np.float64) @ x.astype(np.float64), rtol=0, atol=1e-9)


# ------------------------------------------------------------------- Q4_K
def _onehot_positions(orc, qt, block, n=256):
    """w_e of one block via one-hot x (the dot with e_i picks w_i)."""
    blk = np.frombuffer(block, np.uint8)
    out = np.zeros(n)
    for i in range(n):
        x = np.zeros(n, np.float32)
        x[i] = 1.0
        out[i] = orc.matvec(qt, blk, 1, n, x)[0]
    return out


def test_q4_k_nibble_positions(orc):
    """d = 1, dmin = 0, every scale 1: byte 32oi+l of qs with low nibble 3
    gives element 64oi+l = 3; high nibble 5 gives element 64oi+32+l = 5."""
    for oi, l in [(0, 0), (1, 7), (2, 31), (3, 16)]:
        raw = bytearray(B.q4_k(B.f16_bits(1.0), 0, [1] * 8, [0] * 8, [0] * 256))
        raw[16 + 32 * oi + l] = 0x53
        w = _onehot_positions(orc, orc.Q4_K, bytes(raw))
        want = np.zeros(256)
        want[64 * oi + l], want[64 * oi + 32 + l] = 3.0, 5.0
        assert np.array_equal(w, want)


def test_q4_k_scale_and_min_closed_form(orc):
    """value = (d*sc)*q - dmin*m with d = 1, dmin = 1/2: exact integers and
    halves; sub-block j = 2oi (low nibbles) / 2oi+1 (high nibbles)."""
    sc = [1, 2, 3, 5, 7, 11, 13, 63]
    m = [0, 1, 2, 4, 8, 16, 32, 63]
    q = [(7 * e + 3) % 16 for e in range(256)]
    out = orc.decode_block(orc.Q4_K, np.frombuffer(
        B.q4_k(B.f16_bits(1.0), B.f16_bits(0.5), sc, m, q), np.uint8))
    for e in range(256):
        j = 2 * (e // 64) + ((e % 64) >= 32)
        assert out[e] == sc[j] * q[e] - 0.5 * m[j], e


def test_q4_k_zero_scale_gives_constant_min(orc):
    out = orc.decode_block(orc.Q4_K, np.frombuffer(
        B.q4_k(B.f16_bits(0.25), B.f16_bits(2.0), [0] * 8, [3] * 8, list(range(16)) * 16),
        np.uint8))
    assert np.all(out == -6.0)


# ------------------------------------------------------------------- Q5_K
def test_q5_k_high_bit_planes(orc):
    """qh[l] bit 2oi adds 16 to element 64oi+l; bit 2oi+1 adds 16 to element
    64oi+32+l (d = 1, dmin = 0, scales 1, all nibbles 0)."""
    for oi in range(4):
        for l in (0, 13, 31):
            for hi in (0, 1):
                raw = bytearray(B.q5_k(B.f16_bits(1.0), 0, [1] * 8, [0] * 8, [0] * 256))
                raw[16 + l] = 1 << (2 * oi + hi)
                out = orc.decode_block(orc.Q5_K, np.frombuffer(bytes(raw), np.uint8))
                want = np.zeros(256, np.float32)
                want[64 * oi + 32 * hi + l] = 16.0
                assert np.array_equal(out, want)


def test_q5_k_closed_form(orc):
    sc = [3, 1, 4, 1, 5, 9, 2, 6]
    m = [2, 7, 1, 8, 2, 8, 1, 8]
    q = [(11 * e + 5) % 32 for e in range(256)]
    out = orc.decode_block(orc.Q5_K, np.frombuffer(
        B.q5_k(B.f16_bits(2.0), B.f16_bits(0.25), sc, m, q), np.uint8))
    for e in range(256):
        j = 2 * (e // 64) + ((e % 64) >= 32)
        assert out[e] == 2.0 * sc[j] * q[e] - 0.25 * m[j], e


# ------------------------------------------------------------------- Q6_K
def test_q6_k_signed_scales(orc):
    """The 16 scales are signed int8 (the page's signed-scale fix): with
    d = 1 and stored value v, element weight = sc * (v - 32)."""
    v = [(5 * e + 1) % 64 for e in range(256)]
    scales = [1, -1, 2, -2, 127, -128, 3, -3, 5, -5, 7, -7, 11, -11, 13, -13]
    out = orc.decode_block(orc.Q6_K, np.frombuffer(B.q6_k(B.f16_bits(1.0), scales, v), np.uint8))
    for e in range(256):
        h, t = divmod(e, 128)
        l = t % 32
        quarter = t // 32
        s = scales[8 * h + l // 16 + 2 * quarter]
        assert out[e] == s * (v[e] - 32), e


def test_q6_k_value_32_is_zero(orc):
    out = orc.decode_block(orc.Q6_K, np.frombuffer(
        B.q6_k(B.f16_bits(3.0), [-7] * 16, [32] * 256), np.uint8))
    assert np.all(out == 0.0)


def test_q6_k_bit_planes_by_bytes(orc):
    """Raw byte probes: ql[64h+l] low nibble -> element 128h+l, high nibble ->
    128h+l+64; ql[64h+32+l] -> 128h+l+32 / +96; qh[32h+l] bits 2t..2t+1 are
    the top bits of element 128h+l+32t.  Scales all +1, d = 1."""
    base = bytearray(B.q6_k(B.f16_bits(1.0), [1] * 16, [32] * 256))
    for h in (0, 1):
        for l in (0, 9, 31):
            for which, elem in ((0, 0), (1, 64)):
                raw = bytearray(base)
                # v = 32 is 10_0000b: low nibble 0, top bits 10b.  Setting the
                # probed element's low nibble to 1 makes v = 33, weight +1.
                raw[64 * h + l] = 0x01 if which == 0 else 0x10
                out = orc.decode_block(orc.Q6_K, np.frombuffer(bytes(raw), np.uint8))
                want = np.zeros(256, np.float32)
                want[128 * h + l + elem] = 1.0
                assert np.array_equal(out, want), (h, l, which)
            for t in range(4):
                raw = bytearray(base)
                cur = raw[128 + 32 * h + l]
                # top bits of element +32t from 10b (v=32) to 11b (v=48): +16
                raw[128 + 32 * h + l] = cur | (1 << (2 * t))
                out = orc.decode_block(orc.Q6_K, np.frombuffer(bytes(raw), np.uint8))
                want = np.zeros(256, np.float32)
                want[128 * h + l + 32 * t] = 16.0
                assert np.array_equal(out, want), (h, l, t)


# ---------------------------------------------- fused vs decode-then-dot
@pytest.mark.parametrize("qt", [1, 2, 3, 4, 5])
def test_fused_equals_decode_then_dot(orc, qt):
    """Decoding inside the dot loop (the page kernels' structure) and
    decoding a row first give bit-identical double sums."""
    from moe_ffn_gb300 import synth
    g = synth.rng(10 + qt)
    rows, cols = 9, 768
    W = synth.quant_matrix(g, qt, rows, cols, nan_row=3)
    x = synth.normal(g, cols)
    a = orc.matvec(qt, W, rows, cols, x)
    b = orc.matvec_fused(qt, W, rows, cols, x)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    assert np.isnan(a[3])
    ok = ~np.isnan(a)
    assert np.array_equal(a[ok], b[ok])


@pytest.mark.parametrize("qt", [1, 2, 3, 4, 5])
def test_linearity_in_x(orc, qt):
    from moe_ffn_gb300 import synth
    g = synth.rng(20 + qt)
    rows, cols = 5, 512
    W = synth.quant_matrix(g, qt, rows, cols)
    x1, x2 = synth.normal(g, cols), synth.normal(g, cols)
    al, be = 0.75, -2.5  # exact in f32: alpha*x1 + beta*x2 is formed in double below
    y1, s1 = orc.matvec(qt, W, rows, cols, x1, with_sabs=True)
    y2, s2 = orc.matvec(qt, W, rows, cols, x2, with_sabs=True)
    dense = orc.dequant(qt, W, rows, cols).astype(np.float64)
    x3 = al * x1.astype(np.float64) + be * x2.astype(np.float64)
    assert np.allclose(dense @ x3, al * y1 + be * y2, rtol=0,
                       atol=1e-12 * float(np.max(abs(al) * s1 + abs(be) * s2)))


def test_row_bytes(orc):
    assert orc.row_bytes(orc.Q4_K, 4096) == 16 * 144
    assert orc.row_bytes(orc.Q6_K, 768) == 630
    assert orc.row_bytes(orc.Q8_0, 64) == 68
    assert orc.row_bytes(orc.Q4_0, 48) == -1


# ---------------------------------------------------------------- routing
def test_route_k_equals_e_is_softmax(orc):
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    lg = rng.standard_normal(16) * 3
    idx, w = orc.route(lg, 16)
    p = softmax(lg)
    assert np.allclose(w, p[idx], rtol=1e-13, atol=0)
    assert list(idx) == list(np.argsort(-p, kind="stable"))


def test_route_topk_matches_sort_and_renormalises(orc):
    from scipy.special import softmax
    rng = np.random.default_rng(4)
    for E, k in [(128, 8), (64, 8), (8, 1), (5, 3), (256, 16)]:
        lg = rng.standard_normal(E)
        idx, w = orc.route(lg, k)
        p = softmax(lg)
        order = np.argsort(-p, kind="stable")[:k]
        assert list(idx) == list(order)
        assert abs(w.sum() - 1.0) < 1e-12
        assert np.all(np.diff(w) <= 0)
        assert np.allclose(w, p[order] / p[order].sum(), rtol=1e-13)
    idx, w = orc.route(rng.standard_normal(9), 1)
    assert w[0] == 1.0


def test_route_ties_prefer_lower_index(orc):
    lg = np.array([0.5, 2.0, 2.0, -1.0, 2.0, 0.5])
    idx, w = orc.route(lg, 4)
    assert list(idx) == [1, 2, 4, 0]
    assert np.allclose(w[:3], w[0])


def test_route_brute_force_small(orc):
    """The selected set maximises the sum of probabilities over all k-subsets."""
    rng = np.random.default_rng(5)
    E, k = 7, 3
    lg = rng.standard_normal(E)
    idx, _ = orc.route(lg, k)
    p = np.exp(lg - lg.max())
    best = max(itertools.combinations(range(E), k), key=lambda c: sum(p[list(c)]))
    assert sorted(idx) == sorted(best)


def test_route_without_renormalisation_is_softmax_restricted(orc):
    """renormalize=False: the same experts, weighted by their softmax
    probability over all E experts (scipy), so the weights sum to the mass of
    the top k; k = E sums to 1; two experts, top-1: the logistic function of
    the logit difference."""
    from scipy.special import expit, softmax
    rng = np.random.default_rng(6)
    for E, k in [(128, 8), (64, 8), (8, 1), (5, 3), (256, 16)]:
        lg = rng.standard_normal(E) * 2
        idx, w = orc.route(lg, k, renormalize=False)
        idx_r, w_r = orc.route(lg, k)
        p = softmax(lg)
        order = np.argsort(-p, kind="stable")[:k]
        assert list(idx) == list(order) == list(idx_r)
        assert np.allclose(w, p[order], rtol=1e-13, atol=0)
        assert abs(w.sum() - p[order].sum()) < 1e-13
        assert w.sum() < 1.0 or k == E
    lg = rng.standard_normal(12)
    _, w = orc.route(lg, 12, renormalize=False)
    assert abs(w.sum() - 1.0) < 1e-13
    for a, b in [(0.3, -1.2), (2.0, 1.5), (-4.0, 3.0)]:
        idx, w = orc.route(np.array([a, b]), 1, renormalize=False)
        assert idx[0] == (0 if a >= b else 1)
        assert abs(w[0] - expit(abs(a - b))) < 1e-15
    # equal logits: 1/E each (1/k with renormalisation)
    _, w = orc.route(np.zeros(10), 4, renormalize=False)
    assert np.allclose(w, 0.1, rtol=1e-15)


def test_route_rejects_bad_shape(orc):
    with pytest.raises(ValueError):
        orc.route(np.zeros(4), 5)
    with pytest.raises(ValueError):
        orc.route(np.zeros(4), 0)
