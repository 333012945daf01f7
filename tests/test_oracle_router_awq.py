"""Pins for the oracle's router-logits product and AWQ checkpoint import,
against what the definitions fix: exact rational arithmetic on tiny inputs,
one-hot inputs, the library matrix product, hand-derived packed words, and
invariants of the repack."""
from fractions import Fraction

import numpy as np
import pytest

import oracle

# ---------------------------------------------------------------- router logits


def _half(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def test_router_logits_exact_on_tiny_input(m=oracle):
    """T=2, E=3, H=5: every logit against the exact rational sum of the
    fp16 products (fp16 values are dyadic rationals)."""
    rng = np.random.default_rng(5)
    x, wr = _half(rng, (2, 5)), _half(rng, (3, 5))
    got = m.router_logits(x, wr)
    for t in range(2):
        for e in range(3):
            exact = sum(Fraction(float(x[t, c])) * Fraction(float(wr[e, c])) for c in range(5))
            assert abs(got[t, e] - float(exact)) <= 1e-15 * max(1.0, abs(float(exact)))


def test_router_logits_one_hot_picks_a_column(m=oracle):
    """x[t] = unit vector at h_t: logits[t][e] = wr[e][h_t] exactly."""
    rng = np.random.default_rng(6)
    T, E, H = 4, 7, 96
    wr = _half(rng, (E, H))
    hs = [0, 17, 95, 40]
    x = np.zeros((T, H), np.float16)
    for t, h in enumerate(hs):
        x[t, h] = 1.0
    got = m.router_logits(x, wr)
    for t, h in enumerate(hs):
        assert np.array_equal(got[t], wr[:, h].astype(np.float64))


def test_router_logits_match_library_product(m=oracle):
    """Non-square shapes (E != H, T != E): the library float64 product of
    the fp16 values, within a few units of rounding of the sum of |terms|."""
    rng = np.random.default_rng(7)
    T, E, H = 5, 24, 160
    x, wr = _half(rng, (T, H)), _half(rng, (E, H), 1 / np.sqrt(H))
    got = m.router_logits(x, wr)
    ref = x.astype(np.float64) @ wr.astype(np.float64).T
    bound = 1e-13 * (np.abs(x.astype(np.float64)) @ np.abs(wr.astype(np.float64)).T)
    assert got.shape == (T, E)
    assert np.all(np.abs(got - ref) <= bound)


def test_router_logits_rejects_transposed_matrix(m=oracle):
    with pytest.raises(ValueError):
        m.router_logits(np.zeros((2, 8), np.float16), np.zeros((8, 3), np.float16))


# ---------------------------------------------------------------- AWQ import
# AWQ layer: qweight u32 [E][K][N/8], qzeros u32 [E][K/32][N/8], scales f16 [E][K/32][N]


def _awq_zero(E, K, N):
    return (np.zeros((E, K, N // 8), np.uint32), np.zeros((E, K // 32, N // 8), np.uint32),
            np.zeros((E, K // 32, N), np.float16))


def _dst(E, Ndst, K):
    return (np.zeros((E, Ndst, K // 8), np.uint32), np.zeros((E, Ndst, K // 32), np.float16),
            np.zeros((E, Ndst // 8, K // 32), np.uint32))


def test_awq_order_word_gives_column_index(m=oracle):
    """Every AWQ qweight word = 0x75316420 (hand-derived: nibble i holds the
    column ORDER[i] = 0,2,4,6,1,3,5,7 of its group of eight, so the value
    stored for column 8c + j is j): after import every code of row n is
    n % 8, i.e. every word of row n is (n % 8) * 0x11111111."""
    E, K, N = 2, 64, 32
    awq = _awq_zero(E, K, N)
    awq[0][:] = 0x75316420
    q, _, _ = m.awq_import(awq, _dst(E, N, K))
    for n in range(N):
        assert np.all(q[:, n, :] == (n % 8) * 0x11111111)


def test_awq_single_nibbles_land_where_derived(m=oracle):
    """Hand-derived single elements:
    qweight[0][kk=3][c=0] = 0x50 (nibble 1 -> column 2)  -> q(2, 3) = 5,
        layer word [0][2][0] = 5 << 12 = 0x5000;
    qweight[1][kk=9][c=1] = 0x30000000 (nibble 7 -> column 15)
        -> layer word [1][15][1] = 3 << 4 = 0x30;
    qzeros[0][g=1][c=0] = 0x700 (nibble 2 -> column 4)
        -> layer zero word [0][0][1] = 7 << 16 = 0x70000;
    every other word stays zero."""
    E, K, N = 2, 64, 16
    awq = _awq_zero(E, K, N)
    awq[0][0, 3, 0] = 0x50
    awq[0][1, 9, 1] = 0x30000000
    awq[1][0, 1, 0] = 0x700
    q, _, z = m.awq_import(awq, _dst(E, N, K))
    expect_q = np.zeros_like(q)
    expect_q[0, 2, 0] = 0x5000
    expect_q[1, 15, 1] = 0x30
    expect_z = np.zeros_like(z)
    expect_z[0, 0, 1] = 0x70000
    assert np.array_equal(q, expect_q)
    assert np.array_equal(z, expect_z)


def test_awq_scales_are_transposed(m=oracle):
    E, K, N = 2, 96, 24
    awq = _awq_zero(E, K, N)
    vals = np.arange(E * (K // 32) * N, dtype=np.float16).reshape(E, K // 32, N)
    awq = (awq[0], awq[1], vals)
    _, s, _ = m.awq_import(awq, _dst(E, N, K))
    assert np.array_equal(s, np.transpose(vals, (0, 2, 1)))


def test_awq_import_preserves_every_dequantised_weight(m=oracle):
    """Random AWQ layer: the layer's dequant of the imported matrices equals
    (q - z) * s read from the AWQ layer, element by element."""
    rng = np.random.default_rng(9)
    E, K, N = 2, 64, 24
    awq = (rng.integers(0, 1 << 32, (E, K, N // 8), dtype=np.uint32),
           rng.integers(0, 1 << 32, (E, K // 32, N // 8), dtype=np.uint32),
           (0.002 + 0.018 * rng.random((E, K // 32, N))).astype(np.float16))
    q, s, z = m.awq_import(awq, _dst(E, N, K))
    for e in range(E):
        for n in range(N):
            for kk in range(K):
                aq, az, asb = m.awq_element(awq, K, N, e, n, kk)
                expect = (aq - az) * m.half_to_double(asb)
                assert m.dequant(q, s, z, N, K, e, n, kk) == expect


def test_awq_import_into_upper_half_leaves_lower_half(m=oracle):
    """Importing an up layer into rows [I, 2I) of W13 changes only those
    rows: gate rows, their scales and their zero nibbles keep the values
    written before; the gate-then-up import equals importing a layer whose
    columns are the two side by side."""
    rng = np.random.default_rng(10)
    E, K, I = 2, 64, 16

    def layer(n):
        return (rng.integers(0, 1 << 32, (E, K, n // 8), dtype=np.uint32),
                rng.integers(0, 1 << 32, (E, K // 32, n // 8), dtype=np.uint32),
                (0.002 + 0.018 * rng.random((E, K // 32, n))).astype(np.float16))
    gate, up = layer(I), layer(I)
    dst = _dst(E, 2 * I, K)
    m.awq_import(gate, dst, row0=0)
    before = tuple(a.copy() for a in dst)
    m.awq_import(up, dst, row0=I)
    assert np.array_equal(dst[0][:, :I], before[0][:, :I])
    assert np.array_equal(dst[1][:, :I], before[1][:, :I])
    assert np.array_equal(dst[2][:, :I // 8], before[2][:, :I // 8])
    both = tuple(np.concatenate([g, u], axis=2) for g, u in zip(gate, up))
    ref = m.awq_import(both, _dst(E, 2 * I, K))
    for a, b in zip(dst, ref):
        assert np.array_equal(a, b)


def test_awq_import_rejects_misplaced_rows(m=oracle):
    awq = _awq_zero(1, 32, 8)
    with pytest.raises(ValueError):
        m.awq_import(awq, _dst(1, 16, 32), row0=4)
    with pytest.raises(ValueError):
        m.awq_import(awq, _dst(1, 8, 32), row0=8)
