"""Check (c): each compressed entry equals its closed-form gated sum; special cases of the gate."""

import math

import numpy as np
import pytest

from oracle.compress import compress_blocks, compress_prefix, gated_block_sum


def _closed_form(Kb, Vb, g):
    """Closed form written with math.fsum / math.exp, element by element."""
    m, d = Kb.shape
    z = [math.fsum(float(Kb[t, i]) * float(g[i]) for i in range(d)) for t in range(m)]
    zmax = max(z)
    e = [math.exp(zt - zmax) for zt in z]
    s = math.fsum(e)
    w = [et / s for et in e]
    ck = [math.fsum(w[t] * float(Kb[t, i]) for t in range(m)) for i in range(d)]
    cv = [math.fsum(w[t] * float(Vb[t, i]) for t in range(m)) for i in range(d)]
    return np.array(ck), np.array(cv), np.array(w)


@pytest.mark.parametrize("m,d", [(4, 16), (4, 64), (128, 8), (16, 32)])
def test_gated_sum_closed_form(m, d):
    rng = np.random.default_rng(m * 1000 + d)
    Kb = rng.standard_normal((m, d))
    Vb = rng.standard_normal((m, d))
    g = rng.standard_normal(d) * 0.3
    ck, cv = gated_block_sum(Kb, Vb, g)
    rck, rcv, w = _closed_form(Kb, Vb, g)
    assert abs(sum(w) - 1.0) < 1e-14
    np.testing.assert_allclose(ck, rck, rtol=0, atol=1e-13)
    np.testing.assert_allclose(cv, rcv, rtol=0, atol=1e-13)


def test_zero_gate_gives_block_mean():
    rng = np.random.default_rng(5)
    Kb = rng.standard_normal((4, 12))
    Vb = rng.standard_normal((4, 12))
    ck, cv = gated_block_sum(Kb, Vb, np.zeros(12))
    np.testing.assert_allclose(ck, Kb.mean(axis=0), atol=1e-15)
    np.testing.assert_allclose(cv, Vb.mean(axis=0), atol=1e-15)


def test_identical_rows_give_that_row():
    rng = np.random.default_rng(6)
    row_k = rng.standard_normal(10)
    row_v = rng.standard_normal(10)
    ck, cv = gated_block_sum(np.tile(row_k, (128, 1)), np.tile(row_v, (128, 1)), rng.standard_normal(10))
    np.testing.assert_allclose(ck, row_k, atol=1e-14)
    np.testing.assert_allclose(cv, row_v, atol=1e-14)


def test_dominant_logit_selects_that_token():
    rng = np.random.default_rng(7)
    Kb = rng.standard_normal((4, 6)) * 0.01
    Vb = rng.standard_normal((4, 6))
    g = np.zeros(6)
    g[0] = 1.0
    Kb[2, 0] = 2000.0                    # z_2 exceeds every other logit by ~2000
    ck, cv = gated_block_sum(Kb, Vb, g)
    np.testing.assert_array_equal(ck, Kb[2])
    np.testing.assert_array_equal(cv, Vb[2])


def test_permutation_invariance_and_gate_shift():
    rng = np.random.default_rng(8)
    Kb = rng.standard_normal((16, 8))
    Vb = rng.standard_normal((16, 8))
    g = rng.standard_normal(8)
    perm = rng.permutation(16)
    a = gated_block_sum(Kb, Vb, g)
    b = gated_block_sum(Kb[perm], Vb[perm], g)
    np.testing.assert_allclose(a[0], b[0], atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], atol=1e-14)


@pytest.mark.parametrize("m", [4, 128])
def test_vectorised_blocks_equal_per_block_definition(m):
    rng = np.random.default_rng(9 + m)
    L = 3 * m + m // 2 + 1
    d = 8
    rawK = rng.standard_normal((L, d))
    rawV = rng.standard_normal((L, d))
    g = rng.standard_normal(d)
    CK, CV = compress_prefix(rawK, rawV, L, m, g, "f64")
    assert CK.shape == (L // m, d)
    for j in range(L // m):
        ck, cv = gated_block_sum(rawK[m * j:m * j + m], rawV[m * j:m * j + m], g)
        np.testing.assert_allclose(CK[j], ck, atol=1e-14)
        np.testing.assert_allclose(CV[j], cv, atol=1e-14)
    CK2, _ = compress_blocks(rawK, rawV, 1, L // m, m, g, "f64")
    np.testing.assert_allclose(CK2, CK[1:], atol=1e-14)


def test_many_blocks_span_several_slabs():
    # 9000 C4 entries: the compressor widens the raw rows slab by slab (4096 entries per slab);
    # entries at the slab edges, and a range that starts past entry 0, equal the closed form of
    # their own block
    rng = np.random.default_rng(21)
    m, d, n = 4, 4, 9000
    rawK = rng.standard_normal((m * n, d))
    rawV = rng.standard_normal((m * n, d))
    g = rng.standard_normal(d)
    CK, CV = compress_prefix(rawK, rawV, m * n, m, g, "f64")
    for j in (0, 1, 4095, 4096, 4097, 8191, 8192, 8999):
        ck, cv, _ = _closed_form(rawK[m * j:m * j + m], rawV[m * j:m * j + m], g)
        np.testing.assert_allclose(CK[j], ck, rtol=0, atol=1e-12)
        np.testing.assert_allclose(CV[j], cv, rtol=0, atol=1e-12)
    CK2, CV2 = compress_blocks(rawK, rawV, 100, n, m, g, "f64")
    assert np.array_equal(CK2, CK[100:]) and np.array_equal(CV2, CV[100:])
