"""Pins of the oracle's building blocks: brute force in f64, closed forms,
invariants and special cases (no retyping of the oracle's own expressions)."""
import numpy as np
import pytest

import oracle.core as O

RNG = np.random.default_rng(11)


def test_matvec_exact_on_integer_valued_inputs():
    # integer-valued floats with small magnitudes sum exactly in any order
    W = RNG.integers(-8, 9, size=(37, 53)).astype(np.float32)
    x = RNG.integers(-8, 9, size=53).astype(np.float32)
    y = O.matvec(W, x)
    assert np.array_equal(y, (W.astype(np.int64) @ x.astype(np.int64)).astype(np.float32))


def test_matvec_close_to_f64_and_not_transposed():
    W = RNG.standard_normal((40, 70)).astype(np.float32)
    x = RNG.standard_normal(70).astype(np.float32)
    y = O.matvec(W, x)
    ref = W.astype(np.float64) @ x.astype(np.float64)
    bound = 70 * 2.0**-23 * (np.abs(W) @ np.abs(x))
    assert np.all(np.abs(y - ref) <= bound)


def test_panel_equals_rowwise_matvec_bitwise():
    W = RNG.standard_normal((33, 29)).astype(np.float32)
    X = RNG.standard_normal((5, 29)).astype(np.float32)
    Y = O.matmul_panel(W, X)
    for b in range(5):
        assert np.array_equal(Y[b], O.matvec(W, X[b]))


def test_rmsnorm_closed_forms():
    d, eps = 64, 1e-5
    g = np.ones(d, dtype=np.float32)
    # constant vector c: y = c / sqrt(c^2 + eps)
    for c in (0.5, -3.0, 1e-3):
        y = O.rmsnorm(np.full(d, c, dtype=np.float32), g, eps)
        assert np.allclose(y, c / np.sqrt(c * c + eps), rtol=1e-6)
    # f64 brute force with a non-trivial gain, and mean(y^2) ~ 1 for g = 1
    x = RNG.standard_normal(d).astype(np.float32)
    gg = RNG.uniform(0.5, 2, d).astype(np.float32)
    ref = x / np.sqrt(np.mean(x.astype(np.float64) ** 2) + eps) * gg
    assert np.allclose(O.rmsnorm(x, gg, eps), ref, rtol=3e-6, atol=1e-7)
    assert abs(np.mean(O.rmsnorm(x, g, eps).astype(np.float64) ** 2) - 1) < 1e-4


def _rope_complex(v, hd, pos, theta):
    """Rotate-half RoPE written as complex multiplication, f64."""
    half = hd // 2
    v = v.reshape(-1, hd).astype(np.float64)
    z = v[:, :half] + 1j * v[:, half:]
    ang = pos * theta ** (-2.0 * np.arange(half) / hd)
    z = z * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag], axis=1).reshape(-1)


def test_rope_position_zero_is_identity():
    v = RNG.standard_normal(4 * 16).astype(np.float32)
    assert np.array_equal(O.rope(v, 4, 16, 0, 1e4), v)


@pytest.mark.parametrize("hd,theta", [(16, 1e4), (64, 1e4), (128, 1e6)])
def test_rope_matches_complex_rotation(hd, theta):
    v = RNG.standard_normal(3 * hd).astype(np.float32)
    for pos in (1, 7, 100, 4095):
        got = O.rope(v, 3, hd, pos, theta)
        ref = _rope_complex(v, hd, pos, theta)
        assert np.allclose(got, ref, rtol=0, atol=2e-6 * (1 + pos / 1000))
        # each (i, i+hd/2) pair keeps its length
        a = got.reshape(3, hd)
        b = v.reshape(3, hd)
        h = hd // 2
        n_got = a[:, :h] ** 2 + a[:, h:] ** 2
        n_ref = b[:, :h].astype(np.float64) ** 2 + b[:, h:] ** 2
        assert np.allclose(n_got, n_ref, rtol=1e-5, atol=1e-6)


def test_rope_relative_position_property():
    hd = 64
    q = RNG.standard_normal(hd).astype(np.float32)
    k = RNG.standard_normal(hd).astype(np.float32)
    d1 = np.dot(O.rope(q, 1, hd, 10, 1e4), O.rope(k, 1, hd, 7, 1e4))
    d2 = np.dot(O.rope(q, 1, hd, 103, 1e4), O.rope(k, 1, hd, 100, 1e4))
    assert abs(d1 - d2) < 1e-4


def test_softmax_brute_force_and_invariants():
    s = RNG.standard_normal(50).astype(np.float32) * 3
    p = O.softmax(s)
    e = np.exp(s.astype(np.float64) - s.max())
    assert np.allclose(p, e / e.sum(), rtol=1e-5, atol=1e-8)
    assert abs(p.astype(np.float64).sum() - 1) < 1e-5
    assert np.allclose(O.softmax(s + 100), p, rtol=1e-5, atol=1e-8)
    assert np.all(O.softmax(np.zeros(8, dtype=np.float32)) == np.float32(1 / 8))


def test_attention_special_cases_and_brute_force():
    hd = 16
    q = RNG.standard_normal(hd).astype(np.float32)
    K = RNG.standard_normal((1, hd)).astype(np.float32)
    V = RNG.standard_normal((1, hd)).astype(np.float32)
    # one key: softmax weight is exactly 1, so o == v bit for bit
    assert np.array_equal(O.attend_head(q, K, V), V[0])
    # zero query: uniform weights, o = mean of V
    K = RNG.standard_normal((9, hd)).astype(np.float32)
    V = RNG.standard_normal((9, hd)).astype(np.float32)
    o = O.attend_head(np.zeros(hd, np.float32), K, V)
    assert np.allclose(o, V.astype(np.float64).mean(0), atol=1e-6)
    # brute force f64: softmax(q.K^T / sqrt(hd)) @ V
    s = (K.astype(np.float64) @ q) / np.sqrt(hd)
    w = np.exp(s - s.max())
    w /= w.sum()
    assert np.allclose(O.attend_head(q, K, V), w @ V, atol=2e-6)
    # keys are not transposed with values: swapping rows of K alone changes o
    o2 = O.attend_head(q, K[::-1].copy(), V)
    assert not np.allclose(o2, O.attend_head(q, K, V))


def test_silu_closed_form():
    for z in (-20.0, -1.5, 0.0, 0.3, 4.0, 30.0):
        assert abs(O.silu(z) - z / (1 + np.exp(-z))) <= 1e-6 * max(1, abs(z))
    assert O.silu(0.0) == 0.0


def test_greedy_sampler_lowest_index_on_ties():
    lg = np.array([0.1, 3.0, -1.0, 3.0, 2.9], dtype=np.float32)
    assert O.sample(lg, 0.0) == 1
    assert O.sample(np.zeros(7, np.float32), 0.0) == 0


def test_temperature_sampler_frequencies_chi_square():
    lg = np.array([1.0, 0.0, -1.0, 0.5, 2.0, -3.0], dtype=np.float32)
    T = 0.8
    n = 20000
    counts = np.zeros(lg.size)
    for c in range(n):
        counts[O.sample(lg, T, 99, c)] += 1
    z = lg.astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    chi2 = ((counts - n * p) ** 2 / (n * p)).sum()
    assert chi2 < 25.0  # 5 dof: p(chi2 > 25) ~ 1.4e-4


def test_temperature_sampler_inverse_cdf():
    # the drawn index is the first one whose cumulative mass reaches u
    lg = np.array([0.0, 0.0, 0.0, 0.0], dtype=np.float32)
    for c in range(200):
        u = O.uniform(7, c)
        assert O.sample(lg, 1.0, 7, c) == min(3, int(np.floor(u * 4)))
    # a dominant logit is always drawn; a -inf-like logit never
    lg = np.array([-1e30, 50.0, -1e30], dtype=np.float32)
    assert all(O.sample(lg, 1.0, 3, c) == 1 for c in range(50))
