"""Pins of the oracle's pre-RoPE key path (KVQuant notes, mechanism two: keys are
cached before the rotary position embedding and rotated when attended).

Each check ties the oracle to something outside its own formula: the textbook 2-D
rotation, the complex-number form of RoPE with the page's printed theta_i (1-based
index), the relative-position property that motivates RoPE, norm preservation, the
group law of rotations, and attention over an unquantized cache computed here with
numpy.
"""
import numpy as np
import pytest

import oracle
from oracle import OracleCache


def test_two_dims_is_the_textbook_rotation():
    # D = 2: theta_1 = base^0 = 1, so position t turns (1, 0) by t radians
    t = np.arange(0, 50)
    K = np.tile([[1.0, 0.0]], (len(t), 1))
    out = oracle.rope(K, base=10000.0, t0=0)
    assert np.allclose(out[:, 0], np.cos(t), atol=1e-14)
    assert np.allclose(out[:, 1], np.sin(t), atol=1e-14)


@pytest.mark.parametrize("D,base", [(128, 10000.0), (64, 500000.0), (8, 10.0)])
def test_complex_form_with_printed_theta(D, base):
    """Pair (x_{2i-1}, x_{2i}) (1-based) is the complex number x_{2i-1} + i x_{2i},
    multiplied by exp(i m theta_i), theta_i = base^(-2(i-1)/d)."""
    rng = np.random.default_rng(1)
    L, t0 = 40, 1000
    K = rng.standard_normal((L, D))
    idx = np.arange(1, D // 2 + 1)                      # 1-based i of the page
    theta = base ** (-2.0 * (idx - 1) / D)
    m = (t0 + np.arange(L))[:, None]
    z = (K[:, 0::2] + 1j * K[:, 1::2]) * np.exp(1j * m * theta[None, :])
    want = np.empty_like(K)
    want[:, 0::2], want[:, 1::2] = z.real, z.imag
    assert np.allclose(oracle.rope(K, base, t0), want, atol=1e-12)


def test_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(2)
    D = 128
    q, k = rng.standard_normal((1, D)), rng.standard_normal((1, D))
    s = []
    for m, n in [(5, 2), (13, 10), (1003, 1000), (3, 0)]:
        s.append(float((oracle.rope(q, t0=m) @ oracle.rope(k, t0=n).T)[0, 0]))
    assert np.allclose(s, s[0], rtol=1e-11, atol=1e-11)
    # and differ for another offset
    assert abs(float((oracle.rope(q, t0=7) @ oracle.rope(k, t0=2).T)[0, 0]) - s[0]) > 1e-6


def test_norms_pairs_and_group_law():
    rng = np.random.default_rng(3)
    D, L = 64, 17
    K = rng.standard_normal((L, D))
    R = oracle.rope(K, t0=123)
    # each pair keeps its length
    assert np.allclose(np.hypot(R[:, 0::2], R[:, 1::2]), np.hypot(K[:, 0::2], K[:, 1::2]), atol=1e-12)
    # rotating by a then by b is rotating by a + b (row i: positions 40 + i, then 60 + i)
    twice = oracle.rope(oracle.rope(K, t0=40), t0=60)
    rows = np.stack([oracle.rope(K[i:i + 1], t0=100 + 2 * i)[0] for i in range(L)])
    assert np.allclose(twice, rows, atol=1e-10)
    # only channels 2j and 2j+1 mix
    K2 = K.copy()
    K2[:, 7] += 1.0                                      # channel 7 = pair (6, 7)
    d = np.abs(oracle.rope(K2, t0=5) - oracle.rope(K, t0=5)).max(axis=0)
    assert np.all(d[[6, 7]] > 1e-3) and np.all(np.delete(d, [6, 7]) == 0.0)
    # position 0 is the identity
    assert np.array_equal(oracle.rope(K[:1], t0=0), K[:1])


def test_attention_over_fp16_cache_with_rope_matches_numpy():
    """KIVI cache with every token in the fp16 residual (L0 < G): attention rotates
    each key by its position; compared with numpy attention over complex-rotated keys."""
    rng = np.random.default_rng(4)
    B, H_q, H_kv, D, G = 1, 4, 2, 64, 128
    L0, base = 90, 10000.0
    K = rng.standard_normal((B, H_kv, L0, D)).astype(np.float16)
    V = rng.standard_normal((B, H_kv, L0, D)).astype(np.float16)
    q = rng.standard_normal((B, H_q, D)).astype(np.float16)
    c = OracleCache(B, H_q, H_kv, D, G, 2, R=G, rope_base=base)
    c.prefill(K, V)
    assert c.T_k == 0 and c.n_kres == L0
    got = c.attend(q)
    theta = base ** (-2.0 * np.arange(D // 2) / D)
    pos = np.arange(L0)[:, None]
    g = H_q // H_kv
    for h in range(H_kv):
        k = K[0, h].astype(np.float64)
        z = (k[:, 0::2] + 1j * k[:, 1::2]) * np.exp(1j * pos * theta)
        kr = np.empty_like(k)
        kr[:, 0::2], kr[:, 1::2] = z.real, z.imag
        s = q[0, h * g:(h + 1) * g].astype(np.float64) @ kr.T / np.sqrt(D)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        want = (p / p.sum(axis=1, keepdims=True)) @ V[0, h].astype(np.float64)
        assert np.allclose(got[0, h * g:(h + 1) * g], want, atol=1e-12)


def test_packed_keys_rotate_by_logical_position():
    """Sink, packed and residual keys are rotated by their position in the sequence:
    attention equals the textbook over the dequantized rows rotated in numpy."""
    rng = np.random.default_rng(5)
    B, H_q, H_kv, D, G = 1, 2, 1, 32, 32
    L0, S, base = 3 * G + 11 + 4, 4, 10000.0
    K = rng.standard_normal((B, H_kv, L0, D)).astype(np.float16)
    V = rng.standard_normal((B, H_kv, L0, D)).astype(np.float16)
    q = rng.standard_normal((B, H_q, D)).astype(np.float16)
    c = OracleCache(B, H_q, H_kv, D, G, 2, S=S, R=G, rope_base=base)
    c.prefill(K, V)
    assert c.n_sink == S and c.T_k == 3 * G and c.n_kres == 11
    Kd, Vd = c.rows(0, 0)                  # dequantized, unrotated, logical order
    theta = base ** (-2.0 * np.arange(D // 2) / D)
    z = (Kd[:, 0::2] + 1j * Kd[:, 1::2]) * np.exp(1j * np.arange(L0)[:, None] * theta)
    kr = np.empty_like(Kd)
    kr[:, 0::2], kr[:, 1::2] = z.real, z.imag
    s = q[0].astype(np.float64) @ kr.T / np.sqrt(D)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    want = (p / p.sum(axis=1, keepdims=True)) @ Vd
    assert np.allclose(c.attend(q)[0], want, atol=1e-12)
    # without RoPE the result differs
    c.rope_base = 0.0
    assert np.abs(c.attend(q)[0] - want).max() > 1e-3
