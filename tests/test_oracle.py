"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests re-types the oracle's formulas: each checks a property that
a plausible mistake (wrong step, floor instead of round-half-even, dropped min,
wrong pack shift or axis, wrong top-k tie rule, missing 1/sqrt(d), ...) breaks.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import OracleCache

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- #
# fp16 conversions: numpy's float16 cast is the library routine they reduce to  #
# --------------------------------------------------------------------------- #

def test_h2f_exhaustive_matches_numpy():
    h = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.h2f(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f2h_matches_numpy_rne():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    # every tie between adjacent finite fp16 values (and the overflow tie)
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    ties = ((lo + hi) / 2).astype(np.float32)
    ties = ties[np.isfinite(ties)]
    extra = np.array([65504, 65519.99, 65520, 65536, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8,
                      1e-8, 0.0, -0.0], np.float32)
    for arr in (f, ties, -ties, extra):
        ours = oracle.f2h(arr)
        with np.errstate(over="ignore"):
            ref = arr.astype(np.float16).view(np.uint16)
        assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------- #
# The quantizer of one group                                                   #
# --------------------------------------------------------------------------- #

def _slack(bits):
    """Relative slack on half a step.  The code is rint(v) with v = fl32(fl32(x - mn) / s):
    two fp32 roundings of a quotient below max_int (1 + 2^-11) (s is the fp16 rounding of
    (mx - mn) / max_int, at most 2^-11 below it), so v is within max_int (1 + 2^-10) 2^-23
    of the exact quotient, and x - (code s + mn) within s/2 (1 + max_int (1 + 2^-10) 2^-22)."""
    return ((1 << bits) - 1) * (1 + 2.0 ** -10) * 2.0 ** -22


def _err_bound_ok(x16, bits):
    s, mn, c = oracle.quant_group(x16, bits)
    xh = oracle.dequant(c, s, mn)
    x = x16.astype(np.float64)
    sf = float(s)
    mi = (1 << bits) - 1
    assert c.max(initial=0) <= mi
    if sf == 0.0:
        # zero scale: every code is 0, the error is at most the group's range
        assert not c.any()
        assert np.all(np.abs(x - xh) <= x.max() - x.min())
        return
    bound = sf / 2 * (1 + _slack(bits))
    if abs(sf) < 2.0 ** -14:
        # A subnormal scale is (mx - mn) / max_int rounded to a multiple of 2^-24: up to
        # 2^-25 off, an unbounded fraction of the scale.  Values that clamp to the top code
        # then sit up to max_int (2^-25 + 2^-24 s) above it; interior codes keep the bound.
        bound += mi * (2.0 ** -25 + 2.0 ** -24 * sf)
    assert np.all(np.abs(x - xh) <= bound), (x16, s, mn, c)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_quant_error_bound_random(bits):
    rng = np.random.default_rng(bits)
    for trial in range(3000):
        n = int(rng.integers(1, 160))
        scale = 10.0 ** rng.uniform(-3, 3)
        x = (rng.standard_normal(n) * scale).astype(np.float16)
        _err_bound_ok(x, bits)


def test_quant_error_bound_wide_and_tiny():
    from kvq_synth import random_fp16
    rng = np.random.default_rng(7)
    for special in ("wide", "tiny"):
        for _ in range(500):
            x = random_fp16(rng, (64,), special=special)
            for bits in (2, 4):
                _err_bound_ok(x, bits)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_quant_exact_grid_gives_every_level(bits):
    """x = mn + k*s with exactly representable grid points: code == k, 2^b levels."""
    rng = np.random.default_rng(11 + bits)
    mi = (1 << bits) - 1
    for _ in range(200):
        e = int(rng.integers(-8, 4))
        s = np.float16(2.0 ** e * rng.choice([1.0, 1.25, 1.5, 1.75]))
        mn = np.float16(rng.integers(-64, 64) * 2.0 ** e)
        k = np.arange(mi + 1)
        vals = (np.float64(mn) + k * np.float64(s))
        x = vals.astype(np.float16)
        if not np.array_equal(x.astype(np.float64), vals):
            continue  # grid not representable in fp16
        perm = rng.permutation(mi + 1)
        sq, mq, c = oracle.quant_group(x[perm], bits)
        assert sq == s and mq == mn
        assert np.array_equal(c, k[perm])
        assert len(set(c.tolist())) == mi + 1


def test_quant_round_half_to_even():
    """Exact midpoints between levels go to the even code (torch .round semantics)."""
    # mn=0, mx=3 -> s=1; x = 0.5, 1.5, 2.5 are exact ties
    x = np.array([0.0, 3.0, 0.5, 1.5, 2.5, 1.0], np.float16)
    s, mn, c = oracle.quant_group(x, 2)
    assert float(s) == 1.0 and float(mn) == 0.0
    assert c.tolist() == [0, 3, 0, 2, 2, 1]


def test_quant_constant_and_negative_zero():
    for v in (0.0, -0.0, 1.5, -7.25, 65504.0):
        x = np.full(17, v, np.float16)
        s, mn, c = oracle.quant_group(x, 2)
        assert float(s) == 0.0 and not c.any()
        assert oracle.dequant(c, s, mn).tolist() == x.astype(np.float64).tolist()
        assert np.float16(mn).view(np.uint16) != 0x8000  # -0.0 min stored as +0.0


def test_quant_scale_underflow_gives_code_zero():
    # range 2^-24: (max-min)/3 rounds to fp16 0 -> all codes 0
    x = np.array([0.0, 2.0 ** -24], np.float16)
    s, mn, c = oracle.quant_group(x, 2)
    assert float(s) == 0.0 and not c.any()


def test_quant_brute_force_small_alphabet():
    """Every group of 3 drawn from an alphabet spanning signs, zeros, subnormals and
    normals: codes in range, monotone in x, extremes mapped to 0 and (near) max."""
    alphabet = np.array([0.0, -0.0, 2 ** -24, -(2 ** -20), 2 ** -14, 0.1, -0.1, 0.3333,
                         1.0, -1.0, 2.5, 100.0, -60000.0], np.float16)
    for bits in (2, 4):
        mi = (1 << bits) - 1
        for combo in itertools.product(range(len(alphabet)), repeat=3):
            x = alphabet[list(combo)]
            s, mn, c = oracle.quant_group(x, bits)
            xf = x.astype(np.float64)
            assert float(mn) == xf.min()
            order = np.argsort(xf, kind="stable")
            assert np.all(np.diff(c[order].astype(int)) >= 0)      # monotone
            if float(s) > 0:
                assert c[np.argmin(xf)] == 0
                assert c[np.argmax(xf)] >= mi - 1
            _err_bound_ok(x, bits)


# --------------------------------------------------------------------------- #
# pack_tensor layouts                                                          #
# --------------------------------------------------------------------------- #

def _unpack_along(words, bits, axis):
    """Independent decoder: element j of a word at bits [b*j, b*j+b)."""
    fpi = 32 // bits
    w = np.moveaxis(words.view(np.uint32), axis, -1)
    sh = (np.arange(fpi, dtype=np.uint32) * bits)
    c = (w[..., None] >> sh) & np.uint32((1 << bits) - 1)
    c = c.reshape(w.shape[:-1] + (w.shape[-1] * fpi,))
    return np.moveaxis(c, -1, axis)


def test_pack_worked_example_column_19():
    """KIVI page, Step 4: 2-bit logical column 19 lives in word 19//16 = 1 at shift 6."""
    G = 32
    K = np.zeros((1, 1, G, 4), np.float16)
    K[0, 0, 19, 2] = 1.0          # only token 19 of channel 2 is non-zero -> code 3
    codes, meta = oracle.quant_k(K, G=G, bits=2)
    assert codes.shape == (1, 1, 2, 4)                          # [B,nh,T/16,D]
    w = codes.view(np.uint32)
    assert w[0, 0, 1, 2] == 3 << 6 and w[0, 0, 0, 2] == 0
    assert not w[..., [0, 1, 3]].any()
    # values pack along channels: channel 19 of a token -> word 1, shift 6
    V = np.zeros((1, 1, 1, 32), np.float16)
    V[0, 0, 0, 19] = 1.0
    vc, _ = oracle.quant_v(V, Gv=32, bits=2)
    assert vc.view(np.uint32)[0, 0, 0].tolist() == [0, 3 << 6]
    # 4-bit: 8 codes per word -> column 19 is word 2, shift 12
    vc4, _ = oracle.quant_v(V, Gv=32, bits=4)
    assert vc4.view(np.uint32)[0, 0, 0].tolist() == [0, 0, 15 << 12, 0]


def test_pack_shape_example():
    """[B, nh, T, D] keys packed along T at 2 bits become [B, nh, T/16, D] words."""
    K = np.random.default_rng(0).standard_normal((2, 3, 64, 8)).astype(np.float16)
    codes, meta = oracle.quant_k(K, G=32, bits=2)
    assert codes.shape == (2, 3, 4, 8) and meta.shape == (2, 3, 2, 8, 2)
    codes4, _ = oracle.quant_k(K, G=32, bits=4)
    assert codes4.shape == (2, 3, 8, 8)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_round_trip_equals_group_codes(bits):
    rng = np.random.default_rng(100 + bits)
    G, Gv, D = 32, 32, 64
    K = rng.standard_normal((2, 2, 3 * G, D)).astype(np.float16)
    codes, meta = oracle.quant_k(K, G=G, bits=bits)
    unpacked = _unpack_along(codes, bits, axis=2)               # [B,H,T,D]
    for b, h, gi, d in itertools.product(range(2), range(2), range(3), range(D)):
        s, mn, c = oracle.quant_group(K[b, h, gi * G:(gi + 1) * G, d], bits)
        assert np.array_equal(unpacked[b, h, gi * G:(gi + 1) * G, d], c)
        assert meta[b, h, gi, d, 0] == s and meta[b, h, gi, d, 1] == mn
    V = rng.standard_normal((2, 2, 40, D)).astype(np.float16)
    vc, vm = oracle.quant_v(V, Gv=Gv, bits=bits)
    vu = _unpack_along(vc, bits, axis=3)
    for b, h, t, gv in itertools.product(range(2), range(2), range(40), range(D // Gv)):
        s, mn, c = oracle.quant_group(V[b, h, t, gv * Gv:(gv + 1) * Gv], bits)
        assert np.array_equal(vu[b, h, t, gv * Gv:(gv + 1) * Gv], c)
        assert vm[b, h, t, gv, 0] == s and vm[b, h, t, gv, 1] == mn


def test_kitty_byte_view_of_low_plane():
    """Kitty stores 4 two-bit codes per byte with shifts [0,2,4,6]; the same bits read
    as little-endian int32 are the 16-code words used here."""
    rng = np.random.default_rng(5)
    K = rng.standard_normal((1, 1, 128, 16)).astype(np.float16)
    lo, hi, bidx, meta = oracle.quant_k_kitty(K, G=128, n_boost=0)
    codes2, _ = oracle.quant_k(K, G=128, bits=2)
    by = lo.view(np.uint8).reshape(1, 1, 8, 16, 4)                 # [.., tb, d, byte]
    c = (by[..., None] >> np.array([0, 2, 4, 6], np.uint8)) & 3     # [.., tb, d, byte, j]
    c = c.transpose(0, 1, 2, 4, 5, 3).reshape(1, 1, 128, 16)        # token = 16tb+4byte+j
    assert np.array_equal(c, _unpack_along(codes2, 2, axis=2))


# --------------------------------------------------------------------------- #
# Kitty channel boost                                                          #
# --------------------------------------------------------------------------- #

def _brute_topk(page, n_boost):
    G, D = page.shape
    score = [sum(int(abs(float(page[t, d])) * 2 ** 24) for t in range(G)) for d in range(D)]
    order = sorted(range(D), key=lambda d: (-score[d], d))
    return score, sorted(order[:n_boost])


@pytest.mark.parametrize("n_boost", [0, 1, 3, 8, 16])
def test_kitty_select_brute_force(n_boost):
    rng = np.random.default_rng(n_boost)
    for trial in range(40):
        D = 16
        page = rng.standard_normal((8, D)).astype(np.float16)
        if trial % 3 == 0:        # force ties between channels
            page[:, 5] = page[:, 2]
            page[:, 11] = -page[:, 2]
        if trial % 5 == 0:        # subnormals and zeros
            page[:, 7] = np.float16(2 ** -24)
            page[:, 9] = 0
        score, idx = oracle.kitty_select(page, n_boost)
        bscore, chosen = _brute_topk(page, n_boost)
        assert score.tolist() == bscore
        slots = [int(bidx) for bidx in idx]
        got = [d for d in range(D) if slots[d] < n_boost]
        assert got == chosen
        assert [slots[d] for d in got] == list(range(n_boost))      # ascending slots
        assert all(slots[d] == n_boost + 1 for d in range(D) if d not in chosen)


def test_kitty_zero_boost_equals_kivi_2bit():
    rng = np.random.default_rng(21)
    K = (rng.standard_normal((2, 2, 256, 32)) * 3).astype(np.float16)
    lo, hi, bidx, meta = oracle.quant_k_kitty(K, G=128, n_boost=0)
    c2, m2 = oracle.quant_k(K, G=128, bits=2)
    assert np.array_equal(lo, c2) and np.array_equal(meta.view(np.uint16), m2.view(np.uint16))
    assert np.all(bidx == 1)


def test_kitty_full_boost_equals_kivi_4bit():
    rng = np.random.default_rng(22)
    D = 32
    K = (rng.standard_normal((2, 2, 256, D)) * 3).astype(np.float16)
    lo, hi, bidx, meta = oracle.quant_k_kitty(K, G=128, n_boost=D)
    c4, m4 = oracle.quant_k(K, G=128, bits=4)
    assert np.all(bidx == np.arange(D, dtype=np.uint8))
    low = _unpack_along(lo, 2, axis=2)
    high = _unpack_along(hi, 2, axis=2)        # slot order == channel order here
    assert np.array_equal(low | (high << 2), _unpack_along(c4, 4, axis=2))
    assert np.array_equal(meta.view(np.uint16), m4.view(np.uint16))


def test_kitty_boosted_channels_have_smaller_error():
    """An outlier channel is boosted and its 4-bit error bound is 1/5 of the 2-bit one."""
    rng = np.random.default_rng(3)
    K = rng.standard_normal((1, 1, 128, 16)).astype(np.float16)
    K[..., 6] = (K[..., 6].astype(np.float32) * 10).astype(np.float16)
    lo, hi, bidx, meta = oracle.quant_k_kitty(K, G=128, n_boost=2)
    assert bidx[0, 0, 0, 6] < 2
    c = OracleCache(1, 1, 1, 16, 128, 2, n_boost=2, mode="kitty", R=16)
    c.prefill(K, K)
    Kh, _ = c.rows(0, 0)
    Kt = K[0, 0, : c.T_k].astype(np.float64)
    s6 = float(meta[0, 0, 0, 6, 0])
    assert np.abs(Kh[: c.T_k, 6] - Kt[:, 6]).max() <= s6 / 2 * (1 + 2 ** -16)
    assert s6 <= (Kt[:, 6].max() - Kt[:, 6].min()) / 15 * (1 + 2 ** -10)


# --------------------------------------------------------------------------- #
# Attention                                                                    #
# --------------------------------------------------------------------------- #

def _textbook(q, K, V):
    out = np.zeros(q.shape)
    for h in range(q.shape[0]):
        z = [sum(float(q[h, d]) * float(K[t, d]) for d in range(K.shape[1])) / math.sqrt(K.shape[1])
             for t in range(K.shape[0])]
        e = [math.exp(v) for v in z]
        tot = sum(e)
        for d in range(K.shape[1]):
            out[h, d] = sum(e[t] * float(V[t, d]) for t in range(K.shape[0])) / tot
    return out


def test_attention_quantization_off_equals_textbook():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, D, G = 2, 4, 2, 16, 32
    K = rng.standard_normal((B, Hkv, 20, D)).astype(np.float16)
    V = rng.standard_normal((B, Hkv, 20, D)).astype(np.float16)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    c = OracleCache(B, Hq, Hkv, D, G, 2, R=G)
    c.prefill(K, V)                       # 20 < G: nothing is quantized
    assert c.T_k == 0 and c.n_kres == 20
    out = c.attend(q)
    g = Hq // Hkv
    for b in range(B):
        for hq in range(Hq):
            ref = _textbook(q[b, hq:hq + 1], K[b, hq // g], V[b, hq // g])
            assert np.allclose(out[b, hq], ref[0], rtol=1e-13, atol=1e-13)


def test_attention_one_token_uniform_and_permutation():
    rng = np.random.default_rng(10)
    D = 32
    v = rng.standard_normal((1, D))
    k = rng.standard_normal((1, D))
    q = rng.standard_normal((3, D))
    assert np.array_equal(oracle.attend(q, k, v), np.repeat(v, 3, 0))
    K = rng.standard_normal((50, D))
    V = rng.standard_normal((50, D))
    out0 = oracle.attend(np.zeros((1, D)), K, V)
    assert np.allclose(out0[0], V.mean(0), rtol=1e-14, atol=1e-14)
    p = rng.permutation(50)
    a = oracle.attend(q, K, V)
    assert np.allclose(a, oracle.attend(q, K[p], V[p]), rtol=1e-13, atol=1e-13)
    # 1/sqrt(d) scaling: doubling q equals attention with keys doubled
    assert np.allclose(oracle.attend(2 * q, K, V), oracle.attend(q, 2 * K, V), rtol=1e-13)


def test_attention_long_double_cross_check():
    rng = np.random.default_rng(12)
    D, L = 16, 64
    q = rng.standard_normal((2, D)) * 3
    K = rng.standard_normal((L, D)) * 3
    V = rng.standard_normal((L, D))
    ql, Kl, Vl = (a.astype(np.longdouble) for a in (q, K, V))
    z = ql @ Kl.T / np.sqrt(np.longdouble(D))
    z = np.exp(z - z.max(1, keepdims=True))
    ref = (z @ Vl) / z.sum(1, keepdims=True)
    assert np.allclose(oracle.attend(q, K, V), ref.astype(np.float64), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- #
# The cache pipeline                                                           #
# --------------------------------------------------------------------------- #

def test_kivi_prefill_append_flush_equals_one_shot_quant():
    rng = np.random.default_rng(30)
    B, H, D, G, bits = 1, 2, 32, 32, 2
    L = 5 * G + 7
    K = rng.standard_normal((B, H, L, D)).astype(np.float16)
    V = rng.standard_normal((B, H, L, D)).astype(np.float16)
    c = OracleCache(B, H, H, D, G, bits, R=G)
    c.prefill(K[:, :, :2 * G + 5], V[:, :, :2 * G + 5])
    assert (c.T_k, c.n_kres, c.T_v, c.n_vres) == (2 * G, 5, 2 * G, 5)
    for t in range(2 * G + 5, L):
        c.append(K[:, :, t], V[:, :, t])
        c.flush()
    assert c.T_k == 5 * G and c.n_kres == 7
    ck, mk = oracle.quant_k(K, G, bits, 0, 5 * G)
    cv, mv = oracle.quant_v(V, min(G, D), bits, 0, 5 * G)
    assert np.array_equal(c.k_codes, ck) and np.array_equal(c.v_codes, cv)
    assert np.array_equal(c.k_meta.view(np.uint16), mk.view(np.uint16))
    assert np.array_equal(c.v_meta.view(np.uint16), mv.view(np.uint16))
    assert np.array_equal(c.k_res[:, :, :7], K[:, :, 5 * G:])


def test_kitty_buffers_keep_chronological_order():
    rng = np.random.default_rng(31)
    B, H, D, G, S, R = 1, 1, 16, 16, 4, 16
    L = S + 7 * G + 9
    K = rng.standard_normal((B, H, L, D)).astype(np.float16)
    V = rng.standard_normal((B, H, L, D)).astype(np.float16)
    c = OracleCache(B, 2, H, D, G, 2, S=S, R=R, n_boost=4, mode="kitty")
    c.prefill(K[:, :, :S + 2 * G + 3], V[:, :, :S + 2 * G + 3])
    for t in range(S + 2 * G + 3, L):
        c.append(K[:, :, t], V[:, :, t])
        assert c.n_kres <= G and c.n_vres <= G
        _, Vh = c.rows(0, 0)
        n_fp16_v = c.n_vres + c.n_local
        # the fp16 value tail is exactly the most recent tokens, oldest first
        assert np.array_equal(Vh[c.L - n_fp16_v:], V[0, 0, c.L - n_fp16_v:c.L].astype(np.float64))
        assert np.array_equal(Vh[:S], V[0, 0, :S].astype(np.float64))
        c.flush()
    assert c.n_local == R and c.L == L


def test_sink_fills_before_buffers():
    rng = np.random.default_rng(32)
    K = rng.standard_normal((1, 1, 3, 16)).astype(np.float16)
    c = OracleCache(1, 1, 1, 16, 16, 2, S=8, R=16, mode="kitty")
    c.prefill(K, K)
    assert c.n_sink == 3 and c.T_k == 0 and c.n_kres == 0 and c.n_local == 0
    for t in range(6):
        c.append(K[0, :, 0], K[0, :, 0])
    assert c.n_sink == 8 and c.n_kres == 1 and c.n_local == 1


# --------------------------------------------------------------------------- #
# Bytes accounting: the KV-cache size formula against the pages' tables         #
# --------------------------------------------------------------------------- #

def test_cache_bytes_formula_against_pages():
    with open(os.path.join(GOLDEN, "cache_bytes.json")) as f:
        gold = json.load(f)
    for row in gold["fp16_cache_gib"]:
        got = oracle.fp16_cache_bytes(row["layers"], 1, row["tokens"], row["kv_heads"],
                                      row["head_dim"]) / 2 ** 30
        assert round(got, 0) == row["gib"], row
    per_tok = oracle.fp16_cache_bytes(32, 1, 1, 32, 128)
    assert per_tok == gold["llama7b_bytes_per_token"]
    kitty = gold["llama3_70b_32x128k"]
    tb = oracle.fp16_cache_bytes(80, 32, 131072, 8, 128) / 1e12
    assert tb > kitty["exceeds_tb"]
    kb = gold["kivi_avg_bits"]
    assert round(oracle.kivi_avg_bits(kb["bits"], kb["G"], kb["R"], kb["L"]), 2) == kb["avg_bits"]


def test_packed_sizes_match_accounting():
    """Measured sizes of the oracle's packed arrays equal the bytes accounting:
    b/8 bytes per element of codes plus 4 bytes (fp16 scale + min) per group."""
    rng = np.random.default_rng(40)
    B, H, D, G = 2, 2, 64, 32
    for bits in (2, 4, 8):
        K = rng.standard_normal((B, H, 4 * G, D)).astype(np.float16)
        ck, mk = oracle.quant_k(K, G, bits)
        cv, mv = oracle.quant_v(K, G, bits)
        n = B * H * 4 * G * D
        assert ck.nbytes == cv.nbytes == n * bits // 8
        assert mk.nbytes == mv.nbytes == n // G * 4


def test_signed_zero_groups_store_positive_zero():
    """Groups of +0/-0 in any order: scale and min are +0.0 (no sign from the order)."""
    for vals in ([0.0, -0.0], [-0.0, 0.0], [-0.0, -0.0, 0.0], [-0.0]):
        s, mn, c = oracle.quant_group(np.array(vals, np.float16), 2)
        assert np.float16(s).view(np.uint16) == 0 and np.float16(mn).view(np.uint16) == 0
    s, mn, c = oracle.quant_group(np.array([-1.0, -0.0], np.float16), 2)
    assert float(mn) == -1.0 and c.tolist() == [0, 3]


# --------------------------------------------------------------------------- #
# Separate key and value widths (K4V2, K2V4, K8V8, K2V2 with sinks)            #
# --------------------------------------------------------------------------- #

def _unpack_rows(words: np.ndarray, bits: int, along_last: bool) -> np.ndarray:
    """Codes from packed int32 words, element j of a word at bit bits*j (numpy)."""
    fpi = 32 // bits
    w = words.astype(np.int64) & 0xFFFFFFFF
    shifts = (np.arange(fpi) * bits).astype(np.int64)
    c = (w[..., None] >> shifts) & ((1 << bits) - 1)           # [..., words, fpi]
    if along_last:
        return c.reshape(c.shape[:-2] + (-1,))                 # values: along channels
    c = np.moveaxis(c, -1, -2)                                 # keys: [T/fpi, fpi, D]
    return c.reshape(c.shape[:-3] + (-1, c.shape[-1]))


@pytest.mark.parametrize("kb,vb,S", [(4, 2, 0), (2, 4, 0), (8, 8, 0), (2, 2, 4)])
def test_mixed_widths_codes_and_attention(kb, vb, S):
    rng = np.random.default_rng(40 + kb + vb + S)
    B, Hq, Hkv, D, G = 1, 4, 2, 32, 32
    L = S + 3 * G + 9
    K = rng.standard_normal((B, Hkv, L, D)).astype(np.float16)
    V = rng.standard_normal((B, Hkv, L, D)).astype(np.float16)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    c = OracleCache(B, Hq, Hkv, D, G, kb, S=S, R=G, v_bits=vb)
    c.prefill(K, V)
    T = 3 * G
    assert (c.n_sink, c.T_k, c.T_v, c.n_kres, c.n_vres) == (S, T, T, 9, 9)
    # the packed parts are the one-shot quantizers at their own widths
    ck, mk = oracle.quant_k(K, G, kb, S, T)
    cv, mv = oracle.quant_v(V, min(G, D), vb, S, T)
    assert c.v_codes.shape[-1] == D * vb // 32
    assert np.array_equal(c.k_codes, ck) and np.array_equal(c.v_codes, cv)
    # attention equals a textbook softmax over rows dequantized here with numpy
    kc = _unpack_rows(c.k_codes, kb, along_last=False)         # [B,H,T,D]
    vc = _unpack_rows(c.v_codes, vb, along_last=True)          # [B,H,T,D]
    km = c.k_meta.astype(np.float64)                           # [B,H,T/G,D,2]
    vm = c.v_meta.astype(np.float64)                           # [B,H,T,1,2]
    kd = kc * np.repeat(km[..., 0], G, axis=2) + np.repeat(km[..., 1], G, axis=2)
    vd = vc * vm[..., 0] + vm[..., 1]
    Kf = np.concatenate([K[:, :, :S].astype(np.float64), kd, K[:, :, S + T:].astype(np.float64)], 2)
    Vf = np.concatenate([V[:, :, :S].astype(np.float64), vd, V[:, :, S + T:].astype(np.float64)], 2)
    out = c.attend(q)
    g = Hq // Hkv
    for hq in range(Hq):
        z = Kf[0, hq // g] @ q[0, hq].astype(np.float64) / math.sqrt(D)
        p = np.exp(z - z.max())
        ref = (p / p.sum()) @ Vf[0, hq // g]
        assert np.allclose(out[0, hq], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_quant_error_bound_subnormal_scales(bits):
    """Groups whose scale is an fp16 subnormal (ranges below max_int 2^-14): the interior
    bound plus the clamp term of the rounded scale; the case is hit, not skipped."""
    rng = np.random.default_rng(40 + bits)
    hit = 0
    for _ in range(2000):
        n = int(rng.integers(2, 64))
        span = 2.0 ** rng.uniform(-24, -14) * ((1 << bits) - 1)
        base = float(rng.choice([0.0, 1.0, -3.5e-3, 2.0 ** -10]))
        x = (base + rng.uniform(0, span, n)).astype(np.float16)
        s, _, _ = oracle.quant_group(x, bits)
        hit += 0.0 < float(s) < 2.0 ** -14
        _err_bound_ok(x, bits)
    assert hit > 100


def test_oracle_attend_threads_equal_single_thread():
    """The all-cores form of the oracle (units on a thread pool) gives the same numbers."""
    import kvq_synth
    wl = kvq_synth.WORKLOADS["llama3_8b_gqa_b2"].replace(B=2, H_q=8, H_kv=4, T=512)
    K, V = kvq_synth.prefill_kv(wl, 512 + 70)
    o = OracleCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, R=wl.R)
    o.prefill(K, V)
    q = kvq_synth.queries(wl, 1)[0]
    assert np.array_equal(o.attend(q), o.attend(q, threads=4))
