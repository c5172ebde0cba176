"""Pins of the oracle's NVFP4 pages (BitDecoding notes, Sec. V-D: Blackwell's native
mxfp4 / nvfp4 formats; the format itself is the reading stated in the oracle).

The small-float rounding is checked by brute force against every representable value
(nearest, ties to the even code, saturation), the page quantizer against scale and
code choices recomputed here in numpy float32, and attention over an NVFP4 cache
against the textbook formula over the dequantized rows.
"""
import numpy as np
import pytest

import oracle
from oracle import OracleCache


def _values(ebits, mbits, bias, nan_codes=()):
    n = 1 << (1 + ebits + mbits)
    return {c: oracle.small_float_value(c, ebits, mbits, bias) for c in range(n) if c not in nan_codes}


E2M1 = _values(2, 1, 1)
E4M3 = _values(4, 3, 7, nan_codes=(0x7F, 0xFF))


def test_e2m1_table():
    mags = [E2M1[c] for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert all(E2M1[c + 8] == -E2M1[c] for c in range(8))


def test_e4m3_extremes_and_subnormals():
    assert E4M3[0x7E] == 448.0                      # largest finite
    assert E4M3[0x01] == 2.0 ** -9                  # smallest subnormal
    assert E4M3[0x08] == 2.0 ** -6                  # smallest normal
    assert E4M3[0x38] == 1.0


def _brute(x, table, maxv):
    a = min(abs(x), maxv)
    best = None
    for c, v in table.items():
        if (c >> (len(bin(max(table))) - 3)) & 1 != 0:   # positive codes only
            continue
        d = abs(v - a)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c)
    c = best[1]
    sign_bit = (max(table) + 1) // 2
    return c | (sign_bit if np.signbit(x) else 0)


@pytest.mark.parametrize("fmt", ["e2m1", "e4m3"])
def test_rounding_is_nearest_even_and_saturating(fmt):
    rng = np.random.default_rng(1)
    if fmt == "e2m1":
        table, maxv, enc = E2M1, 6.0, oracle.e2m1_code
        xs = list(rng.uniform(-8, 8, 3000)) + [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, 6.0, 6.5, 100.0]
    else:
        table, maxv, enc = E4M3, 448.0, oracle.e4m3_code
        xs = list(np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), 4000)))
        # every midpoint between neighbouring positive values: ties
        vals = sorted(v for c, v in table.items() if c < 0x80)
        xs += [(a + b) / 2 for a, b in zip(vals, vals[1:])] + [448.0, 470.0, 1e6]
    for x in xs:
        x = float(np.float32(x))
        assert enc(x) == _brute(x, table, maxv), x


def test_round_trip_of_every_finite_code():
    for c, v in E4M3.items():
        if c in (0x80,):            # -0 encodes as itself
            assert oracle.e4m3_code(-0.0) == 0x80
            continue
        assert oracle.e4m3_code(v) == c
    for c, v in E2M1.items():
        assert oracle.e2m1_code(v if c != 8 else -0.0) == c


def _recompute_page(x16, values):
    """Scale and code choices of one page, recomputed in numpy float32."""
    x = x16.astype(np.float32)
    G, D = x.shape
    amax = np.float32(np.abs(x).max())
    S = np.float32(amax / np.float32(2688.0))
    blocks = x.T.reshape(D, G // 16, 16) if values else x.reshape(G, D // 16, 16)
    scales = np.zeros(blocks.shape[:2], np.uint8)
    codes = np.zeros(blocks.shape, np.uint8)
    for i in range(blocks.shape[0]):
        for j in range(blocks.shape[1]):
            blk = blocks[i, j]
            if S == 0:
                continue
            sb = np.float32(np.float32(np.abs(blk).max() / np.float32(6.0)) / S)
            sc = _brute(float(sb), E4M3, 448.0)
            scales[i, j] = sc
            d = np.float32(np.float32(E4M3[sc]) * S)
            for k in range(16):
                codes[i, j, k] = 0 if d == 0 else _brute(float(np.float32(blk[k] / d)), E2M1, 6.0)
    return S, scales, codes


@pytest.mark.parametrize("values", [False, True])
def test_page_quantizer_recomputed_in_float32(values):
    rng = np.random.default_rng(2 + values)
    G, D = 32, 32
    x = (rng.standard_normal((G, D)) * np.exp(rng.uniform(-3, 3, (1, D)))).astype(np.float16)
    x[3, :] = 0.0                      # an all-zero row / part of a block
    codes, scales, S = oracle.nvfp4_page(x, values)
    S_ref, sc_ref, c_ref = _recompute_page(x, values)
    assert S == S_ref
    # unpack codes [G][D/2] to logical [G][D]
    logical = np.zeros((G, D), np.uint8)
    logical[:, 0::2], logical[:, 1::2] = codes & 15, codes >> 4
    if values:
        assert np.array_equal(scales, sc_ref.T)                 # [G/16][D]
        assert np.array_equal(logical.T.reshape(D, G // 16, 16), c_ref)
    else:
        assert np.array_equal(scales, sc_ref)                   # [G][D/16]
        assert np.array_equal(logical.reshape(G, D // 16, 16), c_ref)


def test_page_layout_zero_page_and_error():
    G, D = 16, 32
    x = np.zeros((G, D), np.float16)
    codes, scales, S = oracle.nvfp4_page(x, False)
    assert S == 0 and not codes.any() and not scales.any()
    assert not oracle.nvfp4_dequant(codes, scales, S, False).any()
    x[5, 3] = 6.0                       # channel 3: byte 1, high nibble
    codes, scales, S = oracle.nvfp4_page(x, False)
    assert codes[5, 1] >> 4 == 7 and (codes[5, 1] & 15) == 0
    assert oracle.nvfp4_dequant(codes, scales, S, False)[5, 3] == pytest.approx(6.0, rel=2e-7)
    # dequantization error of random pages: within half an e2m1 step of each element,
    # with the block's e4m3 scale (<= 1/8 relative of the block maximum / 6 * 2)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 64)).astype(np.float16)
    for values in (False, True):
        codes, scales, S = oracle.nvfp4_page(x, values)
        xh = oracle.nvfp4_dequant(codes, scales, S, values)
        err = np.abs(xh - x.astype(np.float64))
        assert err.max() <= np.abs(x).max() * 0.5 / 6 * 2 * 1.25


def test_attention_over_nvfp4_cache_matches_textbook():
    rng = np.random.default_rng(4)
    B, H_q, H_kv, D, G = 1, 4, 2, 64, 32
    L0 = 2 * G + 9
    K = rng.standard_normal((B, H_kv, L0, D)).astype(np.float16)
    V = rng.standard_normal((B, H_kv, L0, D)).astype(np.float16)
    q = rng.standard_normal((B, H_q, D)).astype(np.float16)
    c = OracleCache(B, H_q, H_kv, D, G, 4, R=G, mode="nvfp4")
    c.prefill(K, V)
    assert c.T_k == 2 * G and c.n_kres == 9
    got = c.attend(q)
    g = H_q // H_kv
    for h in range(H_kv):
        Kd, Vd = c.rows(0, h)
        # packed rows are the page dequantization; residual rows are the fp16 inputs
        assert np.array_equal(Kd[2 * G:], K[0, h, 2 * G:].astype(np.float64))
        s = q[0, h * g:(h + 1) * g].astype(np.float64) @ Kd.T / np.sqrt(D)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        want = (p / p.sum(axis=1, keepdims=True)) @ Vd
        assert np.allclose(got[0, h * g:(h + 1) * g], want, atol=1e-12)
