"""The division-free quantizer of the CUDA kernels, restated in numpy float32, against
the oracle (CPU only).

The quantize/pack kernels do not divide per value.  They form r = (x - min) * rcp(scale)
in fp32, round it by adding 1.5 * 2^23 (the integer lands in the low mantissa bits,
ties to even), clamp, and recompute with IEEE division every value whose r lies within
2^-14 of a half-integer.  Because |r - fl(d / s)| is a few ulp of r, a value farther from
a tie than that margin rounds the same either way.  The oracle quantizes with IEEE
division (KIVI notes, Step 1).  numpy's float32 operations round like the kernels', so
the same steps here must give the oracle's codes for every value: on random groups, on
groups built to sit on and next to rounding ties, and at every code width.  The last
test checks that it is the recompute that makes them agree: without it, the near-tie
groups differ.
"""
import numpy as np
import pytest

import oracle

MAGIC = np.float32(1.5 * 2.0 ** 23)


def fast_codes(x16: np.ndarray, bits: int, margin: float = 0.5 - 2.0 ** -14) -> np.ndarray:
    """The kernels' steps for one group (fp16 values): exact min/max, the fp16 scale,
    then multiply by the fp32 reciprocal, round by the magic add, recompute near ties."""
    max_int = (1 << bits) - 1
    x = x16.astype(np.float32)
    mn, mx = np.float32(x.min()), np.float32(x.max())
    if mn == 0:
        mn = np.float32(0.0)          # -0 -> +0
    if mx == 0:
        mx = np.float32(0.0)
    s32 = np.float32(mx - mn) / np.float32(max_int)
    s = np.float32(np.float16(s32))
    if s == 0:
        return np.zeros(x.size, np.uint8)
    inv = np.float32(1.0) / s
    d = x - mn                        # exact: both are fp16 values
    r = d * inv
    k = (r + MAGIC) - MAGIC           # rint(r), ties to even
    near = np.abs(r - k) > np.float32(margin)
    k = np.where(near, np.rint(d / s), k)
    return np.minimum(k, np.float32(max_int)).astype(np.uint8)


def oracle_codes(x16: np.ndarray, bits: int) -> np.ndarray:
    return oracle.quant_group(x16, bits)[2]


def random_groups(rng, n, size):
    scale = np.float32(2.0) ** rng.integers(-12, 6, size=(n, 1)).astype(np.float32)
    x = rng.standard_normal((n, size)).astype(np.float32) * scale
    return x.astype(np.float16)


def tie_groups(rng, n, size, bits):
    """Groups whose values sit on, or one fp16 step beside, min + (k + 1/2) * scale."""
    max_int = (1 << bits) - 1
    out = np.empty((n, size), np.float16)
    for i in range(n):
        mn = np.float16(rng.standard_normal() * 2.0 ** rng.integers(-6, 4))
        step = np.float16(abs(rng.standard_normal()) * 2.0 ** rng.integers(-8, 2) + 1e-3)
        mx = np.float16(np.float32(mn) + max_int * np.float32(step))
        s = np.float32(np.float16((np.float32(mx) - np.float32(mn)) / np.float32(max_int)))
        k = rng.integers(0, max_int, size=size).astype(np.float32)
        v = (np.float32(mn) + (k + np.float32(0.5)) * s).astype(np.float16)
        nudge = rng.integers(-1, 2, size=size)
        v = np.where(nudge < 0, np.nextafter(v, np.float16(-np.inf)),
                     np.where(nudge > 0, np.nextafter(v, np.float16(np.inf)), v))
        v[0], v[1] = mn, mx           # the group's min and max stay as built
        v = np.clip(v, mn, mx)
        out[i] = v
    return out


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_fast_path_equals_oracle_on_random_groups(bits):
    rng = np.random.default_rng(100 + bits)
    for g in random_groups(rng, 400, 128):
        assert np.array_equal(fast_codes(g, bits), oracle_codes(g, bits))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_fast_path_equals_oracle_on_ties(bits):
    rng = np.random.default_rng(200 + bits)
    groups = tie_groups(rng, 300, 64, bits)
    for g in groups:
        assert np.array_equal(fast_codes(g, bits), oracle_codes(g, bits))


def test_the_recompute_is_what_makes_ties_agree():
    """With the near-tie recompute switched off (a margin no rounding error reaches), the
    tie groups give other codes than the oracle for some values."""
    rng = np.random.default_rng(7)
    diff = 0
    for bits in (2, 4, 8):
        for g in tie_groups(rng, 200, 64, bits):
            diff += int(np.count_nonzero(fast_codes(g, bits, margin=1.0) != oracle_codes(g, bits)))
    assert diff > 0
