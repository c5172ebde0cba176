"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

This module holds NO arithmetic of the quantization method: it only draws
random fp16 tensors with the shapes and value structure of the workloads the
KV-cache pages evaluate on (LLaMA / Llama-3 / Qwen3-class attention layers).
Those pages run real models on real datasets; neither is available here, so
these tensors stand in for them:

* K: N(0,1) with a fixed set of "outlier" channels per KV head, shared by all
  batch rows and tokens, multiplied by a constant.  This mirrors the observation
  on the KIVI and KVQuant pages that a few fixed key channels carry very large
  magnitudes (KIVI notes, Step 1; KVQuant, per-channel key quantization).
* V: N(0,1); optionally each (batch, head, token) vector is an outlier with a
  small probability and is multiplied by a constant (no channel pattern, as the
  KIVI page reports for the value cache).
* q: N(0,1), one query token per sequence (decode).

Every draw is float32 from numpy's PCG64, then rounded to fp16 (round to
nearest even, numpy's float16 cast).  Generation is per (b, h) row so that the
128K-token case does not need a multi-GB float32 temporary; the draw order is
part of the recipe: outlier channels first (one ``choice`` per KV head), then
for b, then for h: K rows, V rows, V outlier mask.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic KV-cache workload."""

    name: str
    B: int
    H_q: int
    H_kv: int
    D: int
    T: int            # packed (quantized) tokens per (b, h_kv) at measurement
    G: int            # quantization group / page size in tokens
    R: int            # KIVI residual capacity, or Kitty local-window size
    bits: int
    S: int = 0        # fp16 attention-sink tokens
    n_boost: int = 0  # Kitty: key channels kept at INT4 per page
    mode: str = "kivi"  # "kivi" or "kitty"
    seed: int = 0
    k_outlier_channels: int = 0
    k_outlier_scale: float = 1.0
    v_outlier_prob: float = 0.0
    v_outlier_scale: float = 1.0
    v_bits: int = 0   # value code width; 0: the same as bits
    ragged: float = 0.0  # paged cache: slot lengths spread uniformly over T (1 +- ragged)
    rope_base: float = 0.0  # > 0: keys cached before RoPE (rotated in decode attention)

    @property
    def vbits(self) -> int:
        return self.v_bits or self.bits

    @property
    def g(self) -> int:
        return self.H_q // self.H_kv

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the study (shapes of the pages' LLaMA-7B, Llama-3-8B and
# Qwen3-8B-class layers; sizes and seeds fixed here).
WORKLOADS = {
    "tiny_kivi": Workload("tiny_kivi", B=1, H_q=4, H_kv=4, D=128, T=256, G=32, R=32,
                          bits=2, seed=0, k_outlier_channels=4, k_outlier_scale=10.0),
    "llama7b_mha": Workload("llama7b_mha", B=8, H_q=32, H_kv=32, D=128, T=4096, G=128,
                            R=128, bits=2, seed=2, k_outlier_channels=8,
                            k_outlier_scale=8.0),
    "llama3_8b_gqa_b2": Workload("llama3_8b_gqa_b2", B=4, H_q=32, H_kv=8, D=128, T=32768,
                                 G=128, R=128, bits=2, seed=3, k_outlier_channels=6,
                                 k_outlier_scale=10.0, v_outlier_prob=0.001,
                                 v_outlier_scale=20.0),
    "llama3_8b_gqa_b4": Workload("llama3_8b_gqa_b4", B=4, H_q=32, H_kv=8, D=128, T=32768,
                                 G=128, R=128, bits=4, seed=3, k_outlier_channels=6,
                                 k_outlier_scale=10.0, v_outlier_prob=0.001,
                                 v_outlier_scale=20.0),
    "kitty": Workload("kitty", B=16, H_q=32, H_kv=8, D=128, T=16384, G=128, R=128, bits=2,
                      S=32, n_boost=16, mode="kitty", seed=4, k_outlier_channels=6,
                      k_outlier_scale=10.0, v_outlier_prob=0.001, v_outlier_scale=20.0),
    "long_128k": Workload("long_128k", B=1, H_q=32, H_kv=8, D=128, T=131072, G=128, R=128,
                          bits=2, seed=5, k_outlier_channels=6, k_outlier_scale=10.0),
}

# Key / value width variants of the Llama-3-8B GQA layer (the Kitty notes' K4V2,
# K2V4 and K2V2-with-sinks variants, Sec. 3.1, and 8-bit codes).
_GQA = dict(B=4, H_q=32, H_kv=8, D=128, T=32768, G=128, R=128, k_outlier_channels=6,
            k_outlier_scale=10.0, v_outlier_prob=0.001, v_outlier_scale=20.0)
WORKLOADS.update({
    "llama3_8b_gqa_k4v2": Workload("llama3_8b_gqa_k4v2", bits=4, v_bits=2, seed=6, **_GQA),
    "llama3_8b_gqa_k2v4": Workload("llama3_8b_gqa_k2v4", bits=2, v_bits=4, seed=7, **_GQA),
    "llama3_8b_gqa_k8v8": Workload("llama3_8b_gqa_k8v8", bits=8, seed=8, **_GQA),
    "llama3_8b_gqa_k2v2s": Workload("llama3_8b_gqa_k2v2s", bits=2, S=32, seed=9, **_GQA),
})

# Paged cache with per-sequence lengths: eight slots of the Llama-3-8B GQA heads whose
# lengths spread uniformly over 32768 * (1 +- 0.75) tokens (a continuous-batching mix).
WORKLOADS["llama3_8b_gqa_paged"] = Workload("llama3_8b_gqa_paged", bits=2, seed=10, ragged=0.75,
                                            **dict(_GQA, B=8))


# Pre-RoPE keys (KVQuant notes, mechanism two) on the Llama-3-8B GQA layer, with
# Llama-3's RoPE base.
WORKLOADS["llama3_8b_gqa_rope"] = Workload("llama3_8b_gqa_rope", bits=2, seed=11, rope_base=500000.0, **_GQA)

# NVFP4 pages (BitDecoding notes, Sec. V-D) on the Llama-3-8B GQA layer.
WORKLOADS["llama3_8b_gqa_nvfp4"] = Workload("llama3_8b_gqa_nvfp4", bits=4, seed=12, mode="nvfp4", **_GQA)


def slot_lengths(wl: Workload) -> np.ndarray:
    """Seeded per-slot prefill lengths of a paged workload: T * (1 + ragged * u),
    u uniform in [-1, 1], at least one token."""
    rng = _rng(wl, 7)
    u = rng.uniform(-1.0, 1.0, wl.B)
    return np.maximum(1, np.round(wl.T * (1.0 + wl.ragged * u))).astype(np.int64)


def _rng(wl: Workload, stream: int) -> np.random.Generator:
    # Independent, reproducible streams per purpose (prefill, decode tokens, queries).
    return np.random.Generator(np.random.PCG64([wl.seed, stream]))


def outlier_channels(wl: Workload) -> np.ndarray:
    """[H_kv, n] key channels that carry the large magnitudes (fixed per head)."""
    rng = _rng(wl, 0)
    n = wl.k_outlier_channels
    if n == 0:
        return np.zeros((wl.H_kv, 0), dtype=np.int64)
    return np.stack([rng.choice(wl.D, n, replace=False) for _ in range(wl.H_kv)])


def _fill_kv(wl: Workload, rng: np.random.Generator, L: int, chans: np.ndarray
             ) -> Tuple[np.ndarray, np.ndarray]:
    K = np.empty((wl.B, wl.H_kv, L, wl.D), dtype=np.float16)
    V = np.empty((wl.B, wl.H_kv, L, wl.D), dtype=np.float16)
    for b in range(wl.B):
        for h in range(wl.H_kv):
            k = rng.standard_normal((L, wl.D), dtype=np.float32)
            if chans.shape[1]:
                k[:, chans[h]] *= np.float32(wl.k_outlier_scale)
            K[b, h] = k.astype(np.float16)
            v = rng.standard_normal((L, wl.D), dtype=np.float32)
            if wl.v_outlier_prob > 0:
                m = rng.random(L) < wl.v_outlier_prob
                v[m] *= np.float32(wl.v_outlier_scale)
            V[b, h] = v.astype(np.float16)
    return K, V


def prefill_kv(wl: Workload, L0: int, replica: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """fp16 K, V of shape [B, H_kv, L0, D] for the prefill of one layer cache.

    ``replica`` selects an independent draw with the same recipe (used for the
    several layer caches a benchmark rotates through)."""
    return _fill_kv(wl, _rng(wl, 1 + 16 * replica), L0, outlier_channels(wl))


def decode_tokens(wl: Workload, n_steps: int, replica: int = 0
                  ) -> Tuple[np.ndarray, np.ndarray]:
    """fp16 new-token K, V of shape [n_steps, B, H_kv, D] (same recipe as prefill)."""
    K, V = _fill_kv(wl, _rng(wl, 2 + 16 * replica), n_steps, outlier_channels(wl))
    return (np.ascontiguousarray(K.transpose(2, 0, 1, 3)),
            np.ascontiguousarray(V.transpose(2, 0, 1, 3)))


def queries(wl: Workload, n_steps: int, replica: int = 0) -> np.ndarray:
    """fp16 queries of shape [n_steps, B, H_q, D], N(0,1)."""
    rng = _rng(wl, 3 + 16 * replica)
    return rng.standard_normal((n_steps, wl.B, wl.H_q, wl.D), dtype=np.float32).astype(np.float16)


def small(wl: Workload, **kw) -> Workload:
    """A reduced copy of a workload (same structure), for oracle-sized tests."""
    return wl.replace(**kw)


def random_fp16(rng: np.random.Generator, shape, scale: float = 1.0,
                special: Optional[str] = None) -> np.ndarray:
    """fp16 test values: N(0, scale^2), or a special pattern for edge cases.

    special: None | "const" (one value repeated per last axis) |
    "wide" (random magnitudes over the whole fp16 exponent range, both signs) |
    "tiny" (values near the fp16 subnormal range)."""
    if special is None:
        return (rng.standard_normal(shape, dtype=np.float32) * np.float32(scale)).astype(np.float16)
    if special == "const":
        base = rng.standard_normal(shape[:-1], dtype=np.float32).astype(np.float16)
        return np.repeat(base[..., None], shape[-1], axis=-1)
    if special == "wide":
        bits = rng.integers(0, 0x7C00, size=shape, dtype=np.uint16)  # finite magnitudes
        sign = rng.integers(0, 2, size=shape, dtype=np.uint16) << 15
        return (bits | sign).view(np.float16)
    if special == "tiny":
        bits = rng.integers(0, 0x0800, size=shape, dtype=np.uint16)  # |x| < 2^-13
        sign = rng.integers(0, 2, size=shape, dtype=np.uint16) << 15
        return (bits | sign).view(np.float16)
    raise ValueError(special)
