"""CPU oracle for the low-bit KV cache (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` leg of ``bench.py`` import this package.  It never imports
the CUDA package and shares no code with it.

The arithmetic lives in ``kvq_oracle.c`` (plain single-threaded C, fp32
quantizer with IEEE division, fp64 dequantization and attention).  This module
compiles it with the host ``cc``, loads it with ctypes, and adds the cache
bookkeeping of the three-stage decode pipeline described on the Kitty page
(Sec. 4.3: insert the new token into a full-precision buffer, attend, then
quantize a buffer that has filled up) and the prefill split of the KIVI page
(Step 3: after prefill the cache is divided into a low-bit part and an FP16
residual part).

Oracle functions and their pins (``tests/test_oracle.py``):
  f16 <-> f32 conversions   -- exhaustive / sampled against numpy's float16 cast
  quant_group               -- error bound, exact level grids, constant groups,
                               brute force over a small fp16 alphabet, zero range
  pack layout (quant_k/v)   -- the KIVI page's worked example (column 19 -> word 1,
                               shift 6), the [B,nh,T,D] -> [B,nh,T/16,D] shape
                               example, round trip
  Kitty select / planes     -- brute-force top-k, n_boost=0 equals KIVI 2-bit,
                               n_boost=D equals KIVI 4-bit after lo|hi<<2
  attend                    -- quantization off equals a textbook loop on tiny
                               inputs, one-token cache, uniform logits, permutation
                               invariance, long-double cross-check
  bytes accounting          -- the KV-cache size formula and the pages' tables
  rope (``tests/test_oracle_rope.py``)
                            -- D = 2 is the textbook rotation, the complex form with
                               the KVQuant page's theta_i, scores depend only on the
                               relative position, norms, pairs and the group law,
                               attention against numpy over complex-rotated keys
  e2m1 / e4m3, nvfp4_page, nvfp4_dequant (``tests/test_oracle_nvfp4.py``)
                            -- brute force over every representable value (nearest,
                               ties to even, saturation), page scales and codes
                               recomputed in numpy float32, the error bound, attention
                               over an NVFP4 cache against the textbook formula

Parity unpinned: the codes that running the KIVI page's fp16 quantization snippet
literally would give in near-tie cases.  The oracle follows the fp32 definition
(scale rounded once to fp16, then fp32 IEEE division) instead, and the pins above
tie that definition down.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkvq_oracle.so")
_CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-Wall", "-shared", "-fPIC"]

_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False) -> str:
    """Compile the oracle library (cc, no GPU).  Returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call(["cc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Seq(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("D", "G", "bits", "Gv", "n_boost", "kitty", "vbits")] + \
               [(n, ctypes.c_long) for n in ("n_sink", "T_k", "n_kres", "T_v", "n_vres",
                                             "n_local", "local_head", "local_cap")] + \
               [(n, ctypes.c_void_p) for n in ("k_sink", "v_sink", "k_codes", "k_hi", "k_bidx",
                                               "k_meta", "k_res", "v_codes", "v_meta", "v_res",
                                               "v_local")] + [("rope_base", ctypes.c_double)]


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I, Lg = ctypes.c_int, ctypes.c_long
        L.kvq_or_h2f_array.argtypes = [P, P, Lg]
        L.kvq_or_f2h_array.argtypes = [P, P, Lg]
        L.kvq_or_quant_group.argtypes = [P, Lg, I, I, P, P, P]
        L.kvq_or_quant_k.argtypes = [P, I, Lg, I, I, I, Lg, Lg, P, P]
        L.kvq_or_quant_v.argtypes = [P, I, Lg, I, I, I, Lg, Lg, P, P]
        L.kvq_or_quant_k_kitty.argtypes = [P, I, Lg, I, I, I, Lg, Lg, P, P, P, P]
        L.kvq_or_kitty_select.argtypes = [P, I, I, I, P, P]
        L.kvq_or_seq_rows.argtypes = [ctypes.POINTER(_Seq), P, P]
        L.kvq_or_seq_len.argtypes = [ctypes.POINTER(_Seq)]
        L.kvq_or_seq_len.restype = Lg
        L.kvq_or_attend.argtypes = [P, I, P, P, Lg, I, P]
        L.kvq_or_rope.argtypes = [P, Lg, I, ctypes.c_double, Lg]
        L.kvq_or_seq_attend.argtypes = [ctypes.POINTER(_Seq), P, I, P]
        L.kvq_or_seq_attend.restype = I
        D_ = ctypes.c_double
        L.kvq_or_small_float_value.argtypes = [I, I, I, I]
        L.kvq_or_small_float_value.restype = D_
        L.kvq_or_small_float_code.argtypes = [D_, I, I, I, D_]
        L.kvq_or_small_float_code.restype = I
        L.kvq_or_nvfp4_page_k.argtypes = [P, I, I, P, P, P]
        L.kvq_or_nvfp4_page_v.argtypes = [P, I, I, P, P, P]
        L.kvq_or_nvfp4_dequant.argtypes = [P, P, ctypes.c_float, I, I, I, P]
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _u16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    assert x.dtype == np.uint16
    return x


# --------------------------------------------------------------------------- #
# Element functions                                                            #
# --------------------------------------------------------------------------- #

def h2f(h: np.ndarray) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, np.float32)
    lib().kvq_or_h2f_array(_p(h), _p(out), h.size)
    return out


def f2h(f: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 bits (uint16), round to nearest even."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().kvq_or_f2h_array(_p(f), _p(out), f.size)
    return out


def quant_group(x: np.ndarray, bits: int = 2, max_int: Optional[int] = None):
    """Quantize one 1-D fp16 group.  Returns (scale fp16, min fp16, codes uint8)."""
    x = _u16(x)
    mi = (1 << bits) - 1 if max_int is None else max_int
    s = np.zeros(1, np.uint16)
    m = np.zeros(1, np.uint16)
    c = np.zeros(x.size, np.uint8)
    lib().kvq_or_quant_group(_p(x), 1, x.size, mi, _p(s), _p(m), _p(c))
    return s.view(np.float16)[0], m.view(np.float16)[0], c


def dequant(codes, scale, mn) -> np.ndarray:
    """code*scale + min in fp64 (the page's dequantization)."""
    return np.asarray(codes, np.float64) * np.float64(scale) + np.float64(mn)


# --------------------------------------------------------------------------- #
# Tensor quantizers (layouts of the KIVI page: K packed along tokens,          #
# V packed along channels)                                                     #
# --------------------------------------------------------------------------- #

def quant_k(k: np.ndarray, G: int, bits: int, t0: int = 0, T: Optional[int] = None):
    """k: fp16 [B,H,L,D].  Returns codes int32 [B,H,T/fpi,D], meta fp16 [B,H,T/G,D,2]."""
    B, H, L, D = k.shape
    T = L - t0 if T is None else T
    fpi = 32 // bits
    assert T % G == 0 and G % fpi == 0
    k = _u16(k)
    codes = np.zeros((B, H, T // fpi, D), np.int32)
    meta = np.zeros((B, H, T // G, D, 2), np.uint16)
    lib().kvq_or_quant_k(_p(k), B * H, L, D, G, bits, t0, T, _p(codes), _p(meta))
    return codes, meta.view(np.float16)


def quant_v(v: np.ndarray, Gv: int, bits: int, t0: int = 0, T: Optional[int] = None):
    """v: fp16 [B,H,L,D].  Returns codes int32 [B,H,T,D/fpi], meta fp16 [B,H,T,D/Gv,2]."""
    B, H, L, D = v.shape
    T = L - t0 if T is None else T
    fpi = 32 // bits
    assert D % Gv == 0 and Gv % fpi == 0
    v = _u16(v)
    codes = np.zeros((B, H, T, D // fpi), np.int32)
    meta = np.zeros((B, H, T, D // Gv, 2), np.uint16)
    lib().kvq_or_quant_v(_p(v), B * H, L, D, Gv, bits, t0, T, _p(codes), _p(meta))
    return codes, meta.view(np.float16)


def quant_k_kitty(k: np.ndarray, G: int, n_boost: int, t0: int = 0, T: Optional[int] = None):
    """Kitty key pages.  Returns lo int32 [B,H,T/16,D], hi int32 [B,H,T/16,n_boost],
    bidx uint8 [B,H,T/G,D], meta fp16 [B,H,T/G,D,2]."""
    B, H, L, D = k.shape
    T = L - t0 if T is None else T
    assert T % G == 0 and G % 16 == 0
    k = _u16(k)
    lo = np.zeros((B, H, T // 16, D), np.int32)
    hi = np.zeros((B, H, T // 16, max(n_boost, 0)), np.int32)
    bidx = np.zeros((B, H, T // G, D), np.uint8)
    meta = np.zeros((B, H, T // G, D, 2), np.uint16)
    lib().kvq_or_quant_k_kitty(_p(k), B * H, L, D, G, n_boost, t0, T, _p(lo),
                               _p(hi) if n_boost else 0, _p(bidx), _p(meta))
    return lo, hi, bidx, meta.view(np.float16)


def kitty_select(page: np.ndarray, n_boost: int):
    """page: fp16 [G, D].  Returns (score int64 [D] in units of 2^-24, bidx uint8 [D])."""
    page = _u16(page)
    G, D = page.shape
    score = np.zeros(D, np.int64)
    bidx = np.zeros(D, np.uint8)
    lib().kvq_or_kitty_select(_p(page), G, D, n_boost, _p(score), _p(bidx))
    return score, bidx


def rope(K: np.ndarray, base: float = 10000.0, t0: int = 0) -> np.ndarray:
    """Rotary position embedding of K [L, D] (row i at position t0 + i), fp64: channel
    pair (2j, 2j+1) turns by (t0 + i) * base^(-2j/D) (KVQuant notes, mechanism two)."""
    out = np.array(K, np.float64, copy=True, order="C")
    lib().kvq_or_rope(_p(out), out.shape[0], out.shape[1], float(base), int(t0))
    return out


# --------------------------------------------------------------------------- #
# NVFP4 pages (see kvq_oracle.c for the reading of the format)                 #
# --------------------------------------------------------------------------- #

def small_float_value(code: int, ebits: int, mbits: int, bias: int) -> float:
    return lib().kvq_or_small_float_value(int(code), ebits, mbits, bias)


def small_float_code(x: float, ebits: int, mbits: int, bias: int, maxv: float) -> int:
    return lib().kvq_or_small_float_code(float(x), ebits, mbits, bias, float(maxv))


def e2m1_code(x: float) -> int:
    return small_float_code(x, 2, 1, 1, 6.0)


def e4m3_code(x: float) -> int:
    return small_float_code(x, 4, 3, 7, 448.0)


def nvfp4_page(x: np.ndarray, values: bool):
    """One page fp16 [G][D] -> (codes uint8 [G][D/2], scales uint8 ([G][D/16] for keys,
    [G/16][D] for values), S float32)."""
    x = np.ascontiguousarray(_u16(x))
    G, D = x.shape
    codes = np.zeros((G, D // 2), np.uint8)
    scales = np.zeros((G // 16, D) if values else (G, D // 16), np.uint8)
    S = ctypes.c_float(0.0)
    fn = lib().kvq_or_nvfp4_page_v if values else lib().kvq_or_nvfp4_page_k
    fn(_p(x), G, D, _p(codes), _p(scales), ctypes.byref(S))
    return codes, scales, np.float32(S.value)


def nvfp4_dequant(codes: np.ndarray, scales: np.ndarray, S: float, values: bool) -> np.ndarray:
    G, D = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((G, D), np.float64)
    lib().kvq_or_nvfp4_dequant(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(scales)),
                               float(S), G, D, int(values), _p(out))
    return out


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """fp64 softmax attention. q: [n_heads, D], K, V: [L, D] (any float dtype)."""
    q = np.ascontiguousarray(q, np.float64)
    K = np.ascontiguousarray(K, np.float64)
    V = np.ascontiguousarray(V, np.float64)
    out = np.zeros(q.shape, np.float64)
    lib().kvq_or_attend(_p(q), q.shape[0], _p(K), _p(V), K.shape[0], K.shape[1], _p(out))
    return out


# --------------------------------------------------------------------------- #
# The cache: prefill split, append, flush, attend                              #
# --------------------------------------------------------------------------- #

class OracleCache:
    """The whole cache of one attention layer, in the oracle's own layouts.

    Modes:
      "kivi":  keys and values each keep [sink | packed | fp16 residual (cap R)];
               a residual that holds R tokens is quantized into R/G groups.
      "kitty": keys keep [sink | packed | Q-buffer (cap G)]; values keep
               [sink | packed | Q-buffer (cap G) | local window (last R tokens)];
               a new value enters the local window, whose oldest token moves into
               the value Q-buffer once the window is full (Kitty page, Sec. 4.3,
               step (1)); keys use the two-plane INT4/INT2 pages when n_boost > 0.
    The per-sequence lengths are the same for every (b, h_kv).
    """

    def __init__(self, B, H_q, H_kv, D, G, bits, S=0, R=None, n_boost=0, mode="kivi",
                 max_T=None, v_bits=None, rope_base=0.0):
        assert mode in ("kivi", "kitty", "nvfp4")
        self.nvfp4 = mode == "nvfp4"
        assert not self.nvfp4 or (bits == 4 and (not v_bits or v_bits == 4)), "NVFP4 codes are 4-bit"
        self.B, self.H_q, self.H_kv, self.D, self.G, self.bits = B, H_q, H_kv, D, G, bits
        self.vbits = bits if not v_bits else v_bits  # value codes may use their own width
        self.rope_base = float(rope_base)  # > 0: keys stored before RoPE, rotated when attended
        self.S, self.R, self.n_boost, self.mode = S, (G if R is None else R), n_boost, mode
        self.Gv = min(G, D)
        self.kitty = mode == "kitty"
        assert not self.kitty or bits == 2, "Kitty pages are 2-bit planes"
        self.cap_kres = G if self.kitty else self.R
        self.cap_vres = G if self.kitty else self.R
        U = (B, H_kv)
        z16 = lambda n: np.zeros(U + (n, D), np.float16)
        self.k_sink, self.v_sink = z16(S), z16(S)
        self.k_res, self.v_res = z16(self.cap_kres), z16(self.cap_vres)
        self.v_local = z16(self.R if self.kitty else 0)
        fpi = 32 // self.vbits
        self.k_codes = np.zeros(U + (0, D), np.int32)
        self.k_hi = np.zeros(U + (0, n_boost), np.int32)
        self.k_bidx = np.zeros(U + (0, D), np.uint8)
        self.k_meta = np.zeros(U + (0, D, 2), np.float16)
        self.v_codes = np.zeros(U + (0, D // fpi), np.int32)
        self.v_meta = np.zeros(U + (0, D // self.Gv, 2), np.float16)
        self.n_sink = self.T_k = self.n_kres = self.T_v = self.n_vres = 0
        self.n_local = self.local_head = 0
        if self.nvfp4:  # codes [T][D/2]; key scales [T][D/16], value scales [T/16][D]; S per page
            self.k_codes = np.zeros(U + (0, D // 2), np.uint8)
            self.k_scales = np.zeros(U + (0, D // 16), np.uint8)
            self.k_S = np.zeros(U + (0,), np.float32)
            self.v_codes = np.zeros(U + (0, D // 2), np.uint8)
            self.v_scales = np.zeros(U + (0, D), np.uint8)
            self.v_S = np.zeros(U + (0,), np.float32)

    # -- packing helpers ---------------------------------------------------- #
    def _pack_nvfp4(self, src: np.ndarray, values: bool):
        B, H, n, D = src.shape
        G = self.G
        c = np.zeros((B, H, n, D // 2), np.uint8)
        sc = np.zeros((B, H, n // 16, D) if values else (B, H, n, D // 16), np.uint8)
        S = np.zeros((B, H, n // G), np.float32)
        for b in range(B):
            for h in range(H):
                for j in range(n // G):
                    cc, ss, S[b, h, j] = nvfp4_page(src[b, h, j * G:(j + 1) * G], values)
                    c[b, h, j * G:(j + 1) * G] = cc
                    if values:
                        sc[b, h, j * G // 16:(j + 1) * G // 16] = ss
                    else:
                        sc[b, h, j * G:(j + 1) * G] = ss
        return c, sc, S

    def _pack_k(self, src: np.ndarray):
        """Quantize src fp16 [B,H,n*G,D] as n key groups appended at the tail."""
        if src.shape[2] == 0:
            return
        if self.nvfp4:
            c, sc, S = self._pack_nvfp4(src, False)
            self.k_codes = np.concatenate([self.k_codes, c], 2)
            self.k_scales = np.concatenate([self.k_scales, sc], 2)
            self.k_S = np.concatenate([self.k_S, S], 2)
            self.T_k += src.shape[2]
            return
        if self.kitty:
            lo, hi, bi, mt = quant_k_kitty(src, self.G, self.n_boost)
            self.k_codes = np.concatenate([self.k_codes, lo], 2)
            self.k_hi = np.concatenate([self.k_hi, hi], 2)
            self.k_bidx = np.concatenate([self.k_bidx, bi], 2)
        else:
            c, mt = quant_k(src, self.G, self.bits)
            self.k_codes = np.concatenate([self.k_codes, c], 2)
        self.k_meta = np.concatenate([self.k_meta, mt], 2)
        self.T_k += src.shape[2]

    def _pack_v(self, src: np.ndarray):
        if src.shape[2] == 0:
            return
        if self.nvfp4:
            c, sc, S = self._pack_nvfp4(src, True)
            self.v_codes = np.concatenate([self.v_codes, c], 2)
            self.v_scales = np.concatenate([self.v_scales, sc], 2)
            self.v_S = np.concatenate([self.v_S, S], 2)
            self.T_v += src.shape[2]
            return
        c, mt = quant_v(src, self.Gv, self.vbits)
        self.v_codes = np.concatenate([self.v_codes, c], 2)
        self.v_meta = np.concatenate([self.v_meta, mt], 2)
        self.T_v += src.shape[2]

    # -- the API ------------------------------------------------------------ #
    def prefill(self, K: np.ndarray, V: np.ndarray):
        """Split an fp16 prefill [B,H_kv,L0,D] into sink, packed groups and buffers."""
        L0 = K.shape[2]
        ns = min(self.S, L0)
        self.k_sink[:, :, :ns] = K[:, :, :ns]
        self.v_sink[:, :, :ns] = V[:, :, :ns]
        self.n_sink = ns
        rest = L0 - ns
        tk = rest // self.G * self.G
        self._pack_k(np.ascontiguousarray(K[:, :, ns:ns + tk]))
        self.n_kres = rest - tk
        assert self.n_kres <= self.cap_kres
        self.k_res[:, :, :self.n_kres] = K[:, :, ns + tk:]
        if not self.kitty:
            self._pack_v(np.ascontiguousarray(V[:, :, ns:ns + tk]))
            self.n_vres = rest - tk
            self.v_res[:, :, :self.n_vres] = V[:, :, ns + tk:]
        else:
            nl = min(self.R, rest)
            older = rest - nl
            tv = older // self.G * self.G
            self._pack_v(np.ascontiguousarray(V[:, :, ns:ns + tv]))
            self.n_vres = older - tv
            self.v_res[:, :, :self.n_vres] = V[:, :, ns + tv:ns + older]
            self.v_local[:, :, :nl] = V[:, :, ns + older:]
            self.n_local, self.local_head = nl, 0

    def append(self, k_new: np.ndarray, v_new: np.ndarray):
        """Insert one token (fp16 [B,H_kv,D]) into the full-precision buffers."""
        if self.n_sink < self.S:
            self.k_sink[:, :, self.n_sink] = k_new
            self.v_sink[:, :, self.n_sink] = v_new
            self.n_sink += 1
            return
        assert self.n_kres < self.cap_kres, "key buffer full: flush first"
        self.k_res[:, :, self.n_kres] = k_new
        self.n_kres += 1
        if not self.kitty:
            assert self.n_vres < self.cap_vres
            self.v_res[:, :, self.n_vres] = v_new
            self.n_vres += 1
        elif self.n_local < self.R:
            self.v_local[:, :, (self.local_head + self.n_local) % self.R] = v_new
            self.n_local += 1
        else:
            assert self.n_vres < self.cap_vres, "value Q-buffer full: flush first"
            self.v_res[:, :, self.n_vres] = self.v_local[:, :, self.local_head]
            self.n_vres += 1
            self.v_local[:, :, self.local_head] = v_new
            self.local_head = (self.local_head + 1) % self.R

    def flush(self):
        """Quantize every buffer that is full.  Returns (flushed_k, flushed_v)."""
        fk = fv = False
        if self.n_kres == self.cap_kres:
            self._pack_k(np.ascontiguousarray(self.k_res))
            self.n_kres, fk = 0, True
        if self.n_vres == self.cap_vres:
            self._pack_v(np.ascontiguousarray(self.v_res))
            self.n_vres, fv = 0, True
        return fk, fv

    @property
    def L(self) -> int:
        return self.n_sink + self.T_k + self.n_kres

    def _seq(self, b: int, h: int, keep: List):
        def ptr(a):
            a = np.ascontiguousarray(a)
            keep.append(a)
            return a.ctypes.data if a.size else None
        s = _Seq()
        s.D, s.G, s.bits, s.Gv, s.n_boost, s.kitty = (self.D, self.G, self.bits, self.Gv,
                                                       self.n_boost, int(self.kitty))
        s.vbits = self.vbits
        s.n_sink, s.T_k, s.n_kres = self.n_sink, self.T_k, self.n_kres
        s.T_v, s.n_vres, s.n_local = self.T_v, self.n_vres, self.n_local
        s.local_head, s.local_cap = self.local_head, max(self.v_local.shape[2], 1)
        s.k_sink, s.v_sink = ptr(self.k_sink[b, h]), ptr(self.v_sink[b, h])
        s.k_codes, s.k_hi = ptr(self.k_codes[b, h]), ptr(self.k_hi[b, h])
        s.k_bidx, s.k_meta = ptr(self.k_bidx[b, h]), ptr(self.k_meta[b, h])
        s.k_res = ptr(self.k_res[b, h])
        s.v_codes, s.v_meta = ptr(self.v_codes[b, h]), ptr(self.v_meta[b, h])
        s.v_res, s.v_local = ptr(self.v_res[b, h]), ptr(self.v_local[b, h])
        s.rope_base = self.rope_base
        return s

    def _nvfp4_rows(self, b: int, h: int):
        G, D = self.G, self.D
        parts_k = [self.k_sink[b, h, :self.n_sink].astype(np.float64)]
        parts_v = [self.v_sink[b, h, :self.n_sink].astype(np.float64)]
        for j in range(self.T_k // G):
            parts_k.append(nvfp4_dequant(self.k_codes[b, h, j * G:(j + 1) * G],
                                         self.k_scales[b, h, j * G:(j + 1) * G], self.k_S[b, h, j], False))
            parts_v.append(nvfp4_dequant(self.v_codes[b, h, j * G:(j + 1) * G],
                                         self.v_scales[b, h, j * G // 16:(j + 1) * G // 16], self.v_S[b, h, j], True))
        parts_k.append(self.k_res[b, h, :self.n_kres].astype(np.float64))
        parts_v.append(self.v_res[b, h, :self.n_vres].astype(np.float64))
        return np.concatenate(parts_k, 0), np.concatenate(parts_v, 0)

    def rows(self, b: int, h: int):
        """Dequantized fp64 keys and values [L, D] of one sequence, logical order."""
        if self.nvfp4:
            return self._nvfp4_rows(b, h)
        keep: List = []
        s = self._seq(b, h, keep)
        Kh = np.zeros((self.L, self.D), np.float64)
        Vh = np.zeros((self.L, self.D), np.float64)
        lib().kvq_or_seq_rows(ctypes.byref(s), _p(Kh), _p(Vh))
        return Kh, Vh

    def attend(self, q: np.ndarray, units: Optional[Sequence] = None, threads: int = 1) -> np.ndarray:
        """q fp16 [B,H_q,D] -> fp64 [B,H_q,D] (NaN for units not requested).  threads > 1
        runs the (b, h_kv) units on a thread pool (each unit's arithmetic unchanged)."""
        g = self.H_q // self.H_kv
        out = np.full((self.B, self.H_q, self.D), np.nan)
        if units is None:
            units = [(b, h) for b in range(self.B) for h in range(self.H_kv)]
        if threads > 1 and len(units) > 1:
            from concurrent.futures import ThreadPoolExecutor
            with ThreadPoolExecutor(min(threads, len(units))) as ex:
                parts = list(ex.map(lambda u: self.attend(q, [u]), units))
            for (b, h), o in zip(units, parts):
                out[b, h * g:(h + 1) * g] = o[b, h * g:(h + 1) * g]
            return out
        for b, h in units:
            if self.nvfp4:
                Kh, Vh = self._nvfp4_rows(b, h)
                if self.rope_base > 0:
                    Kh = rope(Kh, self.rope_base, 0)
                out[b, h * g:(h + 1) * g] = attend(q[b, h * g:(h + 1) * g].astype(np.float64), Kh, Vh)
                continue
            keep: List = []
            s = self._seq(b, h, keep)
            qh = np.ascontiguousarray(_u16(q[b, h * g:(h + 1) * g]))
            o = np.zeros((g, self.D), np.float64)
            rc = lib().kvq_or_seq_attend(ctypes.byref(s), _p(qh), g, _p(o))
            assert rc == 0, "oracle out of memory"
            out[b, h * g:(h + 1) * g] = o
        return out


# --------------------------------------------------------------------------- #
# Bytes accounting (the KV-cache size formula of the KIVI / KVQuant pages)      #
# --------------------------------------------------------------------------- #

def fp16_cache_bytes(layers: int, batch: int, seq_len: int, kv_heads: int, head_dim: int,
                     elem_bytes: float = 2) -> float:
    """2 * layers * batch * seq_len * kv_heads * head_dim * bytes (K and V)."""
    return 2 * layers * batch * seq_len * kv_heads * head_dim * elem_bytes


def kivi_avg_bits(bits: int, G: int, R: int, L: int) -> float:
    """Average stored bits per element of a KIVI cache of length L: b-bit codes plus an
    fp16 (scale, min) pair per group of G, with the last R tokens kept in fp16."""
    packed = bits + 32.0 / G
    return (packed * (L - R) + 16.0 * R) / L
