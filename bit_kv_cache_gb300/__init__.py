"""Python binding of libkvq (GB300 low-bit KV cache).

Argument marshalling only: every step of quantization, packing, buffer updates
and attention runs in the library's CUDA kernels, reached through the C ABI in
``include/kvq.h``.  PyTorch provides device memory and the current stream.  There
is no CPU fallback: importing this package fails if ``libkvq.so`` is missing
(build it with ``python bit_kv_cache_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")

KVQ_MODE_KIVI, KVQ_MODE_KITTY = 0, 1
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported configuration",
          -3: "capacity exceeded", -4: "workspace missing or too small", -5: "CUDA error",
          -6: "device-side error reported"}
BUFFERS = ("k_codes", "k_hi", "k_bidx", "k_meta", "v_codes", "v_meta", "k_sink", "k_res",
           "v_res", "v_local")
EXPORTS = ("kvq_status_str", "kvq_config_check", "kvq_buffer_bytes", "kvq_quant_pack_k",
           "kvq_quant_pack_v", "kvq_append_token", "kvq_flush_group",
           "kvq_decode_attn_workspace_bytes", "kvq_workspace_init", "kvq_decode_attn",
           "kvq_read_status", "kvq_decode_attn_noalloc")


class KvqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s: %s (%d)" % (what, STATUS.get(code, "unknown"), code))
        self.code = code


class Config(ctypes.Structure):
    """kvq_config"""
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "H_q", "H_kv", "D", "G", "bits", "S", "R",
                                              "n_boost", "mode", "v_bits")] + [("max_T", ctypes.c_int64)]


class Cache(ctypes.Structure):
    """kvq_cache"""
    _fields_ = [(n, ctypes.c_void_p) for n in ("k_codes", "k_hi", "k_bidx", "k_meta", "v_codes",
                                               "v_meta", "k_sink", "v_sink", "k_res", "v_res",
                                               "v_local", "status")] + \
               [(n, ctypes.c_int64) for n in ("n_sink", "T_k", "n_kres", "T_v", "n_vres",
                                              "n_local", "local_head")]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError("libkvq.so not built (%s); run: python bit_kv_cache_gb300/build.py" % path)
    L = ctypes.CDLL(path)
    P, I, I64, Sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    CP, KP = ctypes.POINTER(Config), ctypes.POINTER(Cache)
    sig = {
        "kvq_status_str": ([I], ctypes.c_char_p),
        "kvq_config_check": ([CP], I),
        "kvq_buffer_bytes": ([CP, I], Sz),
        "kvq_quant_pack_k": ([CP, KP, P, I64, P], I),
        "kvq_quant_pack_v": ([CP, KP, P, I64, P], I),
        "kvq_append_token": ([CP, KP, P, P, P], I),
        "kvq_flush_group": ([CP, KP, ctypes.POINTER(I), ctypes.POINTER(I), P], I),
        "kvq_decode_attn_workspace_bytes": ([CP], Sz),
        "kvq_workspace_init": ([P, Sz, P], I),
        "kvq_decode_attn": ([CP, KP, P, P, P, Sz, P], I),
        "kvq_read_status": ([KP, P, ctypes.POINTER(ctypes.c_int32), P], I),
        "kvq_decode_attn_noalloc": ([CP, KP, P, P, P], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    return L


lib = load_library()


def _check(code: int, what: str):
    if code != 0:
        raise KvqError(code, what)


def make_config(B, H_q, H_kv, D, G, bits, S=0, R=None, n_boost=0, mode="kivi", max_T=0,
                v_bits=0) -> Config:
    m = {"kivi": KVQ_MODE_KIVI, "kitty": KVQ_MODE_KITTY}[mode]
    return Config(B, H_q, H_kv, D, G, bits, S, G if R is None else R, n_boost, m, v_bits or 0, max_T)


class KVQCache:
    """One attention layer's low-bit KV cache in device memory.

    Buffers are allocated with torch on ``device`` at the sizes the library reports
    (kvq_buffer_bytes); the library itself never allocates.  All calls enqueue on the
    current torch stream."""

    def __init__(self, B, H_q, H_kv, D, G, bits, S=0, R=None, n_boost=0, mode="kivi",
                 max_T=0, device="cuda", v_bits=0):
        import torch
        self.torch = torch
        self.cfg = make_config(B, H_q, H_kv, D, G, bits, S, R, n_boost, mode, max_T, v_bits)
        _check(lib.kvq_config_check(ctypes.byref(self.cfg)), "config")
        self.device = torch.device(device)
        self.c = Cache()
        self.buf = {}
        for i, name in enumerate(BUFFERS):
            n = lib.kvq_buffer_bytes(ctypes.byref(self.cfg), i)
            t = torch.zeros(max(n, 16), dtype=torch.uint8, device=self.device)
            self.buf[name] = t
            setattr(self.c, name, t.data_ptr() if n else None)
        vs = torch.zeros(max(self.buf["k_sink"].numel(), 16), dtype=torch.uint8, device=self.device)
        self.buf["v_sink"] = vs
        self.c.v_sink = vs.data_ptr() if self.cfg.S else None
        self.status = torch.zeros(4, dtype=torch.int32, device=self.device)
        self.c.status = self.status.data_ptr()
        wsb = lib.kvq_decode_attn_workspace_bytes(ctypes.byref(self.cfg))
        self.ws = torch.zeros(wsb, dtype=torch.uint8, device=self.device)  # zero-filled

    # -- helpers ------------------------------------------------------------- #
    @staticmethod
    def _stream():
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def _ptr(self, t, shape=None, what="tensor"):
        torch = self.torch
        if t.device != self.device or t.dtype != torch.float16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous float16 tensor on %s" % (what, self.device))
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError("%s has shape %s, expected %s" % (what, tuple(t.shape), tuple(shape)))
        return ctypes.c_void_p(t.data_ptr())

    @property
    def lengths(self) -> dict:
        c = self.c
        return dict(n_sink=c.n_sink, T_k=c.T_k, n_kres=c.n_kres, T_v=c.T_v, n_vres=c.n_vres,
                    n_local=c.n_local, local_head=c.local_head)

    @property
    def L(self) -> int:
        return self.c.n_sink + self.c.T_k + self.c.n_kres

    # -- the ABI ------------------------------------------------------------- #
    def quant_pack_k(self, k):
        B, Hkv, D = self.cfg.B, self.cfg.H_kv, self.cfg.D
        if k.dim() != 4 or tuple(k.shape[:2]) != (B, Hkv) or k.shape[3] != D:
            raise ValueError("k must be [B, H_kv, L0, D]")
        _check(lib.kvq_quant_pack_k(ctypes.byref(self.cfg), ctypes.byref(self.c),
                                    self._ptr(k, what="k"), k.shape[2], self._stream()),
               "kvq_quant_pack_k")

    def quant_pack_v(self, v):
        B, Hkv, D = self.cfg.B, self.cfg.H_kv, self.cfg.D
        if v.dim() != 4 or tuple(v.shape[:2]) != (B, Hkv) or v.shape[3] != D:
            raise ValueError("v must be [B, H_kv, L0, D]")
        _check(lib.kvq_quant_pack_v(ctypes.byref(self.cfg), ctypes.byref(self.c),
                                    self._ptr(v, what="v"), v.shape[2], self._stream()),
               "kvq_quant_pack_v")

    def prefill(self, k, v):
        self.quant_pack_k(k)
        self.quant_pack_v(v)

    def append_token(self, k_new, v_new):
        shp = (self.cfg.B, self.cfg.H_kv, self.cfg.D)
        _check(lib.kvq_append_token(ctypes.byref(self.cfg), ctypes.byref(self.c),
                                    self._ptr(k_new, shp, "k_new"), self._ptr(v_new, shp, "v_new"),
                                    self._stream()), "kvq_append_token")

    def flush_group(self) -> Tuple[bool, bool]:
        fk, fv = ctypes.c_int(0), ctypes.c_int(0)
        _check(lib.kvq_flush_group(ctypes.byref(self.cfg), ctypes.byref(self.c), ctypes.byref(fk),
                                   ctypes.byref(fv), self._stream()), "kvq_flush_group")
        return bool(fk.value), bool(fv.value)

    def decode_attn(self, q, out=None):
        torch = self.torch
        shp = (self.cfg.B, self.cfg.H_q, self.cfg.D)
        if out is None:
            out = torch.empty(shp, dtype=torch.float16, device=self.device)
        _check(lib.kvq_decode_attn(ctypes.byref(self.cfg), ctypes.byref(self.c),
                                   self._ptr(q, shp, "q"), self._ptr(out, shp, "out"),
                                   ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(),
                                   self._stream()), "kvq_decode_attn")
        return out

    def step(self, q, k_new, v_new, out=None):
        """One decode step in the Kitty pipeline order: insert, attend, flush."""
        self.append_token(k_new, v_new)
        out = self.decode_attn(q, out)
        self.flush_group()
        return out

    def read_status(self) -> int:
        st = ctypes.c_int32(0)
        lib.kvq_read_status(ctypes.byref(self.c), ctypes.c_void_p(self.ws.data_ptr()),
                            ctypes.byref(st), self._stream())
        return st.value

    # -- typed views of the buffers (for inspection and tests) ---------------- #
    def view(self, name: str):
        torch = self.torch
        cfg = self.cfg
        U, D, T, G = cfg.B * cfg.H_kv, cfg.D, cfg.max_T, cfg.G
        kitty = cfg.mode == KVQ_MODE_KITTY
        kfpi = 16 if kitty else 32 // cfg.bits
        vfpi = 32 // (cfg.v_bits or cfg.bits)
        Gv = min(G, D)
        b = self.buf[name]
        if name == "k_codes":
            return b.view(torch.int32).view(cfg.B, cfg.H_kv, T // kfpi, D)
        if name == "k_hi":
            return b[: U * (T // 16) * cfg.n_boost * 4].view(torch.int32).view(cfg.B, cfg.H_kv, T // 16, cfg.n_boost)
        if name == "k_bidx":
            return b[: U * (T // G) * D].view(cfg.B, cfg.H_kv, T // G, D)
        if name == "k_meta":
            return b.view(torch.float16).view(cfg.B, cfg.H_kv, T // G, D, 2)
        if name == "v_codes":
            return b.view(torch.int32).view(cfg.B, cfg.H_kv, T // G, D // vfpi, G)
        if name == "v_meta":
            return b.view(torch.float16).view(cfg.B, cfg.H_kv, T, D // Gv, 2)
        rows = {"k_sink": cfg.S, "v_sink": cfg.S, "k_res": G if kitty else cfg.R,
                "v_res": G if kitty else cfg.R, "v_local": cfg.R if kitty else 0}[name]
        return b[: U * rows * D * 2].view(torch.float16).view(cfg.B, cfg.H_kv, rows, D)
