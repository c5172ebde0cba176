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

KVQ_MODE_KIVI, KVQ_MODE_KITTY, KVQ_MODE_NVFP4 = 0, 1, 2
KVQ_DEV_TIMEOUT, KVQ_DEV_BAD_STATE = 1, 2  # device status-word bits
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported configuration",
          -3: "capacity exceeded", -4: "workspace missing or too small", -5: "CUDA error",
          -6: "device-side error reported"}
BUFFERS = ("k_codes", "k_hi", "k_bidx", "k_meta", "v_codes", "v_meta", "k_sink", "k_res",
           "v_res", "v_local")
EXPORTS = ("kvq_status_str", "kvq_config_check", "kvq_buffer_bytes", "kvq_quant_pack_k",
           "kvq_quant_pack_v", "kvq_append_token", "kvq_flush_group",
           "kvq_decode_attn_workspace_bytes", "kvq_workspace_init", "kvq_decode_attn",
           "kvq_read_status", "kvq_decode_attn_noalloc", "kvq_step_io_bytes", "kvq_decode_step_host",
           "kvq_decode_step_host_wait", "kvq_selftest_wait_timeout", "kvq_append_decode",
           "kvq_paged_bytes", "kvq_paged_init",
           "kvq_paged_prefill", "kvq_paged_append", "kvq_paged_flush_plan", "kvq_paged_flush",
           "kvq_paged_release", "kvq_paged_workspace_bytes", "kvq_paged_decode_attn",
           "kvq_paged_read_status")
PAGED_MAX_B = 512


class KvqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s: %s (%d)" % (what, STATUS.get(code, "unknown"), code))
        self.code = code


class Config(ctypes.Structure):
    """kvq_config"""
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "H_q", "H_kv", "D", "G", "bits", "S", "R",
                                              "n_boost", "mode", "v_bits")] + [("max_T", ctypes.c_int64)] + \
               [("rope", ctypes.c_int32), ("rope_base", ctypes.c_float)]


class Cache(ctypes.Structure):
    """kvq_cache"""
    _fields_ = [(n, ctypes.c_void_p) for n in ("k_codes", "k_hi", "k_bidx", "k_meta", "v_codes",
                                               "v_meta", "k_sink", "v_sink", "k_res", "v_res",
                                               "v_local", "status")] + \
               [(n, ctypes.c_int64) for n in ("n_sink", "T_k", "n_kres", "T_v", "n_vres",
                                              "n_local", "local_head")]


class Paged(ctypes.Structure):
    """kvq_paged"""
    _fields_ = [(n, ctypes.c_void_p) for n in ("k_codes", "k_meta", "v_codes", "v_meta")] + \
               [("n_pages", ctypes.c_int64)] + \
               [(n, ctypes.c_void_p) for n in ("page_table", "k_sink", "v_sink", "k_res", "v_res", "lens",
                                               "lens_host", "status")]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError("libkvq.so not built (%s); run: python bit_kv_cache_gb300/build.py" % path)
    L = ctypes.CDLL(path)
    P, I, I64, Sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    CP, KP, PP = ctypes.POINTER(Config), ctypes.POINTER(Cache), ctypes.POINTER(Paged)
    IP = ctypes.POINTER(I)
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
        "kvq_step_io_bytes": ([CP], Sz),
        "kvq_append_decode": ([CP, KP, P, P, P, P, P, Sz, IP, P], I),
        "kvq_decode_step_host": ([CP, KP, P, P, P, P, P, Sz, P, Sz, IP, IP, P], I),
        "kvq_decode_step_host_wait": ([CP, KP, P, P, P, P, P, P, Sz, IP, IP, P], I),
        "kvq_selftest_wait_timeout": ([P, P], I),
        "kvq_paged_bytes": ([CP, I64, I], Sz),
        "kvq_paged_init": ([CP, PP, P], I),
        "kvq_paged_prefill": ([CP, PP, I, P, P, I64, P], I),
        "kvq_paged_append": ([CP, PP, P, P, P], I),
        "kvq_paged_flush_plan": ([CP, PP, ctypes.POINTER(ctypes.c_int32), IP], I),
        "kvq_paged_flush": ([CP, PP, IP, P], I),
        "kvq_paged_release": ([CP, PP, I, P], I),
        "kvq_paged_workspace_bytes": ([CP], Sz),
        "kvq_paged_decode_attn": ([CP, PP, P, P, P, Sz, P], I),
        "kvq_paged_read_status": ([PP, P, ctypes.POINTER(ctypes.c_int32), P], I),
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


def v_tile_tokens(cfg) -> int:
    """Tokens per value tile of a page (the library's value pages are tile-major): 256 /
    key bits when that divides G, else G."""
    t = 256 // (2 if cfg.mode == KVQ_MODE_KITTY else cfg.bits)
    return t if cfg.G % t == 0 else cfg.G


def make_config(B, H_q, H_kv, D, G, bits, S=0, R=None, n_boost=0, mode="kivi", max_T=0,
                v_bits=0, rope_base=0.0) -> Config:
    """rope_base > 0: keys are stored before RoPE and rotated in decode attention."""
    m = {"kivi": KVQ_MODE_KIVI, "kitty": KVQ_MODE_KITTY, "nvfp4": KVQ_MODE_NVFP4}[mode]
    return Config(B, H_q, H_kv, D, G, bits, S, G if R is None else R, n_boost, m, v_bits or 0, max_T,
                  1 if rope_base else 0, float(rope_base or 0.0))


class KVQCache:
    """One attention layer's low-bit KV cache in device memory.

    Buffers are allocated with torch on ``device`` at the sizes the library reports
    (kvq_buffer_bytes); the library itself never allocates.  All calls enqueue on the
    current torch stream."""

    def __init__(self, B, H_q, H_kv, D, G, bits, S=0, R=None, n_boost=0, mode="kivi",
                 max_T=0, device="cuda", v_bits=0, rope_base=0.0):
        import torch
        self.torch = torch
        self.cfg = make_config(B, H_q, H_kv, D, G, bits, S, R, n_boost, mode, max_T, v_bits, rope_base)
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
        # staging of kvq_decode_step_host (q, k_new, v_new, out of one step)
        self.io = torch.empty(lib.kvq_step_io_bytes(ctypes.byref(self.cfg)), dtype=torch.uint8,
                              device=self.device)
        self.done = None  # completion count of kvq_decode_step_host_wait (page-locked, made on first use)

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

    def append_decode(self, q, k_new, v_new, out=None) -> Tuple[object, bool]:
        """Insert the token and attend (kvq_append_decode); returns (out, fused), fused
        telling whether one launch did both."""
        torch = self.torch
        shp, shk = (self.cfg.B, self.cfg.H_q, self.cfg.D), (self.cfg.B, self.cfg.H_kv, self.cfg.D)
        if out is None:
            out = torch.empty(shp, dtype=torch.float16, device=self.device)
        fused = ctypes.c_int(0)
        _check(lib.kvq_append_decode(ctypes.byref(self.cfg), ctypes.byref(self.c),
                                     self._ptr(k_new, shk, "k_new"), self._ptr(v_new, shk, "v_new"),
                                     self._ptr(q, shp, "q"), self._ptr(out, shp, "out"),
                                     ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(),
                                     ctypes.byref(fused), self._stream()), "kvq_append_decode")
        return out, bool(fused.value)

    def step(self, q, k_new, v_new, out=None):
        """One decode step in the Kitty pipeline order: insert, attend, flush."""
        out, _ = self.append_decode(q, k_new, v_new, out)
        self.flush_group()
        return out

    def step_host(self, q, k_new, v_new, out, wait=False):
        """One decode step from host tensors (kvq_decode_step_host): q, out [B, H_q, D],
        k_new, v_new [B, H_kv, D], contiguous float16 on the CPU (page-locked for the
        copies to be asynchronous).  Enqueued on the current stream; out holds the
        result once the stream is synchronized.  wait (kvq_decode_step_host_wait; all
        four tensors page-locked): returns once out holds the result.  Returns
        (flushed_k, flushed_v)."""
        torch = self.torch
        for t, shp, what in ((q, (self.cfg.B, self.cfg.H_q, self.cfg.D), "q"),
                             (out, (self.cfg.B, self.cfg.H_q, self.cfg.D), "out"),
                             (k_new, (self.cfg.B, self.cfg.H_kv, self.cfg.D), "k_new"),
                             (v_new, (self.cfg.B, self.cfg.H_kv, self.cfg.D), "v_new")):
            if t.device.type != "cpu" or t.dtype != torch.float16 or not t.is_contiguous() or \
                    tuple(t.shape) != shp:
                raise ValueError("%s must be a contiguous float16 CPU tensor of shape %s" % (what, shp))
        fk, fv = ctypes.c_int(0), ctypes.c_int(0)
        if wait:
            if self.done is None:
                self.done = torch.zeros(1, dtype=torch.int32).pin_memory()
            _check(lib.kvq_decode_step_host_wait(ctypes.byref(self.cfg), ctypes.byref(self.c),
                                                 ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_new.data_ptr()),
                                                 ctypes.c_void_p(v_new.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                                 ctypes.c_void_p(self.done.data_ptr()),
                                                 ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(),
                                                 ctypes.byref(fk), ctypes.byref(fv), self._stream()),
                   "kvq_decode_step_host_wait")
            return bool(fk.value), bool(fv.value)
        _check(lib.kvq_decode_step_host(ctypes.byref(self.cfg), ctypes.byref(self.c),
                                        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_new.data_ptr()),
                                        ctypes.c_void_p(v_new.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                        ctypes.c_void_p(self.io.data_ptr()), self.io.numel(),
                                        ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(),
                                        ctypes.byref(fk), ctypes.byref(fv), self._stream()),
               "kvq_decode_step_host")
        return bool(fk.value), bool(fv.value)

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
        if cfg.mode == KVQ_MODE_NVFP4:  # codes [B][H][T][D/2]; page records of 16 + G*D/16 bytes
            b = self.buf[name]
            ms = 16 + G * D // 16
            if name in ("k_codes", "v_codes"):
                return b[: U * T * D // 2].view(cfg.B, cfg.H_kv, T, D // 2)
            if name in ("k_meta", "v_meta"):
                return b[: U * (T // G) * ms].view(cfg.B, cfg.H_kv, T // G, ms)
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
        if name == "v_codes":  # tile-major pages: [G / TV][D / fpi rows][TV words]
            TV = v_tile_tokens(cfg)
            return b.view(torch.int32).view(cfg.B, cfg.H_kv, T // G, G // TV, D // vfpi, TV)
        if name == "v_meta":
            return b.view(torch.float16).view(cfg.B, cfg.H_kv, T, D // Gv, 2)
        rows = {"k_sink": cfg.S, "v_sink": cfg.S, "k_res": G if kitty else cfg.R,
                "v_res": G if kitty else cfg.R, "v_local": cfg.R if kitty else 0}[name]
        return b[: U * rows * D * 2].view(torch.float16).view(cfg.B, cfg.H_kv, rows, D)


class KVQPagedCache:
    """A paged low-bit KV cache (KIVI mode): B batch slots of their own lengths over a
    pool of n_pages physical pages, each holding one group of G tokens of all H_kv
    heads of one slot.  The page table and the pool live in torch device memory; this
    class keeps the free list on the host and writes the table rows a slot needs before
    the library packs into them (prefill, flush).  ``max_T`` is the packed-token
    capacity of one slot."""

    def __init__(self, B, H_q, H_kv, D, G, bits, n_pages, max_T, S=0, R=None, device="cuda", v_bits=0):
        import torch
        self.torch = torch
        self.cfg = make_config(B, H_q, H_kv, D, G, bits, S, R, 0, "kivi", max_T, v_bits)
        self.device = torch.device(device)
        self.n_pages = n_pages
        cp = ctypes.byref(self.cfg)
        self.p = Paged()
        self.buf = {}
        for name, which in (("k_codes", 0), ("k_meta", 3), ("v_codes", 4), ("v_meta", 5), ("k_sink", 6),
                            ("v_sink", 6), ("k_res", 7), ("v_res", 8)):
            n = lib.kvq_paged_bytes(cp, n_pages, which)
            if n == 0 and which in (0, 3, 4, 5, 7, 8) and n_pages > 0:
                raise KvqError(-2, "paged config")
            t = torch.zeros(max(n, 16), dtype=torch.uint8, device=self.device)
            self.buf[name] = t
            setattr(self.p, name, t.data_ptr() if n else None)
        self.max_pages = max_T // G
        self.table = torch.zeros((B, self.max_pages), dtype=torch.int32, device=self.device)
        self.lens = torch.zeros((B, 4), dtype=torch.int32, device=self.device)
        self.lens_host = (ctypes.c_int32 * (4 * B))()
        self.status = torch.zeros(4, dtype=torch.int32, device=self.device)
        self.p.n_pages = n_pages
        self.p.page_table = self.table.data_ptr()
        self.p.lens = self.lens.data_ptr()
        self.p.lens_host = ctypes.cast(self.lens_host, ctypes.c_void_p)
        self.p.status = self.status.data_ptr()
        self.ws = torch.zeros(lib.kvq_paged_workspace_bytes(cp), dtype=torch.uint8, device=self.device)
        self.free = list(range(n_pages - 1, -1, -1))  # pop() hands out the lowest id first
        self.pages = [[] for _ in range(B)]           # physical pages of each slot, logical order
        _check(lib.kvq_paged_init(cp, ctypes.byref(self.p), KVQCache._stream()), "paged init")

    def _ptr(self, t, shape, what):
        return KVQCache._ptr(self, t, shape, what)

    def lengths(self, b) -> dict:
        l = self.lens_host[4 * b: 4 * b + 4]
        return {"n_sink": l[0], "T": l[1], "n_res": l[2], "active": l[3]}

    def _map(self, b, n):
        """Maps the next n logical pages of slot b to free physical pages."""
        if len(self.free) < n:
            raise KvqError(-3, "page pool exhausted")
        j0 = len(self.pages[b])
        new = [self.free.pop() for _ in range(n)]
        self.pages[b].extend(new)
        if n:
            self.table[b, j0:j0 + n] = self.torch.tensor(new, dtype=self.torch.int32)

    def prefill(self, b, k, v):
        """k, v: float16 [H_kv][L0][D] of batch slot b (empty)."""
        cfg = self.cfg
        L0 = k.shape[1]
        self._ptr(k, (cfg.H_kv, L0, cfg.D), "k")
        self._ptr(v, (cfg.H_kv, L0, cfg.D), "v")
        if self.lens_host[4 * b + 3]:
            raise KvqError(-1, "prefill of an occupied slot")
        ns = min(cfg.S, L0)
        self._map(b, (L0 - ns) // cfg.G)
        _check(lib.kvq_paged_prefill(ctypes.byref(self.cfg), ctypes.byref(self.p), b, ctypes.c_void_p(k.data_ptr()),
                                     ctypes.c_void_p(v.data_ptr()), L0, KVQCache._stream()), "paged prefill")

    def append(self, k_new, v_new):
        cfg = self.cfg
        kp = self._ptr(k_new, (cfg.B, cfg.H_kv, cfg.D), "k_new")
        vp = self._ptr(v_new, (cfg.B, cfg.H_kv, cfg.D), "v_new")
        _check(lib.kvq_paged_append(ctypes.byref(self.cfg), ctypes.byref(self.p), kp, vp, KVQCache._stream()),
               "paged append")

    def flush(self) -> list:
        """Packs every full residual into new pages; returns the flushed slots."""
        cfg = self.cfg
        seqs = (ctypes.c_int32 * cfg.B)()
        n = ctypes.c_int(0)
        _check(lib.kvq_paged_flush_plan(ctypes.byref(self.cfg), ctypes.byref(self.p), seqs, ctypes.byref(n)),
               "flush plan")
        out = list(seqs[: n.value])
        for b in out:
            self._map(b, cfg.R // cfg.G)
        nf = ctypes.c_int(0)
        _check(lib.kvq_paged_flush(ctypes.byref(self.cfg), ctypes.byref(self.p), ctypes.byref(nf),
                                   KVQCache._stream()), "paged flush")
        return out

    def release(self, b):
        self.free.extend(reversed(self.pages[b]))
        self.pages[b] = []
        _check(lib.kvq_paged_release(ctypes.byref(self.cfg), ctypes.byref(self.p), b, KVQCache._stream()),
               "paged release")

    def decode_attn(self, q, out=None):
        cfg = self.cfg
        qp = self._ptr(q, (cfg.B, cfg.H_q, cfg.D), "q")
        if out is None:
            out = self.torch.zeros_like(q)
        op = self._ptr(out, (cfg.B, cfg.H_q, cfg.D), "out")
        _check(lib.kvq_paged_decode_attn(ctypes.byref(self.cfg), ctypes.byref(self.p), qp, op,
                                         ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(),
                                         KVQCache._stream()), "paged decode")
        return out

    def read_status(self) -> int:
        st = ctypes.c_int32(0)
        lib.kvq_paged_read_status(ctypes.byref(self.p), ctypes.c_void_p(self.ws.data_ptr()), ctypes.byref(st),
                                  KVQCache._stream())
        return st.value

    def view(self, name: str):
        """Typed views of the page pools ([n_pages][H_kv] ...) and the fp16 buffers."""
        torch = self.torch
        cfg = self.cfg
        P, H, D, G = self.n_pages, cfg.H_kv, cfg.D, cfg.G
        kfpi, vfpi, Gv = 32 // cfg.bits, 32 // (cfg.v_bits or cfg.bits), min(G, D)
        b = self.buf[name]
        if name == "k_codes":
            return b.view(torch.int32).view(P, H, G // kfpi, D)
        if name == "k_meta":
            return b.view(torch.float16).view(P, H, D, 2)
        if name == "v_codes":  # tile-major pages: [G / TV][D / fpi rows][TV words]
            TV = v_tile_tokens(cfg)
            return b.view(torch.int32).view(P, H, G // TV, D // vfpi, TV)
        if name == "v_meta":
            return b.view(torch.float16).view(P, H, G, D // Gv, 2)
        rows = {"k_sink": cfg.S, "v_sink": cfg.S, "k_res": cfg.R, "v_res": cfg.R}[name]
        return b[: cfg.B * H * rows * D * 2].view(torch.float16).view(cfg.B, H, rows, D)
