"""Host-side checks of the C ABI: the library loads, exports every declared entry
point, and rejects bad arguments before touching the GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(kvq):
    names = _declared()
    assert "kvq_decode_attn" in names and len(names) >= 11
    for n in names:
        assert hasattr(kvq.lib, n), n
    assert sorted(kvq.EXPORTS) == names


def test_status_strings(kvq):
    for code, text in kvq.STATUS.items():
        assert kvq.lib.kvq_status_str(code).decode() == text


def _cfg(kvq, **kw):
    base = dict(B=2, H_q=8, H_kv=2, D=128, G=128, bits=2, S=0, R=128, n_boost=0, mode="kivi",
                max_T=1024)
    base.update(kw)
    return kvq.make_config(**base)


def test_config_check(kvq):
    ok = lambda **kw: kvq.lib.kvq_config_check(ctypes.byref(_cfg(kvq, **kw)))
    assert ok() == 0
    assert ok(bits=4) == 0 and ok(G=32, R=32) == 0
    assert ok(mode="kitty", S=32, n_boost=16) == 0
    assert ok(bits=3) == -2 and ok(bits=8) == 0 and ok(bits=1) == -2
    assert ok(v_bits=4) == 0 and ok(v_bits=8) == 0 and ok(v_bits=3) == -2
    assert ok(bits=4, v_bits=2) == 0 and ok(mode="kitty", S=32, v_bits=4) == 0
    assert ok(mode="kitty", bits=4) == -2
    assert ok(H_q=7) == -1                 # H_q % H_kv
    assert ok(H_q=32, H_kv=2) == -2        # 16 query heads per KV head
    assert ok(G=24, R=24) == -1            # G % 16 at 2 bits
    assert ok(R=100) == -1                 # KIVI residual must be a multiple of G
    assert ok(max_T=1000) == -1
    assert ok(n_boost=4) == -1             # boost only in Kitty mode
    assert ok(mode="kitty", n_boost=200) == -1
    assert ok(D=96) == -2
    assert ok(B=0) == -1
    assert kvq.lib.kvq_config_check(None) == -1


def test_buffer_bytes_match_layouts(kvq):
    c = _cfg(kvq, bits=2)
    bb = [kvq.lib.kvq_buffer_bytes(ctypes.byref(c), i) for i in range(10)]
    U, T, D, G = 4, 1024, 128, 128
    assert bb[0] == U * T * D * 2 // 8          # 2-bit key codes
    assert bb[1] == 0 and bb[2] == 0 and bb[9] == 0
    assert bb[3] == U * (T // G) * D * 4        # fp16 (scale, min) per channel per group
    assert bb[4] == U * T * D * 2 // 8
    assert bb[5] == U * T * 4                   # one (scale, min) per token
    assert bb[7] == bb[8] == U * 128 * D * 2
    k = _cfg(kvq, mode="kitty", S=32, n_boost=16)
    kb = [kvq.lib.kvq_buffer_bytes(ctypes.byref(k), i) for i in range(10)]
    assert kb[1] == U * (T // 16) * 16 * 4 and kb[2] == U * (T // G) * D
    assert kb[6] == U * 32 * D * 2 and kb[9] == U * 128 * D * 2


def test_buffer_bytes_of_separate_widths(kvq):
    U, T, D = 4, 1024, 128
    for kb, vb in ((4, 2), (2, 4), (8, 8), (2, 8)):
        c = _cfg(kvq, bits=kb, v_bits=vb)
        assert kvq.lib.kvq_buffer_bytes(ctypes.byref(c), 0) == U * T * D * kb // 8
        assert kvq.lib.kvq_buffer_bytes(ctypes.byref(c), 4) == U * T * D * vb // 8
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(_cfg(kvq, bits=4, v_bits=0)), 4) == U * T * D * 4 // 8


def test_argument_errors_before_any_launch(kvq):
    c = _cfg(kvq)
    cache = kvq.Cache()
    L = kvq.lib
    # null cache pointers, null inputs, zero length: all INVALID_ARG, nothing enqueued
    assert L.kvq_quant_pack_k(ctypes.byref(c), ctypes.byref(cache), None, 10, None) == -1
    assert L.kvq_append_token(ctypes.byref(c), ctypes.byref(cache), None, None, None) == -1
    assert L.kvq_decode_attn(ctypes.byref(c), ctypes.byref(cache), None, None, None, 0, None) == -1
    fk = ctypes.c_int(7)
    assert L.kvq_flush_group(ctypes.byref(c), None, ctypes.byref(fk), None, None) == -1
    assert fk.value == 7
    # misaligned pointers are rejected
    for name in ("k_codes", "k_meta", "v_codes", "v_meta", "k_res", "v_res"):
        setattr(cache, name, 0x1000)
    cache.k_codes = 0x1004
    assert L.kvq_quant_pack_k(ctypes.byref(c), ctypes.byref(cache), ctypes.c_void_p(0x2000), 10, None) == -1
    cache.k_codes = 0x1000
    # lengths inconsistent with the config
    cache.T_k = 100
    assert L.kvq_flush_group(ctypes.byref(c), ctypes.byref(cache), None, None, None) == -1
    cache.T_k = 0
    # empty cache cannot be attended
    assert L.kvq_decode_attn(ctypes.byref(c), ctypes.byref(cache), ctypes.c_void_p(0x3000),
                             ctypes.c_void_p(0x4000), ctypes.c_void_p(0x5000), 1 << 30, None) == -1
    # capacity: an append into a full residual is refused and lengths stay unchanged
    cache.T_k = cache.T_v = 128
    cache.n_kres = cache.n_vres = 128
    assert L.kvq_append_token(ctypes.byref(c), ctypes.byref(cache), ctypes.c_void_p(0x6000),
                              ctypes.c_void_p(0x7000), None) == -3
    assert cache.n_kres == 128
    # a too-small workspace is refused
    assert L.kvq_decode_attn(ctypes.byref(c), ctypes.byref(cache), ctypes.c_void_p(0x3000),
                             ctypes.c_void_p(0x4000), ctypes.c_void_p(0x5000), 16, None) == -4
    # flush past max_T
    cache.T_k = cache.T_v = 1024
    assert L.kvq_flush_group(ctypes.byref(c), ctypes.byref(cache), None, None, None) == -3


def test_workspace_size_grows_with_sequences(kvq):
    a = kvq.lib.kvq_decode_attn_workspace_bytes(ctypes.byref(_cfg(kvq, B=1)))
    b = kvq.lib.kvq_decode_attn_workspace_bytes(ctypes.byref(_cfg(kvq, B=8)))
    assert 0 < a < b


def test_step_io_bytes_and_refusals_before_any_copy(kvq):
    c = _cfg(kvq)                                   # B=2, H_q=8, H_kv=2, D=128
    nq, nk = 2 * 8 * 128 * 2, 2 * 2 * 128 * 2       # q / out and k_new / v_new bytes
    r256 = lambda n: (n + 255) // 256 * 256
    assert kvq.lib.kvq_step_io_bytes(ctypes.byref(c)) == 2 * r256(nq) + 2 * r256(nk)
    odd = _cfg(kvq, B=3, H_q=3, H_kv=1, D=64, G=32, R=32)
    assert kvq.lib.kvq_step_io_bytes(ctypes.byref(odd)) == 2 * r256(3 * 3 * 64 * 2) + 2 * r256(3 * 64 * 2)
    assert kvq.lib.kvq_step_io_bytes(ctypes.byref(_cfg(kvq, H_q=7))) == 0
    need = kvq.lib.kvq_step_io_bytes(ctypes.byref(c))
    f = kvq.lib.kvq_decode_step_host
    P = ctypes.c_void_p
    cache = kvq.Cache()
    host = P(0x1000)                                # never dereferenced: every case is refused first
    io = P(0x10000)

    def call(q=host, io_=io, io_bytes=need, cfg=c):
        return f(ctypes.byref(cfg), ctypes.byref(cache), q, host, host, host, io_, io_bytes, P(0x20000),
                 1 << 20, None, None, None)
    assert call(q=P(0)) == -1                       # a missing host buffer
    assert call(io_=P(0x10010)) == -1               # staging not 256-byte aligned
    assert call(io_bytes=need - 1) == -4            # staging too small
    assert call(cfg=_cfg(kvq, H_q=7)) == -1         # invalid configuration


def test_append_decode_refusals_before_any_launch(kvq):
    c = _cfg(kvq)
    P = ctypes.c_void_p
    f = kvq.lib.kvq_append_decode
    fused = ctypes.c_int(7)

    def call(cache, kn=P(0x1000), vn=P(0x2000), cfg=c):
        return f(ctypes.byref(cfg), ctypes.byref(cache), kn, vn, P(0x3000), P(0x4000), P(0x5000), 1 << 20,
                 ctypes.byref(fused), None)
    empty = kvq.Cache()                              # no buffers: refused by the pointer check
    assert call(empty) == -1 and fused.value == 0    # *fused is cleared first
    full = kvq.Cache()
    for name in ("k_codes", "k_meta", "v_codes", "v_meta", "k_res", "v_res"):
        setattr(full, name, 0x10000)                 # never dereferenced
    assert call(full, kn=P(0)) == -1                 # a missing new token
    assert call(full, vn=P(0x2008)) == -1            # misaligned value row
    assert call(full, cfg=_cfg(kvq, H_q=7)) == -1    # invalid configuration
    assert f(ctypes.byref(c), None, P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000), 1 << 20,
             None, None) == -1                       # no cache; fused may be NULL


def test_noalloc_refusals_before_any_launch(kvq):
    """The no-allocation decode entry point checks everything before it looks up its
    region or enqueues anything (fake pointers, never dereferenced)."""
    P = ctypes.c_void_p
    f = kvq.lib.kvq_decode_attn_noalloc
    c = _cfg(kvq)
    assert f(ctypes.byref(c), ctypes.byref(kvq.Cache()), P(0x3000), P(0x4000), None) == -1
    full = kvq.Cache()
    for name in ("k_codes", "k_meta", "v_codes", "v_meta", "k_res", "v_res"):
        setattr(full, name, 0x10000)
    full.T_k = full.T_v = 128
    full.n_kres = full.n_vres = 5
    assert f(ctypes.byref(c), ctypes.byref(full), P(0x3008), P(0x4000), None) == -1   # misaligned q
    assert f(ctypes.byref(c), ctypes.byref(full), P(0x3000), P(0x4000), None) == -1   # no status word
    full.status = 0x20000
    big = _cfg(kvq, B=512, H_q=32, H_kv=32, max_T=1024)
    assert kvq.lib.kvq_decode_attn_workspace_bytes(ctypes.byref(big)) > 16 * 1024 * 1024
    assert f(ctypes.byref(big), ctypes.byref(full), P(0x3000), P(0x4000), None) == -4


def test_step_host_wait_refusals_before_any_launch(kvq):
    """The blocking host step refuses missing, unaligned or unmapped buffers (fake
    pointers, never dereferenced) before it writes the count or enqueues anything."""
    P = ctypes.c_void_p
    f = kvq.lib.kvq_decode_step_host_wait
    c = _cfg(kvq)
    cache = kvq.Cache()
    done = ctypes.c_uint(7)

    def call(q=P(0x1000), d=ctypes.cast(ctypes.byref(done), P), cfg=c):
        return f(ctypes.byref(cfg), ctypes.byref(cache), q, P(0x1000), P(0x1000), P(0x1000), d, P(0x20000),
                 1 << 20, None, None, None)
    assert call(d=P(0)) == -1                         # no count word
    assert call(d=P(0x1002)) == -1                    # count word not 4-byte aligned
    assert call(q=P(0)) == -1                         # a missing host buffer
    assert call() == -1                               # not page-locked mapped memory
    assert call(cfg=_cfg(kvq, H_q=7)) == -1           # invalid configuration
    assert done.value == 7                            # the count was never written


def test_selftest_wait_refusals(kvq):
    """The bounded-wait self-test refuses a missing or misaligned status word before it
    launches anything."""
    P = ctypes.c_void_p
    f = kvq.lib.kvq_selftest_wait_timeout
    assert f(None, None) == -1
    assert f(P(0x1002), None) == -1
