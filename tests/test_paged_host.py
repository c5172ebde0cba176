"""Host-side checks of the paged-cache ABI (no GPU): buffer sizes follow the page-major
layouts, unsupported shapes are refused, the flush plan lists the slots whose residual
is full, and argument and capacity errors come back before anything is enqueued."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_gb300 as m
    return m


def _cfg(kvq, B=4, H_q=32, H_kv=8, D=128, G=128, bits=2, S=0, R=128, mode="kivi", max_T=4096, v_bits=0):
    return kvq.make_config(B, H_q, H_kv, D, G, bits, S, R, 0, mode, max_T, v_bits)


def _fake(kvq, cfg, lens):
    """A kvq_paged whose device pointers are aligned placeholders (never dereferenced
    by the host checks) and whose host lengths are `lens`."""
    p = kvq.Paged()
    for i, name in enumerate(("k_codes", "k_meta", "v_codes", "v_meta", "page_table", "k_sink", "v_sink",
                              "k_res", "v_res", "lens", "status")):
        setattr(p, name, 0x10000 * (i + 1))
    p.n_pages = 64
    host = (ctypes.c_int32 * (4 * cfg.B))(*[x for l in lens for x in l])
    p.lens_host = ctypes.cast(host, ctypes.c_void_p)
    return p, host


def test_paged_bytes_follow_page_layout(kvq):
    c = _cfg(kvq)
    L = kvq.lib
    P, H, D, G = 10, 8, 128, 128
    assert L.kvq_paged_bytes(ctypes.byref(c), P, 0) == P * H * (G // 16) * D * 4   # key codes
    assert L.kvq_paged_bytes(ctypes.byref(c), P, 3) == P * H * D * 4                # key (scale, min)
    assert L.kvq_paged_bytes(ctypes.byref(c), P, 4) == P * H * (D // 16) * G * 4    # value codes
    assert L.kvq_paged_bytes(ctypes.byref(c), P, 5) == P * H * G * 1 * 4            # value (scale, min)
    assert L.kvq_paged_bytes(ctypes.byref(c), P, 7) == 4 * H * 128 * D * 2          # key residual
    assert L.kvq_paged_bytes(ctypes.byref(c), P, 10) == 4 * 16
    assert L.kvq_paged_bytes(ctypes.byref(c), P, 11) == 4 * (4096 // 128) * 4
    # 4-bit keys, 8-bit values: the widths of each side
    c48 = _cfg(kvq, bits=4, v_bits=8)
    assert L.kvq_paged_bytes(ctypes.byref(c48), P, 0) == P * H * (G // 8) * D * 4
    assert L.kvq_paged_bytes(ctypes.byref(c48), P, 4) == P * H * (D // 4) * G * 4
    # the same codes as the dense layout: a page is 1/(max_T/G) of a dense sequence
    dense = L.kvq_buffer_bytes(ctypes.byref(c), 0) // (4 * 8)  # per (b, h)
    assert L.kvq_paged_bytes(ctypes.byref(c), 1, 0) == 8 * dense // (4096 // 128)


@pytest.mark.parametrize("kw", [dict(mode="kitty", R=64), dict(D=64), dict(B=513), dict(G=32, R=128),
                                dict(H_q=64, H_kv=8), dict(G=96, R=192)])
def test_paged_unsupported_shapes(kvq, kw):
    c = _cfg(kvq, **kw)
    assert kvq.lib.kvq_paged_bytes(ctypes.byref(c), 4, 0) == 0
    assert kvq.lib.kvq_paged_workspace_bytes(ctypes.byref(c)) == 0


def test_flush_plan_lists_full_residuals(kvq):
    c = _cfg(kvq)
    p, host = _fake(kvq, c, [(0, 256, 128, 1), (0, 0, 5, 1), (0, 0, 0, 0), (0, 128, 128, 1)])
    seqs = (ctypes.c_int32 * 4)()
    n = ctypes.c_int(-1)
    assert kvq.lib.kvq_paged_flush_plan(ctypes.byref(c), ctypes.byref(p), seqs, ctypes.byref(n)) == 0
    assert n.value == 2 and list(seqs[:2]) == [0, 3]


def test_paged_errors_before_any_launch(kvq):
    c = _cfg(kvq)
    L = kvq.lib
    full = [(0, 256, 128, 1), (0, 0, 5, 1), (0, 0, 0, 0), (0, 0, 7, 1)]
    p, host = _fake(kvq, c, full)
    before = list(host)
    # an append with a full residual is refused; the host lengths stay
    assert L.kvq_paged_append(ctypes.byref(c), ctypes.byref(p), ctypes.c_void_p(0x900000),
                              ctypes.c_void_p(0xA00000), None) == -3
    assert list(host) == before
    # prefill of an occupied slot, of a slot out of range, of zero tokens
    args = (ctypes.c_void_p(0x900000), ctypes.c_void_p(0xA00000))
    assert L.kvq_paged_prefill(ctypes.byref(c), ctypes.byref(p), 0, *args, 10, None) == -1
    assert L.kvq_paged_prefill(ctypes.byref(c), ctypes.byref(p), 4, *args, 10, None) == -1
    assert L.kvq_paged_prefill(ctypes.byref(c), ctypes.byref(p), 2, *args, 0, None) == -1
    # a packed part past max_T
    assert L.kvq_paged_prefill(ctypes.byref(c), ctypes.byref(p), 2, *args, 4096 + 128, None) == -3
    # misaligned pool pointer, null host lengths
    p.v_codes = 0x30004
    assert L.kvq_paged_flush(ctypes.byref(c), ctypes.byref(p), None, None) == -1
    p.v_codes = 0x30000
    # a too-small workspace
    q, out = ctypes.c_void_p(0xB00000), ctypes.c_void_p(0xC00000)
    assert L.kvq_paged_decode_attn(ctypes.byref(c), ctypes.byref(p), q, out, ctypes.c_void_p(0xD00000), 16,
                                   None) == -4
    # inconsistent host lengths (T not a multiple of G, a flag other than 0/1)
    bad, _h = _fake(kvq, c, [(0, 100, 0, 1), (0, 0, 0, 0), (0, 0, 0, 0), (0, 0, 0, 0)])
    assert L.kvq_paged_flush(ctypes.byref(c), ctypes.byref(bad), None, None) == -1
    bad2, _h2 = _fake(kvq, c, [(0, 0, 0, 2), (0, 0, 0, 0), (0, 0, 0, 0), (0, 0, 0, 0)])
    assert L.kvq_paged_flush(ctypes.byref(c), ctypes.byref(bad2), None, None) == -1
    # flush past max_T
    cap, _h3 = _fake(kvq, c, [(0, 4096, 128, 1), (0, 0, 0, 0), (0, 0, 0, 0), (0, 0, 0, 0)])
    assert L.kvq_paged_flush(ctypes.byref(c), ctypes.byref(cap), None, None) == -3


def test_paged_decode_of_no_active_slot_enqueues_nothing(kvq):
    c = _cfg(kvq)
    p, host = _fake(kvq, c, [(0, 0, 0, 0)] * 4)
    wsb = kvq.lib.kvq_paged_workspace_bytes(ctypes.byref(c))
    assert wsb > 0
    q, out, ws = ctypes.c_void_p(0xB00000), ctypes.c_void_p(0xC00000), ctypes.c_void_p(0xD00000)
    assert kvq.lib.kvq_paged_decode_attn(ctypes.byref(c), ctypes.byref(p), q, out, ws, wsb, None) == 0
