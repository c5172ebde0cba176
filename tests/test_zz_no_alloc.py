"""kvq_decode_attn_noalloc (decode attention on the library's own fixed scratch
region, for callers that cannot hand out device memory) against kvq_decode_attn with
a caller workspace and against the CPU oracle, through the C ABI.

Decode is deterministic (a CTA's partial goes to a slot fixed by the schedule, and the
slots are combined in order), so the two entry points must agree bit for bit.

Collected last on purpose: it must pass both in a fresh process (its first call
sets the region up) and after every other GPU test has run in the same process."""
import ctypes

import numpy as np
import pytest

import kvq_synth
import oracle
from kvq_synth import WORKLOADS
from parity_util import TOL_ABS, TOL_REL, to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

CASES = {
    "gqa_b2": (WORKLOADS["llama3_8b_gqa_b2"].replace(B=2, H_q=16, H_kv=4, T=1024), 1024 + 100),
    "gqa_b4": (WORKLOADS["llama3_8b_gqa_b4"].replace(B=2, H_q=16, H_kv=4, T=1024), 1024 + 100),
    "kitty": (WORKLOADS["kitty"].replace(B=2, H_q=16, H_kv=4, T=1024), 32 + 1024 + 128 + 60),
    "tiny_kivi": (WORKLOADS["tiny_kivi"], 256 + 31),
    # 128 sequences: their counters reach past where a 4-sequence call puts partials
    "many_seqs": (WORKLOADS["llama3_8b_gqa_b2"].replace(B=16, H_q=32, H_kv=8, T=256), 256 + 40),
}


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_gb300 as m
    return m


def _noalloc(kvq, cache, q, out):
    import torch
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return kvq.lib.kvq_decode_attn_noalloc(ctypes.byref(cache.cfg), ctypes.byref(cache.c),
                                           ctypes.c_void_p(q.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()), stream)


def _setup(kvq, name):
    wl, L0 = CASES[name]
    K, V = kvq_synth.prefill_kv(wl, L0)
    cache = kvq.KVQCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R,
                         n_boost=wl.n_boost, mode=wl.mode, max_T=wl.T + 4 * wl.G, device=DEV)
    cache.prefill(to_dev(K, DEV), to_dev(V, DEV))
    ora = oracle.OracleCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R,
                             n_boost=wl.n_boost, mode=wl.mode)
    ora.prefill(K, V)
    qh = kvq_synth.queries(wl, 1, replica=5)[0]
    return cache, qh, ora.attend(qh)


def _check(kvq, cache, qh, want, calls=2):
    """`calls` no-alloc calls in a row, each equal bit for bit to kvq_decode_attn with a
    fresh caller workspace and within tolerance of the oracle."""
    import torch
    q = to_dev(qh, DEV)
    ref = cache.decode_attn(q)
    outs = []
    for _ in range(calls):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(kvq, cache, q, out) == 0
        outs.append(out)
    torch.cuda.synchronize()
    assert cache.read_status() == 0          # the no-alloc calls report into cache->status
    r = ref.cpu().numpy()
    for out in outs:
        o = out.cpu().numpy()
        assert np.array_equal(o.view(np.uint16), r.view(np.uint16))
        err = np.abs(o.astype(np.float64) - want)
        assert (err <= TOL_ABS + TOL_REL * np.abs(want)).all(), float(err.max())


@pytest.mark.parametrize("name", list(CASES))
def test_matches_workspace_entry_twice(kvq, name):
    cache, qh, want = _setup(kvq, name)
    _check(kvq, cache, qh, want)


def test_configurations_in_turn(kvq):
    """Small, large, small sequence counts one after the other on the shared region: each
    call finds its counters at zero although the previous call laid the region out
    differently."""
    small = _setup(kvq, "tiny_kivi")
    large = _setup(kvq, "many_seqs")
    for c in (small, large, small, large):
        _check(kvq, *c, calls=1)


def test_refuses_a_workspace_beyond_the_region(kvq):
    cfg = kvq.make_config(B=512, H_q=32, H_kv=32, D=128, G=128, bits=2, R=128, max_T=1024)
    need = kvq.lib.kvq_decode_attn_workspace_bytes(ctypes.byref(cfg))
    assert need > 16 * 1024 * 1024
    cache, _, _ = _setup(kvq, "tiny_kivi")   # real buffers; only the configuration is too large
    rc = kvq.lib.kvq_decode_attn_noalloc(ctypes.byref(cfg), ctypes.byref(cache.c),
                                         ctypes.c_void_p(cache.buf["k_res"].data_ptr()),
                                         ctypes.c_void_p(cache.buf["v_res"].data_ptr()), None)
    assert rc == -4
