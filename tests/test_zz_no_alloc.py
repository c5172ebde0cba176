"""kvq_decode_attn_noalloc (decode attention on the library's own fixed scratch
region) against kvq_decode_attn with a caller workspace, through the C ABI.

Collected last on purpose: it must pass both in a fresh process (its first call
sets the region up) and after every other GPU test has run in the same process."""
import ctypes

import numpy as np
import pytest

import kvq_synth
from kvq_synth import WORKLOADS
from parity_util import TOL_ABS, TOL_REL, to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

CASES = {
    "gqa_b2": (WORKLOADS["llama3_8b_gqa_b2"].replace(B=2, H_q=16, H_kv=4, T=1024), 1024 + 100),
    "gqa_b4": (WORKLOADS["llama3_8b_gqa_b4"].replace(B=2, H_q=16, H_kv=4, T=1024), 1024 + 100),
    "kitty": (WORKLOADS["kitty"].replace(B=2, H_q=16, H_kv=4, T=1024), 32 + 1024 + 128 + 60),
    "tiny_kivi": (WORKLOADS["tiny_kivi"], 256 + 31),
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


def _close(a, ref):
    a = a.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    err = np.abs(a - r)
    assert (err <= TOL_ABS + TOL_REL * np.abs(r)).all(), float(err.max())


@pytest.mark.parametrize("name", list(CASES))
def test_matches_workspace_entry_twice(kvq, name):
    import torch
    wl, L0 = CASES[name]
    K, V = kvq_synth.prefill_kv(wl, L0)
    cache = kvq.KVQCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R,
                         n_boost=wl.n_boost, mode=wl.mode, max_T=wl.T + 4 * wl.G, device=DEV)
    cache.prefill(to_dev(K, DEV), to_dev(V, DEV))
    q = to_dev(kvq_synth.queries(wl, 1, replica=5)[0], DEV)
    ref = cache.decode_attn(q)
    outs = []
    for _ in range(2):                                   # two calls in a row
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(kvq, cache, q, out) == 0
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        _close(out, ref)
    assert cache.read_status() == 0


def test_refuses_a_workspace_beyond_the_region(kvq):
    cfg = kvq.make_config(B=512, H_q=32, H_kv=32, D=128, G=128, bits=2, R=128, max_T=1024)
    need = kvq.lib.kvq_decode_attn_workspace_bytes(ctypes.byref(cfg))
    assert need > 16 * 1024 * 1024
    rc = kvq.lib.kvq_decode_attn_noalloc(ctypes.byref(cfg), ctypes.byref(kvq.Cache()),
                                         ctypes.c_void_p(0), ctypes.c_void_p(0), None)
    assert rc == -4
