"""kvq_decode_step_host (one decode step from host buffers: inputs in, append,
attend, flush, output out) against the same steps through the device-buffer calls (bit
for bit: decode is deterministic) and against the CPU oracle, over steps that cross a
flush of the residual."""
import numpy as np
import pytest

import kvq_synth
from kvq_synth import WORKLOADS
import oracle
from parity_util import assert_close, to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

CASES = {
    # prefill leaves R - 3 tokens in the residual: the fourth step flushes it
    "gqa_b2": (WORKLOADS["llama3_8b_gqa_b2"].replace(B=2, H_q=16, H_kv=4, T=1024), 1024 + 128 - 3),
    "kitty": (WORKLOADS["kitty"].replace(B=2, H_q=16, H_kv=4, T=1024), 32 + 1024 + 128 + 125),
    "tiny_kivi": (WORKLOADS["tiny_kivi"], 256 + 29),
}
STEPS = 6


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_gb300 as m
    return m


def _cache(kvq, wl, K, V):
    c = kvq.KVQCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R, n_boost=wl.n_boost,
                     mode=wl.mode, max_T=wl.T + 4 * wl.G, device=DEV)
    c.prefill(to_dev(K, DEV), to_dev(V, DEV))
    return c


@pytest.mark.parametrize("mode", ["mapped", "pageable", "wait"])
@pytest.mark.parametrize("name", list(CASES))
def test_host_step_matches_device_steps(kvq, name, mode):
    """Page-locked (mapped) host buffers are read and written by the kernels in place;
    pageable ones go through copies into the staging buffer.  wait: the blocking entry
    point, whose output is read as soon as the call returns (no synchronization)."""
    import torch
    pinned, wait = mode != "pageable", mode == "wait"

    def host_mem(t):
        return t.pin_memory() if pinned else t
    wl, L0 = CASES[name]
    K, V = kvq_synth.prefill_kv(wl, L0)
    kn, vn = kvq_synth.decode_tokens(wl, STEPS)
    qs = kvq_synth.queries(wl, STEPS, replica=3)
    dev, host = _cache(kvq, wl, K, V), _cache(kvq, wl, K, V)
    ora = oracle.OracleCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R,
                             n_boost=wl.n_boost, mode=wl.mode)
    ora.prefill(K, V)
    flushes = 0
    for i in range(STEPS):
        dev.append_token(to_dev(kn[i], DEV), to_dev(vn[i], DEV))
        ref = dev.decode_attn(to_dev(qs[i], DEV))
        fd = dev.flush_group()
        out = host_mem(torch.full(tuple(qs[i].shape), float("nan"), dtype=torch.float16))
        ref_u16 = ref.cpu().numpy().view(np.uint16)     # the device path, synchronized
        fh = host.step_host(host_mem(torch.from_numpy(qs[i])), host_mem(torch.from_numpy(kn[i])),
                            host_mem(torch.from_numpy(vn[i])), out, wait=wait)
        if wait:
            a = out.numpy().copy()                     # read before any synchronization
        torch.cuda.synchronize()
        assert fh == fd
        flushes += fd[0] or fd[1]
        if not wait:
            a = out.numpy()
        assert np.array_equal(a.view(np.uint16), ref_u16)
        ora.append(kn[i], vn[i])
        assert_close(a, ora.attend(qs[i]), what="host step %d" % i)
        assert ora.flush() == fh
        assert host.lengths == dev.lengths
    assert flushes >= 1
    for name_ in host.buf:                                # packed state and buffers: bit-exact
        assert torch.equal(host.buf[name_], dev.buf[name_]), name_
    assert host.read_status() == 0 and dev.read_status() == 0


def test_host_step_wait_refuses_unmapped(kvq):
    """The blocking entry point wants page-locked buffers and a page-locked count word;
    otherwise it refuses before it enqueues anything (the cache is unchanged)."""
    import torch
    wl, L0 = CASES["tiny_kivi"]
    K, V = kvq_synth.prefill_kv(wl, L0)
    c = _cache(kvq, wl, K, V)
    kn, vn = kvq_synth.decode_tokens(wl, 1)
    q = kvq_synth.queries(wl, 1)[0]
    out = torch.empty(tuple(q.shape), dtype=torch.float16).pin_memory()
    before = c.lengths
    with pytest.raises(kvq.KvqError):
        c.step_host(torch.from_numpy(q), torch.from_numpy(kn[0]).pin_memory(),
                    torch.from_numpy(vn[0]).pin_memory(), out, wait=True)   # q pageable
    assert c.lengths == before
    torch.cuda.synchronize()
    assert c.read_status() == 0
