"""The kernels' bounded waits on a GPU, without a fault: a wait on an mbarrier that
nothing completes runs out, sets the timeout bit in the status word the host reads, and
the context stays usable (a decode call afterwards matches the oracle)."""
import time

import numpy as np
import pytest

import kvq_synth
from kvq_synth import WORKLOADS
from parity_util import assert_close, make_pair, prefill_both, to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_gb300 as m
    return m


def test_wait_runs_out_and_reports(kvq):
    import ctypes
    import torch
    status = torch.zeros(4, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    assert kvq.lib.kvq_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), stream) == 0
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status[0].item()) & kvq.KVQ_DEV_TIMEOUT
    assert int(status[1:].abs().sum().item()) == 0
    assert 0.5 < dt < 30.0                            # the kernels' bound: about 2 s
    # the context is still usable: one decode call against the oracle
    wl = WORKLOADS["tiny_kivi"]
    gpu, ora = make_pair(wl, wl.T + 4 * wl.G, DEV)
    K, V = kvq_synth.prefill_kv(wl, wl.T + 29)
    prefill_both(gpu, ora, K, V, DEV)
    q = kvq_synth.queries(wl, 1)[0]
    out = gpu.decode_attn(to_dev(q, DEV)).float().cpu().numpy()
    assert_close(out, ora.attend(q))
    assert gpu.read_status() == 0
