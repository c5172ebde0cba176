"""kvq_append_decode (insert the token and attend, in one launch where the tile path
serves the call) against the oracle's append + attend, step by step across a flush,
and the cache state after the steps bit for bit."""
import numpy as np
import pytest

import kvq_synth
from kvq_synth import WORKLOADS
from parity_util import assert_close, assert_state_equal, make_pair, prefill_both, to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

# name: (workload, prefill length, steps, launches fused on every step?)
CASES = {
    # the prefill leaves R - 3 tokens in the residual: the third step fills it, the flush empties it
    "gqa_b2": (WORKLOADS["llama3_8b_gqa_b2"].replace(B=2, H_q=16, H_kv=4, T=512), 512 + 125, 6, True),
    "k4v4_pairs": (WORKLOADS["llama3_8b_gqa_b4"].replace(B=2, H_q=16, H_kv=4, T=512), 512 + 125, 5, True),
    "k8v2": (WORKLOADS["llama3_8b_gqa_b2"].replace(B=2, H_q=8, H_kv=2, T=256, bits=8, v_bits=2), 256 + 126, 4, True),
    "mha": (WORKLOADS["llama7b_mha"].replace(B=2, H_q=8, H_kv=8, T=256), 256 + 125, 5, True),
    "rope": (WORKLOADS["llama3_8b_gqa_rope"].replace(B=2, H_q=16, H_kv=4, T=512), 512 + 126, 4, True),
    "nvfp4": (WORKLOADS["llama3_8b_gqa_nvfp4"].replace(B=2, H_q=16, H_kv=4, T=256), 256 + 125, 5, True),
    # the sink fills during the first steps (those append separately), then one launch
    "sink_filling": (WORKLOADS["llama3_8b_gqa_b2"].replace(B=1, H_q=8, H_kv=2, T=256, S=8), 5, 6, None),
    # not served in one launch: Kitty (local window), the CUDA-core path (G = 32)
    "kitty": (WORKLOADS["kitty"].replace(B=2, H_q=16, H_kv=4, T=256), 32 + 256 + 128 + 126, 4, False),
    "tiny_generic": (WORKLOADS["tiny_kivi"], 256 + 29, 4, False),
}


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_gb300 as m
    return m


@pytest.mark.parametrize("name", list(CASES))
def test_append_decode_matches_oracle(kvq, name):
    wl, L0, steps, fused_expected = CASES[name]
    gpu, ora = make_pair(wl, wl.T + 4 * wl.G, DEV)
    K, V = kvq_synth.prefill_kv(wl, L0)
    prefill_both(gpu, ora, K, V, DEV)
    kn, vn = kvq_synth.decode_tokens(wl, steps)
    qs = kvq_synth.queries(wl, steps)
    flushes = 0
    for i in range(steps):
        sink_full = gpu.lengths["n_sink"] >= wl.S
        out, fused = gpu.append_decode(to_dev(qs[i], DEV), to_dev(kn[i], DEV), to_dev(vn[i], DEV))
        ora.append(kn[i], vn[i])
        want = sink_full if fused_expected is None else fused_expected
        assert fused == want, (i, fused)
        assert_close(out.float().cpu().numpy(), ora.attend(qs[i]), what="step %d" % i)
        fk, fv = gpu.flush_group()
        assert (fk, fv) == ora.flush()
        flushes += fk or fv
    if name not in ("sink_filling",):
        assert flushes >= 1
    assert_state_equal(gpu, ora)
    assert gpu.read_status() == 0
