"""GPU (CUDA kernels through the C ABI) against the CPU oracle.

Codes, scales, mins, boost indices and fp16 buffers must match bit for bit;
attention must satisfy |err| <= 2e-3 + 2e-3 |ref| element-wise.  Small cases span
several tiles and a ragged tail; the full-size cases use the workloads' own
shapes and the launch configuration bench.py times, and compare sampled
sequences (the oracle's attention over 32K-128K tokens is computed per sequence).
"""
import numpy as np
import pytest

import kvq_synth
from kvq_synth import WORKLOADS
from parity_util import (assert_close, assert_state_equal, make_pair, prefill_both, run_steps,
                         to_dev)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


# Reduced copies of the five workloads: same structure, several tiles, ragged tails.
SMALL = {
    "tiny_kivi": (WORKLOADS["tiny_kivi"], 256 + 31, 3),
    "llama7b_mha": (WORKLOADS["llama7b_mha"].replace(B=2, H_q=8, H_kv=8, T=512), 512 + 77, 4),
    "gqa_b2": (WORKLOADS["llama3_8b_gqa_b2"].replace(B=2, H_q=16, H_kv=4, T=1024), 1024 + 100, 4),
    "gqa_b4": (WORKLOADS["llama3_8b_gqa_b4"].replace(B=2, H_q=16, H_kv=4, T=1024), 1024 + 100, 4),
    "kitty": (WORKLOADS["kitty"].replace(B=2, H_q=16, H_kv=4, T=1024), 32 + 1024 + 128 + 60, 4),
    "long": (WORKLOADS["long_128k"].replace(T=2048), 2048 + 64, 3),
    # key / value width variants, all on the tensor-core tiles (keys set the tile:
    # 128, 64 or 32 tokens; values the PV steps)
    "k4v2": (WORKLOADS["llama3_8b_gqa_k4v2"].replace(B=2, H_q=16, H_kv=4, T=512), 512 + 70, 3),
    "k2v4": (WORKLOADS["llama3_8b_gqa_k2v4"].replace(B=2, H_q=16, H_kv=4, T=512), 512 + 70, 3),
    "k8v8": (WORKLOADS["llama3_8b_gqa_k8v8"].replace(B=2, H_q=16, H_kv=4, T=512), 512 + 70, 3),
    "k2v2s": (WORKLOADS["llama3_8b_gqa_k2v2s"].replace(B=2, H_q=16, H_kv=4, T=1024), 32 + 1024 + 70, 3),
    "k2v8": (WORKLOADS["llama3_8b_gqa_k8v8"].replace(B=2, H_q=16, H_kv=4, T=512, bits=2), 512 + 70, 2),
    "k8v2": (WORKLOADS["llama3_8b_gqa_k8v8"].replace(B=2, H_q=16, H_kv=4, T=512, v_bits=2), 512 + 70, 2),
    "k4v8": (WORKLOADS["llama3_8b_gqa_k8v8"].replace(B=2, H_q=16, H_kv=4, T=512, bits=4), 512 + 70, 2),
    "k8v4": (WORKLOADS["llama3_8b_gqa_k8v8"].replace(B=2, H_q=16, H_kv=4, T=512, v_bits=4), 512 + 70, 2),
    # G = 32: 8-bit keys fill one 32-token tile per page; 2-bit keys take the CUDA-core path
    "tiny_k8v2": (WORKLOADS["tiny_kivi"].replace(bits=8, v_bits=2), 256 + 31, 3),
    "tiny_k2v4": (WORKLOADS["tiny_kivi"].replace(v_bits=4), 256 + 31, 3),
    # pre-RoPE keys: the tile path (fp32 rotated QK on the CUDA cores, rotated fp16
    # tokens on tensor cores), widths, sinks, one query head per KV head, and the
    # CUDA-core path (G = 32 below a 2-bit tile)
    "rope_k2v2": (WORKLOADS["llama3_8b_gqa_rope"].replace(B=2, H_q=16, H_kv=4, T=1024), 1024 + 100, 4),
    "rope_k4v4_sink": (WORKLOADS["llama3_8b_gqa_rope"].replace(B=2, H_q=16, H_kv=4, T=512, bits=4, S=8,
                                                             rope_base=10000.0), 8 + 512 + 70, 3),
    "rope_k8v2": (WORKLOADS["llama3_8b_gqa_rope"].replace(B=2, H_q=16, H_kv=4, T=512, bits=8, v_bits=2),
                  512 + 70, 3),
    "rope_mha": (WORKLOADS["llama7b_mha"].replace(B=2, H_q=8, H_kv=8, T=512, rope_base=10000.0), 512 + 77, 3),
    "rope_tiny": (WORKLOADS["tiny_kivi"].replace(rope_base=10000.0), 256 + 31, 3),
    # NVFP4 pages (e2m1 codes, e4m3 block scales, fp32 page scale), CUDA-core decode
    "nvfp4": (WORKLOADS["llama3_8b_gqa_nvfp4"].replace(B=2, H_q=16, H_kv=4, T=256), 256 + 70, 3),
    "nvfp4_sink_g32": (WORKLOADS["llama3_8b_gqa_nvfp4"].replace(B=1, H_q=8, H_kv=2, T=128, G=32, R=64, S=4),
                       4 + 128 + 40, 3),
    "nvfp4_rope": (WORKLOADS["llama3_8b_gqa_nvfp4"].replace(B=1, H_q=8, H_kv=2, T=256, rope_base=10000.0),
                   256 + 50, 2),
    # three sequences of 20 tiles over ~56 warps: ranges cross sequences after odd
    # tile counts, so a unit's second segment starts with its mbarriers mid-phase
    "nvfp4_cross": (WORKLOADS["llama3_8b_gqa_nvfp4"].replace(B=3, H_q=4, H_kv=1, T=1280), 1280 + 30, 3),
    "k4v4_cross": (WORKLOADS["llama3_8b_gqa_b4"].replace(B=3, H_q=4, H_kv=1, T=1280), 1280 + 30, 3),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_prefill_state_and_attention(name):
    wl, L0, steps = SMALL[name]
    K, V = kvq_synth.prefill_kv(wl, L0)
    gpu, ora = make_pair(wl, max_T=wl.T + 4 * wl.G, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    assert_state_equal(gpu, ora)
    q = kvq_synth.queries(wl, 1, replica=7)[0]
    out = gpu.decode_attn(to_dev(q, DEV)).float().cpu().numpy()
    assert_close(out, ora.attend(q))
    run_steps(gpu, ora, wl, steps, DEV)
    assert_state_equal(gpu, ora)
    assert gpu.read_status() == 0


@pytest.mark.parametrize("name", ["gqa_b2", "kitty", "tiny_kivi", "rope_k2v2", "nvfp4_sink_g32", "nvfp4"])
def test_decode_loop_crosses_flushes(name):
    """Enough steps that every buffer fills and is flushed at least once."""
    wl, L0, _ = SMALL[name]
    K, V = kvq_synth.prefill_kv(wl, L0)
    gpu, ora = make_pair(wl, max_T=wl.T + 4 * wl.G, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    n = wl.G + 40
    run_steps(gpu, ora, wl, n, DEV, check_every=9)
    assert_state_equal(gpu, ora)


def test_long_decode_flush_on_step_64():
    """The long-context pattern: prefill T + 64, then 64 steps; the flush fires at 64."""
    wl = SMALL["long"][0]
    K, V = kvq_synth.prefill_kv(wl, wl.T + 64)
    gpu, ora = make_pair(wl, max_T=wl.T + 2 * wl.G, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    run_steps(gpu, ora, wl, 64, DEV, check_every=16)
    assert gpu.lengths["T_k"] == wl.T + wl.G and gpu.lengths["n_kres"] == 0
    assert_state_equal(gpu, ora)


@pytest.mark.parametrize("L0", [1, 5, 127, 128, 129, 256])
@pytest.mark.parametrize("mode", ["kivi", "kitty"])
def test_edge_lengths(L0, mode):
    """Single token, residual only, exact multiples of G, sink partly filled,
    local window not full."""
    base = WORKLOADS["kitty"] if mode == "kitty" else WORKLOADS["llama3_8b_gqa_b2"]
    wl = base.replace(B=1, H_q=8, H_kv=2, T=256)
    K, V = kvq_synth.prefill_kv(wl, L0)
    gpu, ora = make_pair(wl, max_T=1024, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    assert_state_equal(gpu, ora)
    run_steps(gpu, ora, wl, 40, DEV, check_every=7)
    assert_state_equal(gpu, ora)


def test_capacity_is_refused_and_state_kept():
    import bit_kv_cache_gb300 as kvq
    wl = WORKLOADS["llama3_8b_gqa_b2"].replace(B=1, H_q=8, H_kv=2, T=256)
    K, V = kvq_synth.prefill_kv(wl, 256 + 127)
    gpu, ora = make_pair(wl, max_T=256, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    kn, vn = kvq_synth.decode_tokens(wl, 2)
    gpu.append_token(to_dev(kn[0], DEV), to_dev(vn[0], DEV))
    before = gpu.lengths
    with pytest.raises(kvq.KvqError) as e:
        gpu.flush_group()
    assert e.value.code == -3 and gpu.lengths == before
    with pytest.raises(kvq.KvqError) as e:
        gpu.append_token(to_dev(kn[1], DEV), to_dev(vn[1], DEV))
    assert e.value.code == -3 and gpu.lengths == before


@pytest.mark.parametrize("special", ["wide", "tiny", "const", "ties"])
@pytest.mark.parametrize("bits,mode", [(2, "kivi"), (4, "kivi"), (2, "kitty")])
def test_quantizer_edge_values(special, bits, mode):
    """Bit-exact codes for values over the whole fp16 range, near-subnormal values,
    constant groups (scale 0, -0.0) and exact rounding ties (the IEEE-division path)."""
    rng = np.random.default_rng(hash((special, bits, mode)) % 2 ** 32)
    wl = WORKLOADS["kitty"].replace(B=1, H_q=2, H_kv=2, T=256, S=0, bits=bits, mode=mode,
                                    n_boost=16 if mode == "kitty" else 0)
    shape = (1, 2, 256 + 128, 128)
    if special == "ties":
        # groups whose values sit on exact half-steps: mn=0, mx=3*s, x = (k+0.5)*s
        s = np.float16(2.0 ** -3)
        k = rng.integers(0, 6, size=shape).astype(np.float64) * 0.5
        K = (k * float(s)).astype(np.float16)
        K[:, :, ::16, :] = 0.0
        K[:, :, 1::16, :] = np.float16(3 * float(s))
        V = K.copy()
    elif special == "const":
        K = kvq_synth.random_fp16(rng, shape, special="const")
        K[:, :, :64] = np.float16(-0.0)
        K[:, :, 64:128:2] = np.float16(0.0)
        V = K.copy()
    else:
        K = kvq_synth.random_fp16(rng, shape, special=special)
        V = kvq_synth.random_fp16(rng, shape, special=special)
    gpu, ora = make_pair(wl, max_T=1024, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    assert_state_equal(gpu, ora)


def test_decode_is_deterministic():
    wl, L0, _ = SMALL["gqa_b2"]
    K, V = kvq_synth.prefill_kv(wl, L0)
    gpu, _ = make_pair(wl, max_T=wl.T + 4 * wl.G, device=DEV)
    gpu.prefill(to_dev(K, DEV), to_dev(V, DEV))
    q = to_dev(kvq_synth.queries(wl, 1)[0], DEV)
    a = gpu.decode_attn(q).clone()
    for _ in range(3):
        assert bool((gpu.decode_attn(q) == a).all())


# ----------------------------------------------------------------------------- #
# Full sizes (the workloads' own shapes), sampled                                #
# ----------------------------------------------------------------------------- #

FULL = ["llama7b_mha", "llama3_8b_gqa_b2", "llama3_8b_gqa_b4", "kitty", "long_128k"]


def _full_state(name):
    wl = WORKLOADS[name]
    if wl.mode == "kitty":
        L0 = wl.S + wl.T + wl.R + 127   # K Q-buffer 127 after prefill; one append fills it
    else:
        L0 = wl.T + wl.R - 2            # the residual fills on the second step: one flush
    return wl, L0


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    wl, L0 = _full_state(name)
    K, V = kvq_synth.prefill_kv(wl, L0)
    gpu, ora = make_pair(wl, max_T=wl.T + 2 * wl.G + wl.R, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    del K, V
    rng = np.random.default_rng(0)
    U = [(b, h) for b in range(wl.B) for h in range(wl.H_kv)]
    units = [U[i] for i in sorted(rng.choice(len(U), size=min(4, len(U)), replace=False))]
    assert_state_equal(gpu, ora)          # every code, scale, min: bit-exact
    run_steps(gpu, ora, wl, 2, DEV, units=units)
    run_steps(gpu, ora, wl, 2, DEV, units=units, fused=True)   # insert and attend in one call
    assert gpu.read_status() == 0


@pytest.mark.parametrize("wl", [WORKLOADS["llama3_8b_gqa_rope"],
                                WORKLOADS["long_128k"].replace(rope_base=500000.0)],
                         ids=["gqa_rope_32k", "rope_128k"])
def test_full_size_pre_rope_sampled(wl):
    """Pre-RoPE keys at full size: positions up to 131K, where an angle t * theta
    evaluated in plain fp32 would be off by ~1e-2 rad."""
    L0 = wl.T + 64
    K, V = kvq_synth.prefill_kv(wl, L0)
    gpu, ora = make_pair(wl, max_T=wl.T + 2 * wl.G + wl.R, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    del K, V
    rng = np.random.default_rng(1)
    U = [(b, h) for b in range(wl.B) for h in range(wl.H_kv)]
    units = [U[i] for i in sorted(rng.choice(len(U), size=min(3, len(U)), replace=False))]
    run_steps(gpu, ora, wl, 2, DEV, units=units)
    run_steps(gpu, ora, wl, 2, DEV, units=units, fused=True)   # insert and attend in one call
    assert gpu.read_status() == 0


def test_full_size_nvfp4_sampled():
    """NVFP4 pages at the Llama-3-8B GQA shape (32K tokens): every code, block scale and
    page scale bit-exact; attention of sampled sequences."""
    wl = WORKLOADS["llama3_8b_gqa_nvfp4"]
    L0 = wl.T + 64
    K, V = kvq_synth.prefill_kv(wl, L0)
    gpu, ora = make_pair(wl, max_T=wl.T + 2 * wl.G + wl.R, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    del K, V
    assert_state_equal(gpu, ora)
    run_steps(gpu, ora, wl, 2, DEV, units=[(0, 1), (3, 6)])
    run_steps(gpu, ora, wl, 2, DEV, units=[(0, 1), (3, 6)], fused=True)   # insert and attend in one call
    assert gpu.read_status() == 0


def test_long_context_sequence_full_size():
    """The long-context workload as specified: kvq_quant_pack_k / _v over a 131072 + 64
    token prefill (B=1, H_kv=8), then 64 steps of insert-and-attend and flush, the flush
    firing on step 64.  Attention of two sampled sequences at steps 1, 32, 63 and 64;
    every code, scale and min bit-exact after the flush."""
    wl = WORKLOADS["long_128k"]
    L0 = wl.T + 64
    K, V = kvq_synth.prefill_kv(wl, L0)
    gpu, ora = make_pair(wl, max_T=wl.T + 2 * wl.G, device=DEV)
    prefill_both(gpu, ora, K, V, DEV)
    del K, V
    assert gpu.lengths["n_kres"] == 64
    run_steps(gpu, ora, wl, 64, DEV, check_every=31, units=[(0, 2), (0, 7)], fused=True)
    assert gpu.lengths["T_k"] == wl.T + wl.G and gpu.lengths["n_kres"] == 0
    assert_state_equal(gpu, ora)
    assert gpu.read_status() == 0
