"""The benchmark's byte accounting against the oracle cache (CPU only).

bench.py reports bandwidth as algorithmic bytes per step over time.  Those bytes come
from its own length bookkeeping (`after_append`, the flush rule that `replay_steps`
replays) and its per-step formula (`decode_bytes`).  Here both are checked against an
independent source: the oracle cache's lengths after the same appends and flushes, and
the sizes of the arrays the oracle actually holds for those lengths (packed codes,
scales and mins, fp16 rows), plus the query and output of the step.
"""
import numpy as np
import pytest

import bench
import kvq_synth
import oracle
from kvq_synth import WORKLOADS

CASES = {
    "kivi_2bit": WORKLOADS["tiny_kivi"].replace(H_kv=2, T=128),
    "kivi_k4v2_sink": WORKLOADS["tiny_kivi"].replace(H_kv=2, T=128, bits=4, v_bits=2, S=8),
    "kivi_k8v8": WORKLOADS["tiny_kivi"].replace(H_kv=2, T=128, bits=8),
    "kitty": WORKLOADS["kitty"].replace(B=1, H_q=4, H_kv=2, T=256, G=32, R=32, S=4, n_boost=8),
}


def _lengths(o):
    return {"n_sink": o.n_sink, "T_k": o.T_k, "n_kres": o.n_kres, "T_v": o.T_v, "n_vres": o.n_vres,
            "n_local": o.n_local}


def _held_bytes(o, wl):
    """Bytes of what the oracle cache holds for its current lengths, plus q and out."""
    kfpi = 16 if o.kitty else 32 // o.bits
    b = o.k_codes[:, :, : o.T_k // kfpi].nbytes + o.k_meta[:, :, : o.T_k // o.G].nbytes
    if o.kitty and o.n_boost:
        b += o.k_hi[:, :, : o.T_k // 16].nbytes + o.k_bidx[:, :, : o.T_k // o.G].nbytes
    b += o.v_codes[:, :, : o.T_v].nbytes + o.v_meta[:, :, : o.T_v].nbytes
    rows = 2 * o.n_sink + o.n_kres + o.n_vres + o.n_local
    b += o.B * o.H_kv * rows * o.D * 2
    b += 2 * wl.B * wl.H_q * wl.D * 2
    return b


def _oracle(wl):
    return oracle.OracleCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R, n_boost=wl.n_boost,
                              mode=wl.mode, v_bits=wl.v_bits)


@pytest.mark.parametrize("name", list(CASES))
def test_step_bytes_follow_the_cache(name):
    """Over enough steps to fill and flush every buffer: the lengths bench.py predicts
    after each append equal the oracle's, and decode_bytes of them equals the bytes the
    oracle cache holds at that point."""
    wl = CASES[name]
    o = _oracle(wl)
    L0 = wl.T + wl.G // 2 + 3
    K, V = kvq_synth.prefill_kv(wl, L0)
    o.prefill(K, V)
    n = 2 * wl.G + 5
    kn, vn = kvq_synth.decode_tokens(wl, n)
    st = _lengths(o)
    flushes = 0
    for i in range(n):
        st = bench.after_append(wl, st)
        o.append(kn[i], vn[i])
        assert st == _lengths(o), (i, st, _lengths(o))
        assert bench.decode_bytes(wl, st) == _held_bytes(o, wl), i
        fk, fv = o.flush()
        flushes += fk or fv
        # the flush rule of the one-launch loop (KIVI: both residuals at once)
        if not o.kitty and (st["n_kres"] == wl.R or st["n_vres"] == wl.R):
            st["T_k"] += st["n_kres"]
            st["T_v"] += st["n_vres"]
            st["n_kres"] = st["n_vres"] = 0
        if o.kitty:
            st = _lengths(o)
        assert st == _lengths(o), (i, st, _lengths(o))
    assert flushes >= 2


def test_replay_matches_stepping_each_layer():
    """replay_steps over rotating layer states gives the per-step sum of decode_bytes
    after append and the same final lengths as stepping each layer's oracle cache."""
    wl = CASES["kivi_2bit"]
    layers = 3
    saved = bench.N_LAYERS
    bench.N_LAYERS = layers
    try:
        caches = []
        for li in range(layers):
            o = _oracle(wl)
            K, V = kvq_synth.prefill_kv(wl, wl.T + 7 * li, replica=li)
            o.prefill(K, V)
            caches.append(o)
        states = [_lengths(o) for o in caches]
        first, K_steps = 5, 3 * wl.G + 2
        total = bench.replay_steps(wl, states, first, K_steps, wl.R)
        kn, vn = kvq_synth.decode_tokens(wl, 4)
        want = 0
        for s in range(first, first + K_steps):
            o = caches[s % layers]
            o.append(kn[s % 4], vn[s % 4])
            want += _held_bytes(o, wl)
            o.flush()
        assert total == want
        assert states == [_lengths(o) for o in caches]
    finally:
        bench.N_LAYERS = saved


def test_headline_step_bytes():
    """The headline configuration with a full residual: 72 bytes per packed token
    (codes 32 + 32, scales and mins 4 + 4), the fp16 residual rows, q and out."""
    wl = WORKLOADS["llama3_8b_gqa_b2"]
    U = wl.B * wl.H_kv
    st = {"n_sink": 0, "T_k": wl.T, "n_kres": wl.R, "T_v": wl.T, "n_vres": wl.R, "n_local": 0}
    packed = U * wl.T * 72
    rows = U * 2 * wl.R * wl.D * 2
    qo = 2 * wl.B * wl.H_q * wl.D * 2
    assert bench.decode_bytes(wl, st) == packed + rows + qo
    assert abs(bench.decode_bytes(wl, st) / 1e6 - 77.66) < 0.01
