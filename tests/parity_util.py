"""Shared helpers for the GPU-vs-oracle parity tests."""
import numpy as np

import kvq_synth
import oracle

TOL_ABS = 2e-3
TOL_REL = 2e-3


# The library keeps pack_tensor's words but orders them within a page for its decode
# tiles: the 16-byte chunks of key word row r (0-based in its page) are permuted by XOR
# with r mod 8, and value pages are tile-major ([G/TV][D/fpi rows][TV words]) with the
# chunks of row b permuted by XOR with b mod 8 when TV is a multiple of 32.  These undo
# that, giving the oracle's (the pages') layouts.
def keys_logical(kc, G, kfpi):
    """[..., T/fpi, D] words as stored -> pack_tensor's [..., T/fpi, D]."""
    rows, D = kc.shape[-2:]
    r = (np.arange(rows) % (G // kfpi)) & 7
    pos = np.arange(D)[None, :] ^ (r[:, None] << 2)
    return np.take_along_axis(kc, np.broadcast_to(pos, kc.shape), axis=-1)


def values_logical(vc):
    """[..., P, G/TV, D/fpi, TV] words as stored -> [..., P * G, D/fpi] (token-major)."""
    rows, TV = vc.shape[-2:]
    if TV % 32 == 0:
        b = np.arange(rows) & 7
        pos = np.arange(TV)[None, :] ^ (b[:, None] << 2)
        vc = np.take_along_axis(vc, np.broadcast_to(pos, vc.shape), axis=-1)
    vc = np.swapaxes(vc, -1, -2)
    sh = vc.shape
    return vc.reshape(sh[:-4] + (sh[-4] * sh[-3] * sh[-2], sh[-1]))


def make_pair(wl, max_T, device):
    import bit_kv_cache_gb300 as kvq
    gpu = kvq.KVQCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R,
                       n_boost=wl.n_boost, mode=wl.mode, max_T=max_T, device=device, v_bits=wl.v_bits,
                       rope_base=wl.rope_base)
    ora = oracle.OracleCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R,
                             n_boost=wl.n_boost, mode=wl.mode, v_bits=wl.v_bits, rope_base=wl.rope_base)
    return gpu, ora


def to_dev(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def prefill_both(gpu, ora, K, V, device):
    gpu.prefill(to_dev(K, device), to_dev(V, device))
    ora.prefill(K, V)


def assert_lengths(gpu, ora):
    got = gpu.lengths
    want = dict(n_sink=ora.n_sink, T_k=ora.T_k, n_kres=ora.n_kres, T_v=ora.T_v,
                n_vres=ora.n_vres, n_local=ora.n_local, local_head=ora.local_head)
    assert got == want, (got, want)


def _np(t):
    return t.cpu().numpy()


def _u16(a):
    return np.ascontiguousarray(a).view(np.uint16)


def _assert_nvfp4_state(gpu, ora, pick):
    cfg = gpu.cfg
    T, G, D = ora.T_k, cfg.G, cfg.D
    assert ora.T_v == T
    P = T // G
    raw = {s: _np(gpu.view(s + "_codes")).reshape(cfg.B, cfg.H_kv, -1)[:, :, : P * G * D // 2]
           for s in ("k", "v")}
    # keys: [P][D/32][G][16] -> token-major [T][D/2]
    kc = raw["k"].reshape(cfg.B, cfg.H_kv, P, D // 32, G, 16).transpose(0, 1, 2, 4, 3, 5)
    kc = kc.reshape(cfg.B, cfg.H_kv, T, D // 2)
    # values: [P][G/32][D][16] (byte = tokens 2m, 2m+1 of a channel) -> token-major [T][D/2]
    vr = raw["v"].reshape(cfg.B, cfg.H_kv, P, G // 32, D, 16)
    nib = np.stack([vr & 15, vr >> 4], axis=-1)                               # [.., tg, c, m, 2]
    nib = nib.transpose(0, 1, 2, 3, 5, 6, 4).reshape(cfg.B, cfg.H_kv, T, D)     # token-major nibbles
    vc = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    for side, codes in (("k", kc), ("v", vc)):
        assert np.array_equal(pick(codes), pick(getattr(ora, side + "_codes"))), side + " codes differ"
        rec = _np(gpu.view(side + "_meta")[:, :, : T // G])                     # [B,H,P,16 + G*D/16]
        S = np.ascontiguousarray(rec[..., :4]).view(np.float32)[..., 0]
        assert np.array_equal(pick(S).view(np.uint32), pick(getattr(ora, side + "_S")).view(np.uint32)), \
            side + " page scales differ"
        sc = rec[..., 16:]
        if side == "k":
            sc = sc.reshape(cfg.B, cfg.H_kv, T, D // 16)
        else:
            sc = sc.reshape(cfg.B, cfg.H_kv, T // 16, D)
        assert np.array_equal(pick(sc), pick(getattr(ora, side + "_scales"))), side + " block scales differ"


def assert_state_equal(gpu, ora, units=None):
    """Bit-exact comparison of every cache buffer (optionally for some (b, h) only)."""
    assert_lengths(gpu, ora)
    cfg = gpu.cfg
    kitty = ora.kitty
    kfpi = 16 if kitty else 32 // cfg.bits
    vfpi = 32 // (cfg.v_bits or cfg.bits)

    def pick(a):
        if units is None:
            return a
        return np.stack([a[b, h] for b, h in units])

    T_k, T_v, G = ora.T_k, ora.T_v, cfg.G
    if getattr(ora, "nvfp4", False):
        _assert_nvfp4_state(gpu, ora, pick)
        for name, n in (("k_res", ora.n_kres), ("v_res", ora.n_vres), ("k_sink", ora.n_sink),
                        ("v_sink", ora.n_sink)):
            if n:
                assert np.array_equal(pick(_u16(_np(gpu.view(name)[:, :, :n]))),
                                      pick(_u16(getattr(ora, name)[:, :, :n]))), name + " differs"
        return
    kc = keys_logical(_np(gpu.view("k_codes")[:, :, : T_k // kfpi]), G, kfpi)
    assert np.array_equal(pick(kc), pick(ora.k_codes)), "key codes differ"
    km = _u16(_np(gpu.view("k_meta")[:, :, : T_k // G]))
    assert np.array_equal(pick(km), pick(_u16(ora.k_meta))), "key scale/min differ"
    vc = values_logical(_np(gpu.view("v_codes")[:, :, : T_v // G]))  # [B,H,T_v,D/fpi]
    assert np.array_equal(pick(vc), pick(ora.v_codes)), "value codes differ"
    vm = _u16(_np(gpu.view("v_meta")[:, :, :T_v]))
    assert np.array_equal(pick(vm), pick(_u16(ora.v_meta))), "value scale/min differ"
    if kitty:
        bi = _np(gpu.view("k_bidx")[:, :, : T_k // G])
        assert np.array_equal(pick(bi), pick(ora.k_bidx)), "boost index differs"
        if cfg.n_boost:
            hi = _np(gpu.view("k_hi")[:, :, : T_k // 16])
            assert np.array_equal(pick(hi), pick(ora.k_hi)), "high plane differs"
        # the whole ring: slots never written are zero on both sides
        lo = _u16(_np(gpu.view("v_local")))
        assert np.array_equal(pick(lo), pick(_u16(ora.v_local))), "local window differs"
    for name, n in (("k_res", ora.n_kres), ("v_res", ora.n_vres), ("k_sink", ora.n_sink),
                    ("v_sink", ora.n_sink)):
        if n == 0:
            continue
        g = _u16(_np(gpu.view(name)[:, :, :n]))
        o = _u16(getattr(ora, name)[:, :, :n])
        assert np.array_equal(pick(g), pick(o)), name + " differs"


def assert_close(out, ref, what="attention"):
    """|out - ref| <= 2e-3 + 2e-3 |ref| for every element the oracle computed."""
    out = np.asarray(out, np.float64)
    mask = ~np.isnan(ref)
    err = np.abs(out - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = mask & ~(err <= bound)
    assert not bad.any(), "%s: %d elements out of tolerance, max err %.3g (ref %.3g)" % (
        what, bad.sum(), err[mask].max(), np.abs(ref[mask]).max())
    return float(err[mask].max()) if mask.any() else 0.0


def run_steps(gpu, ora, wl, n_steps, device, check_every=1, units=None, fused=False):
    """n decode steps (append, attend, flush) on both sides; compares outputs.  fused:
    the GPU side inserts and attends with one kvq_append_decode call per step."""
    kn, vn = kvq_synth.decode_tokens(wl, n_steps)
    qs = kvq_synth.queries(wl, n_steps)
    worst = 0.0
    for i in range(n_steps):
        if fused:
            out_t, _ = gpu.append_decode(to_dev(qs[i], device), to_dev(kn[i], device), to_dev(vn[i], device))
        else:
            gpu.append_token(to_dev(kn[i], device), to_dev(vn[i], device))
        ora.append(kn[i], vn[i])
        if i % check_every == 0 or i == n_steps - 1:
            out = _np((out_t if fused else gpu.decode_attn(to_dev(qs[i], device))).float())
            ref = ora.attend(qs[i], units=units)
            worst = max(worst, assert_close(out, ref, what="step %d" % i))
        fk, fv = gpu.flush_group()
        ofk, ofv = ora.flush()
        assert (fk, fv) == (ofk, ofv)
    return worst
