"""Paged cache (per-sequence lengths, physical pages through a page table) on the GPU
against one CPU oracle cache per batch slot.

Every slot's packed pages, read back through its page table, must equal the oracle's
codes and scales bit for bit; attention must satisfy |err| <= 2e-3 + 2e-3 |ref|.
Physical pages are handed out in a shuffled order, so logical and physical order
differ; slots have different lengths (one empty, some still filling their sink), so
the decode ranges cross sequences of different item counts, and the steps run until
every slot has flushed a group.
"""
import numpy as np
import pytest

import kvq_synth
import oracle
from kvq_synth import WORKLOADS
from parity_util import _np, _u16, assert_close, keys_logical, to_dev, values_logical

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


BASE = WORKLOADS["llama3_8b_gqa_b2"]
CASES = {
    "k2v2_gqa": BASE.replace(B=7, H_q=16, H_kv=4),
    "k4v4_gqa": BASE.replace(B=7, H_q=16, H_kv=4, bits=4),
    "k2v4_sink": BASE.replace(B=7, H_q=16, H_kv=4, v_bits=4, S=8),
    # 8-bit keys (32-token tiles, four per page), a residual of two pages
    "k8v2_mha_r256": BASE.replace(B=7, H_q=4, H_kv=4, bits=8, v_bits=2, R=256),
}
LENS = [1000, 129, 0, 2048 + 17, 300, 5, 40]  # 0: an empty slot


def slot_workload(wl, b):
    return wl.replace(B=1, seed=1000 + 17 * b + wl.seed)


class Pair:
    """The paged GPU cache and one oracle cache per active slot."""

    def __init__(self, wl, n_pages, max_T, seed=5):
        import bit_kv_cache_gb300 as kvq
        self.wl = wl
        self.gpu = kvq.KVQPagedCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, n_pages=n_pages, max_T=max_T,
                                     S=wl.S, R=wl.R, device=DEV, v_bits=wl.v_bits)
        rng = np.random.default_rng(seed)
        self.gpu.free = [int(x) for x in rng.permutation(n_pages)]
        self.ora = {}

    def new_oracle(self):
        wl = self.wl
        return oracle.OracleCache(1, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R, v_bits=wl.v_bits)

    def prefill(self, b, L0, replica=0):
        K, V = kvq_synth.prefill_kv(slot_workload(self.wl, b), L0, replica=replica)
        o = self.new_oracle()
        o.prefill(K, V)
        self.ora[b] = o
        self.gpu.prefill(b, to_dev(K[0], DEV), to_dev(V[0], DEV))

    def release(self, b):
        self.gpu.release(b)
        del self.ora[b]

    def check_state(self):
        g, cfg = self.gpu, self.gpu.cfg
        H, D, G = cfg.H_kv, cfg.D, cfg.G
        kfpi, vfpi, Gv = 32 // cfg.bits, 32 // (cfg.v_bits or cfg.bits), min(G, D)
        for b in range(cfg.B):
            if b not in self.ora:
                assert g.lengths(b)["active"] == 0
                continue
            o = self.ora[b]
            assert o.T_k == o.T_v and o.n_kres == o.n_vres
            assert g.lengths(b) == {"n_sink": o.n_sink, "T": o.T_k, "n_res": o.n_kres, "active": 1}
            T = o.T_k
            pages = g.pages[b][: T // G]
            assert len(pages) == T // G
            if T:
                idx = np.asarray(pages)
                kc = keys_logical(_np(g.view("k_codes"))[idx], G, kfpi).transpose(1, 0, 2, 3).reshape(H, T // kfpi, D)
                assert np.array_equal(kc, o.k_codes[0][:, : T // kfpi]), "slot %d: key codes" % b
                km = _u16(_np(g.view("k_meta"))[idx].transpose(1, 0, 2, 3))
                assert np.array_equal(km, _u16(o.k_meta[0][:, : T // G])), "slot %d: key scale/min" % b
                vc = values_logical(_np(g.view("v_codes"))[idx].swapaxes(0, 1))
                assert np.array_equal(vc, o.v_codes[0][:, :T]), "slot %d: value codes" % b
                vm = _u16(_np(g.view("v_meta"))[idx].transpose(1, 0, 2, 3, 4).reshape(H, T, D // Gv, 2))
                assert np.array_equal(vm, _u16(o.v_meta[0][:, :T])), "slot %d: value scale/min" % b
            for name, n in (("k_res", o.n_kres), ("v_res", o.n_vres), ("k_sink", o.n_sink), ("v_sink", o.n_sink)):
                if n:
                    got = _u16(_np(g.view(name)[b][:, :n]))
                    assert np.array_equal(got, _u16(getattr(o, name)[0][:, :n])), "slot %d: %s" % (b, name)

    def check_attention(self, q):
        out = _np(self.gpu.decode_attn(to_dev(q, DEV)).float())
        for b, o in self.ora.items():
            assert_close(out[b: b + 1], o.attend(q[b: b + 1]), what="slot %d" % b)

    def steps(self, n, replica=0, check_every=1, state_every=16):
        wl = self.wl
        kn, vn = kvq_synth.decode_tokens(wl, n, replica=replica)
        qs = kvq_synth.queries(wl, n, replica=replica)
        for i in range(n):
            self.gpu.append(to_dev(kn[i], DEV), to_dev(vn[i], DEV))
            for b, o in self.ora.items():
                o.append(kn[i][b: b + 1], vn[i][b: b + 1])
            if i % check_every == 0 or i == n - 1:
                self.check_attention(qs[i])
            flushed = self.gpu.flush()
            want = []
            for b in sorted(self.ora):
                fk, fv = self.ora[b].flush()
                assert fk == fv
                if fk:
                    want.append(b)
            assert flushed == want, (i, flushed, want)
            if i % state_every == state_every - 1:
                self.check_state()
        self.check_state()
        assert self.gpu.read_status() == 0


def make(name, lens=LENS, n_pages=96, max_T=4096):
    wl = CASES[name]
    pr = Pair(wl, n_pages, max_T)
    for b, L0 in enumerate(lens):
        if L0:
            pr.prefill(b, L0)
    return pr


@pytest.mark.parametrize("name", list(CASES))
def test_paged_prefill_state_and_attention(name):
    pr = make(name)
    pr.check_state()
    q = kvq_synth.queries(pr.wl, 1, replica=3)[0]
    pr.check_attention(q)
    assert pr.gpu.read_status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_paged_steps_cross_every_flush(name):
    """R + 2 steps: every slot's residual fills and flushes at its own step."""
    pr = make(name)
    pr.steps(pr.wl.R + 2, check_every=3)


def test_paged_release_and_reuse():
    """A slot is emptied, its pages return to the pool and serve new sequences."""
    pr = make("k2v2_gqa")
    pr.steps(20, check_every=5)
    big = max(pr.ora, key=lambda b: pr.ora[b].T_k)
    pages_before = set(pr.gpu.pages[big])
    pr.release(big)
    assert pr.gpu.lengths(big)["active"] == 0
    pr.check_attention(kvq_synth.queries(pr.wl, 1, replica=9)[0])  # the released slot is skipped
    pr.prefill(2, 1500, replica=1)                                   # the empty slot
    pr.prefill(big, 777, replica=2)
    reused = set(pr.gpu.pages[2]) | set(pr.gpu.pages[big])
    assert reused & pages_before, "released pages were not reused"
    pr.check_state()
    pr.steps(40, replica=4, check_every=4)


def test_paged_single_token_and_sink_only_slots():
    """Slots holding one token, or only sink tokens, next to a long one."""
    wl = CASES["k2v4_sink"]
    pr = Pair(wl, 64, 4096)
    for b, L0 in enumerate([1, 3, 8, 2000, 0, 9, 1]):
        if L0:
            pr.prefill(b, L0)
    pr.check_state()
    pr.steps(12, check_every=1)


def test_paged_full_size_ragged_sampled():
    """Llama-3-8B GQA heads, four slots of 33K, 8K, 20K and 1 tokens; two slots checked
    against the oracle (their attention over every cached token), every slot's state
    sampled through its page table."""
    wl = BASE.replace(B=4)
    lens = [32768 + 100, 8192 + 5, 20000 + 77, 1]
    pr = Pair(wl, 520, 34 * 1024)
    for b, L0 in enumerate(lens):
        pr.prefill(b, L0)
    q = kvq_synth.queries(wl, 1, replica=11)[0]
    out = _np(pr.gpu.decode_attn(to_dev(q, DEV)).float())
    for b in (1, 3):
        assert_close(out[b: b + 1], pr.ora[b].attend(q[b: b + 1]), what="slot %d" % b)
    # slot 0: heads 0 and 5 only (the oracle's attention over 33K tokens per head)
    ref = pr.ora[0].attend(q[0:1], units=[(0, 0), (0, 5)])
    assert_close(out[0:1], ref, what="slot 0")
    pr.check_state()
    assert pr.gpu.read_status() == 0
