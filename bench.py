"""Decode-step benchmark of the GB300 low-bit KV cache.

Default workload: the Llama-3-8B-shaped GQA layer (B=4, H_q=32, H_kv=8, D=128,
T=32768 packed 2-bit tokens, G=R=128).  One step = one decode step of one layer
in the Kitty pipeline order: append the new token and attend (kvq_append_decode:
one launch for KIVI caches on the packed-tile path, else kvq_append_token then
kvq_decode_attn), quantize the residual when it is full (kvq_flush_group).  The
benchmark rotates through 16 layer caches (16 x 77.7 MB > 2 x L2), so no step
finds its cache in L2.  Layer l's prefill is the seeded draw rolled by l*977
tokens (same distribution, different pages); residual fills are staggered.

value  = effective packed-KV bandwidth: algorithmic bytes of all timed steps
         (codes + fp16 scales/mins + fp16 sink/residual + q + out, summed per step
         from the cache state) / device time.  Whole job: summed over ranks.
e2e    = the same through host buffers: per step one kvq_decode_step_host_wait call
         (pinned q / k_new / v_new read and out written by the kernels in place; the
         call returns once out holds the step's result).
roofline: the decode kernel, CUDA events on its stream, against the measured HBM
         copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import kvq_synth  # noqa: E402

N_LAYERS = 16


# The headline metric this harness reports (the name every JSON line carries).
METRIC = "2-bit KV decode-attn \u00b5s/step & packed-KV GB/s (% of GB300 HBM peak)"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def decode_bytes(wl, lengths) -> int:
    """Algorithmic bytes one decode_attn call reads and writes for a cache state."""
    U = wl.B * wl.H_kv
    D, G = wl.D, wl.G
    Gv = min(G, D)
    kb = 2 if wl.mode == "kitty" else wl.bits
    T_k, T_v = lengths["T_k"], lengths["T_v"]
    if wl.mode == "nvfp4":   # 4-bit codes, one e4m3 scale per 16 elements, 16-byte page records
        b = U * (T_k + T_v) * D // 2 + U * (T_k + T_v) * D // 16 + U * (T_k // G + T_v // G) * 16
        n16 = lengths["n_sink"] * 2 + lengths["n_kres"] + lengths["n_vres"]
        return b + U * n16 * D * 2 + 2 * wl.B * wl.H_q * D * 2
    b = U * T_k * D * kb // 8 + U * (T_k // G) * D * 4              # key codes + (scale, min)
    if wl.mode == "kitty" and wl.n_boost:
        b += U * T_k * wl.n_boost * 2 // 8 + U * (T_k // G) * D      # high plane + boost index
    b += U * T_v * D * wl.vbits // 8 + U * T_v * (D // Gv) * 4      # value codes + (scale, min)
    n16 = lengths["n_sink"] * 2 + lengths["n_kres"] + lengths["n_vres"] + lengths["n_local"]
    b += U * n16 * D * 2                                           # fp16 sink / buffers
    b += 2 * wl.B * wl.H_q * D * 2                                 # q in, out
    return b


def after_append(wl, lengths) -> dict:
    """Cache lengths after one kvq_append_token (its rule, on the host-side lengths):
    sink first, then the key residual and the value residual (KIVI) or the local
    window, whose oldest value moves to the value buffer once it is full (Kitty)."""
    n = dict(lengths)
    if n["n_sink"] < wl.S:
        n["n_sink"] += 1
        return n
    n["n_kres"] += 1
    if wl.mode != "kitty":
        n["n_vres"] += 1
    elif n["n_local"] < wl.R:
        n["n_local"] += 1
    else:
        n["n_vres"] += 1
    return n


def replay_steps(wl, states, first, K, cap) -> int:
    """Algorithmic bytes of steps first .. first + K - 1 of the one-launch loop (step s
    appends to and attends over layer s % N_LAYERS, then flushes a full residual),
    replayed on host copies of the lengths; `states` (one dict per layer) advances.
    KIVI caches only: a flush packs the cap residual tokens of keys and values."""
    total = 0
    for s in range(first, first + K):
        li = s % N_LAYERS
        st = after_append(wl, states[li])
        total += decode_bytes(wl, st)
        if st["n_kres"] == cap or st["n_vres"] == cap:
            st["T_k"] += st["n_kres"]
            st["T_v"] += st["n_vres"]
            st["n_kres"] = st["n_vres"] = 0
        states[li] = st
    return total


def decode_bytes_struct(wl, st) -> int:
    """decode_bytes for the lengths held in a kvq_cache struct."""
    return decode_bytes(wl, {"T_k": st.T_k, "T_v": st.T_v, "n_sink": st.n_sink, "n_kres": st.n_kres,
                             "n_vres": st.n_vres, "n_local": st.n_local})


DECODE_SOURCES = ("kvq_decode.cu", "kvq_decode.cuh", "kvq_decode_fast.cuh", "kvq_device.cuh", "kvq_internal.h",
                  "kvq_api.cu", "kvq_host.h", "kvq_paged.cu", "kvq_decode_paged.cu", "kvq_decode_rope.cu",
                  "kvq_decode_nvfp4.cu")
QUANT_SOURCES = ("kvq_quant.cu", "kvq_device.cuh", "kvq_internal.h", "kvq_api.cu", "kvq_host.h")


def kernel_hash(sources=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "bit_kv_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """dram bytes per decode launch from the committed ncu summary, if it still
    describes the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    src = QUANT_SOURCES if workload.startswith("quant_") else DECODE_SOURCES
    if not e or e.get("kernel_hash") != kernel_hash(src):
        return None
    return e.get("dram_bytes_per_launch")


class Clocks:
    """nvidia-smi sampling; summary() keeps the samples taken inside [t0, t1]."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None
        self.rows = []

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "20"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        time.sleep(0.5)

    def stop(self):
        if self.p is None:
            return
        time.sleep(0.1)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        import datetime
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            self.rows.append([ts] + parts[1:])

    def summary(self, t0: float, t1: float):
        rows = [r for r in self.rows if t0 - 0.025 <= r[0] <= t1 + 0.025]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no sample in timed region"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[2]) for r in rows) if v is not None]
        mx = [v for v in (num(r[3]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def reduce_over_ranks(ms: float, nbytes: float, world: int, device=None):
    """Whole-job numbers of a timed region: the slowest rank's time and the bytes
    of all ranks (each rank works on its own shard; this is the only collective,
    and it runs after the timed region)."""
    if world <= 1:
        return ms, nbytes
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, nbytes], dtype=torch.float64, device=device)
    mx = t[:1].clone()
    sm = t[1:].clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[0])


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_oracle_rate(wl, max_seconds: float, threads: int = 1):
    """The oracle (fp64 attention) on a bounded sample of the workload: decode attention
    over `threads` independent (b, h_kv) sequences of the workload's length, one per
    thread, repeated for about max_seconds.  Returns (GB/s in the benchmark's byte
    accounting, seconds, repetitions, sample description)."""
    import oracle
    L0 = wl.T + 64
    n_units = max(1, threads)
    sub = wl.replace(B=1, H_kv=n_units, H_q=n_units * wl.g)
    K, V = kvq_synth.prefill_kv(sub, L0)
    ora = oracle.OracleCache(sub.B, sub.H_q, sub.H_kv, sub.D, sub.G, sub.bits, S=sub.S, R=sub.R,
                             n_boost=sub.n_boost, mode=sub.mode, v_bits=sub.v_bits, rope_base=sub.rope_base)
    ora.prefill(K, V)
    del K, V
    q = kvq_synth.queries(sub, 1)[0]
    lengths = dict(n_sink=ora.n_sink, T_k=ora.T_k, n_kres=ora.n_kres, T_v=ora.T_v,
                   n_vres=ora.n_vres, n_local=ora.n_local)
    per = decode_bytes(sub, lengths)
    t0 = time.perf_counter()
    steps = 0
    while True:
        ora.attend(q, threads=threads)
        steps += 1
        if time.perf_counter() - t0 >= max_seconds:
            break
    dt = time.perf_counter() - t0
    desc = ("oracle decode attention (fp64, %d thread%s, one (b,h_kv) sequence each) over %d sequences "
            "of %d tokens, %d repetitions" % (threads, "s" if threads > 1 else "", n_units, L0, steps))
    return per * steps / dt / 1e9, dt, steps, desc


def cpu_quant_rate(wl, max_seconds: float, threads: int = 1):
    """The oracle's prefill quantizer (keys per channel, values per token, packing) over
    `threads` independent sequences of n tokens each, n sized for about max_seconds."""
    import oracle
    probe_n = 4 * wl.G
    sub = wl.replace(B=1, H_kv=1, H_q=wl.g)
    K, V = kvq_synth.prefill_kv(sub, probe_n)
    o = oracle.OracleCache(1, wl.g, 1, wl.D, wl.G, wl.bits, R=wl.R, v_bits=wl.v_bits)
    t0 = time.perf_counter()
    o.prefill(K, V)
    per_tok = (time.perf_counter() - t0) / probe_n
    n = max(wl.G, int(max_seconds / max(per_tok, 1e-9)) // wl.G * wl.G)
    n = min(n, wl.T)
    n_units = max(1, threads)
    sub = wl.replace(B=1, H_kv=n_units, H_q=n_units * wl.g)
    K, V = kvq_synth.prefill_kv(sub, n)

    def one(h):
        oc = oracle.OracleCache(1, wl.g, 1, wl.D, wl.G, wl.bits, R=wl.R, v_bits=wl.v_bits)
        oc.prefill(np.ascontiguousarray(K[:, h:h + 1]), np.ascontiguousarray(V[:, h:h + 1]))
    t0 = time.perf_counter()
    if threads > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(n_units)))
    else:
        one(0)
    dt = time.perf_counter() - t0
    b = quant_pack_bytes(sub, n)
    return (b["k"] + b["v"]) / dt / 1e9, dt, ("oracle kvq_quant_pack_k + _v (fp32 quantizer, %d thread%s) "
                                              "over %d sequence%s of %d tokens" % (
                                                  threads, "s" if threads > 1 else "", n_units,
                                                  "s" if n_units > 1 else "", n))


def cpu_baseline(wl, seconds: float) -> dict:
    """The oracle timed on this host: single-threaded, and on all cores over independent
    (b, h_kv) sequences (results identical: the same code per sequence)."""
    nproc = os.cpu_count() or 1
    v1, dt1, n1, d1 = cpu_oracle_rate(wl, seconds * 0.4, 1)
    va, dta, na, da = cpu_oracle_rate(wl, seconds * 0.3, nproc)
    q1, qdt1, qd1 = cpu_quant_rate(wl, seconds * 0.15, 1)
    qa, qdta, qda = cpu_quant_rate(wl, seconds * 0.15, nproc)
    return {"value": v1, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": d1, "seconds": dt1,
            "cpu_model": cpu_model(), "nproc": nproc,
            "all_cores": {"value": va, "unit": "GB/s", "cores": nproc, "sample": da, "seconds": dta},
            "quant_pack": {"value": q1, "unit": "GB/s", "cores": 1, "sample": qd1, "seconds": qdt1,
                           "all_cores": {"value": qa, "unit": "GB/s", "cores": nproc, "sample": qda,
                                         "seconds": qdta}}}


def reference_arm(args, wl, rank, world, budget_s: float = 150.0):
    """--impl reference: the CPU oracle as it stands, on the host cores.

    One step = the oracle's decode attention over the first n tokens of one
    (b, h_kv) sequence of the workload (all g query heads), with n chosen from a
    calibration run so that warm-up + timed steps take about budget_s seconds."""
    if rank != 0:
        return 0
    K, W = args.steps, args.warmup
    import oracle
    sub = wl.replace(B=1, H_kv=1, H_q=wl.g)

    def make(n_tok):
        Kx, Vx = kvq_synth.prefill_kv(sub, n_tok)
        ora = oracle.OracleCache(sub.B, sub.H_q, sub.H_kv, sub.D, sub.G, sub.bits, S=sub.S,
                                 R=sub.R, n_boost=sub.n_boost, mode=sub.mode, v_bits=sub.v_bits)
        ora.prefill(Kx, Vx)
        return ora

    L_full = wl.T + 64
    probe = make(min(L_full, 8 * wl.G + 64))
    qs = kvq_synth.queries(sub, 4)
    t0 = time.perf_counter()
    probe.attend(qs[0])
    per_tok = (time.perf_counter() - t0) / probe.L
    n_tok = int(budget_s / (K + W) / max(per_tok, 1e-9))
    n_tok = max(wl.G + 1, min(L_full, n_tok // wl.G * wl.G + 64))
    ora = make(n_tok)
    lengths = dict(n_sink=ora.n_sink, T_k=ora.T_k, n_kres=ora.n_kres, T_v=ora.T_v,
                   n_vres=ora.n_vres, n_local=ora.n_local)
    per = decode_bytes(sub, lengths)
    for i in range(W):
        ora.attend(qs[i % 4])
    t0 = time.perf_counter()
    for i in range(K):
        ora.attend(qs[i % 4])
    dt = time.perf_counter() - t0
    val = per * K / dt / 1e9
    sample = ("per step: oracle decode attention (fp64, single thread) over the first %d of "
              "%d tokens of 1 of %d (b,h_kv) sequences, %d query heads" % (
                  ora.L, L_full, wl.B * wl.H_kv, wl.g))
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": dt / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, shapes of the workload)",
            "config": {"workload": wl.name, "B": wl.B, "H_q": wl.H_q, "H_kv": wl.H_kv, "D": wl.D,
                       "T": wl.T, "G": wl.G, "bits": wl.bits, "v_bits": wl.vbits},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def quant_pack_bytes(wl, L0) -> dict:
    """Algorithmic bytes of the prefill calls over L0 tokens (no sink): the fp16 input read
    once; packed codes, per-group (scale, min) and the fp16 residual rows written."""
    U, D, G = wl.B * wl.H_kv, wl.D, wl.G
    T = L0 // G * G
    res = L0 - T
    k = U * L0 * D * 2 + U * T * D * wl.bits // 8 + U * (T // G) * D * 4 + U * res * D * 2
    v = U * L0 * D * 2 + U * T * D * wl.vbits // 8 + U * T * (D // min(G, D)) * 4 + U * res * D * 2
    return {"k": k, "v": v}


def quant_pack_measure(kvq, dev, peak, reps: int = 5) -> dict:
    """kvq_quant_pack_k and kvq_quant_pack_v over the long-context prefill (B=1, H_kv=8,
    131072 + 64 tokens, 2-bit): CUDA events around each call, a 512 MB write between calls
    so that the input is not in L2; the median of `reps` calls."""
    import torch
    wl = kvq_synth.WORKLOADS["long_128k"]
    L0 = wl.T + 64
    K, V = kvq_synth.prefill_kv(wl, L0)
    Kd, Vd = torch.from_numpy(K).to(dev), torch.from_numpy(V).to(dev)
    del K, V
    c = kvq.KVQCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, R=wl.R, max_T=wl.T + wl.G, device=dev)
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ts = {"k": [], "v": []}
    for r in range(reps + 1):
        for name in ("n_sink", "T_k", "n_kres", "T_v", "n_vres", "n_local", "local_head"):
            setattr(c.c, name, 0)       # an empty cache again (host-side lengths)
        for side, fn, x in (("k", c.quant_pack_k, Kd), ("v", c.quant_pack_v, Vd)):
            scrub.fill_(r & 255)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn(x)
            b.record(stream)
            torch.cuda.synchronize()
            if r > 0:                   # the first call warms up
                ts[side].append(a.elapsed_time(b))
    assert c.read_status() == 0
    nb = quant_pack_bytes(wl, L0)
    outp = {"workload": "long_128k prefill: B=1, H_kv=8, D=128, %d tokens, 2-bit, G=128 (%d MB fp16 per side)" % (
        L0, nb["k"] // 2**20 // 1), "timing": "median of %d calls, CUDA events, L2 scrubbed before each" % reps}
    for side in ("k", "v"):
        ms = statistics.median(ts[side])
        gbs = nb[side] / (ms * 1e-3) / 1e9
        outp["kvq_quant_pack_" + side] = {"us": ms * 1e3, "algorithmic_bytes": nb[side], "achieved": gbs,
                                          "frac": gbs / peak, "traffic": profiled_traffic("quant_" + side)}
    del Kd, Vd, c, scrub
    torch.cuda.empty_cache()
    return outp


def long_sequence_measure(kvq, dev, peak, reps: int = 3) -> dict:
    """The long-context workload as a whole: kvq_quant_pack_k + _v over the 131072 + 64
    token prefill, then 64 decode steps (kvq_append_decode + kvq_flush_group; the flush
    fires on step 64).  CUDA events around the prefill and around the 64 steps; L2
    scrubbed before each repetition; the median of `reps`."""
    import ctypes
    import torch
    wl = kvq_synth.WORKLOADS["long_128k"]
    L0 = wl.T + 64
    K, V = kvq_synth.prefill_kv(wl, L0)
    Kd, Vd = torch.from_numpy(K).to(dev), torch.from_numpy(V).to(dev)
    del K, V
    kn, vn = kvq_synth.decode_tokens(wl, 64)
    qs = kvq_synth.queries(wl, 64)
    kn_d, vn_d, q_d = (torch.from_numpy(a).to(dev) for a in (kn, vn, qs))
    out = torch.empty((wl.B, wl.H_q, wl.D), dtype=torch.float16, device=dev)
    c = kvq.KVQCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, R=wl.R, max_T=wl.T + 2 * wl.G, device=dev)
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    lib = kvq.lib
    args = (ctypes.byref(c.cfg), ctypes.byref(c.c))
    ws, wsb = ctypes.c_void_p(c.ws.data_ptr()), c.ws.numel()
    fk, fv, fu = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    pre, seq, flush_at, step_bytes = [], [], [], 0
    for r in range(reps + 1):
        for name in ("n_sink", "T_k", "n_kres", "T_v", "n_vres", "n_local", "local_head"):
            setattr(c.c, name, 0)
        scrub.fill_(r & 255)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        c.prefill(Kd, Vd)
        e[1].record(stream)
        nbytes, fl = 0, []
        for j in range(64):
            nbytes += decode_bytes(wl, after_append(wl, c.lengths))
            rc = lib.kvq_append_decode(*args, ctypes.c_void_p(kn_d[j].data_ptr()), ctypes.c_void_p(vn_d[j].data_ptr()),
                                       ctypes.c_void_p(q_d[j].data_ptr()), ctypes.c_void_p(out.data_ptr()), ws, wsb,
                                       ctypes.byref(fu), sp)
            rc |= lib.kvq_flush_group(*args, ctypes.byref(fk), ctypes.byref(fv), sp)
            if rc:
                raise RuntimeError("long-context step %d failed: %d" % (j, rc))
            if fk.value:
                fl.append(j + 1)
        e[2].record(stream)
        torch.cuda.synchronize()
        if r > 0:
            pre.append(e[0].elapsed_time(e[1]))
            seq.append(e[1].elapsed_time(e[2]))
            flush_at, step_bytes = fl, nbytes
    assert c.read_status() == 0
    nb = quant_pack_bytes(wl, L0)
    p_ms, s_ms = statistics.median(pre), statistics.median(seq)
    res = {"workload": "long_128k: B=1, H_q=32, H_kv=8, D=128, prefill 131072 + 64 tokens, then 64 decode steps",
           "timing": "median of %d sequences, CUDA events, L2 scrubbed before each" % reps,
           "prefill_us": p_ms * 1e3, "prefill_bytes": nb["k"] + nb["v"],
           "prefill_GBps": (nb["k"] + nb["v"]) / (p_ms * 1e-3) / 1e9,
           "prefill_frac": (nb["k"] + nb["v"]) / (p_ms * 1e-3) / 1e9 / peak,
           "steps_us": s_ms * 1e3, "us_per_step": s_ms * 1e3 / 64, "steps_bytes": step_bytes,
           "steps_GBps": step_bytes / (s_ms * 1e-3) / 1e9, "flush_on_steps": flush_at,
           "total_us": (p_ms + s_ms) * 1e3}
    del Kd, Vd, c, scrub
    torch.cuda.empty_cache()
    return res


def paged_bytes(wl, lens_host) -> int:
    """decode_bytes of a paged cache: the sum over active slots of each slot's bytes."""
    H, D, G = wl.H_kv, wl.D, wl.G
    Gv = min(G, D)
    b = 0
    for s in range(wl.B):
        ns, T, nr, act = lens_host[4 * s: 4 * s + 4]
        if not act:
            continue
        b += H * T * D * wl.bits // 8 + H * (T // G) * D * 4
        b += H * T * D * wl.vbits // 8 + H * T * (D // Gv) * 4
        b += H * (2 * ns + 2 * nr) * D * 2
    return b + 2 * wl.B * wl.H_q * D * 2


def paged_main(args, wl, rank, world, dev):
    """The paged cache: B slots of different lengths (kvq_synth.slot_lengths) over a
    page pool, N_LAYERS layer caches rotated; a step is kvq_paged_append +
    kvq_paged_decode_attn + kvq_paged_flush.  Every slot's logical pages are mapped to
    shuffled physical pages at set-up, so flushes find their pages mapped."""
    import ctypes
    import torch
    import torch.distributed as dist
    import bit_kv_cache_gb300 as kvq
    lens0 = kvq_synth.slot_lengths(wl)
    grow = -(-(args.steps + args.warmup + 256) // N_LAYERS)
    max_T = (int(lens0.max()) + grow + 3 * wl.G) // wl.G * wl.G
    mp = max_T // wl.G
    K0, V0 = kvq_synth.prefill_kv(wl.replace(B=1), int(lens0.max()) + wl.G, replica=rank)
    K0 = torch.from_numpy(K0[0]).to(dev)
    V0 = torch.from_numpy(V0[0]).to(dev)
    rng = np.random.default_rng(wl.seed + 31 * rank)
    caches = []
    for li in range(N_LAYERS):
        c = kvq.KVQPagedCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, n_pages=wl.B * mp, max_T=max_T,
                              S=wl.S, R=wl.R, device=dev, v_bits=wl.v_bits)
        perm = rng.permutation(wl.B * mp).astype(np.int32).reshape(wl.B, mp)
        c.table.copy_(torch.from_numpy(perm))
        for b in range(wl.B):
            c.pages[b] = [int(x) for x in perm[b]]
        c.free = []
        for b in range(wl.B):
            L0 = int(lens0[b]) + (li * wl.G) // N_LAYERS
            Kb = torch.roll(K0, shifts=977 * (b + 3 * li), dims=1)[:, :L0].contiguous()
            Vb = torch.roll(V0, shifts=977 * (b + 3 * li), dims=1)[:, :L0].contiguous()
            rc = kvq.lib.kvq_paged_prefill(ctypes.byref(c.cfg), ctypes.byref(c.p), b,
                                           ctypes.c_void_p(Kb.data_ptr()), ctypes.c_void_p(Vb.data_ptr()), L0,
                                           kvq.KVQCache._stream())
            if rc:
                raise RuntimeError("paged prefill of slot %d failed: %d" % (b, rc))
            del Kb, Vb
        caches.append(c)
    del K0, V0
    kn, vn = kvq_synth.decode_tokens(wl, 64, replica=rank)
    qs = kvq_synth.queries(wl, 64, replica=rank)
    kn_d, vn_d, q_d = (torch.from_numpy(a).to(dev) for a in (kn, vn, qs))
    out = torch.empty((wl.B, wl.H_q, wl.D), dtype=torch.float16, device=dev)
    torch.cuda.synchronize()
    assert sum(c.read_status() for c in caches) == 0
    stream = torch.cuda.current_stream()
    lib = kvq.lib
    sp = ctypes.c_void_p(stream.cuda_stream)
    la = [(ctypes.byref(c.cfg), ctypes.byref(c.p), ctypes.c_void_p(c.ws.data_ptr()), c.ws.numel(), c.lens_host)
          for c in caches]
    knp = [ctypes.c_void_p(kn_d[j].data_ptr()) for j in range(64)]
    vnp = [ctypes.c_void_p(vn_d[j].data_ptr()) for j in range(64)]
    qp = [ctypes.c_void_p(q_d[j].data_ptr()) for j in range(64)]
    outp = ctypes.c_void_p(out.data_ptr())
    nfl = ctypes.c_int(0)
    nflr = ctypes.byref(nfl)

    def step(i, ev=None, inputs=None):
        cfg, pc, ws, wsb, lh = la[i % N_LAYERS]
        j = i % 64
        k_, v_, q_ = inputs if inputs else (knp[j], vnp[j], qp[j])
        rc = lib.kvq_paged_append(cfg, pc, k_, v_, sp)
        b = paged_bytes(wl, lh)
        if ev is not None:
            ev[0].record(stream)
        rc |= lib.kvq_paged_decode_attn(cfg, pc, q_, outp, ws, wsb, sp)
        if ev is not None:
            ev[1].record(stream)
        rc |= lib.kvq_paged_flush(cfg, pc, nflr, sp)
        if rc:
            raise RuntimeError("libkvq call failed in step %d" % i)
        return b, nfl.value

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total_bytes, flushes = 0, 0
    clk = Clocks(dev.index or 0)
    clk.start()
    torch.cuda.synchronize()
    w0 = time.time()
    t_start.record(stream)
    for i in range(K):
        b, f = step(args.warmup + i, evs[i])
        total_bytes += b
        flushes += 2 if f else 0  # a flush is one value and one key launch
    t_end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    clk.stop()
    ms = t_start.elapsed_time(t_end)
    dec_ms = [a.elapsed_time(bb) for a, bb in evs]
    # tens of thousands of live events slow down later runtime calls on the host
    # (one host-buffer step went from about 42 to 226 us of host time): free them
    # before the end-to-end leg
    del evs
    st = sum(c.read_status() for c in caches)
    if st != 0:
        print("device status %d" % st, file=sys.stderr)
    launches = 2 * K + flushes
    ms_max, bytes_all = reduce_over_ranks(ms, float(total_bytes), world, dev)

    # ---- end to end through the C ABI with pinned host buffers ----
    kn_h, vn_h, q_h = (torch.from_numpy(a).pin_memory() for a in (kn, vn, qs))
    out_h = torch.empty((wl.B, wl.H_q, wl.D), dtype=torch.float16).pin_memory()
    kn_s, vn_s, q_s = torch.empty_like(kn_d[0]), torch.empty_like(vn_d[0]), torch.empty_like(q_d[0])
    ins = (ctypes.c_void_p(kn_s.data_ptr()), ctypes.c_void_p(vn_s.data_ptr()), ctypes.c_void_p(q_s.data_ptr()))
    Ke = max(1, min(K, args.e2e_steps))
    e_bytes = 0
    for i in range(Ke + 3):
        if i == 3:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e_bytes = 0
        j = (args.warmup + K + i) % 64
        kn_s.copy_(kn_h[j], non_blocking=True)
        vn_s.copy_(vn_h[j], non_blocking=True)
        q_s.copy_(q_h[j], non_blocking=True)
        b, _ = step(args.warmup + K + i, inputs=ins)
        e_bytes += b
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()
    e_dt = time.perf_counter() - t0
    h2d = (kn_s.numel() + vn_s.numel() + q_s.numel()) * 2
    d2h = out.numel() * 2
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_kind = measured_peaks()
    value = bytes_all / (ms_max * 1e-3) / 1e9
    dec_avg_ms = statistics.mean(dec_ms)
    dec_bytes = total_bytes / K
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_max / K,
        "us_per_step": ms_max * 1e3 / K, "hbm_frac_step": value / world / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; shapes and outlier structure of the workload, ragged slot lengths)",
        "config": {"workload": wl.name, "B": wl.B, "H_q": wl.H_q, "H_kv": wl.H_kv, "D": wl.D,
                   "T_mean": wl.T, "slot_lengths": [int(x) for x in lens0], "G": wl.G, "R": wl.R,
                   "bits": wl.bits, "v_bits": wl.vbits, "S": wl.S, "mode": "kivi", "cache": "paged",
                   "step": "paged append + paged decode_attn + paged flush (when full), one layer",
                   "l2": "%d layer caches rotated (%.0f MB each, %.2f GB > 2 x L2)" % (
                       N_LAYERS, dec_bytes / 1e6, N_LAYERS * dec_bytes / 1e9),
                   "parallelism": "independent replicas per GPU" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": "decode_kernel (paged)", "us_per_launch": dec_avg_ms * 1e3,
                     "algorithmic_bytes_per_launch": dec_bytes, "traffic": profiled_traffic(wl.name)},
        "gpu_launches": launches,
        "clocks": clk.summary(w0, w1),
        "e2e": {"value": e_bytes / e_dt / 1e9 * world, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": e_dt / Ke * 1e6},
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama3_8b_gqa_b2", choices=sorted(kvq_synth.WORKLOADS))
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=24.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-quant-pack", action="store_true", help="skip the prefill quant/pack measurement")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--min-seconds", type=float, default=0.5,
                    help="repeat the K-step timed region until this much device time")
    ap.add_argument("--max-timed-steps", type=int, default=24000,
                    help="cap on the steps of all timed regions (sets the caches' capacity)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    wl = kvq_synth.WORKLOADS[args.workload]

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, wl, rank, world)

    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_gb300 as kvq
    if wl.ragged:
        return paged_main(args, wl, rank, world, dev)

    # ---- N_LAYERS layer caches: one seeded draw, rolled per layer; staggered fills ----
    extra = (wl.S + wl.R) if wl.mode == "kitty" else 0
    max_timed_steps = max(args.steps, args.max_timed_steps)
    grow = -(-(max_timed_steps + args.steps + args.warmup + args.e2e_steps + 256) // N_LAYERS)  # appends per layer
    max_T = wl.T + wl.G * (grow // wl.G + 3)
    L0 = wl.T + extra + wl.G - 1
    K0, V0 = kvq_synth.prefill_kv(wl, L0, replica=rank)
    K0 = torch.from_numpy(K0).to(dev)
    V0 = torch.from_numpy(V0).to(dev)
    caches = []
    for li in range(N_LAYERS):
        fill = (li * wl.G) // N_LAYERS              # residual fill after prefill
        Kl = torch.roll(K0, shifts=li * 977, dims=2)[:, :, : L0 - (wl.G - 1) + fill].contiguous()
        Vl = torch.roll(V0, shifts=li * 977, dims=2)[:, :, : L0 - (wl.G - 1) + fill].contiguous()
        c = kvq.KVQCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R,
                         n_boost=wl.n_boost, mode=wl.mode, max_T=max_T, device=dev, v_bits=wl.v_bits,
                         rope_base=wl.rope_base)
        c.prefill(Kl, Vl)
        caches.append(c)
        del Kl, Vl
    del K0, V0
    kn, vn = kvq_synth.decode_tokens(wl, 64, replica=rank)
    qs = kvq_synth.queries(wl, 64, replica=rank)
    kn_d = torch.from_numpy(kn).to(dev)
    vn_d = torch.from_numpy(vn).to(dev)
    q_d = torch.from_numpy(qs).to(dev)
    out = torch.empty((wl.B, wl.H_q, wl.D), dtype=torch.float16, device=dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    # The timed steps call the C ABI directly with prepared arguments, so that the
    # host enqueues ahead of the GPU and the device time is the kernels' own.
    import ctypes
    lib = kvq.lib
    sp = ctypes.c_void_p(stream.cuda_stream)
    layer_args = [(ctypes.byref(c.cfg), ctypes.byref(c.c), ctypes.c_void_p(c.ws.data_ptr()), c.ws.numel(), c.c)
                  for c in caches]
    knp = [ctypes.c_void_p(kn_d[j].data_ptr()) for j in range(64)]
    vnp = [ctypes.c_void_p(vn_d[j].data_ptr()) for j in range(64)]
    qp = [ctypes.c_void_p(q_d[j].data_ptr()) for j in range(64)]
    outp = ctypes.c_void_p(out.data_ptr())
    fk, fv = ctypes.c_int(0), ctypes.c_int(0)
    fkr, fvr = ctypes.byref(fk), ctypes.byref(fv)

    # KIVI caches on the packed-tile path insert and attend in one launch
    # (kvq_append_decode); the others append, then attend.
    tok = 256 // wl.bits
    one_launch = wl.mode != "kitty" and wl.D == 128 and wl.H_q // wl.H_kv <= 4 and wl.G % tok == 0
    fused = ctypes.c_int(0)
    fusedr = ctypes.byref(fused)
    cap = wl.G if wl.mode == "kitty" else wl.R

    f_ad, f_fl = lib.kvq_append_decode, lib.kvq_flush_group

    def step_one(i, fl_ev):
        """One-launch step with nothing but the two C-ABI calls (and events around a
        flush launch): the host stays ahead of the device.  Bytes: replay_steps."""
        cfg, cc, ws, wsb, st = layer_args[i % N_LAYERS]
        j = i & 63
        rc = f_ad(cfg, cc, knp[j], vnp[j], qp[j], outp, ws, wsb, fusedr, sp)
        if not fused.value:
            raise RuntimeError("step %d was not one launch" % i)
        if st.n_kres == cap:    # the flush below launches
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record(stream)
            rc |= f_fl(cfg, cc, fkr, fvr, sp)
            ev[1].record(stream)
            fl_ev.append(ev)
        else:
            rc |= f_fl(cfg, cc, fkr, fvr, sp)
        if rc:
            raise RuntimeError("libkvq call failed in step %d" % i)
        return fk.value + fv.value

    def step(i, fl_ev=None, dec_ev=None):
        """One step; fl_ev / dec_ev (lists) receive event pairs around a flush launch and
        around the attention launch (dec_ev only where the step has separate launches)."""
        cfg, cc, ws, wsb, st = layer_args[i % N_LAYERS]
        j = i % 64
        if one_launch:
            b = decode_bytes(wl, after_append(wl, caches[i % N_LAYERS].lengths))
            rc = lib.kvq_append_decode(cfg, cc, knp[j], vnp[j], qp[j], outp, ws, wsb, fusedr, sp)
            if not fused.value:
                raise RuntimeError("step %d was not one launch" % i)
        else:
            rc = lib.kvq_append_token(cfg, cc, knp[j], vnp[j], sp)
            b = decode_bytes_struct(wl, st)
            ev = None
            if dec_ev is not None:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record(stream)
            rc |= lib.kvq_decode_attn(cfg, cc, qp[j], outp, ws, wsb, sp)
            if ev is not None:
                ev[1].record(stream)
                dec_ev.append(ev)
        full = st.n_kres == cap or st.n_vres == cap     # the flush below launches
        ev = None
        if full and fl_ev is not None:
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record(stream)
        rc |= lib.kvq_flush_group(cfg, cc, fkr, fvr, sp)
        if ev is not None:
            ev[1].record(stream)
            fl_ev.append(ev)
        if rc:
            raise RuntimeError("libkvq call failed in step %d" % i)
        return b, fk.value + fv.value

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # Timed regions of K steps, repeated until about min_seconds of device time (at least
    # one region).  Only flush launches (rare) and, where a step has separate append and
    # attention launches, the attention launch carry events inside a region: events between
    # kernels would stop one decode launch from starting as the previous one drains.
    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    region_ms, region_bytes = [], []
    flush_ms, dec_ms = [], []
    flushes = 0
    done = 0
    clk = Clocks(local)
    clk.start()
    torch.cuda.synchronize()
    w0 = time.time()
    reps = None
    states = [dict(c.lengths) for c in caches] if one_launch else None
    while True:
        fl_ev, dec_ev = [], ([] if not one_launch else None)
        nbytes = 0
        s0 = args.warmup + done
        if one_launch:
            t_start.record(stream)
            for s in range(s0, s0 + K):
                flushes += step_one(s, fl_ev)
            t_end.record(stream)
            nbytes = replay_steps(wl, states, s0, K, cap)
        else:
            t_start.record(stream)
            for s in range(K):
                b, f = step(s0 + s, fl_ev, dec_ev)
                nbytes += b
                flushes += f
            t_end.record(stream)
        torch.cuda.synchronize()
        done += K
        region_ms.append(t_start.elapsed_time(t_end))
        region_bytes.append(nbytes)
        flush_ms.append(sum(a.elapsed_time(bb) for a, bb in fl_ev))
        if dec_ev is not None:
            dec_ms.extend(a.elapsed_time(bb) for a, bb in dec_ev)
        del fl_ev, dec_ev
        if reps is None:      # regions to run: enough for min_seconds, within the cache capacity
            want = int(np.ceil(args.min_seconds * 1e3 / max(region_ms[0], 1e-3)))
            reps = max(1, min(want, max_timed_steps // K))
            if world > 1:
                r = torch.tensor([reps], dtype=torch.int64, device=dev)
                dist.all_reduce(r, op=dist.ReduceOp.MAX)
                reps = int(r[0])
        if len(region_ms) >= reps:
            break
    w1 = time.time()
    clk.stop()
    if one_launch:      # the replayed lengths are the caches' own
        for c, st in zip(caches, states):
            if dict(c.lengths) != st:
                raise RuntimeError("replayed lengths %s differ from the cache's %s" % (st, c.lengths))
    ms = sum(region_ms)
    total_bytes = sum(region_bytes)
    steps_timed = K * len(region_ms)
    st = sum(c.read_status() for c in caches)
    if st != 0:
        print("device status %d" % st, file=sys.stderr)
    launches = (1 if one_launch else 2) * steps_timed + flushes
    ms_max, bytes_all = reduce_over_ranks(ms, float(total_bytes), world, dev)
    per_step = sorted(r / K for r in region_ms)

    # ---- end to end through host buffers: one kvq_decode_step_host_wait call per step
    # (inputs in, append, attend, flush, output out; pinned memory, which the kernels
    # read and write in place; the call returns once the output is in host memory),
    # through the C ABI with prepared arguments ----
    kn_h = torch.from_numpy(kn).pin_memory()
    vn_h = torch.from_numpy(vn).pin_memory()
    q_h = torch.from_numpy(qs).pin_memory()
    out_h = torch.empty((wl.B, wl.H_q, wl.D), dtype=torch.float16).pin_memory()
    hk = [ctypes.c_void_p(kn_h[j].data_ptr()) for j in range(64)]
    hv = [ctypes.c_void_p(vn_h[j].data_ptr()) for j in range(64)]
    hq = [ctypes.c_void_p(q_h[j].data_ptr()) for j in range(64)]
    ho = ctypes.c_void_p(out_h.data_ptr())
    done_h = torch.zeros(1, dtype=torch.int32).pin_memory()     # the call's completion count
    hd = ctypes.c_void_p(done_h.data_ptr())
    Ke = max(1, min(steps_timed, args.e2e_steps))
    first = args.warmup + done
    e_bytes = 0
    if one_launch:      # the timed steps' bytes, replayed from the lengths before the loop
        st_e = [dict(c.lengths) for c in caches]
        replay_steps(wl, st_e, first, 3, caches[0].cfg.R)
        e_bytes = replay_steps(wl, st_e, first + 3, Ke, caches[0].cfg.R)
    for i in range(Ke + 3):
        if i == 3:
            t0 = time.perf_counter()
        li = (first + i) % N_LAYERS
        cfg, cc, ws, wsb, _ = layer_args[li]
        j = i % 64
        if not one_launch and i >= 3:
            e_bytes += decode_bytes(wl, after_append(wl, caches[li].lengths))
        rc = lib.kvq_decode_step_host_wait(cfg, cc, hq[j], hk[j], hv[j], ho, hd, ws, wsb, fkr, fvr, sp)
        if rc:
            raise RuntimeError("kvq_decode_step_host_wait failed: %d" % rc)
    e_dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    h2d = (kn_h[0].numel() + vn_h[0].numel() + q_h[0].numel()) * 2
    d2h = out_h.numel() * 2

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_kind = measured_peaks()
    value = bytes_all / (ms_max * 1e-3) / 1e9
    dec_bytes = total_bytes / steps_timed
    if one_launch:      # the step's own launch, without the flushes
        dec_avg_ms = (ms - sum(flush_ms)) / steps_timed
    else:
        dec_avg_ms = statistics.mean(dec_ms)
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = profiled_traffic(wl.name)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": statistics.median(per_step),
        "ms_per_step_min": per_step[0], "ms_per_step_max": per_step[-1],
        "us_per_step": statistics.median(per_step) * 1e3, "hbm_frac_step": value / world / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; shapes and outlier structure of the workload)",
        "config": {"workload": wl.name, "B": wl.B, "H_q": wl.H_q, "H_kv": wl.H_kv, "D": wl.D,
                   "T": wl.T, "G": wl.G, "R": wl.R, "bits": wl.bits, "v_bits": wl.vbits, "S": wl.S,
                   "n_boost": wl.n_boost, "mode": wl.mode, "rope_base": wl.rope_base,
                   "step": ("append_decode (one launch)" if one_launch else "append_token + decode_attn")
                           + " + flush_group (when full), one layer",
                   "l2": "%d layer caches rotated (%.0f MB each, %.2f GB > 2 x L2)" % (
                       N_LAYERS, dec_bytes / 1e6, N_LAYERS * dec_bytes / 1e9),
                   "parallelism": "independent replicas per GPU" if world > 1 else "single GPU"},
        "timing": {"regions": len(region_ms), "steps_timed": steps_timed, "device_s": ms * 1e-3,
                   "per_region": "K steps between two events; median / min / max of region time / K"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": "decode_kernel", "us_per_launch": dec_avg_ms * 1e3,
                     "algorithmic_bytes_per_launch": dec_bytes, "traffic": traffic,
                     "launch_time": ("(timed regions - flush launches) / steps" if one_launch
                                     else "mean of events around each attention launch")},
        "gpu_launches": launches,
        "clocks": clk.summary(w0, w1),
        "e2e": {"value": e_bytes / e_dt / 1e9 * world, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": e_dt / Ke * 1e6,
                "call": "kvq_decode_step_host_wait (returns with the output in host memory)"},
    }
    if not args.no_quant_pack and world == 1:
        line["quant_pack"] = quant_pack_measure(kvq, dev, peak)
    if wl.name == "long_128k" and world == 1:
        line["sequence"] = long_sequence_measure(kvq, dev, peak)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
