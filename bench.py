"""Decode-step benchmark of the GB300 low-bit KV cache.

Default workload: the Llama-3-8B-shaped GQA layer (B=4, H_q=32, H_kv=8, D=128,
T=32768 packed 2-bit tokens, G=R=128).  One step = one decode step of one layer
in the Kitty pipeline order: append the new token (kvq_append_token), attend
(kvq_decode_attn), quantize the residual when it is full (kvq_flush_group).  The
benchmark rotates through four independent layer caches (4 x 77.7 MB > 2 x L2),
so no step finds its cache in L2.

value  = effective packed-KV bandwidth: algorithmic bytes of all timed steps
         (codes + fp16 scales/mins + fp16 sink/residual + q + out, summed per step
         from the cache state) / device time.  Whole job: summed over ranks.
e2e    = the same through host buffers: per step, pinned q / k_new / v_new copied
         in, the step run, out copied back, stream synchronized.
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

N_LAYERS = 4
METRIC = None


def load_baseline():
    with open(os.path.join(ROOT, "BASELINE.json")) as f:
        return json.load(f)


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
    b = U * T_k * D * kb // 8 + U * (T_k // G) * D * 4              # key codes + (scale, min)
    if wl.mode == "kitty" and wl.n_boost:
        b += U * T_k * wl.n_boost * 2 // 8 + U * (T_k // G) * D      # high plane + boost index
    b += U * T_v * D * wl.bits // 8 + U * T_v * (D // Gv) * 4       # value codes + (scale, min)
    n16 = lengths["n_sink"] * 2 + lengths["n_kres"] + lengths["n_vres"] + lengths["n_local"]
    b += U * n16 * D * 2                                           # fp16 sink / buffers
    b += 2 * wl.B * wl.H_q * D * 2                                 # q in, out
    return b


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in ("kvq_decode.cu", "kvq_device.cuh", "kvq_internal.h"):
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
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.p is None:
            return
        time.sleep(0.15)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def cpu_oracle_rate(wl, max_seconds: float, n_units: int = 1):
    """The oracle (single thread, fp64) on a bounded sample: decode attention over
    n_units (b, h_kv) sequences of the workload.  Returns (GB/s in the benchmark's
    byte accounting, seconds, steps, sample description)."""
    import oracle
    L0 = wl.T + 64
    rng = np.random.default_rng(1)
    sub = wl.replace(B=1, H_kv=n_units, H_q=n_units * wl.g)
    K, V = kvq_synth.prefill_kv(wl.replace(B=1, H_kv=min(wl.H_kv, n_units)), L0)
    ora = oracle.OracleCache(sub.B, sub.H_q, sub.H_kv, sub.D, sub.G, sub.bits, S=sub.S, R=sub.R,
                             n_boost=sub.n_boost, mode=sub.mode)
    ora.prefill(K, V)
    q = kvq_synth.queries(sub, 1)[0]
    lengths = dict(n_sink=ora.n_sink, T_k=ora.T_k, n_kres=ora.n_kres, T_v=ora.T_v,
                   n_vres=ora.n_vres, n_local=ora.n_local)
    per = decode_bytes(sub, lengths)
    t0 = time.perf_counter()
    steps = 0
    while True:
        ora.attend(q)
        steps += 1
        if time.perf_counter() - t0 >= max_seconds:
            break
    dt = time.perf_counter() - t0
    desc = ("oracle decode attention (fp64, 1 thread) over %d of %d (b,h_kv) sequences, "
            "%d tokens each, %d repetitions" % (n_units, wl.B * wl.H_kv, L0, steps))
    del rng
    return per * steps / dt / 1e9, dt, steps, desc


def reference_arm(args, wl, baseline, rank, world):
    """--impl reference: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return 0
    K, W = args.steps, args.warmup
    import oracle
    L0 = wl.T + 64
    sub = wl.replace(B=1, H_kv=1, H_q=wl.g)
    Kx, Vx = kvq_synth.prefill_kv(sub, L0)
    ora = oracle.OracleCache(sub.B, sub.H_q, sub.H_kv, sub.D, sub.G, sub.bits, S=sub.S, R=sub.R,
                             n_boost=sub.n_boost, mode=sub.mode)
    ora.prefill(Kx, Vx)
    qs = kvq_synth.queries(sub, 4)
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
    sample = ("per step: oracle decode attention over 1 of %d (b,h_kv) sequences (%d tokens, "
              "fp64, single thread)" % (wl.B * wl.H_kv, L0))
    line = {"impl": "reference", "metric": baseline["metric"], "value": val, "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": dt / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, shapes of the workload)",
            "config": {"workload": wl.name, "B": wl.B, "H_q": wl.H_q, "H_kv": wl.H_kv, "D": wl.D,
                       "T": wl.T, "G": wl.G, "bits": wl.bits},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama3_8b_gqa_b2", choices=sorted(kvq_synth.WORKLOADS))
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    baseline = load_baseline()
    wl = kvq_synth.WORKLOADS[args.workload]

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, wl, baseline, rank, world)

    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_gb300 as kvq

    # ---- N_LAYERS independent layer caches, residual fills staggered ----
    caches = []
    L_fill = [64, 96, 0, 32]
    for li in range(N_LAYERS):
        Kx, Vx = kvq_synth.prefill_kv(wl, wl.T + L_fill[li] + (wl.S if wl.mode == "kitty" else 0)
                                      + (wl.R if wl.mode == "kitty" else 0), replica=li + 16 * rank)
        c = kvq.KVQCache(wl.B, wl.H_q, wl.H_kv, wl.D, wl.G, wl.bits, S=wl.S, R=wl.R,
                         n_boost=wl.n_boost, mode=wl.mode, max_T=wl.T + 8 * wl.G, device=dev)
        c.prefill(torch.from_numpy(Kx).to(dev), torch.from_numpy(Vx).to(dev))
        del Kx, Vx
        caches.append(c)
    n_tok = args.steps + args.warmup + 8
    kn, vn = kvq_synth.decode_tokens(wl, 64, replica=rank)
    qs = kvq_synth.queries(wl, 64, replica=rank)
    kn_d = torch.from_numpy(kn).to(dev)
    vn_d = torch.from_numpy(vn).to(dev)
    q_d = torch.from_numpy(qs).to(dev)
    out = torch.empty((wl.B, wl.H_q, wl.D), dtype=torch.float16, device=dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        c = caches[i % N_LAYERS]
        j = i % 64
        c.append_token(kn_d[j], vn_d[j])
        b = decode_bytes(wl, c.lengths)
        if ev is not None:
            ev[0].record(stream)
        c.decode_attn(q_d[j], out)
        if ev is not None:
            ev[1].record(stream)
        fk, fv = c.flush_group()
        return b, int(fk) + int(fv)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total_bytes = 0
    flushes = 0
    with Clocks(local) as clk:
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(K):
            b, f = step(args.warmup + i, evs[i])
            total_bytes += b
            flushes += f
        t_end.record(stream)
        torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_end)
    dec_ms = [a.elapsed_time(bb) for a, bb in evs]
    st = sum(c.read_status() for c in caches)
    if st != 0:
        print("device status %d" % st, file=sys.stderr)
    launches = 2 * K + flushes
    if world > 1:
        t = torch.tensor([ms, float(total_bytes)], dtype=torch.float64, device=dev)
        mx = t.clone()
        dist.all_reduce(mx[:1], op=dist.ReduceOp.MAX)
        dist.all_reduce(t[1:], op=dist.ReduceOp.SUM)
        ms_max, bytes_all = float(mx[0]), float(t[1])
    else:
        ms_max, bytes_all = ms, float(total_bytes)

    # ---- end to end through host buffers (public API, pinned memory) ----
    kn_h = torch.from_numpy(kn).pin_memory()
    vn_h = torch.from_numpy(vn).pin_memory()
    q_h = torch.from_numpy(qs).pin_memory()
    out_h = torch.empty((wl.B, wl.H_q, wl.D), dtype=torch.float16).pin_memory()
    kn_s = torch.empty_like(kn_d[0])
    vn_s = torch.empty_like(vn_d[0])
    q_s = torch.empty_like(q_d[0])
    Ke = min(K, 200)
    e_bytes = 0
    for i in range(Ke + 3):
        if i == 3:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e_bytes = 0
        c = caches[i % N_LAYERS]
        j = i % 64
        kn_s.copy_(kn_h[j], non_blocking=True)
        vn_s.copy_(vn_h[j], non_blocking=True)
        q_s.copy_(q_h[j], non_blocking=True)
        c.append_token(kn_s, vn_s)
        e_bytes += decode_bytes(wl, c.lengths)
        c.decode_attn(q_s, out)
        c.flush_group()
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
    us_step = ms_max * 1e3 / K
    value = bytes_all / (ms_max * 1e-3) / 1e9
    dec_avg_ms = statistics.mean(dec_ms)
    dec_bytes = total_bytes / K
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = profiled_traffic(wl.name)
    line = {
        "metric": baseline["metric"], "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_max / K,
        "us_per_step": us_step, "hbm_frac_step": value / world / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; shapes and outlier structure of the workload)",
        "config": {"workload": wl.name, "B": wl.B, "H_q": wl.H_q, "H_kv": wl.H_kv, "D": wl.D,
                   "T": wl.T, "G": wl.G, "R": wl.R, "bits": wl.bits, "S": wl.S,
                   "n_boost": wl.n_boost, "mode": wl.mode,
                   "step": "append_token + decode_attn + flush_group (when full), one layer",
                   "l2": "%d layer caches rotated (%.0f MB each, > 2 x L2)" % (
                       N_LAYERS, dec_bytes / 1e6),
                   "parallelism": "independent replicas per GPU" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": "decode_kernel", "us_per_launch": dec_avg_ms * 1e3,
                     "algorithmic_bytes_per_launch": dec_bytes, "traffic": traffic},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": {"value": e_bytes / e_dt / 1e9 * world, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": e_dt / Ke * 1e6},
    }
    if not args.no_cpu_baseline and world == 1:
        v, dt, n, desc = cpu_oracle_rate(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
