"""Benchmark of one delta-rule token-mixer layer: forward + backward tokens/s.

One step = dr_fwd + dr_bwd (the backward reusing the forward's residuals)
through the C ABI over one batch of synthetic inputs already resident in HBM.
Prints ONE JSON line (rank 0).  With --impl reference the fp64 CPU oracle is
timed instead, on a bounded sample of the same workload, on the host cores.

Multi-GPU: the layer has no cross-sequence exchange, so N ranks run N
independent replicas of the workload (weak scaling); the only collectives are
the timing barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "gdn_h0_b8_t4096_h16_d128"
METRIC = "fwd+bwd tokens/s per delta-rule layer (T=4096,H=16,d=128)"


def algorithmic(w, N):
    """Per-step algorithmic FLOPs and bytes of the whole path (fwd + bwd), per
    token per head: F = 24 C dk + 14 C dv + 22 dk dv + 16/3 C^2 and
    bytes = 3 s (2 dk + dv) + 2 s dv + 12 + 3 G (s = io bytes, G = gate bytes),
    plus 5 dk dv 4 bytes of state per sequence and head when states are used."""
    C, dk, dv = w.chunk, w.dk, w.dv
    s = 2 if w.io == "bf16" else 4
    G = {"deltanet": 0, "gdn": 4, "kda": 4 * dk}[w.variant]
    th = w.B * w.T * w.H
    flops = th * (24 * C * dk + 14 * C * dv + 22 * dk * dv + 16.0 / 3.0 * C * C)
    byts = th * (3 * s * (2 * dk + dv) + 2 * s * dv + 12 + 3 * G)
    if w.h0:
        byts += 5 * dk * dv * 4 * N * w.H
    return flops, byts


_FWD_SRC = ("delta_rule_recurrent_gated_gb300/csrc/tc_fwd.cu",
            "cc35122664e52feb61b1e5bc8fceccfdd30e7d046d1767f11a1e4d53cd275fc8")
_BWD_SRC = ("delta_rule_recurrent_gated_gb300/csrc/tc_bwd.cu",
            "da69fd81708bc3ef9f74f066f270bd673f5db1a4875a46a25e1090022b9b71bc")
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of each kernel,
# from an ncu capture of the timed step of the full-size workload (profiles/
# dram_traffic_gdn_kda_b8_t4096_h16_d128.md), with the source file it was taken on
MEASURED_TRAFFIC = {
    ("gdn_h0_b8_t4096_h16_d128", "tc_prep"): (430136832 + 686508800, _FWD_SRC),
    ("gdn_h0_b8_t4096_h16_d128", "tc_scan_fwd"): (687477504 + 495796992, _FWD_SRC),
    ("gdn_h0_b8_t4096_h16_d128", "tc_scan_bwd"): (541128192 + 360294912, _BWD_SRC),
    ("gdn_h0_b8_t4096_h16_d128", "tc_bwd_chunk"): (1418410240 + 383005184, _BWD_SRC),
    ("kda_b8_t4096_h16_d128", "tc_prep"): (693737472 + 691343360, _FWD_SRC),
    ("kda_b8_t4096_h16_d128", "tc_scan_fwd"): (679206400 + 497192192, _FWD_SRC),
    ("kda_b8_t4096_h16_d128", "tc_scan_bwd"): (541140224 + 360376832, _BWD_SRC),
    ("kda_b8_t4096_h16_d128", "tc_bwd_chunk"): (1691225856 + 637511680, _BWD_SRC),
}


def measured_traffic(name, w):
    """DRAM bytes of one launch of `name` on workload w from the recorded capture, or None
    (no capture of that workload, or the kernel's source changed since)."""
    rec = MEASURED_TRAFFIC.get((w.name, name))
    if rec is None:
        return None
    byts, (src, sha) = rec
    try:
        with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), src), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha:
                return None
    except OSError:
        return None
    return byts


def kernel_bytes(name, w, N):
    """Bytes a kernel must move by design (its inputs and outputs), per launch."""
    D, H, th = w.dk, w.H, w.B * w.T * w.H
    chunks = (w.T + 63) // 64 * w.B
    recs = chunks * H
    tile, dd = 64 * D * 2, D * D * 2
    g = {"deltanet": 0, "gdn": 4, "kda": 4 * D}[w.variant]
    if name == "tc_prep":            # q, k, v, beta, g in; Wy, Qt, KC, Ut, Ot, T, gC out
        return th * (3 * D * 2 + 4 + g) + recs * (5 * tile + 8192 + D * 4)
    if name == "tc_scan_fwd":        # Wy, Qt, KC, Ut, Ot, gC in; o, U, S out
        return recs * (5 * tile + D * 4) + th * D * 2 + recs * (tile + dd)
    if name == "tc_scan_bwd":        # KC, Qt, Wy, gC, dO in; dU, dS out
        return recs * (3 * tile + D * 4) + th * D * 2 + recs * (tile + dd)
    if name == "tc_bwd_chunk":       # q, k, v, dO, beta, g, U, -dU^T, S, dS, T, gC in;
        return (th * (4 * D * 2 + 4 + g) + recs * (2 * tile + 2 * dd + 8192 + D * 4)
                + th * (3 * D * 2 + 4 + g))             # dq, dk, dv, dbeta, dg out
    return 0


def kernel_algorithmic_bytes(name, w, N):
    """The part of the whole path's algorithmic bytes (the formula of `algorithmic`) that
    each kernel of the step owns, per launch: tc_prep reads q, k, v, beta, g; the forward
    scan writes o (and reads h0, writes hT); the backward scan reads dhT and h0 and writes
    dh0; tc_bwd_chunk reads q, k, v, dO, beta, g and writes dq, dk, dv, dbeta, dg.  The
    four add up to `algorithmic`'s bytes."""
    s = 2 if w.io == "bf16" else 4
    G = {"deltanet": 0, "gdn": 4, "kda": 4 * w.dk}[w.variant]
    th = w.B * w.T * w.H
    st = w.dk * w.dv * 4 * N * w.H if w.h0 else 0
    if name == "tc_prep":
        return th * (s * (2 * w.dk + w.dv) + 4 + G)
    if name == "tc_scan_fwd":
        return th * s * w.dv + 2 * st
    if name == "tc_scan_bwd":
        return 3 * st
    if name == "tc_bwd_chunk":
        return th * (s * (4 * w.dk + 3 * w.dv) + 8 + 2 * G)
    return 0


def config_of(w, world):
    """The `config` object of both arms' JSON lines."""
    return {"workload": w.name, "variant": w.variant, "global_batch": w.B * world,
            "seq_len": w.T, "heads": w.H, "d_k": w.dk, "d_v": w.dv, "chunk": w.chunk,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (no flush needed)"}


DECODE_B, DECODE_H, DECODE_D = 256, 16, 128


def decode_bench(dev, stream, max_over_ranks, barrier, steps=20, warmup=3):
    """The recurrent step (dr_decode) at serving batch: GDN, 256 sequences x 16 heads,
    d = 128, one bf16 token per sequence per call, state [256, 16, 128, 128] fp32
    (256 MiB, larger than L2) updated in place.  HBM-bound on the state: the roofline
    bytes of a call are one read and one write of the state plus the token rows."""
    import torch
    from delta_rule_recurrent_gated_gb300 import binding
    B, H, D = DECODE_B, DECODE_H, DECODE_D
    gen = torch.Generator().manual_seed(0)
    q = torch.nn.functional.normalize(torch.randn(B, 1, H, D, generator=gen), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(B, 1, H, D, generator=gen), dim=-1)
    v = torch.randn(B, 1, H, D, generator=gen)
    beta = torch.sigmoid(torch.randn(B, 1, H, generator=gen))
    g = -torch.nn.functional.softplus(torch.randn(B, 1, H, generator=gen)) * 0.1
    state = torch.randn(B, H, D, D, generator=gen) * 0.02
    q, k, v = (t.to(torch.bfloat16).to(dev) for t in (q, k, v))
    beta, g, state = beta.to(dev), g.to(dev), state.to(dev)
    dec = binding.Decoder("gdn", B, 1, H, D, D, io="bf16", out="bf16", device=dev)
    o = torch.empty(B, 1, H, D, dtype=torch.bfloat16, device=dev)
    for _ in range(warmup):
        dec.step(q, k, v, beta, g, state, o=o)
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        dec.step(q, k, v, beta, g, state, o=o)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps)
    nbytes = 2 * B * H * D * D * 4 + B * H * (4 * D * 2 + 8)
    hbm, _, peak_src = measured_peaks()
    ach = nbytes / (ms / 1e3) / 1e9
    return {"workload": f"gdn_decode_b{B}_h{H}_d{D}_1tok", "value": B / (ms / 1e3),
            "unit": "tokens/s", "ms_per_call": ms, "steps": steps, "warmup": warmup,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                         "frac": ach / hbm, "bytes_per_call": nbytes,
                         "peak_source": f"{peak_src} hbm_gbs (copy, burst)"}}


def gdn2_flops_per_chunk(C, d):
    """FLOPs of one (chunk, head) of the Gated DeltaNet-2 forward + backward in the
    chunkwise form as run with DR_FLAG_REUSE_FWD (dense products, triangular ones counted
    in full, each product once): the forward's chunk-local products (11 of C x C x d), the
    inverse (C^3 / 3) and the state products (4 of C x d x d); the backward, which reads
    the forward's per-chunk records, adds 20 C x C x d, 8 C x d x d and 2 C x C x C
    products."""
    fwd = 22 * C * C * d + C ** 3 / 3 + 8 * C * d * d
    return fwd + 40 * C * C * d + 16 * C * d * d + 4 * C ** 3


def fp32_alu_peak_tflops(sm_mhz):
    """fp32 FMA peak: 152 SMs x 128 fp32 lanes x 2 flops x the SM clock under load."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


def gdn2_bench(dev, stream, max_over_ranks, barrier, sm_mhz, steps=3, warmup=3):
    """Gated DeltaNet-2 forward + backward (dr_gdn2_fwd / dr_gdn2_bwd) on its workload,
    device-resident inputs, CUDA events on the launching stream."""
    import torch
    from delta_rule_recurrent_gated_gb300 import binding, inputs
    w = inputs.get("gdn2_b4_t2048_h8_d64")
    x = inputs.make_gdn2(w, seed=0)
    t = {n: (v.to(dev) if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    prob = binding.Gdn2Problem(w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io, out="bf16",
                               grad="bf16", scale=w.scale, device=dev)
    o = torch.empty(w.B, w.T, w.H, w.dv, dtype=torch.bfloat16, device=dev)
    hT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)

    def step():
        prob.forward(t["q"], t["k"], t["v"], t["erase"], t["write"], t["g"], t["h0"], o=o, hT=hT)
        prob.backward(t["q"], t["k"], t["v"], t["erase"], t["write"], t["g"], t["h0"], t["dO"],
                      t["dhT"], reuse_fwd=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    binding.trace_enable(3 * steps + 3)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    assert prob.status() == binding.DR_OK
    launches = binding.trace_read()
    binding.trace_enable(0)
    ms = max_over_ranks(e0.elapsed_time(e1) / steps)
    chunks = w.B * w.H * ((w.T + w.chunk - 1) // w.chunk)
    flops = chunks * gdn2_flops_per_chunk(w.chunk, w.dk)
    peak = fp32_alu_peak_tflops(sm_mhz)
    ach = flops / (ms / 1e3) / 1e12
    kern = {}
    for nm, kms in launches:
        tot, n = kern.get(nm, (0.0, 0))
        kern[nm] = (tot + kms, n + 1)
    return {"workload": w.name, "value": w.tokens / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "steps": steps, "warmup": warmup, "dtype": "f32 (bf16 io)",
            "kernels": {nm: {"launches": n, "ms_per_launch": tot / n} for nm, (tot, n) in kern.items()},
            "roofline": {"bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                         "frac": ach / peak, "flops_per_step": flops,
                         "peak_source": f"fp32 FMA: 152 SMs x 128 lanes x 2 x {sm_mhz:.0f} MHz"}}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def prepare_bench(args, w, rank, world, dev, stream, plain_ms, o, hT, grads, max_over_ranks,
                  barrier):
    import torch
    from delta_rule_recurrent_gated_gb300 import binding, inputs
    xr = inputs.make_raw(w, seed=rank)
    tr = {n: (v.to(dev) if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in xr.items()}
    prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io,
                           out="bf16", grad="bf16", scale=w.scale,
                           cu_seqlens=xr["cu_seqlens"], device=dev, prepare=True)

    def step_p(src):
        prob.forward(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"], o=o, hT=hT)
        prob.backward(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"], src["dO"],
                      src["dhT"], reuse_fwd=True, out=grads)

    for _ in range(args.warmup):
        step_p(tr)
    torch.cuda.synchronize(dev)
    binding.trace_enable(12 * args.steps + 12)
    barrier()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        step_p(tr)
    p1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    st = prob.status()
    assert st == binding.DR_OK, binding.error_string(st)
    launches = binding.trace_read()
    binding.trace_enable(0)
    p_ms = max_over_ranks(p0.elapsed_time(p1) / args.steps)
    kern = {}
    for nm, kms in launches:
        tot, n = kern.get(nm, (0.0, 0))
        kern[nm] = (tot + kms, n + 1)
    kern = {nm: {"launches": n, "ms_per_launch": tot / n} for nm, (tot, n) in kern.items()}
    del prob
    torch.cuda.empty_cache()
    return {"value": w.tokens * world / (p_ms / 1e3), "unit": "tokens/s", "ms_per_step": p_ms,
            "ms_over_plain_step": p_ms - plain_ms, "kernels": kern,
            "fused": "the maps run inside tc_prep and tc_bwd_chunk on the raw tiles",
            "inputs": "raw q, k ~ N(0,1), beta logits ~ N(0,1), gate arguments ~ N(0,1)"}


def oracle_step(w, x, units):
    """One timed pass of the fp64 oracle (forward + backward, as it stands) over the given
    (sequence, head) units of the workload; returns (seconds, token-equivalents), a token
    of the layer carrying H heads."""
    import numpy as np
    import oracle
    a = dict(q=x["q"], k=x["k"], v=x["v"], beta=x["beta"], g=x["g"], h0=x["h0"],
             cu_seqlens=x["cu_seqlens"], scale=w.scale)
    u = np.asarray(units, dtype=np.int32)
    t0 = time.perf_counter()
    oracle.forward(w.variant, units=u, **a)
    oracle.backward(w.variant, dO=x["dO"], dhT=x["dhT"], units=u, **a)
    secs = time.perf_counter() - t0
    N = x["N"]
    tok_per_unit = w.T if x["cu_seqlens"] is None else w.T / max(N, 1)
    return secs, len(u) * tok_per_unit / w.H


def cpu_baseline(w, x, budget_s=12.0):
    """Time the fp64 oracle (forward + backward, as it stands) on whole (sequence, head)
    units of the workload on the host cores, one unit per thread per pass, for about
    budget_s seconds, and express it as tokens/s of the layer."""
    import oracle
    threads = oracle.max_threads()
    total = x["N"] * w.H
    secs = toks = 0.0
    done = 0
    while done < total and (secs < budget_s or done == 0):
        n = min(threads, total - done)
        dt, tk = oracle_step(w, x, range(done, done + n))
        secs, toks, done = secs + dt, toks + tk, done + n
    return {"value": toks / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} of {total} (sequence, head) units of {w.name}, "
                      f"fp64 forward+backward, {secs:.1f} s on {threads} threads"}


def run_reference(args, w):
    """The reference arm: the fp64 oracle as it stands on the host cores.  Each step is
    one pass over `threads` (sequence, head) units of the workload (a bounded sample,
    different units every step); ms_per_step is that pass's wall time and value the
    token-equivalents it processed per second."""
    from delta_rule_recurrent_gated_gb300.replicas import Replicas
    if not Replicas.from_env().is_root:  # the oracle runs once, on rank 0's host cores
        return
    import oracle
    from delta_rule_recurrent_gated_gb300 import inputs
    x = inputs.make(w, seed=0)
    threads = oracle.max_threads()
    total = x["N"] * w.H
    n = min(threads, total)
    secs = toks = 0.0
    for i in range(args.warmup + args.steps):
        units = [(i * n + j) % total for j in range(n)]
        dt, tk = oracle_step(w, x, units)
        if i >= args.warmup:
            secs, toks = secs + dt, toks + tk
    value = toks / secs
    ms = 1e3 * secs / args.steps
    base = {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {total} (sequence, head) units of {w.name} per step "
                      f"({toks / args.steps:.0f} token-equivalents), fp64 forward+backward "
                      f"on {threads} threads"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, 1),
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def time_workload(name, dev, stream, steps, warmup, max_over_ranks, barrier, seed=0):
    """Forward + backward (dr_fwd, dr_bwd reusing the forward) of a workload on device-
    resident inputs: ms per step from CUDA events on the launching stream, the path's
    roofline fraction and the per-kernel device times."""
    import torch
    from delta_rule_recurrent_gated_gb300 import binding, inputs
    w = inputs.get(name)
    x = inputs.make(w, seed=seed)
    N = x["N"]
    t = {n: (v.to(dev) if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    del x
    prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io,
                           out="bf16", grad="bf16", scale=w.scale, device=dev)
    o = torch.empty(w.B, w.T, w.H, w.dv, dtype=torch.bfloat16, device=dev)
    hT = torch.empty(N, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)

    def step():
        prob.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], o=o, hT=hT)
        prob.backward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], t["dO"], t["dhT"],
                      reuse_fwd=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    binding.trace_enable(8 * steps + 8)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    assert prob.status() == binding.DR_OK
    launches = binding.trace_read()
    binding.trace_enable(0)
    ms = max_over_ranks(e0.elapsed_time(e1) / steps)
    hbm, tflops, _ = measured_peaks()
    flops, byts = algorithmic(w, N)
    t_roof = max(flops / (tflops * 1e12), byts / (hbm * 1e9))
    kern = {}
    for nm, kms in launches:
        tot, n = kern.get(nm, (0.0, 0))
        kern[nm] = (tot + kms, n + 1)
    del prob, t, o, hT
    torch.cuda.empty_cache()
    trs = {nm: measured_traffic(nm, w) for nm in kern}
    traffic = (sum(trs[nm] * n / steps for nm, (tot, n) in kern.items())
               if kern and all(v is not None for v in trs.values()) else None)
    return {"workload": w.name, "value": w.tokens / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "steps": steps, "warmup": warmup,
            "roofline_frac": t_roof / (ms / 1e3), "t_roof_ms": t_roof * 1e3,
            "traffic_bytes_per_step": traffic, "algorithmic_bytes_per_step": byts,
            "kernels_ms": {nm: tot / n for nm, (tot, n) in kern.items()}}


def sweep_bench(dev, stream, max_over_ranks, barrier, steps=5, warmup=3):
    """The sequence-length sweep: every variant at T = 4096 .. 32768 with B T = 65536
    tokens, H = 16, d = 128; tokens/s, the path roofline fraction and the iteration-time
    ratio t(T) / t(4096)."""
    out = {}
    for variant in ("deltanet", "gdn", "kda"):
        rows = []
        for T, B in ((4096, 16), (8192, 8), (16384, 4), (32768, 2)):
            r = time_workload(f"sweep_{variant}_b{B}_t{T}_h16_d128", dev, stream, steps, warmup,
                              max_over_ranks, barrier)
            rows.append(r)
        t0 = rows[0]["ms_per_step"]
        out[variant] = [{"T": int(r["workload"].split("_t")[1].split("_")[0]),
                         "ms_per_step": r["ms_per_step"], "tokens_per_s": r["value"],
                         "roofline_frac": r["roofline_frac"],
                         "ratio_vs_t4096": r["ms_per_step"] / t0,
                         "scan_ms": r["kernels_ms"].get("tc_scan_fwd", 0.0)
                         + r["kernels_ms"].get("tc_scan_bwd", 0.0)} for r in rows]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-write", action="store_true",
                    help="skip the step that emits the write u and takes its gradient")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the recurrent-step (dr_decode) measurement")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="copy streams per direction in the end-to-end measurement")
    ap.add_argument("--no-gdn2", action="store_true",
                    help="skip the Gated DeltaNet-2 measurement")
    ap.add_argument("--no-prepare", action="store_true",
                    help="skip the step with input preparation (DR_FLAG_PREPARE_INPUTS)")
    ap.add_argument("--no-kda", action="store_true",
                    help="skip the KDA step at the headline shape")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the sequence-length sweep (all variants, T = 4096 .. 32768)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from delta_rule_recurrent_gated_gb300 import inputs
    w = inputs.get(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    from delta_rule_recurrent_gated_gb300 import binding

    from delta_rule_recurrent_gated_gb300.replicas import Replicas
    rep = Replicas.from_env()
    world, rank = rep.world, rep.rank
    torch.cuda.set_device(rep.local_rank)
    dev = torch.device("cuda", rep.local_rank)
    rep.init("nccl", dev)

    x = inputs.make(w, seed=rep.seed())
    N = x["N"]
    prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io,
                           out="bf16", grad="bf16", scale=w.scale,
                           cu_seqlens=x["cu_seqlens"], device=dev)
    t = {n: (v.to(dev) if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    o = torch.empty(w.B, w.T, w.H, w.dv, dtype=torch.bfloat16, device=dev)
    hT = torch.empty(N, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)
    grads = {
        "dq": torch.empty(w.B, w.T, w.H, w.dk, dtype=torch.bfloat16, device=dev),
        "dk": torch.empty(w.B, w.T, w.H, w.dk, dtype=torch.bfloat16, device=dev),
        "dv": torch.empty(w.B, w.T, w.H, w.dv, dtype=torch.bfloat16, device=dev),
        "dbeta": torch.empty(w.B, w.T, w.H, dtype=torch.float32, device=dev),
        "dg": None if t["g"] is None else torch.empty_like(t["g"]),
        "dh0": torch.empty(N, w.H, w.dk, w.dv, dtype=torch.float32, device=dev),
    }

    def step(src):
        prob.forward(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"], o=o, hT=hT)
        prob.backward(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"], src["dO"],
                      src["dhT"], reuse_fwd=True, out=grads)

    stream = torch.cuda.current_stream(dev)

    barrier = rep.barrier

    def max_over_ranks(v):
        return rep.max_over_ranks(v, dev)

    for _ in range(args.warmup):
        step(t)
    torch.cuda.synchronize(dev)
    assert prob.status() == binding.DR_OK

    # timed region: K steps, per-kernel events recorded on the launching stream
    binding.trace_enable(8 * args.steps + 8)
    clocks = ClockSampler(rep.local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step(t)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    st = prob.status()
    assert st == binding.DR_OK, binding.error_string(st)
    launches = binding.trace_read()
    binding.trace_enable(0)
    per = {}
    for nm, kms in launches:
        tot, n = per.get(nm, (0.0, 0))
        per[nm] = (tot + kms, n + 1)

    tokens = rep.total_units(w.tokens)
    value = tokens / (ms / 1e3)
    hbm, tflops, peak_src = measured_peaks()
    flops, byts = algorithmic(w, N)
    t_roof = max(flops / (tflops * 1e12), byts / (hbm * 1e9))
    # the roofline of the whole step: its algorithmic bytes (every kernel's inputs and
    # outputs, no intermediates) over its measured time, against the HBM copy peak; the
    # FLOP leg is below it at the measured bf16 peak
    roof = {"bound": "hbm" if byts / (hbm * 1e9) >= flops / (tflops * 1e12) else "tensor",
            "achieved": byts / (ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
            "frac": t_roof / (ms / 1e3), "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
            "bytes_per_step": byts, "flops_per_step": flops, "t_roof_ms": t_roof * 1e3,
            "tflops_achieved": flops / (ms / 1e3) / 1e12, "tflops_peak": tflops,
            "traffic": None}
    dom = None
    if per:
        name, (tot, n) = max(per.items(), key=lambda kv: kv[1][0])
        avg_s = tot / n / 1e3
        ab = kernel_algorithmic_bytes(name, w, N)
        db = kernel_bytes(name, w, N)
        tr = measured_traffic(name, w)
        dom = {"kernel": name, "avg_launch_ms": tot / n, "launches_per_step": n / args.steps,
               "algorithmic_bytes_per_launch": ab, "achieved": ab / avg_s / 1e9,
               "frac": ab / avg_s / 1e9 / hbm, "unit": "GB/s",
               "traffic": tr,
               "design_bytes_per_launch": db,
               "design_bytes_gbs": db / avg_s / 1e9, "design_bytes_frac": db / avg_s / 1e9 / hbm}
        roof["dominant_kernel"] = dom
        # DRAM traffic of the whole step, when every kernel of it has a recorded capture
        trs = [measured_traffic(k, w) for k in per]
        if all(x is not None for x in trs):
            roof["traffic"] = sum(x * per[k][1] / args.steps for x, k in zip(trs, per))
    kern = {k: {"launches": n, "ms_per_launch": tot / n, "share": tot / sum(v[0] for v in per.values()),
                "algorithmic_bytes_per_launch": kernel_algorithmic_bytes(k, w, N),
                "design_bytes_per_launch": kernel_bytes(k, w, N)}
            for k, (tot, n) in per.items()}

    # end to end through the public API from pinned host buffers, copies inside: every
    # step copies its inputs in and all its outputs and gradients out.  Two buffer sets
    # and two copy streams let step s+1's inputs and step s-1's results move while step
    # s computes (the way a training loop feeds a layer); the timed region runs from
    # before the first input copy to after the last result copy.
    e2e = None
    if not args.no_e2e:
        names = [n for n, v in x.items() if torch.is_tensor(v) and n != "cu_seqlens"]
        host_in = {n: x[n].pin_memory() for n in names}
        dev_in = [dict(t), dict(t)]
        for n in names:
            dev_in[1][n] = torch.empty_like(t[n])
        out_sets = [(o, hT, grads),
                    (torch.empty_like(o), torch.empty_like(hT),
                     {n: (None if v is None else torch.empty_like(v)) for n, v in grads.items()})]

        def flat(os_):
            oo, hh, gg = os_
            return [oo, hh] + [gg[n] for n in ("dq", "dk", "dv", "dbeta", "dg", "dh0")
                               if gg[n] is not None]

        outs_host = [[torch.empty(v.shape, dtype=v.dtype).pin_memory() for v in flat(os_)]
                     for os_ in out_sets]
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in outs_host[0])
        ncs = max(1, args.copy_streams)

        def spread(sizes):
            """Tensor indices per copy stream, balancing bytes (largest first)."""
            parts, load = [[] for _ in range(ncs)], [0] * ncs
            for i in sorted(range(len(sizes)), key=lambda i: -sizes[i]):
                j = load.index(min(load))
                parts[j].append(i)
                load[j] += sizes[i]
            return parts

        in_parts = spread([host_in[n].numel() * host_in[n].element_size() for n in names])
        out_parts = spread([v.numel() * v.element_size() for v in outs_host[0]])
        s_in = [torch.cuda.Stream(dev) for _ in range(ncs)]
        s_out = [torch.cuda.Stream(dev) for _ in range(ncs)]
        ev_in = [[torch.cuda.Event() for _ in range(ncs)] for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [[torch.cuda.Event() for _ in range(ncs)] for _ in range(2)]
        used = [False, False]

        def e2e_step(i):
            bi = i % 2
            src, (oo, hh, gg) = dev_in[bi], out_sets[bi]
            for j in range(ncs):
                with torch.cuda.stream(s_in[j]):
                    if used[bi]:
                        s_in[j].wait_event(ev_comp[bi])  # step i-2 has read this input set
                    for ti in in_parts[j]:
                        src[names[ti]].copy_(host_in[names[ti]], non_blocking=True)
                    ev_in[bi][j].record(s_in[j])
                stream.wait_event(ev_in[bi][j])
                if used[bi]:
                    stream.wait_event(ev_out[bi][j])  # step i-2's results have left this set
            prob.forward(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"], o=oo, hT=hh)
            prob.backward(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"], src["dO"],
                          src["dhT"], reuse_fwd=True, out=gg)
            ev_comp[bi].record(stream)
            dsts, srcs = outs_host[bi], flat(out_sets[bi])
            for j in range(ncs):
                with torch.cuda.stream(s_out[j]):
                    s_out[j].wait_event(ev_comp[bi])
                    for ti in out_parts[j]:
                        dsts[ti].copy_(srcs[ti], non_blocking=True)
                    ev_out[bi][j].record(s_out[j])
            used[bi] = True

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for j in range(ncs):
            s_in[j].wait_event(e0)
        for i in range(args.steps):
            e2e_step(i)
        for bi in range(2):
            for j in range(ncs):
                stream.wait_event(ev_out[bi][j])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
        e2e = {"value": tokens / (e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "h2d_gbs": h2d / (e_ms / 1e3) / 1e9, "d2h_gbs": d2h / (e_ms / 1e3) / 1e9,
               "pipelining": f"2 buffer sets; inputs in on {ncs} copy streams, results out on "
                             f"{ncs} others, tensors spread over them by size"}

    dec = None if args.no_decode else decode_bench(dev, stream, max_over_ranks, barrier)

    # the same step emitting every token's write u = beta r (dr_fwd_u) and taking a
    # gradient for it (dr_bwd_u), device-resident like the headline value
    wr = None
    if not args.no_write:
        u = torch.empty_like(o)
        dU = torch.randn(t["v"].shape, generator=torch.Generator().manual_seed(1)).to(
            t["v"].dtype).to(dev)

        def step_w(src):
            prob.forward(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"], o=o,
                         hT=hT, u=u)
            prob.backward(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"],
                          src["dO"], src["dhT"], reuse_fwd=True, out=grads, dU=dU)

        for _ in range(args.warmup):
            step_w(t)
        torch.cuda.synchronize(dev)
        barrier()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for _ in range(args.steps):
            step_w(t)
        w1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        assert prob.status() == binding.DR_OK
        w_ms = max_over_ranks(w0.elapsed_time(w1) / args.steps)
        wr = {"value": tokens / (w_ms / 1e3), "unit": "tokens/s", "ms_per_step": w_ms,
              "ms_over_plain_step": w_ms - ms,
              "extra_bytes_per_step": 2 * u.numel() * u.element_size()}

    # the same step on raw inputs (q, k unnormalised, beta logits, gate arguments) with
    # the library preparing them (DR_FLAG_PREPARE_INPUTS): its cost over the plain step,
    # and each preparation kernel against the HBM roofline
    g2 = None
    if not args.no_gdn2:
        sm = (clk or {}).get("sm_mhz") or 2070.0
        g2 = gdn2_bench(dev, stream, max_over_ranks, barrier, sm)

    pr = None
    if not args.no_prepare:
        pr = prepare_bench(args, w, rank, world, dev, stream, ms, o, hT, grads, max_over_ranks,
                           barrier)

    # KDA at the headline shape and the sequence-length sweep (same step, own workloads)
    kda = None if args.no_kda else time_workload("kda_b8_t4096_h16_d128", dev, stream, args.steps,
                                                  args.warmup, max_over_ranks, barrier, rep.seed())
    sweep = None if args.no_sweep else sweep_bench(dev, stream, max_over_ranks, barrier)

    if not rep.is_root:
        rep.shutdown()
        return
    base = None if args.no_cpu_baseline else cpu_baseline(w, x)
    in_bytes = sum(v.numel() * v.element_size() for n, v in t.items()
                   if torch.is_tensor(v) and n != "cu_seqlens")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": config_of(w, world),
        "inputs_mib_per_step": in_bytes / 2**20,
        "roofline": roof,
        "kernels": kern,
        "cpu_baseline": base,
        "e2e": e2e,
        "decode": dec,
        "emit_write": wr,
        "prepare_inputs": pr,
        "gdn2": g2,
        "kda": kda,
        "sweep": sweep,
        "gpu_launches": len(launches),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    rep.shutdown()


if __name__ == "__main__":
    main()
