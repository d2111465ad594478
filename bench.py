"""Benchmark of the context-parallel Gated DeltaNet forward on GB300.

One step = one gdn_shard_fwd call (plan, conv + SiLU with halo, chunked gated
delta rule, and for P > 1 the prefix merge and second pass) over one batch of
seeded synthetic input resident in HBM.  Prints ONE JSON line (rank 0).

The default workload is the largest bf16 d = 128 configuration, the
million-token sequence (T = 1048576, 32 heads, 64 virtual shards, h0 != 0);
--config picks another (packed_varlen, long, ragged, tiny).  The line's
"kernels" entry gives each phase of the step (plan + conv, chunk pass 1,
merge, chunk pass 2, final states), timed with CUDA events recorded between
the step's own launches; "roofline" rates the two chunk passes together.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--impl ours|reference] [--no-cpu-baseline] [--pass forward|backward]

--pass backward times the backward of the recurrence (gdn_chunk_bwd, or
gdn_shard_bwd on the config's shards) instead of the forward step.

With N > 1 (launched by torch.distributed.run) every rank runs an
independent replica of the workload on its own GPU (weak scaling, no
collective on the data path); value = total tokens of all ranks / the
slowest rank's time.  --impl reference times the fp64 CPU oracle (the only
reference implementation that exists for this path) on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN fwd tokens/s at 1 GB300 (bf16, d=128) and % of roofline; oracle tokens/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def workload(name):
    import workloads as W
    return W.CONFIGS[name]()


def algorithmic(w, spanning_tokens=0, n_affine=0):
    """Algorithmic bytes and FLOPs of the chunk passes (real tokens, C = 64);
    the UT triangular solve is ALU work and not credited.  On P > 1 shards
    the M chain adds 4 K^2 Hv FLOPs per token of a spanning shard and the
    merge 2 K^2 V Hv per affine shard carry."""
    e = 2 if w.dtype == "bf16" else 4
    T, Hk, Hv, K, V, C = w.T, w.Hk, w.Hv, w.dk, w.dv, 64
    chunk_bytes = T * (2 * Hk * K * e + Hv * V * e      # q, k, v in
                       + Hv * V * e                      # o out
                       + Hv * (4 + e))                   # g fp32, beta
    chunk_bytes += w.N * Hv * K * V * 4                  # h_final
    if w.h0_std:
        chunk_bytes += w.N * Hv * K * V * 4
    flops = T * (4 * C * K * Hk + (2 * C * K + 4 * C * V + 6 * K * V) * Hv)
    flops += spanning_tokens * 4 * K * K * Hv + n_affine * 2 * K * K * V * Hv
    conv_bytes = 2 * T * w.Cch * e
    return chunk_bytes, flops, conv_bytes


def shard_extras(recs):
    """Tokens of spanning shards and affine carries, from the device plan."""
    part_tokens, span, aff = 0, 0, 0
    for r in recs:
        part_tokens = r["local_cu"][-1]
        if r["local_num_seqs"] == 1 and not r["is_first_rank"] and r["post_num_ranks"] > 0:
            span += part_tokens
            aff += 1
    return span, aff


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        self.first = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            # its first sample means the sampler has finished starting up, so
            # its start-up does not fall inside the timed region
            self.first = self.proc.stdout.readline()
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.samples = []
        if self.proc is None:
            return
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        for line in ((self.first or "") + out).strip().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) >= 8:
                self.samples.append(parts)

    def summary(self):
        if not getattr(self, "samples", None):
            return None
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if s[4 + i].lower().startswith("active")})
        pw = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(self.samples)}


KERNEL_SOURCES = ["chunk_tc.cu", "chunk_common.cuh", "tc_util.cuh", "gdn_internal.cuh"]


def kernel_sources_sha256():
    """Hash of the dominant kernel's sources (ties stored ncu counters to them)."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "linear_attention_sequence_device_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def time_loop(fn, n, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(n):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / n  # ms


def to_dev(a, dtype, dev):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def oracle_prefix_runner(w):
    """Returns run(S): the fp64 oracle (whole path) on the first S tokens."""
    import oracle
    import workloads as W
    cu = w.cu_seqlens()

    def run(S):
        cu_s = np.concatenate([cu[cu < S], [S]]).astype(np.int64)
        x = W.as_f64(w.x(rows=(0, S)), w.dtype)
        cw = W.as_f64(w.conv_w(), w.dtype)
        g = w.g(rows=(0, S)).astype(np.float64)
        b = W.as_f64(w.beta(rows=(0, S)), w.dtype)
        h0 = w.h0()
        h0 = None if h0 is None else h0[: len(cu_s) - 1].astype(np.float64)
        t0 = time.perf_counter()
        oracle.path_forward(x, cw, None, g, b, h0, cu_s, w.Hk, w.Hv, w.dk, w.dv, w.scale)
        return time.perf_counter() - t0
    return run


def calibrate(run, T, budget_s):
    S = 256
    dt = run(S)
    while dt < budget_s / 2.5 and S * 2 <= T:
        S *= 2
        dt = run(S)
    return S, dt


def cpu_baseline(w, budget_s=20.0):
    """The fp64 oracle (whole path) on a bounded prefix of the workload."""
    import oracle
    run = oracle_prefix_runner(w)
    S, dt = calibrate(run, w.T, budget_s)
    threads = oracle.max_threads()
    return {"value": S / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"first {S} tokens of the {w.name} workload (all {w.Hv} value heads, "
                      f"conv + L2 norm + token recurrence in fp64), {dt:.2f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = workload(args.config)
    import oracle
    oracle.build()
    import workloads as W
    W.build_synth()
    run = oracle_prefix_runner(w)
    S, _ = calibrate(run, w.T, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        run(S)
    per = [run(S) for _ in range(args.steps)]
    dt = float(np.median(per))
    v = S / dt
    cb = {"value": v, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
          "sample": f"first {S} tokens of the {w.name} workload per step (all {w.Hv} value heads, "
                    f"conv + L2 norm + token recurrence in fp64), median {dt:.2f} s"}
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
            "config": config_dict(w), "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(w):
    return {"workload": w.name, "T": w.T, "num_seqs": w.N, "Hk": w.Hk, "Hv": w.Hv, "dk": w.dk,
            "dv": w.dv, "n_shards": w.n_shards, "conv_k": w.conv_k, "dtype": w.dtype,
            "l2": "inputs larger than L2 (raw qkv %.0f MiB)" % (w.T * w.Cch * (2 if w.dtype == "bf16" else 4) / 2**20)}


def run_backward(args, rank, world, local_rank):
    """--pass backward: the backward of the recurrence (gdn_chunk_bwd, or
    gdn_shard_bwd on the config's P shards) on the config's q, k, v, gates,
    h0 and seeded output gradients; one JSON line, tokens/s of the backward
    step with its inputs resident in HBM."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import linear_attention_sequence_device_gb300 as g
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workload(args.config)
    if rank:
        w = w.replace(seed=w.seed + 1000 * rank)
    P = w.n_shards
    q = to_dev(w.q(), w.dtype, dev).view(w.T, w.Hk, w.dk)
    k = to_dev(w.k(), w.dtype, dev).view(w.T, w.Hk, w.dk)
    v = to_dev(w.v(), w.dtype, dev).view(w.T, w.Hv, w.dv)
    gg, bb = to_dev(w.g(), "f32", dev), to_dev(w.beta(), w.dtype, dev)
    h0_h = w.h0()
    h0 = None if h0_h is None else to_dev(h0_h, "f32", dev)
    cu = torch.from_numpy(w.cu_seqlens()).to(dev)
    gen = torch.Generator(device=dev).manual_seed(w.seed + 7)
    do = torch.randn((w.T, w.Hv, w.dv), generator=gen, device=dev).to(v.dtype)
    dh = torch.randn((w.N, w.Hv, w.dk, w.dv), generator=gen, device=dev)
    if P > 1:
        wsz = g.load().gdn_shard_bwd_workspace_size(w.T, w.N, P, w.Hk, w.Hv, w.dk, w.dv)
    else:
        wsz = g.chunk_bwd_workspace_size(w.T, w.N, w.Hk, w.Hv, w.dk, w.dv)
    ws = torch.empty(wsz, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        g.gdn_chunk_bwd(q, k, v, gg, bb, cu, do, h0=h0, dh_final=dh, workspace=ws,
                        n_shards=P if P > 1 else None)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(local_rank) as clk:
        ms = time_loop(step, args.steps, stream)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    e = 2 if w.dtype == "bf16" else 4
    # algorithmic bytes: q, k, v, dout, g, beta read; fp32 dq, dk, dv, dg, dbeta written;
    # h0, dh_final read and dh0 written per sequence
    byts = w.T * (2 * w.Hk * w.dk * e + 2 * w.Hv * w.dv * e + w.Hv * (4 + e)
                  + 4 * (2 * w.Hk * w.dk + w.Hv * w.dv + 2 * w.Hv)) + 3 * w.N * w.Hv * w.dk * w.dv * 4
    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    ach = byts / (ms * 1e-3) / 1e9
    line = {"metric": "GDN backward tokens/s at 1 GB300", "value": world * w.T / (ms * 1e-3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded counter-based generator; no dataset)", "config": config_dict(w),
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                         "traffic": None, "kernel": "bwd_job_kernel", "peak_source": src,
                         "algorithmic_bytes": byts},
            "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import linear_attention_sequence_device_gb300 as g

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workload(args.config)
    P = w.n_shards
    # inputs: rank-specific seed so replicas are independent problems
    if rank:
        w = w.replace(seed=w.seed + 1000 * rank)
    x_h, cw_h, g_h, b_h = w.x(), w.conv_w(), w.g(), w.beta()
    h0_h = w.h0()
    x, cw = to_dev(x_h, w.dtype, dev), to_dev(cw_h, w.dtype, dev)
    gg, bb = to_dev(g_h, "f32", dev), to_dev(b_h, w.dtype, dev)
    h0 = None if h0_h is None else to_dev(h0_h, "f32", dev)
    cu = torch.from_numpy(w.cu_seqlens()).to(dev)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ws = torch.empty(g.shard_fwd_workspace_size(w.T, w.N, P, w.Hk, w.Hv, w.dk, w.dv, tdt),
                     dtype=torch.uint8, device=dev)
    o = torch.empty((w.T, w.Hv, w.dv), dtype=tdt, device=dev)
    hf_d = torch.empty((w.N, w.Hv, w.dk, w.dv), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        g.gdn_shard_fwd(x, cw, None, gg, bb, cu, w.Hk, w.Hv, w.dk, w.dv, P, h0=h0, workspace=ws,
                        out=o, h_final=hf_d)

    # plan, conv, pass 1, empty-seq final (+ merge, pass 2); the tensor-core
    # chunk path (bf16, d = 128) sorts each pass's work queue first (order
    # kernel) and, on P > 1 shards, runs the summaries' M chains apart (one
    # more launch in pass 1)
    tc_path = w.dtype == "bf16" and w.dk == 128 and w.dv == 128
    passes = 2 if P > 1 else 1
    launches_per_step = (3 + passes + (1 if P > 1 else 0) + (passes if tc_path else 0)
                         + (1 if tc_path and P > 1 else 0))

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    g.binding.device_timeouts(reset=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        ms = time_loop(step, args.steps, stream)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    value = world * w.T / (ms * 1e-3)

    # ---- end to end through the public API with host buffers ----
    # Every step copies all of its inputs up from pinned host memory, runs the
    # public entry point, and copies its outputs back down.  Consecutive steps
    # overlap the way a serving loop would: step k+1's inputs go up on one copy
    # stream and step k-1's outputs come down on another while step k
    # computes (the two copy directions run concurrently).  Device buffers are
    # double-buffered and events order every reuse.
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    xh = pin(x_h.view(np.int16) if w.dtype == "bf16" else x_h)
    gh, bh = pin(g_h), pin(b_h.view(np.int16) if w.dtype == "bf16" else b_h)
    cuh = pin(w.cu_seqlens())
    oh = torch.empty((w.T, w.Hv, w.dv), dtype=tdt).pin_memory()
    hfh = torch.empty((w.N, w.Hv, w.dk, w.dv), dtype=torch.float32).pin_memory()
    ibuf = torch.int16 if w.dtype == "bf16" else tdt
    bufs = [dict(x=torch.empty_like(x), g=torch.empty_like(gg), b=torch.empty_like(bb), cu=torch.empty_like(cu),
                 o=torch.empty_like(o), hf=torch.empty_like(hf_d)) for _ in range(2)]
    NUP = 1  # input copy streams (more did not raise the host link's rate on GB300)
    s_ups = [torch.cuda.Stream() for _ in range(NUP)]
    s_up, s_down = s_ups[0], torch.cuda.Stream()
    rows = [(i * w.T) // NUP for i in range(NUP + 1)]
    ev_in = [[torch.cuda.Event() for _ in range(NUP)] for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(k):
        bi = k & 1
        B = bufs[bi]
        for i, su in enumerate(s_ups):
            with torch.cuda.stream(su):
                if used[bi]:
                    su.wait_event(ev_comp[bi])  # step k-2 is done reading these inputs
                B["x"].view(ibuf)[rows[i]:rows[i + 1]].copy_(xh[rows[i]:rows[i + 1]], non_blocking=True)
                if i == 0:
                    B["g"].copy_(gh, non_blocking=True)
                    B["b"].view(ibuf).copy_(bh, non_blocking=True)
                    B["cu"].copy_(cuh, non_blocking=True)
                ev_in[bi][i].record(su)
        for i in range(NUP):
            stream.wait_event(ev_in[bi][i])
        if used[bi]:
            stream.wait_event(ev_out[bi])  # step k-2's outputs have been copied down
        g.gdn_shard_fwd(B["x"], cw, None, B["g"], B["b"], B["cu"], w.Hk, w.Hv, w.dk, w.dv, P, h0=h0,
                        workspace=ws, out=B["o"], h_final=B["hf"])
        ev_comp[bi].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev_comp[bi])
            oh.copy_(B["o"], non_blocking=True)
            hfh.copy_(B["hf"], non_blocking=True)
            ev_out[bi].record(s_down)
        used[bi] = True

    for k in range(2):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 20))
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for su in s_ups:
        su.wait_event(t_start)
    for k in range(2, 2 + e2e_steps):
        e2e_step(k)
    stream.wait_stream(s_down)
    for su in s_ups:
        stream.wait_stream(su)
    t_end.record(stream)
    t_end.synchronize()
    e2e_ms = t_start.elapsed_time(t_end) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    h2d = xh.numel() * xh.element_size() + gh.numel() * 4 + bh.numel() * bh.element_size() + cuh.numel() * 4
    d2h = oh.numel() * oh.element_size() + hfh.numel() * 4
    # the host link's own rate: one plain pinned-to-device copy of a slice of
    # the input, so that the end-to-end figure can be read against it
    link_n = min(xh.numel(), (1 << 30) // xh.element_size())
    link_dst = torch.empty(link_n, dtype=xh.dtype, device=dev)
    link_src = xh.view(-1)[:link_n]
    for _ in range(2):
        link_dst.copy_(link_src, non_blocking=True)
    torch.cuda.synchronize()
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            link_dst.copy_(link_src, non_blocking=True)
    l1.record(stream)
    l1.synchronize()
    link_gbps = 3 * link_n * xh.element_size() / (l0.elapsed_time(l1) * 1e6)
    del link_dst
    e2e_gbps = (h2d + d2h) / (e2e_ms * 1e6)

    # ---- per-phase times of the same step (events between its kernels) ----
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize()
    g.binding.debug_set_phase_events(evs)
    phases = []
    try:
        for _ in range(max(5, min(args.steps, 30))):
            step()
            evs[-1].synchronize()
            phases.append([evs[i].elapsed_time(evs[i + 1]) for i in range(5)])
    finally:
        g.binding.debug_set_phase_events(None)
    ph = np.median(np.array(phases), axis=0)
    conv_ms, pass1_ms, combine_ms, pass2_ms, final_ms = (float(x) for x in ph)
    chunk_ms = pass1_ms + pass2_ms
    timeouts = g.binding.device_timeouts(reset=True)
    if timeouts:
        raise RuntimeError(f"{timeouts} bounded device waits expired during the bench: outputs incomplete")

    _, _, plan = g.gdn_shard_fwd(x, cw, None, gg, bb, cu, w.Hk, w.Hv, w.dk, w.dv, P, h0=h0, workspace=ws,
                                 out=o, h_final=hf_d, want_plan=True)
    _, recs = g.decode_plan(plan, w.N, P)
    span_tokens, n_affine = shard_extras(recs)

    peaks, peak_src = load_peaks()
    chunk_bytes, flops, conv_bytes = algorithmic(w, span_tokens, n_affine)
    hbm = float(peaks["hbm_gbs"])
    tfl = float(peaks["bf16_tflops_sustained" if chunk_ms > 50 else "bf16_tflops"])
    t_bytes = chunk_bytes / (hbm * 1e9)
    t_flops = flops / (tfl * 1e12)
    traffic = None
    tp = os.path.join(ROOT, "profiles", f"chunk_traffic_{w.name}.json")
    if os.path.exists(tp):
        rec = json.load(open(tp))
        # counters are only valid for the kernel sources they were taken on
        if rec.get("kernel_sources_sha256") == kernel_sources_sha256():
            traffic = rec.get("bytes_per_step")
    if t_bytes >= t_flops:
        ach = chunk_bytes / (chunk_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": traffic}
    else:
        ach = flops / (chunk_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": tfl, "unit": "TFLOP/s",
                "frac": ach / tfl, "traffic": traffic}
    roof.update({"kernel": ("chunk_tc_kernel" if (w.dtype == "bf16" and w.dk == 128 and w.dv == 128)
                            else "chunk_bf16_kernel" if w.dtype == "bf16" else "chunk_f32_kernel"),
                 "kernel_ms": chunk_ms, "launches_per_step": (3 if tc_path else 2) if P > 1 else 1,
                 # the launches the chunk passes' time covers (the M chains of the
                 # summaries run in their own kernel on the tensor-core path)
                 "pass_kernels": (["chunk_tc_kernel", "mchain_kernel"] if tc_path and P > 1 else None),
                 "peak_source": peak_src + (" (sustained)" if chunk_ms > 50 else " (burst)"),
                 "algorithmic_bytes": chunk_bytes, "algorithmic_flops": flops,
                 "tensor_frac": (flops / (chunk_ms * 1e-3) / 1e12) / tfl,
                 "roofline_ms": max(t_bytes, t_flops) * 1e3,
                 "step_frac": max(t_bytes, t_flops) * 1e3 / ms})

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded counter-based generator; no dataset)",
            "config": config_dict(w),
            "e2e": {"value": world * w.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "host_GBps": e2e_gbps, "host_link_GBps": link_gbps},
            "gpu_launches": launches_per_step * args.steps,
            "roofline": roof,
            "kernels": {"plan_conv_ms": conv_ms, "pass1_ms": pass1_ms, "combine_ms": combine_ms,
                        "pass2_ms": pass2_ms, "final_ms": final_ms, "chunk_ms": chunk_ms,
                        "conv_GBps": conv_bytes / (conv_ms * 1e-3) / 1e9,
                        "conv_frac_hbm": conv_bytes / (conv_ms * 1e-3) / 1e9 / hbm},
            "device_timeouts": timeouts,
            "clocks": clk.summary()}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(workload(args.config))
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="million")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward"])
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        (run_backward if args.which == "backward" else run_ours)(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
