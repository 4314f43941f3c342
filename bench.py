"""Benchmark: exact tiled attention on GB300, one JSON line on stdout.

A step is one pass of the whole hot path over one batch: fa_fwd then fa_bwd
(schedule, TMA loads, S = QK^T, masking, online softmax, PV, epilogue; then
D, recompute of S and P, dV, dP, dS, dK, dQ and the dQ conversion) on the
training workload: B=8, H=16, N=2048, d=128, bf16, causal, synthetic
iid N(0,1) inputs (seeded).  The metric is attention TFLOP/s counted the
pages' way: 4*N^2*d per head for the forward, 14*N^2*d for forward+backward
(the backward's five matmuls), halved under the causal mask.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`value` is device-timed (inputs resident in HBM; every input tensor is
larger than L2, so no flush is needed between steps); `e2e` times the same
step through the public API with pinned host buffers: every step copies its
inputs in and its results out inside the timed region, pipelined so that one
step's copies overlap its neighbours' kernels;
`fwd` holds forward-only TFLOP/s of the Llama-3.1-8B-shaped and long-context
workloads.  `--impl reference` times the fp64 CPU oracle (the only other
implementation of this computation) on a bounded sample of the same
workload on the host cores.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd and fwd+bwd at 1 GB300; % of dense BF16 tensor peak"
WORKLOAD = "train_fwd_bwd"
FALLBACK_BF16_TFLOPS = 1900.0


def attn_flops(B, H, N, d, causal, passes):
    per_head = (4 if passes == "fwd" else 14) * N * N * d
    if causal:
        per_head /= 2
    return per_head * B * H


def window_pairs(N, w):
    """Visible (query, key) pairs of one head under the causal sliding window
    of w keys: sum over rows r of min(r + 1, w)."""
    if w >= N:
        return N * (N + 1) // 2
    return w * (w + 1) // 2 + (N - w) * w


def window_flops(B, H, N, d, w, passes):
    """The metric's convention applied to the visible pairs: 4*d per pair for
    the forward, 14*d for forward+backward."""
    return (4 if passes == "fwd" else 14) * d * window_pairs(N, w) * B * H


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", 0) or 0), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# kernel key (as in profiles/traffic.txt) -> the source file that defines it
KERNEL_SOURCES = {"bwd_kernel": "fa_bwd_tc.cu", "fwd_kernel": "fa_fwd_tc.cu",
                  "fwd256_kernel": "fa_fwd256_tc.cu", "bwd256_kernel": "fa_bwd256_tc.cu"}


def kernel_digest(kernel_key):
    """sha256 (first 16 hex digits) of the kernel's .cu file and every shared
    header of csrc/: the sources a capture of that kernel depends on."""
    import hashlib
    src = os.path.join(ROOT, "exact_tiled_attention_sm_gb300", "csrc")
    cu = next(v for k, v in KERNEL_SOURCES.items() if kernel_key.startswith(k))
    files = [cu] + sorted(f for f in os.listdir(src) if f.endswith((".cuh", ".h")))
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(src, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_key):
    """Per-launch DRAM bytes of a kernel from a committed ncu summary, if the
    summary was taken on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    digest = kernel_digest(kernel_key)
    try:
        for line in open(path):
            parts = line.split()
            if len(parts) >= 3 and parts[0] == kernel_key and parts[2] == digest:
                return float(parts[1])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed regions run."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sms, maxs, reasons, n = [], [], set(), 0
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx, pw = float(parts[0]), float(parts[1]), float(parts[2])
            except ValueError:
                continue
            n += 1
            maxs.append(mx)
            if pw > 250:  # under load
                sms.append(sm)
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(name)
        sms.sort()
        med = sms[len(sms) // 2] if sms else None
        return {"sm_mhz": med, "sm_max_mhz": max(maxs) if maxs else None,
                "reasons": sorted(reasons), "samples": n, "samples_under_load": len(sms)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world, device="cuda"):
    """Device work done and every rank here (device "cpu": host-only ranks,
    as in the gloo tests of this logic)."""
    import torch
    if device == "cuda":
        torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """The largest of the ranks' values of x (a time: the job is as slow as
    its slowest replica)."""
    import torch
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def bench_config(w, world):
    """The `config` of the bench line, identical in both arms."""
    return {"workload": "train_fwd_bwd: B=8 H=16 N=2048 d=128 bf16 causal, fa_fwd + fa_bwd",
            "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": True, "scale": w.scale,
            "parallelism": f"replicas x{world} (heads independent; no collective)",
            "l2": "no flush: inputs larger than L2 (Q, K, V, dO, O are 64 MiB each; 320 MiB read per step)"}


def job_tflops(world, flops_per_rank, ms):
    """Whole-job throughput: every rank processes its own replica of the
    workload (weak scaling), the job takes the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------ profile
def run_profile(args):
    """Only the launches of one workload (for ncu): W warm-up steps then K
    steps, nothing else on the GPU.  `train_fwd_bwd` runs fa_fwd + fa_bwd
    (4 launches a step); a forward workload runs fa_fwd (1 launch a step).
    --window and --dropout select those variants, --fp8 the 8-bit forward
    (forward workloads only)."""
    import torch
    import exact_tiled_attention_sm_gb300 as fa
    from exact_tiled_attention_sm_gb300 import inputs
    torch.cuda.set_device(0)
    w = inputs.WORKLOADS[args.workload]
    x = inputs.workload_inputs(w)
    q, k, v = (x[n].cuda() for n in ("Q", "K", "V"))
    causal = args.causal if w.passes == "fwd" else True
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
    if w.passes == "fwd+bwd":
        do = x["dO"].cuda()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = fa.workspace(w.B, w.H, w.N, w.d)
    opt = {"window": args.window, "dropout_p": args.dropout, "seed": 1234}
    if args.fp8:
        x8, fac = inputs.e4m3_inputs(w.B, w.H, w.N, w.d, w.seed)
        q8, k8, v8 = (x8[n].cuda() for n in ("Q", "K", "V"))
        dsc = (fac["Q"], fac["K"], fac["V"])
        for _ in range(args.warmup + args.steps):
            fa.fwd_fp8(q8, k8, v8, w.scale, dsc, causal, out=o, lse=lse,
                       window=args.window)
    for _ in range(0 if args.fp8 else args.warmup + args.steps):
        fa.fwd(q, k, v, w.scale, causal, out=o, lse=lse, **opt)
        if w.passes == "fwd+bwd":
            fa.bwd(q, k, v, o, do, lse, w.scale, causal, dq=dq, dk=dk, dv=dv, ws=ws,
                   **opt)
    torch.cuda.synchronize()
    st = fa.last_device_status()
    if st != fa.FA_OK:
        raise SystemExit(f"device status: {fa.status_string(st)}")
    return {"profile": args.workload, "causal": causal, "steps": args.steps,
            "warmup": args.warmup, "window": args.window, "dropout": args.dropout,
            "fp8": bool(args.fp8)}


# ------------------------------------------------------------------ balance
BALANCE_CASES = (("llama3_8b_fwd", True, "fwd"), ("llama3_8b_fwd", False, "fwd"),
                 ("gpt2_medium_fwd", True, "fwd"), ("gpt2_medium_fwd", False, "fwd"),
                 ("long_ctx_32k", True, "fwd"), ("train_fwd_bwd", True, "fwd"),
                 ("train_fwd_bwd", True, "bwd"), ("d256_train", True, "bwd"))


def run_balance(args):
    """How evenly the schedulers spread the work: the trace build of the
    library (libfa_trace.so, built on demand) records each CTA's start and
    end; for every case, three traced launches after three warm-up launches,
    summarised per launch (exact_tiled_attention_sm_gb300.trace.summarize).
    Inputs are drawn on the device (no parity check here)."""
    import torch
    import exact_tiled_attention_sm_gb300 as fa
    from exact_tiled_attention_sm_gb300 import _build, inputs, trace
    fa.use_library(_build.build(trace=True))
    L = fa.lib()
    torch.cuda.set_device(0)
    out = {}
    for name, causal, which in BALANCE_CASES:
        w = inputs.WORKLOADS[name]
        x = inputs.seeded_inputs_cuda(w.B, w.H, w.N, w.d, w.seed, with_dO=(which == "bwd"))
        q, k, v = x["Q"], x["K"], x["V"]
        o, lse = fa.fwd(q, k, v, w.scale, causal)
        if which == "bwd":
            do = x["dO"]
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            ws = fa.workspace(w.B, w.H, w.N, w.d)

        def call():
            if which == "bwd":
                fa.bwd(q, k, v, o, do, lse, w.scale, causal, dq=dq, dk=dk, dv=dv, ws=ws)
            else:
                fa.fwd(q, k, v, w.scale, causal, out=o, lse=lse)

        runs = []
        for rep in range(6):
            call()
            # the kernel that ran: d = 256 and (backward) d = 64 have their own
            marks = trace.read(L, which + ("256" if w.d == 256 else
                                           "64" if (w.d == 64 and which == "bwd") else ""))
            if rep >= 3:
                runs.append(trace.summarize(marks))
        st = fa.last_device_status()
        if st != fa.FA_OK:
            raise SystemExit(f"device status: {fa.status_string(st)}")
        out[f"{name}{'_causal' if causal else ''}_{which}"] = {
            "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal, "launches": runs}
        del x, q, k, v, o, lse
    return {"balance": out, "note": "per-CTA global-timer marks from libfa_trace.so "
            "(FA_CTA_TRACE build); times in microseconds relative to the launch's first CTA start"}


# --------------------------------------------------------------------- ours
def run_ours(args):
    import torch
    import exact_tiled_attention_sm_gb300 as fa
    from exact_tiled_attention_sm_gb300 import inputs

    world, rank, local = dist_setup()
    w = inputs.WORKLOADS[WORKLOAD]
    B, H, N, d, sc = w.B, w.H, w.N, w.d, w.scale
    causal = True
    stream = torch.cuda.current_stream()
    host = inputs.workload_inputs(w)  # every rank: its own replica of the batch
    q, k, v, do = (host[n].cuda() for n in ("Q", "K", "V", "dO"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = fa.workspace(B, H, N, d)

    def step():
        fa.fwd(q, k, v, sc, causal, out=o, lse=lse)
        fa.bwd(q, k, v, o, do, lse, sc, causal, dq=dq, dk=dk, dv=dv, ws=ws)

    sampler = ClockSampler(local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = fa.last_device_status()
    if st != fa.FA_OK:
        raise SystemExit(f"device status after warm-up: {fa.status_string(st)}")

    sampler.start()
    time.sleep(0.3)
    # --- device-timed region: K steps, per-call events on the launch stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        fa.fwd(q, k, v, sc, causal, out=o, lse=lse)
        ev[i][1].record(stream)
        fa.bwd(q, k, v, o, do, lse, sc, causal, dq=dq, dk=dk, dv=dv, ws=ws)
        ev[i][2].record(stream)
    t1.record(stream)
    barrier(world)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world)
    fwd_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / args.steps
    bwd_ms = sum(b.elapsed_time(c) for _, b, c in ev) / args.steps
    launches = args.steps * (1 + 3)  # fwd kernel; bwd pre, main, convert

    # --- e2e: pinned host buffers -> device -> fwd + bwd -> host, per step.
    # Every step copies its own inputs in and its own results out inside the
    # timed region; the steps are pipelined over two device buffer sets and
    # three streams (copy in, compute, copy out), so the copies of one step
    # overlap the kernels of its neighbours.
    pin = {n: host[n].pin_memory() for n in ("Q", "K", "V", "dO")}
    outs = {n: torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=True)
            for n in ("O", "dQ", "dK", "dV")}
    lse_h = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in outs.values()) + lse_h.numel() * 4
    bufs = [dict(Q=q, K=k, V=v, dO=do, O=o, LSE=lse, dQ=dq, dK=dk, dV=dv)]
    bufs.append({n: torch.empty_like(t) for n, t in bufs[0].items()})
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(kstep):
        b = kstep & 1
        t = bufs[b]
        with torch.cuda.stream(s_in):
            if kstep >= 2:
                s_in.wait_event(ev_cmp[b])  # step k-2 is done reading set b
            for n in ("Q", "K", "V", "dO"):
                t[n].copy_(pin[n], non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if kstep >= 2:
            stream.wait_event(ev_out[b])  # step k-2's results have left set b
        fa.fwd(t["Q"], t["K"], t["V"], sc, causal, out=t["O"], lse=t["LSE"])
        fa.bwd(t["Q"], t["K"], t["V"], t["O"], t["dO"], t["LSE"], sc, causal,
               dq=t["dQ"], dk=t["dK"], dv=t["dV"], ws=ws)  # one compute stream: one workspace
        ev_cmp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            for n in ("O", "dQ", "dK", "dV"):
                outs[n].copy_(t[n], non_blocking=True)
            lse_h.copy_(t["LSE"], non_blocking=True)
            ev_out[b].record(s_out)

    def e2e_run(nsteps, k0):
        for kk in range(nsteps):
            e2e_step(k0 + kk)
        # the timed region ends when the last results are on the host
        stream.wait_event(ev_out[(k0 + nsteps - 1) & 1])
        stream.wait_event(ev_out[(k0 + nsteps - 2) & 1])

    # at least 20 timed steps: the pipeline's fill (the first step's copy-in)
    # and drain (the last step's copy-out) are not overlapped, and over a
    # handful of steps they dominate the per-step figure
    e2e_steps = max(20, args.steps)
    e2e_run(2, 0)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    e2e_run(e2e_steps, 0)
    e1.record(stream)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps

    # --- forward-only workloads (the forward metric), each timed on its own
    fwd_results = {}
    for name, causal_list in (("llama3_8b_fwd", (False, True)), ("long_ctx_32k", (True,)),
                              ("gpt2_medium_fwd", (False, True))):
        wf = inputs.WORKLOADS[name]
        xf = inputs.workload_inputs(wf, with_dO=False)
        qf, kf, vf = (xf[n].cuda() for n in ("Q", "K", "V"))
        of = torch.empty_like(qf)
        lf = torch.empty((wf.B, wf.H, wf.N), dtype=torch.float32, device="cuda")
        # inputs smaller than L2 (the GPT-2-shaped workload, 48 MiB): each
        # timed call is preceded by a 256 MiB write that evicts them, outside
        # its own pair of events
        small = (3 * qf.numel() * qf.element_size()) < (129 << 20)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if small else None
        for c in causal_list:
            reps = max(5, args.steps // 2)
            for _ in range(3):
                fa.fwd(qf, kf, vf, wf.scale, c, out=of, lse=lf)
            barrier(world)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fa.fwd(qf, kf, vf, wf.scale, c, out=of, lse=lf)
            b.record(stream)
            barrier(world)
            ms = max_over_ranks(a.elapsed_time(b), world) / reps
            fl = attn_flops(wf.B, wf.H, wf.N, wf.d, c, "fwd")
            key = f"{name}{'_causal' if c else ''}"
            launches += reps
            if small:
                warm_ms = ms
                evs = [(torch.cuda.Event(enable_timing=True),
                        torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
                barrier(world)
                for i in range(reps):
                    flush.fill_(i & 0xFF)
                    evs[i][0].record(stream)
                    fa.fwd(qf, kf, vf, wf.scale, c, out=of, lse=lf)
                    evs[i][1].record(stream)
                barrier(world)
                ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in evs), world) / reps
                launches += reps
            fwd_results[key] = {"tflops": round(job_tflops(world, fl, ms), 1),
                                "ms": round(ms, 4), "launches": reps}
            if small:
                fwd_results[key]["l2"] = ("flushed: a 256 MiB write before each call, "
                                          "outside its timed events")
                fwd_results[key]["tflops_warm_l2"] = round(job_tflops(world, fl, warm_ms), 1)
        del qf, kf, vf, of, lf, flush

    def time_variant(name, passes, causal_v, win=0, drop=0.0, seed=0):
        """Device time of one fa_fwd (+ fa_bwd) call pair of a mask or dropout
        variant on workload `name`; returns (ms per call pair, launches timed)."""
        wf = inputs.WORKLOADS[name]
        xf = inputs.workload_inputs(wf, with_dO=(passes != "fwd"))
        qf, kf, vf = (xf[n].cuda() for n in ("Q", "K", "V"))
        of = torch.empty_like(qf)
        lf = torch.empty((wf.B, wf.H, wf.N), dtype=torch.float32, device="cuda")
        if passes != "fwd":
            dof = xf["dO"].cuda()
            dqf, dkf, dvf = torch.empty_like(qf), torch.empty_like(qf), torch.empty_like(qf)
            wsf = fa.workspace(wf.B, wf.H, wf.N, wf.d)

        def vstep():
            fa.fwd(qf, kf, vf, wf.scale, causal_v, out=of, lse=lf, window=win,
                   dropout_p=drop, seed=seed)
            if passes != "fwd":
                fa.bwd(qf, kf, vf, of, dof, lf, wf.scale, causal_v, dq=dqf, dk=dkf,
                       dv=dvf, ws=wsf, window=win, dropout_p=drop, seed=seed)

        reps = max(5, args.steps // 4)
        for _ in range(3):
            vstep()
        barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            vstep()
        b.record(stream)
        barrier(world)
        ms = max_over_ranks(a.elapsed_time(b), world) / reps
        return ms, reps * (1 if passes == "fwd" else 4)

    # --- causal sliding window ("LLM Architecture Refresh [3]", section 5):
    # a long-context forward with a 4096-key window, and the training step's
    # shape with a 512-key window (fwd + bwd); FLOPs over the visible pairs
    window_results = {}
    for name, win, passes in (("long_ctx_32k", 4096, "fwd"), (WORKLOAD, 512, "fwd+bwd")):
        wf = inputs.WORKLOADS[name]
        ms, nl = time_variant(name, passes, True, win=win)
        fl = window_flops(wf.B, wf.H, wf.N, wf.d, win, passes)
        window_results[f"{name}_w{win}_{passes.replace('+', '_')}"] = {
            "tflops": round(job_tflops(world, fl, ms), 1), "ms": round(ms, 4),
            "window": win, "launches": nl}
        launches += nl

    # --- attention dropout (p = 0.1; the backward regenerates the keep mask
    # from the seed): the 4096-token forward without a mask and the training
    # step; FLOPs those of the same computation without dropout
    dropout_results = {}
    for name, causal_v, passes in (("llama3_8b_fwd", False, "fwd"), (WORKLOAD, True, "fwd+bwd")):
        wf = inputs.WORKLOADS[name]
        ms, nl = time_variant(name, passes, causal_v, drop=0.1, seed=1234)
        fl = attn_flops(wf.B, wf.H, wf.N, wf.d, causal_v, passes)
        dropout_results[f"{name}{'_causal' if causal_v else ''}_p0.1_{passes.replace('+', '_')}"] = {
            "tflops": round(job_tflops(world, fl, ms), 1), "ms": round(ms, 4),
            "dropout_p": 0.1, "launches": nl}
        launches += nl
    # --- the 8-bit forward (E4M3 inputs with per-tensor factors): the 4096-
    # token shape both ways and the 32K causal context; FLOPs as the bf16
    # forward's
    fp8_results = {}
    for name, causal_list in (("llama3_8b_fwd", (False, True)), ("long_ctx_32k", (True,))):
        wf = inputs.WORKLOADS[name]
        x8, fac = inputs.e4m3_inputs(wf.B, wf.H, wf.N, wf.d, wf.seed)
        q8, k8, v8 = (x8[n].cuda() for n in ("Q", "K", "V"))
        of = torch.empty((wf.B, wf.H, wf.N, wf.d), dtype=torch.bfloat16, device="cuda")
        lf = torch.empty((wf.B, wf.H, wf.N), dtype=torch.float32, device="cuda")
        dsc = (fac["Q"], fac["K"], fac["V"])
        for c in causal_list:
            reps = max(5, args.steps // 2)
            for _ in range(3):
                fa.fwd_fp8(q8, k8, v8, wf.scale, dsc, c, out=of, lse=lf)
            barrier(world)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fa.fwd_fp8(q8, k8, v8, wf.scale, dsc, c, out=of, lse=lf)
            b.record(stream)
            barrier(world)
            ms = max_over_ranks(a.elapsed_time(b), world) / reps
            fl = attn_flops(wf.B, wf.H, wf.N, wf.d, c, "fwd")
            fp8_results[f"{name}{'_causal' if c else ''}_e4m3"] = {
                "tflops": round(job_tflops(world, fl, ms), 1), "ms": round(ms, 4),
                "launches": reps}
            launches += reps
        del q8, k8, v8, of, lf
    # --- head dimension 256: the tensor-core forward (one query block per
    # item) both ways, and the training step at d = 256 (tensor-core backward:
    # one pass per half of d over 64-query blocks)
    d256_results = {}
    for name, causal_v, passes in (("d256_fwd", False, "fwd"), ("d256_fwd", True, "fwd"),
                                   ("d256_train", True, "fwd+bwd")):
        wf = inputs.WORKLOADS[name]
        ms, nl = time_variant(name, passes, causal_v)
        fl = attn_flops(wf.B, wf.H, wf.N, wf.d, causal_v, passes)
        d256_results[f"{name}{'_causal' if causal_v else ''}_{passes.replace('+', '_')}"] = {
            "tflops": round(job_tflops(world, fl, ms), 1), "ms": round(ms, 4),
            "launches": nl}
        launches += nl
    clocks = sampler.stop()
    st = fa.last_device_status()
    if st != fa.FA_OK:
        raise SystemExit(f"device status after timing: {fa.status_string(st)}")

    if rank != 0:
        return None
    peak, peak_sustained, peak_src = measured_peaks()
    step_flops = attn_flops(B, H, N, d, causal, "fwd+bwd")
    ms_per_step = elapsed_ms / args.steps
    value = job_tflops(world, step_flops, ms_per_step)
    bwd_flops = step_flops - attn_flops(B, H, N, d, causal, "fwd")
    bwd_tflops = bwd_flops / (bwd_ms * 1e-3) / 1e12
    fwd_tflops = attn_flops(B, H, N, d, causal, "fwd") / (fwd_ms * 1e-3) / 1e12
    for r in (list(fwd_results.values()) + list(window_results.values())
              + list(dropout_results.values()) + list(d256_results.values())):
        r["frac_of_peak"] = round(r["tflops"] / world / peak, 4)
    for r in fp8_results.values():  # against the 8-bit peak: 2x the bf16 one
        r["frac_of_fp8_peak"] = round(r["tflops"] / world / (2 * peak), 4)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded iid N(0,1) bf16 tensors of the workload's shape",
        "config": bench_config(w, world),
        "frac_of_peak": round(value / world / peak, 4),
        "roofline": {
            "bound": "tensor",
            "kernel": "fa_bwd call (bwd_pre + bwd_kernel<128> + dq_convert launches)",
            "achieved": round(bwd_tflops, 1),
            "peak": peak,
            "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback 1.9 PFLOP/s",
            "unit": "TFLOP/s",
            "frac": round(bwd_tflops / peak, 4),
            "traffic": profile_traffic("bwd_kernel_train"),
            "algorithmic_flops_per_launch": bwd_flops,
        },
        "roofline_fwd": {
            "bound": "tensor",
            "kernel": "fwd_kernel<128> (one launch per fa_fwd)",
            "achieved": round(fwd_tflops, 1),
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": round(fwd_tflops / peak, 4),
            "traffic": profile_traffic("fwd_kernel_train"),
            "algorithmic_flops_per_launch": attn_flops(B, H, N, d, causal, "fwd"),
        },
        "fwd": fwd_results,
        "window": window_results,
        "dropout": dropout_results,
        "fp8": fp8_results,
        "d256": d256_results,
        "fp8_peak_note": "8-bit dense peak taken as 2 x the measured bf16 burst peak (the nominal 4.5 / 2.25 PFLOP/s ratio)",
        "e2e": {"value": round(job_tflops(world, step_flops, e2e_ms), 2),
                "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    return line


# ------------------------------------------------------- the oracle on CPU
def oracle_sample_step(w, heads, nthreads):
    """One bounded sample of the workload through the fp64 oracle: forward
    and backward of `heads` whole heads, one head per host thread."""
    import numpy as np
    import oracle
    from exact_tiled_attention_sm_gb300 import inputs
    x = inputs.seeded_inputs(1, heads, w.N, w.d, w.seed, w.dtype, with_dO=True)
    Q, K, V, dO = (inputs.to_f64(x[n]) for n in ("Q", "K", "V", "dO"))
    t = time.perf_counter()
    oracle.fwd(Q, K, V, w.scale, True, nthreads=nthreads)
    oracle.bwd(Q, K, V, dO, w.scale, True, nthreads=nthreads)
    return time.perf_counter() - t, attn_flops(1, heads, w.N, w.d, True, "fwd+bwd")


def cpu_baseline(w, budget_s=15.0):
    """The oracle on the host cores: a first batch of one head per core sizes
    the sample so that the timed batch takes about `budget_s` seconds (at most
    the whole workload)."""
    import oracle
    cores = oracle.cores()
    t1, _ = oracle_sample_step(w, cores, cores)
    total = w.B * w.H
    heads = max(cores, int(cores * budget_s / max(t1, 1e-3)) // cores * cores)
    heads = min(heads, total)
    secs, flops = oracle_sample_step(w, heads, cores)
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{heads} of the {total} heads of {w.name} (N={w.N}, d={w.d}, causal), "
                      f"fp64 forward + backward, one head per thread at a time, {secs:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    from exact_tiled_attention_sm_gb300 import inputs
    w = inputs.WORKLOADS[WORKLOAD]
    cores = oracle.cores()
    heads = cores
    for _ in range(args.warmup):
        oracle_sample_step(w, heads, cores)
    tot_s, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        s, f = oracle_sample_step(w, heads, cores)
        tot_s += s
        tot_f += f
    value = tot_f / tot_s / 1e12
    sample = (f"{heads} of the {w.B * w.H} heads of {w.name} per step (N={w.N}, d={w.d}, "
              f"causal), fp64 forward + backward, one head per host thread")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic: seeded iid N(0,1), rounded to bf16, widened to fp64",
        "config": bench_config(w, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--profile", action="store_true",
                    help="run only --workload's launches (for ncu captures)")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--causal", type=int, default=1)
    ap.add_argument("--window", type=int, default=0, help="profile: sliding window")
    ap.add_argument("--dropout", type=float, default=0.0, help="profile: dropout p")
    ap.add_argument("--fp8", action="store_true", help="profile: the 8-bit forward")
    ap.add_argument("--balance", action="store_true",
                    help="per-CTA balance of the schedulers (trace build)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.balance:
        line = run_balance(args)
    elif args.profile:
        line = run_profile(args)
    elif args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
