"""Throughput of diagonal-aware sparse decode attention on GB300.

A bench step is one decode step of the whole hot path for every layer of the
workload: 32 per-layer handles, each one fused kernel launch (plus a small
merge launch when streams are split) over batch x heads streams (append +
evict, index set from the skip bitmask, gather, split-K softmax.V, fused
argmin).  The metric counts stream-steps (sequence x layer x head) per second.

Default workload: the high-resolution stress stack (32 layers x 32 heads x
head_dim 128, bf16 KV, L_p 96, 90x90 grid = 8100 decode tokens, N_r 4050,
95 % sparsity -> N_att 405) at batch 64, about 139 GB of KV resident in HBM,
in the phase-3 steady state (t >= N_r).  Inputs are seeded synthetic traces
resident in HBM; each step reads every layer's KV (about 17 GB), far more
than the 129 MB L2.  The same line carries the dense setting of the same
kernel at the largest batch whose 32 layers of dense KV fit on the device,
and the Janus-Pro-7B-shaped stack at batch 96 as an extra key.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
sequences (weak scaling, no data-path collective); the time is the max over
ranks and the value counts all ranks' stream-steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode attn steps/s (batch·layers·heads) and HBM GB/s vs peak @95%"
UNIT = "stream-steps/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["ar_image_gen_gb300/csrc/dsa_decode.cuh", "ar_image_gen_gb300/csrc/dsa_ptx.cuh"]


def code_tokens(src: str) -> str:
    """C / CUDA source without its comments and with whitespace collapsed, so
    that a comment-only edit keeps the identity of the compiled kernel."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash() -> str:
    """Identity of the decode kernel's device code (comments and layout
    excluded): profile figures stored under profiles/ apply while it and the
    launch plan they were taken with are unchanged."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops() -> float:
    """Burst bf16 dense-GEMM TFLOP/s of this machine's GPUs (cuBLAS, measured),
    else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def profiled_traffic(workload: str, plan=None):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, or None when the kernel's code or the launch plan (pipeline,
    work items per stream, grid) changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"decode_kernel_{workload}.json")
    try:
        with open(path) as f:
            prof = json.load(f)
    except Exception:
        return None
    if prof.get("kernel_source_hash") != kernel_source_hash():
        return None
    if plan is not None:
        for key in ("pipeline", "nsplit", "grid"):
            if prof.get(key) != getattr(plan, key):
                return None
    return prof.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.proc = None
        self.uuid = gpu_uuid

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, flag in zip(names, f[4:8]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(c: dict) -> str | None:
    """Why a timed region's clock record disqualifies its number (a thermal
    or hardware slowdown, or SM clocks well below their maximum with no
    reason given, as a leftover clock lock would leave them), else None.
    sw_power_cap is kept: it is normal under a long bandwidth-bound load."""
    bad = [r for r in BAD_REASONS if r in c.get("reasons", [])]
    if bad:
        return "throttled: " + ", ".join(bad)
    sm, mx = c.get("sm_mhz"), c.get("sm_max_mhz")
    if sm and mx and not c.get("reasons") and sm < 0.9 * mx:
        return f"SM clock {sm:.0f} of {mx:.0f} MHz with no throttle reason"
    return None


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, ws


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_config(wl, phase: str) -> dict:
    return {
        "workload": (f"{wl.name}: {wl.layers} layers x {wl.heads} heads x head_dim {wl.head_dim}, "
                     f"batch {wl.batch}, {wl.dtype} KV, L_p {wl.L_p}, L_dec {wl.L_dec} "
                     f"({wl.grid}x{wl.grid} grid), N_r {wl.N_r}, N_att {wl.N_att}, sink {wl.sink}; {phase}"),
        "streams_per_layer": wl.streams,
        "layers": wl.layers,
        "l2": "no flush: each step reads every layer's KV (working set >> 129 MB L2)",
    }


# ----------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same workload
# ----------------------------------------------------------------------------

class OracleArm:
    """The C oracle (fp64, as it stands) on `n` streams of layer 0 of the
    workload; steps stay inside the trace (0 .. L_dec - 1): past its last
    step the sample is prefilled again and brought back, untimed, to the
    step it is timed from."""

    def __init__(self, wl, n: int, device: str):
        from ar_image_gen_gb300.synth import TraceGen
        from oracle.oracle import max_threads

        self.wl = wl
        self.gen = TraceGen(wl.with_batch(max(1, (n + wl.heads - 1) // wl.heads)), layer=0, device=device)
        self.n = min(n, self.gen.S)
        self.threads = max_threads()
        self.restart()

    def restart(self):
        from oracle.oracle import OracleBatch

        wl = self.wl
        ks = vs = None
        if wl.dtype == "fp8e4m3":
            ks, vs = (x[: self.n] for x in self.gen.kv_scales())
        self.orc = OracleBatch(self.n, wl.head_dim, wl.L_p, wl.N_r, wl.N_att, wl.sink, k_scales=ks, v_scales=vs)
        Kp, Vp = self.gen.prompt()
        self.orc.prefill(Kp[: self.n].double().cpu().numpy(), Vp[: self.n].double().cpu().numpy())
        self.t = 0

    def inputs(self):
        return [x[: self.n].double().cpu().numpy() for x in self.gen.step(self.t)]

    def advance(self, t_end: int):
        while self.t < t_end:
            self.orc.step(*self.inputs(), threads=self.threads)
            self.t += 1

    def timed_step(self, t_from: int) -> tuple[float, int]:
        """One decode step of the sample (from step t_from again once the
        trace is exhausted); returns its seconds (input generation and any
        restart excluded) and the step it ran."""
        if self.t >= self.wl.L_dec:
            self.restart()
            self.advance(t_from)
        q, k, v = self.inputs()
        t0 = time.perf_counter()
        self.orc.step(q, k, v, threads=self.threads)
        el = time.perf_counter() - t0
        self.t += 1
        return el, self.t - 1


def cpu_sample_streams(wl) -> int:
    """Streams of the oracle sample: as many as keep its untimed approach to
    the steady state (steps 0 .. N_r + sink - 1) near 1.5e8 row visits
    (a few seconds on the host cores), at least 32."""
    t0 = wl.N_r + wl.sink
    rows = sum(wl.L_p + min(t + 1, wl.N_att) for t in range(t0))
    return int(min(wl.streams, max(32, 1.5e8 // max(rows, 1))))


def step_ranges(steps: list[int]) -> str:
    """'a..b, c..d' for the runs of consecutive steps in `steps`."""
    runs, start, prev = [], None, None
    for t in steps:
        if start is None:
            start = prev = t
        elif t == prev + 1:
            prev = t
        else:
            runs.append((start, prev))
            start = prev = t
    if start is not None:
        runs.append((start, prev))
    return ", ".join(f"{a}..{b}" for a, b in runs)


def oracle_baseline(wl, n_streams: int = 0, budget_s: float = 10.0, device: str = "cuda") -> dict:
    """Stream-steps/s of the oracle on phase-3 steps of a sample of layer 0,
    timed until about `budget_s` seconds of oracle work have run."""
    arm = OracleArm(wl, n_streams or cpu_sample_streams(wl), device)
    t0 = wl.N_r + wl.sink
    arm.advance(t0)
    spent, ran = 0.0, []
    while spent < budget_s:
        el, t = arm.timed_step(t0)
        spent += el
        ran.append(t)
    steps = len(ran)
    return {"value": arm.n * steps / spent, "unit": UNIT, "cores": arm.threads, "kind": "oracle",
            "sample": f"{arm.n} streams of layer 0, phase-3 steps {step_ranges(ran)} of the {wl.L_dec}-step trace "
                      f"({arm.n * steps} stream-steps in {spent:.1f} s of oracle time, fp64 C oracle, "
                      f"input generation excluded)"}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

class Stack:
    """Per-layer handles of one workload, prefilled and advanced to a step."""

    def __init__(self, wl, pool_steps: int, device: str = "cuda"):
        import torch

        from ar_image_gen_gb300.dsa import DSA
        from ar_image_gen_gb300.synth import TraceGen

        self.wl = wl
        self.handles = []
        self.gens = []
        self.outs = []
        self.pool_steps = pool_steps
        self.pool = None
        try:
            for layer in range(wl.layers):
                gen = TraceGen(wl, layer=layer, device=device)
                h = DSA(wl.streams, wl.head_dim, wl.L_p, wl.N_r, wl.N_att, wl.sink, wl.dtype)
                self.handles.append(h)
                if wl.dtype == "fp8e4m3":
                    h.set_kv_scales(*gen.kv_scales())
                Kp, Vp = gen.prompt()
                h.prefill(Kp, Vp)
                self.gens.append(gen)
                self.outs.append(torch.empty((wl.streams, wl.head_dim), dtype=Kp.dtype, device=device))
                del Kp, Vp
        except BaseException:
            self.close()
            raise

    def advance(self, t_end: int, generate: bool = True):
        """Decode steps t = current .. t_end - 1 with freshly drawn inputs."""
        t = self.handles[0].t
        while t < t_end:
            for layer, h in enumerate(self.handles):
                q, k, v = self.gens[layer].step(min(t, self.wl.L_dec - 1)) if generate else self.pool[t % self.pool_steps][layer]
                h.decode_step(q, k, v, self.outs[layer])
            t += 1

    def make_pool(self, t0: int):
        """Inputs of pool_steps consecutive steps from t0, resident in HBM."""
        self.pool = []
        for i in range(self.pool_steps):
            t = min(t0 + i, self.wl.L_dec - 1)
            self.pool.append([self.gens[layer].step(t) for layer in range(self.wl.layers)])

    def reprefill(self):
        """Prefills every layer again (t = 0, empty skip sets)."""
        for layer, h in enumerate(self.handles):
            Kp, Vp = self.gens[layer].prompt()
            h.prefill(Kp, Vp)

    def close(self):
        for h in self.handles:
            h.close()
        self.handles = []
        self.pool = None
        self.outs = []


def time_steps(stack, steps: int, per_launch: bool):
    """Runs `steps` bench steps from the input pool; returns (elapsed_ms,
    mean per-launch ms or None, launches)."""
    import torch

    wl = stack.wl
    stream = torch.cuda.current_stream()
    launches = 0
    evs = []
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    t = stack.handles[0].t
    for i in range(steps):
        inputs = stack.pool[(t + i) % stack.pool_steps]
        for layer, h in enumerate(stack.handles):
            q, k, v = inputs[layer]
            if per_launch:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                h.decode_step(q, k, v, stack.outs[layer], stream)
                e1.record(stream)
                evs.append((e0, e1))
            else:
                h.decode_step(q, k, v, stack.outs[layer], stream)
            launches += 1
    end.record(stream)
    torch.cuda.synchronize()
    el = start.elapsed_time(end)
    per = statistics.fmean(a.elapsed_time(b) for a, b in evs) if evs else None
    return el, per, launches


def time_trace(stack, runs: int):
    """The whole decode trace (steps 0 .. L_dec - 1 of every layer: fill,
    selection and eviction phases) from a fresh prefill, `runs` times, inputs
    cycled from the pool.  Returns a summary dict: stream-steps/s and GB/s of
    algorithmic bytes, mean with min and max over the runs."""
    import torch

    wl = stack.wl
    stream = torch.cuda.current_stream()
    nbytes = sum(stack.handles[0].plan(t).algo_bytes for t in range(wl.L_dec)) * wl.layers
    times = []
    for _ in range(runs):
        stack.reprefill()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for t in range(wl.L_dec):
            inputs = stack.pool[t % stack.pool_steps]
            for layer, h in enumerate(stack.handles):
                q, k, v = inputs[layer]
                h.decode_step(q, k, v, stack.outs[layer], stream)
        end.record(stream)
        torch.cuda.synchronize()
        times.append(start.elapsed_time(end))
    rates = [wl.streams * wl.layers * wl.L_dec / (ms / 1e3) for ms in times]
    gbs = [nbytes / (ms / 1e3) / 1e9 for ms in times]
    return {"steps": f"0..{wl.L_dec - 1}", "layers": wl.layers, "runs": runs,
            "value": statistics.fmean(rates), "min": min(rates), "max": max(rates), "unit": UNIT,
            "hbm_gbs": statistics.fmean(gbs), "ms_per_trace": statistics.fmean(times),
            "algo_bytes_per_trace": nbytes}


def time_graph(stack, steps: int, ws: int) -> dict:
    """Steady-state steps replayed from a CUDA graph that holds one decode
    step of every layer (graph mode), timed with CUDA events; returns
    stream-steps/s and the average launch time.  The handles return to host
    steps afterwards."""
    import torch

    wl = stack.wl
    for h in stack.handles:
        h.set_graph_mode(True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for layer, h in enumerate(stack.handles):
            q, k, v = stack.pool[0][layer]
            h.decode_step(q, k, v, stack.outs[layer])
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s)
    with torch.cuda.stream(s):
        for _ in range(steps):
            g.replay()
    end.record(s)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), ws)
    for h in stack.handles:
        h.sync_step()
        h.set_graph_mode(False)
    return {"value": wl.streams * wl.layers * steps * ws / (ms / 1e3), "unit": UNIT, "steps": steps,
            "ms_per_step": ms / steps, "launch_ms": ms / (steps * wl.layers)}


def time_e2e(stack, steps: int):
    """Same metric through the public API with host-resident inputs, as a
    pipelined caller would run it: every step copies q, k_new, v_new of all
    layers from pinned host memory (one copy, on a copy stream, overlapping
    the previous step's kernels; device buffers double-buffered), decodes all
    layers, and copies all layers' outputs back to pinned host memory (one
    copy, on a third stream).  Returns (elapsed_ms, h2d bytes per step, d2h
    bytes per step); the elapsed time spans the first copy in to the last
    copy out."""
    import torch

    wl = stack.wl
    L, S, d = wl.layers, wl.streams, wl.head_dim
    dt = stack.outs[0].dtype
    compute = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    host_in = []
    for i in range(2):  # two distinct steps of inputs, cycled
        x = torch.empty((L, 3, S, d), dtype=dt).pin_memory()
        for layer in range(L):
            for j in range(3):
                x[layer, j].copy_(stack.pool[i % stack.pool_steps][layer][j])
        host_in.append(x)
    dev_in = [torch.empty((L, 3, S, d), dtype=dt, device="cuda") for _ in range(2)]
    dev_out = [torch.empty((L, S, d), dtype=dt, device="cuda") for _ in range(2)]
    host_out = [torch.empty((L, S, d), dtype=dt).pin_memory() for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    h2d = host_in[0].numel() * host_in[0].element_size()
    d2h = host_out[0].numel() * host_out[0].element_size()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    start.record(compute)
    h2d_s.wait_stream(compute)
    d2h_s.wait_stream(compute)
    with torch.cuda.stream(h2d_s):
        dev_in[0].copy_(host_in[0], non_blocking=True)
        in_ready[0].record(h2d_s)
    for i in range(steps):
        b = i % 2
        if i + 1 < steps:  # next step's inputs, once the step that last used the buffer is done
            nb = (i + 1) % 2
            if i >= 1:
                h2d_s.wait_event(done[nb])
            with torch.cuda.stream(h2d_s):
                dev_in[nb].copy_(host_in[(i + 1) % 2], non_blocking=True)
                in_ready[nb].record(h2d_s)
        compute.wait_event(in_ready[b])
        if i >= 2:
            compute.wait_event(out_read[b])  # dev_out[b] has been copied out
        for layer, h in enumerate(stack.handles):
            x = dev_in[b][layer]
            h.decode_step(x[0], x[1], x[2], dev_out[b][layer], compute)
        done[b].record(compute)
        d2h_s.wait_event(done[b])
        with torch.cuda.stream(d2h_s):
            host_out[b].copy_(dev_out[b], non_blocking=True)
            out_read[b].record(d2h_s)
    compute.wait_stream(d2h_s)
    end.record(compute)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) * 1e3
    return max(start.elapsed_time(end), wall), h2d, d2h


def kernels_per_step(stack, t: int) -> int:
    """Kernel launches of one decode step of every layer at step t: the
    decode kernel, plus the merge kernel where streams are split."""
    p = stack.handles[0].plan(t)
    return stack.wl.layers * (2 if p.nsplit > 1 else 1)


def dense_stack(wl, pool_steps: int):
    """The dense setting (N_r = N_att = L_dec) of the workload at the largest
    batch, from the workload's own down, whose layers all fit on the device.
    Returns (stack, batches tried that did not fit)."""
    import torch

    from ar_image_gen_gb300.dsa import DSA_ERR_OOM, DSAError

    tried, b = [], wl.batch
    while b >= 1:
        st = None
        try:
            st = Stack(wl.dense().with_batch(b), pool_steps=pool_steps)
            st.make_pool(0)
            return st, tried
        except (DSAError, torch.cuda.OutOfMemoryError) as e:
            if isinstance(e, DSAError) and e.code != DSA_ERR_OOM:
                raise
            if st is not None:
                st.close()
            del st
            torch.cuda.empty_cache()
            tried.append(b)
            b = b - 8 if b > 16 else b // 2
    raise RuntimeError("no batch of the dense setting fits on the device")


def time_dense(wl, args, peak: float, last_sparse_ms: float) -> dict:
    """The 0 % sparsity setting of the same kernel at the largest batch that
    fits: the last `dense_steps` steps of the trace (every layer, back to
    back) and the last step alone.  The handles jump to the first timed step
    (dsa_debug_set_step: the entries before it are zero rows, which move the
    same bytes through the same launches as real ones)."""
    import torch

    dstack, tried = dense_stack(wl, args.pool)
    dwl = dstack.wl
    d_steps = max(2, min(args.dense_steps, dwl.L_dec - 1))
    t_first = dwl.L_dec - 1 - d_steps
    for h in dstack.handles:
        h.debug_set_step(t_first)
    time_steps(dstack, 1, per_launch=False)  # warm-up step t_first
    t_first += 1
    d_steps -= 1
    d_ms, _, _ = time_steps(dstack, d_steps, per_launch=False)
    d_bytes = sum(dstack.handles[0].plan(t_first + i).algo_bytes for i in range(d_steps))
    last_dense_ms = _last_step_ms(dstack)
    dplan_last = dstack.handles[0].plan(dwl.L_dec - 1)
    status = max((h.sync_status() for h in dstack.handles), key=abs)
    kv_gb = sum(1 for _ in dstack.handles) * dstack.handles[0].state_bytes() / 1e9
    dstack.close()
    del dstack
    torch.cuda.empty_cache()
    res = {
        "workload": f"{dwl.name}: N_r = N_att = L_dec = {dwl.L_dec}, batch {dwl.batch} (largest that fits; "
                    f"{kv_gb:.1f} GB of KV over {dwl.layers} layers), steps {t_first}..{t_first + d_steps - 1}",
        "batch": dwl.batch, "batches_that_did_not_fit": tried, "kv_gb": kv_gb,
        "value": dwl.streams * dwl.layers * d_steps / (d_ms / 1e3), "unit": UNIT,
        "hbm_gbs": d_bytes * dwl.layers / (d_ms / 1e3) / 1e9,
        "frac": d_bytes * dwl.layers / (d_ms / 1e3) / 1e9 / peak,
        "last_step_ms": last_dense_ms,
        "last_step_gbs": dplan_last.algo_bytes * dwl.layers / (last_dense_ms / 1e3) / 1e9,
        "device_status": status,
    }
    if dwl.batch == wl.batch:
        res["last_step_speedup_sparse_vs_dense"] = last_dense_ms / last_sparse_ms
    else:
        res["last_step_speedup_sparse_vs_dense_per_stream"] = (last_dense_ms / dwl.batch) / (last_sparse_ms / wl.batch)
    return res


def time_extra(key: str, args, ws: int, peak: float) -> dict:
    """Another workload's sparse steady state (all its layers), timed like the
    main line: stream-steps/s and the decode kernel's roofline fraction."""
    import torch

    from ar_image_gen_gb300.synth import WORKLOADS

    wl = WORKLOADS[key]
    if args.kv == "fp8":
        wl = wl.fp8()
    stack = Stack(wl, pool_steps=args.pool)
    t_start = wl.N_r + wl.sink
    stack.advance(t_start)
    stack.make_pool(t_start)
    plan = stack.handles[0].plan(t_start)
    time_steps(stack, args.warmup, per_launch=False)
    barrier(ws)
    steps = max(20, args.steps)
    el_ms, _, launches = time_steps(stack, steps, per_launch=False)
    el_ms = max_over_ranks(el_ms, ws)
    per_launch_ms = el_ms / launches
    achieved = plan.algo_bytes / (per_launch_ms / 1e3) / 1e9
    status = max((h.sync_status() for h in stack.handles), key=abs)
    stack.close()
    del stack
    torch.cuda.empty_cache()
    return {"workload": workload_config(wl, f"phase-3 steady state from t = {t_start}")["workload"],
            "value": wl.streams * wl.layers * steps * ws / (el_ms / 1e3), "unit": UNIT, "steps": steps,
            "ms_per_step": el_ms / steps, "launch_ms": per_launch_ms, "algo_bytes_per_launch": plan.algo_bytes,
            "achieved_gbs": achieved, "frac": achieved / peak, "traffic": profiled_traffic(wl.name, plan),
            "pipeline": plan.pipeline, "nsplit": plan.nsplit, "device_status": status}


def run_ours(args, rank: int, ws: int) -> dict | None:
    import torch

    from __graft_entry__ import build

    build()
    torch.cuda.init()
    wl = _workload(args)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    peak, peak_kind = measured_peak()

    # --- sparse setting, phase-3 steady state
    stack = Stack(wl, pool_steps=args.pool)
    t_start = wl.N_r + wl.sink
    stack.advance(t_start)
    stack.make_pool(t_start)
    plan = stack.handles[0].plan(t_start)
    _, _, _ = time_steps(stack, args.warmup, per_launch=False)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(uuid) as clk:
        torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed region's launches
        el_ms, _, launches = time_steps(stack, args.steps, per_launch=False)
        torch.cuda.nvtx.range_pop()
    clocks = clk.summary()
    why = clocks_rejected(clocks)
    if why:  # measured again, once, and the second number reported
        barrier(ws)
        torch.cuda.synchronize()
        with ClockSampler(uuid) as clk:
            el_ms, _, launches = time_steps(stack, args.steps, per_launch=False)
        clocks = dict(clk.summary(), first_run_rejected=why)
    el_ms = max_over_ranks(el_ms, ws)
    # The timed region launches only the decode kernel (and, where streams
    # are split, its merge kernel), back to back (each launch may overlap the
    # previous one's tail): its average duration is the region's time over
    # the decode launches.  A second pass with events around every launch
    # gives the duration of a launch that cannot overlap.
    per_launch_ms = el_ms / launches
    gpu_launches = kernels_per_step(stack, t_start) * args.steps
    _, isolated_ms, _ = time_steps(stack, max(4, min(args.steps, 50)), per_launch=True)
    stream_steps = wl.streams * wl.layers * args.steps * ws
    value = stream_steps / (el_ms / 1e3)
    achieved = plan.algo_bytes / (per_launch_ms / 1e3) / 1e9
    whole = plan.algo_bytes * wl.layers * args.steps * ws / (el_ms / 1e3) / 1e9
    traffic = profiled_traffic(wl.name, plan)

    # --- the same steady state replayed from a CUDA graph (graph mode: the
    # step lives on the device; one capture of all layers, replayed per step;
    # inputs are the pool's first step in every replay, which does not change
    # the work)
    graph = None
    if args.graph:
        graph = time_graph(stack, max(4, min(args.steps, 200)), ws)
        graph["frac"] = plan.algo_bytes / (graph["launch_ms"] / 1e3) / 1e9 / peak

    # --- end to end through the public API with host buffers
    e2e_steps = max(50, min(args.steps, 200))
    e2e_ms, h2d, d2h = time_e2e(stack, e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, ws)
    e2e_value = wl.streams * wl.layers * e2e_steps * ws / (e2e_ms / 1e3)

    # last step of the trace, sparse
    stack.advance(wl.L_dec - 1, generate=False)
    last_sparse_ms = _last_step_ms(stack)
    status = max((h.sync_status() for h in stack.handles), key=abs)
    # the whole trace, all phases: three runs where a run is short, else one
    trace = None
    if not args.no_trace:
        est_s = sum(stack.handles[0].plan(t).algo_bytes for t in range(wl.L_dec)) * wl.layers / (0.8 * peak * 1e9)
        trace = time_trace(stack, 3 if est_s < 20 else 1)
        trace["frac"] = trace["hbm_gbs"] / peak
        status = max([status] + [h.sync_status() for h in stack.handles], key=abs)
    stack.close()
    del stack
    torch.cuda.empty_cache()

    # --- dense setting (0 % sparsity) of the same kernel: N_r = N_att = L_dec
    dense = None if args.no_dense else time_dense(wl, args, peak, last_sparse_ms)

    # --- other workloads' steady state, as extra keys
    extra = {}
    for key in ([] if args.no_extra else [k for k in args.extra.split(",") if k and k != args.workload]):
        extra[key] = time_extra(key, args, ws, peak)

    if rank != 0:
        return None
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": workload_config(wl, f"phase-3 steady state from t = {t_start}"),
        "hbm_gbs": whole,
        "roofline": {"bound": "hbm", "kernel": f"dsa::decode_kernel<{wl.dtype},{wl.head_dim},{(plan.pipeline - 1) & 1}>, "
                                                  f"{2 + (plan.pipeline - 1) // 2} stages per warp",
                     "achieved": achieved,
                     "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algo_bytes_per_launch": plan.algo_bytes, "launch_ms": per_launch_ms,
                     "launch_ms_note": "timed region / decode launches (merge launches of split streams included)",
                     "isolated_launch_ms": isolated_ms,
                     "grid": plan.grid, "nsplit": plan.nsplit, "pipeline": plan.pipeline},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "last_step": {"sparse_ms": last_sparse_ms},
        "trace": trace,
        "graph": graph,
        "dense": dense,
        "extra": extra,
        "device_status": status,
    }
    if dense is not None:
        res["config"]["dense_batch"] = dense["batch"]
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = oracle_baseline(wl, budget_s=args.cpu_budget)
    if args.layers:
        res["config"]["layers_override"] = args.layers
    return res


def _last_step_ms(stack) -> float:
    """Duration of the final decode step of the trace (all layers)."""
    import torch

    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t = stack.handles[0].t
    a.record(stream)
    for layer, h in enumerate(stack.handles):
        q, k, v = stack.pool[t % stack.pool_steps][layer]
        h.decode_step(q, k, v, stack.outs[layer], stream)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def run_reference(args, rank: int, ws: int) -> dict | None:
    """The reference arm: the CPU oracle, as it stands, on this workload.
    Each bench step is one phase-3 decode step of a fixed sample of streams."""
    if rank != 0:
        return None
    import torch

    from ar_image_gen_gb300.synth import WORKLOADS
    from oracle.oracle import build as build_oracle

    build_oracle()
    wl = _workload(args)
    device = "cuda" if torch.cuda.is_available() else "cpu"
    arm = OracleArm(wl, args.ref_streams or cpu_sample_streams(wl), device)
    t0 = wl.N_r + wl.sink
    arm.advance(t0)
    for _ in range(args.warmup):
        arm.timed_step(t0)
    spent, ran = 0.0, []
    for _ in range(args.steps):
        el, t = arm.timed_step(t0)
        spent += el
        ran.append(t)
    value = arm.n * args.steps / spent
    sample = (f"each step: one phase-3 decode step of {arm.n} streams of layer 0 "
              f"(steps {step_ranges(ran)} of the {wl.L_dec}-step trace), fp64 C oracle, "
              f"input generation excluded")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, f"phase-3 steady state from t = {t0}"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": arm.threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _workload(args):
    from dataclasses import replace

    from ar_image_gen_gb300.synth import WORKLOADS

    wl = WORKLOADS[args.workload]
    if args.layers:
        wl = replace(wl, layers=args.layers)
    if getattr(args, "calibrated", False):
        wl = wl.calibrated()
    if args.kv == "fp8":
        wl = wl.fp8()
    return wl


SWEEP = ["janus-b32", "janus-b96", "sweep512-s50", "sweep512-s75", "sweep512-s90", "sweep512-s95",
         "sweep512-sink4-s95", "lumina-s90-b16", "lumina-s90-b32", "lumina-s90-b54", "lumina-s95-b16", "lumina-s95-b32",
         "lumina-s95-b54", "stress-s95"]


def run_sweep(args) -> None:
    """One JSON line per workload (sparse, phase-3 steady state) and per dense
    setting (last steps of the trace): average launch time back to back over
    `layers` distinct layers, GB/s of algorithmic bytes and the fraction of
    the measured peak.  Not the benchmark contract's line."""
    import torch
    from dataclasses import replace

    from __graft_entry__ import build
    from ar_image_gen_gb300.synth import WORKLOADS

    build()
    peak, peak_kind = measured_peak()
    layers = args.layers or 4
    for key in (args.sweep_only.split(",") if args.sweep_only else SWEEP):
        base = replace(WORKLOADS[key], layers=layers)
        if args.kv == "fp8":
            base = base.fp8()
        for dense in ((False,) if args.sparse_only else (False, True)):
            wl = base.dense() if dense else base
            steps = max(8, min(args.steps, 40))
            st = Stack(wl, pool_steps=4)
            for h in st.handles:
                if args.splits:
                    h.set_splits(args.splits)
                if args.pipeline:
                    h.set_pipeline(args.pipeline)
            t0 = (wl.L_dec - steps) if dense else wl.N_r + wl.sink
            st.make_pool(min(t0, wl.L_dec - 1))
            if dense:  # jump to the last steps (the entries before them are zero rows: same bytes, same launches)
                for h in st.handles:
                    h.debug_set_step(t0)
            else:
                st.advance(t0, generate=False)
                time_steps(st, 3, per_launch=False)
            t_first = st.handles[0].t
            plan = st.handles[0].plan(t_first)
            el, _, n = time_steps(st, steps, per_launch=False)
            nbytes = sum(st.handles[0].plan(t_first + i).algo_bytes for i in range(steps)) * wl.layers
            gbs = nbytes / (el / 1e3) / 1e9
            line = {"workload": wl.name, "dense": dense, "streams": wl.streams, "layers": wl.layers,
                    "rows_per_stream": plan.n_prefix + plan.n_decode, "nsplit": plan.nsplit,
                    "pipeline": plan.pipeline, "grid": plan.grid,
                    "steps": f"{t_first}..{t_first + steps - 1}", "ms_per_launch": el / n,
                    "stream_steps_per_s": wl.streams * n / (el / 1e3), "gbs": gbs,
                    "frac": gbs / peak, "peak": f"{peak} ({peak_kind})"}
            if args.trace:
                line["trace"] = time_trace(st, 3)
                line["trace"]["frac"] = line["trace"]["hbm_gbs"] / peak
            line["status"] = max((h.sync_status() for h in st.handles), key=abs)
            print(json.dumps(line), flush=True)
            st.close()
            del st
            torch.cuda.empty_cache()


def run_fused(args) -> None:
    """The fused layer step (QKV projection with RoPE on the tensor cores,
    then the decode kernel on its output) for every layer of the workload,
    phase-3 steady state; plus the projection kernel alone, back to back over
    the layers (each layer's W is read from HBM: 30 x 100 MB per step at
    janus-b96) and with events around each launch.  One JSON line; not the
    benchmark contract's line."""
    import numpy as np
    import torch

    from __graft_entry__ import build
    from ar_image_gen_gb300.dsa import Proj
    from ar_image_gen_gb300.synth import ProjGen
    from oracle.proj import qkv_rope as oracle_qkv_rope

    build()
    wl = _workload(args)
    peak, peak_kind = measured_peak()
    stack = Stack(wl, pool_steps=args.pool)
    t_start = wl.N_r + wl.sink
    stack.advance(t_start)
    pgens = [ProjGen(wl, layer=layer, device="cuda") for layer in range(wl.layers)]
    Ws = [g.weight() for g in pgens]
    projs = [Proj(wl.batch, wl.heads, wl.head_dim, g.hidden) for g in pgens]
    xpool = [[g.x(t_start + i) for g in pgens] for i in range(args.pool)]
    hidden, HD, B = pgens[0].hidden, wl.heads * wl.head_dim, wl.batch
    # the projection alone (dsa_qkv_rope): W and x read, q, k, v written (bf16)
    proj_bytes = 3 * HD * hidden * 2 + B * hidden * 2 + 3 * B * HD * 2
    proj_flops = 2.0 * B * hidden * 3 * HD
    # the fused layer step: the projection writes q (bf16) and the newest entry
    # in its stored form straight into the decode state; the decode kernel
    # reads q, the attended rows (the newest entry among them) and writes out
    e = 1 if wl.dtype == "fp8e4m3" else 2
    d = wl.head_dim
    pl0 = stack.handles[0].plan(t_start)
    rows = pl0.n_prefix + pl0.n_decode
    fused_bytes = (3 * HD * hidden * 2 + B * hidden * 2
                   + wl.streams * (2 * d + 2 * d * e + 2 * d * e * rows + 2 * d + 2 * d))
    stream = torch.cuda.current_stream()
    q, k, v = (torch.empty((wl.streams, wl.head_dim), dtype=torch.bfloat16, device="cuda") for _ in range(3))

    def fused_steps(n):
        t = stack.handles[0].t
        for i in range(n):
            xs = xpool[(t + i - t_start) % args.pool]
            for layer, h in enumerate(stack.handles):
                h.decode_step_fused(projs[layer], xs[layer], Ws[layer], stack.outs[layer], stream)

    def proj_steps(n, events=False):
        evs = []
        for i in range(n):
            xs = xpool[i % args.pool]
            for layer in range(wl.layers):
                if events:
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                projs[layer].qkv_rope(xs[layer], Ws[layer], wl.L_p + t_start + i, q, k, v, stream)
                if events:
                    e1.record(stream)
                    evs.append((e0, e1))
        return evs

    def timed(fn, *a):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        r = fn(*a)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), r

    fused_steps(args.warmup)
    plan = stack.handles[0].plan()
    steps = max(3, min(args.steps, 200))
    with ClockSampler(None) as clk:
        el_fused, _ = timed(fused_steps, steps)
        proj_steps(args.warmup)
        el_proj, _ = timed(proj_steps, steps)
    _, evs = timed(proj_steps, max(3, min(steps, 20)), True)
    iso = statistics.fmean(a.elapsed_time(b) for a, b in evs)
    per_proj = el_proj / (steps * wl.layers)

    # for context: the library GEMM of the same shapes (torch.matmul on
    # cuBLAS, x W^T without RoPE), back to back over the layers
    def lib_steps(n):
        for i in range(n):
            xs = xpool[i % args.pool]
            for layer in range(wl.layers):
                torch.matmul(xs[layer], Ws[layer].t())

    lib_steps(args.warmup)
    el_lib, _ = timed(lib_steps, steps)
    per_lib = el_lib / (steps * wl.layers)
    status = max([h.sync_status() for h in stack.handles] + [p.sync_status() for p in projs], key=abs)
    # the oracle's projection (numpy fp64) on one layer, for scale
    x0 = xpool[0][0].double().cpu().numpy()
    W0 = Ws[0].double().cpu().numpy()
    t0 = time.perf_counter()
    oracle_qkv_rope(x0, W0, wl.heads, wl.head_dim, wl.L_p + t_start)
    cpu_s = time.perf_counter() - t0
    n_fused = wl.streams * wl.layers * steps
    line = {
        "mode": "fused layer step (QKV projection + RoPE on tcgen05, then sparse decode attention)",
        "config": workload_config(wl, f"phase-3 steady state from t = {t_start}; hidden {hidden}"),
        "fused": {"value": n_fused / (el_fused / 1e3), "unit": UNIT, "ms_per_step": el_fused / steps,
                  "ms_per_layer": el_fused / (steps * wl.layers),
                  "hbm_gbs": fused_bytes * wl.layers * steps / (el_fused / 1e3) / 1e9,
                  "frac": fused_bytes * wl.layers * steps / (el_fused / 1e3) / 1e9 / peak,
                  "algo_bytes_per_layer": fused_bytes, "launches_per_layer": 2 if plan.nsplit == 1 else 3},
        "projection": {"kernel": "dsa_proj_k::qkv_rope_kernel", "bound": "hbm", "launch_ms": per_proj,
                       "isolated_launch_ms": iso, "algo_bytes_per_launch": proj_bytes,
                       "achieved": proj_bytes / (per_proj / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                       "peak_kind": f"{peak_kind} hbm_gbs", "frac": proj_bytes / (per_proj / 1e3) / 1e9 / peak,
                       "tflops": proj_flops / (per_proj / 1e3) / 1e12,
                       "tensor_frac_of_bf16_peak": proj_flops / (per_proj / 1e3) / 1e12 / measured_bf16_tflops(),
                       "library_gemm_ms": per_lib,
                       "library_gemm_note": "torch.matmul (cuBLAS) of x by W^T, same shapes, no RoPE, back to back"},
        "clocks": clk.summary(), "steps": steps, "warmup": args.warmup,
        "cpu_baseline": {"seconds_per_layer_projection": cpu_s, "kind": "oracle", "cores": "numpy BLAS",
                         "sample": "layer 0, one step, fp64 x W^T and RoPE"},
        "device_status": status,
    }
    print(json.dumps(line), flush=True)
    for p_ in projs:
        p_.close()
    stack.close()


def run_policies(args) -> None:
    """The score-based eviction baselines (TOVA, H2O) next to the diagonal
    method on the same workload and budget N_att: per workload family and
    policy, `layers` distinct layers stepped back to back in the steady state
    (t >= N_att, every step evicts), average launch time, stream-steps/s and
    GB/s of algorithmic bytes (K|V rows read, q / k_new / v_new read, out and
    the new entry written, plus 4 bytes of slot position per attended decode
    row and, for H2O, 8 bytes of accumulated weight).  One JSON line each;
    not the benchmark contract's line."""
    import torch
    from dataclasses import replace

    from __graft_entry__ import build
    from ar_image_gen_gb300.dsa import Policy
    from ar_image_gen_gb300.synth import WORKLOADS, TraceGen

    build()
    peak, peak_kind = measured_peak()
    layers = args.layers or 4
    steps = max(8, min(args.steps, 40))
    for key in (args.sweep_only.split(",") if args.sweep_only else ["janus-b96", "sweep512-s95", "lumina-s95-b32"]):
        wl = replace(WORKLOADS[key], layers=layers)
        d, e, a = wl.head_dim, 2, wl.N_att
        for policy in ("tova", "h2o"):
            hs, gens, outs = [], [], []
            for layer in range(layers):
                gen = TraceGen(wl, layer=layer, device="cuda")
                h = Policy(wl.streams, d, wl.L_p, wl.N_att, policy, wl.dtype)
                Kp, Vp = gen.prompt()
                h.prefill(Kp, Vp)
                hs.append(h)
                gens.append(gen)
                outs.append(torch.empty((wl.streams, d), dtype=Kp.dtype, device="cuda"))
            pool = [[gens[l].step(t) for l in range(layers)] for t in range(4)]
            stream = torch.cuda.current_stream()

            def go(n):
                for i in range(n):
                    for l, h in enumerate(hs):
                        q, k, v = pool[i % 4][l]
                        h.decode_step(q, k, v, outs[l], stream)

            go(wl.N_att + 3)  # fill the caches; every later step evicts
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            go(steps)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / (steps * layers)
            per_stream = 2 * d * e * (wl.L_p + a - 1) + 4 * d * e + 2 * d * e + 4 * (a - 1) + (8 * (a - 1) if policy == "h2o" else 0)
            nbytes = per_stream * wl.streams
            status = max((h.sync_status() for h in hs), key=abs)
            line = {"workload": key, "policy": policy, "streams": wl.streams, "layers": layers, "N_att": a,
                    "L_p": wl.L_p, "ms_per_launch": ms, "stream_steps_per_s": wl.streams / (ms / 1e3),
                    "algo_bytes_per_launch": nbytes, "gbs": nbytes / (ms / 1e3) / 1e9,
                    "frac": nbytes / (ms / 1e3) / 1e9 / peak, "peak": f"{peak} ({peak_kind})", "status": status}
            print(json.dumps(line), flush=True)
            for h in hs:
                h.close()
            del hs, pool, outs
            torch.cuda.empty_cache()


def run_diag(args) -> None:
    """Attention diagnostics (section 3.4: Fig. 8 prompt / local / middle
    weight, Fig. 10 vertical vs diagonal score-vector similarity) of the dense
    trace of layer 0, batch 1, of each workload family: one JSON line each,
    with the call's wall time and the oracle's time on one head for scale.
    Not the benchmark contract's line."""
    import torch

    from __graft_entry__ import build
    from ar_image_gen_gb300.dsa import diag_trace
    from ar_image_gen_gb300.synth import WORKLOADS, TraceGen
    from oracle.oracle import diag_stream

    build()
    for key, heads in (("janus-b32", 32), ("sweep512-s95", 32), ("lumina-s95-b16", 32), ("stress-s95", 8)):
        wl = WORKLOADS[key].with_batch(1)
        if args.calibrated:
            wl = wl.calibrated()
        g = wl.grid
        dists = sorted({d for d in (1, 2, 4, g - 1, g, g + 1, 2 * g, 4 * g) if 1 <= d < wl.L_dec})
        gen = TraceGen(wl, device="cuda")
        Kp, _ = gen.prompt()
        steps = [gen.step(t) for t in range(wl.L_dec)]
        Q = torch.stack([x[0] for x in steps], 1)[:heads].contiguous()
        Kd = torch.stack([x[1] for x in steps], 1)[:heads].contiguous()
        Kp = Kp[:heads].contiguous()
        del steps
        diag_trace(Q[:1], Kp[:1], Kd[:1], dists)  # warm-up
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        mass, vert, diag = diag_trace(Q, Kp, Kd, dists)
        el = time.perf_counter() - t0
        flops = 2.0 * heads * wl.head_dim * sum(wl.L_p + i + 1 for i in range(wl.L_dec))
        line = {"diagnostic": "attention mass and score-vector similarity", "workload": f"{wl.name}, layer 0, batch 1",
                "heads": heads, "L_p": wl.L_p, "L_dec": wl.L_dec,
                "mass": {"prompt": mass[0], "local": mass[1], "middle": mass[2]},
                "similarity": {str(d): {"vertical": v, "diagonal": dg} for d, v, dg in zip(dists, vert, diag)},
                "seconds": el, "logit_gflops_per_s": flops / el / 1e9,
                "page": "middle weight 6.2 % (Janus-Pro), 8.1 % (NextStep-1), 8.5 % (Lumina-mGPT) on real "
                        "traces (Fig. 8); diagonal above vertical similarity for image models (Fig. 10)"}
        if wl.L_dec <= 1024:
            t0 = time.perf_counter()
            diag_stream(Q[0].double().cpu().numpy(), Kp[0].double().cpu().numpy(), Kd[0].double().cpu().numpy(), dists)
            line["cpu_baseline"] = {"seconds_per_head": time.perf_counter() - t0, "kind": "oracle", "cores": 1,
                                    "sample": "head 0 of the same trace"}
        print(json.dumps(line), flush=True)
        del Q, Kd, Kp
        torch.cuda.empty_cache()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stress-s95")
    ap.add_argument("--extra", default="janus-b96", help="comma-separated workloads timed as extra keys")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--pool", type=int, default=8, help="distinct input steps kept in HBM and cycled")
    ap.add_argument("--dense-steps", type=int, default=16)
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-trace", action="store_true", help="skip the whole-trace timing")
    ap.add_argument("--graph", action="store_true", help="also time the steady state replayed from a CUDA graph")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-streams", type=int, default=0,
                    help="streams per step of the reference arm (0: as many as keep its untimed approach short)")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling runs)")
    ap.add_argument("--kv", choices=["native", "fp8"], default="native",
                    help="fp8: store the KV state as FP8 E4M3 (q, k, v, out stay bf16)")
    ap.add_argument("--sweep", action="store_true", help="time every workload family (one JSON line each)")
    ap.add_argument("--sweep-only", default="", help="comma-separated workloads for --sweep")
    ap.add_argument("--splits", type=int, default=0, help="--sweep: force this many work items per stream")
    ap.add_argument("--pipeline", type=int, default=0, help="--sweep: force this launch pipeline (1 .. 4)")
    ap.add_argument("--trace", action="store_true", help="--sweep: also time whole traces (all phases, 3 runs)")
    ap.add_argument("--sparse-only", action="store_true", help="--sweep: sparse rows only")
    ap.add_argument("--diag", action="store_true", help="attention diagnostics of each workload family's dense trace")
    ap.add_argument("--fused", action="store_true", help="fused layer step: QKV projection + decode, and the projection alone")
    ap.add_argument("--policies", action="store_true", help="score-based baselines (TOVA, H2O) on the same workloads")
    ap.add_argument("--calibrated", action="store_true",
                    help="use the calibrated traces (Fig. 8 attention split) for --diag and the decode bench")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.sweep:
        run_sweep(args)
        return
    if args.diag:
        run_diag(args)
        return
    if args.fused:
        run_fused(args)
        return
    if args.policies:
        run_policies(args)
        return
    rank, ws = dist_setup()
    res = run_reference(args, rank, ws) if args.impl == "reference" else run_ours(args, rank, ws)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
