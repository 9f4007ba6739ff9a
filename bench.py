#!/usr/bin/env python
"""DFlash draft + verify step throughput on GB300 (steps/s, tokens/s, HBM GB/s).

One step = inject the S newest target-feature rows of every sequence into the paged
KV cache (fuse + K/V + RoPE), draft the block (all drafter layers), LM head + argmax,
verify (greedy, or temperature 1 with supplied uniforms).  The default workload is the
Qwen3-8B-shaped batch-1 drafter (context 2048, block 16, bf16).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...      # the fp64 CPU oracle on the host cores

Under torchrun each rank runs the whole workload on its own GPU (replicas, no
collective on the data path); rank 0 prints one JSON line with the job's aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft+verify steps/sec and tokens/sec; achieved HBM GB/s vs ~8 TB/s (1 GB300)"
DEFAULT_CONFIG = "qwen3-8b-shaped-b1"
# DRAM read + write bytes of one LM-head launch on this workload, from an ncu capture of
# the current kernel (None until the kernel has been captured since its last change)
LM_HEAD_TRAFFIC = 1249930312


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other workloads after the headline one")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the input-fusion variant and the speculative loop")
    ap.add_argument("--cpu-budget", type=float, default=120.0,
                    help="seconds of oracle time the reference arm may spend")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------------ clocks
class Clocks:
    """Samples nvidia-smi every 200 ms while running."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, uuid):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
               "-lms", "200"]
        if uuid:
            cmd[1:1] = ["-i", uuid]
        try:
            self.p = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[0]) for r in rows) if v is not None]
        mx = [v for v in (num(r[1]) for r in rows) if v is not None]
        reasons = sorted({self.NAMES[i] for r in rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------------ oracle
def oracle_timing(w, budget, max_steps, warmup, one_thread=False):
    """Times the fp64 oracle step of sequence 0 on the host cores (context K/V of the
    earlier positions prepared untimed).  Returns (seconds per oracle step, steps); with
    one_thread the timed steps run with BLAS limited to one thread (None when no limit
    could be applied)."""
    import numpy as np
    from oracle import run as orun
    from workload import inputs

    W = orun.host_weights(w)
    T = int(inputs.ctx_lens(w)[0])
    _, K, V = orun.context(w, W, 0, 0, T - w.block_size)
    logits = inputs.logits_noise(w, 0, 1)
    inputs.plant(w, logits, inputs.decoy_drafts(w)[:1], inputs.plant_mask(w)[:1])
    row = logits[0].float().numpy().astype(np.float64)
    u = inputs.uniforms(w)[0].numpy()
    for _ in range(min(warmup, 1)):
        orun.step_sequence(w, W, 0, (K, V), row, u)
    if one_thread:
        with blas_threads(1) as lim:
            if not lim.ok:
                return None, 0
            return oracle_timing_loop(w, W, K, V, row, u, budget, max_steps)
    return oracle_timing_loop(w, W, K, V, row, u, budget, max_steps)


def oracle_timing_loop(w, W, K, V, row, u, budget, max_steps):
    from oracle import run as orun
    times = []
    t_all = time.perf_counter()
    while len(times) < max(1, max_steps):
        t0 = time.perf_counter()
        orun.step_sequence(w, W, 0, (K, V), row, u)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > budget:
            break
    return sum(times) / len(times), len(times)


class blas_threads:
    """Limits the BLAS library numpy uses to n threads inside a with-block (through
    threadpoolctl when it is installed, else the OpenBLAS thread-count call found among
    the loaded libraries).  `ok` tells whether a limit could be applied."""

    SYMS = ("openblas_set_num_threads", "scipy_openblas_set_num_threads64_",
            "openblas_set_num_threads64_", "scipy_openblas_set_num_threads")
    GET = ("openblas_get_num_threads", "scipy_openblas_get_num_threads64_",
           "openblas_get_num_threads64_", "scipy_openblas_get_num_threads")

    def __init__(self, n):
        self.n, self.ok, self._undo = n, False, None

    def __enter__(self):
        try:
            from threadpoolctl import threadpool_limits
            self._undo = threadpool_limits(limits=self.n, user_api="blas")
            self.ok = True
            return self
        except Exception:
            pass
        import ctypes
        try:
            libs = {ln.split()[-1] for ln in open("/proc/self/maps") if "blas" in ln.lower()}
        except OSError:
            libs = set()
        for path in libs:
            try:
                lib = ctypes.CDLL(path)
            except OSError:
                continue
            for s, g in zip(self.SYMS, self.GET):
                if hasattr(lib, s) and hasattr(lib, g):
                    prev = getattr(lib, g)()
                    getattr(lib, s)(self.n)
                    self._undo = lambda f=getattr(lib, s), p=prev: f(p)
                    self.ok = True
                    return self
        return self

    def __exit__(self, *exc):
        if self._undo is None:
            return
        if callable(self._undo):
            self._undo()
        else:
            self._undo.restore_original_limits()


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


def run_reference(args):
    from workload.configs import BY_NAME
    if int(os.environ.get("RANK", "0")) != 0:
        return
    w = BY_NAME[args.config]
    t, n = oracle_timing(w, args.cpu_budget, args.steps, args.warmup)
    steps_per_s = 1.0 / (t * w.batch)
    sample = (f"{n} oracle step(s) of sequence 0 of {w.batch} (fuse+inject S rows, draft, "
              "LM head, verify; context K/V prepared untimed); value scaled to whole steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": steps_per_s, "unit": "steps/s",
        "n_gpus": args.gpus, "steps": n, "warmup": min(args.warmup, 1),
        "ms_per_step": 1e3 / steps_per_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "block": w.block_size,
                   "ctx_len": w.max_ctx, "parallelism": "host cores"},
        "cpu_baseline": {"value": steps_per_s, "unit": "steps/s", "cores": cpu_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": steps_per_s, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------ per config
def measure_config(w, steps, warmup, hbm, bf16_tf):
    """One workload timed on its own: the step in a CUDA graph (K replays between CUDA
    events), its step roofline, and each library call of an eager step timed between
    events (no programmatic overlap between calls there, so they sum to more than the
    graph step).  Returns a dict for the bench line's per_config object."""
    import torch

    from block_diffusion_drafter_concat_gb300.runner import (StepRunner, lm_head_bytes,
                                                            step_bytes, step_flops)
    r = StepRunner(w)
    r.keep_fused = False
    r.step()
    torch.cuda.synchronize()
    r.plant(r.draft.cpu())
    r.capture()
    for _ in range(max(3, warmup)):
        r.replay()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(steps):
        r.replay()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    calls = r.timed_calls(reps=3)
    if r.drafter.device_error():
        raise RuntimeError(f"device error on {w.name}")
    sb, fl = step_bytes(w), step_flops(w)
    t_roof = max(sb / (hbm * 1e9), fl / (bf16_tf * 1e12))
    lm_us = calls["lm_head_argmax"]
    lm_gbs = lm_head_bytes(w) / (lm_us * 1e-6) / 1e9
    lm_tf = 2.0 * w.rows * w.vocab * w.d_model / (lm_us * 1e-6) / 1e12
    lm_tensor = (2.0 * w.rows * w.vocab * w.d_model / lm_head_bytes(w)
                 > bf16_tf * 1e12 / (hbm * 1e9))
    out = {
        "ms_per_step": ms, "steps_per_s": 1e3 / ms, "batch": w.batch,
        "mean_emitted": float(r.n_emit.float().mean()),
        "tokens_per_s": 1e3 / ms * w.batch * float(r.n_emit.float().mean()),
        "step_roofline": {"bytes": sb, "flops": fl, "t_roof_us": t_roof * 1e6,
                          "frac": t_roof / (ms / 1e3)},
        "eager_call_us": calls,
        "lm_head": ({"bound": "tensor", "achieved": lm_tf, "unit": "TFLOP/s",
                     "frac": lm_tf / bf16_tf, "us_per_launch": lm_us} if lm_tensor else
                    {"bound": "hbm", "achieved": lm_gbs, "unit": "GB/s", "frac": lm_gbs / hbm,
                     "us_per_launch": lm_us}),
        "launches_per_step": r.launches,
        "steps": steps,
    }
    del r
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------ NEXT rows
def measure_input_fusion(w, steps, warmup, hbm, bf16_tf):
    """The input-fusion variant of the headline workload: its graph step beside the KV
    injection step, and the context prefill of sequence 0 both ways."""
    import torch

    from block_diffusion_drafter_concat_gb300.runner import StepRunner, step_bytes
    from workload import inputs as winputs
    r = StepRunner(w, variant="input")
    r.step()
    torch.cuda.synchronize()
    r.plant(r.draft.cpu())
    r.capture()
    for _ in range(max(3, warmup)):
        r.replay()
    st = torch.cuda.current_stream()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    torch.cuda.synchronize()
    e[0].record(st)
    for _ in range(steps):
        r.replay()
    e[1].record(st)
    torch.cuda.synchronize()
    ms = e[0].elapsed_time(e[1]) / steps
    # prefill of sequence 0's context through the layer stack (chunks of S rows)
    S = w.block_size
    T = int(r.lens[0]) - S
    x = torch.empty(w.rows, w.fuse_in, dtype=r.dt, device="cuda")
    chunks = list(range(0, T, S))
    xs = [winputs.ctx_hidden(w, 0, c0, c0 + S, "cuda") for c0 in chunks]
    ctx = [torch.tensor([c0] * w.batch, dtype=torch.int32, device="cuda") for c0 in chunks]
    torch.cuda.synchronize()
    e[2].record(st)
    for xc, cc in zip(xs, ctx):
        x[:S].copy_(xc)
        r.drafter.inject_inputs(x, cc, r.page_table, r.cache, r.ws)
    e[3].record(st)
    torch.cuda.synchronize()
    pf_us = e[2].elapsed_time(e[3]) * 1e3
    if r.drafter.device_error():
        raise RuntimeError("device error in the input-fusion variant")
    out = {"ms_per_step": ms, "steps_per_s": 1e3 / ms,
           "step_hbm_gbs": step_bytes(w) / (ms / 1e3) / 1e9,
           "prefill": {"rows": T, "us": pf_us, "chunks": len(chunks),
                       "note": "context of sequence 0 through the layer stack, causal "
                               "chunks of S rows (input fusion), timed with the copies "
                               "of the chunk inputs"},
           "note": "fused features as the drafter's input: the S new context rows run "
                   "through every layer (causal) instead of being injected as K/V"}
    del r
    torch.cuda.empty_cache()
    return out


def measure_spec_loop(sw, steps, warmup):
    """The greedy speculative loop with a random causal target: prefill (untimed), a
    few eager steps, then one step captured in a CUDA graph and replayed; tokens/s from
    the tokens the timed steps emitted (planted agreement, see the workload)."""
    import torch

    from block_diffusion_drafter_concat_gb300.spec import SpecRunner
    steps = max(1, min(steps, sw.steps - warmup - 1))
    r = SpecRunner(sw)
    r.prefill()
    for _ in range(warmup):
        r.step()
    torch.cuda.synchronize()
    n0 = int(r.n_generated.sum())
    r.capture()
    st = torch.cuda.current_stream()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    torch.cuda.synchronize()
    e[0].record(st)
    for _ in range(steps):
        r.replay()
    e[1].record(st)
    torch.cuda.synchronize()
    ms = e[0].elapsed_time(e[1]) / steps
    emitted = int(r.n_generated.sum()) - n0
    if r.drafter.device_error() or r.target.device_error():
        raise RuntimeError("device error in the speculative loop")
    # one target pass over a block alone (what one greedy token costs without drafting
    # at batch 1, where the pass streams the target's weights whatever its row count)
    w = sw.drafter
    ids = torch.zeros(w.batch, w.block_size, dtype=torch.int32, device="cuda")
    ctx = r.ctx_lens.clone()
    for _ in range(2):
        r.target.target_forward(ids, ctx, r.table, r.tcache, r.tws)
    torch.cuda.synchronize()
    e[2].record(st)
    for _ in range(5):
        r.target.target_forward(ids, ctx, r.table, r.tcache, r.tws)
    e[3].record(st)
    torch.cuda.synchronize()
    t_pass = e[2].elapsed_time(e[3]) / 5
    tok_s = emitted / (ms * steps / 1e3)
    out = {"workload": sw.name, "target_layers": sw.target_layers,
           "tap_layers": list(sw.tap_layers), "batch": w.batch, "prompt": sw.prompt_len,
           "steps": steps, "ms_per_step": ms, "tokens_per_s": tok_s,
           "mean_emitted": emitted / (steps * w.batch), "plant_p": sw.plant_p,
           "launches_per_step": r.launches,
           "target_pass_ms": t_pass,
           "tokens_per_s_one_target_pass_per_token": w.batch * 1e3 / t_pass,
           "note": "draft -> target pass -> verify -> commit -> inject in one CUDA graph per "
                   "step; random weights, so acceptance comes from planted agreement"}
    del r
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------ ours
def run_ours(args):
    import torch
    import torch.distributed as dist

    from block_diffusion_drafter_concat_gb300 import build
    from block_diffusion_drafter_concat_gb300 import replicas
    from workload.configs import BY_NAME

    build.build()
    from block_diffusion_drafter_concat_gb300.runner import (PREFILL_CHUNK, StepRunner,
                                                            lm_head_bytes,
                                                            step_bytes, step_flops)

    rep = replicas.from_env()
    world, rank, local = rep.world, rep.rank, rep.local
    torch.cuda.set_device(local)
    if rep.distributed:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        replicas.barrier(rep)

    def max_over_ranks(t):
        return replicas.max_over_ranks(rep, t, device="cuda")

    w = BY_NAME[args.config]
    r = StepRunner(replicas.shard(w, rank))
    r.keep_fused = False   # the fused rows are an optional output the step does not need
    # one eager step, then plant the verify logits' agreement with this step's drafts
    r.step()
    torch.cuda.synchronize()
    r.plant(r.draft.cpu())
    r.capture()
    for _ in range(args.warmup):
        r.replay()
    torch.cuda.synchronize()
    if r.drafter.device_error():
        raise RuntimeError("device error during warm-up")

    uuid = None
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    st = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]

    # ---- device-resident inputs: K graph replays, an event between consecutive replays
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    torch.cuda.synchronize()
    clk = Clocks(uuid)
    ev[0].record(st)
    step_ev[0].record(st)
    for i in range(args.steps):
        r.replay()
        step_ev[i + 1].record(st)
    ev[1].record(st)
    torch.cuda.synchronize()
    clocks = clk.stop()
    barrier()
    t = max_over_ranks(ev[0].elapsed_time(ev[1]) / 1e3)
    per_step = sorted(step_ev[i].elapsed_time(step_ev[i + 1]) * 1e3 for i in range(args.steps))

    def pct(q):
        return per_step[min(len(per_step) - 1, int(q * len(per_step)))]

    # ---- the same steps with L2 flushed before each one (256 MB written, untimed)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    k_fl = max(3, min(20, args.steps))
    fl_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * k_fl)]
    for i in range(k_fl):
        flush.zero_()
        fl_ev[2 * i].record(st)
        r.replay()
        fl_ev[2 * i + 1].record(st)
    torch.cuda.synchronize()
    fl_us = sorted(fl_ev[2 * i].elapsed_time(fl_ev[2 * i + 1]) * 1e3 for i in range(k_fl))
    del flush
    mean_emit = float(r.n_emit.float().mean())
    value = replicas.aggregate(args.steps, rep, t)
    ms = t / args.steps * 1e3

    # ---- end to end through the public API: pinned host inputs in, results out
    x_h = r.x_step.cpu().pin_memory()
    lg_h = r.logits.cpu().pin_memory()
    out_h = torch.empty(r.out_tokens.shape, dtype=torch.int32).pin_memory()
    ne_h = torch.empty(r.n_emit.shape, dtype=torch.int32).pin_memory()
    k_e2e = max(1, args.steps // 2)
    barrier()
    torch.cuda.synchronize()
    ev[2].record(st)
    for _ in range(k_e2e):
        r.x_step.copy_(x_h, non_blocking=True)
        r.logits.copy_(lg_h, non_blocking=True)
        r.replay()
        out_h.copy_(r.out_tokens, non_blocking=True)
        ne_h.copy_(r.n_emit, non_blocking=True)
        st.synchronize()
    ev[3].record(st)
    torch.cuda.synchronize()
    te = max_over_ranks(ev[2].elapsed_time(ev[3]) / 1e3)
    h2d = x_h.numel() * x_h.element_size() + lg_h.numel() * lg_h.element_size()
    d2h = (out_h.numel() + ne_h.numel()) * 4

    # ---- dominant kernel: the LM head (weight-streaming GEMM + argmax epilogue)
    g = torch.cuda.CUDAGraph()
    s2 = torch.cuda.Stream()
    s2.wait_stream(st)
    with torch.cuda.stream(s2):
        r.drafter.lm_head_argmax(r.hidden, r.draft.view(-1), r.ws, r.dmax, None, 1.0)
    st.wait_stream(s2)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        r.drafter.lm_head_argmax(r.hidden, r.draft.view(-1), r.ws, r.dmax, None, 1.0)
    for _ in range(3):
        g.replay()
    k_lm = 50
    torch.cuda.synchronize()
    ev[4].record(st)
    for _ in range(k_lm):
        g.replay()
    ev[5].record(st)
    torch.cuda.synchronize()
    t_lm = ev[4].elapsed_time(ev[5]) / 1e3 / k_lm
    if r.drafter.device_error():
        raise RuntimeError("device error during the timed region")

    # ---- context prefill by injection: fuse + K/V of sequence 0's context (one chunk)
    from workload import inputs as winputs
    rows_pf = min(int(r.lens[0]) - w.block_size, PREFILL_CHUNK)
    x_pf = winputs.ctx_hidden(r.w, 0, 0, rows_pf, "cuda")
    p_pf = torch.arange(0, rows_pf)
    s_pf = winputs.slots_for(r.w, r.table_host, 0, p_pf).to(torch.int32).cuda()
    p_pf = p_pf.to(torch.int32).cuda()
    for _ in range(2):
        r.drafter.inject_kv(p_pf, s_pf, r.cache, r.ws, x_cat=x_pf)
    k_pf = 5
    torch.cuda.synchronize()
    ev[4].record(st)
    for _ in range(k_pf):
        r.drafter.inject_kv(p_pf, s_pf, r.cache, r.ws, x_cat=x_pf)
    ev[5].record(st)
    torch.cuda.synchronize()
    t_pf = ev[4].elapsed_time(ev[5]) / 1e3 / k_pf
    pf_flops = 2.0 * rows_pf * (w.fuse_in * w.d_model + w.n_layers * 2 * w.kv_width * w.d_model)
    if r.drafter.device_error():
        raise RuntimeError("device error during the prefill timing")

    hbm, bf16_tf, src = peaks()
    sb, fl = step_bytes(w), step_flops(w)
    t_roof = max(sb / (hbm * 1e9), fl / (bf16_tf * 1e12))
    lm_gbs = lm_head_bytes(w) / t_lm / 1e9
    # the LM head is a contraction of `rows` hidden rows with the whole head: HBM-bound
    # below the ridge intensity (peak FLOP/s over peak bytes/s), tensor-bound above it
    lm_flops = 2.0 * w.rows * w.vocab * w.d_model
    lm_tensor = lm_flops / lm_head_bytes(w) > bf16_tf * 1e12 / (hbm * 1e9)
    lm_kind = ("argmax finished in the projection (packed keys)"
               if w.rows <= 128 and w.temperature == 0 and w.dtype == "bf16" else
               "per-tile argmax partials + reduction launch")
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "block": w.block_size,
                   "ctx_len": w.max_ctx, "d_model": w.d_model, "layers": w.n_layers,
                   "vocab": w.vocab, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({sb / 1e9:.2f} GB streamed per step)",
                   "graph": "one CUDA graph per step, programmatic dependent launch"},
        "tokens_per_s": value * w.batch * mean_emit,
        "mean_emitted": mean_emit,
        "step_hbm_gbs": sb / (ms / 1e3) / 1e9,
        "step_roofline": {"bytes": sb, "flops": fl, "t_roof_us": t_roof * 1e6,
                          "frac": t_roof / (ms / 1e3), "peak_gbs": hbm, "peak_src": src},
        "roofline": ({"kernel": f"LM-head projection, {lm_kind}",
                      "bound": "tensor", "achieved": lm_flops / t_lm / 1e12, "peak": bf16_tf,
                      "unit": "TFLOP/s", "frac": lm_flops / t_lm / 1e12 / bf16_tf,
                      "traffic": None, "peak_src": src, "us_per_launch": t_lm * 1e6}
                     if lm_tensor else
                     {"kernel": f"LM-head projection, {lm_kind}",
                      "bound": "hbm", "achieved": lm_gbs, "peak": hbm, "unit": "GB/s",
                      "frac": lm_gbs / hbm,
                      "traffic": LM_HEAD_TRAFFIC if w.name == DEFAULT_CONFIG else None,
                      "peak_src": src, "us_per_launch": t_lm * 1e6}),
        "e2e": {"value": replicas.aggregate(k_e2e, rep, te), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "step_us": {"median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9)},
        "l2_flushed": {"ms_per_step": statistics.median(fl_us) / 1e3,
                       "value": 1e6 / statistics.median(fl_us), "unit": "steps/s",
                       "note": f"256 MB written before each of {k_fl} timed steps"},
        "prefill": {"rows": rows_pf, "us": t_pf * 1e6, "rows_per_s": rows_pf / t_pf,
                    "tflops": pf_flops / t_pf / 1e12,
                    "note": "fuse + K/V injection of sequence 0's context, all layers"},
        "gpu_launches": r.launches * args.steps,
        "launches_per_step": r.launches,
        "clocks": clocks,
    }
    if not args.no_per_config:
        from workload.configs import ALL
        per = {w.name: {"headline": True, "ms_per_step": ms,
                        "step_roofline": {"frac": t_roof / (ms / 1e3)}}}
        for wo in ALL:
            if wo.name == w.name:
                continue
            per[wo.name] = measure_config(replicas.shard(wo, rank), min(args.steps, 30),
                                          args.warmup, hbm, bf16_tf)
        line["per_config"] = per
    if not args.no_next and w.name == DEFAULT_CONFIG:
        from workload.configs import SPEC_QWEN3_8B
        line["input_fusion"] = measure_input_fusion(replicas.shard(w, rank), min(args.steps, 50),
                                                    args.warmup, hbm, bf16_tf)
        line["input_fusion"]["kv_injection_ms_per_step"] = ms
        line["spec_loop"] = measure_spec_loop(SPEC_QWEN3_8B, args.steps, 3)
        from workload.configs import FP8
        f8 = measure_config(replicas.shard(FP8[w.name + "-fp8"], rank), min(args.steps, 50),
                            args.warmup, hbm, bf16_tf)
        f8["note"] = ("the same step with FP8 e4m3 projection weights (per-row power-of-two "
                      "scales; activations and the rounding points as in bf16); roofline "
                      "on the FP8 step's own bytes")
        f8["bf16_ms_per_step"] = ms
        line["fp8_weights"] = f8
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tc, n = oracle_timing(w, 30.0, 3, 1)
        line["cpu_baseline"] = {
            "value": 1.0 / (tc * w.batch), "unit": "steps/s", "cores": cpu_threads(),
            "kind": "oracle",
            "sample": f"{n} fp64 oracle step(s) of sequence 0 of {w.batch}, context K/V "
                      "prepared untimed; scaled to whole steps"}
        # the same oracle with BLAS on one thread, on the tiny and the headline workload
        one = {}
        for wo in (BY_NAME["tiny-f32"], w):
            t1, n1 = oracle_timing(wo, 30.0, 3 if wo.name == "tiny-f32" else 1, 1,
                                   one_thread=True)
            one[wo.name] = (None if t1 is None else
                            {"value": 1.0 / (t1 * wo.batch), "unit": "steps/s", "cores": 1,
                             "sample": f"{n1} oracle step(s) of sequence 0"})
        line["cpu_baseline"]["one_thread"] = one
    if rank == 0:
        print(json.dumps(line), flush=True)
    if rep.distributed:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
