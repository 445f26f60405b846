"""Benchmark of the fused mixed-precision optimizer step on GB300.

Default workload: the 8B Llama-3-shaped parameter set (8,030,261,248 params in
291 tensors; hidden 4096, 32 layers, GQA 32q/8kv, ffn 14336, vocab 128256),
fp32 master + m + v, fp16 gradients scaled by a dynamic loss scale, AdamW
emitting the bf16 working copy and, for the 224 linear weights, e4m3fn copies
with their transposed (column-major) copies.  One step = unscale/check ->
AdamW (+bf16, +amax) -> FP8 quantization -> scale update, all resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3_8b|llama_1b|gpt2_small|fp8_sweep] [--no-e2e]
                    [--no-configs]

Prints one JSON line.  At N = 1 the default run also times, after freeing the
8B state, the GPT-2-small and 1B Llama sets and the FP8 quantizer sweep
(tensorwise, rowwise, g128), each under "configs" with its own roofline
fraction and CPU-oracle baseline; the headline keys stay on the 8B step.  Under torchrun (N > 1) every rank holds its own
parameter shard of the same size (weak scaling) and the per-step non-finite
flag is combined across ranks with an all-reduce(MAX) before the update.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HBM_FALLBACK_GBS = 6800.0
HBM_NOMINAL_GBS = 8000.0      # the HBM3e figure the target is stated against (~7.9-8 TB/s)
BF16_FALLBACK_TFLOPS = 1900.0
L2_BYTES = 129 * 2 ** 20


def profiled_traffic(kernel: str, units: int):
    """DRAM bytes per launch of `kernel` from its committed ncu capture, scaled
    by units processed; None when the kernel source changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        m = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                m.update(f.read())
        if m.hexdigest() != rec["source_sha256"]:
            return None
        return rec["dram_bytes_per_param"] * units
    except Exception:
        return None


METRIC = ("fused AMP step params/s (unscale/check + FP32-master AdamW + bf16 emit "
          "+ tensorwise FP8 e4m3fn with transposed copy)")


def workload_config(workload: str, world: int) -> dict:
    from workloads import amp_config
    cfg = amp_config(workload)
    n = sum(s.numel for s in cfg.specs)
    n8 = sum(s.numel for s in cfg.specs if s.fp8) if cfg.fp8_weights else 0
    return {"workload": f"{workload}: {n:,} params in {len(cfg.specs)} tensors, {n8:,} FP8-emitted",
            "grad_dtype": cfg.grad_dtype, "parallelism": f"dp{world} (sharded, weak)",
            "l2": "inputs larger than L2 (no flush needed)"}


def storage_desc(workload: str) -> str:
    """What the step reads and writes, from the workload's own recipe."""
    from workloads import amp_config
    cfg = amp_config(workload)
    fp8 = cfg.fp8_weights and any(s.fp8 for s in cfg.specs)
    return (f"f32 master/m/v, {cfg.grad_dtype} grads in, bf16"
            + (" + e4m3fn (+ transposed) copies out" if fp8 else " copy out"))


def adamw_traffic(delayed: bool, n_params: int, n_fp8: int):
    """DRAM bytes of the AdamW call from the committed captures: the chunked
    kernel for every parameter, or (delayed FP8) the chunked kernel for the
    plain parameters plus the tile kernel for the FP8 weights."""
    if not delayed:
        return profiled_traffic("adamw_bulk_kernel", n_params)
    a = profiled_traffic("adamw_bulk_kernel", n_params - n_fp8)
    b = profiled_traffic("adamw_fp8_tile_kernel", n_fp8)
    return None if a is None or b is None else a + b


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def host_facts() -> dict:
    """nproc and CPU model of the host the CPU baseline runs on."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"host_nproc": os.cpu_count(), "cpu_model": model or platform.machine()}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc = index, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 8:
                try:
                    rows.append((float(f[0]), float(f[1]), f[4:8]))
                except ValueError:
                    pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, v in enumerate(fl)
                          if v.lower() == "active"})
        load = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- workloads
def build_step(workload: str, device, seed: int, fp8_scaling: str = "dynamic", sr_seed=None):
    """Allocate a workload's device state; returns (step_obj, info).  sr_seed:
    the step object's own step() rounds both copies stochastically."""
    import torch

    from loss_scaling_master_gb300 import AmpOptimizerStep
    from workloads import amp_config, device_fill_normal, device_generator, tensor_sigmas

    cfg = amp_config(workload)
    gdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[cfg.grad_dtype]
    gen = device_generator(device, seed, 1)
    # flat master and gradient buffers with one view per tensor, as sharded
    # data-parallel optimizers keep them (every offset is a multiple of 8
    # elements, so every view stays 16-byte aligned)
    n_all = sum(s.numel for s in cfg.specs)
    master_flat = torch.empty(n_all, device=device)
    grads_flat = torch.empty(n_all, dtype=gdt, device=device)
    master, grads, off = [], [], 0
    sig = tensor_sigmas(cfg, seed)
    for i, s in enumerate(cfg.specs):
        master.append(device_fill_normal(master_flat[off:off + s.numel], cfg.master_sigma, gen))
        grads.append(device_fill_normal(grads_flat[off:off + s.numel],
                                        float(sig[i] * cfg.init_scale), gen))
        off += s.numel
    fp8_shapes = [(s.rows, s.cols) if s.fp8 else None for s in cfg.specs] \
        if cfg.fp8_weights else None
    step = AmpOptimizerStep(master, grads, lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2,
                            eps=cfg.eps, weight_decay=cfg.weight_decay,
                            init_scale=cfg.init_scale, growth_factor=cfg.growth_factor,
                            backoff_factor=cfg.backoff_factor,
                            growth_interval=cfg.growth_interval, fp8_shapes=fp8_shapes,
                            fp8_scaling=fp8_scaling if fp8_shapes is not None else "dynamic",
                            sr_seed=sr_seed)
    n = sum(s.numel for s in cfg.specs)
    n8 = sum(s.numel for s in cfg.specs if s.fp8) if cfg.fp8_weights else 0
    gbytes = {"f16": 2, "bf16": 2, "f32": 4}[cfg.grad_dtype]
    info = {"cfg": cfg, "params": n, "fp8_params": n8, "tensors": len(cfg.specs),
            # algorithmic bytes per step, per kernel
            "bytes_check": gbytes * n,
            "bytes_adamw": (gbytes + 12) * n + 12 * n + 2 * n,
            "bytes_quant": 4 * n8,
            "grad_bytes": gbytes * n, "grads_flat": grads_flat}
    return step, info


def run_ours(args, rank, world, device):
    import torch
    import torch.distributed as dist

    import loss_scaling_master_gb300 as A

    torch.cuda.set_device(device)
    if args.workload == "fp8_sweep":
        return run_fp8_sweep(args, rank, world, device)
    step, info = build_step(args.workload, device, seed=1234 + rank, fp8_scaling=args.fp8_scaling)
    step.max_norm = args.clip
    delayed = step.fp8_scaling == "delayed"
    if delayed and args.clip is not None:
        raise SystemExit("--clip with --fp8-scaling delayed is not supported")
    sr = args.sr_seed is not None
    if delayed:
        info["bytes_adamw"] += 2 * info["fp8_params"]       # fp8 + fp8T written in the same pass
        info["bytes_quant"] = 0
    n_params = info["params"]
    stream = torch.cuda.Stream(device=device)
    comb = None
    if world > 1:
        from loss_scaling_master_gb300.sharded import combine_found_inf, combine_grad_sumsq
        step.data_parallel = True      # the e2e leg's step() exchanges the same values

        def comb():
            combine_found_inf(step.found_inf)
            if args.clip is not None:
                combine_grad_sumsq(step.grad_sumsq)

    def one_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if args.clip is None:
            A.amp_unscale_check(step.L_g, step.scale, step.found_inf, stream=stream)
        else:
            A.amp_unscale_check_norm(step.L_g, step.scale, step.found_inf, step.grad_sumsq,
                                     stream=stream)
        if comb is not None:
            with torch.cuda.stream(stream):
                comb()
        if ev is not None:
            ev[1].record(stream)
        amax = step.amax if step.n_fp8 else None
        if delayed:
            P, F = step.delayed_groups[0]
            if sr:
                A.amp_adamw_master_step_fp8_delayed_sr(P, F, step.L_q, step.L_qt, "e4m3fn",
                                                       step.amax_history, step.hist_len,
                                                       step.amax, step.inv_scale, step.scale,
                                                       step.found_inf, step.step_count,
                                                       *step.hyper, args.sr_seed,
                                                       fp8_eps=step.fp8_eps, stream=stream)
            else:
                A.amp_adamw_master_step_fp8_delayed(P, F, step.L_q, step.L_qt, "e4m3fn",
                                                    step.amax_history, step.hist_len, step.amax,
                                                    step.inv_scale, step.scale, step.found_inf,
                                                    step.step_count, *step.hyper,
                                                    fp8_eps=step.fp8_eps, stream=stream)
        elif args.clip is None:
            if sr:
                A.amp_adamw_master_step_sr(step.L_master, step.L_m, step.L_v, step.L_g, step.L_b,
                                           step.scale, step.found_inf, step.step_count,
                                           *step.hyper, args.sr_seed, amax=amax, stream=stream)
            else:
                A.amp_adamw_master_step(step.L_master, step.L_m, step.L_v, step.L_g, step.L_b,
                                        step.scale, step.found_inf, step.step_count, *step.hyper,
                                        amax=amax, stream=stream)
        elif sr:
            A.amp_adamw_master_step_clip_sr(step.L_master, step.L_m, step.L_v, step.L_g,
                                            step.L_b, step.scale, step.found_inf,
                                            step.step_count, *step.hyper, step.grad_sumsq,
                                            args.clip, args.sr_seed, amax=amax, stream=stream)
        else:
            A.amp_adamw_master_step_clip(step.L_master, step.L_m, step.L_v, step.L_g, step.L_b,
                                         step.scale, step.found_inf, step.step_count,
                                         *step.hyper, step.grad_sumsq, args.clip, amax=amax,
                                         stream=stream)
        if ev is not None:
            ev[2].record(stream)
        if step.n_fp8 and not delayed:
            if sr:
                A.fp8_quant_tensorwise_list_sr(step.L_x8, step.L_q, step.L_qt, "e4m3fn",
                                               step.amax, step.inv_scale, args.sr_seed,
                                               step.step_count, eps=step.fp8_eps,
                                               skip_if=step.found_inf, stream=stream)
            else:
                A.fp8_quant_tensorwise_list(step.L_x8, step.L_q, step.L_qt, "e4m3fn", step.amax,
                                            step.inv_scale, eps=step.fp8_eps,
                                            skip_if=step.found_inf, stream=stream)
        if ev is not None:
            ev[3].record(stream)
        if delayed:
            A.amp_update_scale_fp8_history(step.scale, step.growth_tracker, step.found_inf,
                                           step.growth, step.backoff, step.interval, step.amax,
                                           step.amax_history, step.n_fp8, step.hist_len,
                                           stream=stream)
        else:
            A.amp_update_scale(step.scale, step.growth_tracker, step.found_inf, step.growth,
                               step.backoff, step.interval,
                               amax=step.amax if step.n_fp8 else None, n_amax=step.n_fp8,
                               stream=stream)
        if ev is not None:
            ev[4].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    st0 = step.state()
    # the clock sampler starts first, so the timed steps follow the warm-up
    # steps without an idle gap
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(args.warmup):
            one_step()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_begin.record(stream)
        for k in range(args.steps):
            one_step(evs[k])
        t_end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms_total = t_begin.elapsed_time(t_end)
    st1 = step.state()
    assert st1["step"] - st0["step"] == args.steps + args.warmup, "a step was skipped"
    k_check = [e[0].elapsed_time(e[1]) for e in evs]
    k_adamw = [e[1].elapsed_time(e[2]) for e in evs]
    k_quant = [e[2].elapsed_time(e[3]) for e in evs]
    ms_t = torch.tensor([ms_total], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(ms_t, op=dist.ReduceOp.MAX)
    ms_total = float(ms_t.item())
    ms_step = ms_total / args.steps

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, step, info, stream, world)

    if rank != 0:
        step.close()
        return None
    peak, peak_kind = measured_peaks()
    adamw_ms = statistics.mean(k_adamw)
    achieved = info["bytes_adamw"] / (adamw_ms * 1e-3) / 1e9
    total_bytes = info["bytes_check"] + info["bytes_adamw"] + info["bytes_quant"]
    line = {
        "metric": METRIC,
        "value": n_params * args.steps * world / (ms_total * 1e-3),
        "unit": "params/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "storage": storage_desc(args.workload),
        "data": "synthetic (seeded N(0,0.02) masters and seeded gradients of the workload's "
                "recipe; no trained weights)",
        "config": dict(workload_config(args.workload, world), per_step_bytes=total_bytes),
        "hbm_gbs_step": total_bytes / (ms_step * 1e-3) / 1e9,
        "grad_clip": args.clip,
        "rounding": ("stochastic (bf16 and FP8 copies)" if args.sr_seed is not None
                     else "nearest-even"),
        "fp8_scaling": step.fp8_scaling,
        "kernels_ms": {"unscale_check": statistics.mean(k_check),
                       "adamw_master_step": adamw_ms,
                       "fp8_quant_list": statistics.mean(k_quant)},
        "fp8_quant_gbs": (info["bytes_quant"] / (statistics.mean(k_quant) * 1e-3) / 1e9)
        if info["bytes_quant"] else None,
        "adamw_gbs": info["bytes_adamw"] / (statistics.mean(k_adamw) * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "amp_adamw_master_step",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "frac_of_nominal": achieved / HBM_NOMINAL_GBS,
                     "nominal_gbs": HBM_NOMINAL_GBS,
                     "bytes_per_param": info["bytes_adamw"] / n_params,
                     "traffic": adamw_traffic(delayed, n_params, info["fp8_params"]),
                     "traffic_note": "ncu dram read+write per param of a smaller launch of the "
                                     "same kernel(s), scaled by params (profiles/traffic.json)"},
        "clocks": clk.summary(),
        "gpu_launches": args.steps * step.launches_per_step,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    step.close()
    return line


def run_e2e(args, step, info, stream, world):
    """The same step through the public API, with every step's gradients
    copied from pinned host memory by the C ABI (amp_tensor_list_copy_from_host:
    one copy per tensor) and the scaler state read back, all inside the timed
    region.  Two device gradient buffers let the copy of step k+1 (on its own
    stream) overlap the update of step k."""
    import torch
    import torch.distributed as dist

    import loss_scaling_master_gb300 as A

    nbytes = info["grad_bytes"]
    bufs = [info["grads_flat"], torch.empty_like(info["grads_flat"])]
    views, off = [], 0
    for g in step.grads:
        views.append(bufs[1][off:off + g.numel()])
        off += g.numel()
    b1 = step.add_grad_buffer(views)
    from loss_scaling_master_gb300.hostmem import pinned_empty
    hbuf = pinned_empty(bufs[0].numel(), bufs[0].dtype)
    host = hbuf.tensor
    host.copy_(bufs[0])      # finite gradients of the workload's recipe
    state_host = torch.empty(4, dtype=torch.int32, pin_memory=True)   # an amp_scaler_state
    copy_stream = torch.cuda.Stream(device=step.scale.device)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    free = [torch.cuda.Event(), torch.cuda.Event()]
    for e in free:
        e.record(stream)
    host_ptrs, off = [], 0
    for g in step.grads:
        host_ptrs.append(host.data_ptr() + off * host.element_size() if g.numel() else None)
        off += g.numel()
    grad_lists = [step.grad_lists[0], step.grad_lists[b1]]
    torch.cuda.synchronize()

    copy_ev = []   # (start, end) of each timed step's host->device copy

    def e2e_step(k, timed=False):
        b = k % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(free[b])
            if timed:
                ce = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ce[0].record(copy_stream)
            A.amp_tensor_list_copy_from_host(grad_lists[b], host_ptrs, stream=copy_stream)
            if timed:
                ce[1].record(copy_stream)
                copy_ev.append(ce)
            ready[b].record(copy_stream)
        stream.wait_event(ready[b])
        step.step(stream=stream, grad_buffer=(0 if b == 0 else b1))
        free[b].record(stream)
        A.amp_read_state(step.scale, step.growth_tracker, step.step_count, step.found_inf,
                         state_host.data_ptr(), stream=stream)

    for k in range(max(2, args.warmup // 2)):
        e2e_step(k)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    copy_stream.wait_event(t0)
    for k in range(args.steps):
        e2e_step(k, timed=True)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    # Each copy's events bracket only its copies: the start event follows the
    # wait for its buffer on the copy stream, so it completes once that wait
    # is satisfied.  The copies run back to back on one stream inside the
    # timed region, so their mean (the copy stream's busy time per step)
    # cannot exceed ms_per_step.
    copy_ms = sorted(a.elapsed_time(b) for a, b in copy_ev)
    busy = sum(copy_ms) / len(copy_ms)
    del host, bufs
    hbuf.close()
    return {"value": info["params"] * args.steps * world / (ms * 1e-3), "unit": "params/s",
            "ms_per_step": ms / args.steps, "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": 16,
            "h2d_copy_ms": {"min": copy_ms[0], "mean_busy": busy, "max": copy_ms[-1]},
            "h2d_gbs_best": nbytes / copy_ms[0] / 1e6,
            "h2d_gbs_mean": nbytes / busy / 1e6,
            "api": "amp_tensor_list_copy_from_host (one H2D copy per tensor from pinned huge-page "
                   "host memory, on a copy stream, double-buffered) + AmpOptimizerStep.step() "
                   "(C-ABI calls) + amp_read_state (D2H of {scale, tracker, step, found_inf})",
            "host_huge_pages": hbuf.huge_pages}


def run_fp8_sweep(args, rank, world, device):
    """Standalone quantizer on the sweep matrices (bf16, row-major + transposed)."""
    import torch

    import loss_scaling_master_gb300 as A
    from workloads import (FP8_SWEEP_SHAPES, FP8_SWEEP_ZERO_SHAPE, device_fill_sweep,
                           device_generator)

    gen = device_generator(device, 99 + rank, 4)
    mats = []
    for (r, c) in FP8_SWEEP_SHAPES + [FP8_SWEEP_ZERO_SHAPE]:
        x = torch.empty((r, c), dtype=torch.bfloat16, device=device)
        if (r, c) == FP8_SWEEP_ZERO_SHAPE and len(mats) == len(FP8_SWEEP_SHAPES):
            x.zero_()
        else:
            device_fill_sweep(x, gen)
        mats.append(x)
    outs = [(torch.empty(x.shape, dtype=torch.uint8, device=device),
             torch.empty((x.shape[1], x.shape[0]), dtype=torch.uint8, device=device))
            for x in mats]
    inv = torch.zeros(len(mats), device=device)
    amax = torch.zeros(len(mats), device=device)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)
    fmts = ["e4m3fn", "e5m2"]
    rowwise = args.fp8_granularity == "rowwise"
    groupwise = args.fp8_granularity == "groupwise"
    if groupwise:
        G = 128
        gw = [{k: torch.empty(n, device=device) for k, n in
               (("ar", x.shape[0] * -(-x.shape[1] // G)), ("sr", x.shape[0] * -(-x.shape[1] // G)),
                ("ir", x.shape[0] * -(-x.shape[1] // G)), ("ac", x.shape[1] * -(-x.shape[0] // G)),
                ("sc", x.shape[1] * -(-x.shape[0] // G)), ("ic", x.shape[1] * -(-x.shape[0] // G)))}
              for x in mats]
    if rowwise:
        rc = [{k: torch.empty(n, device=device) for k, n in
               (("ar", x.shape[0]), ("sr", x.shape[0]), ("ir", x.shape[0]),
                ("ac", x.shape[1]), ("sc", x.shape[1]), ("ic", x.shape[1]))} for x in mats]

    def one(ev=None):
        for f in fmts:
            for i, x in enumerate(mats):
                if ev is not None:
                    ev[(f, i)][0].record(stream)
                if groupwise:
                    d = gw[i]
                    A.fp8_quant_groupwise(x, f, G, outs[i][0], outs[i][1], d["ar"], d["sr"],
                                          d["ir"], d["ac"], d["sc"], d["ic"], stream=stream)
                elif rowwise:
                    d = rc[i]
                    A.fp8_quant_rowwise(x, f, outs[i][0], outs[i][1], d["ar"], d["sr"], d["ir"],
                                        d["ac"], d["sc"], d["ic"], stream=stream)
                else:
                    A.fp8_quant_tensorwise(x, f, outs[i][0], outs[i][1], inv[i:i + 1],
                                           amax[i:i + 1], stream=stream)
                if ev is not None:
                    ev[(f, i)][1].record(stream)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    times = []
    per_call = {(f, i): [] for f in fmts for i in range(len(mats))}
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(args.steps):
            with torch.cuda.stream(stream):
                flush.fill_(1)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            one()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
    # the per-call breakdown comes from separate steps: events between the
    # calls end each call's overlap with the next one's launch, so they are
    # kept out of the timed steps above
    for _ in range(max(3, args.steps // 2)):
        with torch.cuda.stream(stream):
            flush.fill_(1)
        ev = {key: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for key in per_call}
        one(ev)
        torch.cuda.synchronize()
        for key, (e0, e1) in ev.items():
            per_call[key].append(e0.elapsed_time(e1))
    ms = statistics.mean(times)
    elems = sum(x.numel() for x in mats) * len(fmts)
    peak, kind = measured_peaks()
    # algorithmic bytes: two passes (amax, then cast) read x twice; the
    # group-wise cast reads it once (its groups lie inside one tile)
    per_elt = 4 if groupwise else 6
    gbs = per_elt * elems / (ms * 1e-3) / 1e9
    if rank != 0:
        return None
    gran = ("rowwise (per-row / per-column scales)" if rowwise else
            "group-wise (g128 along rows / along columns for the copy)" if groupwise else "tensorwise")
    return {"metric": f"FP8 {gran} quant GB/s (amax + e4m3fn/e5m2 cast + transposed copy)",
            "value": gbs * world, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "storage": "bf16 in, e4m3fn/e5m2 out",
            "data": "synthetic N(0,1) bf16 with 0.1 % of positions x100, + one all-zero matrix",
            "config": {"workload": "fp8_sweep [4096,4096],[8192,8192],[16384,5120],zero[4096,4096] "
                                   "x {e4m3fn,e5m2}", "l2": "flushed between steps"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_kind": kind, "traffic": None},
            "clocks": clk.summary(),
            "bytes_per_elt": per_elt,
            # each call's own time (CUDA events around it, in extra steps
            # after the timed ones; the first call of a step follows the L2
            # flush) and its algorithmic rate
            "per_call": {f"{'zero ' if i == len(mats) - 1 else ''}{mats[i].shape[0]}x"
                         f"{mats[i].shape[1]} {f}": {
                             "us": 1e3 * statistics.mean(v),
                             "gbs": per_elt * mats[i].numel() / (statistics.mean(v) * 1e-3) / 1e9}
                         for (f, i), v in per_call.items()},
            "gpu_launches": args.steps * len(mats) * len(fmts) * (4 if rowwise else 1 if groupwise else 3)}


# ------------------------------------------------- the other configs, 1 GPU
def _condense(line: dict) -> dict:
    keep = ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "hbm_gbs_step",
            "kernels_ms", "adamw_gbs", "bytes_per_elt", "per_call", "roofline", "clocks",
            "gpu_launches", "cpu_baseline", "storage")
    d = {k: line[k] for k in keep if k in line}
    d["workload"] = line["config"]["workload"]
    if "per_step_bytes" in line["config"]:
        d["per_step_bytes"] = line["config"]["per_step_bytes"]
    return d


def run_configs(args, device) -> dict:
    """The configurations besides the 8B set, timed on one GPU in the same
    process after the 8B state is freed: the GPT-2-small and 1B Llama
    parameter sets (each its own device-timed step line; every timed step
    updates, none is skipped) and the FP8 quantizer sweep at tensorwise,
    rowwise and group-wise (g128) granularity.  Each carries its roofline
    fraction and a CPU-oracle baseline."""
    import gc

    import torch
    out = {}
    for wl, steps in (("gpt2_small", 10), ("llama_1b", 50)):
        gc.collect()
        torch.cuda.empty_cache()
        a = argparse.Namespace(**vars(args))
        a.workload, a.steps, a.warmup = wl, steps, 3
        a.no_e2e, a.clip, a.sr_seed, a.fp8_scaling = True, None, None, "dynamic"
        a.cpu_seconds = min(args.cpu_seconds, 4.0)
        out[wl] = _condense(run_ours(a, 0, 1, device))
    for gran in ("tensorwise", "rowwise", "groupwise"):
        gc.collect()
        torch.cuda.empty_cache()
        a = argparse.Namespace(**vars(args))
        a.workload, a.fp8_granularity, a.steps, a.warmup = "fp8_sweep", gran, 30, 5
        out[f"fp8_sweep_{gran}"] = _condense(run_fp8_sweep(a, 0, 1, device))
    if not args.no_cpu_baseline:
        out["fp8_sweep_tensorwise"]["cpu_baseline"] = cpu_baseline_sweep(min(args.cpu_seconds, 4.0))
    return out


# ------------------------------------------------------------ CPU baseline
def _oracle_sample(workload: str, names):
    """Oracle state for a named subset of the workload's tensors."""
    import numpy as np

    import oracle as O
    from workloads import amp_config

    cfg = amp_config(workload if workload != "fp8_sweep" else "llama3_8b")
    specs = [s for s in cfg.specs if names(s.name)] or cfg.specs[:3]
    rng = np.random.default_rng(5)
    master = [(rng.standard_normal(s.numel, dtype=np.float32) * np.float32(0.02)) for s in specs]
    sig = 1e-4 if isinstance(cfg.grad_sigma, str) else float(cfg.grad_sigma)
    grads = [(rng.standard_normal(s.numel, dtype=np.float32) * np.float32(sig * cfg.init_scale))
             .astype(np.float16).view(np.uint16) for s in specs]
    if cfg.grad_dtype == "bf16":
        grads = [O.encode("bf16", O.decode("f16", g)) for g in grads]
    fp8_shapes = [(s.rows, s.cols) if s.fp8 else None for s in specs] if cfg.fp8_weights else None
    orc = O.AmpStepOracle(master, cfg.grad_dtype, cfg.lr, cfg.beta1, cfg.beta2, cfg.eps,
                          cfg.weight_decay, cfg.init_scale, cfg.growth_factor, cfg.backoff_factor,
                          cfg.growth_interval, fp8_shapes=fp8_shapes)
    n = sum(s.numel for s in specs)
    n8 = sum(s.numel for s in specs if s.fp8) if cfg.fp8_weights else 0
    return cfg, specs, orc, grads, n, n8


def cpu_baseline(workload: str, seconds: float):
    """The CPU oracle as it stands, single-threaded, on a bounded sample of
    the workload: layer 0 of the parameter set (all of its tensors, FP8
    copies included), timed for whole steps until ~`seconds` have passed."""
    cfg, specs, orc, grads, n, n8 = _oracle_sample(workload, lambda nm: nm.startswith(("l0.", "h0.")))
    steps, t0 = 0, time.perf_counter()
    while True:
        orc.run(grads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds or steps >= 50:
            break
    return dict({"value": n * steps / el, "unit": "params/s", "cores": 1, "kind": "oracle",
                 "sample": f"{len(specs)} tensors of {cfg.name} layer 0 ({n:,} params, {n8:,} "
                           f"FP8-emitted), {steps} full step(s) in {el:.1f} s, single-threaded "
                           f"C oracle"}, **host_facts())


def cpu_baseline_sweep(seconds: float):
    """The oracle's tensorwise quantizer (amax, fp64 scale, e4m3fn cast,
    transposed copy) on the sweep's [4096, 4096] matrix, single-threaded,
    repeated until ~`seconds` have passed; GB/s at 6 bytes per element."""
    import oracle as O
    from workloads import fp8_sweep_host
    r, c = 4096, 4096
    x = fp8_sweep_host(r, c, seed=0)
    calls, t0 = 0, time.perf_counter()
    while True:
        O.fp8_quant_tensorwise(x, "bf16", r, c, "e4m3fn", 1e-12, True)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds or calls >= 50:
            break
    return dict({"value": 6 * r * c * calls / el / 1e9, "unit": "GB/s", "cores": 1,
                 "kind": "oracle",
                 "sample": f"{calls} tensorwise e4m3fn quantizations (with the transposed copy) "
                           f"of one [4096, 4096] bf16 matrix in {el:.1f} s, single-threaded "
                           f"C oracle"}, **host_facts())


def run_reference(args, rank, world):
    """The reference arm: the pages ship no runnable code, so it is the CPU
    oracle, timed for W untimed + K timed steps on a bounded sample of the
    workload (the attention block of layer 0), on one host core."""
    if rank != 0:
        return None
    attn = ("l0.attn_norm", "l0.q", "l0.k", "l0.v", "l0.o", "l0.ffn_norm",
            "h0.ln_1.w", "h0.ln_1.b", "h0.attn.c_attn.w", "h0.attn.c_proj.w")
    cfg, specs, orc, grads, n, n8 = _oracle_sample(args.workload, lambda nm: nm in attn)
    for _ in range(args.warmup):
        orc.run(grads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.run(grads)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    sample = (f"{len(specs)} tensors of {cfg.name} layer 0 attention ({n:,} params, {n8:,} "
              f"FP8-emitted) per step, single-threaded C oracle")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "storage": storage_desc(args.workload),
            "data": "synthetic", "config": workload_config(args.workload, world),
            "cpu_baseline": dict({"value": value, "unit": "params/s", "cores": 1,
                                  "kind": "oracle", "sample": sample}, **host_facts()),
            "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "note": "the pages ship no runnable code; the reference arm is the CPU oracle"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b",
                    choices=["llama3_8b", "llama_1b", "gpt2_small", "fp8_sweep",
                             "llama3_8b_2layers"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only --workload (by default the 8B run also times the GPT-2, 1B "
                         "and FP8-sweep configurations on one GPU, under 'configs')")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--fp8-scaling", default="dynamic", choices=["dynamic", "delayed"],
                    help="FP8 weight scaling: this step's amax (a separate cast pass) or the "
                         "previous step's (cast fused into the AdamW pass)")
    ap.add_argument("--fp8-granularity", default="tensorwise",
                    choices=["tensorwise", "rowwise", "groupwise"],
                    help="scale granularity of the fp8_sweep workload")
    ap.add_argument("--sr-seed", type=int, default=None,
                    help="round the bf16 and FP8 copies stochastically (Philox4x32-10 with this "
                         "seed)")
    ap.add_argument("--clip", type=float, default=None,
                    help="also clip the unscaled gradients to this global L2 norm")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        import torch
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        line = run_ours(args, rank, world, torch.device("cuda", local))
        if (world == 1 and args.workload == "llama3_8b" and not args.no_configs
                and line is not None):
            line["configs"] = run_configs(args, torch.device("cuda", local))
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
