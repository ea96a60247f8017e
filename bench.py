"""Benchmark of the blockwise-FP8 ZeRO-1 optimizer step on one GB300.

One step = one pass of the whole hot path over the shard, through the C-ABI:
fold the row-major FP32 grads into blocks -> global grad norm + inf flag ->
fused unscale + clip + AdamW + per-block E4M3 quantise -> unfold the codes
into the row-major FP8 weights -> host reads found_inf and updates the loss
scale.  Workload (default): 32 experts x gate_up [7168,4096] + down [2048,7168]
(86016 blocks, 1.41 G padded elements, ~31 GB resident), one DP rank owning the
whole buffer.  Inputs are larger than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs the same
single-GPU workload as an independent replica; the timing is the max over
ranks and ``value`` counts the elements of all ranks.  ``--impl reference``
times the CPU oracle on a bounded sample of the same workload.
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

METRIC = "fp8z1_step elements/s and achieved HBM GB/s (fraction of ~8 TB/s) per shard, 1 GB300"
# bytes the step must move per real element: read grad, master, m, v (16) +
# write master, m, v (12) + write the E4M3 code (1); plus 4 per block (scale).
# The padding of grad / master / m / v is zero and stays zero, and is not moved;
# a folded code shard also gets its padding codes (1 byte per padded element).
STEP_BYTES_PER_ELEM = 29
STEP_BYTES_PER_BLOCK = 4
FALLBACK_HBM_GBS = 6800.0


def _peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _ncu_traffic():
    """Per-launch DRAM bytes of the step kernel from the committed ncu summary."""
    p = os.path.join(ROOT, "profiles", "step_kernel_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d
    except Exception:
        return None


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's ``x`` (the slowest rank sets the time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, steps: int, seconds: float) -> float:
    """Units processed by all ranks per second of the slowest rank."""
    return world * units_per_rank * steps / seconds


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def _workload(args, synth):
    """The named workload, cut to its first --experts experts of each 3-D
    param and/or its first --params params when asked (smaller cases)."""
    w = synth.workload(args.workload, dp=1, rank=0)
    shapes = w.shapes
    if args.experts:
        shapes = [(min(e, args.experts), r, c) for e, r, c in shapes]
    if args.params:
        shapes = shapes[:args.params]
    return w if shapes == w.shapes else synth.workload(args.workload, dp=1, rank=0, shapes=shapes)


def _config(args, shapes, dp, shard_rank, b0, b1, n_real, world) -> dict:
    """The workload the line measures; both arms report this same record."""
    whole = dp == 1
    return {
        "workload": _workload_label(args, shapes),
        "blocks": b1 - b0, "elems_padded": (b1 - b0) * 16384, "elems_real": n_real,
        "dp": "whole buffer (1 rank)" if whole else
              f"rank {shard_rank} of {dp}: blocks [{b0}, {b1}) (this rank's norm partial; no all-reduce on one GPU)",
        "parallelism": f"replicas{world}" if world > 1 else "single",
        "l2": _l2_note(b1 - b0, n_real),
        "value_counts": "padded elements per second through the whole step",
    }


def _l2_note(nblk, n_real) -> str:
    """How the timed steps avoid L2 reuse: the state a fused step touches
    (master / m / v folded, grads and FP8 weights row-major) against L2."""
    gb = (12 * nblk * 16384 + 5 * (n_real or nblk * 16384)) / 1e9
    if gb > 0.129 * 4:
        return f"inputs larger than L2 (~{gb:.0f} GB resident per step), no flush"
    return f"inputs ({gb * 1e3:.1f} MB) fit in L2: a latency-bound case, not a bandwidth figure"


def _time_layout_build(F, shapes, dp, reps=3):
    """Host wall time of the one-time layout build (block table, run table,
    shard ranges) and of the build plus its upload to the device; medians."""
    host, full = [], []
    for _ in range(reps):
        t = time.perf_counter()
        L = F.fp8z1_build_layout(shapes, dp_size=dp, host_only=True)
        host.append((time.perf_counter() - t) * 1e3)
        del L
        t = time.perf_counter()
        L = F.fp8z1_build_layout(shapes, dp_size=dp)
        full.append((time.perf_counter() - t) * 1e3)
        del L
    return {"host": statistics.median(host), "host_and_upload": statistics.median(full)}


def _workload_label(args, shapes) -> str:
    cut = "".join([f"[{args.experts} experts]" if args.experts else "",
                   f"[first {args.params} params]" if args.params else ""])
    if len(shapes) <= 8:
        body = " + ".join(f"{e}x[{r},{c}]" for e, r, c in shapes)
    else:
        body = f"{len(shapes)} params, " + " + ".join(f"{e}x[{r},{c}]" for e, r, c in shapes[:3]) + " + ..."
    return f"{args.workload}{cut}: {body}"


def bench_ours(args, rank, world, dist):
    import torch

    from blockwise_fp8_zero_fold_gb300 import build as fp8build
    from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
    from blockwise_fp8_zero_fold_gb300 import synth
    from blockwise_fp8_zero_fold_gb300.optimizer import ShardOptimizer

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fp8build.build()
    if dist is not None:
        dist.barrier()
    F.lib()

    w = _workload(args, synth)
    dp, shard_rank = (int(x) for x in args.shard.split(":")) if args.shard else (1, 0)
    opt = ShardOptimizer(w.shapes, dp_size=dp, rank=shard_rank, device=dev, loss_scale=w.loss_scale,
                         growth_interval=w.growth_interval,
                         **{k: v for k, v in w.hp().items() if k != "loss_scale"})
    for kind, buf in (("master", None), ("m", None), ("v", None)):
        rm = synth.make_state(w, kind, dev)
        opt.fold_into(rm, {"master": opt.master, "m": opt.m, "v": opt.v}[kind])
        del rm
    grads = synth.make_grads(w, 1, dev)
    fp8 = [torch.zeros(s, dtype=torch.uint8, device=dev) for s in w.shapes]
    torch.cuda.synchronize()
    layout_ms = _time_layout_build(F, w.shapes, dp)
    stream = torch.cuda.current_stream()
    # the shard's blocks, padded elements and real elements (whole buffer: all)
    nblk = opt.b1 - opt.b0
    n_pad = nblk * F.BLOCK_ELEMS
    lut = F.fp8z1_copy_lut(opt.layout)[opt.b0:opt.b1]
    n_real = int((lut["rows_real"].astype("int64") * lut["cols_real"].astype("int64")).sum())
    whole = (opt.b0, opt.b1) == (0, opt.nblk)
    b0, b1 = opt.b0, opt.b1

    def stages(path):
        """The kernels of one step on ``path``, as (label, launch) pairs."""
        def norm_fused():
            F.fp8z1_norm_reset(opt.sumsq, opt.found_inf)
            F.fp8z1_fold_norm(opt.layout, gptrs, None, opt.b0, opt.b1, opt.sumsq, opt.found_inf)

        def step_fused():
            hp = F.make_hp(step=opt.scaler.step + 1, loss_scale=opt.scaler.scale, **opt.hp)
            F.fp8z1_step_fused(opt.layout, hp, d_grad_params=gptrs, master_shard=opt.master,
                               m_shard=opt.m, v_shard=opt.v, d_fp8_params=fptrs,
                               scale_shard=opt.scales, b0=opt.b0, b1=opt.b1, d_sumsq=opt.sumsq,
                               d_found_inf=opt.found_inf)

        def fold():
            F.fp8z1_fold(opt.layout, gptrs, gbuf, 4, opt.b0, opt.b1)

        def norm():
            F.fp8z1_norm_reset(opt.sumsq, opt.found_inf)
            F.fp8z1_grad_norm(opt.layout, gbuf, opt.b0, opt.b1, opt.sumsq, opt.found_inf)

        def step():
            hp = F.make_hp(step=opt.scaler.step + 1, loss_scale=opt.scaler.scale, **opt.hp)
            F.fp8z1_step(opt.layout, hp, gbuf, opt.master, opt.m, opt.v, opt.codes, opt.scales,
                         opt.b0, opt.b1, opt.sumsq, opt.found_inf)

        def unfold():
            F.fp8z1_unfold(opt.layout, opt.codes, fptrs, 1, opt.b0, opt.b1)

        if path == "fused":
            return [("fold_norm", norm_fused), ("step", step_fused)]
        return [("fold", fold), ("norm", norm), ("step", step), ("unfold", unfold)]

    def run_steps(path, k, events=None):
        skipped = 0
        if path == "fused" and args.pipeline:
            # each step enqueued before the previous one's found_inf is read:
            # the kernel picks t and S by that flag, the host reads it a step late
            for i in range(k):
                ev = None if events is None else {"norm": events["fold_norm"][i], "step": events["step"][i]}
                skipped += sum(opt.launch_step_async(gptrs, fptrs, stream, ev))
            return skipped + sum(opt.drain())
        for i in range(k):
            for name, fn in stages(path):
                if events is not None:
                    events[name][i][0].record(stream)
                fn()
                if events is not None:
                    events[name][i][1].record(stream)
            skipped += opt.finish_step()  # host reads found_inf (a10)
        return skipped

    def timed(path, k):
        names = [n for n, _ in stages(path)]
        ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(k)] for n in names}
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("timed")
        n0 = F.fp8z1_kernel_launches()
        t0.record(stream)
        sk = run_steps(path, k, ev)
        t1.record(stream)
        launches = F.fp8z1_kernel_launches() - n0
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        ms = max_over_ranks(t0.elapsed_time(t1), dist, dev)
        kern = {n: statistics.mean(a.elapsed_time(b) for a, b in ev[n]) for n in names}
        kern_med = {n: statistics.median(a.elapsed_time(b) for a, b in ev[n]) for n in names}
        return ms, kern, sk, launches, kern_med

    gptrs = opt._ptrs(grads)
    fptrs = opt._ptrs(fp8)
    gbuf = torch.empty(opt.master.numel(), dtype=torch.float32, device=dev) if args.path == "unfused" \
        or args.compare else None

    # warm-up, then the timed region with clocks sampled during it
    run_steps(args.path, args.warmup)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    elapsed_ms, kern, skipped, launches, kern_med = timed(args.path, args.steps)
    clk = clocks.stop()
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_rate(n_pad, world, args.steps, elapsed_ms / 1e3)
    other = None
    if args.compare:
        alt = "unfused" if args.path == "fused" else "fused"
        run_steps(alt, 2)
        a_ms, a_kern, _, _, _ = timed(alt, max(3, args.steps // 4))
        other = {"path": alt, "ms_per_step": a_ms / max(3, args.steps // 4), "kernels_ms": a_kern}
    if gbuf is not None:
        del gbuf

    peak, peak_kind = _peak_hbm()
    # algorithmic bytes of the dominant kernel (the step): grads read and
    # master/m/v read and written on the real elements, one code byte per real
    # (row-major codes) or padded (folded codes) element
    if args.path == "fused":
        step_bytes = STEP_BYTES_PER_ELEM * n_real + STEP_BYTES_PER_BLOCK * nblk
        gbs = {"fold_norm": 4 * n_real / kern["fold_norm"] / 1e6}
    else:
        step_bytes = (STEP_BYTES_PER_ELEM - 1) * n_real + 1 * n_pad + STEP_BYTES_PER_BLOCK * nblk
        gbs = {"fold": 4 * (n_real + n_pad) / kern["fold"] / 1e6, "norm": 4 * n_pad / kern["norm"] / 1e6,
               "unfold": 1 * (n_real + n_pad) / kern["unfold"] / 1e6}
    achieved = step_bytes / (kern["step"] / 1e3) / 1e9
    gbs["step"] = achieved
    tr = _ncu_traffic()
    traffic = None
    traffic_basis = None
    if tr and tr.get("workload") == args.workload and tr.get("path") == args.path and \
            bool(tr.get("pipelined")) == bool(args.pipeline and args.path == "fused") and \
            tr.get("source_sha") == _step_source_sha() and not args.experts and not args.params and whole:
        traffic = tr.get("bytes_per_launch")
        traffic_basis = (f"extrapolated: ncu DRAM read + write of {tr.get('captured_on')}, "
                         f"scaled {tr.get('scale')}")

    # bf16 fold / unfold of the weights over the shard (2-byte elements)
    bf16 = None
    if args.bf16_fold:
        wb = [torch.empty(sh, dtype=torch.bfloat16, device=dev).normal_(0, 0.02) for sh in w.shapes]
        folded = torch.empty(n_pad, dtype=torch.bfloat16, device=dev)
        bptrs = opt._ptrs(wb)
        fold_b = lambda: F.fp8z1_fold(opt.layout, bptrs, folded, 2, opt.b0, opt.b1)  # noqa: E731
        unfold_b = lambda: F.fp8z1_unfold(opt.layout, folded, bptrs, 2, opt.b0, opt.b1)  # noqa: E731
        bf16 = {}
        for name, fn in (("fold", fold_b), ("unfold", unfold_b)):
            for _ in range(3):
                fn()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.bf16_fold)]
            for a, b in evs:
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
            bf16[name + "_ms"] = ms
            bf16[name + "_gbs"] = 2 * (n_real + n_pad) / ms / 1e6
        bf16["bytes_per_launch"] = 2 * (n_real + n_pad)
        del wb, folded

    # the fused step with the per-block quantisation monitors (underflow count
    # and cosine distortion), and the host-side greedy param-wise split
    monitors = None
    if args.monitors:
        bcos = torch.empty(nblk, dtype=torch.float32, device=dev)
        bund = torch.empty(nblk, dtype=torch.int32, device=dev)

        def step_mon():
            hp = F.make_hp(step=opt.scaler.step + 1, loss_scale=opt.scaler.scale, **opt.hp)
            F.fp8z1_step_fused(opt.layout, hp, d_grad_params=gptrs, master_shard=opt.master,
                               m_shard=opt.m, v_shard=opt.v, d_fp8_params=fptrs,
                               scale_shard=opt.scales, block_cos=bcos, block_underflow=bund,
                               b0=opt.b0, b1=opt.b1, d_sumsq=opt.sumsq, d_found_inf=opt.found_inf)

        for _ in range(3):
            step_mon()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.monitors)]
        for a, b in evs:
            a.record(stream)
            step_mon()
            b.record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        t = time.perf_counter()
        F.fp8z1_paramwise_split(w.shapes, max(dp, 8))
        split_ms = (time.perf_counter() - t) * 1e3
        monitors = {"step_ms": ms, "step_gbs": (step_bytes + 8 * nblk) / ms / 1e6,
                    "bytes_per_launch": step_bytes + 8 * nblk,
                    "paramwise_split_ms": split_ms, "paramwise_split_dp": max(dp, 8)}
        del bcos, bund

    # e2e: the same step through the public API, grads from pinned host memory
    # and the FP8 weights + scales + found flag read back every step
    e2e = None
    if args.e2e_steps > 0 and whole:
        # every rank pins its own host buffers (7 GB for MoE): all ranks go on,
        # or all report e2e unavailable, so none waits at a barrier alone
        why = ""
        try:
            hgrads = [torch.empty(s, dtype=torch.float32, pin_memory=True) for s in w.shapes]
            hfp8 = [torch.empty(s, dtype=torch.uint8, pin_memory=True) for s in w.shapes]
            hscales = torch.empty(nblk, dtype=torch.float32, pin_memory=True)
        except RuntimeError as exc:
            why = str(exc).strip().splitlines()[0][:200] if str(exc).strip() else type(exc).__name__
            hgrads = hfp8 = hscales = None
        ok = torch.tensor([0 if why else 1], dtype=torch.int32, device=dev)
        if dist is not None:
            dist.all_reduce(ok, op=dist.ReduceOp.MIN)
        if not int(ok.item()):
            e2e = {"value": None, "unit": "elem/s",
                   "unavailable": "pinned host buffers could not be allocated" + (f": {why}" if why else " on another rank")}
    if e2e is None and args.e2e_steps > 0 and whole:
        for h, d in zip(hgrads, grads):
            h.copy_(d)
        h2d = sum(h.numel() * 4 for h in hgrads)
        d2h = sum(h.numel() for h in hfp8) + nblk * 4 + 4

        def e2e_step(wait):
            # the public API's host path: chunked copies overlapped with the norm
            # and the update (ShardOptimizer.step_from_host); without waiting,
            # the next step's grads go in while this step's FP8 weights come out
            return opt.step_from_host(hgrads, hfp8, hscales, grads=grads, fp8_params=fp8, wait=wait)

        e2e_step(True)
        # the host link is shared with the machine's other tenants: each form
        # runs e2e_reps times, the two forms alternating, and the medians count
        sync_ms, pipe_ms = [], []
        for _ in range(max(1, args.e2e_reps)):
            if dist is not None:
                dist.barrier()
            t0 = time.perf_counter()
            for _ in range(args.e2e_steps):
                e2e_step(True)
            sync_ms.append(max_over_ranks(time.perf_counter() - t0, dist, dev) / args.e2e_steps * 1e3)
            if dist is not None:
                dist.barrier()
            t0 = time.perf_counter()
            for _ in range(args.e2e_steps):
                e2e_step(False)
            opt.finish_host_step()
            pipe_ms.append(max_over_ranks(time.perf_counter() - t0, dist, dev) / args.e2e_steps * 1e3)
        ms = statistics.median(pipe_ms)
        e2e = {"value": whole_job_rate(n_pad, world, 1, ms / 1e3), "unit": "elem/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ms, "steps": args.e2e_steps, "reps": len(pipe_ms),
               "mode": "steps enqueued back to back (step_from_host wait=False), then finish_host_step; "
                       "median of the repetitions",
               "ms_per_step_reps": pipe_ms,
               "ms_per_step_one_at_a_time": statistics.median(sync_ms),
               "ms_per_step_one_at_a_time_reps": sync_ms}
        del hgrads, hfp8

    # the other configurations, each a few steps of the same loop, after the
    # headline's timed region (its buffers freed first)
    others = None
    if args.other_workloads not in ("", "none") and not args.experts and not args.params:
        del opt, grads, fp8, gptrs, fptrs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        others = [other_workload_mx(spec[3:], args.other_steps, dev, dist, peak) if spec.startswith("mx:")
                  else other_workload(spec, args.other_steps, dev, dist, peak)
                  for spec in args.other_workloads.split(",") if spec]

    out = {
        "metric": METRIC,
        "value": value,
        "unit": "elem/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,s) grads/master/moments as the workload states)",
        "config": _config(args, w.shapes, dp, shard_rank, b0, b1, n_real, world),
        "gpu_launches": launches,
        "path": args.path,
        "pipelined": bool(args.pipeline and args.path == "fused"),
        "kernels_ms": kern,
        "kernels_gbs": gbs,
        "other_path": other,
        "step_kernel_elem_per_s": n_pad / (kern["step"] / 1e3),
        "kernels_ms_median": kern_med,
        "real_elem_per_s": whole_job_rate(n_real, world, args.steps, elapsed_ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "traffic_basis": traffic_basis,
                     "kernel": ("fp8z1_step_fused_select" if args.pipeline else "fp8z1_step_fused")
                               if args.path == "fused" else "fp8z1_step",
                     "peak_source": peak_kind,
                     "bytes_per_launch": step_bytes},
        "clocks": clk,
        "skipped_steps": skipped,
        "e2e": e2e,
        "bf16_fold": bf16,
        "layout_build_ms": layout_ms,
        "monitors": monitors,
        "other_workloads": others,
    }
    if rank == 0 and world == 1 and args.cpu_sample_experts > 0:
        out["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_sample_experts)
        out["cpu_baseline_all_cores"] = cpu_baseline_all_cores(args.workload, args.cpu_sample_experts)
    return out


def other_workload(spec: str, steps: int, dev, dist, peak: float) -> dict:
    """One more configuration in the headline's loop (fused path, each step
    enqueued before the previous one's found_inf is read), ``steps`` timed
    steps after 3 warm-up steps.  ``spec`` is a workload name, optionally
    with ``@D:r`` for DP rank r of D's block range.  Reports the whole step
    and each kernel (CUDA events on the launching stream), their bytes per
    real element as GB/s and as a fraction of the measured copy bandwidth."""
    import torch

    from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
    from blockwise_fp8_zero_fold_gb300 import synth
    from blockwise_fp8_zero_fold_gb300.optimizer import ShardOptimizer

    name, _, shard = spec.partition("@")
    dp, shard_rank = (int(x) for x in shard.split(":")) if shard else (1, 0)
    w = synth.workload(name, dp=dp, rank=shard_rank)
    t_setup = time.perf_counter()
    opt = ShardOptimizer(w.shapes, dp_size=dp, rank=shard_rank, device=dev, loss_scale=w.loss_scale,
                         growth_interval=w.growth_interval,
                         **{k: v for k, v in w.hp().items() if k != "loss_scale"})
    for kind in ("master", "m", "v"):
        if {"master": w.master_sigma, "m": w.m_sigma, "v": w.v_sigma}[kind] == 0.0 and not w.zero_tile_frac:
            continue  # the optimizer's buffers start at zero
        rm = synth.make_state(w, kind, dev)
        opt.fold_into(rm, getattr(opt, kind))
        del rm
    grads = synth.make_grads(w, 1, dev)
    fp8 = [torch.zeros(s, dtype=torch.uint8, device=dev) for s in w.shapes]
    gptrs, fptrs = opt.pointers(grads), opt.pointers(fp8)
    nblk = opt.b1 - opt.b0
    lut = F.fp8z1_copy_lut(opt.layout)[opt.b0:opt.b1]
    n_real = int((lut["rows_real"].astype("int64") * lut["cols_real"].astype("int64")).sum())
    n_pad = nblk * F.BLOCK_ELEMS
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup
    stream = torch.cuda.current_stream()
    for _ in range(3):
        opt.launch_step_async(gptrs, fptrs, stream)
    opt.drain()
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)] for k in ("norm", "step")}
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    skipped = 0
    for i in range(steps):
        skipped += sum(opt.launch_step_async(gptrs, fptrs, stream, {"norm": ev["norm"][i], "step": ev["step"][i]}))
    skipped += sum(opt.drain())
    t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), dist, dev) / steps
    kern = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}
    med = {k: statistics.median(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}
    step_bytes = STEP_BYTES_PER_ELEM * n_real + STEP_BYTES_PER_BLOCK * nblk
    norm_bytes = 4 * n_real
    gbs = {"norm": norm_bytes / kern["norm"] / 1e6, "step": step_bytes / kern["step"] / 1e6}
    # the norm alone, launches back to back: in the loop it follows the step,
    # whose dirty lines in L2 it writes back as it evicts them
    sums = torch.zeros(1, dtype=torch.float64, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    alone = []
    for i in range(steps + 3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        F.fp8z1_fold_norm(opt.layout, gptrs, None, opt.b0, opt.b1, sums, flag, stream)
        b.record(stream)
        alone.append((a, b))
    torch.cuda.synchronize()
    norm_alone = statistics.median(a.elapsed_time(b) for a, b in alone[3:])
    out = {"workload": _workload_label(argparse.Namespace(workload=name, experts=0, params=0), w.shapes),
           "dp": "whole buffer (1 rank)" if dp == 1 else f"rank {shard_rank} of {dp}: blocks [{opt.b0}, {opt.b1})",
           "blocks": nblk, "elems_padded": n_pad, "elems_real": n_real, "steps": steps, "warmup": 3,
           "ms_per_step": ms, "value": n_pad / (ms / 1e3), "real_elem_per_s": n_real / (ms / 1e3),
           "kernels_ms": {"fold_norm": kern["norm"], "step": kern["step"]},
           "kernels_ms_median": {"fold_norm": med["norm"], "step": med["step"]},
           "bytes_per_launch": {"fold_norm": norm_bytes, "step": step_bytes},
           "kernels_gbs": {"fold_norm": gbs["norm"], "step": gbs["step"]},
           "frac_of_measured": {"fold_norm": gbs["norm"] / peak, "step": gbs["step"] / peak},
           "fold_norm_alone": {"ms_median": norm_alone, "gbs": norm_bytes / norm_alone / 1e6,
                               "frac_of_measured": norm_bytes / norm_alone / 1e6 / peak,
                               "note": "launches back to back, not after the step: in the loop the norm "
                                       "also writes back the step's dirty L2 lines as it evicts them"},
           "skipped_steps": skipped, "setup_s": setup_s}
    del opt, grads, fp8, gptrs, fptrs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def other_workload_mx(name: str, steps: int, dev, dist, peak: float) -> dict:
    """The MXFP8 variant on workload ``name`` (whole buffer) in its pipelined
    loop, ``steps`` timed steps after 3 warm-up steps; the same record as
    ``other_workload`` (bytes: 4 per element for the norm, 29 per element plus
    the E8M0 scales for the step)."""
    import torch

    from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
    from blockwise_fp8_zero_fold_gb300 import synth
    from blockwise_fp8_zero_fold_gb300.optimizer import MxShardOptimizer

    w = synth.workload(name, dp=1, rank=0)
    t_setup = time.perf_counter()
    opt = MxShardOptimizer(w.shapes, device=dev, loss_scale=w.loss_scale, growth_interval=w.growth_interval,
                           **{k: v for k, v in w.hp().items() if k != "loss_scale"})
    n = opt.n_elems
    for kind, buf in (("master", opt.master), ("m", opt.m), ("v", opt.v)):
        _flat_into(buf, synth.make_state(w, kind, dev))
    grad = torch.empty(n, dtype=torch.float32, device=dev)
    _flat_into(grad, synth.make_grads(w, 1, dev))
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup
    stream = torch.cuda.current_stream()
    for _ in range(3):
        opt.launch_step_async(grad, stream)
    opt.drain()
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)] for k in ("norm", "step")}
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    skipped = 0
    for i in range(steps):
        skipped += sum(opt.launch_step_async(grad, stream, {"norm": ev["norm"][i], "step": ev["step"][i]}))
    skipped += sum(opt.drain())
    t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), dist, dev) / steps
    kern = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}
    med = {k: statistics.median(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}
    step_bytes, norm_bytes = 29 * n + n // 32, 4 * n
    gbs = {"norm": norm_bytes / kern["norm"] / 1e6, "step": step_bytes / kern["step"] / 1e6}
    out = {"workload": _workload_label(argparse.Namespace(workload=name, experts=0, params=0), w.shapes)
                       + " in the MXFP8 layout (E8M0 scale per 32 elements)",
           "scheme": "mx", "dp": "whole buffer (1 rank)", "groups": opt.n_groups, "elems_padded": n,
           "elems_real": n, "steps": steps, "warmup": 3, "ms_per_step": ms, "value": n / (ms / 1e3),
           "real_elem_per_s": n / (ms / 1e3),
           "kernels_ms": {"norm": kern["norm"], "step": kern["step"]},
           "kernels_ms_median": {"norm": med["norm"], "step": med["step"]},
           "bytes_per_launch": {"norm": norm_bytes, "step": step_bytes},
           "kernels_gbs": gbs, "frac_of_measured": {k: v / peak for k, v in gbs.items()},
           "whole_step_gbs": (norm_bytes + step_bytes) / ms / 1e6,
           "skipped_steps": skipped, "setup_s": setup_s}
    del opt, grad
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def _flat_into(dst, tensors):
    """The tensors' elements back to back into the flat buffer ``dst``."""
    off = 0
    for t in tensors:
        dst[off:off + t.numel()].copy_(t.reshape(-1))
        off += t.numel()


def bench_mx(args, rank, world, dist):
    """The MXFP8 variant on the same workload: flat row-major state, a step is
    the grad norm + the fused update with the MX quantiser (no fold, no table)."""
    import torch

    from blockwise_fp8_zero_fold_gb300 import build as fp8build
    from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
    from blockwise_fp8_zero_fold_gb300 import synth
    from blockwise_fp8_zero_fold_gb300.optimizer import MxShardOptimizer

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fp8build.build()
    if dist is not None:
        dist.barrier()
    F.lib()
    w = _workload(args, synth)
    opt = MxShardOptimizer(w.shapes, device=dev, loss_scale=w.loss_scale,
                           growth_interval=w.growth_interval,
                           **{k: v for k, v in w.hp().items() if k != "loss_scale"})
    n = opt.n_elems
    for kind, buf in (("master", opt.master), ("m", opt.m), ("v", opt.v)):
        _flat_into(buf, synth.make_state(w, kind, dev))
    grad = torch.empty(n, dtype=torch.float32, device=dev)
    _flat_into(grad, synth.make_grads(w, 1, dev))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        if args.pipeline:
            opt.launch_step_async(grad)
        else:
            opt.step(grad)
    opt.drain()
    torch.cuda.synchronize()
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for k in ("norm", "step")}
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    n0 = F.fp8z1_kernel_launches()
    t0.record(stream)
    skipped = 0
    for i in range(args.steps if args.pipeline else 0):  # steps ahead of their found_inf
        skipped += sum(opt.launch_step_async(grad, stream, {"norm": ev["norm"][i], "step": ev["step"][i]}))
    skipped += sum(opt.drain())
    for i in range(0 if args.pipeline else args.steps):
        ev["norm"][i][0].record(stream)
        F.fp8z1_norm_reset(opt.sumsq, opt.found_inf)
        F.fp8z1_mx_grad_norm(opt.layout, grad, opt.g0, opt.g1, opt.sumsq, opt.found_inf)
        ev["norm"][i][1].record(stream)
        hp = F.make_hp(step=opt.scaler.step + 1, loss_scale=opt.scaler.scale, **opt.hp)
        ev["step"][i][0].record(stream)
        F.fp8z1_mx_step(opt.layout, hp, grad, opt.master, opt.m, opt.v, opt.codes, opt.scales,
                        opt.g0, opt.g1, opt.sumsq, opt.found_inf)
        ev["step"][i][1].record(stream)
        skipped += opt.finish_step()
    t1.record(stream)
    launches = F.fp8z1_kernel_launches() - n0
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    kern = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}
    peak, peak_kind = _peak_hbm()
    step_bytes = 29 * n + n // 32
    achieved = step_bytes / (kern["step"] / 1e3) / 1e9
    return {
        "metric": METRIC,
        "value": whole_job_rate(n, world, args.steps, elapsed_ms / 1e3),
        "unit": "elem/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,s) grads/master/moments as the workload states)",
        "config": {"workload": _workload_label(args, w.shapes) + " in the MXFP8 layout (E8M0 scale per 32 elements)",
                   "elems": n, "groups": opt.n_groups, "dp": "whole buffer (1 rank)",
                   "l2": "inputs larger than L2, no flush"},
        "scheme": "mx", "gpu_launches": launches, "kernels_ms": kern,
        "kernels_gbs": {"norm": 4 * n / kern["norm"] / 1e6, "step": achieved},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "fp8z1_mx_step_select" if args.pipeline else "fp8z1_mx_step",
                     "peak_source": peak_kind, "bytes_per_launch": step_bytes},
        "clocks": clk, "skipped_steps": skipped, "e2e": None,
    }


def _step_source_sha():
    """Hash of the files holding the step kernel's device code (the entry
    points in step.cu are host code): its traffic is stale once they change."""
    import hashlib
    h = hashlib.sha256()
    for name in ("step_args.h", "step_kernel.cuh", "step_full.cu", "step_pad.cu", "update.cuh"):
        with open(os.path.join(ROOT, "blockwise_fp8_zero_fold_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class OracleSample:
    """The oracle (single thread) on the first ``experts`` experts of each MoE
    param, over the whole path: fold grads, exact norm, step, unfold codes.
    Inputs are drawn once; run() times one pass."""

    def __init__(self, workload: str, experts: int):
        import numpy as np

        import oracle
        from blockwise_fp8_zero_fold_gb300 import synth

        w = synth.workload(workload)
        self.shapes = [(min(e, experts), r, c) for e, r, c in w.shapes]
        self.w = synth.workload(workload, shapes=self.shapes)
        fold = oracle.fold
        self.p = fold(self.shapes, [t.numpy() for t in synth.make_state(self.w, "master", "cpu")])
        self.m = fold(self.shapes, [t.numpy() for t in synth.make_state(self.w, "m", "cpu")])
        self.v = fold(self.shapes, [t.numpy() for t in synth.make_state(self.w, "v", "cpu")])
        self.g_rows = [t.numpy() for t in synth.make_grads(self.w, 1, "cpu")]
        self.outs = [np.zeros(s, np.uint8) for s in self.shapes]
        self.n_pad = self.p.size
        self.t = 0
        self.sample = (f"{workload}, first {experts} expert(s) of each param ({self.n_pad} padded "
                       f"elements); whole path: fold grads, exact norm, step, unfold codes")

    def run(self) -> float:
        import oracle

        self.t += 1
        t0 = time.perf_counter()
        g = oracle.fold(self.shapes, self.g_rows)
        s, f = oracle.sumsq(g)
        q, _, _ = oracle.step(oracle.make_hp(step=self.t, **self.w.hp()), s, f, g, self.p, self.m, self.v)
        oracle.unfold(self.shapes, q, self.outs)
        return time.perf_counter() - t0


    def run_threads(self, threads: int) -> float:
        """The same pass with the oracle's calls on ``threads`` contiguous block
        ranges at once (ctypes releases the GIL during each call; blocks are
        independent once the global sum of squares is known)."""
        from concurrent.futures import ThreadPoolExecutor

        import numpy as np

        import oracle

        self.t += 1
        nb = self.n_pad // 16384
        cuts = [nb * i // threads for i in range(threads + 1)]
        ranges = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
        g = np.empty(self.n_pad, np.float32)
        q = np.empty(self.n_pad, np.uint8)
        hp = oracle.make_hp(step=self.t, **self.w.hp())
        E = 16384
        t0 = time.perf_counter()
        with ThreadPoolExecutor(len(ranges)) as ex:
            def fold(r):
                g[r[0] * E:r[1] * E] = oracle.fold(self.shapes, self.g_rows, r[0], r[1])
            list(ex.map(fold, ranges))
            s, f = oracle.sumsq_parallel([g], threads=len(ranges))

            def step(r):
                sl = slice(r[0] * E, r[1] * E)
                q[sl] = oracle.step(hp, s, f, g[sl], self.p[sl], self.m[sl], self.v[sl])[0]
            list(ex.map(step, ranges))
            list(ex.map(lambda r: oracle.unfold(self.shapes, q[r[0] * E:r[1] * E], self.outs, r[0], r[1]),
                        ranges))
        return time.perf_counter() - t0


def _host_info():
    ram = None
    try:
        with open("/proc/meminfo") as f:
            ram = round(int(f.readline().split()[1]) / 2**20, 1)
    except Exception:
        pass
    return {"cpu": _cpu_name(), "host_cores": os.cpu_count(), "ram_gb": ram}


def cpu_baseline(workload: str, experts: int, min_seconds: float = 10.0):
    """The oracle on one core: passes over the sample until min_seconds of CPU
    work have run (at least two)."""
    s = OracleSample(workload, experts)
    ts = []
    while len(ts) < 2 or sum(ts) < min_seconds:
        ts.append(s.run())
    return {"value": s.n_pad * len(ts) / sum(ts), "unit": "elem/s", "cores": 1, "kind": "oracle",
            "sample": s.sample, "passes": len(ts), "seconds": sum(ts), **_host_info()}


def cpu_baseline_all_cores(workload: str, experts: int):
    """The oracle as it stands, on every host core (one thread per core, each
    on a contiguous block range).  A second reported baseline."""
    s = OracleSample(workload, experts)
    n = os.cpu_count() or 1
    t = s.run_threads(n)
    return {"value": s.n_pad / t, "unit": "elem/s", "cores": n, "kind": "oracle, block ranges on every core",
            "sample": s.sample, "seconds": t, **_host_info()}


_ARM_PARTS = {"0xd4f": "Arm Neoverse V2 (Grace)", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1"}


def _cpu_name():
    """The CPU model: 'model name' on x86, the Arm part number named where known."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    v = line.split(":", 1)[1].strip()
                    return _ARM_PARTS.get(v.lower(), v)
    except Exception:
        pass
    return os.uname().machine


def bench_reference(args, rank, world):
    """The oracle as the reference arm, on the host cores, rank 0 only: the
    same workload record as our arm's line, each step one pass of the oracle
    over a bounded sample -- the cpu_baseline's sample (the first
    --cpu-sample-experts experts of each param) unless the run's W + K passes
    would then exceed --ref-budget-s, in which case fewer experts."""
    if rank != 0:
        return None
    from blockwise_fp8_zero_fold_gb300 import synth

    experts = args.ref_sample_experts if args.ref_sample_experts > 0 else max(1, args.cpu_sample_experts)
    smp = OracleSample(args.workload, experts)
    first = smp.run()  # the first warm-up pass, also sizing the sample
    passes = args.warmup + args.steps
    if args.ref_sample_experts <= 0 and passes * first > args.ref_budget_s and experts > 1:
        experts = max(1, int(experts * args.ref_budget_s / (passes * first)))
        smp = OracleSample(args.workload, experts)
        smp.run()
    for _ in range(args.warmup - 1):
        smp.run()
    ts = [smp.run() for _ in range(args.steps)]
    v = smp.n_pad * len(ts) / sum(ts)
    w = _workload(args, synth)
    dp, shard_rank = (int(x) for x in args.shard.split(":")) if args.shard else (1, 0)
    nblk = sum(e * -(-r // 128) * -(-c // 128) for e, r, c in w.shapes)
    per = -(-nblk // dp)
    b0, b1 = min(per * shard_rank, nblk), min(per * (shard_rank + 1), nblk)
    if dp == 1:
        n_real = w.n_real
    else:
        import oracle
        lut = oracle.build_lut(w.shapes)[b0:b1]
        n_real = int((lut[:, 4] * lut[:, 5]).sum())
    return {
        "impl": "reference",
        "metric": METRIC, "value": v, "unit": "elem/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sum(ts) / len(ts) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,s) grads/master/moments as the workload states)",
        "config": _config(args, w.shapes, dp, shard_rank, b0, b1, n_real, world),
        "sample": smp.sample,
        "cpu_baseline": {"value": v, "unit": "elem/s", "cores": 1, "kind": "oracle",
                         "sample": smp.sample, **_host_info()},
        "e2e": {"value": v, "unit": "elem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


WORKLOADS = ("tiny", "dense", "moe", "ragged", "ragged_literal", "large", "large_literal")


def list_workloads():
    """One JSON line per workload: its shapes (or the rule that draws them),
    sizes, hyper-parameters and input distributions, as synth.py defines them."""
    import dataclasses

    sys.path.insert(0, ROOT)
    from blockwise_fp8_zero_fold_gb300 import synth

    for name in WORKLOADS:
        w = synth.workload(name)
        d = dataclasses.asdict(w)
        shapes = [tuple(int(x) for x in s) for s in w.shapes]
        d["n_params"] = len(shapes)
        d["n_blocks"] = sum(e * -(-r // 128) * -(-c // 128) for e, r, c in shapes)
        d["n_real"] = w.n_real
        if name in ("ragged", "ragged_literal"):
            hi = 690 if name == "ragged" else 3000
            d["shapes"] = f"synth.ragged_shapes(n=4000, lo=17, hi={hi}, seed=0): R, C uniform in [17, {hi}], " \
                          "redrawn while a multiple of 128"
        else:
            d["shapes"] = shapes
        print(json.dumps(d))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="moe")
    ap.add_argument("--scheme", choices=["block", "mx"], default="block",
                    help="block: 128x128 blockwise FP8 (the method); mx: the MXFP8 variant")
    ap.add_argument("--path", choices=["fused", "unfused"], default="fused",
                    help="fused: norm from row-major grads + step with fused fold/unfold (2 passes); "
                         "unfused: fold, norm, step, unfold (4 passes)")
    ap.add_argument("--compare", type=int, default=1, help="also time the other path briefly")
    ap.add_argument("--experts", type=int, default=0,
                    help="keep only the first K experts of each 3-D param (a smaller case)")
    ap.add_argument("--pipeline", type=int, default=-1,
                    help="enqueue each step before the previous one's found_inf is read "
                         "(launch_step_async); -1: on for MX and the block scheme's fused path")
    ap.add_argument("--params", type=int, default=0,
                    help="keep only the first K params of the workload (a smaller case)")
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--e2e-reps", type=int, default=5,
                    help="repetitions of each e2e form (alternating); the medians are reported")
    ap.add_argument("--monitors", type=int, default=0,
                    help="also time N launches of the fused step with the per-block quantisation monitors")
    ap.add_argument("--bf16-fold", type=int, default=0,
                    help="also time N launches each of the bf16 fold and unfold of the weights")
    ap.add_argument("--shard", default="", help="D:r -- time DP rank r's block range of D ranks "
                    "instead of the whole buffer (block scheme)")
    ap.add_argument("--other-workloads", default="dense,ragged,moe@8:3,ragged_literal,large,mx:moe",
                    help="comma-separated configurations (name, name@D:r, or mx:name for the MXFP8 "
                         "variant) timed after the headline for --other-steps steps each in the same "
                         "loop; empty or 'none': none")
    ap.add_argument("--other-steps", type=int, default=20)
    ap.add_argument("--cpu-sample-experts", type=int, default=6)
    ap.add_argument("--ref-sample-experts", type=int, default=0,
                    help="experts per param in the reference arm's sample; 0: the cpu_baseline's, "
                         "fewer when W + K passes would exceed --ref-budget-s")
    ap.add_argument("--ref-budget-s", type=float, default=180.0)
    ap.add_argument("--list-workloads", action="store_true",
                    help="print each workload's configuration as one JSON line and exit")
    args = ap.parse_args()
    if args.list_workloads:
        list_workloads()
        return
    if args.pipeline < 0:
        args.pipeline = int(args.scheme == "mx" or args.path == "fused")
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        out = bench_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as td
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        td.init_process_group("nccl")
        dist = td
    out = bench_mx(args, rank, world, dist) if args.scheme == "mx" else bench_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
