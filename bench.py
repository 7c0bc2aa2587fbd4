#!/usr/bin/env python3
"""Benchmark of the fused, chunked top-K KL loss (forward + backward) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload longctx]
    python bench.py --impl reference ...      # the fp64 CPU oracle, timed on host cores

    python bench.py --sweep                   # output-head-only T sweep, one line per T
    python bench.py --topk-cache              # the teacher-cache builder

One step = one ``kd_topk_kl_fused_step`` over the whole workload: every chunk's
prep, logits GEMM with fused softmax partials and top-K gather, combine,
logits GEMM again with the gradient epilogue (merged with the next chunk's
forward GEMM), dH = G W and dW += G^T H.  Default workload: the long-context
head (T 32768, d 3072, V 128256, K 100, chunk 2048).  Inputs are seeded
synthetic tensors of that shape; W alone (788 MB) is larger than L2, so no
flush is needed between steps.

Prints ONE JSON line (rank 0).  ``value`` is tokens/s of the whole job with
inputs resident in HBM; ``e2e`` repeats the measurement through the public
API with the step's inputs (H, idx, p) copied from pinned host memory (on a
side stream, one step ahead, into two device buffers) and the loss read back
every step; ``variants.fused_norecompute`` times the fused step without the
backward recompute in the same run, and ``variants.separate_forward_backward``
the forward and backward entry points called one after the other.  N > 1 runs one independent replica per
GPU (torchrun; the path needs no data exchange for this metric), timed
between barriers, max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused top-K KL fwd+bwd tokens/s & TFLOP/s (fraction of bf16 peak); peak bytes vs T"

# DRAM traffic per launch of the kernels that can dominate the step, carried
# over from ncu captures (dram__bytes_read.sum + dram__bytes_write.sum), one
# kernel and at most three launches per capture, of the same command at
# T 8192, where every launch does the work of a launch at T 32768; reported
# only while the kernel sources still hash to what was captured.  gemm_dw: one
# launch per group of two 2048-row chunks, the first group of a step stores dW
# ("first"), the others reduce-add into it ("rest").  logits_gf: one chunk's G
# with the next chunk's forward.
TRAFFIC = {"workload": "longctx", "src_sha": "bce7373be8465ed0", "kinds": {
    "gemm_dw": {"first": 1842127872 + 1546414080, "rest": 3012833536 + 1538813696},
    "logits_gf": {"first": 971829504 + 525924352,
                  "rest": (1128472064 + 522564864 + 1067071232 + 522660608) // 2},
}}
# sequence lengths of the peak-bytes-versus-T series (the output-head-only benchmark's range)
PEAK_T = (4096, 8192, 16384, 32768, 65536, 131072, 262144)
KERNEL_SOURCES = ["lm_head_top_tma_b300/csrc/kd_gemm.cuh", "lm_head_top_tma_b300/csrc/kd_ptx.cuh",
                  "lm_head_top_tma_b300/csrc/kdtopk.cu"]


def _code_only(src: str) -> str:
    """C/C++ source without comments and whitespace: what the compiler sees."""
    import re

    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return re.sub(r"\s+", "", src)


def kernel_src_sha(read=None) -> str:
    """Hash of the kernel sources' code (comments and layout excluded)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(ROOT, f)) as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(_code_only(text).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"bf16": float(pk["bf16_tflops"]), "bf16_sustained": float(pk["bf16_tflops_sustained"]),
                "hbm": float(pk["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16": 1800.0, "bf16_sustained": 1400.0, "hbm": 6400.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        # nvidia-smi numbers GPUs physically; CUDA may renumber them (CUDA_VISIBLE_DEVICES),
        # so the sampled GPU is named by its UUID when torch reports one
        self.gpu = str(gpu_index)
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(gpu_index).uuid)
            if uuid:
                self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kd_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in open(self.path).read().splitlines():
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ dist
def dist_setup(n_gpus: int):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=ws)
    return rank, local, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle leg
def oracle_tokens_per_s(H_cpu, W_cpu, idx, p, target_s: float, rows0: int = 128):
    """Time the fp64 oracle (forward + backward incl. dW) on a bounded row sample,
    sized from a first run on `rows0` rows to take about `target_s` seconds."""
    import numpy as np
    from oracle import kd_oracle

    Wd = W_cpu.double().numpy()
    T = H_cpu.shape[0]
    n = min(rows0, T)
    t0 = time.perf_counter()
    kd_oracle(H_cpu[:n], Wd, idx[:n], p[:n])
    dt = time.perf_counter() - t0
    rows = int(min(T, max(n, n * target_s / max(dt, 1e-6))))
    rows = max(n, (rows // 64) * 64)
    t0 = time.perf_counter()
    kd_oracle(H_cpu[:rows], Wd, idx[:rows], p[:rows])
    dt = time.perf_counter() - t0
    cores = _blas_threads()
    return rows / dt, rows, dt, cores


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np
    import torch

    from lm_head_top_tma_b300.inputs import get_workload, make_cache, make_hw
    from oracle import kd_oracle

    wl = get_workload(args.workload)
    if args.T:
        wl = wl.with_T(args.T)
    per_step_s = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    rows = 32
    H, W = make_hw(wl.T, wl.d, wl.V, wl.kind, wl.seed, device="cpu")
    idx, p = make_cache(wl.T, wl.V, wl.K, wl.kind, wl.seed)
    Wd = W.double().numpy()
    t0 = time.perf_counter()
    kd_oracle(H[:rows], Wd, idx[:rows], p[:rows])
    dt = time.perf_counter() - t0
    rows = int(max(32, min(wl.T, rows * per_step_s / max(dt, 1e-6))) // 32 * 32)
    times = []
    for s in range(args.warmup + args.steps):
        r0 = (s * rows) % max(1, wl.T - rows + 1)
        t0 = time.perf_counter()
        kd_oracle(H[r0:r0 + rows], Wd, idx[r0:r0 + rows], p[r0:r0 + rows])
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = rows * len(times) / tot
    cores = _blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} token rows per step of the {wl.name} workload, fp64 forward+backward "
                                   f"(z, lse, loss, G, dH, dW) with the full W[{wl.V},{wl.d}]"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(wl):
    return {"workload": wl.name, "T": wl.T, "d": wl.d, "V": wl.V, "K": wl.K, "chunk": wl.chunk,
            "seed": wl.seed, "l2": "inputs larger than L2 (W alone is %.0f MB), no flush" % (wl.V * wl.d * 2 / 1e6)}


# ------------------------------------------------------------------ our arm
def run_kdtopk(args):
    import numpy as np
    import torch

    from lm_head_top_tma_b300 import api
    from lm_head_top_tma_b300.inputs import get_workload, make_inputs

    rank, local, ws = dist_setup(args.gpus)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    wl = get_workload(args.workload)
    if args.T:
        wl = wl.with_T(args.T)
    inp = make_inputs(wl, device=dev, seed=wl.seed + rank)
    H, W = inp["H"], inp["W"]
    idx = torch.as_tensor(inp["idx"]).to(dev)
    p = torch.as_tensor(inp["p"]).to(dev)
    T, d, V, K, C = wl.T, wl.d, wl.V, wl.K, wl.chunk
    torch.cuda.reset_peak_memory_stats(dev)
    work = api.Workspace(dev)
    out = {"loss": torch.empty(1, device=dev), "lse": torch.empty(T, device=dev),
           "dH": torch.empty(T, d, device=dev), "dW": torch.empty(V, d, device=dev)}
    stream = torch.cuda.current_stream(dev)

    def step(h=H, i=idx, pp=p):
        api.fused_step(h, W, i, pp, C, workspace=work, out=out, check=False)

    for _ in range(args.warmup):
        step()
    from lm_head_top_tma_b300 import _native as N

    N.check(api.device_status(work.buf, dev), "warm-up")
    torch.cuda.synchronize(dev)

    # ---- device-resident timed region (no per-kernel events inside it)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.stop()
    N.check(api.device_status(work.buf, dev), "timed steps")
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, ws)
    tokens_per_s = ws * T / (ms / 1e3)
    peak_bytes = torch.cuda.max_memory_allocated(dev)  # inputs + outputs + workspace of the step

    # ---- the same K steps again with a CUDA event pair around every launch, on the
    # launching stream: the per-kernel breakdown, the launch count and the dominant
    # kernel's roofline come from this second loop
    api.profile_enable(True)
    api.profile_read(reset=True)
    ep0, ep1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ep0.record(stream)
    for _ in range(args.steps):
        step()
    ep1.record(stream)
    torch.cuda.synchronize(dev)
    prof = api.profile_read(reset=True)
    api.profile_enable(False)
    N.check(api.device_status(work.buf, dev), "profiled steps")
    ms_profiled = ep0.elapsed_time(ep1) / args.steps

    # ---- end to end: every step's inputs copied in from pinned host memory and its loss
    # read back.  The copies run on a side stream into two device buffers, so step k+1's
    # inputs arrive while step k computes; the first copy starts after the opening event
    # and every copy completes before the step that consumes it, so all of them are
    # inside the timed region.
    Hh = H.cpu().pin_memory()
    ih = idx.cpu().pin_memory()
    ph = p.cpu().pin_memory()
    bufs = [(torch.empty_like(H), torch.empty_like(idx), torch.empty_like(p)) for _ in range(2)]
    loss_h = torch.empty(1, dtype=torch.float32).pin_memory()
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n_steps, start_event=None):
        if start_event is not None:
            copy_stream.wait_event(start_event)
        used = [False, False]

        def issue(k):
            b = k % 2
            if used[b]:
                copy_stream.wait_event(consumed[b])
            with torch.cuda.stream(copy_stream):
                for dst, src in zip(bufs[b], (Hh, ih, ph)):
                    dst.copy_(src, non_blocking=True)
                copied[b].record(copy_stream)

        for k in range(min(2, n_steps)):
            issue(k)
        for k in range(n_steps):
            b = k % 2
            stream.wait_event(copied[b])
            step(*bufs[b])
            consumed[b].record(stream)
            used[b] = True
            loss_h.copy_(out["loss"], non_blocking=True)
            if k + 2 < n_steps:
                issue(k + 2)

    e2e_run(max(1, args.warmup // 2))
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0.record(stream)
    e2e_run(args.steps, start_event=e0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws)
    h2d = Hh.numel() * Hh.element_size() + ih.numel() * 4 + ph.numel() * 4
    launches = sum(n for _, n in prof.values()) + prof["combine"][1]  # the loss reduction rides with combine

    # ---- the same step without the backward recompute (kept exponentials -> G)
    variants = {}
    if not args.no_variants:
        def step_nr():
            api.fused_step_norecompute(H, W, idx, p, C, workspace=work, out=out, check=False)

        for _ in range(args.warmup):
            step_nr()
        torch.cuda.synchronize(dev)
        api.profile_enable(True)
        api.profile_read(reset=True)
        clocks_nr = ClockSampler(local)
        clocks_nr.start()
        time.sleep(0.3)
        barrier(ws)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            step_nr()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(ws)
        clk_nr = clocks_nr.stop()
        prof_nr = api.profile_read(reset=True)
        api.profile_enable(False)
        N.check(api.device_status(work.buf, dev), "no-recompute steps")
        ms_nr = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws)
        variants["fused_norecompute"] = {
            "value": ws * T / (ms_nr / 1e3), "unit": "tokens/s", "ms_per_step": ms_nr,
            "tflops_actual_6TVd": ws * 6.0 * T * V * d / (ms_nr / 1e3) / 1e12,
            "per_kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof_nr.items() if v[1]},
            "launches_per_step": {k: v[1] // args.steps for k, v in prof_nr.items() if v[1]},
            "clocks": clk_nr}

        # ---- forward and backward as separate calls (kd_topk_kl_forward, then
        # kd_topk_kl_backward with the saved lse), each timed over its own loop
        dW_sep = torch.empty(V, d, dtype=torch.float32, device=dev)
        lse_sep = api.forward(H, W, idx, p, C, workspace=work, check=False)[1]
        for _ in range(args.warmup):
            api.forward(H, W, idx, p, C, workspace=work, check=False)
            api.backward(H, W, idx, p, lse_sep, C, dW=dW_sep, workspace=work, check=False)
        ms_sep = {}
        for name, call in (("forward", lambda: api.forward(H, W, idx, p, C, workspace=work, check=False)),
                           ("backward", lambda: api.backward(H, W, idx, p, lse_sep, C, dW=dW_sep, workspace=work,
                                                             check=False))):
            barrier(ws)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for _ in range(args.steps):
                call()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            barrier(ws)
            ms_sep[name] = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws)
        N.check(api.device_status(work.buf, dev), "separate forward / backward calls")
        ms_fb = ms_sep["forward"] + ms_sep["backward"]
        variants["separate_forward_backward"] = {
            "value": ws * T / (ms_fb / 1e3), "unit": "tokens/s", "ms_per_step": ms_fb,
            "forward_ms": ms_sep["forward"], "backward_ms": ms_sep["backward"],
            "tflops_8TVd": ws * 8.0 * T * V * d / (ms_fb / 1e3) / 1e12}
        del dW_sep

        # ---- the teacher-cache builder (the offline step that produces the cache)
        variants["topk_cache_build"] = time_topk_cache(dev, 32768, 128256, 100, args.steps, args.warmup)
        variants["topk_cache_build_fp32"] = time_topk_cache(dev, 32768, 128256, 100, args.steps, args.warmup,
                                                            dtype="fp32")

    # ---- peak bytes versus T on the benchmark head (one warm-up and one timed step per T)
    peak_vs_T = None
    ws_nbytes = work.nbytes
    if not args.no_variants and not args.no_peak_sweep:
        del out, work
        torch.cuda.empty_cache()
        peak_vs_T = {"head": {"d": d, "V": V, "K": K, "chunk": C},
                     "inputs": f"H, W drawn as the {wl.name} workload's; its teacher cache repeated to T rows",
                     "points": peak_bytes_vs_T(dev, wl, inp["idx"], inp["p"], PEAK_T)}

    flops_8 = 8.0 * T * V * d
    flops_6 = 6.0 * T * V * d
    peaks = load_peaks()
    # dominant kernel: the kind with the largest total time inside the timed region.
    # Per-launch work: a chunk's logits GEMM (forward or G) and its dH GEMM do
    # 2 C V d flops; the merged launch of one chunk's G and the next chunk's
    # forward does 4 C V d; a dW launch covers a group of chunks, 2 T V d per
    # step over its launches.
    dom = max(prof, key=lambda k: prof[k][0])
    dom_ms, dom_n = prof[dom]
    Cc = min(C, T)
    launch_flops = {"logits_fwd": 2.0 * Cc * V * d, "logits_g": 2.0 * Cc * V * d, "logits_gf": 4.0 * Cc * V * d,
                    "gemm_dh": 2.0 * Cc * V * d}
    if dom == "gemm_dw" and dom_n:
        per_launch_flops = 2.0 * T * V * d / (dom_n / args.steps)
    else:
        per_launch_flops = launch_flops.get(dom)
    achieved = per_launch_flops / (dom_ms / dom_n / 1e3) / 1e12 if per_launch_flops and dom_n else None
    traffic = None
    tk = TRAFFIC["kinds"].get(dom)
    if (tk and TRAFFIC["workload"] == wl.name and C == get_workload(wl.name).chunk
            and TRAFFIC["src_sha"] == kernel_src_sha() and dom_n):
        n_launch = dom_n // args.steps  # per step: one "first" launch, the others "rest"
        traffic = (tk["first"] + (n_launch - 1) * tk["rest"]) / n_launch
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peaks["bf16_sustained"],
                "unit": "TFLOP/s", "frac": (achieved / peaks["bf16_sustained"]) if achieved else None,
                "traffic": traffic,
                "traffic_source": ("carried over from an ncu capture at T 8192 (DRAM read + write bytes per launch) "
                                   f"of the same kernel sources (hash {TRAFFIC['src_sha']}), not measured in this run"
                                   if traffic is not None else "no capture of the current kernel sources"),
                "peak_kind": f"bf16 sustained ({peaks['source']})",
                "flops_per_launch": per_launch_flops,
                "frac_of_burst_peak": (achieved / peaks["bf16"]) if achieved else None,
                "timing": "CUDA events around each launch on the launching stream, in a second loop of the same "
                          f"{args.steps} steps after the unprofiled headline loop ({ms_profiled:.2f} ms/step with "
                          "the events)",
                "per_kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]},
                "launches_per_step": {k: v[1] // args.steps for k, v in prof.items() if v[1]}}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        Hc = H[: min(T, 4096)].cpu()
        v, rows, dt, cores = oracle_tokens_per_s(Hc, W.cpu(), inp["idx"], inp["p"], args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"first {rows} token rows of the {wl.name} workload, fp64 forward+backward "
                         f"with the full W[{V},{d}] ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": _config(wl),
            "tflops_8TVd": ws * flops_8 / (ms / 1e3) / 1e12,
            "tflops_6TVd": ws * flops_6 / (ms / 1e3) / 1e12,
            "frac_of_bf16_peak": {"burst": ws * flops_8 / (ms / 1e3) / 1e12 / ws / peaks["bf16"],
                                  "sustained": ws * flops_8 / (ms / 1e3) / 1e12 / ws / peaks["bf16_sustained"],
                                  "source": peaks["source"]},
            "workspace_bytes": ws_nbytes, "peak_bytes": peak_bytes,
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": ws * T / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": 4},
            "gpu_launches": launches,
            "clocks": clk,
            "variants": variants,
            "peak_bytes_vs_T": peak_vs_T,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_sweep(args):
    """Output-head-only scaling sweep (d 4096, V 128256, K 100, chunk 4096, T 4K..256K):
    one JSON line per T with tokens/s, TFLOP/s, library workspace and device peak bytes."""
    import torch

    from lm_head_top_tma_b300 import _native as N
    from lm_head_top_tma_b300 import api
    from lm_head_top_tma_b300.inputs import SWEEP_T, make_inputs, sweep_workload

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    for T in SWEEP_T:
        wl = sweep_workload(T)
        inp = make_inputs(wl, device=dev)
        H, W = inp["H"], inp["W"]
        idx = torch.as_tensor(inp["idx"]).to(dev)
        p = torch.as_tensor(inp["p"]).to(dev)
        del inp
        torch.cuda.synchronize(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        work = api.Workspace(dev)
        out = {"loss": torch.empty(1, device=dev), "lse": torch.empty(T, device=dev),
               "dH": torch.empty(T, wl.d, device=dev), "dW": torch.empty(wl.V, wl.d, device=dev)}
        for _ in range(max(1, args.warmup)):
            api.fused_step(H, W, idx, p, wl.chunk, workspace=work, out=out, check=False)
        N.check(api.device_status(work.buf, dev), "sweep warm-up")
        steps = max(1, min(args.steps, 5))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(steps):
            api.fused_step(H, W, idx, p, wl.chunk, workspace=work, out=out, check=False)
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        peak = torch.cuda.max_memory_allocated(dev)
        print(json.dumps({
            "sweep": wl.name, "T": T, "d": wl.d, "V": wl.V, "K": wl.K, "chunk": wl.chunk,
            "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3),
            "tflops_8TVd": 8.0 * T * wl.V * wl.d / (ms / 1e3) / 1e12,
            "workspace_bytes": work.nbytes, "peak_bytes": peak, "inputs_bytes": base,
            "peak_GiB": peak / 2**30}), flush=True)
        del H, W, idx, p, out, work
        torch.cuda.empty_cache()
    return 0


def time_topk_cache(dev, T, V, K, steps, warmup, dtype="bf16"):
    """Teacher-cache builder on synthetic teacher logits Z [T, V] (bf16 or fp32):
    CUDA-event time of `steps` launches on the launching stream, and the HBM
    roofline.  Algorithmic bytes per launch: one read of Z plus the cache
    written (idx, p) and lse."""
    import torch

    from lm_head_top_tma_b300 import api
    from lm_head_top_tma_b300.inputs import make_teacher_logits

    Z = make_teacher_logits(T, V, seed=7, device=dev, dtype=dtype)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    p = torch.empty(T, K, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    for _ in range(max(3, warmup)):
        api.topk_cache_build(Z, K, out=(idx, p, lse))
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        api.topk_cache_build(Z, K, out=(idx, p, lse))
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    bytes_alg = T * V * Z.element_size() + T * K * 8 + T * 4
    peaks = load_peaks()
    achieved = bytes_alg / (ms / 1e3) / 1e9
    del Z, idx, p, lse
    torch.cuda.empty_cache()
    return {"value": T / (ms / 1e3), "unit": "rows/s", "ms_per_launch": ms, "launches": steps,
            "config": {"workload": "teacher_logits", "T": T, "V": V, "K": K, "logits_dtype": dtype,
                       "l2": "logits larger than L2, no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm"], "traffic": None, "bytes_per_launch": bytes_alg,
                         "peak_kind": f"HBM copy ({peaks['source']})"},
            "clocks": clk}


def run_topk_cache(args):
    """Teacher-cache builder: top-K ids and probabilities of every row of
    synthetic teacher logits Z [T, V] (bf16, or fp32 with --logits-dtype fp32),
    one JSON line."""
    import torch

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    r = time_topk_cache(dev, args.T or 32768, 128256, 100, args.steps, args.warmup, args.logits_dtype)
    print(json.dumps({
        "metric": "teacher top-K cache build rows/s", "value": r["value"], "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_launch"], "higher_is_better": True,
        "dtype": args.logits_dtype, "data": "synthetic", "config": r["config"], "roofline": r["roofline"],
        "clocks": r["clocks"]}), flush=True)
    return 0


def peak_bytes_vs_T(dev, wl, idx_host, p_host, Ts):
    """Library workspace and device peak of one fused step at each sequence
    length T on the given head (d, V, K, chunk): H and W drawn as the
    workload's, the teacher cache the workload's own rows repeated to T rows.
    One warm-up step, then one step timed with CUDA events.  ``peak_bytes`` is
    the allocator's peak during the step minus what was allocated before its
    inputs existed, so it counts exactly the step's inputs, outputs and
    workspace."""
    import numpy as np
    import torch

    from lm_head_top_tma_b300 import _native as N
    from lm_head_top_tma_b300 import api
    from lm_head_top_tma_b300.inputs import make_hw

    rows = []
    for T in Ts:
        torch.cuda.synchronize(dev)
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        H, W = make_hw(T, wl.d, wl.V, wl.kind, wl.seed, device=dev)
        reps = -(-T // idx_host.shape[0])
        idx = torch.as_tensor(np.tile(idx_host, (reps, 1))[:T]).to(dev)
        p = torch.as_tensor(np.tile(p_host, (reps, 1))[:T]).to(dev)
        work = api.Workspace(dev)
        out = {"loss": torch.empty(1, device=dev), "lse": torch.empty(T, device=dev),
               "dH": torch.empty(T, wl.d, device=dev), "dW": torch.empty(wl.V, wl.d, device=dev)}
        api.fused_step(H, W, idx, p, wl.chunk, workspace=work, out=out, check=False)
        N.check(api.device_status(work.buf, dev), f"peak-bytes step at T {T}")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        api.fused_step(H, W, idx, p, wl.chunk, workspace=work, out=out, check=False)
        e1.record()
        torch.cuda.synchronize(dev)
        N.check(api.device_status(work.buf, dev), f"peak-bytes step at T {T}")
        ms = e0.elapsed_time(e1)
        peak = torch.cuda.max_memory_allocated(dev) - base
        rows.append({"T": T, "workspace_bytes": work.nbytes, "peak_bytes": peak, "ms_per_step": ms,
                     "tokens_per_s": T / (ms / 1e3), "tflops_8TVd": 8.0 * T * wl.V * wl.d / (ms / 1e3) / 1e12})
        del H, W, idx, p, out, work
        torch.cuda.empty_cache()
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kdtopk", choices=["kdtopk", "reference"])
    ap.add_argument("--workload", default="longctx")
    ap.add_argument("--T", type=int, default=None, help="override the sequence length (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=25.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip everything but the fused step (variants, peak bytes versus T)")
    ap.add_argument("--no-peak-sweep", action="store_true", help="skip the peak-bytes-versus-T series")
    ap.add_argument("--sweep", action="store_true", help="output-head-only T sweep, one line per T")
    ap.add_argument("--topk-cache", action="store_true", help="teacher-cache builder over synthetic logits")
    ap.add_argument("--logits-dtype", default="bf16", choices=["bf16", "fp32"],
                    help="teacher logits' type for --topk-cache")
    args = ap.parse_args()
    if args.sweep:
        return run_sweep(args)
    if args.topk_cache:
        return run_topk_cache(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_kdtopk(args)


if __name__ == "__main__":
    sys.exit(main())
