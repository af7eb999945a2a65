#!/usr/bin/env python3
"""Throughput of the top-k gated MoE FFN layer forward pass on GB300.

One step = one ``moe_layer_forward`` (router, dispatch, expert FFN, combine,
load-balancing loss) over one batch resident in HBM.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Multi-GPU (torchrun): every rank runs its own batch through its own copy of the
layer (weak scaling, no collective on the data path); rank 0 reports the
aggregate tokens/s over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# the oracle's numpy BLAS uses every host core; set before numpy loads
_CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mixture_experts_topk_gb300 import workloads as W  # noqa: E402

METRIC = "MoE layer tokens/s at 1 GB300; % of bf16 tensor peak (GEMM) and HBM BW"
FLUSH_BYTES = 512 << 20          # > 129 MB L2
# --gemm: the library's choice, or one expert GEMM kernel forced (descriptor
# flags: single-SM tiles; SM pairs; SM pairs with token rows on the MMA's M
# side for every product; SM pairs with one launch per product; the library's
# choice with one launch per product)
GEMM_FLAGS = {"auto": 0, "single": 1 << 4, "pair": 1 << 5, "pair-rows": (1 << 5) | (1 << 8),
              "pair-split": (1 << 5) | (1 << 9), "split": 1 << 9}
STAGES = ["router", "dispatch", "ffn_first", "ffn_second", "combine"]


def peaks():
    """HBM copy GB/s, bf16 TFLOP/s burst and sustained, the SM clock the burst
    figure was taken at, and where they come from."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        burst = float(d["bf16_tflops"])
        return (float(d["hbm_gbs"]), burst, float(d.get("bf16_tflops_sustained", burst)),
                float(d.get("sm_max_mhz", 2070.0)), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, 2070.0, "fallback"


def tensor_peak(burst: float, sustained: float, burst_mhz: float, clk, src: str):
    """The bf16 peak a GEMM timed in this run is held to.  With no power cap
    seen during the timed region the GPU ran its kernels at full clock, so the
    burst figure applies.  With the power cap active the burst figure is scaled
    by the median SM clock sampled during the timed region (tensor throughput
    is proportional to the SM clock).  Returns (peak, why)."""
    reasons = (clk or {}).get("reasons") or []
    mhz = (clk or {}).get("sm_mhz")
    if "sw_power_cap" not in reasons:
        return burst, f"{src} bf16 burst (no power cap during the timed region)"
    if mhz:
        return burst * min(1.0, mhz / burst_mhz), \
            f"{src} bf16 burst x median SM clock {mhz:.0f}/{burst_mhz:.0f} MHz (power cap active)"
    return sustained, f"{src} bf16 sustained (power cap active, no clock samples)"


def config_of(w: W.Workload, world: int, rows: int, used: int, gemm: str):
    """The workload description both arms print (same keys, same values)."""
    return {"workload": describe(w), "global_batch_tokens": world * w.T,
            "l2": f"flushed between timed steps ({FLUSH_BYTES >> 20} MB write, then "
                  f"{FLUSH_BYTES >> 20} MB read so the written lines are back in DRAM)",
            "parallelism": f"replicas x{world}", "kept_rows": rows, "used_experts": used, "gemm": gemm}


def gemm_desc(args) -> str:
    return args.gemm + ("+fused-combine" if getattr(args, "fused_combine", False) else "") + \
        ("+decode-split" if getattr(args, "decode_split", False) else "") + \
        ("+gather-gemm" if getattr(args, "gather_gemm", False) else "")


def describe(w: W.Workload) -> str:
    cap = f" capacity={w.capacity}" if w.capacity > 0 else ""
    return f"{w.name}: T={w.T} H={w.H} E={w.E} k={w.K} F={w.F} {w.dtype}{cap}"


def work_counts(w: W.Workload, rows: int, used_experts: int):
    """Algorithmic work of one layer pass: FLOPs of each expert product over
    the kept rows, and the bytes each stage must move once."""
    es = 2 if w.dtype == W.BF16 else 4
    S = w.S
    up = 2 if w.act == "swiglu" else 1        # SwiGLU: the first product has W1 and W3
    return {
        "ffn_flops_first": 2.0 * rows * w.H * w.F * up,
        "ffn_flops_second": 2.0 * rows * w.H * w.F,
        "router": w.T * w.H * es + w.E * w.H * es + S * 8,                 # x, Wg; ids + w
        "dispatch": w.T * w.H * es + rows * w.H * es + S * 4 * 2 + S * 4,  # x, x_perm, pos+src, ids
        "combine": rows * w.H * es + w.T * w.H * es + S * 8,               # y_perm, out; pos + w
        "ffn_first_bytes": used_experts * up * w.F * w.H * es + rows * (w.H + w.F) * es,
        "ffn_second_bytes": used_experts * w.F * w.H * es + rows * (w.H + w.F) * es,
        # the whole layer in one launch: x and Wg in, the used experts' weights, out
        "layer_bytes": 2 * w.T * w.H * es + w.E * w.H * es + used_experts * (up + 1) * w.F * w.H * es,
    }


class Clocks:
    """nvidia-smi samples (arrival time, fields) while the GPU works."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.p.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self, t0: float, t1: float):
        def pick(a, b):
            return [f for (t, f) in self.samples if a <= t <= b and len(f) >= 7]
        sel = pick(t0, t1)
        window = "timed region"
        if len(sel) < 3:                       # short region: add the loaded second before it
            sel = pick(t0 - 1.5, t1)
            window = "timed region + 1.5 s of warm-up under the same load"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(f[0]) for f in sel if num(f[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for f in sel for i in range(4) if f[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(sel[0][1]), "power_w_max": max(num(f[2]) or 0 for f in sel),
                "reasons": reasons, "samples": len(sel), "window": window}


GEMM_SOURCES = ("ffn_tc.cu", "ffn_tc2.cu", "tc_ptx.cuh", "common.cuh")
STREAM_SOURCES = ("ffn_stream.cu", "stream_body.cuh", "bf16_dot.cuh", "tc_ptx.cuh", "common.cuh")
DECODE_SOURCES = ("decode_layer.cu", "stream_body.cuh", "router_body.cuh", "combine.cuh", "bf16_dot.cuh",
                  "tc_ptx.cuh", "common.cuh")


def source_hash(files=GEMM_SOURCES) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "sparse_mixture_experts_topk_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, files=GEMM_SOURCES):
    """DRAM bytes per launch of each expert product from the committed ncu
    summary (profiles/traffic.json), if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
        e = d[workload]
        if e.get("source_hash") == source_hash(files):
            return e
    except Exception:
        pass
    return None


# ---------------------------------------------------------------- CPU oracle

def widen_inputs(inp: W.LayerInputs):
    from oracle import moe_oracle as O
    dt = inp.w.dtype
    return (O.widen(inp.x, dt), O.widen(inp.Wg, dt), O.widen(inp.W1, dt), O.widen(inp.W2, dt))


def oracle_rate(inp: W.LayerInputs, wide, n_tokens: int, reps: int = 1):
    """Seconds for reps calls of the oracle's whole layer on the first n tokens of the batch."""
    from oracle import moe_oracle as O
    x, Wg, W1, W2 = wide
    w = inp.w
    assert 0 < n_tokens <= w.T
    cap = W.capacity_ceil(n_tokens, w.E, w.K) if w.capacity > 0 else 0
    t0 = time.perf_counter()
    for _ in range(reps):
        O.layer_forward(x[:n_tokens], Wg, W1, W2, w.K, capacity=cap, gate_bias=inp.gate_bias,
                        bf16=(w.dtype == W.BF16), reroute_over=w.reroute, act=w.act, temperature=w.temperature)
    return time.perf_counter() - t0


def cpu_baseline(inp: W.LayerInputs, target_s: float):
    wide = widen_inputs(inp)
    n = min(64, inp.w.T)
    dt = oracle_rate(inp, wide, n)
    while dt < target_s / 3 and n < inp.w.T:
        n = min(inp.w.T, n * 4 if dt < target_s / 12 else n * 2)
        dt = oracle_rate(inp, wide, n)
    reps = 1
    if dt < target_s / 3:       # the whole batch is small (decode): repeat the call
        reps = max(1, min(1000, int(target_s / 3 / max(dt, 1e-6))))
        dt = oracle_rate(inp, wide, n, reps)
    return {"value": n * reps / dt, "unit": "tokens/s", "cores": _CORES, "kind": "oracle",
            "sample": f"fp64 numpy oracle, whole layer on the first {n} of {inp.w.T} tokens, "
                      f"{reps} call(s) ({dt:.1f} s); weights widened to fp64 beforehand (untimed)"}


def run_reference(args, w: W.Workload):
    from oracle import moe_oracle as O
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    inp = W.generate(w)
    wide = widen_inputs(inp)
    # the whole batch's routing (cheap) for the kept rows and used experts
    ids, _, _ = O.route(O.gate_logits(wide[0], wide[1], inp.gate_bias), w.K, w.temperature)
    dd = O.dispatch_rerouted(ids, O.gate_logits(wide[0], wide[1], inp.gate_bias), w.E, w.capacity) \
        if (w.reroute and w.capacity > 0) else O.dispatch(ids, w.E, w.capacity)
    budget = 150.0 / max(1, args.steps + args.warmup)     # seconds per step
    n = min(16, w.T)
    while n < w.T and oracle_rate(inp, wide, n) < budget / 2.5:
        n = min(w.T, n * 2)
    for _ in range(args.warmup):
        oracle_rate(inp, wide, n)
    times = [oracle_rate(inp, wide, n) for _ in range(args.steps)]
    tot = sum(times)
    value = n * args.steps / tot
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": config_of(w, world, int(dd["offs"][-1]), int((dd["count"] > 0).sum()), gemm_desc(args)),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _CORES, "kind": "oracle",
                             "sample": f"fp64 numpy oracle, whole layer on the first {n} of {w.T} "
                                       f"tokens per step ({n} tokens timed per step)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU path

def to_dev(a, torch):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_ours(args, w: W.Workload):
    import torch
    import torch.distributed as dist
    import sparse_mixture_experts_topk_gb300 as moe
    from sparse_mixture_experts_topk_gb300 import build as _b

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    if rank == 0:
        _b.build()
    if world > 1:
        dist.barrier()
    moe.lib()

    # every rank has its own batch (weak scaling); weights are replicated
    wr = W.Workload(**{**w.__dict__, "seed": w.seed + rank}) if world > 1 else w
    inp = W.generate(wr)
    x, Wg, W1, W2 = (to_dev(a, torch) for a in (inp.x, inp.Wg, inp.W1, inp.W2))
    gb = to_dev(inp.gate_bias, torch)
    dt = torch.bfloat16 if w.dtype == W.BF16 else torch.float32
    flags = (moe.MOE_FLAG_SWIGLU if w.act == "swiglu" else 0) | (moe.MOE_FLAG_REROUTE if w.reroute else 0) | \
        (moe.MOE_FLAG_FUSED_COMBINE if args.fused_combine else 0) | \
        (moe.MOE_FLAG_DECODE_SPLIT if args.decode_split else 0) | \
        (moe.MOE_FLAG_GATHER_GEMM if args.gather_gemm else 0) | GEMM_FLAGS[args.gemm]
    d = moe.make_desc(w.T, w.H, w.E, w.K, w.F, w.capacity,
                      moe.MOE_BF16 if w.dtype == W.BF16 else moe.MOE_F32, flags, w.temperature)
    launches_per_step = moe.moe_layer_launches(d)
    ffn_kind = moe.moe_ffn_kernel(d)
    fused = ffn_kind in (moe.MOE_FFN_TC_FUSED, moe.MOE_FFN_STREAM)   # both products in one launch
    one_launch = moe.moe_layer_decode_fused(d)                        # the whole decode layer in one launch
    ws = moe.workspace(d)
    out = torch.empty((w.T, w.H), dtype=dt, device="cuda")
    aux = torch.empty(1, device="cuda")
    count = torch.empty(w.E, dtype=torch.int32, device="cuda")
    dropped = torch.empty(1, dtype=torch.int32, device="cuda")
    flush = L2Flush(torch)
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_layer_forward(d, x, Wg, gb, W1, None, W2, None, out, aux, count, dropped, ws)

    clocks = Clocks(local) if rank == 0 else None
    # warm-up: W steps, and at least 1.5 s under load so clocks settle
    t_w = time.time()
    i = 0
    while i < args.warmup or time.time() - t_w < args.min_warmup_s:
        flush()
        step()
        i += 1
        if i % 20 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if moe.moe_get_device_error(ws) != 0:
        raise RuntimeError("device error flag set during warm-up")
    c = count.cpu().numpy()
    rows = w.S - int(dropped.item())         # kept rows (moved ones included under drop_tokens=False)
    used = int((c > 0).sum())

    # Timed region.  Loop A (the headline): CUDA events around each whole layer
    # call only, so the library's kernels chain with programmatic dependent
    # launch as they do for a user.  Loop B: the same steps with events at
    # every stage boundary (which break that chaining) for per-kernel times.
    ev_a = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for k in range(args.steps):
        flush()                           # L2 flushed between timed steps
        ev_a[k][0].record()
        step()
        ev_a[k][1].record()
    for k in range(args.steps):
        flush()
        moe.moe_profile_events(evs[k])
        step()
    moe.moe_profile_events(None)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t1 = time.time()
    per_step = [a.elapsed_time(b) for a, b in ev_a]
    stage_ms = {name: statistics.mean(evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(args.steps))
                for j, name in enumerate(STAGES)}
    staged_step_ms = statistics.mean(evs[k][0].elapsed_time(evs[k][5]) for k in range(args.steps))
    total_ms = sum(per_step)
    if world > 1:
        tt = torch.tensor([total_ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    if moe.moe_get_device_error(ws) != 0:
        raise RuntimeError("device error flag set in the timed region")

    # end to end: pinned host x in, host out back, through the public call
    e2e_line = None
    if not args.no_e2e:
        e2e_line = run_e2e(args, moe, torch, w, d, x, Wg, gb, W1, W2, aux, flush, stream, world, dist)
    if clocks:
        clocks.stop()
    clk = clocks.summary(t0, t1) if clocks else None
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    hbm, tflops_burst, tflops_sus, burst_mhz, src = peaks()
    tflops, tflops_why = tensor_peak(tflops_burst, tflops_sus, burst_mhz, clk, src)
    work = work_counts(w, rows, used)
    value = world * w.T * args.steps / (total_ms / 1e3)
    f1, f2 = stage_ms["ffn_first"], stage_ms["ffn_second"]
    flops = {"ffn_first": work["ffn_flops_first"], "ffn_second": work["ffn_flops_second"],
             "ffn": work["ffn_flops_first"] + work["ffn_flops_second"]}
    work["ffn_bytes"] = work["ffn_first_bytes"] + work["ffn_second_bytes"]
    if one_launch:
        # one launch runs the whole layer (after a one-block counter reset):
        # its time is the headline's, events around each whole call
        dom, dom_ms = "layer", total_ms / args.steps
    elif fused:
        # one launch runs both products: its time is the whole span between the
        # dispatch and the combine marks (the second mark follows it directly)
        dom, dom_ms = "ffn", f1 + f2
    else:
        dom, dom_ms = ("ffn_first", f1) if f1 >= f2 else ("ffn_second", f2)
    # decode-sized batches run the weight-streaming kernel: bound by HBM
    streaming = ffn_kind in (moe.MOE_FFN_STREAM, moe.MOE_FFN_STREAM_SPLIT)
    if one_launch:
        achieved = work["layer_bytes"] / (dom_ms / 1e3) / 1e9
        roof = {"kernel": "one-launch decode layer (gate scores, routing, both expert products, combine; "
                          "timed with its counter reset)", "bound": "hbm", "achieved": achieved,
                "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "peak_source": f"{src} HBM copy",
                "traffic": (ncu_traffic(w.name, DECODE_SOURCES) or {}).get(dom),
                "algorithmic_bytes_per_launch": work["layer_bytes"]}
    elif streaming:
        achieved = work[dom + "_bytes"] / (dom_ms / 1e3) / 1e9
        roof = {"kernel": "weight-streaming expert kernel (both products, one launch)" if fused
                else f"weight-streaming expert kernel ({dom})", "bound": "hbm", "achieved": achieved,
                "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "peak_source": f"{src} HBM copy",
                "traffic": (ncu_traffic(w.name, STREAM_SOURCES) or {}).get(dom),
                "algorithmic_bytes_per_launch": work[dom + "_bytes"]}
    else:
        achieved = flops[dom] / (dom_ms / 1e3) / 1e12
        traffic = ncu_traffic(w.name)
        roof = {"kernel": "expert grouped GEMM (both products, one launch)" if fused
                else f"expert grouped GEMM ({dom})", "bound": "tensor", "achieved": achieved,
                "peak": tflops, "unit": "TFLOP/s", "frac": achieved / tflops,
                "peak_source": tflops_why,
                "frac_of_burst_peak": achieved / tflops_burst, "burst_peak": tflops_burst,
                "frac_of_sustained_peak": achieved / tflops_sus, "sustained_peak": tflops_sus,
                "traffic": traffic.get(dom) if traffic else None, "algorithmic_flops_per_launch": flops[dom]}
    stages = {}
    stage_names = ["router", "dispatch", "ffn", "combine"] if fused else STAGES
    if fused:
        stage_ms = dict(stage_ms, ffn=f1 + f2)
    if one_launch:
        stage_names = []
        stages["layer"] = {"ms": dom_ms, "gbs": achieved, "frac_hbm": achieved / hbm}
    for name in stage_names:
        ms = stage_ms[name]
        if name.startswith("ffn"):
            tf = flops[name] / (ms / 1e3) / 1e12
            gbs = work[name + "_bytes"] / (ms / 1e3) / 1e9
            stages[name] = {"ms": ms, "tflops": tf, "frac_bf16_peak": tf / tflops, "gbs": gbs,
                            "frac_hbm": gbs / hbm}
        else:
            gbs = work[name] / (ms / 1e3) / 1e9
            stages[name] = {"ms": ms, "gbs": gbs, "frac_hbm": gbs / hbm}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == W.BF16 else "f32",
        "data": "synthetic",
        "config": config_of(w, world, rows, used, gemm_desc(args)),
        "roofline": roof,
        "stages": stages,
        "stage_timing": {"ms_per_step_with_stage_events": staged_step_ms,
                         "note": "per-stage CUDA events break kernel chaining; ms_per_step is timed "
                                 "with events around whole layer calls only"},
        "e2e": e2e_line,
        "gpu_launches": launches_per_step * args.steps * 2,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        del x, W1, W2
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


class L2Flush:
    """Between timed steps: write a buffer larger than L2, which evicts the
    layer's data, then read a second one, so that the written lines reach
    DRAM before the next step instead of being written back while the
    step's first kernels run."""

    def __init__(self, torch):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(FLUSH_BYTES // 8, dtype=torch.int64, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.r.max()


def run_e2e(args, moe, torch, w, d, x, Wg, gb, W1, W2, aux, flush, stream, world, dist):
    dh = moe.make_desc(w.T, w.H, w.E, w.K, w.F, w.capacity, d.dtype, d.flags | moe.MOE_FLAG_HOST_IO,
                       w.temperature)
    wsh = moe.workspace(dh)
    xh = x.cpu().pin_memory()
    outh = torch.empty_like(xh).pin_memory()
    for _ in range(3):
        moe.moe_layer_forward(dh, xh, Wg, gb, W1, None, W2, None, outh, aux, None, None, wsh)
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 50))
    tot = 0.0
    for _ in range(n):
        flush()
        torch.cuda.synchronize()
        a = time.perf_counter()
        moe.moe_layer_forward(dh, xh, Wg, gb, W1, None, W2, None, outh, aux, None, None, wsh)
        stream.synchronize()
        tot += time.perf_counter() - a
    if world > 1:
        tt = torch.tensor([tot], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        tot = float(tt.item())
    if moe.moe_get_device_error(wsh) != 0:
        raise RuntimeError("device error flag set in the end-to-end loop")
    return {"value": world * w.T * n / tot, "unit": "tokens/s",
            "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
            "d2h_bytes_per_step": int(outh.numel() * outh.element_size()),
            "steps": n, "timing": "wall clock per call: H2D of x from pinned memory, the layer, "
                                  "D2H of out, stream sync"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill", choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--min-warmup-s", type=float, default=1.5)
    ap.add_argument("--gemm", default="auto", choices=sorted(GEMM_FLAGS),
                    help="expert GEMM kernel for bf16 prefill: the library's choice, or one forced")
    ap.add_argument("--fused-combine", action="store_true",
                    help="fold the weighted combine into the second expert product's epilogue")
    ap.add_argument("--decode-split", action="store_true",
                    help="decode-sized batches: the layer's separate steps instead of the one-launch layer")
    ap.add_argument("--gather-gemm", action="store_true",
                    help="the first expert product reads its token rows from x (no gather kernel, no x_perm)")
    args = ap.parse_args()
    w = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
