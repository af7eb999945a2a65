"""Shared helpers of the GPU parity tests: move workload arrays to the device,
run the library's entry points, and bring results back as float64 / int64
numpy arrays for comparison with the oracle."""
from __future__ import annotations

import numpy as np

import sparse_mixture_experts_topk_gb300 as moe
from sparse_mixture_experts_topk_gb300 import workloads as W
from oracle import moe_oracle as O


def torch():
    import torch as _t
    return _t


def to_dev(a, dtype: str):
    t = torch()
    if a is None:
        return None
    if a.dtype == np.uint16:
        return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(t.bfloat16).cuda()
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def to_np(t_):
    """Device tensor -> numpy (bf16 as uint16 bits)."""
    t = torch()
    if t_.dtype == t.bfloat16:
        return t_.view(t.int16).cpu().numpy().view(np.uint16)
    return t_.cpu().numpy()


def as_f64(t_):
    t = torch()
    a = to_np(t_)
    if t_.dtype == t.bfloat16:
        return O.widen(a, "bf16")
    return a.astype(np.float64)


def tdtype(w: W.Workload):
    t = torch()
    return t.bfloat16 if w.dtype == W.BF16 else t.float32


def desc_of(w: W.Workload, flags: int = 0):
    if w.act == "swiglu":
        flags |= moe.MOE_FLAG_SWIGLU
    if w.reroute:
        flags |= moe.MOE_FLAG_REROUTE
    return moe.make_desc(w.T, w.H, w.E, w.K, w.F, w.capacity,
                         moe.MOE_BF16 if w.dtype == W.BF16 else moe.MOE_F32, flags, w.temperature)


class Dev:
    """Device copies of one workload's inputs."""

    def __init__(self, inp: W.LayerInputs):
        self.inp = inp
        w = inp.w
        self.w = w
        self.x = to_dev(inp.x, w.dtype)
        self.Wg = to_dev(inp.Wg, w.dtype)
        self.W1 = to_dev(inp.W1, w.dtype)
        self.W2 = to_dev(inp.W2, w.dtype)
        self.gb = to_dev(inp.gate_bias, "f32")
        self.b1 = to_dev(inp.b1, "f32")
        self.b2 = to_dev(inp.b2, "f32")

    def f64(self, name):
        a = getattr(self.inp, name)
        if a is None:
            return None
        return O.widen(a, self.w.dtype) if a.dtype in (np.uint16,) or name in ("x", "Wg", "W1", "W2") \
            else a.astype(np.float64)


def run_stages(dev: Dev, flags: int = 0):
    """Router -> dispatch -> expert FFN -> combine -> aux through the separate
    entry points; returns every intermediate as a device tensor."""
    t = torch()
    w = dev.w
    d = desc_of(w, flags)
    ws = moe.workspace(d)
    R = max(moe.moe_max_rows(d), 1)
    T, E, K, H, F = w.T, w.E, w.K, w.H, w.F
    dt = tdtype(w)
    r = {}
    r["logits"] = t.empty((T, E), dtype=t.float32, device="cuda")
    r["ids"] = t.empty((T, K), dtype=t.int32, device="cuda")
    r["w"] = t.empty((T, K), dtype=t.float32, device="cuda")
    r["psum"] = t.empty((E,), dtype=t.float32, device="cuda")
    moe.moe_router_topk(d, dev.x, dev.Wg, dev.gb, r["logits"], r["ids"], r["w"], r["psum"], ws)
    r["count"] = t.empty((E,), dtype=t.int32, device="cuda")
    r["offs"] = t.empty((E + 1,), dtype=t.int32, device="cuda")
    r["src"] = t.full((R,), -7, dtype=t.int32, device="cuda")
    r["pos"] = t.empty((T * K,), dtype=t.int32, device="cuda")
    r["x_perm"] = t.zeros((R, H), dtype=dt, device="cuda")
    r["dropped"] = t.empty((1,), dtype=t.int32, device="cuda")
    moe.moe_dispatch(d, r["ids"], dev.x, r["count"], r["offs"], r["src"], r["pos"], r["x_perm"],
                     r["dropped"], ws)
    if w.reroute and w.capacity > 0:
        # drop_tokens=False: move the slots the capacity dropped, then group
        # the moved routing (the routing's own counts stay in r["count"])
        r["ids_final"] = t.empty((T, K), dtype=t.int32, device="cuda")
        moe.moe_reroute(d, r["logits"], r["ids"], r["pos"], r["offs"], r["ids_final"], r["dropped"], ws)
        r["count_final"] = t.empty((E,), dtype=t.int32, device="cuda")
        moe.moe_dispatch(d, r["ids_final"], dev.x, r["count_final"], r["offs"], r["src"], r["pos"],
                         r["x_perm"], None, ws)
    r["h_perm"] = t.zeros((R, F), dtype=dt, device="cuda")
    r["y_perm"] = t.zeros((R, H), dtype=dt, device="cuda")
    moe.moe_expert_ffn(d, r["x_perm"], r["offs"], dev.W1, dev.b1, dev.W2, dev.b2, r["h_perm"],
                       r["y_perm"], ws)
    r["out"] = t.empty((T, H), dtype=dt, device="cuda")
    moe.moe_combine(d, r["y_perm"], r["pos"], r["w"], r["out"])
    r["aux"] = t.empty((1,), dtype=t.float32, device="cuda")
    moe.moe_aux_loss(d, r["psum"], r["count"], r["aux"])
    t.cuda.synchronize()
    r["device_error"] = moe.moe_get_device_error(ws)
    return r


def run_layer(dev: Dev, flags: int = 0, ws=None):
    t = torch()
    w = dev.w
    d = desc_of(w, flags)
    if ws is None:
        ws = moe.workspace(d)
    out = t.empty((w.T, w.H), dtype=tdtype(w), device="cuda")
    aux = t.empty((1,), dtype=t.float32, device="cuda")
    count = t.empty((w.E,), dtype=t.int32, device="cuda")
    dropped = t.empty((1,), dtype=t.int32, device="cuda")
    moe.moe_layer_forward(d, dev.x, dev.Wg, dev.gb, dev.W1, dev.b1, dev.W2, dev.b2, out, aux, count,
                          dropped, ws)
    t.cuda.synchronize()
    return dict(out=out, aux=aux, count=count, dropped=dropped, device_error=moe.moe_get_device_error(ws))


def logits_rel_err(gpu_l: np.ndarray, ref_l: np.ndarray) -> float:
    """max over rows of max|diff| / max|ref| in that row."""
    num = np.abs(gpu_l - ref_l).max(axis=1)
    den = np.maximum(np.abs(ref_l).max(axis=1), 1e-30)
    return float((num / den).max()) if gpu_l.size else 0.0


def out_errors(gpu: np.ndarray, ref: np.ndarray):
    """(max-abs, relative-L2) of the layer output."""
    if gpu.size == 0:
        return 0.0, 0.0
    diff = gpu - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    return float(np.abs(diff).max()), rel


def product_tol(ref, A, B, slope=1.0):
    """Tolerance of one bf16 expert product ``bf16(act(A @ B^T))`` computed with
    fp32 accumulation, against the oracle's fp64 product rounded to bf16:
    one bf16 ulp (each side rounds once; at most |ref| 2^-7) plus the fp32
    accumulation error carried through the activation.  The tensor cores add
    16 products exactly per step and then round into the fp32 accumulator, so
    over n = A.shape[1] terms the accumulated error is modelled as
    sqrt(ceil(n / 16)) roundings of at most 2^-23 relative to sum_i |a_i b_i|,
    which is bounded by |a| |b| (Cauchy-Schwarz), times the activation's
    largest slope.  A dropped or doubled term moves a result by about one
    product |a_i b_i|, hundreds of times this bound at the layer sizes."""
    n = A.shape[1]
    acc = np.sqrt(np.ceil(n / 16.0)) * 2.0 ** -23 * np.outer(np.linalg.norm(A, axis=1), np.linalg.norm(B, axis=1))
    return np.abs(ref) * 2.0 ** -7 + slope * acc


# largest slope of the activations: GELU'(a) = Phi(a) + a phi(a) <= 1.129
GELU_SLOPE = 1.13


# tolerances (floating point); integer outputs are compared bit-exactly
LOGITS_REL = 1e-4          # router scores, max|d| / max|ref| per row
W_ABS = 2e-6               # renormalised weights from the same fp32 scores
PSUM_REL = 2e-5            # fp32 sums of T probabilities
OUT_MAXABS_BF16 = 2e-2     # layer output vs the bf16-rounded oracle
OUT_REL_L2_BF16 = 1e-2
OUT_REL_L2_F32 = 1e-4


def oracle_dispatch(w: W.Workload, ids_o, scores):
    """The oracle's dispatch of the routing ids_o (from the GPU's scores):
    with drop_tokens=False the rerouted one."""
    if w.reroute and w.capacity > 0:
        return O.dispatch_rerouted(ids_o, scores, w.E, w.capacity)
    return O.dispatch(ids_o, w.E, w.capacity)
