"""Seeded synthetic inputs for the top-k gated MoE FFN layer.

This module only draws random numbers and packs them into the storage formats
the layer reads (fp32, or bf16 bit patterns held in ``uint16``).  It holds none
of the layer's arithmetic: both the CUDA path and the CPU oracle take their
inputs from here, so they read identical bytes.

Streams: every tensor has its own PCG64 stream, ``default_rng([seed, stream,
expert])``, so the weights of one expert can be regenerated alone.

Shapes follow the Qwen2-MoE module article (mlqm.cn), section 2.2 (config
fields ``num_experts``, ``num_experts_per_tok``, ``expert_capacity``) and the
Qwen2-MoE code walkthrough (jsqmd.com), section 3.1 (the gate is a bias-free
``nn.Linear(hidden, num_experts)`` with Xavier-uniform init).  Weights use the
``nn.Linear`` ``[out, in]`` layout: ``Wg[E, H]``, ``W1[E, F, H]``, ``W2[E, H, F]``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# stream ids (one per tensor kind)
_S_X, _S_WG, _S_W1, _S_W2, _S_BG, _S_B1, _S_B2 = range(7)

F32 = "f32"
BF16 = "bf16"


@dataclasses.dataclass(frozen=True)
class Workload:
    """One layer configuration.  ``capacity <= 0`` means no per-expert limit."""
    name: str
    T: int
    H: int
    E: int
    K: int
    F: int
    dtype: str = BF16
    capacity: int = 0
    x_kind: str = "normal"        # "normal" | "decode_distinct"
    gate_bias: str = "none"       # "none" | "zipf"
    zipf_s: float = 1.2
    ffn_bias: bool = False
    temperature: float = 1.0      # router softmax temperature
    act: str = "gelu"             # "gelu" (Linear-GELU-Linear) | "swiglu" (W2 (SiLU(W1 x) * W3 x))
    reroute: bool = False         # drop_tokens=False: over-capacity slots move to the next-best expert
    seed: int = 0

    @property
    def S(self) -> int:
        return self.T * self.K


def capacity_ceil(T: int, E: int, K: int) -> int:
    """``ceil(T / E) * K`` -- the capacity the Qwen2-MoE module article
    (mlqm.cn, section 2.2) gives for ``expert_capacity``."""
    return -(-T // E) * K


WORKLOADS = {
    # tiny fp32 layer, every step checkable by the oracle in full
    "tiny": Workload("tiny", T=64, H=256, E=8, K=2, F=512, dtype=F32),
    # batch 4 x seq 2048 prefill at the pages' layer sizes
    "prefill": Workload("prefill", T=8192, H=3584, E=32, K=2, F=2560),
    # decode-sized batches; x is built so token t routes to experts 2t, 2t+1
    "decode1": Workload("decode1", T=1, H=3584, E=32, K=2, F=2560, x_kind="decode_distinct"),
    "decode8": Workload("decode8", T=8, H=3584, E=32, K=2, F=2560, x_kind="decode_distinct"),
    # a 16-token decode batch routed by the gate as it falls: experts get 0-3 rows
    "decode16r": Workload("decode16r", T=16, H=3584, E=32, K=2, F=2560),
    # top-4 with a Zipf(1.2) gate bias and capacity ceil(T/E)*k = 2048
    "zipf_cap": Workload("zipf_cap", T=16384, H=3584, E=32, K=4, F=2560,
                         capacity=capacity_ceil(16384, 32, 4), gate_bias="zipf"),
    # the same with drop_tokens=False: the slots over capacity move to the next-best expert with room
    "zipf_reroute": Workload("zipf_reroute", T=16384, H=3584, E=32, K=4, F=2560,
                             capacity=capacity_ceil(16384, 32, 4), gate_bias="zipf", reroute=True),
    # long prefill with wide hidden and many narrow experts
    "wide": Workload("wide", T=32768, H=4096, E=64, K=2, F=1408),
    # the prefill layer with SwiGLU experts (W1, W2, W3)
    "prefill_swiglu": Workload("prefill_swiglu", T=8192, H=3584, E=32, K=2, F=2560, act="swiglu"),
    # profiler-sized case: prefill layer dims with 8 experts (weights 294 MB > L2)
    "ncu_medium": Workload("ncu_medium", T=4096, H=3584, E=8, K=2, F=2560),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Pack finite fp32 values as bf16 bit patterns, round-to-nearest-even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _pack(a32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(a32) if dtype == BF16 else np.ascontiguousarray(a32, dtype=np.float32)


def xavier_bound(fan_in: int, fan_out: int) -> float:
    """Bound of ``torch.nn.init.xavier_uniform_`` with gain 1."""
    return math.sqrt(6.0 / (fan_in + fan_out))


def _rng(seed: int, stream: int, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, stream, sub])


def gen_gate(w: Workload) -> np.ndarray:
    b = xavier_bound(w.H, w.E)
    return _pack(_rng(w.seed, _S_WG).uniform(-b, b, size=(w.E, w.H)).astype(np.float32), w.dtype)


def gen_w1(w: Workload, e: int) -> np.ndarray:
    """Expert e's first linear, ``[F, H]``; for SwiGLU experts W1 and W3
    stacked, ``[2F, H]`` (each an ``[F, H]`` Xavier-uniform linear)."""
    b = xavier_bound(w.H, w.F)
    rows = 2 * w.F if w.act == "swiglu" else w.F
    return _pack(_rng(w.seed, _S_W1, e).uniform(-b, b, size=(rows, w.H)).astype(np.float32), w.dtype)


def gen_w2(w: Workload, e: int) -> np.ndarray:
    """Expert e's second linear, ``[H, F]``."""
    b = xavier_bound(w.F, w.H)
    return _pack(_rng(w.seed, _S_W2, e).uniform(-b, b, size=(w.H, w.F)).astype(np.float32), w.dtype)


def gen_gate_bias(w: Workload):
    """Optional per-expert gate bias (fp32 ``[E]``) or None.

    ``zipf``: ``b_e = ln(p_e)`` with ``p_e`` proportional to ``(e+1)^-s``, so
    that the softmax prior over experts is Zipf(s).
    ``hot``: +20 on the first K experts and 0 elsewhere, so that every token
    picks experts 0..K-1 (the most unbalanced routing: K long segments, the
    other experts empty)."""
    if w.gate_bias == "none":
        return None
    if w.gate_bias == "zipf":
        p = (np.arange(1, w.E + 1, dtype=np.float64)) ** (-w.zipf_s)
        p /= p.sum()
        return np.log(p).astype(np.float32)
    if w.gate_bias == "hot":
        b = np.zeros(w.E, dtype=np.float32)
        b[:w.K] = 20.0
        return b
    raise ValueError(w.gate_bias)


def gen_ffn_bias(w: Workload):
    if not w.ffn_bias:
        return None, None
    b1 = _rng(w.seed, _S_B1).uniform(-0.1, 0.1, size=(w.E, 2 * w.F if w.act == "swiglu" else w.F)).astype(np.float32)
    b2 = _rng(w.seed, _S_B2).uniform(-0.1, 0.1, size=(w.E, w.H)).astype(np.float32)
    return b1, b2


def gen_x(w: Workload, Wg: np.ndarray | None = None) -> np.ndarray:
    """Token activations ``[T, H]``.

    ``normal``: x ~ N(0, 1).
    ``decode_distinct``: ``x_t = alpha * (g_{2t} + g_{2t+1}) + N(0, 1)`` where
    ``g_e`` is the unit-norm gate row e, so token t's two largest gate scores
    are experts 2t and 2t+1 by a wide margin (needs 2T <= E)."""
    r = _rng(w.seed, _S_X)
    if w.x_kind == "normal":
        return _pack(r.standard_normal(size=(w.T, w.H), dtype=np.float32), w.dtype)
    if w.x_kind == "decode_distinct":
        if 2 * w.T > w.E:
            raise ValueError("decode_distinct needs 2T <= E")
        if Wg is None:
            Wg = gen_gate(w)
        g = bf16_bits_to_f32(Wg).astype(np.float64) if w.dtype == BF16 else Wg.astype(np.float64)
        g = g / np.linalg.norm(g, axis=1, keepdims=True)
        alpha = 64.0
        noise = r.standard_normal(size=(w.T, w.H)).astype(np.float64)
        x = np.empty((w.T, w.H), dtype=np.float64)
        for t in range(w.T):
            x[t] = alpha * (g[2 * t] + g[2 * t + 1]) + noise[t]
        return _pack(x.astype(np.float32), w.dtype)
    raise ValueError(w.x_kind)


@dataclasses.dataclass
class LayerInputs:
    w: Workload
    x: np.ndarray
    Wg: np.ndarray
    W1: np.ndarray      # [E, F, H]
    W2: np.ndarray      # [E, H, F]
    gate_bias: np.ndarray | None
    b1: np.ndarray | None
    b2: np.ndarray | None


def generate(w: Workload) -> LayerInputs:
    Wg = gen_gate(w)
    x = gen_x(w, Wg)
    store = np.uint16 if w.dtype == BF16 else np.float32
    W1 = np.empty((w.E, 2 * w.F if w.act == "swiglu" else w.F, w.H), dtype=store)
    W2 = np.empty((w.E, w.H, w.F), dtype=store)
    for e in range(w.E):
        W1[e] = gen_w1(w, e)
        W2[e] = gen_w2(w, e)
    b1, b2 = gen_ffn_bias(w)
    return LayerInputs(w, x, Wg, W1, W2, gen_gate_bias(w), b1, b2)


def small(name: str, T: int, H: int, E: int, K: int, F: int, dtype: str = BF16, **kw) -> Workload:
    """A parity-test sized workload (shapes chosen by the test)."""
    return Workload(name, T=T, H=H, E=E, K=K, F=F, dtype=dtype, **kw)
