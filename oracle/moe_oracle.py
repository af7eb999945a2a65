"""Plain fp64 CPU oracle of the top-k gated MoE FFN layer forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product path
(the CUDA library and its Python binding) never calls it, and it imports
nothing from the product: it reads plain numpy arrays (fp32 values, or bf16 bit
patterns in ``uint16``) and computes every step in float64 with numpy, one step
per function, in the order the pages give them.

Sources (page title, section):
  [W]  "Qwen2-MoE代码解析：MoE架构原理、工程实现与部署避坑指南" (jsqmd.com; the same
       article is mirrored at ksqn.cn), section 3.1 (gate, softmax, top-k,
       renormalisation, grouping by expert), 3.3 (load-balancing loss),
       3.4 (expert capacity and token dropping).
  [M]  Qwen2-MoE module article (mlqm.cn), section 2.2 (experts are
       Linear-GELU-Linear FFNs; expert_capacity = ceil(total_tokens /
       num_experts) * num_experts_per_tok), section 3.2 (forward pass: router
       logits, softmax, top-k, per-expert gather, per-expert FFN).
  [A]  MoE sparse-activation article (wmrh.cn), section 2.2 (Router, Experts,
       Dispatcher; the k expert outputs are summed with their weights),
       section 5.2 (the router softmax temperature, 1.0 by default).

Readings taken where the pages are silent or garbled:
  * top-k is chosen on the logits (softmax is monotone), ties to the lower
    expert index, output in descending order;
  * the capacity keeps, per expert, its first C slots in (token, rank) order;
    dropped slots add nothing and the surviving weights are not renormalised;
  * the load-balancing frequency is count_i / (T*k) with counts taken before
    any drop, so the loss is exactly 1 under uniform routing;
  * with drop_tokens=False the slots the capacity would drop move, one at a
    time in slot order, to their token's best-scored unused expert with room
    (``reroute``);
  * GELU is the erf form; on the bf16 path the GELU output h and the expert
    output y are rounded to bf16 (round-to-nearest-even), everything else is
    carried in float64; the fp32 path rounds nowhere.

Every function below is pinned by ``tests/test_oracle_pins.py`` against values
the pages print, closed forms, brute force on tiny inputs or library routines.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

# ---------------------------------------------------------------------------
# storage formats


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Input values as float64.  bf16 arrays arrive as uint16 bit patterns."""
    if dtype == "bf16":
        u = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned
    as float64.  bf16 keeps 8 significant bits, exponent range as fp32; the
    subnormal quantum is 2^-133."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)                     # a = m * 2^e, 0.5 <= |m| < 1
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)
    return np.rint(a / q) * q


# ---------------------------------------------------------------------------
# router  ([W] 3.1; [M] 3.2 step 1-2)


def gate_logits(x: np.ndarray, Wg: np.ndarray, gate_bias=None) -> np.ndarray:
    """Router scores ``l = x Wg^T`` of the bias-free gate ``nn.Linear(H, E)``
    ([W] 3.1 item 1), plus an optional per-expert bias (default: none)."""
    l = x @ Wg.T
    if gate_bias is not None:
        l = l + np.asarray(gate_bias, dtype=np.float64)[None, :]
    return l


def softmax(l: np.ndarray, temperature: float = 1.0) -> np.ndarray:
    """Softmax over the expert axis ([W] 3.1; [M] 3.2 step 2) of ``l / tau``;
    the router temperature tau is 1 unless set ([A] 5.2: 2.0 flattens the
    distribution, 0.5 sharpens it)."""
    a = l / temperature
    m = a.max(axis=1, keepdims=True)
    z = np.exp(a - m)
    return z / z.sum(axis=1, keepdims=True)


def topk_select(l: np.ndarray, k: int) -> np.ndarray:
    """The k experts with the largest score per token, largest first; equal
    scores are ordered by ascending expert index ([W] 3.1, ``torch.topk``)."""
    order = np.argsort(-l, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def renormalised_weights(p: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """``w = p_sel / sum(p_sel)``: the k selected probabilities rescaled to sum
    to one ([W] 3.1 item 2)."""
    sel = np.take_along_axis(p, ids, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def route(l: np.ndarray, k: int, temperature: float = 1.0):
    """Softmax (at the given temperature), top-k and renormalisation from
    given logits.  Returns ``(ids [T,k], w [T,k], p [T,E])``.  The k experts
    are the k largest scores whatever the temperature (tau > 0 keeps the
    order); the temperature changes the probabilities and so the weights."""
    p = softmax(l, temperature)
    ids = topk_select(l, k)
    return ids, renormalised_weights(p, ids), p


# ---------------------------------------------------------------------------
# dispatch  ([W] 3.1 item 3 grouping; [W] 3.4 capacity; [M] 2.2 capacity)


def capacity_ceil(T: int, E: int, k: int) -> int:
    """``expert_capacity = ceil(total_tokens / num_experts) * num_experts_per_tok``
    ([M] 2.2)."""
    return math.ceil(T / E) * k


def dispatch(ids: np.ndarray, E: int, capacity: int = 0):
    """Group slots by expert.  Slot ``s = t*k + j`` is token t's j-th choice.

    Slots of one expert keep their (token, rank) order -- the order a stable
    sort of the expert ids gives ([W] 3.1 item 3).  With ``capacity > 0`` an
    expert keeps only its first ``capacity`` slots; the rest are dropped
    ([W] 3.4).  Returns a dict with
      count [E]   slots routed to each expert (before dropping)
      kept  [E]   slots each expert keeps
      offs  [E+1] first permuted row of each expert
      src   [R]   slot held by permuted row r (R = offs[E])
      pos   [T*k] permuted row of slot s, or -1 if dropped
      dropped     number of dropped slots
    """
    T, k = ids.shape
    flat = ids.reshape(-1)
    count = np.bincount(flat, minlength=E).astype(np.int64)
    kept = np.minimum(count, capacity) if capacity > 0 else count.copy()
    offs = np.zeros(E + 1, dtype=np.int64)
    offs[1:] = np.cumsum(kept)
    pos = np.full(T * k, -1, dtype=np.int64)
    src = np.empty(int(offs[E]), dtype=np.int64)
    for e in range(E):
        slots = np.nonzero(flat == e)[0]          # ascending slot order
        keep = slots[: kept[e]]
        rows = offs[e] + np.arange(keep.size)
        pos[keep] = rows
        src[offs[e]:offs[e + 1]] = keep
    return dict(count=count, kept=kept, offs=offs, src=src, pos=pos,
                dropped=int((count - kept).sum()))


def reroute(ids: np.ndarray, l: np.ndarray, E: int, capacity: int):
    """``drop_tokens=False`` ([W] 3.4: with it, slots over an expert's
    capacity go to the next-best expert instead of being dropped).

    Reading taken where the page stops: the slots the capacity keeps are those
    ``dispatch`` keeps (each expert's first ``capacity`` slots in (token, rank)
    order); only the slots it would drop move.  They are taken one at a time in
    slot order; each goes to its token's best-scored expert (score descending,
    index ascending) that the token does not already use -- neither among its
    k choices nor as the target of an earlier move -- and that still has room
    (``capacity`` minus the slots it already holds); with no such expert the
    slot is dropped.  A moved slot keeps its routing weight.

    Returns ``(final [T, k], dropped)``: each slot's expert after the moves,
    -1 for a dropped slot."""
    T, k = ids.shape
    d = dispatch(ids, E, capacity)
    room = (capacity - d["kept"]).astype(np.int64)
    final = np.asarray(ids, dtype=np.int64).copy()
    dropped = 0
    for t in range(T):
        used = set(int(e) for e in ids[t])
        for j in range(k):
            if d["pos"][t * k + j] >= 0:
                continue
            best = -1
            for e in range(E):
                if e in used or room[e] <= 0:
                    continue
                if best < 0 or l[t, e] > l[t, best]:      # equal scores keep the lower index
                    best = e
            final[t, j] = best
            if best < 0:
                dropped += 1
            else:
                room[best] -= 1
                used.add(best)
    return final, dropped


def dispatch_rerouted(ids: np.ndarray, l: np.ndarray, E: int, capacity: int):
    """Dispatch with ``drop_tokens=False``: ``reroute`` then group the slots by
    their final expert, stable in slot order (no expert exceeds its capacity
    any more).  ``count`` stays the count of the routing's own choices (before
    any move or drop: the load-balancing frequency); ``dropped`` counts the
    slots left without an expert."""
    T, k = ids.shape
    final, dropped = reroute(ids, l, E, capacity)
    flat = final.reshape(-1)
    load = np.bincount(flat[flat >= 0], minlength=E).astype(np.int64)
    offs = np.zeros(E + 1, dtype=np.int64)
    offs[1:] = np.cumsum(load)
    pos = np.full(T * k, -1, dtype=np.int64)
    src = np.empty(int(offs[E]), dtype=np.int64)
    for e in range(E):
        slots = np.nonzero(flat == e)[0]              # ascending slot order
        pos[slots] = offs[e] + np.arange(slots.size)
        src[offs[e]:offs[e + 1]] = slots
    count = np.bincount(np.asarray(ids).reshape(-1), minlength=E).astype(np.int64)
    return dict(count=count, kept=load, offs=offs, src=src, pos=pos, dropped=dropped, final=final)


# ---------------------------------------------------------------------------
# experts  ([M] 2.2: each expert is Linear - GELU - Linear; [A] 2.2)


def gelu(a: np.ndarray) -> np.ndarray:
    """GELU, erf form: ``a * Phi(a) = 0.5 a (1 + erf(a / sqrt 2))``."""
    return 0.5 * a * (1.0 + _erf(a / math.sqrt(2.0)))


def silu(a: np.ndarray) -> np.ndarray:
    """SiLU: ``a * sigmoid(a) = a / (1 + exp(-a))`` (exp overflows to inf for
    very negative a, giving the exact limit -0)."""
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def expert_ffn(xr: np.ndarray, W1e: np.ndarray, W2e: np.ndarray,
               b1e=None, b2e=None, bf16: bool = False, act: str = "gelu") -> np.ndarray:
    """One expert on rows ``xr [n, H]``: ``y = W2 GELU(W1 x + b1) + b2``.
    ``W1e [F, H]`` and ``W2e [H, F]`` use the nn.Linear ``[out, in]`` layout.
    On the bf16 path h and y are rounded to bf16.

    ``act="swiglu"``: the three-matrix expert (W1, W2, W3) of the Qwen2-MoE
    walkthrough, section 4.6, read as ``y = W2 (SiLU(W1 x) * (W3 x))``; here
    ``W1e [2F, H]`` stacks W1 (rows 0..F-1) over W3 (rows F..2F-1) and ``b1e``
    is ``[2F]``."""
    a = xr @ W1e.T
    if b1e is not None:
        a = a + b1e[None, :]
    if act == "swiglu":
        F = W1e.shape[0] // 2
        h = silu(a[:, :F]) * a[:, F:]
    else:
        h = gelu(a)
    if bf16:
        h = round_bf16(h)
    y = h @ W2e.T
    if b2e is not None:
        y = y + b2e[None, :]
    if bf16:
        y = round_bf16(y)
    return y


# ---------------------------------------------------------------------------
# combine  ([W] 3.1 item 2; [A] 2.2)


def combine(y_perm: np.ndarray, pos: np.ndarray, w: np.ndarray) -> np.ndarray:
    """``out[t] = sum_j w[t,j] * y_perm[pos[t*k+j]]``; a dropped slot
    (``pos = -1``) adds nothing."""
    T, k = w.shape
    out = np.zeros((T, y_perm.shape[1]), dtype=np.float64)
    p = pos.reshape(T, k)
    for j in range(k):
        keep = p[:, j] >= 0
        out[keep] += w[keep, j:j + 1] * y_perm[p[keep, j]]
    return out


# ---------------------------------------------------------------------------
# load-balancing loss  ([W] 3.3)


def aux_loss(p: np.ndarray, count: np.ndarray, k: int) -> float:
    """``L = E * sum_i f_i P_i`` with ``P_i`` the mean router probability of
    expert i over tokens and ``f_i = count_i / (T k)`` the share of slots routed
    to it ([W] 3.3).  The caller scales L by ``router_aux_loss_coef``."""
    T, E = p.shape
    P = p.sum(axis=0) / T
    f = np.asarray(count, dtype=np.float64) / (T * k)
    return float(E * np.sum(f * P))


def aux_loss_from_psum(psum: np.ndarray, count: np.ndarray, T: int, k: int) -> float:
    """The same loss from per-expert probability sums ``psum[i] = sum_t p[t,i]``."""
    E = psum.shape[0]
    P = np.asarray(psum, dtype=np.float64) / T
    f = np.asarray(count, dtype=np.float64) / (T * k)
    return float(E * np.sum(f * P))


# ---------------------------------------------------------------------------
# whole layer


def expert_outputs(x, d, W1, W2, b1=None, b2=None, bf16=False, E=None, ids=None, act="gelu"):
    """``y_perm [R, H]``: every kept slot through its expert, rows in permuted order."""
    E = W1.shape[0] if E is None else E
    R = int(d["offs"][E])
    H = W2.shape[1]
    y_perm = np.zeros((R, H), dtype=np.float64)
    k = ids.shape[1]
    for e in range(E):
        r0, r1 = int(d["offs"][e]), int(d["offs"][e + 1])
        if r1 == r0:
            continue
        toks = d["src"][r0:r1] // k
        y_perm[r0:r1] = expert_ffn(x[toks], W1[e], W2[e],
                                   None if b1 is None else b1[e],
                                   None if b2 is None else b2[e], bf16, act)
    return y_perm


def layer_forward(x, Wg, W1, W2, k, capacity=0, gate_bias=None, b1=None, b2=None,
                  bf16=False, logits=None, temperature=1.0, act="gelu", reroute_over=False):
    """The full forward pass of [M] 3.2 with the weighted combine of [W] 3.1.

    All arrays are float64 values.  If ``logits`` is given (e.g. the GPU's fp32
    router output widened to float64), routing starts from them instead of
    from ``x Wg^T``.  ``reroute_over``: slots over capacity move to the next
    best expert with room (``dispatch_rerouted``) instead of being dropped.
    Returns a dict with every intermediate."""
    T = x.shape[0]
    E = Wg.shape[0]
    l = gate_logits(x, Wg, gate_bias) if logits is None else np.asarray(logits, np.float64)
    ids, w, p = route(l, k, temperature)
    if reroute_over and capacity > 0:
        d = dispatch_rerouted(ids, l, E, capacity)
    else:
        d = dispatch(ids, E, capacity)
    y_perm = expert_outputs(x, d, W1, W2, b1, b2, bf16, E, ids, act)
    out = combine(y_perm, d["pos"], w)
    return dict(logits=l, ids=ids, w=w, p=p, y_perm=y_perm, out=out,
                aux=aux_loss(p, d["count"], k), **d)


def token_outputs(x, ids, w, pos, W1, W2, tokens, b1=None, b2=None, bf16=False, act="gelu"):
    """``out`` rows for a subset of tokens only, given the routing.  A token's
    output depends on its own row, its k choices and their kept/dropped state,
    so this is exact for each listed token."""
    k = ids.shape[1]
    H = W2.shape[1]
    out = np.zeros((len(tokens), H), dtype=np.float64)
    for i, t in enumerate(tokens):
        for j in range(k):
            if pos[t * k + j] < 0:
                continue
            e = int(ids[t, j])
            y = expert_ffn(x[t:t + 1], W1[e], W2[e],
                           None if b1 is None else b1[e],
                           None if b2 is None else b2[e], bf16, act)
            out[i] += w[t, j] * y[0]
    return out
