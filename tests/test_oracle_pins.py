"""Pins for the CPU oracle: each function is checked against something other
than itself -- values the pages print (tests/golden/page_values.json), closed
forms, brute-force enumeration on tiny inputs, and library routines -- so that
a dropped term, a wrong sign or index, or a transposed operand fails here."""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")))


# ---------------------------------------------------------------- formats

def test_widen_bf16_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F, 0x8000, 0x4049], dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127, -0.0, 3.140625]
    got = O.widen(bits, "bf16")
    assert got.dtype == np.float64
    assert list(got) == want


def test_round_bf16_ties_and_exact_values():
    one = 1.0
    cases = [
        (one, one),
        (-2.0, -2.0),
        (one + 2.0 ** -7, one + 2.0 ** -7),            # representable
        (one + 2.0 ** -8, one),                          # tie -> even (mantissa 0)
        (one + 3 * 2.0 ** -8, one + 2.0 ** -6),          # tie -> even (mantissa 2)
        (-(one + 2.0 ** -8), -one),
        (one + 2.0 ** -8 + 2.0 ** -40, one + 2.0 ** -7),  # just above the tie
        (one + 2.0 ** -8 - 2.0 ** -40, one),              # just below the tie
        (3.0 * 2.0 ** -134, 2.0 * 2.0 ** -133),           # subnormal tie 1.5 q -> 2 q
        (2.0 ** 100 * (1 + 2.0 ** -9), 2.0 ** 100),
        (0.0, 0.0),
    ]
    for a, want in cases:
        assert O.round_bf16(np.array([a]))[0] == want, a


def test_round_bf16_matches_torch_on_fp32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    a = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # fp32 subnormals
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
    ])
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(a.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


# ---------------------------------------------------------------- router

def test_gate_logits_brute_force_integer():
    rng = np.random.default_rng(1)
    T, H, E = 5, 7, 3
    x = rng.integers(-4, 5, size=(T, H)).astype(np.float64)
    Wg = rng.integers(-4, 5, size=(E, H)).astype(np.float64)
    b = np.array([0.5, -1.0, 2.0])
    l = O.gate_logits(x, Wg, b)
    assert l.shape == (T, E)
    for t in range(T):
        for e in range(E):
            assert l[t, e] == sum(int(x[t, h]) * int(Wg[e, h]) for h in range(H)) + b[e]


def test_softmax_closed_forms():
    p = O.softmax(np.array([[0.0, math.log(2.0), math.log(3.0)]]))
    np.testing.assert_allclose(p[0], [1 / 6, 2 / 6, 3 / 6], rtol=0, atol=1e-15)
    q = O.softmax(np.full((2, 8), 3.25))
    assert np.all(q == 0.125)
    rng = np.random.default_rng(2)
    l = rng.standard_normal((4, 9)) * 10
    np.testing.assert_allclose(O.softmax(l), O.softmax(l + 123.0), rtol=1e-13)
    np.testing.assert_allclose(O.softmax(l).sum(1), 1.0, rtol=1e-15)
    # two-way softmax is the logistic function
    a, b = 0.7, -1.3
    assert abs(O.softmax(np.array([[a, b]]))[0, 0] - 1 / (1 + math.exp(b - a))) < 1e-15


def _brute_topk(row, k):
    """Best k-subset by sum of scores, then ordered; ties to lower indices.
    Enumerates every ordered k-tuple and picks the lexicographically best key
    (scores descending, then indices ascending)."""
    best = None
    for tup in itertools.permutations(range(len(row)), k):
        key = tuple(-row[i] for i in tup) + tup
        # only tuples sorted by (score desc, index asc) are candidate outputs
        if any((row[tup[i]] < row[tup[i + 1]]) or
               (row[tup[i]] == row[tup[i + 1]] and tup[i] > tup[i + 1]) for i in range(k - 1)):
            continue
        if best is None or key < best[0]:
            best = (key, tup)
    return list(best[1])


@pytest.mark.parametrize("E,k", [(4, 1), (4, 2), (5, 2), (5, 3), (6, 4), (3, 3)])
def test_topk_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    # random scores plus heavy ties drawn from a tiny alphabet
    rows = [rng.standard_normal(E) for _ in range(20)] + \
           [rng.integers(0, 3, size=E).astype(np.float64) for _ in range(40)]
    l = np.array(rows)
    ids = O.topk_select(l, k)
    for t in range(l.shape[0]):
        assert list(ids[t]) == _brute_topk(l[t], k), l[t]


def test_topk_all_tied_gives_lowest_indices():
    for E, k in [(8, 2), (32, 4), (64, 2)]:
        ids = O.topk_select(np.zeros((3, E)), k)
        assert (ids == np.arange(k)[None, :]).all()


def test_renormalised_weights_hand_values():
    p = np.array([[0.1, 0.2, 0.3, 0.4]])
    ids = O.topk_select(np.log(p), 2)
    assert list(ids[0]) == [3, 2]
    w = O.renormalised_weights(p, ids)
    np.testing.assert_allclose(w[0], [0.4 / 0.7, 0.3 / 0.7], rtol=1e-15)
    g = GOLDEN["renorm_example"]
    p2 = np.array([g["p_selected"] + [0.25, 0.25]])
    ids2 = np.array([[0, 1]])
    assert abs(sum(g["p_selected"]) - g["sum_before"]) < 1e-15
    np.testing.assert_allclose(O.renormalised_weights(p2, ids2)[0], g["w"], rtol=1e-15)


def test_route_special_cases():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((50, 8))
    ids, w, p = O.route(l, 1)
    assert np.all(w == 1.0)
    assert (ids[:, 0] == l.argmax(1)).all()
    ids, w, p = O.route(l, 8)                      # k = E: w is the full softmax
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-14)
    ids, w, p = O.route(l, 3)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-15)
    # w equals a softmax over the selected logits alone
    sel = np.take_along_axis(l, ids, 1)
    np.testing.assert_allclose(w, O.softmax(sel), rtol=1e-14)
    assert (np.diff(np.take_along_axis(l, ids, 1), axis=1) <= 0).all()


# ---------------------------------------------------------------- dispatch

def test_capacity_formula_page_values():
    for T, E, k, cap in GOLDEN["capacity_default"]["cases"]:
        assert O.capacity_ceil(T, E, k) == cap
        if k == 2 and T % E == 0:                  # the other default of the page
            assert cap == 2 * (T // E)


def _dispatch_brute(ids, E, C):
    """Walk the slots in order keeping a running count per expert."""
    T, k = ids.shape
    run = [0] * E
    kept_slots = [[] for _ in range(E)]
    pos_local = {}
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if C <= 0 or run[e] < C:
                pos_local[t * k + j] = (e, len(kept_slots[e]))
                kept_slots[e].append(t * k + j)
            run[e] += 1
    offs = [0]
    for e in range(E):
        offs.append(offs[-1] + len(kept_slots[e]))
    pos = [-1] * (T * k)
    for s, (e, r) in pos_local.items():
        pos[s] = offs[e] + r
    src = [s for e in range(E) for s in kept_slots[e]]
    return run, offs, src, pos, sum(run) - offs[-1]


def _check_dispatch(ids, E, C):
    d = O.dispatch(ids, E, C)
    count, offs, src, pos, dropped = _dispatch_brute(ids, E, C)
    assert list(d["count"]) == count
    assert list(d["offs"]) == offs
    assert list(d["src"]) == src
    assert list(d["pos"]) == pos
    assert d["dropped"] == dropped
    T, k = ids.shape
    assert d["count"].sum() == T * k
    # src is a permutation of the kept slots and pos inverts it
    kept = [s for s in range(T * k) if d["pos"][s] >= 0]
    assert sorted(d["src"].tolist()) == kept
    for r, s in enumerate(d["src"]):
        assert d["pos"][s] == r and ids.reshape(-1)[s] == np.searchsorted(d["offs"], r, side="right") - 1


def test_dispatch_exhaustive_tiny():
    # every assignment of distinct experts to T tokens, E <= 4, k <= 2
    for E, k, T in [(3, 1, 3), (3, 2, 3), (4, 2, 3), (4, 1, 4)]:
        choices = list(itertools.permutations(range(E), k))
        for combo in itertools.product(choices, repeat=T):
            ids = np.array(combo, dtype=np.int64)
            for C in (0, 1, 2):
                _check_dispatch(ids, E, C)


def test_dispatch_random_with_capacity():
    rng = np.random.default_rng(4)
    for _ in range(30):
        T, E, k = int(rng.integers(1, 40)), int(rng.integers(2, 9)), 0
        k = int(rng.integers(1, min(E, 4) + 1))
        l = rng.standard_normal((T, E)) + np.linspace(2, 0, E)[None, :]
        ids = O.topk_select(l, k)
        C = int(rng.integers(0, T + 1))
        _check_dispatch(ids, E, C)


def test_dispatch_page_slot_count():
    g = GOLDEN["slot_count"]
    rng = np.random.default_rng(5)
    for k, want in ((g["k"], g["slots"]), (1, g["slots_k1"])):
        ids = O.topk_select(rng.standard_normal((g["T"], 32)), k)
        d = O.dispatch(ids, 32, 0)
        assert d["count"].sum() == want and d["offs"][-1] == want and d["dropped"] == 0


def test_dispatch_page_capacity_collapse():
    g = GOLDEN["capacity_collapse"]
    T, E, k, C = g["T"], g["E"], g["k"], g["capacity"]
    # perfectly balanced routing: token t takes experts (2t, 2t+1) mod E
    t = np.arange(T)
    ids = np.stack([(2 * t) % E, (2 * t + 1) % E], axis=1)
    d = O.dispatch(ids, E, C)
    assert (d["count"] == T * k // E).all()
    assert d["dropped"] / (T * k) == g["dropped_fraction"]
    assert (d["kept"] == C).all()
    # earliest tokens win: the kept slots are exactly the first C tokens' slots per expert
    assert d["pos"][: C * E // k * k].min() >= 0 and d["pos"][C * E:].max() == -1


# ---------------------------------------------------------------- reroute (drop_tokens=False)

def _check_greedy(ids, l, E, C, final, dropped):
    """An independent description of the rerouting the walkthrough's 3.4
    describes (with the reading of the oracle's docstring), checked on a
    result instead of constructed: kept slots stay; a moved slot's expert was,
    at that slot's turn, the best-scored expert with room that its token did
    not use, and every better one was full; a dropped slot had no such expert
    at all.  "At a slot's turn" an expert holds the slots the capacity kept
    plus the moves of earlier slots.  These conditions determine the result
    uniquely, so they pin it."""
    T, k = ids.shape
    d = O.dispatch(ids, E, C)
    kept = d["kept"]
    assert dropped == int((final < 0).sum())
    load = np.bincount(final[final >= 0], minlength=E)
    assert (load <= C).all()
    for t in range(T):
        got = [int(e) for e in final[t] if e >= 0]
        assert len(got) == len(set(got))                   # a token never uses an expert twice
        for j in range(k):
            s = t * k + j
            if d["pos"][s] >= 0:
                assert final[t, j] == ids[t, j]           # kept slots stay
                continue
            e_new = int(final[t, j])
            assert e_new not in ids[t].tolist()
            moved_before = [(s2, int(final.reshape(-1)[s2])) for s2 in range(s)
                            if d["pos"][s2] < 0 and final.reshape(-1)[s2] >= 0]
            held = kept.copy()
            for _, e2 in moved_before:
                held[e2] += 1
            used = set(ids[t].tolist()) | {e2 for s2, e2 in moved_before if s2 // k == t}
            free = [e for e in range(E) if e not in used and held[e] < C]
            if e_new < 0:
                assert free == []
            else:
                assert e_new in free
                # no free expert ranks above it (score, then lower index)
                for e in free:
                    assert (l[t, e], -e) <= (l[t, e_new], -e_new)


def test_reroute_hand_example():
    """Four tokens that all prefer expert 0, capacity 1: token 1 moves to its
    second-best expert 2, token 2 to its second-best expert 1, token 3 finds
    both full and is dropped."""
    l = np.array([[3., 2., 1.], [3., 1., 2.], [3., 2., 1.], [3., 2., 1.]])
    ids, _, _ = O.route(l, 1)
    assert ids.reshape(-1).tolist() == [0, 0, 0, 0]
    final, dropped = O.reroute(ids, l, 3, 1)
    assert final.reshape(-1).tolist() == [0, 2, 1, -1] and dropped == 1
    d = O.dispatch_rerouted(ids, l, 3, 1)
    assert d["offs"].tolist() == [0, 1, 2, 3]
    assert d["src"].tolist() == [0, 2, 1] and d["pos"].tolist() == [0, 2, 1, -1]
    assert d["count"].tolist() == [4, 0, 0] and d["dropped"] == 1


@pytest.mark.parametrize("seed", range(40))
def test_reroute_tiny_random_satisfies_the_greedy_conditions(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 6))
    k = int(rng.integers(1, E + 1))
    T = int(rng.integers(1, 7))
    C = int(rng.integers(1, 4))
    # few distinct score values, so ties between experts are common
    l = rng.integers(-2, 3, size=(T, E)).astype(np.float64)
    if seed % 2:
        l[:, 0] += 2.0                                     # crowd the first expert
    ids, _, _ = O.route(l, k)
    final, dropped = O.reroute(ids, l, E, C)
    _check_greedy(ids, l, E, C, final, dropped)


def test_reroute_larger_random_satisfies_the_greedy_conditions():
    rng = np.random.default_rng(5)
    T, E, k = 60, 8, 3
    l = rng.standard_normal((T, E)) + np.log(np.arange(1, E + 1) ** -1.5)[None, :]
    C = O.capacity_ceil(T, E, k) // 2
    ids, _, _ = O.route(l, k)
    final, dropped = O.reroute(ids, l, E, C)
    assert dropped < O.dispatch(ids, E, C)["dropped"]        # rerouting saves slots here
    _check_greedy(ids, l, E, C, final, dropped)


def test_reroute_special_cases():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((20, 6))
    ids, _, _ = O.route(l, 2)
    # ample capacity: nothing moves
    final, dropped = O.reroute(ids, l, 6, 40)
    assert (final == ids).all() and dropped == 0
    # k = E: no other expert exists, so reroute drops exactly what dispatch drops
    ids6, _, _ = O.route(l, 6)
    final, dropped = O.reroute(ids6, l, 6, 10)
    d = O.dispatch(ids6, 6, 10)
    assert dropped == d["dropped"]
    assert ((final.reshape(-1) >= 0) == (d["pos"] >= 0)).all()
    # total capacity E * C >= T * k: every slot finds an expert
    final, dropped = O.reroute(ids, l, 6, 7)
    assert dropped == 0 and (np.bincount(final.reshape(-1), minlength=6) <= 7).all()


def test_dispatch_rerouted_groups_final_experts_stably():
    rng = np.random.default_rng(9)
    T, E, k = 40, 5, 2
    l = rng.standard_normal((T, E))
    l[:, 1] += 1.5
    ids, _, _ = O.route(l, k)
    C = 10
    d = O.dispatch_rerouted(ids, l, E, C)
    final = d["final"].reshape(-1)
    R = int(d["offs"][-1])
    assert R == T * k - d["dropped"]
    assert sorted(d["src"].tolist()) == sorted(np.nonzero(final >= 0)[0].tolist())
    for e in range(E):
        seg = d["src"][d["offs"][e]:d["offs"][e + 1]]
        assert (final[seg] == e).all() and (np.diff(seg) > 0).all()
        assert len(seg) <= C
    for s in range(T * k):
        assert (d["pos"][s] >= 0) == (final[s] >= 0)
        if d["pos"][s] >= 0:
            assert d["src"][d["pos"][s]] == s
    assert d["count"].tolist() == np.bincount(ids.reshape(-1), minlength=E).tolist()


def test_layer_forward_reroute_uses_the_new_experts():
    """Each token's output is the weighted sum of its slots' final experts,
    computed here token by token with the routing weights unchanged."""
    rng = np.random.default_rng(11)
    T, H, E, k, F = 24, 8, 4, 2, 6
    x = rng.standard_normal((T, H))
    Wg = rng.standard_normal((E, H))
    Wg[0] *= 0.0
    Wg[0] += 0.5 * x.mean(0) / (np.linalg.norm(x.mean(0)) ** 2)   # tokens lean towards expert 0
    W1 = rng.standard_normal((E, F, H)) * 0.3
    W2 = rng.standard_normal((E, H, F)) * 0.3
    C = 13                                               # 52 places for 48 slots, expert 0 over
    r = O.layer_forward(x, Wg, W1, W2, k, capacity=C, reroute_over=True)
    plain = O.layer_forward(x, Wg, W1, W2, k, capacity=C)
    final, dropped = O.reroute(r["ids"], r["logits"], E, C)
    assert r["dropped"] == dropped < plain["dropped"]
    for t in range(T):
        want = np.zeros(H)
        for j in range(k):
            e = int(final[t, j])
            if e >= 0:
                want += r["w"][t, j] * O.expert_ffn(x[t:t + 1], W1[e], W2[e])[0]
        np.testing.assert_allclose(r["out"][t], want, rtol=1e-12, atol=1e-12)
    assert r["aux"] == plain["aux"]                      # the routing's own counts


# ---------------------------------------------------------------- experts

def test_gelu_normal_cdf_values():
    # GELU(a) = a * Phi(a); Phi from the standard normal table
    Phi = {1.0: 0.8413447460685429, 2.0: 0.9772498680518208, -1.0: 0.15865525393145707,
           0.5: 0.6914624612740131, -2.5: 0.006209665325776132}
    for a, ph in Phi.items():
        assert abs(O.gelu(np.array([a]))[0] - a * ph) < 1e-15
    a = np.linspace(-6, 6, 101)
    np.testing.assert_allclose(O.gelu(a) - O.gelu(-a), a, atol=1e-14)   # Phi(a)+Phi(-a)=1
    assert O.gelu(np.array([0.0]))[0] == 0.0
    assert O.gelu(np.array([40.0]))[0] == 40.0 and O.gelu(np.array([-40.0]))[0] == 0.0


def test_expert_ffn_exact_integer_relu_regime():
    """With |W1 x| >= 20 the erf GELU equals ReLU to double precision, so an
    integer-valued FFN has an exact integer answer computed by brute force."""
    rng = np.random.default_rng(6)
    n, H, F = 4, 5, 7
    for _ in range(20):
        x = rng.integers(-3, 4, size=(n, H)).astype(np.float64)
        W1 = rng.integers(-3, 4, size=(F, H)).astype(np.float64) * 40.0
        W2 = rng.integers(-3, 4, size=(H, F)).astype(np.float64)
        y = O.expert_ffn(x, W1, W2)
        for i in range(n):
            for hh in range(H):
                want = 0
                for f in range(F):
                    a = sum(int(W1[f, c]) * int(x[i, c]) for c in range(H))
                    want += int(W2[hh, f]) * max(a, 0)
                assert abs(y[i, hh] - want) < 1e-9, (y[i, hh], want)


def test_expert_ffn_identity_w2_is_gelu_and_linear_in_w2():
    rng = np.random.default_rng(8)
    n, H = 6, 16
    x = rng.standard_normal((n, H))
    W1 = rng.standard_normal((H, H)) * 0.3
    I = np.eye(H)
    for bf16 in (False, True):
        y = O.expert_ffn(x, W1, I, bf16=bf16)
        h = O.gelu(x @ W1.T)
        np.testing.assert_array_equal(y, O.round_bf16(h) if bf16 else h)
        W2 = rng.standard_normal((H, H))
        np.testing.assert_array_equal(O.expert_ffn(x, W1, 2 * W2, bf16=bf16),
                                      2 * O.expert_ffn(x, W1, W2, bf16=bf16))


def test_expert_ffn_biases():
    H, F = 3, 2
    x = np.zeros((1, H))
    W1 = np.zeros((F, H))
    W2 = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    b1 = np.array([1.0, -1.0])
    b2 = np.array([0.0, 10.0, -5.0])
    y = O.expert_ffn(x, W1, W2, b1, b2)
    p1, pm1 = 0.8413447460685429, 0.15865525393145707
    np.testing.assert_allclose(y[0], [p1, -pm1 + 10.0, p1 - pm1 - 5.0], atol=1e-15)


# ---------------------------------------------------------------- combine

def test_combine_hand_values():
    y = np.array([[1.0], [10.0], [100.0], [1000.0]])
    # token 0 -> rows 2 (j=0) and 0 (j=1); token 1 -> row 3 and a dropped slot;
    # token 2 -> both slots dropped
    pos = np.array([2, 0, 3, -1, -1, -1])
    w = np.array([[0.75, 0.25], [0.5, 0.5], [0.9, 0.1]])
    out = O.combine(y, pos, w)
    assert out[:, 0].tolist() == [75.25, 500.0, 0.0]


# ---------------------------------------------------------------- aux loss

def test_aux_loss_uniform_cases_and_hand_values():
    rng = np.random.default_rng(9)
    T, E, k = 64, 8, 2
    # uniform P (all logits equal) -> L = sum f = 1 whatever the counts
    p = O.softmax(np.zeros((T, E)))
    count = rng.multinomial(T * k, np.ones(E) / E)
    assert O.aux_loss(p, count, k) == pytest.approx(1.0, abs=1e-15)
    # uniform f (balanced counts) -> L = sum P = 1 whatever P is
    p = O.softmax(rng.standard_normal((T, E)) * 3)
    assert O.aux_loss(p, np.full(E, T * k // E), k) == pytest.approx(1.0, abs=1e-14)
    # collapse onto one expert with one-hot probabilities -> L = E
    p = np.zeros((T, E)); p[:, 0] = 1.0
    count = np.zeros(E, dtype=np.int64); count[0] = T
    assert O.aux_loss(p, count, 1) == E
    # T = 2, E = 2 by hand
    p = np.array([[0.7, 0.3], [0.4, 0.6]])
    assert O.aux_loss(p, np.array([1, 1]), 1) == pytest.approx(1.0, abs=1e-15)
    assert O.aux_loss(p, np.array([2, 0]), 1) == pytest.approx(2 * 0.55, abs=1e-15)
    assert O.aux_loss(p, np.array([0, 2]), 1) == pytest.approx(2 * 0.45, abs=1e-15)
    # the psum form agrees
    assert O.aux_loss_from_psum(p.sum(0), np.array([2, 0]), 2, 1) == pytest.approx(1.1, abs=1e-15)


# ---------------------------------------------------------------- whole layer

def test_layer_forward_per_token_path_agrees_and_invariants():
    rng = np.random.default_rng(10)
    T, H, E, k, F = 37, 24, 6, 2, 40
    x = rng.standard_normal((T, H))
    Wg = rng.standard_normal((E, H)) * 0.3
    W1 = rng.standard_normal((E, F, H)) * 0.2
    W2 = rng.standard_normal((E, H, F)) * 0.2
    for C in (0, 9):
        for bf16 in (False, True):
            r = O.layer_forward(x, Wg, W1, W2, k, capacity=C, bf16=bf16)
            toks = list(range(T))
            ref = O.token_outputs(x, r["ids"], r["w"], r["pos"], W1, W2, toks, bf16=bf16)
            np.testing.assert_allclose(r["out"], ref, rtol=1e-13, atol=1e-13)
            assert r["count"].sum() == T * k
    # k = 1 with one expert whose W2 is the identity: out = GELU(W1 x)
    W1s = rng.standard_normal((1, H, H)) * 0.2
    r = O.layer_forward(x, np.zeros((1, H)), W1s, np.eye(H)[None], 1)
    np.testing.assert_allclose(r["out"], O.gelu(x @ W1s[0].T), rtol=1e-14)
    assert r["aux"] == pytest.approx(1.0)


def test_activation_rate_arithmetic():
    g = GOLDEN["activation_rate"]
    per = 2 * g["hidden"] * g["ffn"]
    assert per == g["per_expert"]
    assert per * g["layers"] * g["experts"] == g["total"]
    assert per * g["layers"] * g["active"] == g["active_params"]
    assert 100.0 * g["active"] / g["experts"] == g["rate_percent"]


def test_softmax_temperature_closed_forms():
    # tau scales the scores: softmax([0, ln 2, ln 3] at tau=0.5) = [1, 4, 9] / 14
    p = O.softmax(np.array([[0.0, math.log(2.0), math.log(3.0)]]), temperature=0.5)
    np.testing.assert_allclose(p[0], [1 / 14, 4 / 14, 9 / 14], rtol=0, atol=1e-15)
    p = O.softmax(np.array([[0.0, math.log(4.0)]]), temperature=2.0)       # -> [1, 2] / 3
    np.testing.assert_allclose(p[0], [1 / 3, 2 / 3], rtol=0, atol=1e-15)
    rng = np.random.default_rng(12)
    l = rng.standard_normal((20, 8)) * 3
    np.testing.assert_array_equal(O.softmax(l, 1.0), O.softmax(l))


def test_route_temperature_keeps_experts_changes_weights():
    rng = np.random.default_rng(13)
    l = rng.standard_normal((40, 8)) * 2
    ids1, w1, _ = O.route(l, 3)
    for tau in (0.5, 2.0, 1e6):
        ids, w, p = O.route(l, 3, temperature=tau)
        np.testing.assert_array_equal(ids, ids1)                 # order of scores unchanged
        sel = np.take_along_axis(l, ids, 1) / tau
        np.testing.assert_allclose(w, O.softmax(sel), rtol=1e-13)
        np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-15)
    _, w_flat, _ = O.route(l, 3, temperature=1e6)                # very hot: uniform weights
    np.testing.assert_allclose(w_flat, 1 / 3, atol=1e-5)
    _, w_cold, _ = O.route(l, 3, temperature=1e-3)               # very cold: all on the top score
    srt = np.sort(l, axis=1)
    clear = srt[:, -1] - srt[:, -2] > 0.05                       # rows without a near-tie at the top
    assert clear.sum() > 30
    np.testing.assert_allclose(w_cold[clear, 0], 1.0, atol=1e-6)


def test_silu_closed_forms():
    # sigmoid(ln 3) = 3/4, sigmoid(0) = 1/2; silu(a) - silu(-a) = a
    assert abs(O.silu(np.array([math.log(3.0)]))[0] - 0.75 * math.log(3.0)) < 1e-15
    assert O.silu(np.array([0.0]))[0] == 0.0
    a = np.linspace(-8, 8, 81)
    np.testing.assert_allclose(O.silu(a) - O.silu(-a), a, atol=1e-14)
    assert O.silu(np.array([50.0]))[0] == 50.0 and abs(O.silu(np.array([-50.0]))[0]) < 1e-19


def test_swiglu_expert_exact_integer_relu_regime():
    """With |W1 x| >= 50 SiLU equals ReLU to double precision, so the SwiGLU
    expert W2 (relu(W1 x) * (W3 x)) has an exact integer answer."""
    rng = np.random.default_rng(14)
    n, H, F = 3, 5, 6
    for _ in range(20):
        x = rng.integers(-3, 4, size=(n, H)).astype(np.float64)
        Wgt = rng.integers(-3, 4, size=(F, H)).astype(np.float64) * 50.0
        Wup = rng.integers(-3, 4, size=(F, H)).astype(np.float64)
        W2 = rng.integers(-3, 4, size=(H, F)).astype(np.float64)
        y = O.expert_ffn(x, np.concatenate([Wgt, Wup]), W2, act="swiglu")
        for i in range(n):
            for hh in range(H):
                want = 0
                for f in range(F):
                    g = sum(int(Wgt[f, c]) * int(x[i, c]) for c in range(H))
                    u = sum(int(Wup[f, c]) * int(x[i, c]) for c in range(H))
                    want += int(W2[hh, f]) * max(g, 0) * u
                assert abs(y[i, hh] - want) < 1e-9


def test_swiglu_gate_and_up_roles():
    """Unit up-projection leaves SiLU of the gate; unit gate at +inf leaves the up."""
    rng = np.random.default_rng(15)
    H = 8
    x = rng.standard_normal((4, H))
    Wgt = rng.standard_normal((H, H))
    y = O.expert_ffn(x, np.concatenate([Wgt, np.zeros((H, H))]), np.eye(H), b1e=np.r_[np.zeros(H), np.ones(H)],
                     act="swiglu")
    np.testing.assert_allclose(y, O.silu(x @ Wgt.T), rtol=1e-14)
    Wup = rng.standard_normal((H, H))
    y = O.expert_ffn(x, np.concatenate([np.zeros((H, H)), Wup]), np.eye(H), b1e=np.r_[np.full(H, 60.0), np.zeros(H)],
                     act="swiglu")
    np.testing.assert_allclose(y, 60.0 * (x @ Wup.T), rtol=1e-13)
