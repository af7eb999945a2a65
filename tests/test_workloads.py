"""The seeded input generator: formats, determinism and the workload recipes."""
import numpy as np
import pytest

from sparse_mixture_experts_topk_gb300 import workloads as W
from oracle import moe_oracle as O


def test_bf16_packing_is_rne_like_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(10000), rng.standard_normal(100) * 1e-39]).astype(np.float32)
    bits = W.f32_to_bf16_bits(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    np.testing.assert_array_equal(W.bf16_bits_to_f32(bits).astype(np.float64), O.widen(bits, "bf16"))


def test_generation_is_deterministic_and_per_expert():
    w = W.small("t", T=16, H=32, E=4, K=2, F=48)
    a, b = W.generate(w), W.generate(w)
    for f in ("x", "Wg", "W1", "W2"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    np.testing.assert_array_equal(a.W1[2], W.gen_w1(w, 2))
    assert a.x.dtype == np.uint16 and a.W1.shape == (4, 48, 32) and a.W2.shape == (4, 32, 48)


def test_xavier_bounds_of_the_recipes():
    assert W.xavier_bound(3584, 32) == pytest.approx(0.04074, abs=1e-5)
    assert W.xavier_bound(3584, 2560) == pytest.approx(0.03125, abs=1e-6)
    assert W.xavier_bound(256, 8) == pytest.approx(0.1508, abs=1e-4)
    w = W.small("t", T=4, H=256, E=8, K=2, F=512, dtype=W.F32)
    g = W.gen_gate(w)
    assert np.abs(g).max() <= W.xavier_bound(256, 8)


def test_capacity_recipe():
    assert W.WORKLOADS["zipf_cap"].capacity == 2048
    assert W.capacity_ceil(16384, 32, 4) == O.capacity_ceil(16384, 32, 4)


@pytest.mark.parametrize("T", [1, 4])
def test_decode_recipe_routes_to_distinct_experts(T):
    w = W.small("d", T=T, H=512, E=16, K=2, F=64, x_kind="decode_distinct")
    inp = W.generate(w)
    l = O.gate_logits(O.widen(inp.x, "bf16"), O.widen(inp.Wg, "bf16"))
    ids = O.topk_select(l, 2)
    assert sorted(ids.reshape(-1).tolist()) == list(range(2 * T))
    srt = np.sort(l, axis=1)
    assert (srt[:, -2] - srt[:, -3]).min() > 3.0       # a wide margin to the 3rd choice


def test_zipf_gate_bias_is_log_zipf():
    w = W.small("z", T=4, H=32, E=32, K=4, F=16, gate_bias="zipf")
    b = W.gen_gate_bias(w).astype(np.float64)
    p = np.exp(b)
    assert p.sum() == pytest.approx(1.0, rel=1e-6)
    np.testing.assert_allclose(p[0] / p[1:], np.arange(2, 33) ** 1.2, rtol=1e-5)


def test_hot_gate_bias_sends_every_token_to_the_first_k_experts():
    from oracle import moe_oracle as O
    w = W.small("hot", T=50, H=64, E=8, K=2, F=64, gate_bias="hot")
    inp = W.generate(w)
    l = O.gate_logits(O.widen(inp.x, w.dtype), O.widen(inp.Wg, w.dtype), inp.gate_bias)
    ids, _, _ = O.route(l, w.K)
    assert set(np.unique(ids)) == {0, 1}


def test_decode16r_recipe_gives_experts_several_rows():
    """The 16-token decode batch is routed by the gate as it falls, so some
    experts stream with several activation rows (the streaming kernel's
    per-CTA stage sizing depends on it) and none with more than the batch."""
    w = W.WORKLOADS["decode16r"]
    Wg = W.gen_gate(w)
    x = W.gen_x(w, Wg)
    l = O.gate_logits(O.widen(x, w.dtype), O.widen(Wg, w.dtype))
    count = np.bincount(O.topk_select(l, w.K).ravel(), minlength=w.E)
    assert count.sum() == w.T * w.K
    assert count.max() >= 2 and count.max() <= w.T
    assert (count > 0).sum() < w.T * w.K              # shared experts, not 32 distinct ones
