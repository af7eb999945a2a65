"""The one-launch decode layer against the layer's separate steps.

Batches of at most 16 bf16 tokens run by default as one launch: gate
scores, routing and placement in every CTA, the used experts' weight rows
spread evenly over the CTAs, then the combine, with counters in the
workspace between the steps.  Every value is computed with the same
operations in the same order as the separate steps (router, dispatch,
weight-streaming products, combine: MOE_FLAG_DECODE_SPLIT), so outputs,
counts, dropped slots and the loss are compared bit for bit; the outputs
are also checked against the oracle with the per-element tolerance of the
full-size tests."""
import numpy as np
import pytest

from sparse_mixture_experts_topk_gb300 import workloads as W
import sparse_mixture_experts_topk_gb300 as moe
from oracle import moe_oracle as O

from harness import (Dev, desc_of, run_stages, run_layer, to_np, as_f64, out_errors, oracle_dispatch,
                     OUT_MAXABS_BF16, OUT_REL_L2_BF16)

pytestmark = pytest.mark.gpu

CASES = {
    # one token: two CTAs per SM, two experts over all of them
    "t1_e32": W.small("t1_e32", T=1, H=512, E=32, K=2, F=256),
    "t2_e8": W.small("t2_e8", T=2, H=256, E=8, K=2, F=384),
    # capacity drops (one row per expert)
    "t3_k4_cap": W.small("t3_k4_cap", T=3, H=256, E=8, K=4, F=128, capacity=1, gate_bias="zipf"),
    "t8_distinct": W.small("t8_distinct", T=8, H=512, E=32, K=2, F=256, x_kind="decode_distinct"),
    "t16_routed": W.small("t16_routed", T=16, H=512, E=32, K=2, F=512),
    # every token to both experts: one 16-row expert per product, the largest bodies
    "t16_all": W.small("t16_all", T=16, H=256, E=2, K=2, F=128),
    "t16_hot_cap": W.small("t16_hot_cap", T=16, H=256, E=8, K=2, F=256, gate_bias="hot", capacity=5),
    # 256 gate rows, top-8: the score units cover every CTA
    "e256_k8": W.small("e256_k8", T=5, H=64, E=256, K=8, F=64),
    "swiglu_bias": W.small("swiglu_bias", T=6, H=256, E=16, K=3, F=200, act="swiglu", ffn_bias=True),
    # row sizes that are whole 16-byte vectors but not 128-byte lines
    "h_ragged": W.small("h_ragged", T=5, H=200, E=8, K=2, F=264),
    "temp_zipf": W.small("temp_zipf", T=7, H=128, E=16, K=4, F=96, temperature=0.7, gate_bias="zipf"),
    # four score pieces per gate row, 14 KB token rows
    "wide_h": W.small("wide_h", T=4, H=7168, E=16, K=2, F=512),
    # all kept h rows (128 x 2 KB) do not fit beside the ring: the second
    # product runs expert by expert and the combine reads y back
    "t16_k8_wide_f": W.small("t16_k8_wide_f", T=16, H=256, E=64, K=8, F=1024),
    # top-1 routing (weights all 1), the smallest expert count, one token on both experts
    "t3_k1": W.small("t3_k1", T=3, H=256, E=4, K=1, F=128),
    "t1_e2": W.small("t1_e2", T=1, H=256, E=2, K=2, F=128),
    "t16_e256_k1": W.small("t16_e256_k1", T=16, H=128, E=256, K=1, F=64),
    # capacity 1 with every token preferring the same two experts: most slots dropped
    "t9_hot_cap1": W.small("t9_hot_cap1", T=9, H=128, E=8, K=2, F=96, gate_bias="hot", capacity=1),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_topk_gb300 import build
    build.build()
    moe.lib()


def _same(a, b):
    for k in ("out", "count", "dropped", "aux"):
        np.testing.assert_array_equal(to_np(a[k]), to_np(b[k]), err_msg=k)


@pytest.mark.parametrize("name", list(CASES))
def test_one_launch_equals_separate_steps_and_oracle(name):
    w = CASES[name]
    inp = W.generate(w)
    dev = Dev(inp)
    assert moe.moe_layer_decode_fused(desc_of(w))
    one = run_layer(dev)
    steps = run_layer(dev, flags=moe.MOE_FLAG_DECODE_SPLIT)
    assert one["device_error"] == 0 and steps["device_error"] == 0
    _same(one, steps)

    # the oracle, taking its top-k decisions on the GPU's fp32 scores
    r = run_stages(dev)
    gl = to_np(r["logits"]).astype(np.float64)
    ids_o, w_o, p_o = O.route(gl, w.K, w.temperature)
    d = oracle_dispatch(w, ids_o, gl)
    np.testing.assert_array_equal(to_np(one["count"]), d["count"])
    assert int(to_np(one["dropped"])[0]) == d["dropped"]
    aux_ref = O.aux_loss(p_o, d["count"], w.K)
    assert abs(float(to_np(one["aux"])[0]) - aux_ref) <= 1e-5 * max(1.0, abs(aux_ref))
    x64, Wg64 = O.widen(inp.x, w.dtype), O.widen(inp.Wg, w.dtype)
    ref = O.layer_forward(x64, Wg64, O.widen(inp.W1, w.dtype), O.widen(inp.W2, w.dtype), w.K,
                          capacity=w.capacity, gate_bias=inp.gate_bias,
                          b1=None if inp.b1 is None else inp.b1.astype(np.float64),
                          b2=None if inp.b2 is None else inp.b2.astype(np.float64),
                          bf16=True, logits=gl, temperature=w.temperature, act=w.act)
    # each element within 2e-2 plus one bf16 ulp of its value (the constructed
    # decode inputs give outputs where one ulp is most of 2e-2), rel-L2 1e-2
    out = as_f64(one["out"])
    mx, rel = out_errors(out, ref["out"])
    assert rel <= OUT_REL_L2_BF16, rel
    assert not (np.abs(out - ref["out"]) > OUT_MAXABS_BF16 + np.abs(ref["out"]) * 2.0 ** -7).any(), mx


def test_workspace_content_does_not_matter():
    """The counters are zeroed inside the call: a workspace full of ones
    (its error word read and cleared first) and one reused by earlier calls
    give the same bits."""
    import torch
    w = CASES["t16_routed"]
    dev = Dev(W.generate(w))
    ref = run_layer(dev)
    ws = moe.workspace(desc_of(w))
    ws.fill_(0xFF)
    moe.moe_get_device_error(ws)
    for _ in range(3):
        got = run_layer(dev, ws=ws)
        assert got["device_error"] == 0
        _same(got, ref)
    torch.cuda.synchronize()


def test_back_to_back_calls_on_one_stream():
    """Calls queued without a synchronisation in between (each call's counter
    reset waits for the call before it, which may still be running) give
    the results of the same calls made one at a time."""
    import torch
    base = CASES["t2_e8"]
    devs = [Dev(W.generate(W.Workload(**{**base.__dict__, "seed": s}))) for s in range(6)]
    alone = [run_layer(dv) for dv in devs]
    d = desc_of(base)
    ws = moe.workspace(d)
    outs = []
    for dv in devs:
        o = dict(out=torch.empty((base.T, base.H), dtype=torch.bfloat16, device="cuda"),
                 aux=torch.empty((1,), dtype=torch.float32, device="cuda"),
                 count=torch.empty((base.E,), dtype=torch.int32, device="cuda"),
                 dropped=torch.empty((1,), dtype=torch.int32, device="cuda"))
        moe.moe_layer_forward(d, dv.x, dv.Wg, dv.gb, dv.W1, dv.b1, dv.W2, dv.b2, o["out"], o["aux"], o["count"],
                              o["dropped"], ws)
        outs.append(o)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    for o, a in zip(outs, alone):
        _same(o, a)
