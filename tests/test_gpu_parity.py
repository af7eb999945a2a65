"""GPU parity: every entry point of the CUDA library against the fp64 oracle on
the same seeded inputs.

Integer results (expert ids, counts, offsets, the permutation, dropped slots)
are compared bit-exactly, with the oracle's routing fed the GPU's own fp32
router scores so that both sides take every top-k decision on the same
numbers.  Floating-point results use the tolerances in ``harness``:
  scores        max|d| / max|ref| per row <= 1e-4
  weights       |d| <= 2e-6 (fp32 softmax of the same scores)
  h, y (bf16)   |d| <= 2^-7 |ref| + 1e-6 (one bf16 ulp: the rounding of an
                fp32 vs fp64 accumulation can land on either neighbour)
  out           max-abs <= 2e-2 and rel-L2 <= 1e-2 against the oracle whose
                h and y are rounded to bf16 (fp32 layers: rel-L2 <= 1e-4)
"""
import numpy as np
import pytest

from sparse_mixture_experts_topk_gb300 import workloads as W
import sparse_mixture_experts_topk_gb300 as moe
from oracle import moe_oracle as O

from harness import (Dev, run_stages, run_layer, to_np, as_f64, logits_rel_err, out_errors, oracle_dispatch,
                     LOGITS_REL, W_ABS, PSUM_REL, OUT_MAXABS_BF16, OUT_REL_L2_BF16, OUT_REL_L2_F32)

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny_f32": W.WORKLOADS["tiny"],
    "ragged_bf16": W.small("ragged_bf16", T=333, H=512, E=8, K=2, F=768),
    "cap_zipf_k4": W.small("cap_zipf_k4", T=300, H=256, E=8, K=4, F=384,
                           capacity=W.capacity_ceil(300, 8, 4) // 2, gate_bias="zipf"),
    "ffn_bias": W.small("ffn_bias", T=200, H=256, E=16, K=2, F=256, ffn_bias=True, gate_bias="zipf"),
    "e64_k8": W.small("e64_k8", T=129, H=128, E=64, K=8, F=136),
    "e256_k3": W.small("e256_k3", T=70, H=64, E=256, K=3, F=64),
    "f32_ragged": W.small("f32_ragged", T=150, H=96, E=6, K=2, F=200, dtype=W.F32, ffn_bias=True),
    "decode4": W.small("decode4", T=4, H=512, E=16, K=2, F=256, x_kind="decode_distinct"),
    "one_token": W.small("one_token", T=1, H=256, E=8, K=2, F=128),
    "k1": W.small("k1", T=96, H=128, E=4, K=1, F=64),
    "k_eq_e": W.small("k_eq_e", T=40, H=64, E=4, K=4, F=64),
    "hot_router": W.small("hot_router", T=260, H=256, E=16, K=2, F=128, temperature=2.0),
    "cold_router_f32": W.small("cold_router_f32", T=90, H=64, E=8, K=3, F=64, dtype=W.F32, temperature=0.5),
    "swiglu_ragged": W.small("swiglu_ragged", T=333, H=512, E=8, K=2, F=384, act="swiglu", ffn_bias=True),
    "swiglu_f32": W.small("swiglu_f32", T=120, H=96, E=6, K=2, F=136, dtype=W.F32, act="swiglu"),
    # decode-sized batch (weight-streaming kernel) with x ~ N(0,1): the
    # distinct-expert construction scales x by 64, and SiLU(g) * u would square
    # that into outputs whose bf16 storage alone exceeds the 2e-2 bound
    "swiglu_decode": W.small("swiglu_decode", T=4, H=512, E=16, K=2, F=200, act="swiglu"),
    # one-block dispatch: capacity drops; exactly its slot limit (1024 slots,
    # 256 KB of rows); one slot pair past it (multi-block path)
    "small_cap": W.small("small_cap", T=100, H=128, E=8, K=2, F=64,
                         capacity=W.capacity_ceil(100, 8, 2) // 2, gate_bias="zipf"),
    "slots_1024": W.small("slots_1024", T=512, H=128, E=8, K=2, F=64),
    "slots_1026": W.small("slots_1026", T=513, H=128, E=8, K=2, F=64),
    # small-batch router with the widest cluster (8 CTAs, 4 gate rows a warp)
    "tiny_e256_k8": W.small("tiny_e256_k8", T=5, H=64, E=256, K=8, F=64),
    # every token picks both experts: 16-row segments, the largest streaming body
    "decode16_all": W.small("decode16_all", T=16, H=256, E=2, K=2, F=128),
    # every token to experts 0 and 1: long segments (three 256-row blocks, the
    # last one short), six empty experts
    "hot2": W.small("hot2", T=700, H=256, E=8, K=2, F=384, gate_bias="hot"),
    "hot2_cap": W.small("hot2_cap", T=700, H=256, E=8, K=2, F=384, gate_bias="hot",
                        capacity=W.capacity_ceil(700, 8, 2)),
    # fp32 decode-sized batches: the CUDA-core router and the fp32 streaming kernel
    "decode_f32": W.small("decode_f32", T=3, H=96, E=6, K=2, F=64, dtype=W.F32, ffn_bias=True),
    "swiglu_decode_f32": W.small("swiglu_decode_f32", T=6, H=128, E=8, K=3, F=72, dtype=W.F32, act="swiglu"),
    # hidden size not a multiple of the 64-wide k-block: the tensor-core router's and the first
    # expert product's last k-block is partly zero-filled
    "h_ragged": W.small("h_ragged", T=300, H=200, E=8, K=2, F=264),
    "h_ragged_decode": W.small("h_ragged_decode", T=5, H=200, E=8, K=2, F=264),
    # drop_tokens=False: the slots over capacity move to the next-best expert with room
    "reroute_k4": W.small("reroute_k4", T=300, H=256, E=8, K=4, F=384,
                          capacity=W.capacity_ceil(300, 8, 4) // 2, gate_bias="zipf", reroute=True),
    # every token prefers experts 0 and 1: most slots move, in score order, to the other experts
    "reroute_hot2": W.small("reroute_hot2", T=700, H=256, E=8, K=2, F=384, gate_bias="hot",
                            capacity=W.capacity_ceil(700, 8, 2), reroute=True),
    # one-block dispatch on both sides of the move
    "reroute_small": W.small("reroute_small", T=100, H=128, E=8, K=2, F=64,
                             capacity=W.capacity_ceil(100, 8, 2) // 2, gate_bias="zipf", reroute=True),
    # many experts, top-8: many epochs of the move
    "reroute_e64_k8": W.small("reroute_e64_k8", T=700, H=128, E=64, K=8, F=64, gate_bias="zipf",
                              capacity=W.capacity_ceil(700, 64, 8) // 2, reroute=True),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_topk_gb300 import build
    build.build()
    moe.lib()


def _ulp_tol(ref):
    return np.abs(ref) * 2.0 ** -7 + 1e-6


def _check_routing(w, inp, r, x64, Wg64):
    """Router scores, ids, weights and probability sums."""
    gl = to_np(r["logits"]).astype(np.float64)
    ref_l = O.gate_logits(x64, Wg64, inp.gate_bias)
    assert logits_rel_err(gl, ref_l) <= LOGITS_REL
    ids_o, w_o, p_o = O.route(gl, w.K, w.temperature)
    np.testing.assert_array_equal(to_np(r["ids"]), ids_o)
    np.testing.assert_allclose(to_np(r["w"]), w_o, rtol=0, atol=W_ABS)
    ps = p_o.sum(axis=0)
    np.testing.assert_allclose(to_np(r["psum"]), ps, rtol=PSUM_REL, atol=1e-6)
    return gl, ids_o, w_o, p_o


def _check_dispatch(w, r, ids_o, x_bytes, scores):
    d = oracle_dispatch(w, ids_o, scores)
    if "ids_final" in r:
        np.testing.assert_array_equal(to_np(r["ids_final"]), d["final"])
    np.testing.assert_array_equal(to_np(r["count"]), d["count"])
    np.testing.assert_array_equal(to_np(r["offs"]), d["offs"])
    R = int(d["offs"][-1])
    np.testing.assert_array_equal(to_np(r["src"])[:R], d["src"])
    np.testing.assert_array_equal(to_np(r["pos"]), d["pos"])
    assert int(to_np(r["dropped"])[0]) == d["dropped"]
    xp = to_np(r["x_perm"])[:R]
    np.testing.assert_array_equal(xp, x_bytes[d["src"] // w.K])
    return d


@pytest.mark.parametrize("name", list(SMALL))
def test_stages_and_layer_small(name):
    w = SMALL[name]
    inp = W.generate(w)
    dev = Dev(inp)
    bf = w.dtype == W.BF16
    x64, Wg64 = O.widen(inp.x, w.dtype), O.widen(inp.Wg, w.dtype)
    W164, W264 = O.widen(inp.W1, w.dtype), O.widen(inp.W2, w.dtype)
    r = run_stages(dev)
    assert r["device_error"] == 0
    gl, ids_o, w_o, p_o = _check_routing(w, inp, r, x64, Wg64)
    d = _check_dispatch(w, r, ids_o, inp.x, gl)
    R = int(d["offs"][-1])

    # expert FFN, one product at a time
    xp = as_f64(r["x_perm"])[:R]
    h_gpu = as_f64(r["h_perm"])[:R]
    y_gpu = as_f64(r["y_perm"])[:R]
    for e in range(w.E):
        a, b = int(d["offs"][e]), int(d["offs"][e + 1])
        if a == b:
            continue
        b1 = None if inp.b1 is None else inp.b1[e].astype(np.float64)
        b2 = None if inp.b2 is None else inp.b2[e].astype(np.float64)
        pre = xp[a:b] @ W164[e].T + (0 if b1 is None else b1)
        h_ref = O.silu(pre[:, :w.F]) * pre[:, w.F:] if w.act == "swiglu" else O.gelu(pre)
        y_ref = h_gpu[a:b] @ W264[e].T + (0 if b2 is None else b2)
        if bf:
            h_ref, y_ref = O.round_bf16(h_ref), O.round_bf16(y_ref)
            assert (np.abs(h_gpu[a:b] - h_ref) <= _ulp_tol(h_ref)).all(), name
            assert (np.abs(y_gpu[a:b] - y_ref) <= _ulp_tol(y_ref)).all(), name
        else:
            np.testing.assert_allclose(h_gpu[a:b], h_ref, rtol=1e-5, atol=1e-5)
            np.testing.assert_allclose(y_gpu[a:b], y_ref, rtol=1e-5, atol=1e-5)

    # combine of the GPU's own expert outputs
    out_gpu = as_f64(r["out"])
    out_ref = O.combine(y_gpu, d["pos"], w_o)
    tol = (np.abs(out_ref) * 2.0 ** -8 + 1e-5) if bf else (np.abs(out_ref) * 1e-6 + 1e-6)
    assert (np.abs(out_gpu - out_ref) <= tol).all()
    # load-balancing loss
    aux_ref = O.aux_loss(p_o, d["count"], w.K)
    assert abs(float(to_np(r["aux"])[0]) - aux_ref) <= 1e-5 * max(1.0, abs(aux_ref))

    # the whole layer: identical to the stages, and within tolerance of the oracle
    L = run_layer(dev)
    assert L["device_error"] == 0
    np.testing.assert_array_equal(to_np(L["out"]), to_np(r["out"]))
    np.testing.assert_array_equal(to_np(L["count"]), d["count"])
    assert int(to_np(L["dropped"])[0]) == d["dropped"]
    assert abs(float(to_np(L["aux"])[0]) - aux_ref) <= 1e-5 * max(1.0, abs(aux_ref))
    ref = O.layer_forward(x64, Wg64, W164, W264, w.K, capacity=w.capacity, gate_bias=inp.gate_bias,
                          b1=None if inp.b1 is None else inp.b1.astype(np.float64),
                          b2=None if inp.b2 is None else inp.b2.astype(np.float64),
                          bf16=bf, logits=gl, temperature=w.temperature, act=w.act,
                          reroute_over=w.reroute)
    mx, rel = out_errors(out_gpu, ref["out"])
    if bf:
        assert mx <= OUT_MAXABS_BF16 and rel <= OUT_REL_L2_BF16, (mx, rel)
    else:
        assert rel <= OUT_REL_L2_F32, rel


def test_layer_is_deterministic():
    w = SMALL["cap_zipf_k4"]
    dev = Dev(W.generate(w))
    a = run_layer(dev)
    b = run_layer(dev)
    np.testing.assert_array_equal(to_np(a["out"]), to_np(b["out"]))
    assert to_np(a["aux"])[0] == to_np(b["aux"])[0]


def test_all_logits_tied_pick_lowest_experts():
    w = W.small("tied", T=50, H=64, E=8, K=3, F=64)
    inp = W.generate(w)
    inp.Wg[:] = 0                       # every score is 0
    r = run_stages(Dev(inp))
    ids = to_np(r["ids"])
    assert (ids == np.arange(3)[None, :]).all()
    np.testing.assert_allclose(to_np(r["w"]), 1.0 / 3.0, atol=1e-7)
    assert float(to_np(r["aux"])[0]) == pytest.approx(1.0, abs=1e-6)   # uniform P -> L = 1


def test_empty_batch():
    w = W.small("empty", T=0, H=64, E=4, K=2, F=64)
    inp = W.generate(w)
    dev = Dev(inp)
    r = run_stages(dev)
    assert (to_np(r["count"]) == 0).all() and (to_np(r["offs"]) == 0).all()
    L = run_layer(dev)
    assert L["out"].numel() == 0 and int(to_np(L["dropped"])[0]) == 0


@pytest.mark.parametrize("name", ["ragged_bf16", "one_token", "decode4"])
def test_host_io_layer_matches_device_layer(name):
    """Host x and out, copied through the workspace: the device layer's bits
    (the multi-block path, and decode-sized batches on the one-launch layer)."""
    torch = pytest.importorskip("torch")
    w = SMALL[name]
    dev = Dev(W.generate(w))
    ref = run_layer(dev)
    d = moe.make_desc(w.T, w.H, w.E, w.K, w.F, w.capacity, moe.MOE_BF16, moe.MOE_FLAG_HOST_IO)
    ws = moe.workspace(d)
    xh = dev.x.cpu().pin_memory()
    outh = torch.empty_like(xh).pin_memory()
    aux = torch.empty(1, device="cuda")
    moe.moe_layer_forward(d, xh, dev.Wg, None, dev.W1, None, dev.W2, None, outh, aux, None, None, ws)
    torch.cuda.synchronize()
    assert torch.equal(outh.view(torch.int16), ref["out"].cpu().view(torch.int16))


@pytest.mark.parametrize("name", ["ragged_bf16", "hot2_cap", "swiglu_ragged", "e64_k8", "cap_zipf_k4", "h_ragged"])
def test_fused_combine_matches_oracle(name):
    """MOE_FLAG_FUSED_COMBINE: the weighted combine in the second product's
    epilogue (fp32 vector reductions onto a zeroed copy of out), for K <= 2 on
    the SM-pair kernels; other layers ignore the flag.  Against the oracle
    like the plain layer, and within one bf16 ulp of it (the two add the same
    rounded products in fp32, one with a fused multiply-add)."""
    w = SMALL[name]
    inp = W.generate(w)
    dev = Dev(inp)
    plain = run_layer(dev, flags=moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_NO_DECODE)
    fused = run_layer(dev, flags=moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_NO_DECODE | moe.MOE_FLAG_FUSED_COMBINE)
    assert plain["device_error"] == 0 and fused["device_error"] == 0
    a, b = as_f64(fused["out"]), as_f64(plain["out"])
    # one bf16 ulp, or the fp32 rounding of the two products where they cancel
    assert (np.abs(a - b) <= np.abs(b) * 2.0 ** -7 + 1e-6).all()
    if w.K > 2:
        np.testing.assert_array_equal(to_np(fused["out"]), to_np(plain["out"]))   # not fused: same path
    np.testing.assert_array_equal(to_np(fused["count"]), to_np(plain["count"]))
    r = run_stages(dev, flags=moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_NO_DECODE)
    gl = to_np(r["logits"]).astype(np.float64)
    ref = O.layer_forward(O.widen(inp.x, w.dtype), O.widen(inp.Wg, w.dtype), O.widen(inp.W1, w.dtype),
                          O.widen(inp.W2, w.dtype), w.K, capacity=w.capacity, gate_bias=inp.gate_bias,
                          b1=None if inp.b1 is None else inp.b1.astype(np.float64),
                          b2=None if inp.b2 is None else inp.b2.astype(np.float64),
                          bf16=True, logits=gl, act=w.act)
    mx, rel = out_errors(a, ref["out"])
    assert mx <= OUT_MAXABS_BF16 and rel <= OUT_REL_L2_BF16, (mx, rel)


@pytest.mark.parametrize("T", [2048, 2501])
def test_chunked_host_io_layer_matches_device_layer(T):
    """With host buffers and no capacity the call runs the batch in two
    pieces of tokens, each piece's copies overlapping the other's layer: the
    output is the device layer's bit for bit (a token's output depends on its
    own row only), the counts are equal and the loss is the whole batch's."""
    torch = pytest.importorskip("torch")
    w = W.small("io_chunks", T=T, H=256, E=8, K=2, F=384)
    dev = Dev(W.generate(w))
    ref = run_layer(dev)
    d = moe.make_desc(w.T, w.H, w.E, w.K, w.F, 0, moe.MOE_BF16, moe.MOE_FLAG_HOST_IO)
    ws = moe.workspace(d)
    xh = dev.x.cpu().pin_memory()
    outh = torch.full_like(xh, 7.0).pin_memory()
    aux = torch.full((1,), -1.0, device="cuda")
    count = torch.full((w.E,), -1, dtype=torch.int32, device="cuda")
    dropped = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    moe.moe_layer_forward(d, xh, dev.Wg, None, dev.W1, None, dev.W2, None, outh, aux, count, dropped, ws)
    torch.cuda.current_stream().synchronize()
    assert moe.moe_get_device_error(ws) == 0
    assert torch.equal(outh.view(torch.int16), ref["out"].cpu().view(torch.int16))
    assert torch.equal(count, ref["count"]) and int(dropped.item()) == 0
    assert float(aux.item()) == pytest.approx(float(ref["aux"].item()), rel=2e-6)
    # a second call on the same workspace and streams gives the same bits
    outh2 = torch.empty_like(xh).pin_memory()
    moe.moe_layer_forward(d, xh, dev.Wg, None, dev.W1, None, dev.W2, None, outh2, None, None, None, ws)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(outh2.view(torch.int16), outh.view(torch.int16))


@pytest.mark.parametrize("name", ["ragged_bf16", "e64_k8", "cap_zipf_k4"])
def test_cuda_core_router_and_ffn_match_oracle(name):
    """The CUDA-core router and expert FFN (kept for fp32 layers and as a
    cross-check) on bf16 layers, against the same oracle checks."""
    w = SMALL[name]
    inp = W.generate(w)
    dev = Dev(inp)
    x64, Wg64 = O.widen(inp.x, w.dtype), O.widen(inp.Wg, w.dtype)
    r = run_stages(dev, flags=moe.MOE_FLAG_SIMT_ROUTER | moe.MOE_FLAG_SIMT_FFN)
    assert r["device_error"] == 0
    gl, ids_o, w_o, p_o = _check_routing(w, inp, r, x64, Wg64)
    d = _check_dispatch(w, r, ids_o, inp.x, gl)
    ref = O.layer_forward(x64, Wg64, O.widen(inp.W1, w.dtype), O.widen(inp.W2, w.dtype), w.K,
                          capacity=w.capacity, gate_bias=inp.gate_bias, bf16=True, logits=gl)
    mx, rel = out_errors(as_f64(r["out"]), ref["out"])
    assert mx <= OUT_MAXABS_BF16 and rel <= OUT_REL_L2_BF16, (mx, rel)
    # and the tensor-core path picks the same experts from its own scores
    r2 = run_stages(dev)
    gl2 = to_np(r2["logits"]).astype(np.float64)
    assert logits_rel_err(gl2, gl) <= 2 * LOGITS_REL


def test_heavily_tied_scores_route_like_the_oracle():
    """Small-integer x and gate weights make the fp32 scores exact integers
    with many equal values; the expert ids must still match the oracle's
    (score descending, index ascending) order exactly, on both routers."""
    w = W.small("ties", T=700, H=64, E=16, K=4, F=64)
    inp = W.generate(w)
    rng = np.random.default_rng(99)
    inp.x[:] = W.f32_to_bf16_bits(rng.integers(-1, 2, size=inp.x.shape).astype(np.float32))
    inp.Wg[:] = W.f32_to_bf16_bits(rng.integers(-1, 2, size=inp.Wg.shape).astype(np.float32))
    dev = Dev(inp)
    for flags in (0, moe.MOE_FLAG_SIMT_ROUTER):
        r = run_stages(dev, flags=flags)
        gl = to_np(r["logits"]).astype(np.float64)
        ref = O.gate_logits(O.widen(inp.x, "bf16"), O.widen(inp.Wg, "bf16"))
        np.testing.assert_array_equal(gl, ref)                 # exact integers
        ids_o, w_o, _ = O.route(gl, w.K)
        np.testing.assert_array_equal(to_np(r["ids"]), ids_o)
        np.testing.assert_allclose(to_np(r["w"]), w_o, rtol=0, atol=W_ABS)
        srt = np.sort(gl, axis=1)
        assert (srt[:, :-1] == srt[:, 1:]).any(axis=1).mean() > 0.9   # ties everywhere


@pytest.mark.parametrize("kind", ["single", "pair", "pair_rows", "pair_split"])
@pytest.mark.parametrize("name", ["ragged_bf16", "e64_k8", "ffn_bias", "cap_zipf_k4", "e256_k3", "one_token",
                                  "swiglu_ragged", "h_ragged"])
def test_expert_gemm_kernels_match_oracle(name, kind):
    """The tensor-core GEMM kernels (128x256 tiles per SM; SM pairs with the
    token rows on the MMA's N side, the default, or on its M side; SM pairs
    with both products in one launch, the default, or one launch each)
    against the oracle, product by product, and the layer output."""
    w = SMALL[name]
    inp = W.generate(w)
    dev = Dev(inp)
    flag = {"single": moe.MOE_FLAG_GEMM_SINGLE, "pair": moe.MOE_FLAG_GEMM_PAIR,
            "pair_rows": moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_GEMM_ROWS,
            "pair_split": moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_FFN_SPLIT}[kind]
    flags = flag | moe.MOE_FLAG_NO_DECODE
    r = run_stages(dev, flags=flags)
    assert r["device_error"] == 0
    x64, Wg64 = O.widen(inp.x, w.dtype), O.widen(inp.Wg, w.dtype)
    gl, ids_o, w_o, p_o = _check_routing(w, inp, r, x64, Wg64)
    d = _check_dispatch(w, r, ids_o, inp.x, gl)
    R = int(d["offs"][-1])
    W164, W264 = O.widen(inp.W1, w.dtype), O.widen(inp.W2, w.dtype)
    xp, h_gpu, y_gpu = as_f64(r["x_perm"])[:R], as_f64(r["h_perm"])[:R], as_f64(r["y_perm"])[:R]
    for e in range(w.E):
        a, b = int(d["offs"][e]), int(d["offs"][e + 1])
        if a == b:
            continue
        b1 = 0 if inp.b1 is None else inp.b1[e].astype(np.float64)
        b2 = 0 if inp.b2 is None else inp.b2[e].astype(np.float64)
        pre = xp[a:b] @ W164[e].T + b1
        h_ref = O.round_bf16(O.silu(pre[:, :w.F]) * pre[:, w.F:] if w.act == "swiglu" else O.gelu(pre))
        y_ref = O.round_bf16(h_gpu[a:b] @ W264[e].T + b2)
        assert (np.abs(h_gpu[a:b] - h_ref) <= _ulp_tol(h_ref)).all(), (name, kind, e)
        assert (np.abs(y_gpu[a:b] - y_ref) <= _ulp_tol(y_ref)).all(), (name, kind, e)
    L = run_layer(dev, flags=flags)
    assert L["device_error"] == 0
    np.testing.assert_array_equal(to_np(L["out"]), to_np(r["out"]))
    ref = O.layer_forward(x64, Wg64, W164, W264, w.K, capacity=w.capacity, gate_bias=inp.gate_bias,
                          b1=None if inp.b1 is None else inp.b1.astype(np.float64),
                          b2=None if inp.b2 is None else inp.b2.astype(np.float64),
                          bf16=True, logits=gl, act=w.act)
    mx, rel = out_errors(as_f64(L["out"]), ref["out"])
    assert mx <= OUT_MAXABS_BF16 and rel <= OUT_REL_L2_BF16, (mx, rel)


@pytest.mark.parametrize("name", ["ragged_bf16", "cap_zipf_k4", "swiglu_ragged", "hot2", "hot2_cap", "e64_k8"])
def test_fused_pair_products_equal_split_launches(name):
    """One launch for both SM-pair products (second-product tiles wait on
    their row block's counter) gives the same bits as one launch per
    product: every tile computes the same sums in the same order; only when
    they run changes."""
    w = SMALL[name]
    dev = Dev(W.generate(w))
    base = moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_NO_DECODE
    fused = run_stages(dev, flags=base)
    split = run_stages(dev, flags=base | moe.MOE_FLAG_FFN_SPLIT)
    assert fused["device_error"] == 0 and split["device_error"] == 0
    R = int(to_np(fused["offs"])[-1])
    for key in ("h_perm", "y_perm"):
        np.testing.assert_array_equal(to_np(fused[key])[:R], to_np(split[key])[:R], err_msg=key)
    np.testing.assert_array_equal(to_np(fused["out"]), to_np(split["out"]))


@pytest.mark.parametrize("name", ["decode4", "one_token", "decode16_all", "swiglu_decode", "decode_f32",
                                  "swiglu_decode_f32"])
def test_streamed_products_in_one_launch_equal_two_launches(name):
    """Decode-sized batches: both weight-streaming products in one launch
    (the second's activation rows wait on the expert's counter) give the same
    bits as one launch per product."""
    w = SMALL[name]
    dev = Dev(W.generate(w))
    one = run_stages(dev, flags=0)
    two = run_stages(dev, flags=moe.MOE_FLAG_FFN_SPLIT)
    assert one["device_error"] == 0 and two["device_error"] == 0
    R = int(to_np(one["offs"])[-1])
    for key in ("h_perm", "y_perm"):
        np.testing.assert_array_equal(to_np(one[key])[:R], to_np(two[key])[:R], err_msg=key)
    np.testing.assert_array_equal(to_np(one["out"]), to_np(two["out"]))
    L = run_layer(dev, flags=0)
    assert L["device_error"] == 0
    np.testing.assert_array_equal(to_np(L["out"]), to_np(one["out"]))


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("name", ["ragged_bf16", "cap_zipf_k4", "e64_k8", "hot2", "hot2_cap", "swiglu_ragged",
                                  "h_ragged", "e256_k3"])
def test_layer_equals_separate_steps_on_pair_gemm(name, split):
    """The layer call (router, dispatch, both SM-pair expert products, the
    combine chained by programmatic launch) and the separate entry points
    (moe_router_topk, moe_dispatch, moe_expert_ffn, moe_combine) compute the
    same sums in the same order: the outputs are equal bit for bit, with one
    launch for both products or one per product, empty experts, capacity
    drops and up to 8 slots a token."""
    w = SMALL[name]
    dev = Dev(W.generate(w))
    flags = moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_NO_DECODE | (moe.MOE_FLAG_FFN_SPLIT if split else 0)
    lay = run_layer(dev, flags=flags)
    stg = run_stages(dev, flags=flags)
    assert lay["device_error"] == 0 and stg["device_error"] == 0
    np.testing.assert_array_equal(to_np(lay["out"]), to_np(stg["out"]))
    np.testing.assert_array_equal(to_np(lay["count"]), to_np(stg["count"]))
