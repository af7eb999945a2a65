"""The first expert product reading its token rows from x (MOE_FLAG_GATHER_GEMM).

The layer then runs no gather kernel and never writes x_perm: the SM-pair
kernel's producer warp copies each kept row's token row (slot s = src[r] of
kept row r is token s / K) into the stage in the 128-byte swizzle itself.
Every tile multiplies the same operand values as from x_perm, so the output,
the counts and the loss equal the default layer's bit for bit: on every tile
shape (full row blocks, swapped and wide tails), with SwiGLU experts, with
capacity drops, with a hidden size whose last k-block is partly zero-filled,
with one launch per product, with row orientation forced, through host
buffers, and at the 8192-token layer.  One case is also checked against the
oracle directly."""
import numpy as np
import pytest

from sparse_mixture_experts_topk_gb300 import workloads as W
import sparse_mixture_experts_topk_gb300 as moe
from oracle import moe_oracle as O

from harness import Dev, run_layer, run_stages, desc_of, to_np, as_f64, out_errors, OUT_MAXABS_BF16, OUT_REL_L2_BF16

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": W.small("ragged", T=333, H=512, E=8, K=2, F=768),
    # 16 experts of about 190 rows: swapped and wide tails, most experts one block
    "tails": W.small("tails", T=1500, H=256, E=16, K=2, F=512),
    # every token on experts 0 and 1: three 256-row blocks each, the last short
    "hot2": W.small("hot2", T=700, H=256, E=8, K=2, F=384, gate_bias="hot"),
    "cap_zipf_k4": W.small("cap_zipf_k4", T=300, H=256, E=8, K=4, F=384,
                           capacity=W.capacity_ceil(300, 8, 4) // 2, gate_bias="zipf"),
    "swiglu": W.small("swiglu", T=333, H=512, E=8, K=2, F=384, act="swiglu", ffn_bias=True),
    # H = 200: the last 64-column k-block holds 8 columns, the rest zero-filled
    "h_ragged": W.small("h_ragged", T=300, H=200, E=8, K=2, F=264),
    "e64_k8": W.small("e64_k8", T=129, H=128, E=64, K=8, F=136),
}
BASE = moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_NO_DECODE
VARIANTS = {
    "one_launch": BASE,
    "split": BASE | moe.MOE_FLAG_FFN_SPLIT,
    "rows": BASE | moe.MOE_FLAG_GEMM_ROWS,
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
    np.testing.assert_array_equal(to_np(a["out"]), to_np(b["out"]))
    np.testing.assert_array_equal(to_np(a["count"]), to_np(b["count"]))
    np.testing.assert_array_equal(to_np(a["dropped"]), to_np(b["dropped"]))
    assert float(a["aux"].item()) == float(b["aux"].item())


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("name", list(CASES))
def test_gathered_first_product_equals_x_perm(name, variant):
    w = CASES[name]
    dev = Dev(W.generate(w))
    flags = VARIANTS[variant]
    plain = run_layer(dev, flags=flags)
    gath = run_layer(dev, flags=flags | moe.MOE_FLAG_GATHER_GEMM)
    assert plain["device_error"] == 0 and gath["device_error"] == 0
    _same(gath, plain)
    # one launch fewer: the gather kernel is gone (the one-block dispatch, for
    # at most 1024 slots and 256 KB of rows, gathers in its own launch and
    # skips that part)
    one_block = w.T * w.K <= 1024 and w.T * w.K * w.H * 2 <= 256 * 1024
    n_plain = moe.moe_layer_launches(desc_of(w, flags))
    n_gath = moe.moe_layer_launches(desc_of(w, flags | moe.MOE_FLAG_GATHER_GEMM))
    assert n_gath == n_plain - (0 if one_block else 1)


def test_gathered_layer_matches_oracle():
    w = CASES["tails"]
    inp = W.generate(w)
    dev = Dev(inp)
    gath = run_layer(dev, flags=BASE | moe.MOE_FLAG_GATHER_GEMM)
    assert gath["device_error"] == 0
    r = run_stages(dev, flags=BASE)   # the GPU's router scores decide the routing on both sides
    gl = to_np(r["logits"]).astype(np.float64)
    ref = O.layer_forward(O.widen(inp.x, w.dtype), O.widen(inp.Wg, w.dtype), O.widen(inp.W1, w.dtype),
                          O.widen(inp.W2, w.dtype), w.K, capacity=w.capacity, gate_bias=inp.gate_bias,
                          bf16=True, logits=gl, act=w.act)
    mx, rel = out_errors(as_f64(gath["out"]), ref["out"])
    assert mx <= OUT_MAXABS_BF16 and rel <= OUT_REL_L2_BF16, (mx, rel)
    np.testing.assert_array_equal(to_np(gath["count"]), ref["count"])


def test_reroute_ignores_the_flag():
    """drop_tokens=False dispatches twice; the flag does not apply there and
    the layer keeps its gather kernel."""
    w = W.small("reroute", T=300, H=256, E=8, K=4, F=384, capacity=W.capacity_ceil(300, 8, 4) // 2,
                gate_bias="zipf", reroute=True)
    dev = Dev(W.generate(w))
    plain = run_layer(dev, flags=BASE)
    gath = run_layer(dev, flags=BASE | moe.MOE_FLAG_GATHER_GEMM)
    assert plain["device_error"] == 0 and gath["device_error"] == 0
    _same(gath, plain)
    assert moe.moe_layer_launches(desc_of(w, BASE | moe.MOE_FLAG_GATHER_GEMM)) == \
        moe.moe_layer_launches(desc_of(w, BASE))


def test_host_io_gathered_equals_device_layer():
    """Host buffers in two pieces of tokens: each piece's first product
    gathers from the piece's staged x rows."""
    torch = pytest.importorskip("torch")
    w = W.small("io_gather", T=2501, H=256, E=8, K=2, F=384)
    dev = Dev(W.generate(w))
    ref = run_layer(dev)
    d = moe.make_desc(w.T, w.H, w.E, w.K, w.F, 0, moe.MOE_BF16, moe.MOE_FLAG_HOST_IO | moe.MOE_FLAG_GATHER_GEMM)
    ws = moe.workspace(d)
    xh = dev.x.cpu().pin_memory()
    outh = torch.full_like(xh, 7.0).pin_memory()
    moe.moe_layer_forward(d, xh, dev.Wg, None, dev.W1, None, dev.W2, None, outh, None, None, None, ws)
    torch.cuda.current_stream().synchronize()
    assert moe.moe_get_device_error(ws) == 0
    assert torch.equal(outh.view(torch.int16), ref["out"].cpu().view(torch.int16))


def test_prefill_layer_gathered_equals_x_perm():
    """The 8192-token layer (H=3584 E=32 k=2 F=2560): bit for bit."""
    w = W.WORKLOADS["prefill"]
    dev = Dev(W.generate(w))
    plain = run_layer(dev)
    gath = run_layer(dev, flags=moe.MOE_FLAG_GATHER_GEMM)
    assert plain["device_error"] == 0 and gath["device_error"] == 0
    _same(gath, plain)
