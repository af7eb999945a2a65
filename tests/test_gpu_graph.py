"""The layer call can be captured into a CUDA graph and replayed.

moe_layer_forward only enqueues work on the caller's stream: it never
allocates, never synchronises and never reads device data on the host, and
the tile counters of the expert GEMMs are reset by a kernel inside the call.
So a captured call must replay to the same bits as the eager call, also
after the input buffer has been rewritten in place."""
import numpy as np
import pytest

import sparse_mixture_experts_topk_gb300 as moe
from sparse_mixture_experts_topk_gb300 import workloads as W

from harness import Dev, desc_of, run_layer, to_np, tdtype

pytestmark = pytest.mark.gpu

CASES = {
    # tensor-core router with tile counts, scan+scatter, SM-pair GEMM
    "ragged_bf16": W.small("ragged_bf16", T=333, H=512, E=8, K=2, F=768),
    # the one-launch decode layer: one CTA per SM (4 tokens), two per SM (1 token)
    "decode4": W.small("decode4", T=4, H=512, E=16, K=2, F=256, x_kind="decode_distinct"),
    "decode1": W.small("decode1", T=1, H=512, E=32, K=2, F=256),
    # SwiGLU experts with capacity drops
    "swiglu_cap": W.small("swiglu_cap", T=300, H=256, E=8, K=2, F=384, act="swiglu",
                          capacity=W.capacity_ceil(300, 8, 2) // 2, gate_bias="zipf"),
    # drop_tokens=False: capacity-limited dispatch, the move, the dispatch of the moved routing
    "reroute": W.small("reroute", T=700, H=256, E=8, K=2, F=384, gate_bias="hot",
                       capacity=W.capacity_ceil(700, 8, 2), reroute=True),
}
# the combine folded into the second product's epilogue (flags on top of the case)
FLAGGED = {"fused_combine": ("ragged_bf16", moe.MOE_FLAG_FUSED_COMBINE)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_topk_gb300 import build
    build.build()
    moe.lib()


@pytest.mark.parametrize("name", list(CASES) + list(FLAGGED))
def test_captured_layer_replays_bit_exactly(name):
    import torch
    case, flags = FLAGGED.get(name, (name, 0))
    w = CASES[case]
    inp = W.generate(w)
    dev = Dev(inp)
    eager = run_layer(dev, flags=flags)
    assert eager["device_error"] == 0

    d = desc_of(w, flags)
    ws = moe.workspace(d)
    out = torch.empty((w.T, w.H), dtype=tdtype(w), device="cuda")
    aux = torch.empty((1,), dtype=torch.float32, device="cuda")
    count = torch.empty((w.E,), dtype=torch.int32, device="cuda")
    dropped = torch.empty((1,), dtype=torch.int32, device="cuda")

    def call():
        moe.moe_layer_forward(d, dev.x, dev.Wg, dev.gb, dev.W1, dev.b1, dev.W2, dev.b2, out, aux, count,
                              dropped, ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # one eager call outside the capture
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(3):
        out.zero_()
        aux.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    np.testing.assert_array_equal(to_np(out), to_np(eager["out"]))
    np.testing.assert_array_equal(to_np(count), to_np(eager["count"]))
    np.testing.assert_array_equal(to_np(dropped), to_np(eager["dropped"]))
    np.testing.assert_array_equal(to_np(aux), to_np(eager["aux"]))

    # new input values in the captured buffer: the replay follows them
    inp2 = W.generate(W.Workload(**{**w.__dict__, "seed": w.seed + 7}))
    dev2 = Dev(inp2)
    dev.x.copy_(dev2.x)
    g.replay()
    torch.cuda.synchronize()
    eager2 = run_layer(dev, flags=flags)
    np.testing.assert_array_equal(to_np(out), to_np(eager2["out"]))
