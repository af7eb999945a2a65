"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot
allocate device memory (allocator callbacks, runtimes that reserve all device
memory up front, hosts that forbid allocation on their execution path), gives
the same results as moe_dispatch on two calls in a row.

The two calls use different layers, so stale scratch left by the first call
would show up in the second.  Integer outputs and the gathered rows must match
bit for bit, as in every other dispatch test.  This file is collected last so
that a stop-at-first-failure run has already run everything else."""
import ctypes

import numpy as np
import pytest

import sparse_mixture_experts_topk_gb300 as moe
from sparse_mixture_experts_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_topk_gb300 import build
    build.build()
    moe.lib()


def _route(torch, w, inp):
    from harness import Dev, desc_of
    dev = Dev(inp)
    d = desc_of(w)
    ws = moe.workspace(d)
    ids = torch.empty((w.T, w.K), dtype=torch.int32, device="cuda")
    wts = torch.empty((w.T, w.K), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(d, dev.x, dev.Wg, dev.gb, None, ids, wts, None, ws)
    return dev, d, ws, ids


def _outputs(torch, w, dev):
    R = max(moe.moe_max_rows(moe.make_desc(w.T, w.H, w.E, w.K, w.F, w.capacity)), 1)
    return dict(count=torch.full((w.E,), -9, dtype=torch.int32, device="cuda"),
                offs=torch.full((w.E + 1,), -9, dtype=torch.int32, device="cuda"),
                src=torch.full((R,), -9, dtype=torch.int32, device="cuda"),
                pos=torch.full((w.T * w.K,), -9, dtype=torch.int32, device="cuda"),
                x_perm=torch.zeros((R, w.H), dtype=dev.x.dtype, device="cuda"),
                dropped=torch.full((1,), -9, dtype=torch.int32, device="cuda"))


def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    torch = pytest.importorskip("torch")
    cases = [
        W.small("na_first", T=3000, H=256, E=64, K=4, F=64, gate_bias="zipf",
                capacity=W.capacity_ceil(3000, 64, 4)),
        W.small("na_second", T=700, H=128, E=16, K=2, F=64),
    ]
    for w in cases:
        inp = W.generate(w)
        dev, d, ws, ids = _route(torch, w, inp)
        ref = _outputs(torch, w, dev)
        moe.moe_dispatch(d, ids, dev.x, ref["count"], ref["offs"], ref["src"], ref["pos"],
                         ref["x_perm"], ref["dropped"], ws)
        got = _outputs(torch, w, dev)
        err = torch.full((1,), -5, dtype=torch.int32, device="cuda")
        moe.moe_dispatch_noalloc(d, ids, dev.x, got["count"], got["offs"], got["src"], got["pos"],
                                 got["x_perm"], got["dropped"], err)
        torch.cuda.synchronize()
        R = int(ref["offs"][-1].item())
        assert int(err.item()) == 0
        for k in ("count", "offs", "pos", "dropped"):
            assert torch.equal(got[k], ref[k]), (w.name, k)
        assert torch.equal(got["src"][:R], ref["src"][:R]), w.name
        assert torch.equal(got["x_perm"][:R], ref["x_perm"][:R]), w.name
        if w.capacity > 0:
            assert int(ref["dropped"].item()) > 0


def test_noalloc_rejects_layers_beyond_its_scratch():
    lib = moe.lib()
    d = moe.make_desc(T=100000, H=64, E=256, K=2, F=64)     # 64 blocks x 256 experts
    A = 1 << 20
    rc = lib.moe_dispatch_noalloc(ctypes.byref(d), A, None, A, A, A, A, None, None, None, None)
    assert rc == -2                                           # MOE_ERR_UNSUPPORTED
