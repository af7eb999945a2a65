"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot
allocate device memory (allocator callbacks, runtimes that reserve all device
memory up front, hosts that forbid allocation on their execution path), gives
the same results as moe_dispatch, and as the oracle, on calls in a row.

The calls use different layers, so stale scratch left by one call would show
up in the next: the multi-block path with capacity drops, the one-block path
(at most 1024 slots), and a multi-block call with no error word.  Integer
outputs and the gathered rows must match bit for bit, as in every other
dispatch test.  This file is collected last so that a stop-at-first-failure
run has already run everything else."""
import ctypes

import numpy as np
import pytest

import sparse_mixture_experts_topk_gb300 as moe
from sparse_mixture_experts_topk_gb300 import workloads as W
from oracle import moe_oracle as O

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
    logits = torch.empty((w.T, w.E), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(d, dev.x, dev.Wg, dev.gb, logits, ids, wts, None, ws)
    return dev, d, ws, ids, logits


def _outputs(torch, w, dev):
    R = max(moe.moe_max_rows(moe.make_desc(w.T, w.H, w.E, w.K, w.F, w.capacity)), 1)
    return dict(count=torch.full((w.E,), -9, dtype=torch.int32, device="cuda"),
                offs=torch.full((w.E + 1,), -9, dtype=torch.int32, device="cuda"),
                src=torch.full((R,), -9, dtype=torch.int32, device="cuda"),
                pos=torch.full((w.T * w.K,), -9, dtype=torch.int32, device="cuda"),
                x_perm=torch.zeros((R, w.H), dtype=dev.x.dtype, device="cuda"),
                dropped=torch.full((1,), -9, dtype=torch.int32, device="cuda"))


CASES = [
    # multi-block, capacity drops, error word passed
    (W.small("na_first", T=3000, H=256, E=64, K=4, F=64, gate_bias="zipf",
             capacity=W.capacity_ceil(3000, 64, 4)), True),
    # one-block path (300 slots), error word passed
    (W.small("na_one_block", T=150, H=128, E=8, K=2, F=64, gate_bias="zipf",
             capacity=W.capacity_ceil(150, 8, 2) // 2), True),
    # multi-block, no capacity, no error word
    (W.small("na_second", T=700, H=128, E=16, K=2, F=64), False),
]


def test_noalloc_dispatch_matches_workspace_dispatch_and_oracle():
    torch = pytest.importorskip("torch")
    for w, with_err in CASES:
        inp = W.generate(w)
        dev, d, ws, ids, logits = _route(torch, w, inp)
        ref = _outputs(torch, w, dev)
        moe.moe_dispatch(d, ids, dev.x, ref["count"], ref["offs"], ref["src"], ref["pos"],
                         ref["x_perm"], ref["dropped"], ws)
        got = _outputs(torch, w, dev)
        err = torch.full((1,), -5, dtype=torch.int32, device="cuda") if with_err else None
        moe.moe_dispatch_noalloc(d, ids, dev.x, got["count"], got["offs"], got["src"], got["pos"],
                                 got["x_perm"], got["dropped"], err)
        torch.cuda.synchronize()
        R = int(ref["offs"][-1].item())
        if with_err:
            assert int(err.item()) == 0
        for k in ("count", "offs", "pos", "dropped"):
            assert torch.equal(got[k], ref[k]), (w.name, k)
        assert torch.equal(got["src"][:R], ref["src"][:R]), w.name
        assert torch.equal(got["x_perm"][:R], ref["x_perm"][:R]), w.name
        # and against the oracle's dispatch of the same routing
        ids_o, _, _ = O.route(logits.cpu().numpy().astype(np.float64), w.K, w.temperature)
        assert np.array_equal(ids.cpu().numpy(), ids_o), w.name
        o = O.dispatch(ids_o, w.E, w.capacity)
        for k in ("count", "offs", "pos"):
            assert np.array_equal(got[k].cpu().numpy(), o[k]), (w.name, k)
        assert np.array_equal(got["src"][:R].cpu().numpy(), o["src"]), w.name
        assert int(got["dropped"].item()) == o["dropped"], w.name
        xp = got["x_perm"][:R].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(xp, inp.x[o["src"] // w.K]), w.name
        if w.capacity > 0:
            assert o["dropped"] > 0


def test_noalloc_rejects_layers_beyond_its_scratch():
    """A layer whose per-block tables exceed the fixed scratch is refused
    before anything launches.  Every buffer is real and sized for the call, so
    a regression in the size check gives a wrong return code, never a fault."""
    torch = pytest.importorskip("torch")
    T, E, K = 100000, 256, 2                                  # 64 blocks x 256 experts
    d = moe.make_desc(T=T, H=64, E=E, K=K, F=64)
    R = moe.moe_max_rows(d)
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    ids[:, 1] = 1                                             # valid, distinct experts
    count = torch.empty((E,), dtype=torch.int32, device="cuda")
    offs = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    src = torch.empty((R,), dtype=torch.int32, device="cuda")
    pos = torch.empty((T * K,), dtype=torch.int32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    rc = moe.lib().moe_dispatch_noalloc(ctypes.byref(d), ids.data_ptr(), None, count.data_ptr(),
                                        offs.data_ptr(), src.data_ptr(), pos.data_ptr(), None, None,
                                        err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == -2                                           # MOE_ERR_UNSUPPORTED
