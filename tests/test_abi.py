"""The C ABI library loads, exports every symbol include/moe.h declares, and
rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

import sparse_mixture_experts_topk_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from sparse_mixture_experts_topk_gb300 import build
    build.build()
    return moe.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "moe_layer_forward" in names and len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
        # the binding exposes the same name
        assert hasattr(moe, n), n


def test_header_constants_match_the_binding():
    """Every flag, status and expert-FFN kind that include/moe.h defines has
    the same name and value in the Python binding (parsed from the header's
    text, so a constant added on one side only fails here)."""
    hdr = open(os.path.join(ROOT, "include", "moe.h")).read()
    defs = {n: int(a) << int(b or 0) for n, a, b in
            re.findall(r"#define (MOE_(?:FLAG|FFN)_\w+)\s+\(?(\d+)u?(?:\s*<<\s*(\d+))?", hdr)}
    enums = {n: int(v) for n, v in re.findall(r"\b(MOE_(?:OK|ERR_\w+))\s*=\s*(-?\d+)", hdr)}
    assert len(defs) >= 20 and len(enums) == 7
    for n, v in {**defs, **enums}.items():
        assert getattr(moe, n) == v, n
        assert n in moe.__all__, n


def test_capacity_and_rows(lib):
    assert moe.moe_capacity_default(8192, 32, 2) == 512
    assert moe.moe_capacity_default(16384, 32, 4) == 2048
    assert moe.moe_capacity_default(1, 32, 2) == 2
    assert moe.moe_capacity_default(10, 0, 2) == -1
    d = moe.make_desc(16384, 3584, 32, 4, 2560, capacity=2048)
    assert moe.moe_max_rows(d) == 65536
    d = moe.make_desc(16384, 3584, 32, 4, 2560, capacity=100)
    assert moe.moe_max_rows(d) == 3200
    d = moe.make_desc(8192, 3584, 32, 2, 2560)
    assert moe.moe_max_rows(d) == 16384


def test_workspace_size_grows_with_shape(lib):
    a = moe.moe_workspace_size(moe.make_desc(64, 256, 8, 2, 512))
    b = moe.moe_workspace_size(moe.make_desc(8192, 3584, 32, 2, 2560))
    c = moe.moe_workspace_size(moe.make_desc(8192, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_HOST_IO))
    assert 0 < a < b < c
    # x_perm + h_perm dominate: rows * (H + F) * 2 bytes
    assert b >= 16384 * (3584 + 2560) * 2


def test_layer_launch_count(lib):
    """The kernels one layer call issues, from the shape: router, dispatch
    (one block for a small batch; scan+scatter and gather when the router
    counted its tiles; else histogram, scan, scatter, gather), the expert
    products (one launch on SM pairs, else one per product), combine."""
    prefill = moe.make_desc(8192, 3584, 32, 2, 2560)
    assert moe.moe_ffn_kernel(prefill) == moe.MOE_FFN_TC_FUSED
    assert moe.moe_layer_launches(prefill) == 1 + 2 + 1 + 1
    split = moe.make_desc(8192, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_FFN_SPLIT)
    assert moe.moe_ffn_kernel(split) == moe.MOE_FFN_TC_PAIRS
    assert moe.moe_layer_launches(split) == 1 + 2 + 2 + 1
    single = moe.make_desc(8192, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_GEMM_SINGLE)
    assert moe.moe_ffn_kernel(single) == moe.MOE_FFN_TC_SINGLE
    f32 = moe.make_desc(4096, 256, 8, 2, 512, dtype=moe.MOE_F32)      # CUDA-core router: own histogram
    assert moe.moe_ffn_kernel(f32) == moe.MOE_FFN_SIMT
    assert moe.moe_layer_launches(f32) == 1 + 4 + 2 + 1
    decode = moe.make_desc(8, 3584, 32, 2, 2560)
    assert moe.moe_ffn_kernel(decode) == moe.MOE_FFN_STREAM
    assert moe.moe_layer_decode_fused(decode)
    assert moe.moe_layer_launches(decode) == 2            # counters zeroed, the one-launch layer
    steps = moe.make_desc(8, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_DECODE_SPLIT)
    assert not moe.moe_layer_decode_fused(steps)
    assert moe.moe_layer_launches(steps) == 1 + 1 + 1 + 1
    decode_split = moe.make_desc(8, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_FFN_SPLIT)
    assert moe.moe_ffn_kernel(decode_split) == moe.MOE_FFN_STREAM_SPLIT
    assert not moe.moe_layer_decode_fused(decode_split)
    assert moe.moe_layer_launches(decode_split) == 1 + 1 + 2 + 1
    # fp32, more than 16 tokens, drop_tokens=False with a capacity: the separate steps
    assert not moe.moe_layer_decode_fused(moe.make_desc(8, 256, 8, 2, 256, dtype=moe.MOE_F32))
    assert not moe.moe_layer_decode_fused(moe.make_desc(17, 3584, 32, 2, 2560))
    assert not moe.moe_layer_decode_fused(moe.make_desc(8, 3584, 32, 2, 2560, capacity=1,
                                                        flags=moe.MOE_FLAG_REROUTE))
    assert moe.moe_layer_decode_fused(moe.make_desc(16, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_SWIGLU))
    assert moe.moe_layer_decode_fused(moe.make_desc(1, 3584, 32, 2, 2560))
    assert moe.moe_layer_launches(moe.make_desc(0, 3584, 32, 2, 2560)) == 1
    # host buffers, no capacity: two halves of 4096 tokens (each router, scan+scatter, gather,
    # expert FFN, combine; the second half's combine in two launches), then the statistics merge
    host = moe.make_desc(8192, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_HOST_IO)
    assert moe.moe_layer_launches(host) == 1 + 2 * (1 + 2 + 1 + 1) + 1
    # with a capacity the whole batch runs once between its two copies
    host_cap = moe.make_desc(8192, 3584, 32, 2, 2560, capacity=512, flags=moe.MOE_FLAG_HOST_IO)
    assert moe.moe_layer_launches(host_cap) == moe.moe_layer_launches(
        moe.make_desc(8192, 3584, 32, 2, 2560, capacity=512))
    with pytest.raises(moe.MoeError):
        moe.moe_layer_launches(moe.make_desc(8, 3584, 32, 9, 2560))
    with pytest.raises(moe.MoeError):
        moe.moe_ffn_kernel(moe.make_desc(8, 3584, 32, 9, 2560))


def test_gather_gemm_launch_count(lib):
    """MOE_FLAG_GATHER_GEMM takes the gather kernel out of the layer call on
    the SM-pair kernels (one launch fewer, in each half of a host-I/O call
    too); it does not apply to the one-block dispatch (which has no separate
    gather), to drop_tokens=False, to the single-SM and CUDA-core kernels or
    to the decode layer."""
    G = moe.MOE_FLAG_GATHER_GEMM

    def n(*a, flags=0, **kw):
        return moe.moe_layer_launches(moe.make_desc(*a, flags=flags, **kw))
    assert n(8192, 3584, 32, 2, 2560, flags=G) == n(8192, 3584, 32, 2, 2560) - 1
    assert n(8192, 3584, 32, 2, 2560, flags=G | moe.MOE_FLAG_FFN_SPLIT) == \
        n(8192, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_FFN_SPLIT) - 1
    assert n(8192, 3584, 32, 2, 2560, flags=G | moe.MOE_FLAG_HOST_IO) == \
        n(8192, 3584, 32, 2, 2560, flags=moe.MOE_FLAG_HOST_IO) - 2
    assert n(8192, 3584, 32, 2, 2560, capacity=512, flags=G) == n(8192, 3584, 32, 2, 2560, capacity=512) - 1
    for kw in (dict(flags=moe.MOE_FLAG_GEMM_SINGLE), dict(capacity=512, flags=moe.MOE_FLAG_REROUTE),
               dict(dtype=moe.MOE_F32)):
        f = kw.pop("flags", 0)
        assert n(4096, 256, 8, 2, 512, flags=f | G, **kw) == n(4096, 256, 8, 2, 512, flags=f, **kw), kw
    assert n(300, 200, 8, 2, 264, flags=G | moe.MOE_FLAG_GEMM_PAIR) == n(300, 200, 8, 2, 264, flags=moe.MOE_FLAG_GEMM_PAIR)
    assert n(8, 3584, 32, 2, 2560, flags=G) == 2


@pytest.mark.parametrize("bad", [
    dict(K=0), dict(K=9), dict(E=1, K=2), dict(E=257), dict(H=12), dict(F=4), dict(T=-1),
    dict(dtype=7), dict(T=1 << 30, K=4), dict(temperature=float("nan")), dict(temperature=float("inf")),
])
def test_bad_desc_rejected(lib, bad):
    args = dict(T=64, H=256, E=8, K=2, F=512, capacity=0, dtype=moe.MOE_BF16, flags=0, temperature=1.0)
    args.update(bad)
    d = moe.make_desc(**args)
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(d), ctypes.byref(n)) == -1
    assert lib.moe_max_rows(ctypes.byref(d)) == -1
    rc = lib.moe_layer_forward(ctypes.byref(d), *([256] * 12), 1 << 30, None)
    assert rc == -1


def test_host_checks_before_any_launch(lib):
    d = moe.make_desc(64, 256, 8, 2, 512)
    need = moe.moe_workspace_size(d)
    A = 1 << 20          # fake, aligned addresses: never dereferenced on these paths
    P = [A] * 11         # x .. dropped; the workspace follows
    # workspace missing / too small / misaligned
    assert lib.moe_layer_forward(ctypes.byref(d), *P, None, need, None) == -3
    assert lib.moe_layer_forward(ctypes.byref(d), *P, A, need - 1, None) == -3
    assert lib.moe_layer_forward(ctypes.byref(d), *P, A + 16, need, None) == -3
    # a required pointer missing
    Q = list(P); Q[1] = None          # Wg
    assert lib.moe_layer_forward(ctypes.byref(d), *Q, A, need, None) == -1
    # a misaligned tensor
    Q = list(P); Q[0] = A + 2         # x
    assert lib.moe_layer_forward(ctypes.byref(d), *Q, A, need, None) == -1
    assert lib.moe_combine(ctypes.byref(d), A + 8, A, A, A, None) == -1
    assert lib.moe_aux_loss(ctypes.byref(d), None, A, A, None) == -1
    assert lib.moe_router_topk(ctypes.byref(d), A, A, None, None, None, A, None, A, need, None) == -1
    assert lib.moe_expert_ffn(ctypes.byref(d), A, A, A, None, A, None, A, None, A, need, None) == -1
    assert lib.moe_dispatch(ctypes.byref(d), A, None, None, A, A, A, None, None, A, need, None) == -1
    assert lib.moe_get_device_error(None, None, None) == -1


def test_status_strings(lib):
    for c in (0, -1, -2, -3, -4, -5, -6):
        assert moe.moe_status_string(c).startswith("MOE_")
    assert "unknown" in moe.moe_status_string(42)
