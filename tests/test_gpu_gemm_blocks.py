"""The expert GEMMs on chosen per-expert row counts.

moe_expert_ffn is called directly with an offs table whose experts hold row
counts on both sides of every change of tile shape in the SM-pair kernel: a
last block of at most 48 rows runs wide (two n-tiles a stage), up to 128 rows
swapped (token rows on the MMA's N side), beyond that in row orientation,
and 256 rows fill a block.  N = 768 gives the first product three n-tiles (a
pair and an odd one), N = 512 the second two.  Each product of each expert is
checked against the oracle's fp64 product rounded to bf16 (one bf16 ulp plus
the fp32 accumulation bound), for every GEMM variant."""
import numpy as np
import pytest

from sparse_mixture_experts_topk_gb300 import workloads as W
import sparse_mixture_experts_topk_gb300 as moe
from oracle import moe_oracle as O

from harness import to_dev, to_np, as_f64, product_tol, GELU_SLOPE

pytestmark = pytest.mark.gpu

H, F = 512, 768
# rows per expert: 0 (empty), wide tails alone (1, 16, 32, 33, 48), swapped
# (49, 128), row orientation (129, 255), a full block (256), full blocks with
# a wide tail (256 + 1, 256 + 48, 512 + 48) or a swapped one (256 + 49), and
# two full blocks with tails either side of the swap limit (512 + 128, 512 + 129)
COUNTS = [1, 16, 0, 32, 33, 48, 49, 128, 129, 255, 256, 257, 304, 305, 560, 640, 641]
E = len(COUNTS)

KINDS = {
    "pair": moe.MOE_FLAG_GEMM_PAIR,
    "pair_split": moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_FFN_SPLIT,
    "pair_rows": moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_GEMM_ROWS,
    "single": moe.MOE_FLAG_GEMM_SINGLE,
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_topk_gb300 import build
    build.build()
    moe.lib()


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("kind", list(KINDS))
def test_products_at_every_tile_shape(kind, act):
    import torch
    R = sum(COUNTS)
    rng = np.random.default_rng(20261203)
    xp = W.f32_to_bf16_bits(rng.standard_normal((R, H), dtype=np.float32))
    w = W.small("blocks", T=R, H=H, E=E, K=1, F=F, act=act)
    W1 = np.stack([W.gen_w1(w, e) for e in range(E)])
    W2 = np.stack([W.gen_w2(w, e) for e in range(E)])
    offs = np.concatenate([[0], np.cumsum(COUNTS)]).astype(np.int32)
    flags = KINDS[kind] | moe.MOE_FLAG_NO_DECODE | (moe.MOE_FLAG_SWIGLU if act == "swiglu" else 0)
    d = moe.make_desc(R, H, E, 1, F, 0, moe.MOE_BF16, flags)
    ws = moe.workspace(d)
    x_d, W1_d, W2_d = to_dev(xp, W.BF16), to_dev(W1, W.BF16), to_dev(W2, W.BF16)
    offs_d = torch.from_numpy(offs).cuda()
    h = torch.zeros((R, F), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((R, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn(d, x_d, offs_d, W1_d, None, W2_d, None, h, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    x64, h_gpu, y_gpu = O.widen(xp, W.BF16), as_f64(h), as_f64(y)
    W164, W264 = O.widen(W1, W.BF16), O.widen(W2, W.BF16)
    for e in range(E):
        a, b = int(offs[e]), int(offs[e + 1])
        if a == b:
            continue
        pre = x64[a:b] @ W164[e].T
        if act == "swiglu":
            g, u = pre[:, :F], pre[:, F:]
            h_ref = O.round_bf16(O.silu(g) * u)
            # d(SiLU(g) u) = SiLU'(g) u dg + SiLU(g) du, |SiLU'| <= 1.1
            tol_g = product_tol(0 * g, x64[a:b], W164[e][:F])
            tol_u = product_tol(0 * u, x64[a:b], W164[e][F:])
            tol_h = np.abs(h_ref) * 2.0 ** -7 + 1.1 * np.abs(u) * tol_g + np.abs(O.silu(g)) * tol_u
        else:
            h_ref = O.round_bf16(O.gelu(pre))
            tol_h = product_tol(h_ref, x64[a:b], W164[e], GELU_SLOPE)
        bad = np.abs(h_gpu[a:b] - h_ref) > tol_h
        assert not bad.any(), (kind, act, e, COUNTS[e], "h", int(bad.sum()))
        y_ref = O.round_bf16(h_gpu[a:b] @ W264[e].T)
        bad = np.abs(y_gpu[a:b] - y_ref) > product_tol(y_ref, h_gpu[a:b], W264[e])
        assert not bad.any(), (kind, act, e, COUNTS[e], "y", int(bad.sum()))


def test_one_launch_equals_one_launch_per_product():
    """With every tile shape present, the pair kernel running both products
    in one launch (second-product tiles waiting on their row block's counter,
    which wide tiles advance by two) gives the same bits as one launch per
    product."""
    import torch
    R = sum(COUNTS)
    rng = np.random.default_rng(7)
    xp = W.f32_to_bf16_bits(rng.standard_normal((R, H), dtype=np.float32))
    w = W.small("blocks", T=R, H=H, E=E, K=1, F=F)
    W1 = np.stack([W.gen_w1(w, e) for e in range(E)])
    W2 = np.stack([W.gen_w2(w, e) for e in range(E)])
    offs_d = torch.from_numpy(np.concatenate([[0], np.cumsum(COUNTS)]).astype(np.int32)).cuda()
    x_d, W1_d, W2_d = to_dev(xp, W.BF16), to_dev(W1, W.BF16), to_dev(W2, W.BF16)
    outs = []
    for flags in (moe.MOE_FLAG_GEMM_PAIR, moe.MOE_FLAG_GEMM_PAIR | moe.MOE_FLAG_FFN_SPLIT):
        d = moe.make_desc(R, H, E, 1, F, 0, moe.MOE_BF16, flags | moe.MOE_FLAG_NO_DECODE)
        ws = moe.workspace(d)
        h = torch.zeros((R, F), dtype=torch.bfloat16, device="cuda")
        y = torch.zeros((R, H), dtype=torch.bfloat16, device="cuda")
        moe.moe_expert_ffn(d, x_d, offs_d, W1_d, None, W2_d, None, h, y, ws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
        outs.append((to_np(h), to_np(y)))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])
