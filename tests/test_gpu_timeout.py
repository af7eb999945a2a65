"""Failure detection without a GPU fault: a bounded wait in the tensor-core
expert GEMM is made to run out (the first stage is never filled, so the
barrier it waits on is never signalled).  The kernel must return on its own
with MOE_ERR_TIMEOUT in the workspace error word, and the same process must
then run the layer correctly."""
import time

import numpy as np
import pytest

import sparse_mixture_experts_topk_gb300 as moe
from sparse_mixture_experts_topk_gb300 import workloads as W
from oracle import moe_oracle as O

from harness import Dev, run_stages, run_layer, as_f64, out_errors, OUT_MAXABS_BF16, OUT_REL_L2_BF16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_topk_gb300 import build
    build.build()
    moe.lib()


def test_expired_wait_reports_timeout_and_context_survives():
    w = W.small("stall", T=64, H=256, E=2, K=1, F=256)     # one tile per product
    inp = W.generate(w)
    dev = Dev(inp)
    base = moe.MOE_FLAG_GEMM_SINGLE | moe.MOE_FLAG_NO_DECODE
    t0 = time.time()
    r = run_stages(dev, flags=base | moe.MOE_FLAG_TEST_WAIT_TIMEOUT)
    took = time.time() - t0
    assert r["device_error"] == -5          # MOE_ERR_TIMEOUT
    assert took < 30.0
    # the error word was cleared by the read; the next calls are clean and correct
    ok = run_stages(dev, flags=base)
    assert ok["device_error"] == 0
    L = run_layer(dev, flags=base)
    assert L["device_error"] == 0
    gl = ok["logits"].cpu().numpy().astype(np.float64)
    ref = O.layer_forward(O.widen(inp.x, "bf16"), O.widen(inp.Wg, "bf16"), O.widen(inp.W1, "bf16"),
                          O.widen(inp.W2, "bf16"), w.K, bf16=True, logits=gl)
    mx, rel = out_errors(as_f64(L["out"]), ref["out"])
    assert mx <= OUT_MAXABS_BF16 and rel <= OUT_REL_L2_BF16
