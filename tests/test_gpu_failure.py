"""Failure detection without a GPU fault: a bounded device wait is made to run
out (it waits on a barrier that nothing arrives at), the kernel reports
MOE_ERR_TIMEOUT through the plan's error word, cleans up, and the same CUDA
context then runs the layer correctly."""

import numpy as np
import pytest
import torch

from gpu_case import bits, check_forward, make, run_gpu, to_dev
from parity import compare, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


@pytest.mark.parametrize("precision,pairs", [("bf16", False), ("bf16", True), ("mxfp8", False)])
def test_wait_timeout_is_reported_and_context_survives(moe, orc, precision, pairs):
    """pairs=True runs the CTA-pair W13 kernel; the others the one-CTA kernel."""
    d = I = 256 if pairs else 128
    inp = make(None, seed=31, train=False, T=256, d=d, I=I, E=4, k=2)
    c = inp["cfg"]
    dev = to_dev(inp)
    prec = moe.MOE_PREC_BF16 if precision == "bf16" else moe.MOE_PREC_MXFP8
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], precision=prec, flags=0,
                       cta_pairs=pairs)
    w = dict(w13=dev["w13"], w2=dev["w2"], sf13=None, sf2=None)
    if precision == "mxfp8":
        w["w13"], w["sf13"], w["w2"], w["sf2"] = moe.prepare_weights_mxfp8(dev["w13"], dev["w2"])

    def fwd():
        return plan.forward(dev["x"], dev["ids"], dev["scores"], w["w13"], w["w2"],
                            w13_sf=w["sf13"], w2_sf=w["sf2"])

    plan.set_debug(wait_limit_ns=50_000_000, stall_w13=True)
    fwd()
    rc, where = plan.check()
    assert rc == moe.MOE_ERR_TIMEOUT
    assert where in (1, 2, 3, 4, 5, 9)
    # the context is still usable and the plan recovers
    plan.set_debug(0, False)
    y = fwd()
    rc, _ = plan.check()
    assert rc == 0
    assert torch.isfinite(y.float()).all()
    if precision == "bf16":
        yref = orc.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"])
        compare(f32(bits(y)), f32(yref), what="y after timeout", max_bad_frac=1e-3)
