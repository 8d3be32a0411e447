"""The training step captured in a CUDA graph (nvfp4moe "MoE layer": a warmed
plan does not allocate and can be captured in a CUDA Graph).

A plan's forward + backward are captured once; replays must give the same bits
as eager calls, also after new inputs are copied into the captured buffers
(the graph reads the buffers, it does not freeze their contents)."""

import numpy as np
import pytest
import torch

from gpu_case import make, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


def test_training_step_replays_bit_exact(moe):
    inp = make(None, seed=41, train=True, T=300, d=256, I=256, E=8, k=4)
    inp2 = make(None, seed=42, train=True, T=300, d=256, I=256, E=8, k=4)
    c = inp["cfg"]
    dev = to_dev(inp)
    dev2 = to_dev(inp2)
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], flags=moe.MOE_WS_TRAINING)
    y = torch.empty(c["T"], c["d"], dtype=torch.bfloat16, device="cuda")
    dx = torch.empty_like(y)
    ds = torch.empty(c["T"], c["k"], dtype=torch.float32, device="cuda")
    dw13, dw2 = dev["dw13"].clone(), dev["dw2"].clone()

    def step():
        plan.forward(dev["x"], dev["ids"], dev["scores"], dev["w13"], dev["w2"], y=y, save=True)
        plan.backward(dev["dy"], dev["w13"], dev["w2"], dw13, dw2, dx=dx, dscores=ds)

    def eager(src):
        dw13.copy_(src["dw13"])
        dw2.copy_(src["dw2"])
        for key in ("x", "ids", "scores", "dy"):
            dev[key].copy_(src[key])
        step()
        torch.cuda.synchronize()
        return [t.clone() for t in (y, dx, ds, dw13, dw2)]

    want1 = eager(to_dev(inp))
    want2 = eager(dev2)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm the plan on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for src, want in ((to_dev(inp), want1), (dev2, want2), (to_dev(inp), want1)):
        dw13.copy_(src["dw13"])
        dw2.copy_(src["dw2"])
        for key in ("x", "ids", "scores", "dy"):
            dev[key].copy_(src[key])
        g.replay()
        torch.cuda.synchronize()
        got = (y, dx, ds, dw13, dw2)
        for name, a, b in zip(("y", "dx", "dscores", "dw13", "dw2"), got, want):
            assert torch.equal(a, b), name
    assert plan.check() == (0, 0)
    assert not torch.equal(want1[0], want2[0])
