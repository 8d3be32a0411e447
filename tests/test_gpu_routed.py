"""moe_forward_routed: the expert computation over rows the caller has already
laid out expert-major (nvfp4moe README, "MoE layer": run_routed with m_indptr
and padded offsets), dispatch and gather skipped.

On the layout moe_forward builds itself (its m_indptr, off_pad, gathered rows,
row scores and row_of), the routed call must give the same ys and y bit for
bit.  On a caller layout of its own (segments padded further than needed,
experts without rows, no scores) it must agree with the oracle within the
stated tolerance.  An inconsistent layout or an out-of-range row_of entry is
reported through the device error word and runs nothing out of bounds.
"""

import numpy as np
import pytest
import torch

from gpu_case import bits, make, run_gpu
from parity import compare, f32, term_flips

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


def _tables(plan, c):
    T, k = c["T"], c["k"]
    op = plan.buffer("off_pad", torch.int32).clone()
    mi_ = plan.buffer("m_indptr", torch.int32).clone()
    n = int(op[-1])
    xe = plan.buffer("xe", torch.bfloat16).view(-1, c["d"])[:n].clone()
    so = plan.buffer("score_of", torch.float32)[:n].clone()
    ro = plan.buffer("row_of", torch.int32)[: T * k].clone()
    ys = plan.buffer("ys", torch.bfloat16).view(-1, c["d"])[:n].clone()
    return dict(off_pad=op, m_indptr=mi_, xe=xe, score_of=so, row_of=ro, ys=ys, n=n)


@pytest.mark.parametrize("sizes", [
    dict(T=300, d=256, I=192, E=7, k=3),
    dict(T=400, d=128, I=256, E=12, k=3, routing="zipf", zipf_s=1.2, zipf_support=8),
    dict(T=8192, d=2048, I=768, E=16, k=8),
], ids=["ragged", "skew_empty", "infer_e16_sizes"])
def test_routed_matches_forward_bit_for_bit(moe, sizes):
    inp = make(None, seed=41, train=False, **sizes)
    c = inp["cfg"]
    g = run_gpu(moe, inp, train=False)
    assert g["rc"] == 0
    t = _tables(g["plan"], c)
    plan2 = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], flags=0)
    dev = g["dev"]
    for _ in range(2):                     # twice in a row: the same bits
        ys, y = plan2.forward_routed(t["xe"], t["m_indptr"], t["off_pad"], dev["w13"], dev["w2"],
                                     score_of=t["score_of"], row_of=t["row_of"].view(c["T"], c["k"]))
        torch.cuda.synchronize()
        rc, det = plan2.check()
        assert rc == 0, (rc, det)
        # every routed row of ys, and y
        real = t["row_of"][t["row_of"] >= 0].long()
        assert torch.equal(ys[real].view(torch.int16), t["ys"][real].view(torch.int16))
        assert torch.equal(y.view(torch.int16), g["y"].view(torch.int16))


def test_routed_own_layout_against_oracle(moe, orc):
    """A layout built here: segments padded with extra empty 128-row blocks (more
    than the kernels need), experts without rows, and no routing scores
    (score_of = NULL, so the oracle runs with unit scores)."""
    T, d, I, E, k = 200, 256, 128, 9, 2
    inp = make(None, seed=42, train=False, T=T, d=d, I=I, E=E, k=k, routing="zipf", zipf_s=1.2,
               zipf_support=6)
    ids = inp["ids"]
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    assert np.any(counts == 0)
    seg = (counts + 127) // 128 * 128
    cap = (T * k + E * 127) // 128 * 128
    for e in range(E):                       # extra padding blocks while they fit
        if seg.sum() + 128 <= cap and e % 2 == 0:
            seg[e] += 128
    off_pad = np.concatenate([[0], np.cumsum(seg)]).astype(np.int32)
    m_indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(off_pad[-1])
    # a stable expert-major layout by flat index
    row_of = np.full(T * k, -1, np.int32)
    fill = off_pad[:-1].copy()
    for f in range(T * k):
        e = flat[f]
        row_of[f] = fill[e]
        fill[e] += 1
    x_e = np.zeros((rows, d), np.uint16)
    x_e[row_of] = inp["x"][np.arange(T * k) // k]
    plan = moe.MoePlan(T, d, I, E, k, flags=0)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    w13 = dev(inp["w13"]).view(torch.bfloat16)
    w2 = dev(inp["w2"]).view(torch.bfloat16)
    ys, y = plan.forward_routed(dev(x_e).view(torch.bfloat16), dev(m_indptr), dev(off_pad), w13,
                                w2, row_of=dev(row_of.reshape(T, k)))
    torch.cuda.synchronize()
    rc, det = plan.check()
    assert rc == 0, (rc, det)
    ones = np.ones((T, k), np.float32)
    yref, it = orc.forward(inp["x"], ids, ones, inp["w13"], inp["w2"], intermediates=True)
    compare(f32(bits(y)), f32(yref), what="y routed", flip=term_flips(it["ys"]))
    compare(f32(bits(ys)[row_of]), f32(it["ys"].reshape(T * k, d)), what="ys routed",
            max_bad_frac=1e-3)


def test_routed_rejects_inconsistent_layout(moe):
    T, d, I, E, k = 64, 128, 64, 4, 2
    plan = moe.MoePlan(T, d, I, E, k, flags=0)
    inp = make(None, seed=43, train=False, T=T, d=d, I=I, E=E, k=k)
    w13 = torch.from_numpy(inp["w13"]).cuda().view(torch.bfloat16)
    w2 = torch.from_numpy(inp["w2"]).cuda().view(torch.bfloat16)
    rows = 512
    x_e = torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda")
    m_indptr = torch.tensor([0, 30, 60, 100, 128], dtype=torch.int32, device="cuda")
    # expert 2's segment [256, 256) is shorter than its 40 rows -> expert 2 is reported
    off_pad = torch.tensor([0, 128, 256, 256, 384], dtype=torch.int32, device="cuda")
    ys = torch.full((rows, d), 7.0, dtype=torch.bfloat16, device="cuda")
    plan.forward_routed(x_e, m_indptr, off_pad, w13, w2, ys=ys)
    rc, det = plan.check()
    assert rc == moe.MOE_ERR_INVALID_ARG and det == 2
    assert torch.all(ys == 7.0)                # no tile ran
    # a consistent layout with one out-of-range row_of entry: dropped and reported
    off_pad = torch.tensor([0, 128, 256, 384, 512], dtype=torch.int32, device="cuda")
    row_of = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    row_of[3, 1] = 9999
    row_of[5, 0] = 130
    ys, y = plan.forward_routed(x_e, m_indptr, off_pad, w13, w2, row_of=row_of)
    rc, det = plan.check()
    assert rc == moe.MOE_ERR_INVALID_ARG and det == E + 1 + 3 * k + 1
    assert torch.all(y.float() == 0)           # zero rows in, zero out
    # and the next consistent call reports nothing
    row_of[3, 1] = -1
    plan.forward_routed(x_e, m_indptr, off_pad, w13, w2, row_of=row_of)
    assert plan.check() == (0, 0)
