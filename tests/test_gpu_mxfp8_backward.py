"""MXFP8 training step (saving forward + moe_backward_mxfp8) through the C ABI
against the oracle's MXFP8 backward.

Bit-exact: the weights prepared for the backward (W13^T along 2I, W2^T along
d, codes and scales) and the routed x rows quantised along the rows (the
WGRAD-W13 operand) and along d (the forward's operand, same pass).  Within the MXFP8 tolerance (relative Frobenius 1e-2,
tests/parity.py): dx, dscores, the quantised intermediates (dA along 2I, dA and
hs along the rows; nearly all codes equal), and the weight gradient increments
of every expert (small cases) or of sampled experts (full size).
"""

import numpy as np
import pytest
import torch

from gpu_case import bits, to_dev
from parity import REL_FRO_MXFP8, compare, f32
from test_gpu_mxfp8 import dequant, untile
import moe_inputs as mi

pytestmark = pytest.mark.gpu

NEED = ("x", "ids", "scores", "w13", "w2", "dy", "dw13", "dw2")


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


def train_step(moe, inp, dev):
    c = inp["cfg"]
    prep = moe.prepare_weights_mxfp8(dev["w13"], dev["w2"])
    prep_t = moe.prepare_weights_mxfp8_backward(dev["w13"], dev["w2"])
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], precision=moe.MOE_PREC_MXFP8,
                       clamp=c.get("clamp", 0.0), flags=moe.MOE_WS_TRAINING)
    w13q, w13s, w2q, w2s = prep
    y = plan.forward(dev["x"], dev["ids"], dev["scores"], w13q, w2q, w13_sf=w13s, w2_sf=w2s,
                     save=True)
    dw13, dw2 = dev["dw13"].clone(), dev["dw2"].clone()
    dx, ds = plan.backward_mxfp8(dev["dy"], *prep_t, dw13, dw2)
    torch.cuda.synchronize()
    rc, det = plan.check()
    assert rc == 0, (rc, det)
    return dict(plan=plan, prep=prep, prep_t=prep_t, y=y, dx=dx, ds=ds, dw13=dw13, dw2=dw2)


def oracle_weights(orc, inp, experts=None):
    """Forward and backward prepared weights in the oracle's layout (all experts,
    or zeros except the listed ones)."""
    w13, w2 = inp["w13"], inp["w2"]
    if experts is None:
        fw = orc.quant_mxfp8(w13) + orc.quant_mxfp8(w2)
        bw = orc.prepare_mxfp8_backward_weights(w13, w2)
        return fw, bw
    E, I2, d = w13.shape
    I = I2 // 2
    fw = [np.zeros((E, I2, d), np.uint8), np.zeros((E, I2, d // 32), np.uint8),
          np.zeros((E, d, I), np.uint8), np.zeros((E, d, I // 32), np.uint8)]
    bw = [np.zeros((E, d, I2), np.uint8), np.zeros((E, d, I2 // 32), np.uint8),
          np.zeros((E, I, d), np.uint8), np.zeros((E, I, d // 32), np.uint8)]
    for e in experts:
        fw[0][e], fw[1][e] = orc.quant_mxfp8(w13[e])
        fw[2][e], fw[3][e] = orc.quant_mxfp8(w2[e])
        b = orc.prepare_mxfp8_backward_weights(w13[e:e + 1], w2[e:e + 1])
        for i in range(4):
            bw[i][e] = b[i][0]
    return tuple(fw), tuple(bw)


@pytest.mark.parametrize("sizes", [
    dict(T=64, d=128, I=128, E=4, k=2),
    dict(T=300, d=256, I=256, E=7, k=3),
    dict(T=200, d=384, I=128, E=9, k=2, clamp=1.0, pad=30),
    dict(T=400, d=128, I=128, E=12, k=3, routing="zipf", zipf_s=1.2, zipf_support=8),
    # degenerate routing: one token; k = 8 of 256 experts (most experts hold a few
    # rows, so most 32-row blocks along the rows are mostly padding)
    dict(T=1, d=128, I=128, E=4, k=2),
    dict(T=96, d=128, I=128, E=256, k=8),
], ids=["tiny", "ragged", "clamped_pad", "skew_empty", "one_token", "k8_e256"])
def test_mxfp8_backward_small(moe, orc, sizes):
    inp = mi.make_inputs(None, seed=23, need=NEED, **sizes)
    c = inp["cfg"]
    T, d, I, E, k = c["T"], c["d"], c["I"], c["E"], c["k"]
    L = c.get("clamp", 0.0)
    dev = to_dev(inp)
    g = train_step(moe, inp, dev)
    fw, bw = oracle_weights(orc, inp)
    # prepared backward weights: bit-exact
    w13t, w13ts, w2t, w2ts = (t.cpu().numpy() for t in g["prep_t"])
    assert np.array_equal(w13t, bw[0]) and np.array_equal(w2t, bw[2])
    assert np.array_equal(untile(w13ts, E * d, 2 * I), bw[1].reshape(E * d, 2 * I // 32))
    assert np.array_equal(untile(w2ts, E * I, d), bw[3].reshape(E * I, d // 32))
    # routed x quantised along the rows (WGRAD-W13 operand): bit-exact
    plan = g["plan"]
    n = int(plan.buffer("off_pad", torch.int32).cpu().numpy()[-1])
    tok = plan.buffer("token_of", torch.int32).cpu().numpy()[:n]
    xrows = orc.gather_rows(inp["x"], tok)
    qT, sT = orc.quant_mxfp8(np.ascontiguousarray(xrows.T))
    RP = plan.buffer("xqT", torch.uint8).numel() // d
    gq = plan.buffer("xqT", torch.uint8).cpu().numpy().reshape(d, RP)[:, :n]
    assert np.array_equal(gq, qT)
    gs = untile(plan.buffer("xqTsf", torch.uint8).cpu().numpy(), d, RP)[:, : n // 32]
    assert np.array_equal(gs, sT)
    # ... and along d (the forward's A operand), from the same pass
    qx, sx = orc.quant_mxfp8(xrows)
    assert np.array_equal(plan.buffer("xq", torch.uint8).cpu().numpy()[: n * d].reshape(n, d), qx)
    assert np.array_equal(untile(plan.buffer("xsf", torch.uint8).cpu().numpy(), n, d), sx)
    # outputs and intermediates
    dxr, dsr, bi = orc.backward_mxfp8(inp["x"], inp["ids"], inp["scores"], fw, bw, inp["dy"],
                                      clamp=L, intermediates=True)
    compare(f32(bits(g["dx"])), f32(dxr), bf16_out=True, rel_fro=REL_FRO_MXFP8, what="dx mxfp8",
            max_bad_frac=1.0)
    compare(g["ds"].cpu().numpy(), dsr, rel_fro=REL_FRO_MXFP8, what="dscores mxfp8",
            max_bad_frac=1.0)
    ro = plan.buffer("row_of", torch.int32).cpu().numpy()[: T * k].reshape(T, k)
    ok = ro >= 0
    # dA and hs exist only quantised (the DGRAD-W2 epilogue writes no bf16 copies):
    # dA along 2I (DGRAD-W13 operand), dA and hs along the rows (WGRAD operands).
    # Reference: the oracle's bf16 dA and hs in the padded row order, quantised by
    # the oracle.  The dequantised values agree within tolerance and nearly all
    # codes are equal (a code moves by one step where the two bf16 values differ
    # in their last bit).
    dA_pad = np.zeros((n, 2 * I), np.uint16)
    hs_pad = np.zeros((n, I), np.uint16)
    dA_pad[ro[ok]] = bi["dA"][ok]
    hs_pad[ro[ok]] = bi["hs"][ok]
    for name, sname, ref, rows, cols, transposed in (
            ("dAq", "dAsf", dA_pad, RP, 2 * I, False),
            ("dAqT", "dAqTsf", dA_pad.T, 2 * I, RP, True),
            ("hsqT", "hsqTsf", hs_pad.T, I, RP, True)):
        q = plan.buffer(name, torch.uint8).cpu().numpy().reshape(rows, cols)
        sc = untile(plan.buffer(sname, torch.uint8).cpu().numpy(), rows, cols)
        if transposed:
            q, sc = q[:, :n], sc[:, : n // 32]
        else:
            q, sc = q[:n], sc[:n]
        rq, rs = orc.quant_mxfp8(np.ascontiguousarray(ref))
        compare(dequant(orc, q, sc), dequant(orc, rq, rs), bf16_out=False, rel_fro=REL_FRO_MXFP8,
                what=name + " mxfp8", max_bad_frac=1e-2)
        assert np.mean(q == rq) > 0.99, name
    # weight-gradient increments, every expert (untouched where an expert has no rows)
    d13 = (g["dw13"] - dev["dw13"]).cpu().numpy()
    d2 = (g["dw2"] - dev["dw2"]).cpu().numpy()
    for e in range(E):
        r13, r2, rows = orc.wgrad_expert_mxfp8(inp["x"], inp["ids"], inp["scores"], fw, bw,
                                               inp["dy"], e, clamp=L)
        if rows == 0:
            assert torch.equal(g["dw13"][e], dev["dw13"][e]) and torch.equal(g["dw2"][e],
                                                                             dev["dw2"][e])
            continue
        compare(d13[e], r13, rel_fro=REL_FRO_MXFP8, what="dW13[%d] mxfp8" % e, max_bad_frac=1.0)
        compare(d2[e], r2, rel_fro=REL_FRO_MXFP8, what="dW2[%d] mxfp8" % e, max_bad_frac=1.0)


def test_mxfp8_backward_needs_a_saving_forward(moe):
    inp = mi.make_inputs(None, seed=24, need=NEED, T=64, d=128, I=128, E=4, k=2)
    c = inp["cfg"]
    dev = to_dev(inp)
    prep = moe.prepare_weights_mxfp8(dev["w13"], dev["w2"])
    prep_t = moe.prepare_weights_mxfp8_backward(dev["w13"], dev["w2"])
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], precision=moe.MOE_PREC_MXFP8,
                       flags=moe.MOE_WS_TRAINING)
    with pytest.raises(moe.MoeError) as ei:
        plan.backward_mxfp8(dev["dy"], *prep_t, dev["dw13"], dev["dw2"])
    assert ei.value.code == moe.MOE_ERR_STATE
    plan.forward(dev["x"], dev["ids"], dev["scores"], prep[0], prep[2], w13_sf=prep[1],
                 w2_sf=prep[3], save=False)
    with pytest.raises(moe.MoeError):
        plan.backward_mxfp8(dev["dy"], *prep_t, dev["dw13"], dev["dw2"])
    bf = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], flags=moe.MOE_WS_TRAINING)
    with pytest.raises(moe.MoeError) as ei:
        bf.backward_mxfp8(dev["dy"], *prep_t, dev["dw13"], dev["dw2"])
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED


def test_mxfp8_backward_full_size_sampled(moe, orc):
    inp = mi.make_inputs("mxfp8_e128", need=NEED)
    c = inp["cfg"]
    dev = to_dev(inp)
    g = train_step(moe, inp, dev)
    dx = f32(bits(g["dx"]))
    assert np.all(np.isfinite(dx)) and np.all(np.isfinite(g["ds"].cpu().numpy()))
    rng = np.random.default_rng(6)
    toks = np.array(sorted(set(rng.choice(c["T"], 256, replace=False).tolist())
                           | {0, c["T"] - 1}), np.int32)
    counts = np.bincount(inp["ids"].reshape(-1), minlength=c["E"])
    # the heaviest expert (longest WGRAD K loop) and the lightest
    wg_experts = [int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))]
    fw, bw = oracle_weights(orc, inp)
    dxr, dsr = orc.backward_mxfp8(inp["x"], inp["ids"], inp["scores"], fw, bw, inp["dy"],
                                  toks=toks)
    compare(dx[toks], f32(dxr), bf16_out=True, rel_fro=REL_FRO_MXFP8, what="dx mxfp8 full",
            max_bad_frac=1.0)
    compare(g["ds"].cpu().numpy()[toks], dsr, rel_fro=REL_FRO_MXFP8, what="dscores mxfp8 full",
            max_bad_frac=1.0)
    for e in wg_experts:
        r13, r2, rows = orc.wgrad_expert_mxfp8(inp["x"], inp["ids"], inp["scores"], fw, bw,
                                               inp["dy"], e)
        assert rows == counts[e]
        compare((g["dw13"][e] - dev["dw13"][e]).cpu().numpy(), r13, rel_fro=REL_FRO_MXFP8,
                what="dW13[%d] mxfp8 full" % e, max_bad_frac=1.0)
        compare((g["dw2"][e] - dev["dw2"][e]).cpu().numpy(), r2, rel_fro=REL_FRO_MXFP8,
                what="dW2[%d] mxfp8 full" % e, max_bad_frac=1.0)


@pytest.mark.parametrize("min_rows", [0, 128])
def test_mxfp8_wgrad_interleave_is_bit_identical(moe, min_rows):
    """Block-scaled weight gradients with the heavy experts' tiles interleaved
    with lighter ones: the same bits as the default schedule."""
    inp = mi.make_inputs(None, seed=63, need=NEED, T=4096, d=256, I=256, E=32, k=8,
                         routing="zipf", zipf_s=1.2, zipf_support=24)
    counts = np.bincount(inp["ids"].reshape(-1), minlength=32)
    assert counts.max() > 2560   # the default threshold splits the heaviest experts
    dev = to_dev(inp)
    ref = train_step(moe, inp, dev)
    plan = ref["plan"]
    plan.set_wgrad_interleave(min_rows)
    w13q, w13s, w2q, w2s = ref["prep"]
    plan.forward(dev["x"], dev["ids"], dev["scores"], w13q, w2q, w13_sf=w13s, w2_sf=w2s,
                 save=True)
    dw13, dw2 = dev["dw13"].clone(), dev["dw2"].clone()
    dx, ds = plan.backward_mxfp8(dev["dy"], *ref["prep_t"], dw13, dw2)
    torch.cuda.synchronize()
    assert plan.check()[0] == 0
    assert torch.equal(dx.view(torch.int16), ref["dx"].view(torch.int16))
    assert torch.equal(ds, ref["ds"])
    assert torch.equal(dw13, ref["dw13"]) and torch.equal(dw2, ref["dw2"])
