"""Runs one routed-expert case through the C ABI and through the oracle, and
compares them (shared by the GPU parity tests and the smoke check)."""

import numpy as np
import torch

import moe_inputs as mi
from parity import REL_FRO, WGRAD_FLIP_FRAC, compare, f32, term_flips


def to_dev(inp):
    dev = {}
    for key, v in inp.items():
        if key == "cfg":
            continue
        t = torch.from_numpy(np.ascontiguousarray(v))
        if v.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        dev[key] = t.cuda()
    return dev


def run_gpu(moe, inp, train=True, stream=None):
    c = inp["cfg"]
    dev = to_dev(inp)
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], clamp=c.get("clamp", 0.0),
                       flags=moe.MOE_WS_TRAINING if train else 0,
                       cta_pairs=c.get("cta_pairs", False))
    out = {"plan": plan, "dev": dev}
    out["y"] = plan.forward(dev["x"], dev["ids"], dev["scores"], dev["w13"], dev["w2"], save=train)
    if train:
        dw13, dw2 = dev["dw13"].clone(), dev["dw2"].clone()
        dx, ds = plan.backward(dev["dy"], dev["w13"], dev["w2"], dw13, dw2)
        out.update(dx=dx, dscores=ds, dw13=dw13, dw2=dw2)
    torch.cuda.synchronize()
    rc, detail = plan.check()
    out["rc"], out["detail"] = rc, detail
    return out


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_dispatch(orc, inp, g):
    """Dispatch tables: bit-exact against the oracle's stable counting sort with
    the plan's padding granule."""
    c = inp["cfg"]
    plan = g["plan"]
    r = orc.dispatch(inp["ids"], c["E"], plan.row_granule())
    mi_ = plan.buffer("m_indptr", torch.int32).cpu().numpy()
    op = plan.buffer("off_pad", torch.int32).cpu().numpy()
    ro = plan.buffer("row_of", torch.int32).cpu().numpy()[: c["T"] * c["k"]].reshape(c["T"], c["k"])
    assert np.array_equal(mi_, r["m_indptr"])
    assert np.array_equal(op, r["off_pad"])
    assert np.array_equal(ro, r["row_of"])
    return r


def check_forward(orc, inp, g, toks=None, intermediates=True):
    c = inp["cfg"]
    y_ref, it = orc.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"],
                            clamp=c.get("clamp", 0.0), toks=toks, intermediates=True)
    y = bits(g["y"])
    sel = slice(None) if toks is None else np.asarray(toks)
    compare(f32(y[sel]), f32(y_ref), what="y", flip=term_flips(it["ys"]))
    if intermediates:
        plan = g["plan"]
        ro = plan.buffer("row_of", torch.int32).cpu().numpy()[: c["T"] * c["k"]].reshape(c["T"], c["k"])
        rows = ro[sel]
        ok = rows >= 0
        I, d = c["I"], c["d"]
        h = bits(plan.buffer("h", torch.bfloat16).view(-1, I))
        ys = bits(plan.buffer("ys", torch.bfloat16).view(-1, d))
        compare(f32(h[rows[ok]]), f32(it["h"][ok]), what="h", max_bad_frac=1e-3)
        compare(f32(ys[rows[ok]]), f32(it["ys"][ok]), what="ys", max_bad_frac=1e-3)
        if c.get("train", True) and plan.flags & 1:
            a = bits(plan.buffer("a", torch.bfloat16).view(-1, 2 * I))
            compare(f32(a[rows[ok]]), f32(it["a"][ok]), what="a", max_bad_frac=1e-3)
    return y_ref


def check_backward(orc, inp, g, toks=None, experts=None, intermediates=True):
    c = inp["cfg"]
    clamp = c.get("clamp", 0.0)
    dx_ref, ds_ref, bi = orc.backward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"],
                                      inp["dy"], clamp=clamp, toks=toks, intermediates=True)
    sel = slice(None) if toks is None else np.asarray(toks)
    compare(f32(bits(g["dx"])[sel]), f32(dx_ref), what="dx", flip=term_flips(bi["dxe"]))
    compare(g["dscores"].cpu().numpy()[sel], ds_ref, bf16_out=False, what="dscores")
    if intermediates:
        plan = g["plan"]
        ro = plan.buffer("row_of", torch.int32).cpu().numpy()[: c["T"] * c["k"]].reshape(c["T"], c["k"])
        rows = ro[sel]
        ok = rows >= 0
        I = c["I"]
        dA = bits(plan.buffer("dA", torch.bfloat16).view(-1, 2 * I))
        hs = bits(plan.buffer("hs", torch.bfloat16).view(-1, I))
        compare(f32(dA[rows[ok]]), f32(bi["dA"][ok]), what="dA", max_bad_frac=1e-3)
        compare(f32(hs[rows[ok]]), f32(bi["hs"][ok]), what="hs", max_bad_frac=1e-3)
    E = c["E"]
    experts = range(E) if experts is None else experts
    dw13 = g["dw13"]
    dw2 = g["dw2"]
    plan = g["plan"]
    op = plan.buffer("off_pad", torch.int32).cpu().numpy()
    mi_ = plan.buffer("m_indptr", torch.int32).cpu().numpy()
    for e in experts:
        d13, d2, nrows = orc.wgrad_expert(inp["x"], inp["ids"], inp["scores"], inp["w13"],
                                          inp["w2"], inp["dy"], e, clamp=clamp)
        got13 = (dw13[e].double() - g["dev"]["dw13"][e].double()).cpu().numpy()
        got2 = (dw2[e].double() - g["dev"]["dw2"][e].double()).cpu().numpy()
        if nrows == 0:
            assert np.all(got13 == 0) and np.all(got2 == 0), "expert %d without rows changed" % e
            continue
        # Against the oracle.  A weight gradient sums, over the expert's rows, products
        # of the bf16 operands hs and dA (R7, R4); where one of those flipped to the
        # neighbouring bf16 value (a different fp32 summation order upstream) the
        # difference can pass the literal max-abs bound: at most WGRAD_FLIP_FRAC of
        # the elements may (counts recorded), and the Frobenius bound holds as stated.
        compare(got13, d13, bf16_out=False, what="dW13[%d]" % e, max_bad_frac=WGRAD_FLIP_FRAC)
        compare(got2, d2, bf16_out=False, what="dW2[%d]" % e, max_bad_frac=WGRAD_FLIP_FRAC)
        # The WGRAD GEMMs alone, against an FP64 product of the GPU's own operands
        # (the expert's rows of dY_e, hs, dA and x_e): the bf16 products are exact,
        # so only the fp32 accumulation differs.  Bound: the deterministic error
        # bound n * 2^-24 of an n-term fp32 sum (n = the expert's rows), at least
        # 1e-5; every element also within the literal max-abs bound.
        if plan.flags & 1 and plan.precision == 0:
            r0, r1 = int(op[e]), int(op[e]) + int(mi_[e + 1] - mi_[e])
            I, d = c["I"], c["d"]
            rows = lambda name, w: f32(bits(plan.buffer(name, torch.bfloat16).view(-1, w)[r0:r1])) \
                .astype(np.float64)
            own13 = rows("dA", 2 * I).T @ rows("xe", d)
            own2 = rows("dye", d).T @ rows("hs", I)
            tol = max(1e-5, (r1 - r0) * 2.0 ** -24)
            compare(got13, own13, bf16_out=False, rel_fro=tol, what="dW13[%d] own operands" % e)
            compare(got2, own2, bf16_out=False, rel_fro=tol, what="dW2[%d] own operands" % e)


def make(name=None, seed=0, train=True, **over):
    need = ("x", "ids", "scores", "w13", "w2") + (("dy", "dw13", "dw2") if train else ())
    return mi.make_inputs(name, seed=seed, need=need, **over)


__all__ = ["make", "run_gpu", "check_dispatch", "check_forward", "check_backward", "bits",
           "REL_FRO"]
