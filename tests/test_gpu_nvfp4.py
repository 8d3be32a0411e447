"""NVFP4 inference forward through the C ABI against the oracle.

Prepared weights (packed E2M1 codes, E4M3 block scales, per-expert scales) and
the quantised routed activations must match the oracle's quantiser bit for bit
(the scales after undoing the tiled layout).  The output must be within
relative Frobenius error 1e-2 of the oracle's NVFP4 forward, which quantises the
same way with the same static scales (the bound of the block-scaled MXFP8 path;
a bf16 flip of h upstream can move an E2M1 code of h by one step).  Nearly all
codes of the requantised h must equal the oracle's.
"""

import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_case import bits, to_dev
from parity import REL_FRO_MXFP8, compare, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


def untile16(sf, rows, K, gu_I=0):
    """Tiled NVFP4 scale bytes -> [rows, K/16] (inverse of the documented layout)."""
    kbs, ngr = K // 16, K // 64
    r = np.arange(rows)
    if gu_I:
        e, i = r // (2 * gu_I), r % (2 * gu_I)
        up = i >= gu_I
        ii = np.where(up, i - gu_I, i)
        blk, rin = e * (gu_I // 64) + ii // 64, up * 64 + ii % 64
    else:
        blk, rin = r // 128, r % 128
    kb = np.arange(kbs)
    off = ((blk[:, None] * ngr + kb[None, :] // 4) * 512 + (rin[:, None] % 32) * 16
           + (rin[:, None] // 32) * 4 + kb[None, :] % 4)
    return sf[off]


def calibrated_scales(moe, inp, dev):
    """Static activation scales as a calibration pass would set them: amax / (6 *
    448) of x and of h from the bf16 forward on the same inputs (device amax)."""
    c = inp["cfg"]
    x_amax = float(moe.amax_bf16(dev["x"]).item())
    assert x_amax == float(np.abs(f32(inp["x"])).max())
    bp = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], clamp=c.get("clamp", 0.0), flags=0)
    bp.forward(dev["x"], dev["ids"], dev["scores"], dev["w13"], dev["w2"])
    n = int(bp.buffer("off_pad", torch.int32)[-1].item())
    h = bp.buffer("h", torch.bfloat16)[: n * c["I"]]
    h_amax = float(moe.amax_bf16(h).item())
    torch.cuda.synchronize()
    return np.float32(x_amax) / np.float32(2688.0), np.float32(h_amax) / np.float32(2688.0)


def run_nv(moe, inp, dev, prep, xs, hs):
    c = inp["cfg"]
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], precision=moe.MOE_PREC_NVFP4,
                       clamp=c.get("clamp", 0.0), flags=0)
    plan.set_activation_scales(xs, hs)
    y = plan.forward_nvfp4(dev["x"], dev["ids"], dev["scores"], prep)
    torch.cuda.synchronize()
    rc, det = plan.check()
    assert rc == 0, (rc, det)
    return plan, y


def check_prepared(orc, inp, prep, experts=None):
    c = inp["cfg"]
    E, I, d = c["E"], c["I"], c["d"]
    g13q, g13s, g13c, g2q, g2s, g2c = (t.cpu().numpy() for t in prep)
    o13 = orc.prepare_nvfp4(inp["w13"])
    o2 = orc.prepare_nvfp4(inp["w2"])
    assert np.array_equal(g13c, o13[2]) and np.array_equal(g2c, o2[2])
    assert np.array_equal(g13q, o13[0]) and np.array_equal(g2q, o2[0])
    assert np.array_equal(untile16(g13s, E * 2 * I, d, gu_I=I), o13[1].reshape(E * 2 * I, d // 16))
    assert np.array_equal(untile16(g2s, E * d, I), o2[1].reshape(E * d, I // 16))
    return o13, o2


SMALL = [
    dict(T=64, d=256, I=256, E=4, k=2),
    dict(T=300, d=512, I=256, E=7, k=3),
    dict(T=200, d=256, I=512, E=9, k=2, clamp=1.0, pad=30),
    dict(T=400, d=256, I=256, E=12, k=3, routing="zipf", zipf_s=1.2, zipf_support=8),
    dict(T=1, d=256, I=256, E=4, k=2),
    dict(T=96, d=256, I=256, E=256, k=8),
]


@pytest.mark.parametrize("sizes", SMALL,
                         ids=["tiny", "ragged", "clamped_pad", "skew_empty", "one_token", "k8_e256"])
def test_nvfp4_small(moe, orc, sizes):
    inp = mi.make_inputs(None, seed=51, need=("x", "ids", "scores", "w13", "w2"), **sizes)
    c = inp["cfg"]
    T, d, I, E, k = c["T"], c["d"], c["I"], c["E"], c["k"]
    dev = to_dev(inp)
    prep = moe.prepare_weights_nvfp4(dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    o13, o2 = check_prepared(orc, inp, prep)
    xs, hs = calibrated_scales(moe, inp, dev)
    plan, y = run_nv(moe, inp, dev, prep, xs, hs)
    # quantised routed activations: bit-exact (padding rows zero codes)
    n = int(plan.buffer("off_pad", torch.int32).cpu().numpy()[-1])
    tok = plan.buffer("token_of", torch.int32).cpu().numpy()[:n]
    xrows = orc.gather_rows(inp["x"], tok)
    qx, sx = orc.quant_nvfp4(xrows, np.float32(1.0) / xs)
    assert np.array_equal(plan.buffer("xq", torch.uint8).cpu().numpy()[: n * d // 2]
                          .reshape(n, d // 2), qx)
    assert np.array_equal(untile16(plan.buffer("xsf", torch.uint8).cpu().numpy(), n, d), sx)
    # output and the requantised h
    yref, it = orc.forward_nvfp4(inp["x"], inp["ids"], inp["scores"], o13, o2, xs, hs,
                                 clamp=c.get("clamp", 0.0), intermediates=True)
    assert np.sqrt(np.mean(f32(yref) ** 2)) > 1e-3          # a non-trivial output
    compare(f32(bits(y)), f32(yref), bf16_out=True, rel_fro=REL_FRO_MXFP8, what="y nvfp4",
            max_bad_frac=1.0)
    ro = plan.buffer("row_of", torch.int32).cpu().numpy()[: T * k].reshape(T, k)
    ok = ro >= 0
    RP = plan.buffer("hq", torch.uint8).numel() * 2 // I
    hq = plan.buffer("hq", torch.uint8).cpu().numpy().reshape(RP, I // 2)[ro[ok]]
    hsc = untile16(plan.buffer("hsf", torch.uint8).cpu().numpy(), RP, I)[ro[ok]]
    qh, sh = orc.quant_nvfp4(it["h"][ok], np.float32(1.0) / hs)
    assert np.mean(hq == qh) > 0.99 and np.mean(hsc == sh) > 0.99


def test_nvfp4_refuses_training_and_needs_scales(moe):
    plan = moe.lib().moe_plan_create(64, 256, 256, 4, 2, moe.MOE_PREC_NVFP4)
    assert plan
    L = moe.lib()
    import ctypes
    ws = torch.empty(L.moe_plan_workspace_bytes(plan, 1) + 256, dtype=torch.uint8, device="cuda")
    assert L.moe_plan_set_workspace(plan, ctypes.c_void_p(ws.data_ptr()), ws.numel(), 1) == \
        moe.MOE_ERR_UNSUPPORTED
    L.moe_plan_destroy(plan)
    assert not L.moe_plan_create(64, 128, 256, 4, 2, moe.MOE_PREC_NVFP4)   # d % 256
    inp = mi.make_inputs(None, seed=52, need=("x", "ids", "scores", "w13", "w2"),
                         T=64, d=256, I=256, E=4, k=2)
    dev = to_dev(inp)
    prep = moe.prepare_weights_nvfp4(dev["w13"], dev["w2"])
    p = moe.MoePlan(64, 256, 256, 4, 2, precision=moe.MOE_PREC_NVFP4, flags=0)
    with pytest.raises(moe.MoeError) as ei:
        p.forward_nvfp4(dev["x"], dev["ids"], dev["scores"], prep)
    assert ei.value.code == moe.MOE_ERR_STATE
    with pytest.raises(moe.MoeError) as ei:
        p.forward(dev["x"], dev["ids"], dev["scores"], dev["w13"], dev["w2"])
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED


def test_nvfp4_full_size_sampled(moe, orc):
    """The inference workload (T = 8192, d = 2048, I = 768, E = 16, k = 8) at full
    size in the benchmark's launch configuration; the oracle evaluates 1024
    sampled tokens."""
    inp = mi.make_inputs("infer_e16", need=("x", "ids", "scores", "w13", "w2"))
    c = inp["cfg"]
    dev = to_dev(inp)
    prep = moe.prepare_weights_nvfp4(dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    o13, o2 = check_prepared(orc, inp, prep)
    xs, hs = calibrated_scales(moe, inp, dev)
    plan, y = run_nv(moe, inp, dev, prep, xs, hs)
    yb = f32(bits(y))
    assert np.all(np.isfinite(yb))
    rng = np.random.default_rng(7)
    toks = np.array(sorted(set(rng.choice(c["T"], 1024, replace=False).tolist())
                           | {0, c["T"] - 1}), np.int32)
    yref = orc.forward_nvfp4(inp["x"], inp["ids"], inp["scores"], o13, o2, xs, hs, toks=toks)
    assert np.sqrt(np.mean(f32(yref) ** 2)) > 1e-3
    compare(yb[toks], f32(yref), bf16_out=True, rel_fro=REL_FRO_MXFP8, what="y nvfp4 full",
            max_bad_frac=1.0)
