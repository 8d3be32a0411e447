"""MXFP8 E4M3 forward through the C ABI against the oracle.

Prepared weight codes and scales, and the quantised routed activations, must
match the oracle's quantiser bit for bit (the scales after undoing the tiled
layout); the output must be within relative Frobenius error 1e-2 of the
oracle's MXFP8 forward, which quantises the same way (tests/parity.py).
"""

import numpy as np
import pytest
import torch

from gpu_case import bits, to_dev
from parity import REL_FRO_MXFP8, compare, f32
import moe_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


def untile(sf, rows, K, gu_I=0):
    """Tiled scale bytes -> [rows, K/32] (inverse of the documented layout)."""
    kbs = K // 32
    ngr = K // 128
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


def dequant(orc, codes, scales):
    """E4M3 codes [rows, K] with E8M0 scales [rows, K/32] -> float64 values."""
    return orc.e4m3_decode(codes) * np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32, axis=1)


def prepared(moe, dev):
    w13q, w13s, w2q, w2s = moe.prepare_weights_mxfp8(dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    return w13q, w13s, w2q, w2s


def run_mx(moe, inp, dev, prep):
    c = inp["cfg"]
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"], precision=moe.MOE_PREC_MXFP8,
                       clamp=c.get("clamp", 0.0), flags=0)
    w13q, w13s, w2q, w2s = prep
    y = plan.forward(dev["x"], dev["ids"], dev["scores"], w13q, w2q, w13_sf=w13s, w2_sf=w2s)
    torch.cuda.synchronize()
    rc, det = plan.check()
    assert rc == 0, (rc, det)
    return plan, y


@pytest.mark.parametrize("sizes", [
    dict(T=64, d=128, I=128, E=4, k=2),
    dict(T=300, d=256, I=256, E=7, k=3),
    dict(T=200, d=384, I=128, E=9, k=2, clamp=1.0, pad=30),
    dict(T=400, d=128, I=128, E=12, k=3, routing="zipf", zipf_s=1.2, zipf_support=8),
    dict(T=1, d=128, I=128, E=4, k=2),
    dict(T=96, d=128, I=128, E=256, k=8),
], ids=["tiny", "ragged", "clamped_pad", "skew_empty", "one_token", "k8_e256"])
def test_mxfp8_small(moe, orc, sizes):
    inp = mi.make_inputs(None, seed=21, need=("x", "ids", "scores", "w13", "w2"), **sizes)
    c = inp["cfg"]
    T, d, I, E, k = c["T"], c["d"], c["I"], c["E"], c["k"]
    dev = to_dev(inp)
    prep = prepared(moe, dev)
    # prepared weights: bit-exact against the oracle's quantiser
    oq13, os13 = orc.quant_mxfp8(inp["w13"])
    oq2, os2 = orc.quant_mxfp8(inp["w2"])
    assert np.array_equal(prep[0].cpu().numpy(), oq13)
    assert np.array_equal(prep[2].cpu().numpy(), oq2)
    assert np.array_equal(untile(prep[1].cpu().numpy(), E * 2 * I, d, gu_I=I),
                          os13.reshape(E * 2 * I, d // 32))
    assert np.array_equal(untile(prep[3].cpu().numpy(), E * d, I), os2.reshape(E * d, I // 32))
    plan, y = run_mx(moe, inp, dev, prep)
    # quantised routed activations: bit-exact (padding rows zero)
    op = plan.buffer("off_pad", torch.int32).cpu().numpy()
    n = int(op[-1])
    tok = plan.buffer("token_of", torch.int32).cpu().numpy()[:n]
    xrows = orc.gather_rows(inp["x"], tok)
    qx, sx = orc.quant_mxfp8(xrows)
    gq = plan.buffer("xq", torch.uint8).cpu().numpy()[: n * d].reshape(n, d)
    assert np.array_equal(gq, qx)
    gs = untile(plan.buffer("xsf", torch.uint8).cpu().numpy(), n, d)
    assert np.array_equal(gs, sx)
    # output
    yref, href = orc.forward_mxfp8(inp["x"], inp["ids"], inp["scores"], oq13, os13, oq2, os2,
                                   clamp=c.get("clamp", 0.0), return_h=True)
    compare(f32(bits(y)), f32(yref), bf16_out=True, rel_fro=REL_FRO_MXFP8, what="y mxfp8",
            max_bad_frac=1.0)
    # h quantised along I (the W2 GEMM's A operand): the dequantised codes against
    # the oracle's h quantised by the oracle; a code may differ by one step where
    # the two h values differ in their last bf16 bit
    ro = plan.buffer("row_of", torch.int32).cpu().numpy()[: T * k].reshape(T, k)
    ok = ro >= 0
    rows = ro[ok]
    hq_all = plan.buffer("hq", torch.uint8).cpu().numpy()
    RP = hq_all.size // I
    hq = hq_all.reshape(RP, I)[rows]
    hs = untile(plan.buffer("hsf", torch.uint8).cpu().numpy(), RP, I)[rows]
    qh, sh = orc.quant_mxfp8(href[ok])
    compare(dequant(orc, hq, hs), dequant(orc, qh, sh), bf16_out=False, rel_fro=REL_FRO_MXFP8,
            what="hq mxfp8", max_bad_frac=1e-2)
    assert np.mean(hq == qh) > 0.99


def test_mxfp8_full_size_sampled(moe, orc):
    inp = mi.make_inputs("mxfp8_e128", need=("x", "ids", "scores", "w13", "w2"))
    c = inp["cfg"]
    dev = to_dev(inp)
    prep = prepared(moe, dev)
    plan, y = run_mx(moe, inp, dev, prep)
    yb = f32(bits(y))
    assert np.all(np.isfinite(yb))
    rng = np.random.default_rng(5)
    toks = np.array(sorted(set(rng.choice(c["T"], 1024, replace=False).tolist())
                           | {0, c["T"] - 1}), np.int32)
    # prepared weights of every expert: bit-exact against the oracle's quantiser
    I, d, E = c["I"], c["d"], c["E"]
    oq13, os13 = orc.quant_mxfp8(inp["w13"])
    oq2, os2 = orc.quant_mxfp8(inp["w2"])
    assert np.array_equal(prep[0].cpu().numpy(), oq13)
    assert np.array_equal(untile(prep[1].cpu().numpy(), E * 2 * I, d, gu_I=I),
                          os13.reshape(E * 2 * I, d // 32))
    assert np.array_equal(prep[2].cpu().numpy(), oq2)
    assert np.array_equal(untile(prep[3].cpu().numpy(), E * d, I), os2.reshape(E * d, I // 32))
    yref = orc.forward_mxfp8(inp["x"], inp["ids"], inp["scores"], oq13, os13, oq2, os2, toks=toks)
    compare(yb[toks], f32(yref), bf16_out=True, rel_fro=REL_FRO_MXFP8, what="y mxfp8 full",
            max_bad_frac=1.0)
