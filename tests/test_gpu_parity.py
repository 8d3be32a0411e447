"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Dispatch tables and gathered rows: bit-exact.  Floating-point results: within
the stated tolerance (tests/parity.py).  Small cases compare every output and
every intermediate; they span several GEMM tiles, ragged expert segments, empty
experts, padding tokens and the clamped SwiGLU.
"""

import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_case import bits, check_backward, check_dispatch, check_forward, make, run_gpu
from parity import f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


def test_tiny_forward(moe, orc):
    inp = make("tiny_fwd", train=False)
    g = run_gpu(moe, inp, train=False)
    assert g["rc"] == 0
    check_dispatch(orc, inp, g)
    check_forward(orc, inp, g)


def test_gathered_rows_bit_exact(moe, orc):
    # the gather of a saving forward: bit-exact copies, padding rows zero
    inp = make("tiny_fwd", train=True)
    g = run_gpu(moe, inp, train=True)
    assert g["rc"] == 0
    r = check_dispatch(orc, inp, g)
    c = inp["cfg"]
    tok = g["plan"].buffer("token_of", torch.int32).cpu().numpy()[: r["off_pad"][-1]]
    xe = bits(g["plan"].buffer("xe", torch.bfloat16).view(-1, c["d"]))[: r["off_pad"][-1]]
    assert np.array_equal(xe, orc.gather_rows(inp["x"], tok))


SMALL = [
    # name, sizes, extra
    ("tiny_train", dict(T=64, d=128, I=64, E=4, k=2), {}),
    ("ragged", dict(T=300, d=256, I=192, E=7, k=3), {}),
    ("wide", dict(T=517, d=384, I=128, E=16, k=4), {}),
    ("clamped_pad", dict(T=200, d=256, I=128, E=9, k=2, clamp=1.0, pad=37), {}),
    ("skew_empty", dict(T=400, d=128, I=256, E=12, k=3, routing="zipf", zipf_s=1.2,
                        zipf_support=8), {}),
    ("single_expert", dict(T=130, d=128, I=64, E=1, k=1), {}),
    ("one_token", dict(T=1, d=128, I=64, E=4, k=2), {}),
    ("k8_e256", dict(T=96, d=128, I=64, E=256, k=8), {}),
    # more than eight experts per token: the combine's general-k kernel
    ("k16", dict(T=150, d=128, I=64, E=40, k=16), {}),
    ("k11_pad", dict(T=90, d=256, I=128, E=24, k=11, pad=10), {}),
    # W13, W2 and DGRAD-W13 on CTA pairs (moe_plan_set_cta_pairs): pairs of an
    # expert's m tiles on the pair kernel, an odd last m tile on one CTA
    ("pairs", dict(T=300, d=256, I=256, E=6, k=3, cta_pairs=True), {}),
    ("pairs_odd_tiles", dict(T=700, d=256, I=256, E=6, k=3, cta_pairs=True), {}),
    ("pairs_clamp_pad", dict(T=200, d=512, I=256, E=9, k=2, clamp=1.0, pad=20, cta_pairs=True),
     {}),
    ("pairs_skew", dict(T=400, d=256, I=512, E=12, k=3, routing="zipf", zipf_s=1.2,
                        zipf_support=8, cta_pairs=True), {}),
    ("same_sizes_one_cta", dict(T=300, d=256, I=256, E=6, k=3), {}),
]


@pytest.mark.parametrize("name,sizes,extra", SMALL, ids=[s[0] for s in SMALL])
def test_small_forward_backward(moe, orc, name, sizes, extra):
    inp = make(None, seed=len(name), train=True, **sizes)
    g = run_gpu(moe, inp, train=True)
    assert g["rc"] == 0, g
    check_dispatch(orc, inp, g)
    check_forward(orc, inp, g)
    check_backward(orc, inp, g)


@pytest.mark.parametrize("sizes", [dict(T=300, d=256, I=192, E=7, k=3),
                                   dict(T=2048, d=512, I=256, E=32, k=8, routing="zipf",
                                        zipf_s=1.2, zipf_support=24)], ids=["ragged", "skew"])
def test_backward_split_is_bit_identical(moe, sizes):
    """Weight gradients on their own stream and SMs beside DGRAD-W13: the same bits
    as one stream, for every output, twice in a row."""
    inp = make(None, seed=61, train=True, **sizes)
    ref = run_gpu(moe, inp, train=True)
    assert ref["rc"] == 0
    dev = ref["dev"]
    plan = ref["plan"]
    plan.set_backward_split(plan.num_sms() // 2)
    for _ in range(2):
        dw13, dw2 = dev["dw13"].clone(), dev["dw2"].clone()
        plan.forward(dev["x"], dev["ids"], dev["scores"], dev["w13"], dev["w2"], save=True)
        dx, ds = plan.backward(dev["dy"], dev["w13"], dev["w2"], dw13, dw2)
        torch.cuda.synchronize()
        assert plan.check()[0] == 0
        assert torch.equal(dx.view(torch.int16), ref["dx"].view(torch.int16))
        assert torch.equal(ds, ref["dscores"])
        assert torch.equal(dw13, ref["dw13"]) and torch.equal(dw2, ref["dw2"])


@pytest.mark.parametrize("min_rows,split", [(0, False), (128, False), (1024, False), (128, True)],
                         ids=["plain", "interleave128", "interleave1024", "interleave128_split"])
def test_wgrad_interleave_is_bit_identical(moe, min_rows, split):
    """Weight-gradient tiles of the heavy experts run in pieces interleaved with
    lighter tiles on the other accumulator (the default threshold, 2560 rows,
    splits this case's heaviest experts; 128 rows splits nearly every tile):
    every output has the same bits as with the plain order (0) and as with the
    default, since each tile still sums its K range in order; also with the
    weight gradients on their own stream and half the SMs."""
    sizes = dict(T=4096, d=512, I=256, E=32, k=8, routing="zipf", zipf_s=1.2, zipf_support=24)
    inp = make(None, seed=62, train=True, **sizes)
    counts = np.bincount(inp["ids"].reshape(-1), minlength=sizes["E"])
    assert counts.max() > 2560
    ref = run_gpu(moe, inp, train=True)
    assert ref["rc"] == 0
    dev = ref["dev"]
    plan = ref["plan"]
    plan.set_wgrad_interleave(min_rows)
    if split:   # weight gradients on their own stream and half the SMs
        plan.set_backward_split(plan.num_sms() // 2)
    dw13, dw2 = dev["dw13"].clone(), dev["dw2"].clone()
    plan.forward(dev["x"], dev["ids"], dev["scores"], dev["w13"], dev["w2"], save=True)
    dx, ds = plan.backward(dev["dy"], dev["w13"], dev["w2"], dw13, dw2)
    torch.cuda.synchronize()
    assert plan.check()[0] == 0
    assert torch.equal(dx.view(torch.int16), ref["dx"].view(torch.int16))
    assert torch.equal(ds, ref["dscores"])
    assert torch.equal(dw13, ref["dw13"]) and torch.equal(dw2, ref["dw2"])


def test_wgrad_interleave_rejects_bad_threshold(moe):
    plan = moe.MoePlan(64, 128, 64, 4, 2, flags=moe.MOE_WS_TRAINING)
    with pytest.raises(moe.MoeError):
        plan.set_wgrad_interleave(-1)


def test_zero_score_padding_rows_are_zero(moe):
    inp = make(None, seed=5, train=True, T=160, d=128, I=64, E=6, k=2, pad=40)
    g = run_gpu(moe, inp, train=True)
    y = f32(bits(g["y"]))
    dx = f32(bits(g["dx"]))
    assert np.all(y[-40:] == 0) and np.all(dx[-40:] == 0)
    assert np.all(np.abs(g["dscores"].cpu().numpy()[-40:]) > 0)


def test_forward_is_deterministic(moe):
    inp = make(None, seed=6, train=True, T=300, d=256, I=128, E=8, k=4)
    g1 = run_gpu(moe, inp, train=True)
    g2 = run_gpu(moe, inp, train=True)
    for key in ("y", "dx", "dscores", "dw13", "dw2"):
        assert torch.equal(g1[key], g2[key]), key


def test_weight_gradients_accumulate(moe):
    """Running the backward twice adds the increment twice (in-place +=)."""
    inp = make(None, seed=7, train=True, T=256, d=128, I=64, E=4, k=2)
    g = run_gpu(moe, inp, train=True)
    plan, dev = g["plan"], g["dev"]
    d13_1 = g["dw13"].double() - dev["dw13"].double()
    plan.backward(dev["dy"], dev["w13"], dev["w2"], g["dw13"], g["dw2"])
    torch.cuda.synchronize()
    d13_2 = g["dw13"].double() - dev["dw13"].double()
    assert torch.allclose(d13_2, 2 * d13_1, rtol=1e-5, atol=1e-6)


def test_bad_ids_are_reported(moe):
    inp = make(None, seed=8, train=False, T=100, d=128, I=64, E=8, k=3)
    ids = inp["ids"].copy()
    ids[40, 2] = ids[40, 0]       # repeated id, flat index 122
    ids[70, 1] = 8                # out of range, flat index 211
    inp["ids"] = ids
    g = run_gpu(moe, inp, train=False)
    assert g["rc"] == moe.MOE_ERR_BAD_IDS
    assert g["detail"] == 122
    # the error word is cleared by the check
    assert g["plan"].check() == (0, 0)


def test_all_ids_invalid(moe):
    # every routed element dropped: no rows reach any expert, so the GEMMs have no
    # tiles; y and dx are zero, dscores zero, the weight gradients untouched
    inp = make(None, seed=10, train=True, T=50, d=128, I=64, E=4, k=2)
    inp["ids"] = np.full_like(inp["ids"], 4)       # out of range for E = 4
    g = run_gpu(moe, inp, train=True)
    assert g["rc"] == moe.MOE_ERR_BAD_IDS and g["detail"] == 0
    assert not g["y"].any() and not g["dx"].any() and not g["dscores"].any()
    assert torch.equal(g["dw13"], g["dev"]["dw13"]) and torch.equal(g["dw2"], g["dev"]["dw2"])
    assert int(g["plan"].buffer("off_pad", torch.int32)[-1]) == 0


def test_backward_needs_saving_forward(moe):
    inp = make(None, seed=9, train=True, T=64, d=128, I=64, E=4, k=2)
    dev = {k: v for k, v in __import__("gpu_case").to_dev(inp).items()}
    plan = moe.MoePlan(64, 128, 64, 4, 2, flags=moe.MOE_WS_TRAINING)
    with pytest.raises(moe.MoeError) as ei:
        plan.backward(dev["dy"], dev["w13"], dev["w2"], dev["dw13"], dev["dw2"])
    assert ei.value.code == moe.MOE_ERR_STATE
    plan.forward(dev["x"], dev["ids"], dev["scores"], dev["w13"], dev["w2"], save=False)
    with pytest.raises(moe.MoeError):
        plan.backward(dev["dy"], dev["w13"], dev["w2"], dev["dw13"], dev["dw2"])
    inf_plan = moe.MoePlan(64, 128, 64, 4, 2, flags=0)
    with pytest.raises(moe.MoeError) as ei:
        inf_plan.forward(dev["x"], dev["ids"], dev["scores"], dev["w13"], dev["w2"], save=True)
    assert ei.value.code == moe.MOE_ERR_WORKSPACE


def test_host_step_matches_device_path(moe):
    inp = make(None, seed=10, train=True, T=200, d=256, I=128, E=8, k=4)
    g = run_gpu(moe, inp, train=True)
    c = inp["cfg"]
    dev = g["dev"]
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"],
                       flags=moe.MOE_WS_TRAINING | moe.MOE_WS_HOST_STAGING)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    x_h = pin(inp["x"]).view(torch.bfloat16)
    dy_h = pin(inp["dy"]).view(torch.bfloat16)
    ids_h, sc_h = pin(inp["ids"]), pin(inp["scores"])
    y_h = torch.empty(c["T"], c["d"], dtype=torch.bfloat16).pin_memory()
    dx_h = torch.empty(c["T"], c["d"], dtype=torch.bfloat16).pin_memory()
    ds_h = torch.empty(c["T"], c["k"], dtype=torch.float32).pin_memory()
    dw13, dw2 = dev["dw13"].clone(), dev["dw2"].clone()
    plan.step_host(x_h, ids_h, sc_h, dev["w13"], dev["w2"], y_h, dy_h, dw13, dw2, dx_h, ds_h)
    torch.cuda.synchronize()
    assert torch.equal(y_h, g["y"].cpu())
    assert torch.equal(dx_h, g["dx"].cpu())
    assert torch.equal(ds_h, g["dscores"].cpu())
    assert torch.equal(dw13, g["dw13"]) and torch.equal(dw2, g["dw2"])


def test_host_steps_back_to_back(moe):
    """Training steps from host buffers enqueued without synchronising in between:
    a step's uploads may overlap the previous step's weight gradients, and each
    step must still give the outputs of its own inputs."""
    c0 = dict(T=200, d=256, I=128, E=8, k=4)
    a = make(None, seed=12, train=True, **c0)
    b = make(None, seed=13, train=True, **c0)
    b2 = dict(a)                         # same weights, other tokens, routing and dY
    for key in ("x", "ids", "scores", "dy"):
        b2[key] = b[key]
    inps = [a, b2]
    refs = [run_gpu(moe, inp, train=True) for inp in inps]
    c = inps[0]["cfg"]
    plan = moe.MoePlan(c["T"], c["d"], c["I"], c["E"], c["k"],
                       flags=moe.MOE_WS_TRAINING | moe.MOE_WS_HOST_STAGING)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    dev = refs[0]["dev"]
    dw13, dw2 = dev["dw13"].clone(), dev["dw2"].clone()
    # training steps with alternating inputs, an inference step in between
    order = [(0, True), (1, True), (0, False), (1, True), (0, True)]
    outs = []
    for i, train in order:
        inp = inps[i]
        h = dict(x=pin(inp["x"]).view(torch.bfloat16), dy=pin(inp["dy"]).view(torch.bfloat16),
                 ids=pin(inp["ids"]), sc=pin(inp["scores"]),
                 y=torch.empty(c["T"], c["d"], dtype=torch.bfloat16).pin_memory(),
                 dx=torch.empty(c["T"], c["d"], dtype=torch.bfloat16).pin_memory(),
                 ds=torch.empty(c["T"], c["k"], dtype=torch.float32).pin_memory())
        if train:
            plan.step_host(h["x"], h["ids"], h["sc"], dev["w13"], dev["w2"], h["y"], h["dy"], dw13,
                           dw2, h["dx"], h["ds"])
        else:
            plan.step_host(h["x"], h["ids"], h["sc"], dev["w13"], dev["w2"], h["y"])
        outs.append(h)
    torch.cuda.synchronize()
    for (i, train), h in zip(order, outs):
        assert torch.equal(h["y"], refs[i]["y"].cpu())
        if train:
            assert torch.equal(h["dx"], refs[i]["dx"].cpu())
            assert torch.equal(h["ds"], refs[i]["dscores"].cpu())
    # the weight gradients received every step's increment
    want13 = dev["dw13"] + 2 * (refs[0]["dw13"] - dev["dw13"]) + 2 * (refs[1]["dw13"] - dev["dw13"])
    want2 = dev["dw2"] + 2 * (refs[0]["dw2"] - dev["dw2"]) + 2 * (refs[1]["dw2"] - dev["dw2"])
    # (two training steps of each input)
    assert torch.allclose(dw13, want13, rtol=1e-4, atol=1e-4)
    assert torch.allclose(dw2, want2, rtol=1e-4, atol=1e-4)
    assert plan.check() == (0, 0)


def test_mxfp8_quantiser_bit_exact(moe, orc):
    rng = np.random.default_rng(3)
    w = rng.standard_normal((96, 512)).astype(np.float32) * \
        (2.0 ** rng.integers(-30, 30, (96, 1))).astype(np.float32)
    w[5, 64:96] = 0.0
    wb = mi.to_bf16_bits(w)
    codes, scales = orc.quant_mxfp8(wb)
    t = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).cuda()
    gc, gs = moe.quantize_mxfp8(t)
    torch.cuda.synchronize()
    assert np.array_equal(gc.cpu().numpy(), codes)
    assert np.array_equal(gs.cpu().numpy(), scales)


def _bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_clamp_gradient_boundary(moe, orc):
    """Clamped SwiGLU on the GPU: where the bf16 pre-activation is exactly -L or
    L the gradient passes, one bf16 step outside it is exactly zero (the oracle
    takes the same decisions, pinned on the CPU).  x = e_0 with one expert, so
    every gate and up value is one weight exactly."""
    T, d, I, E, k, L = 1, 128, 64, 1, 1, 1.0
    out = 1.0078125                         # the bf16 value just above 1.0
    gate = np.full(I, 0.5)
    up = np.full(I, 0.5)
    gate[[0, 1, 2, 3]] = [L, -L, out, -out]
    up[[4, 5, 6, 7]] = [L, -L, out, -out]
    x = np.zeros((T, d), np.float32)
    x[0, 0] = 1.0
    w13 = np.zeros((E, 2 * I, d), np.float32)
    w13[0, :I, 0] = gate
    w13[0, I:, 0] = up
    rng = np.random.default_rng(7)
    inp = dict(x=_bf16_bits(x), ids=np.zeros((T, k), np.int32),
               scores=np.ones((T, k), np.float32), w13=_bf16_bits(w13),
               w2=_bf16_bits(rng.normal(0, I ** -0.5, (E, d, I))),
               dy=_bf16_bits(rng.normal(0, 1, (T, d))),
               dw13=np.zeros((E, 2 * I, d), np.float32), dw2=np.zeros((E, d, I), np.float32),
               cfg=dict(T=T, d=d, I=I, E=E, k=k, clamp=L))
    g = run_gpu(moe, inp, train=True)
    assert g["rc"] == 0
    dA = f32(bits(g["plan"].buffer("dA", torch.bfloat16)))[: 2 * I].astype(np.float64)
    dg, du = dA[:I], dA[I:]
    assert np.all(dg[[2, 3]] == 0) and np.all(du[[6, 7]] == 0)
    _, _, bi = orc.backward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"],
                            inp["dy"], clamp=L, intermediates=True)
    ref = f32(bi["dA"])[0, 0].astype(np.float64)
    for i in (0, 1, 8):
        assert dg[i] != 0 and abs(dg[i] - ref[i]) <= 2.0 ** -7 * abs(ref[i]), i
    for i in (4, 5, 8):
        assert du[i] != 0 and abs(du[i] - ref[I + i]) <= 2.0 ** -7 * abs(ref[I + i]), i
