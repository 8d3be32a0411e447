"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks the oracle against a library routine (torch FP64 autograd,
numpy's stable sort, torch's bf16 / float8 conversions), a closed form, an
invariant of the method, or a hand-worked example, chosen so that a plausible
slip (a swapped gate/up, a dropped score, a transposed weight, a wrong rounding
point, an off-by-one in the scan) fails at least one of them.
"""

import json
import os

import numpy as np
import pytest
import torch

import moe_inputs as mi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bits(f):
    return torch.from_numpy(np.ascontiguousarray(f, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def small(T=24, d=64, I=32, E=5, k=3, seed=3, routing="uniform", pad=0, **kw):
    inp = mi.make_inputs(None, seed=seed, T=T, d=d, I=I, E=E, k=k, routing=routing, pad=pad,
                         need=("x", "ids", "scores", "w13", "w2", "dy"), **kw)
    return inp


# ---------------------------------------------------------------------------
# worked example


def test_worked_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    x = bits(np.array(g["x"]))
    w13 = bits(np.array(g["w13"]))
    w2 = bits(np.array(g["w2"]))
    ids = np.array(g["ids"], np.int32)
    sc = np.array(g["scores"], np.float32)
    dy = bits(np.array(g["dy"]))
    ex = {k: np.array(v) for k, v in g["expect"].items()}
    y, it = orc.forward(x, ids, sc, w13, w2, intermediates=True)
    assert np.array_equal(f32(y), ex["y"])
    assert np.array_equal(f32(it["a"]), ex["a"])
    assert np.array_equal(f32(it["h"]), ex["h"])
    assert np.array_equal(f32(it["ys"]), ex["ys"])
    dx, ds, bi = orc.backward(x, ids, sc, w13, w2, dy, intermediates=True)
    assert np.array_equal(f32(dx), ex["dx"])
    assert np.array_equal(ds, ex["dscores"].astype(np.float32))
    assert np.array_equal(f32(bi["dA"]), ex["dA"])
    assert np.array_equal(f32(bi["hs"]), ex["hs"])
    for e in range(2):
        d13, d2, rows = orc.wgrad_expert(x, ids, sc, w13, w2, dy, e)
        assert rows == 2
        assert np.array_equal(d13, ex["dw13_delta"][e].astype(np.float32))
        assert np.array_equal(d2, ex["dw2_delta"][e].astype(np.float32))


# ---------------------------------------------------------------------------
# conversions


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 100000).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1e-40, -1e-40, np.inf, -np.inf], np.float32),
        # exact ties between two bf16 neighbours
        (f32(np.arange(0x3f80, 0x3fa0, dtype=np.uint16)) +
         np.float32(2.0 ** -8)).astype(np.float32),
    ]).astype(np.float32)
    assert np.array_equal(orc.float_to_bf16(v), bits(v))


# ---------------------------------------------------------------------------
# dispatch


@pytest.mark.parametrize("T,k,E,BM", [(64, 2, 4, 128), (300, 8, 128, 128), (257, 3, 17, 64),
                                      (1000, 8, 256, 128), (5, 1, 1, 128)])
def test_dispatch_is_stable_counting_sort(orc, T, k, E, BM):
    ids = mi.draw_ids(T, k, E, seed=T + E)
    r = orc.dispatch(ids, E, BM)
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")          # library stable sort by expert
    counts = np.bincount(flat, minlength=E)
    assert r["first_bad"] == -1
    assert np.array_equal(r["counts"], counts)
    assert r["m_indptr"][0] == 0 and r["m_indptr"][-1] == T * k
    assert np.array_equal(np.diff(r["m_indptr"]), counts)
    padded = -(-counts // BM) * BM
    assert np.array_equal(np.diff(r["off_pad"]), padded)
    # position in the sorted order minus the expert's start = rank within the expert
    rank = np.empty(T * k, np.int64)
    rank[order] = np.arange(T * k) - np.repeat(np.concatenate([[0], np.cumsum(counts)[:-1]]), counts)
    assert np.array_equal(r["rank_of"].reshape(-1), rank)
    rows = r["row_of"].reshape(-1)
    assert np.array_equal(rows, r["off_pad"][flat] + rank)
    assert len(np.unique(rows)) == T * k                       # injective
    assert rows.max() < r["off_pad"][-1]


def test_dispatch_flags_invalid_ids(orc):
    ids = mi.draw_ids(50, 4, 16, seed=1).copy()
    ids[7, 2] = ids[7, 0]          # duplicate within a row (flat 30)
    ids[20, 1] = 16                # out of range (flat 81)
    ids[3, 3] = -1                 # out of range (flat 15)
    r = orc.dispatch(ids, 16, 128)
    assert r["first_bad"] == 15
    bad = {15, 30, 81}
    for f in range(200):
        if f in bad:
            assert r["row_of"].reshape(-1)[f] == -1
        else:
            assert r["row_of"].reshape(-1)[f] >= 0
    assert r["m_indptr"][-1] == 200 - 3


def _token_of(row_of, nrows):
    tok = np.full(nrows, -1, np.int32)
    T, k = row_of.shape
    for t in range(T):
        for j in range(k):
            if row_of[t, j] >= 0:
                tok[row_of[t, j]] = t
    return tok


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_gather_combine_identity_experts(orc, k):
    """Identity experts: combine(gather(x)) with one-hot scores returns x exactly,
    with unit scores k*x exactly (k a power of two)."""
    T, d, E = 40, 64, 8
    inp = mi.make_inputs(None, seed=k, T=T, d=d, I=32, E=E, k=k, need=("x", "ids"))
    r = orc.dispatch(inp["ids"], E, 16)
    nrows = int(r["off_pad"][-1])
    tok = _token_of(r["row_of"], nrows)
    xe = orc.gather_rows(inp["x"], tok)
    assert np.array_equal(xe[tok < 0], np.zeros_like(xe[tok < 0]))
    assert np.array_equal(xe[tok >= 0], inp["x"][tok[tok >= 0]])
    # unit scores
    y = orc.combine_rows(xe, r["row_of"])
    assert np.array_equal(f32(y), f32(inp["x"]) * k)
    # one-hot scores: keep only the column j0 = t % k
    ys = xe.copy()
    for t in range(T):
        for j in range(k):
            if j != t % k:
                ys[r["row_of"][t, j]] = 0
    y1 = orc.combine_rows(ys, r["row_of"])
    assert np.array_equal(y1, inp["x"])


# ---------------------------------------------------------------------------
# forward against an FP64 brute force (every expert for every token, then select)


def _dense_fp64(inp, clamp=0.0):
    x = torch.from_numpy(f32(inp["x"]).astype(np.float64))
    W13 = torch.from_numpy(f32(inp["w13"]).astype(np.float64))
    W2 = torch.from_numpy(f32(inp["w2"]).astype(np.float64))
    I = W2.shape[2]
    gu = torch.einsum("td,eid->eti", x, W13)             # [E, T, 2I]
    g, u = gu[..., :I], gu[..., I:]
    if clamp:
        g, u = g.clamp(-clamp, clamp), u.clamp(-clamp, clamp)
    h = torch.nn.functional.silu(g) * u
    o = torch.einsum("eti,edi->etd", h, W2)              # [E, T, d]
    ids = torch.from_numpy(inp["ids"]).long()
    s = torch.from_numpy(inp["scores"]).double()
    T = x.shape[0]
    sel = o[ids, torch.arange(T)[:, None]]               # [T, k, d]
    return (s[..., None] * sel).sum(1).numpy()


def _rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("clamp", [0.0, 1.0])
def test_forward_matches_fp64_bruteforce(orc, clamp):
    inp = small(T=40, d=128, I=64, E=6, k=3, seed=11)
    y = f32(orc.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"], clamp=clamp))
    ref = _dense_fp64(inp, clamp)
    # bf16 rounding at four points: about 2^-9 relative each
    assert _rel_fro(y, ref) < 8e-3
    assert np.max(np.abs(y - ref)) < 3e-2 * np.sqrt(np.mean(ref ** 2)) + 2 ** -8 * np.abs(ref).max()


def test_forward_single_expert_is_dense_swiglu_mlp(orc):
    """E=1, k=1, score 1: the routed layer is a dense SwiGLU MLP (torch CPU ops,
    rounding to bf16 at the same points)."""
    inp = small(T=33, d=128, I=64, E=1, k=1, seed=5)
    inp["scores"][:] = 1.0
    y = orc.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"])
    x = torch.from_numpy(f32(inp["x"]))
    W13 = torch.from_numpy(f32(inp["w13"][0]))
    W2 = torch.from_numpy(f32(inp["w2"][0]))
    a = (x @ W13.T).to(torch.bfloat16).float()
    h = (torch.nn.functional.silu(a[:, :64]) * a[:, 64:]).to(torch.bfloat16).float()
    ref = (h @ W2.T).to(torch.bfloat16).float().numpy()
    yy = f32(y)
    # the only differences are FP32 summation order -> at most one bf16 step, rarely
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert np.mean(np.abs(yy - ref) <= ulp) == 1.0
    assert np.mean(yy == ref) > 0.97


def test_zero_score_padding_tokens_give_zero(orc):
    inp = small(T=20, d=64, I=32, E=4, k=2, seed=9, pad=6)
    y = f32(orc.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"]))
    assert np.all(y[-6:] == 0)
    assert np.all(np.abs(y[:-6]).sum(1) > 0)


def test_forward_gate_up_order_matters(orc):
    """Swapping the gate and up halves of W13 changes the output by O(1):
    the pins above would catch a swapped reading."""
    inp = small(T=16, d=64, I=32, E=3, k=2, seed=2)
    y = f32(orc.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"]))
    w = inp["w13"].copy()
    w = np.concatenate([w[:, 32:], w[:, :32]], axis=1)
    y2 = f32(orc.forward(inp["x"], inp["ids"], inp["scores"], np.ascontiguousarray(w), inp["w2"]))
    assert _rel_fro(y2, y) > 0.3


# ---------------------------------------------------------------------------
# backward against torch autograd in FP64 (rounding-free)


def _autograd_fp64(inp, clamp=0.0):
    x = torch.from_numpy(f32(inp["x"]).astype(np.float64)).requires_grad_()
    W13 = torch.from_numpy(f32(inp["w13"]).astype(np.float64)).requires_grad_()
    W2 = torch.from_numpy(f32(inp["w2"]).astype(np.float64)).requires_grad_()
    s = torch.from_numpy(inp["scores"].astype(np.float64)).requires_grad_()
    ids = torch.from_numpy(inp["ids"]).long()
    T, k = ids.shape
    I = W2.shape[2]
    Wsel = W13[ids]                                       # [T, k, 2I, d]
    gu = torch.einsum("td,tkid->tki", x, Wsel)
    # the clamp decision is taken on the bf16-rounded pre-activation (R1); round
    # the value, pass the gradient straight through
    gu = gu + (gu.detach().float().to(torch.bfloat16).double() - gu.detach())
    g, u = gu[..., :I], gu[..., I:]
    if clamp:
        g, u = g.clamp(-clamp, clamp), u.clamp(-clamp, clamp)
    h = torch.nn.functional.silu(g) * u
    o = torch.einsum("tki,tkdi->tkd", h, W2[ids])
    y = (s[..., None] * o).sum(1)
    dy = torch.from_numpy(f32(inp["dy"]).astype(np.float64))
    (y * dy).sum().backward()
    return dict(dx=x.grad.numpy(), ds=s.grad.numpy(), dw13=W13.grad.numpy(), dw2=W2.grad.numpy())


@pytest.mark.parametrize("clamp", [0.0, 0.75])
def test_backward_matches_fp64_autograd(orc, clamp):
    inp = small(T=40, d=64, I=32, E=5, k=3, seed=21)
    ref = _autograd_fp64(inp, clamp)
    dx, ds = orc.backward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"], inp["dy"],
                          clamp=clamp)
    assert _rel_fro(f32(dx), ref["dx"]) < 2e-2
    assert _rel_fro(ds, ref["ds"]) < 2e-2
    for e in range(5):
        d13, d2, rows = orc.wgrad_expert(inp["x"], inp["ids"], inp["scores"], inp["w13"],
                                         inp["w2"], inp["dy"], e, clamp=clamp)
        assert rows == int((inp["ids"] == e).sum())
        assert _rel_fro(d13, ref["dw13"][e]) < 2e-2
        assert _rel_fro(d2, ref["dw2"][e]) < 2e-2


def test_clamp_gradient_boundary(orc):
    """Clamped SwiGLU (limit L): the gradient passes where the bf16 pre-activation
    equals -L or L exactly and is exactly zero one bf16 step outside; where it
    passes it is the closed form dh*U*sigma(G)*(1 + G*(1 - sigma(G))) (gate) or
    dh*silu(G)*[G clamped] (up), rounded to bf16.  One token, one expert, x = e_0,
    so every gate and up value is one weight exactly."""
    d, I, L = 64, 32, 1.0
    out = 1.0078125                         # the bf16 value just above 1.0
    gate = np.full(I, 0.5)
    up = np.full(I, 0.5)
    gate[[0, 1, 2, 3]] = [L, -L, out, -out]
    up[[4, 5, 6, 7]] = [L, -L, out, -out]
    x = np.zeros((1, d), np.float32)
    x[0, 0] = 1.0
    w13 = np.zeros((1, 2 * I, d), np.float32)
    w13[0, :I, 0] = gate
    w13[0, I:, 0] = up
    rng = np.random.default_rng(5)
    w2 = rng.normal(0, I ** -0.5, (1, d, I)).astype(np.float32)
    dy = rng.normal(0, 1, (1, d)).astype(np.float32)
    ids = np.zeros((1, 1), np.int32)
    scores = np.ones((1, 1), np.float32)
    args = (bits(x), ids, scores, bits(w13), bits(w2), bits(dy))
    _, _, it = orc.backward(*args, clamp=L, intermediates=True)
    dA = f32(it["dA"])[0, 0].astype(np.float64)
    dg, du = dA[:I], dA[I:]
    dh = it["g"][0, 0].astype(np.float64)           # score 1: dh = g
    assert np.all(dh[:8] != 0)
    assert np.all(dg[[2, 3]] == 0) and np.all(du[[6, 7]] == 0)
    G = np.clip(gate, -L, L)
    U = np.clip(up, -L, L)
    sig = 1.0 / (1.0 + np.exp(-G))
    ref_g = dh * U * sig * (1.0 + G * (1.0 - sig))
    ref_u = dh * G * sig
    for i in (0, 1, 8):                             # gate at +L, -L, inside
        assert dg[i] != 0 and abs(dg[i] - ref_g[i]) <= 2.0 ** -7 * abs(ref_g[i]), i
    for i in (4, 5, 8):                             # up at +L, -L, inside
        assert du[i] != 0 and abs(du[i] - ref_u[i]) <= 2.0 ** -7 * abs(ref_u[i]), i
    # outside the interval the forward uses the clamped value
    _, fi = orc.forward(*args[:5], clamp=L, intermediates=True)
    h = f32(fi["h"])[0, 0].astype(np.float64)
    silu_L = L / (1.0 + np.exp(-L))
    assert abs(h[2] - silu_L * 0.5) <= 2.0 ** -8 * silu_L * 0.5
    assert h[2] == h[0]                             # G = out clamps to the same L


def test_dscores_linearity_invariant(orc):
    """y is linear in each score, so dscores[t,j] = <dY_t, o_j> where o_j = ys_j / s_j."""
    inp = small(T=12, d=64, I=32, E=4, k=2, seed=4)
    _, it = orc.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"],
                        intermediates=True)
    _, ds = orc.backward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"], inp["dy"])
    dy = f32(inp["dy"])
    o = f32(it["ys"]) / inp["scores"][..., None]
    lhs = np.einsum("tkd,td->tk", o, dy)
    assert _rel_fro(ds, lhs) < 1e-2


def test_zero_score_padding_gradients(orc):
    """Padding tokens: no dX, no dW contribution, but their dscores are defined."""
    inp = small(T=20, d=64, I=32, E=4, k=2, seed=9, pad=6)
    dx, ds = orc.backward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"], inp["dy"])
    assert np.all(f32(dx)[-6:] == 0)
    assert np.all(np.abs(ds[-6:]) > 0)
    cut = {k: (v[:-6] if k in ("x", "ids", "scores", "dy") else v) for k, v in inp.items()}
    for e in range(4):
        a13, a2, _ = orc.wgrad_expert(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"],
                                      inp["dy"], e)
        b13, b2, _ = orc.wgrad_expert(cut["x"], cut["ids"], cut["scores"], inp["w13"], inp["w2"],
                                      cut["dy"], e)
        assert np.array_equal(a13, b13) and np.array_equal(a2, b2)


# ---------------------------------------------------------------------------
# the parallel build: every sum keeps its order, so the thread count changes nothing


def test_oracle_results_do_not_depend_on_thread_count(orc):
    inp = small(T=40, d=128, I=64, E=5, k=3, seed=21, clamp=1.0)
    args = (inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"])
    n_all = orc.threads()
    res = []
    try:
        for n in (1, max(n_all, 3)):
            orc.set_threads(n)
            y, fi = orc.forward(*args, clamp=1.0, intermediates=True)
            dx, ds, bi = orc.backward(*args, inp["dy"], clamp=1.0, intermediates=True)
            w = [orc.wgrad_expert(*args, inp["dy"], e, clamp=1.0) for e in range(5)]
            fw = orc.quant_mxfp8(inp["w13"]) + orc.quant_mxfp8(inp["w2"])
            bw = orc.prepare_mxfp8_backward_weights(inp["w13"], inp["w2"])
            mx = args[:3]
            _, _, mi = orc.backward_mxfp8(*mx, fw, bw, inp["dy"], clamp=1.0, intermediates=True)
            bi.update({"mx_" + key: v for key, v in mi.items()})
            w += [orc.wgrad_expert_mxfp8(*mx, fw, bw, inp["dy"], e, clamp=1.0) for e in range(5)]
            res.append((y, fi, dx, ds, bi, w))
    finally:
        orc.set_threads(n_all)
    (y1, f1, dx1, ds1, b1, w1), (yn, fn, dxn, dsn, bn, wn) = res
    assert np.array_equal(y1, yn) and np.array_equal(dx1, dxn) and np.array_equal(ds1, dsn)
    for key in f1:
        assert np.array_equal(f1[key], fn[key]), key
    for key in b1:
        assert np.array_equal(b1[key], bn[key]), key
    for (a13, a2, ra), (b13, b2, rb) in zip(w1, wn):
        assert ra == rb and np.array_equal(a13, b13) and np.array_equal(a2, b2)


# ---------------------------------------------------------------------------
# FP32 working type against the FP64 build of the same definition


def test_fp32_oracle_agrees_with_fp64_oracle(orc, orc64):
    inp = small(T=32, d=256, I=128, E=4, k=2, seed=8)
    y = f32(orc.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"]))
    y64 = f32(orc64.forward(inp["x"], inp["ids"], inp["scores"], inp["w13"], inp["w2"]))
    assert _rel_fro(y, y64) < 2e-3
    ulp = np.abs(y64) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(y - y64) <= 2 * ulp)


# ---------------------------------------------------------------------------
# MXFP8


def test_e4m3_decode_matches_torch_float8(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    ours = orc.e4m3_decode(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(ours, theirs)
    assert ours.max() == 448.0 and ours[codes == 0x01][0] == 2.0 ** -9


def test_e4m3_encode_roundtrip_and_ties(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_decode(codes)
    assert np.array_equal(orc.e4m3_encode(vals), codes)
    pos = np.sort(vals[vals > 0])
    mids = (pos[:-1] + pos[1:]) / 2
    enc = orc.e4m3_encode(mids)
    lo_code = orc.e4m3_encode(pos[:-1])
    expect = np.where(lo_code % 2 == 0, lo_code, lo_code + 1)   # ties to the even code
    assert np.array_equal(enc, expect)
    # saturation
    assert np.array_equal(orc.e4m3_encode(np.array([448.0, 460.0, 1e6, -1e9])),
                          np.array([0x7E, 0x7E, 0x7E, 0xFE], np.uint8))


def test_e4m3_encode_matches_torch_float8(orc):
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(200000) * 2.0 ** rng.uniform(-12, 10, 200000)).astype(np.float32)
    v = np.clip(v, -448, 448).astype(np.float64)
    ours = orc.e4m3_encode(v)
    theirs = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_mxfp8_block_scale_closed_form(orc):
    rng = np.random.default_rng(2)
    m = bits(rng.standard_normal((64, 256)).astype(np.float32) *
             (2.0 ** rng.integers(-20, 20, (64, 1))).astype(np.float32))
    m[3, 32:64] = 0                                   # an all-zero block
    codes, scales = orc.quant_mxfp8(m)
    v = f32(m).reshape(64, 8, 32).astype(np.float64)
    amax = np.abs(v).max(-1)
    _, ex = np.frexp(amax)
    X = np.clip(ex - 1 - 8, -127, 127)
    expect = np.where(amax == 0, 0, X + 127)
    assert np.array_equal(scales, expect.astype(np.uint8))
    scaled = v * 2.0 ** (-X[..., None])
    torch_codes = torch.from_numpy(np.clip(scaled, -448, 448).astype(np.float32).reshape(64, 256)) \
        .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    torch_codes[3, 32:64] = 0
    assert np.array_equal(codes, torch_codes)
    # every block's largest magnitude lands in [256, 448]
    dec = orc.e4m3_decode(codes).reshape(64, 8, 32)
    big = np.abs(dec).max(-1)[amax > 0]
    assert big.min() >= 256 and big.max() <= 448


def _deq_mx(b):
    """FP64 values of bf16 bits after MX quantisation along the last axis (32-element
    blocks; torch's float8_e4m3fn conversion and numpy's frexp for the scale)."""
    v = f32(b).astype(np.float64)
    K = v.shape[-1]
    blk = v.reshape(v.shape[:-1] + (K // 32, 32))
    amax = np.abs(blk).max(-1, keepdims=True)
    _, ex = np.frexp(amax)
    X = ex - 1 - 8
    q = torch.from_numpy(np.clip(blk * 2.0 ** -X, -448, 448).astype(np.float32)) \
        .to(torch.float8_e4m3fn).double().numpy()
    return (q * 2.0 ** X).reshape(v.shape)


def _deq_mx_rows(b):
    """Same, along axis 0 in blocks of 32 rows (zero rows pad the last block)."""
    n = b.shape[0]
    pad = (-n) % 32
    bb = np.concatenate([b, np.zeros((pad,) + b.shape[1:], b.dtype)]) if pad else b
    return _deq_mx(np.ascontiguousarray(bb.T)).T[:n]


def test_mxfp8_backward_matches_fp64_dequantised(orc):
    """MXFP8 DGRAD = FP64 matmuls of operands quantised along each GEMM's K
    (dY and W2^T along d; dA and W13^T along 2I), with the bf16 points."""
    inp = small(T=24, d=128, I=64, E=4, k=2, seed=17)
    fw = orc.quant_mxfp8(inp["w13"]) + orc.quant_mxfp8(inp["w2"])
    bw = orc.prepare_mxfp8_backward_weights(inp["w13"], inp["w2"])
    dx, ds, bi = orc.backward_mxfp8(inp["x"], inp["ids"], inp["scores"], fw, bw, inp["dy"],
                                    intermediates=True)
    xd, w13d = _deq_mx(inp["x"]), _deq_mx(inp["w13"])
    w2d = _deq_mx(inp["w2"])
    w2td = _deq_mx(np.ascontiguousarray(np.swapaxes(inp["w2"], 1, 2)))     # [E, I, d]
    w13td = _deq_mx(np.ascontiguousarray(np.swapaxes(inp["w13"], 1, 2)))   # [E, d, 2I]
    dyd = _deq_mx(inp["dy"])
    T, k = inp["ids"].shape
    I = 64
    ds_ref = np.zeros((T, k))
    dx_ref = np.zeros((T, 128))
    dA_all = []
    for t in range(T):
        for j in range(k):
            e, s = inp["ids"][t, j], float(inp["scores"][t, j])
            a = f32(bits(w13d[e] @ xd[t])).astype(np.float64)
            G, U = a[:I], a[I:]
            sig = 1 / (1 + np.exp(-G))
            h = f32(bits(G * sig * U)).astype(np.float64)
            g = w2td[e] @ dyd[t]
            ds_ref[t, j] = h @ g
            dsilu = sig * (1 + G * (1 - sig))
            dA = bits(np.concatenate([s * g * U * dsilu, s * g * G * sig]))
            dA_all.append(np.mean(dA == bi["dA"][t, j]))
            dxe = bits(w13td[e] @ _deq_mx(dA[None])[0])
            dx_ref[t] += f32(dxe)
    assert np.mean(dA_all) > 0.99
    assert _rel_fro(ds, ds_ref) < 2e-3
    assert _rel_fro(f32(dx), dx_ref) < 5e-3
    # the forward the backward sees is the MXFP8 forward (h via W2 quantised along I)
    assert w2d.shape == inp["w2"].shape


def test_mxfp8_wgrad_matches_fp64_dequantised(orc):
    """MXFP8 WGRAD of each expert = FP64 sums over its rows (dispatch order) of
    operands quantised along the rows in blocks of 32."""
    inp = small(T=90, d=128, I=64, E=3, k=2, seed=19)
    fw = orc.quant_mxfp8(inp["w13"]) + orc.quant_mxfp8(inp["w2"])
    bw = orc.prepare_mxfp8_backward_weights(inp["w13"], inp["w2"])
    _, _, bi = orc.backward_mxfp8(inp["x"], inp["ids"], inp["scores"], fw, bw, inp["dy"],
                                  intermediates=True)
    for e in range(3):
        d13, d2, rows = orc.wgrad_expert_mxfp8(inp["x"], inp["ids"], inp["scores"], fw, bw,
                                               inp["dy"], e)
        sel = [(t, j) for t in range(90) for j in range(2) if inp["ids"][t, j] == e]
        assert rows == len(sel) and rows > 32          # more than one row block
        dA = np.stack([bi["dA"][t, j] for t, j in sel])
        hs = np.stack([bi["hs"][t, j] for t, j in sel])
        dy = np.stack([inp["dy"][t] for t, _ in sel])
        x = np.stack([inp["x"][t] for t, _ in sel])
        r13 = _deq_mx_rows(dA).T @ _deq_mx_rows(x)
        r2 = _deq_mx_rows(dy).T @ _deq_mx_rows(hs)
        assert _rel_fro(d13, r13) < 1e-5 and _rel_fro(d2, r2) < 1e-5
        # quantising along the other axis gives measurably different sums
        assert _rel_fro(d13, (_deq_mx(dA).T @ _deq_mx(x))) > 1e-4


def test_mxfp8_forward_matches_fp64_dequantised(orc):
    """MXFP8 forward = FP64 matmuls of the dequantised operands (quantised with
    torch's float8 conversion and numpy's frexp), with the same bf16 points."""
    inp = small(T=24, d=128, I=64, E=4, k=2, seed=13)
    w13q, w13s = orc.quant_mxfp8(inp["w13"])
    w2q, w2s = orc.quant_mxfp8(inp["w2"])
    y, h = orc.forward_mxfp8(inp["x"], inp["ids"], inp["scores"], w13q, w13s, w2q, w2s,
                             return_h=True)

    def deq(b):
        v = f32(b).astype(np.float64)
        K = v.shape[-1]
        blk = v.reshape(v.shape[:-1] + (K // 32, 32))
        amax = np.abs(blk).max(-1, keepdims=True)
        _, ex = np.frexp(amax)
        X = ex - 1 - 8
        q = torch.from_numpy(np.clip(blk * 2.0 ** -X, -448, 448).astype(np.float32)) \
            .to(torch.float8_e4m3fn).double().numpy()
        return (q * 2.0 ** X).reshape(v.shape)

    xd, w13d, w2d = deq(inp["x"]), deq(inp["w13"]), deq(inp["w2"])
    T, k = inp["ids"].shape
    yref = np.zeros((T, 128))
    for t in range(T):
        for j in range(k):
            e = inp["ids"][t, j]
            a = f32(bits(w13d[e] @ xd[t]))
            G, U = a[:64].astype(np.float64), a[64:].astype(np.float64)
            hh = bits(G / (1 + np.exp(-G)) * U)
            assert np.mean(hh == h[t, j]) > 0.95
            o = w2d[e] @ deq(hh[None])[0]
            yref[t] += f32(bits(inp["scores"][t, j] * o))
    assert _rel_fro(f32(y), yref) < 5e-3


# ---------------------------------------------------------------------------
# NVFP4: E2M1 elements, E4M3 scales per 16 elements, per-tensor scale

# The E2M1 magnitudes in code order (1 sign, 2 exponent bits with bias 1, 1
# mantissa bit; exponent 0 subnormal), written from the format's definition.
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_brute(v):
    """Nearest E2M1 code by brute force over the eight magnitudes (ties to the
    even code, saturation to 6, sign kept)."""
    v = np.asarray(v, np.float64)
    m = np.minimum(np.abs(v), 6.0)
    dist = np.abs(m[..., None] - E2M1_MAG)                      # [..., 8]
    best = dist.min(-1, keepdims=True)
    cand = dist == best
    # among equally near codes prefer an even one (mantissa bit 0)
    even = cand & (np.arange(8) % 2 == 0)
    code = np.where(even.any(-1), even.argmax(-1), cand.argmax(-1))
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def test_e2m1_codes_roundtrip_ties_and_brute_force(orc):
    codes = np.arange(16, dtype=np.uint8)
    vals = orc.e2m1_decode(codes)
    assert np.array_equal(np.abs(vals[:8]), E2M1_MAG) and np.array_equal(vals[8:], -E2M1_MAG)
    assert np.array_equal(orc.e2m1_encode(vals), codes)           # every code round-trips
    # midpoints between neighbours go to the even code
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert orc.e2m1_encode(mids).tolist() == [0, 2, 2, 4, 4, 6, 6]
    assert orc.e2m1_encode(-mids).tolist() == [8, 10, 10, 12, 12, 14, 14]
    # saturation and signed zero
    assert orc.e2m1_encode(np.array([6.0, 7.0, 1e30, -9.0, -0.0, -0.2])).tolist() == \
        [7, 7, 7, 15, 8, 8]
    grid = np.linspace(-8, 8, 64001)
    assert np.array_equal(orc.e2m1_encode(grid), _e2m1_brute(grid))


def _nv_quant_ref(v_bits, g):
    """NVFP4 block quantisation restated in numpy/torch: fp32 arithmetic, torch's
    float8_e4m3fn conversion (after explicit saturation) for the block scale,
    brute-force E2M1 for the elements.  Returns (codes unpacked [..., K], scales)."""
    v = f32(v_bits)
    K = v.shape[-1]
    blk = v.reshape(v.shape[:-1] + (K // 16, 16))
    amax = np.abs(blk).max(-1)
    t = (amax / np.float32(6.0)).astype(np.float32) * np.float32(g)
    t = np.minimum(t.astype(np.float32), np.float32(448.0))
    sf = torch.from_numpy(np.ascontiguousarray(t)).to(torch.float8_e4m3fn)
    S = sf.float().numpy()
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (np.float32(g) / S).astype(np.float32)
        q = _e2m1_brute((blk * r[..., None]).astype(np.float32))
    q = np.where((S == 0)[..., None], 0, q).astype(np.uint8)
    return q.reshape(v.shape), sf.view(torch.uint8).numpy()


def _unpack(p):
    return np.stack([p & 15, p >> 4], -1).reshape(p.shape[:-1] + (2 * p.shape[-1],))


@pytest.mark.parametrize("g", [1.0, 64.0, 1.0 / 3.0, 2688.0 / 5.5])
def test_nvfp4_block_quantiser_matches_restatement(orc, g):
    rng = np.random.default_rng(int(g * 1000) % 97)
    v = rng.standard_normal((40, 128)).astype(np.float32) * \
        np.exp2(rng.integers(-12, 8, (40, 1))).astype(np.float32)
    v[0] = 0.0                                   # all-zero blocks
    v[1, :16] = 1e-30                            # a scale that rounds to zero
    v[2, 16:32] = -v[2, 16:32]
    vb = bits(v)
    codes, scales = orc.quant_nvfp4(vb, g)
    q, sf = _nv_quant_ref(vb, g)
    assert np.array_equal(scales, sf)
    assert np.array_equal(_unpack(codes), q)
    assert np.all(scales[0] == 0) and np.all(codes[0] == 0)


def test_nvfp4_prepared_weights_per_expert_scale(orc):
    inp = small(T=8, d=64, I=32, E=3, k=2, seed=17)
    w = inp["w13"].copy()
    w[1] = 0                                     # an all-zero expert: scale 1
    codes, scales, sc = orc.prepare_nvfp4(w)
    amax = np.abs(f32(w)).reshape(3, -1).max(1)
    want = np.where(amax > 0, (amax / np.float32(2688.0)).astype(np.float32), np.float32(1.0))
    assert np.array_equal(sc, want.astype(np.float32))
    for e in range(3):
        q, sf = _nv_quant_ref(w[e], np.float32(1.0) / sc[e])
        assert np.array_equal(scales[e], sf) and np.array_equal(_unpack(codes[e]), q)
    # the largest block of each non-empty expert uses the top of the E4M3 range
    assert scales[0].max() == 0x7E and scales[2].max() == 0x7E


def _grid_values(rng, shape):
    """E2M1 grid values with +-6 in every 16-element block (so the block amax is 6)."""
    v = rng.choice(np.concatenate([E2M1_MAG, -E2M1_MAG[1:]]), size=shape)
    v[..., ::16] = np.where(rng.random(v[..., ::16].shape) < 0.5, 6.0, -6.0)
    return v.astype(np.float32)


def test_nvfp4_forward_reduces_to_bf16_on_grid_values(orc):
    """Inputs exactly representable with block scale 64 and per-tensor scale
    1/64: the NVFP4 pre-activations a equal the bf16 forward's bit for bit (the
    sums differ only by the exact factor 64 * 64 * 2^-12)."""
    rng = np.random.default_rng(3)
    T, d, I, E, k = 12, 64, 32, 3, 2
    inp = small(T=T, d=d, I=I, E=E, k=k, seed=19)
    x = _grid_values(rng, (T, d))
    w13 = _grid_values(rng, (E, 2 * I, d))
    w2 = _grid_values(rng, (E, d, I))
    xb, w13b, w2b = bits(x), bits(w13), bits(w2)
    pack = lambda q: (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    sf64 = 0x68                                  # E4M3 code of 64 = 2^6
    w13p = (pack(orc.e2m1_encode(w13)), np.full((E, 2 * I, d // 16), sf64, np.uint8),
            np.full(E, 1 / 64, np.float32))
    w2p = (pack(orc.e2m1_encode(w2)), np.full((E, d, I // 16), sf64, np.uint8),
           np.full(E, 1 / 64, np.float32))
    assert orc.e4m3_decode(np.array([sf64], np.uint8))[0] == 64.0
    _, it = orc.forward_nvfp4(xb, inp["ids"], inp["scores"], w13p, w2p, 1 / 64, 1 / 64,
                              intermediates=True)
    _, ib = orc.forward(xb, inp["ids"], inp["scores"], w13b, w2b, intermediates=True)
    assert np.array_equal(it["a"], ib["a"])
    assert np.array_equal(it["h"], ib["h"])


def test_nvfp4_forward_matches_fp64_dequantised(orc):
    """NVFP4 forward = FP64 matmuls of the dequantised operands (quantised by the
    numpy/torch restatement), with the same alpha and bf16 points."""
    T, d, I, E, k = 16, 128, 64, 4, 2
    inp = small(T=T, d=d, I=I, E=E, k=k, seed=23)
    w13p = orc.prepare_nvfp4(inp["w13"])
    w2p = orc.prepare_nvfp4(inp["w2"])
    xs = np.float32(np.abs(f32(inp["x"])).max() / 2688.0)
    hs = np.float32(0.05)
    y, it = orc.forward_nvfp4(inp["x"], inp["ids"], inp["scores"], w13p, w2p, xs, hs,
                              intermediates=True)

    def deq(b, g):
        q, sf = _nv_quant_ref(b, g)
        S = torch.from_numpy(sf).view(torch.float8_e4m3fn).double().numpy()
        val = np.where(q >= 8, -1.0, 1.0) * E2M1_MAG[q & 7]
        return val * np.repeat(S, 16, axis=-1)

    xd = deq(inp["x"], np.float32(1) / xs)
    yref = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            e = inp["ids"][t, j]
            w13d = deq(inp["w13"][e], np.float32(1) / w13p[2][e])
            w2d = deq(inp["w2"][e], np.float32(1) / w2p[2][e])
            a = bits(float(xs * w13p[2][e]) * (w13d @ xd[t]))
            assert np.mean(a == it["a"][t, j]) > 0.97
            G, U = f32(a[:I]).astype(np.float64), f32(a[I:]).astype(np.float64)
            hh = bits(G / (1 + np.exp(-G)) * U)
            assert np.mean(hh == it["h"][t, j]) > 0.95
            o = float(hs * w2p[2][e]) * (w2d @ deq(hh[None], np.float32(1) / hs)[0])
            yref[t] += f32(bits(inp["scores"][t, j] * o))
    assert _rel_fro(f32(y), yref) < 5e-3
    # a wrong nibble order would not pass
    swapped = (w13p[0] >> 4) | ((w13p[0] & 15) << 4)
    y2 = orc.forward_nvfp4(inp["x"], inp["ids"], inp["scores"], (swapped,) + w13p[1:], w2p, xs, hs)
    assert _rel_fro(f32(y2), yref) > 0.1
