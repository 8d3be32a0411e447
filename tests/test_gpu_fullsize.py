"""Parity at the full workload sizes, in the launch configuration the benchmark
times (one plan, forward with saved activations, backward).  The oracle
evaluates sampled tokens one by one and the weight gradients of sampled
experts; dispatch tables are compared in full, bit-exact; properties that hold
at any size (finite outputs, zero output for zero-score padding, untouched
gradients of experts without rows) are checked on every element.
"""

import numpy as np
import pytest
import torch

from gpu_case import bits, check_backward, check_dispatch, check_forward, make, run_gpu
from parity import f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


def _sample_tokens(T, n, seed, must=()):
    rng = np.random.default_rng(seed)
    toks = set(int(t) for t in rng.choice(T, n, replace=False)) | set(must)
    return np.array(sorted(toks), np.int32)


def _sample_experts(ids, E, n_light=1, n_mid=1, include_empty=True):
    counts = np.bincount(ids.reshape(-1), minlength=E)
    order = np.argsort(counts, kind="stable")
    nz = [e for e in order if counts[e] > 0]
    pick = list(nz[:n_light]) + list(nz[len(nz) // 2:len(nz) // 2 + n_mid])
    if include_empty:
        pick += [int(e) for e in order if counts[e] == 0][:1]
    return pick


def test_infer_e16_forward(moe, orc):
    inp = make("infer_e16", train=False)
    g = run_gpu(moe, inp, train=False)
    assert g["rc"] == 0
    check_dispatch(orc, inp, g)
    y = f32(bits(g["y"]))
    assert np.all(np.isfinite(y))
    toks = _sample_tokens(inp["cfg"]["T"], 24, 1, must=(0, inp["cfg"]["T"] - 1))
    check_forward(orc, inp, g, toks=toks)


@pytest.mark.parametrize("pairs", [False, True], ids=["one_cta", "cta_pairs"])
def test_train_e128_forward_backward(moe, orc, pairs):
    inp = make("train_e128", train=True, cta_pairs=pairs)
    g = run_gpu(moe, inp, train=True)
    assert g["rc"] == 0
    check_dispatch(orc, inp, g)
    assert np.all(np.isfinite(f32(bits(g["y"])))) and np.all(np.isfinite(f32(bits(g["dx"]))))
    toks = _sample_tokens(inp["cfg"]["T"], 16, 2, must=(0, inp["cfg"]["T"] - 1))
    check_forward(orc, inp, g, toks=toks)
    experts = _sample_experts(inp["ids"], inp["cfg"]["E"], include_empty=False)
    check_backward(orc, inp, g, toks=toks, experts=experts)


def test_skew_pad_forward_backward(moe, orc):
    inp = make("skew_pad", train=True)
    c = inp["cfg"]
    g = run_gpu(moe, inp, train=True)
    assert g["rc"] == 0
    check_dispatch(orc, inp, g)
    y = f32(bits(g["y"]))
    dx = f32(bits(g["dx"]))
    pad = c["pad"]
    assert np.all(y[-pad:] == 0) and np.all(dx[-pad:] == 0)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(dx))
    toks = _sample_tokens(c["T"] - pad, 12, 3, must=(0,))
    toks = np.concatenate([toks, [c["T"] - pad, c["T"] - 1]]).astype(np.int32)
    check_forward(orc, inp, g, toks=toks)
    experts = _sample_experts(inp["ids"], c["E"], include_empty=True)
    check_backward(orc, inp, g, toks=toks, experts=experts)
    # every expert without rows keeps its gradient bit-for-bit
    counts = np.bincount(inp["ids"].reshape(-1), minlength=c["E"])
    empty = torch.from_numpy(np.flatnonzero(counts == 0)).cuda()
    assert torch.equal(g["dw13"][empty], g["dev"]["dw13"][empty])
    assert torch.equal(g["dw2"][empty], g["dev"]["dw2"][empty])


def test_train_e256_forward_backward(moe, orc):
    """The plan's largest expert count (E = 256, k = 8) at the full d and I: about
    256 routed rows per expert, so most experts end in a part-filled m tile."""
    inp = make(None, seed=31, train=True, T=8192, d=2048, I=768, E=256, k=8)
    c = inp["cfg"]
    g = run_gpu(moe, inp, train=True)
    assert g["rc"] == 0
    check_dispatch(orc, inp, g)
    assert np.all(np.isfinite(f32(bits(g["y"])))) and np.all(np.isfinite(f32(bits(g["dx"]))))
    toks = _sample_tokens(c["T"], 12, 4, must=(0, c["T"] - 1))
    check_forward(orc, inp, g, toks=toks)
    experts = _sample_experts(inp["ids"], c["E"], include_empty=False)
    check_backward(orc, inp, g, toks=toks, experts=experts)
