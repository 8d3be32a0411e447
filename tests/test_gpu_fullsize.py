"""Parity at the full workload sizes, in the launch configuration the benchmark
times (one plan, forward with saved activations, backward).  The oracle
evaluates whole token sets (every token of the training workload, at least 1024
tokens of the others) and the weight gradients of the experts that exercise the
longest and the shortest K loops: the four heaviest experts (for the skewed
workload, 7.7K to 15.7K routed rows each), the lightest, the median one and an
expert without rows.  Dispatch tables are compared in full, bit-exact;
properties that hold at any size (finite outputs, zero output for zero-score
padding, untouched gradients of experts without rows) are checked on every
element.
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
    if n >= T:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    toks = set(int(t) for t in rng.choice(T, n, replace=False)) | set(must)
    return np.array(sorted(toks), np.int32)


def _sample_experts(ids, E, n_heavy=4, include_empty=True):
    """The n_heavy heaviest experts (longest WGRAD K loops), the lightest and the
    median non-empty expert, and one expert without rows if there is one."""
    counts = np.bincount(ids.reshape(-1)[ids.reshape(-1) >= 0], minlength=E)
    order = np.argsort(counts, kind="stable")
    nz = [int(e) for e in order if counts[e] > 0]
    pick = nz[-n_heavy:] + nz[:1] + [nz[len(nz) // 2]]
    if include_empty:
        pick += [int(e) for e in order if counts[e] == 0][:1]
    return sorted(set(pick)), counts


def test_infer_e16_forward(moe, orc):
    inp = make("infer_e16", train=False)
    g = run_gpu(moe, inp, train=False)
    assert g["rc"] == 0
    check_dispatch(orc, inp, g)
    y = f32(bits(g["y"]))
    assert np.all(np.isfinite(y))
    toks = _sample_tokens(inp["cfg"]["T"], 1024, 1, must=(0, inp["cfg"]["T"] - 1))
    check_forward(orc, inp, g, toks=toks)


@pytest.mark.parametrize("pairs", [False, True], ids=["one_cta", "cta_pairs"])
def test_train_e128_forward_backward(moe, orc, pairs):
    inp = make("train_e128", train=True, cta_pairs=pairs)
    c = inp["cfg"]
    g = run_gpu(moe, inp, train=True)
    assert g["rc"] == 0
    check_dispatch(orc, inp, g)
    assert np.all(np.isfinite(f32(bits(g["y"])))) and np.all(np.isfinite(f32(bits(g["dx"]))))
    # one-CTA kernels (the benchmark's configuration): every token; CTA pairs: 1024
    toks = _sample_tokens(c["T"], c["T"] if not pairs else 1024, 2, must=(0, c["T"] - 1))
    check_forward(orc, inp, g, toks=toks)
    experts, counts = _sample_experts(inp["ids"], c["E"], include_empty=False)
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
    toks = _sample_tokens(c["T"] - pad, 1024, 3, must=(0,))
    toks = np.concatenate([toks, [c["T"] - pad, c["T"] - 1]]).astype(np.int32)
    check_forward(orc, inp, g, toks=toks)
    experts, counts = _sample_experts(inp["ids"], c["E"], include_empty=True)
    # the heaviest expert's K loop runs over more than 15K routed rows
    assert counts[experts].max() > 15000
    check_backward(orc, inp, g, toks=toks, experts=experts)
    # every expert without rows keeps its gradient bit-for-bit
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
    toks = _sample_tokens(c["T"], 1024, 4, must=(0, c["T"] - 1))
    check_forward(orc, inp, g, toks=toks)
    experts, _ = _sample_experts(inp["ids"], c["E"], include_empty=False)
    check_backward(orc, inp, g, toks=toks, experts=experts)
