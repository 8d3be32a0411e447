"""Seeded synthetic inputs for the routed-expert hot path.

This module only draws random inputs; it holds none of the method's arithmetic.
Both the CUDA path (tests, benchmark) and the CPU oracle (tests) take their
inputs from here, so the two always see bit-identical tensors.

Recipe (one generator for every workload):
  x       ~ N(0, 1)               rounded to bf16
  W13     ~ N(0, 1/d)             [E, 2I, d] bf16  (rows [0,I) gate, [I,2I) up)
  W2      ~ N(0, 1/I)             [E, d, I]  bf16
  ids     uniform: per token the first k entries of an argsort of E uniforms
          (column order as drawn); zipf: k distinct draws without replacement
          from Zipf(s) over the first `zipf_support` ranks, ranks mapped to
          expert ids through a seeded permutation (Gumbel top-k sampling)
  scores  softmax over the k chosen of N(0, 1) logits, float32; padding tokens
          (the last `pad` rows) get zero scores but keep valid ids
  dY      ~ N(0, 1)               bf16
  dW init ~ N(0, 1e-3^2)          float32 (existing gradient contents)

Normals come from numpy's Philox generator keyed by (seed, tensor tag, chunk),
so the values do not depend on thread count.  bf16 rounding of the drawn
floats uses torch's standard conversion.
"""

from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

# Workloads (sizes and structure of the configurations the method is measured on).
CONFIGS = {
    # tiny correctness case: T=64, d=128, I=64, E=4, k=2, plain SwiGLU, forward
    "tiny_fwd": dict(T=64, d=128, I=64, E=4, k=2, routing="uniform", clamp=0.0, pad=0,
                     precision="bf16", train=False),
    # BF16 inference forward, E=16
    "infer_e16": dict(T=8192, d=2048, I=768, E=16, k=8, routing="uniform", clamp=0.0, pad=0,
                      precision="bf16", train=False),
    # BF16 training forward+backward, E=128
    "train_e128": dict(T=8192, d=2048, I=768, E=128, k=8, routing="uniform", clamp=0.0, pad=0,
                       precision="bf16", train=True),
    # skewed Zipf(1.2) routing, last 2048 of 16384 tokens are zero-score padding,
    # clamped SwiGLU (limit 7), forward+backward
    "skew_pad": dict(T=16384, d=2048, I=768, E=128, k=8, routing="zipf", zipf_s=1.2,
                     zipf_support=102, clamp=7.0, pad=2048, precision="bf16", train=True),
    # MXFP8 E4M3 block-scaled forward, E=128
    "mxfp8_e128": dict(T=8192, d=2048, I=768, E=128, k=8, routing="uniform", clamp=0.0, pad=0,
                       precision="mxfp8", train=False),
}

_TAGS = {"x": 1, "w13": 2, "w2": 3, "ids": 4, "logits": 5, "dy": 6, "dw13": 7, "dw2": 8,
         "perm": 9}
_CHUNK = 1 << 22


def _rng(seed, tag, chunk=0):
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tag, chunk])))


def normal_f32(shape, std, seed, tag):
    """float32 normals N(0, std^2) of the given shape (chunked, thread-parallel)."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        _rng(seed, _TAGS[tag], c).standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    workers = min(nchunks, os.cpu_count() or 1)
    if workers > 1:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    else:
        for c in range(nchunks):
            fill(c)
    return out.reshape(shape)


def to_bf16_bits(f):
    """Round float32 to bf16 with torch's standard conversion; return raw uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(f, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def draw_ids(T, k, E, seed, routing="uniform", zipf_s=1.2, zipf_support=None):
    """int32 [T, k] expert ids, distinct within each row."""
    g = _rng(seed, _TAGS["ids"])
    if routing == "uniform":
        u = g.random((T, E))
        return np.argsort(u, axis=1, kind="stable")[:, :k].astype(np.int32)
    if routing == "zipf":
        R = zipf_support or E
        assert k <= R <= E
        logw = -zipf_s * np.log(np.arange(1, R + 1, dtype=np.float64))
        gumbel = -np.log(-np.log(g.random((T, R))))
        keys = logw[None, :] + gumbel
        ranks = np.argsort(-keys, axis=1, kind="stable")[:, :k]      # draw order
        perm = _rng(seed, _TAGS["perm"]).permutation(E)
        return perm[ranks].astype(np.int32)
    raise ValueError(routing)


def draw_scores(T, k, seed, pad=0):
    """float32 [T, k]: softmax over k N(0,1) logits; the last `pad` rows are zero."""
    z = _rng(seed, _TAGS["logits"]).standard_normal((T, k))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    s = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    if pad:
        s[T - pad:] = 0.0
    return s


def make_inputs(name=None, seed=0, need=("x", "ids", "scores", "w13", "w2"), **over):
    """Inputs of a named workload (or of explicit sizes given as keywords).

    Returns a dict with numpy arrays (bf16 tensors as uint16 bit patterns) and
    the workload description under "cfg".
    """
    cfg = dict(CONFIGS[name]) if name else dict(routing="uniform", clamp=0.0, pad=0,
                                                 precision="bf16", train=False)
    cfg.update(over)
    T, d, I, E, k = cfg["T"], cfg["d"], cfg["I"], cfg["E"], cfg["k"]
    out = {"cfg": cfg}
    if "x" in need:
        out["x"] = to_bf16_bits(normal_f32((T, d), 1.0, seed, "x"))
    if "w13" in need:
        out["w13"] = to_bf16_bits(normal_f32((E, 2 * I, d), d ** -0.5, seed, "w13"))
    if "w2" in need:
        out["w2"] = to_bf16_bits(normal_f32((E, d, I), I ** -0.5, seed, "w2"))
    if "ids" in need:
        out["ids"] = draw_ids(T, k, E, seed, cfg.get("routing", "uniform"),
                              cfg.get("zipf_s", 1.2), cfg.get("zipf_support"))
    if "scores" in need:
        out["scores"] = draw_scores(T, k, seed, cfg.get("pad", 0))
    if "dy" in need:
        out["dy"] = to_bf16_bits(normal_f32((T, d), 1.0, seed, "dy"))
    if "dw13" in need:
        out["dw13"] = normal_f32((E, 2 * I, d), 1e-3, seed, "dw13")
    if "dw2" in need:
        out["dw2"] = normal_f32((E, d, I), 1e-3, seed, "dw2")
    return out
