"""moe_dispatch_static: the allocation-free dispatch entry point.

Callers that cannot allocate device memory (code inside another framework's
allocator or memory-pool callbacks, hosts with device memory already carved
into fixed pools) route tokens through moe_dispatch_static, whose scratch is a
static device array inside the library.  Here it is called through the C ABI
twice in a row, on different routings, and each result must equal, bit for bit,
the dispatch tables that moe_forward builds in its own workspace for the same
inputs.  This file is collected last so a failure here never hides the others.
"""

import ctypes

import numpy as np
import pytest
import torch

from gpu_case import make, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    L = m.lib()
    vp = ctypes.c_void_p
    L.moe_dispatch_static.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      vp, vp, vp, vp, vp, ctypes.c_longlong, vp, vp]
    L.moe_dispatch_static.restype = ctypes.c_int
    return m


def _static_dispatch(moe, dev, T, k, E):
    L = moe.lib()
    BM = L.moe_tile_rows()
    cap = (T * k + E * (BM - 1)) // BM * BM
    out = dict(
        m_indptr=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
        off_pad=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
        row_of=torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
        token_of=torch.full((cap,), -7, dtype=torch.int32, device="cuda"),
        score_of=torch.full((cap,), -7.0, dtype=torch.float32, device="cuda"),
        status=torch.full((2,), -7, dtype=torch.int32, device="cuda"),
    )
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = L.moe_dispatch_static(p(dev["ids"]), p(dev["scores"]), T, k, E, p(out["m_indptr"]),
                               p(out["off_pad"]), p(out["row_of"]), p(out["token_of"]),
                               p(out["score_of"]), cap, p(out["status"]),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, moe.lib().moe_status_string(rc)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


def test_static_dispatch_allocates_nothing(moe):
    # after the first call (the set-up), a call leaves the device's free memory
    # unchanged: it allocates nothing (device allocations are 2 MB granular)
    inp = make(None, seed=15, train=False, T=4096, d=128, I=64, E=64, k=8)
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in inp.items()
           if k in ("ids", "scores")}
    _static_dispatch(moe, dev, 4096, 8, 64)              # set-up (and outputs allocated)
    L = moe.lib()
    BM = L.moe_tile_rows()
    cap = (4096 * 8 + 64 * (BM - 1)) // BM * BM
    outs = [torch.empty(n, dtype=dt, device="cuda") for n, dt in
            ((65, torch.int32), (65, torch.int32), (4096 * 8, torch.int32), (cap, torch.int32),
             (cap, torch.float32), (2, torch.int32))]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for _ in range(3):
        rc = L.moe_dispatch_static(p(dev["ids"]), p(dev["scores"]), 4096, 8, 64, *map(p, outs[:5]),
                                   cap, p(outs[5]),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert outs[5].tolist() == [0, -1]


@pytest.mark.parametrize("sizes", [
    dict(T=300, d=128, I=64, E=7, k=3),
    dict(T=2048, d=128, I=64, E=128, k=8, routing="zipf", zipf_s=1.2, zipf_support=102),
    # at the static scratch's capacity: T*k = MOE_STATIC_MAX_ROUTED, E = 256
    dict(T=32768, d=128, I=64, E=256, k=8),
], ids=["ragged", "skew_e128", "at_capacity"])
def test_static_dispatch_matches_plan_dispatch(moe, sizes):
    cases = [make(None, seed=s, train=False, **sizes) for s in (11, 12)]
    for inp in cases:                     # two calls in a row, different routings
        g = run_gpu(moe, inp, train=False)
        assert g["rc"] == 0
        plan = g["plan"]
        c = inp["cfg"]
        T, k, E = c["T"], c["k"], c["E"]
        got = _static_dispatch(moe, g["dev"], T, k, E)
        mi = plan.buffer("m_indptr", torch.int32).cpu().numpy()
        op = plan.buffer("off_pad", torch.int32).cpu().numpy()
        ro = plan.buffer("row_of", torch.int32).cpu().numpy()[: T * k]
        n = int(op[-1])
        tok = plan.buffer("token_of", torch.int32).cpu().numpy()[:n]
        sco = plan.buffer("score_of", torch.float32).cpu().numpy()[:n]
        assert np.array_equal(got["m_indptr"], mi)
        assert np.array_equal(got["off_pad"], op)
        assert np.array_equal(got["row_of"], ro)
        assert np.array_equal(got["token_of"][:n], tok)
        assert np.array_equal(got["score_of"][:n].view(np.int32), sco.view(np.int32))
        assert got["status"].tolist() == [0, -1]


def test_static_dispatch_reports_bad_ids_and_clears(moe):
    inp = make(None, seed=13, train=False, T=100, d=128, I=64, E=8, k=3)
    ids = inp["ids"].copy()
    ids[40, 2] = ids[40, 0]              # flat index 122 repeats an id of its row
    inp["ids"] = ids
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in inp.items()
           if k in ("ids", "scores")}
    got = _static_dispatch(moe, dev, 100, 3, 8)
    assert got["status"].tolist() == [moe.MOE_ERR_BAD_IDS, 122]
    # the repeated id is dropped; the tables stay consistent without it
    assert got["row_of"][122] == -1
    assert got["m_indptr"][-1] == 100 * 3 - 1
    assert np.all(got["row_of"][np.arange(300) != 122] >= 0)
    dev["ids"] = torch.from_numpy(make(None, seed=14, train=False, T=100, d=128, I=64, E=8,
                                       k=3)["ids"]).cuda()
    got = _static_dispatch(moe, dev, 100, 3, 8)
    assert got["status"].tolist() == [0, -1]


def test_static_dispatch_rejects_oversize(moe):
    L = moe.lib()
    big = 262144 // 8 + 1
    fake = ctypes.c_void_p(1 << 20)
    rc = L.moe_dispatch_static(fake, fake, big, 8, 128, fake, fake, fake, fake, fake,
                               1 << 30, fake, None)
    assert rc == moe.MOE_ERR_WORKSPACE
    rc = L.moe_dispatch_static(fake, fake, 100, 3, 8, fake, fake, fake, fake, fake, 10, fake,
                               None)
    assert rc == moe.MOE_ERR_INVALID_ARG
