"""The C-ABI library builds, loads and exports every entry point of include/moe.h,
and its host-side argument checks behave (CPU only: no compute call)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    from routed_mixture_experts_gb300 import build as b

    b.build()
    from routed_mixture_experts_gb300 import binding

    return binding.lib()


def test_header_declares_the_path(L):
    names = _declared_functions()
    for must in ("moe_plan_create", "moe_forward", "moe_backward", "moe_plan_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_plan_create_validates_shapes(L):
    ok = L.moe_plan_create(64, 128, 64, 4, 2, 0)
    assert ok
    L.moe_plan_destroy(ok)
    for bad in [(0, 128, 64, 4, 2, 0), (64, 96, 64, 4, 2, 0), (64, 128, 48, 4, 2, 0),
                (64, 128, 64, 4, 5, 0), (64, 128, 64, 300, 2, 0), (64, 128, 64, 4, 0, 0),
                (64, 128, 64, 4, 2, 9), (1 << 28, 128, 64, 256, 16, 0)]:
        assert not L.moe_plan_create(*bad), bad


def test_workspace_bytes_cover_worst_case_padding(L):
    p = L.moe_plan_create(8192, 2048, 768, 128, 8, 0)
    try:
        inf = L.moe_plan_workspace_bytes(p, 0)
        tr = L.moe_plan_workspace_bytes(p, 1)
        st = L.moe_plan_workspace_bytes(p, 3)
        assert 0 < inf < tr < st
        R, E, BM = 8192 * 8, 128, L.moe_tile_rows()
        RP = (R + E * (BM - 1)) // BM * BM
        # at least x_e, h, ys for the forward; a, dY_e, dA, hs, dX_e in training
        assert inf >= 2 * RP * (2048 + 768 + 2048)
        assert tr >= inf + 2 * RP * (2 * 768 + 2048 + 2 * 768 + 768 + 2048)
    finally:
        L.moe_plan_destroy(p)


def test_entry_points_reject_bad_arguments_on_host(L):
    vp = ctypes.c_void_p
    assert L.moe_forward(None, *([None] * 8), 0, None) == 1
    assert L.moe_backward(None, *([None] * 8)) == 1
    assert L.moe_plan_set_swiglu_clamp(None, 7.0) == 1
    p = L.moe_plan_create(64, 128, 64, 4, 2, 0)
    try:
        assert L.moe_plan_set_swiglu_clamp(p, -1.0) == 1
        assert L.moe_plan_set_swiglu_clamp(p, 7.0) == 0
        # no workspace yet
        fake = vp(1 << 20)
        assert L.moe_forward(p, fake, fake, fake, fake, fake, None, None, fake, 0, None) == 2
        assert L.moe_backward(p, fake, fake, fake, fake, fake, fake, fake, None) == 2
        # misaligned activation pointer
        assert L.moe_forward(p, vp((1 << 20) + 2), fake, fake, fake, fake, None, None, fake, 0,
                             None) == 1
        assert L.moe_plan_set_workspace(p, vp((1 << 20) + 16), 1 << 30, 0) == 1   # misaligned
        assert L.moe_plan_set_workspace(p, fake, 16, 0) == 2                      # too small
    finally:
        L.moe_plan_destroy(p)
    assert L.moe_quantize_mxfp8(vp(1 << 20), 4, 48, vp(1 << 20), vp(1 << 20), None) == 1
    assert L.moe_gemm_bf16(0, vp(1 << 20), vp(1 << 20), vp(1 << 20), 100, 64, 64, vp(1 << 20),
                           None) == 1


def test_status_strings(L):
    for code, name in [(0, b"MOE_OK"), (4, b"MOE_ERR_BAD_IDS"), (5, b"MOE_ERR_TIMEOUT")]:
        assert L.moe_status_string(code) == name


def test_cta_pairs_option_sizes_the_workspace(L):
    p = L.moe_plan_create(8192, 2048, 768, 128, 8, 0)
    q = L.moe_plan_create(64, 128, 64, 4, 2, 0)
    m = L.moe_plan_create(8192, 2048, 768, 128, 8, 1)
    try:
        assert L.moe_plan_row_granule(p) == 128
        one = L.moe_plan_workspace_bytes(p, 1)
        assert L.moe_plan_set_cta_pairs(p, 1) == 0
        assert L.moe_plan_row_granule(p) == 128                # segments stay 128-row
        assert one < L.moe_plan_workspace_bytes(p, 1) < one + 65536   # + the pair tile lists
        assert L.moe_plan_set_cta_pairs(p, 0) == 0
        assert L.moe_plan_workspace_bytes(p, 1) == one
        assert L.moe_plan_set_cta_pairs(q, 1) == 7             # d, I not multiples of 256
        assert L.moe_plan_set_cta_pairs(m, 1) == 7             # MXFP8 plans: one-CTA only
    finally:
        for x in (p, q, m):
            L.moe_plan_destroy(x)


def test_mxfp8_training_workspace_keeps_dA_and_hs_only_as_codes(L):
    """An MXFP8 training plan adds the saved a, dX_e, the score-gradient partials
    and the E4M3 operands of the backward (dY and dA along K, dY, dA, hs and x
    along the rows, each with 1/32 of scale bytes), but no bf16 dA or hs
    (6*Rpad*I bytes)."""
    T, d, I, E, k = 8192, 2048, 768, 128, 8
    p = L.moe_plan_create(T, d, I, E, k, 1)
    assert p
    try:
        extra = L.moe_plan_workspace_bytes(p, 1) - L.moe_plan_workspace_bytes(p, 0)
        R, BM = T * k, L.moe_tile_rows()
        RP = (R + E * (BM - 1)) // BM * BM
        codes = RP * (d + 2 * I) + RP * (d + 2 * I + I + d)
        expected = 2 * RP * 2 * I + 2 * RP * d + 4 * RP * 2 * (I // 128) + codes * 33 // 32
        assert expected - (1 << 20) <= extra <= expected + (1 << 20)
        assert extra < expected + 6 * RP * I - (1 << 20)
    finally:
        L.moe_plan_destroy(p)
