"""ctypes binding of include/moe.h (argument marshalling only)."""

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_WORKSPACE = 2
MOE_ERR_STATE = 3
MOE_ERR_BAD_IDS = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_CUDA = 6
MOE_ERR_UNSUPPORTED = 7
MOE_PREC_BF16 = 0
MOE_PREC_MXFP8 = 1
MOE_PREC_NVFP4 = 2
MOE_WS_TRAINING = 1
MOE_WS_HOST_STAGING = 2
MOE_BUF = dict(m_indptr=0, off_pad=1, row_of=2, token_of=3, score_of=4, xe=5, a=6, h=7, ys=8,
               dye=9, dA=10, hs=11, dxe=12, xq=13, xsf=14, hq=15, hsf=16, xqT=17, xqTsf=18,
               dAq=19, dAsf=20, dAqT=21, dAqTsf=22, hsqT=23, hsqTsf=24)

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        name = _lib.moe_status_string(code).decode() if _lib is not None else str(code)
        super().__init__("%s%s" % (name, (": " + what) if what else ""))


def _declare(L):
    vp, i32, f32, sz, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_long
    L.moe_plan_create.argtypes = [i32] * 6
    L.moe_plan_create.restype = vp
    L.moe_plan_destroy.argtypes = [vp]
    L.moe_plan_destroy.restype = None
    L.moe_plan_set_swiglu_clamp.argtypes = [vp, f32]
    L.moe_plan_workspace_bytes.argtypes = [vp, i32]
    L.moe_plan_workspace_bytes.restype = sz
    L.moe_plan_set_workspace.argtypes = [vp, vp, sz, i32]
    L.moe_forward.argtypes = [vp] * 9 + [i32, vp]
    L.moe_backward.argtypes = [vp] * 9
    L.moe_forward_routed.argtypes = [vp, vp, ctypes.c_longlong] + [vp] * 9
    L.moe_step_host.argtypes = [vp] * 13
    L.moe_quantize_mxfp8.argtypes = [vp, i64, i32, vp, vp, vp]
    L.moe_plan_check.argtypes = [vp, ctypes.POINTER(ctypes.c_longlong)]
    L.moe_status_string.argtypes = [i32]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_plan_buffer.argtypes = [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(sz)]
    L.moe_tile_rows.restype = i32
    L.moe_plan_set_cta_pairs.argtypes = [vp, i32]
    L.moe_plan_row_granule.argtypes = [vp]
    L.moe_plan_row_granule.restype = i32
    L.moe_gemm_scratch_bytes.argtypes = [i32, i32]
    L.moe_gemm_scratch_bytes.restype = sz
    L.moe_gemm_bf16.argtypes = [i32, vp, vp, vp, i32, i32, i32, vp, vp]
    L.moe_plan_set_timing_events.argtypes = [vp, i32, ctypes.POINTER(vp), i32]
    L.moe_plan_set_debug.argtypes = [vp, ctypes.c_longlong, i32]
    L.moe_mxfp8_weight_scale_bytes.argtypes = [i32, i32, i32, i32]
    L.moe_mxfp8_weight_scale_bytes.restype = sz
    L.moe_prepare_weights_mxfp8.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
    L.moe_prepare_weights_mxfp8_backward.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
    L.moe_backward_mxfp8.argtypes = [vp] * 11
    L.moe_plan_set_activation_scales.argtypes = [vp, f32, f32]
    L.moe_nvfp4_weight_bytes.argtypes = [i32, i32, i32, i32]
    L.moe_nvfp4_weight_bytes.restype = sz
    L.moe_prepare_weights_nvfp4.argtypes = [vp, vp, i32, i32, i32] + [vp] * 7
    L.moe_forward_nvfp4.argtypes = [vp] * 12
    L.moe_amax_bf16.argtypes = [vp, ctypes.c_longlong, vp, vp]
    L.moe_plan_set_backward_split.argtypes = [vp, i32]
    L.moe_plan_set_wgrad_interleave.argtypes = [vp, ctypes.c_longlong]
    L.moe_plan_num_sms.argtypes = [vp]
    L.moe_plan_num_sms.restype = i32
    L.moe_plan_launch_count.argtypes = [vp]
    L.moe_plan_launch_count.restype = ctypes.c_longlong
    for name in ("moe_plan_set_swiglu_clamp", "moe_plan_set_workspace", "moe_forward",
                 "moe_forward_routed",
                 "moe_backward", "moe_step_host", "moe_quantize_mxfp8", "moe_plan_check",
                 "moe_plan_buffer", "moe_gemm_bf16", "moe_plan_set_timing_events",
                 "moe_prepare_weights_mxfp8", "moe_plan_set_debug", "moe_plan_set_cta_pairs",
                 "moe_prepare_weights_mxfp8_backward", "moe_backward_mxfp8",
                 "moe_plan_set_activation_scales", "moe_prepare_weights_nvfp4",
                 "moe_forward_nvfp4", "moe_amax_bf16", "moe_plan_set_backward_split",
                 "moe_plan_set_wgrad_interleave"):
        getattr(L, name).restype = i32
    return L


def lib():
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libmoe_gb300.so is not built; run `python -m routed_mixture_experts_gb300.build` "
                    "(there is no CPU fallback)")
            _lib = _declare(ctypes.CDLL(LIB_PATH))
        return _lib


def _check(rc, what=""):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _stream(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class MoePlan:
    """A routed-expert layer plan with its workspace (a torch uint8 device tensor)."""

    def __init__(self, T, d, I, E, k, precision=MOE_PREC_BF16, clamp=0.0,
                 flags=MOE_WS_TRAINING, device="cuda", cta_pairs=False):
        import torch

        L = lib()
        self.T, self.d, self.I, self.E, self.k = T, d, I, E, k
        self.precision = precision
        self.flags = flags
        self.ptr = L.moe_plan_create(T, d, I, E, k, precision)
        if not self.ptr:
            raise MoeError(MOE_ERR_INVALID_ARG, "moe_plan_create(%d,%d,%d,%d,%d)" % (T, d, I, E, k))
        _check(L.moe_plan_set_swiglu_clamp(self.ptr, float(clamp)), "clamp")
        if cta_pairs:
            _check(L.moe_plan_set_cta_pairs(self.ptr, 1), "cta_pairs")
        nbytes = L.moe_plan_workspace_bytes(self.ptr, flags)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _check(L.moe_plan_set_workspace(self.ptr, _p(self.workspace), nbytes, flags), "workspace")

    def __del__(self):
        if getattr(self, "ptr", None) and _lib is not None:
            _lib.moe_plan_destroy(self.ptr)
            self.ptr = None

    def forward(self, x, ids, scores, w13, w2, y=None, save=False, w13_sf=None, w2_sf=None,
                stream=None):
        import torch

        if y is None:
            y = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=x.device)
        _check(lib().moe_forward(self.ptr, _p(x), _p(ids), _p(scores), _p(w13), _p(w2), _p(w13_sf),
                                 _p(w2_sf), _p(y), 1 if save else 0, _stream(stream)), "forward")
        return y

    def forward_routed(self, x_e, m_indptr, off_pad, w13, w2, score_of=None, ys=None,
                       row_of=None, y=None, stream=None):
        """Forward over caller-laid-out expert-major rows x_e [rows, d] (see
        moe_forward_routed in moe.h).  Returns (ys, y); y only with row_of."""
        import torch

        rows = x_e.shape[0]
        if ys is None:
            ys = torch.empty(rows, self.d, dtype=torch.bfloat16, device=x_e.device)
        if row_of is not None and y is None:
            y = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=x_e.device)
        _check(lib().moe_forward_routed(self.ptr, _p(x_e), rows, _p(m_indptr), _p(off_pad),
                                        _p(score_of), _p(w13), _p(w2), _p(ys), _p(row_of), _p(y),
                                        _stream(stream)), "forward_routed")
        return ys, y

    def set_activation_scales(self, x_scale, h_scale):
        """Static NVFP4 activation dequantisation scales (see moe.h)."""
        _check(lib().moe_plan_set_activation_scales(self.ptr, float(x_scale), float(h_scale)),
               "set_activation_scales")

    def forward_nvfp4(self, x, ids, scores, prepared, y=None, stream=None):
        """NVFP4 inference forward; prepared = prepare_weights_nvfp4(w13, w2)."""
        import torch

        if y is None:
            y = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=x.device)
        w13q, w13s, w13c, w2q, w2s, w2c = prepared
        _check(lib().moe_forward_nvfp4(self.ptr, _p(x), _p(ids), _p(scores), _p(w13q), _p(w13s),
                                       _p(w13c), _p(w2q), _p(w2s), _p(w2c), _p(y),
                                       _stream(stream)), "forward_nvfp4")
        return y

    def backward(self, dy, w13, w2, dw13, dw2, dx=None, dscores=None, stream=None):
        import torch

        if dx is None:
            dx = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=dy.device)
        if dscores is None:
            dscores = torch.empty(self.T, self.k, dtype=torch.float32, device=dy.device)
        _check(lib().moe_backward(self.ptr, _p(dy), _p(w13), _p(w2), _p(dx), _p(dw13), _p(dw2),
                                  _p(dscores), _stream(stream)), "backward")
        return dx, dscores

    def backward_mxfp8(self, dy, w13t, w13t_sf, w2t, w2t_sf, dw13, dw2, dx=None, dscores=None,
                       stream=None):
        """Backward of an MXFP8 plan; w13t.. from prepare_weights_mxfp8_backward."""
        import torch

        if dx is None:
            dx = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=dy.device)
        if dscores is None:
            dscores = torch.empty(self.T, self.k, dtype=torch.float32, device=dy.device)
        _check(lib().moe_backward_mxfp8(self.ptr, _p(dy), _p(w13t), _p(w13t_sf), _p(w2t),
                                        _p(w2t_sf), _p(dx), _p(dw13), _p(dw2), _p(dscores),
                                        _stream(stream)), "backward_mxfp8")
        return dx, dscores

    def step_host(self, x_h, ids_h, scores_h, w13, w2, y_h, dy_h=None, dw13=None, dw2=None,
                  dx_h=None, dscores_h=None, stream=None):
        _check(lib().moe_step_host(self.ptr, _p(x_h), _p(ids_h), _p(scores_h), _p(dy_h), _p(w13),
                                   _p(w2), _p(dw13), _p(dw2), _p(y_h), _p(dx_h), _p(dscores_h),
                                   _stream(stream)), "step_host")

    def set_timing_events(self, which, events):
        """Record `events` (torch.cuda.Event list, None entries skipped; or None) at the
        stage boundaries of every following forward (which=0) or backward (which=1) call."""
        if not events:
            self._ev = getattr(self, "_ev", {})
            self._ev.pop(which, None)
            _check(lib().moe_plan_set_timing_events(self.ptr, which, None, 0), "timing")
            return
        handles = [None if e is None else e.cuda_event for e in events]
        arr = (ctypes.c_void_p * len(events))(*handles)
        self._ev = getattr(self, "_ev", {})
        self._ev[which] = (arr, events)          # keep the handles alive while set
        _check(lib().moe_plan_set_timing_events(self.ptr, which, arr, len(events)), "timing")

    def set_backward_split(self, wgrad_sms):
        """Weight-gradient GEMMs on wgrad_sms SMs beside DGRAD-W13 (0: off); see moe.h."""
        _check(lib().moe_plan_set_backward_split(self.ptr, int(wgrad_sms)), "backward_split")

    def set_wgrad_interleave(self, min_rows):
        """Weight-gradient tiles of experts with more than min_rows rows run
        interleaved with the lighter ones (0: plain order); see moe.h."""
        _check(lib().moe_plan_set_wgrad_interleave(self.ptr, int(min_rows)), "wgrad_interleave")

    def num_sms(self):
        return lib().moe_plan_num_sms(self.ptr)

    def set_debug(self, wait_limit_ns=0, stall_w13=False):
        """Failure-path testing knobs (see moe_plan_set_debug in moe.h)."""
        _check(lib().moe_plan_set_debug(self.ptr, int(wait_limit_ns), 1 if stall_w13 else 0),
               "set_debug")

    def row_granule(self):
        """Padding granule of the expert segments (128, or 256 with CTA-pair GEMMs)."""
        return lib().moe_plan_row_granule(self.ptr)

    def launch_count(self):
        return lib().moe_plan_launch_count(self.ptr)

    def check(self):
        """Synchronise and return (status, detail) of the device error word."""
        det = ctypes.c_longlong(0)
        rc = lib().moe_plan_check(self.ptr, ctypes.byref(det))
        return rc, det.value

    def buffer(self, name, dtype, shape=None):
        """A torch view of one internal workspace tensor (see MOE_BUF_* in moe.h)."""
        import torch

        ptr = ctypes.c_void_p()
        nb = ctypes.c_size_t()
        _check(lib().moe_plan_buffer(self.ptr, MOE_BUF[name], ctypes.byref(ptr), ctypes.byref(nb)),
               name)
        off = ptr.value - self.workspace.data_ptr()
        t = self.workspace[off:off + nb.value].view(dtype)
        return t if shape is None else t[: int(torch.tensor(shape).prod())].view(*shape)


def quantize_mxfp8(w, stream=None):
    """bf16 [..., K] -> (E4M3 codes uint8 [..., K], E8M0 scales uint8 [..., K/32])."""
    import torch

    K = w.shape[-1]
    rows = w.numel() // K
    codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    scales = torch.empty(w.shape[:-1] + (K // 32,), dtype=torch.uint8, device=w.device)
    _check(lib().moe_quantize_mxfp8(_p(w), rows, K, _p(codes), _p(scales), _stream(stream)),
           "quantize_mxfp8")
    return codes, scales


def prepare_weights_mxfp8(w13, w2, stream=None):
    """bf16 W13 [E,2I,d], W2 [E,d,I] -> (w13 codes, w13 tiled scales, w2 codes,
    w2 tiled scales), the prepared MXFP8 weights of moe_forward."""
    import torch

    E, I2, d = w13.shape
    I = I2 // 2
    L = lib()
    w13q = torch.empty(w13.shape, dtype=torch.uint8, device=w13.device)
    w2q = torch.empty(w2.shape, dtype=torch.uint8, device=w2.device)
    w13s = torch.empty(L.moe_mxfp8_weight_scale_bytes(d, I, E, 0), dtype=torch.uint8,
                       device=w13.device)
    w2s = torch.empty(L.moe_mxfp8_weight_scale_bytes(d, I, E, 1), dtype=torch.uint8,
                      device=w2.device)
    _check(L.moe_prepare_weights_mxfp8(_p(w13), _p(w2), d, I, E, _p(w13q), _p(w13s), _p(w2q),
                                       _p(w2s), _stream(stream)), "prepare_weights_mxfp8")
    return w13q, w13s, w2q, w2s


def prepare_weights_nvfp4(w13, w2, stream=None):
    """bf16 W13 [E,2I,d], W2 [E,d,I] -> (w13 codes, w13 tiled scales, w13 per-expert
    scales, w2 codes, w2 tiled scales, w2 per-expert scales), the prepared NVFP4
    weights of moe_forward_nvfp4."""
    import torch

    E, I2, d = w13.shape
    I = I2 // 2
    L = lib()
    dev = w13.device
    nb = lambda which: L.moe_nvfp4_weight_bytes(d, I, E, which)
    w13q = torch.empty(E, I2, d // 2, dtype=torch.uint8, device=dev)
    w13s = torch.empty(nb(1), dtype=torch.uint8, device=dev)
    w2q = torch.empty(E, d, I // 2, dtype=torch.uint8, device=dev)
    w2s = torch.empty(nb(3), dtype=torch.uint8, device=dev)
    w13c = torch.empty(E, dtype=torch.float32, device=dev)
    w2c = torch.empty(E, dtype=torch.float32, device=dev)
    _check(L.moe_prepare_weights_nvfp4(_p(w13), _p(w2), d, I, E, _p(w13q), _p(w13s), _p(w13c),
                                       _p(w2q), _p(w2s), _p(w2c), _stream(stream)),
           "prepare_weights_nvfp4")
    return w13q, w13s, w13c, w2q, w2s, w2c


def amax_bf16(t, stream=None):
    """max |t| of a bf16 device tensor, as a one-element fp32 device tensor."""
    import torch

    out = torch.empty(1, dtype=torch.float32, device=t.device)
    _check(lib().moe_amax_bf16(_p(t), t.numel(), _p(out), _stream(stream)), "amax_bf16")
    return out


def prepare_weights_mxfp8_backward(w13, w2, stream=None):
    """bf16 W13 [E,2I,d], W2 [E,d,I] -> (W13^T codes [E,d,2I], their tiled scales,
    W2^T codes [E,I,d], their tiled scales), the prepared weights of
    moe_backward_mxfp8 (quantised along 2I and along d)."""
    import torch

    E, I2, d = w13.shape
    I = I2 // 2
    L = lib()
    w13t = torch.empty(E, d, I2, dtype=torch.uint8, device=w13.device)
    w2t = torch.empty(E, I, d, dtype=torch.uint8, device=w2.device)
    w13ts = torch.empty(L.moe_mxfp8_weight_scale_bytes(d, I, E, 2), dtype=torch.uint8,
                        device=w13.device)
    w2ts = torch.empty(L.moe_mxfp8_weight_scale_bytes(d, I, E, 3), dtype=torch.uint8,
                       device=w2.device)
    _check(L.moe_prepare_weights_mxfp8_backward(_p(w13), _p(w2), d, I, E, _p(w13t), _p(w13ts),
                                                _p(w2t), _p(w2ts), _stream(stream)),
           "prepare_weights_mxfp8_backward")
    return w13t, w13ts, w2t, w2ts


def gemm_bf16(mode, A, B, C, M, N, K, stream=None):
    """Dense GEMM through the grouped tcgen05 kernels (modes as in moe.h)."""
    import torch

    L = lib()
    scratch = torch.empty(L.moe_gemm_scratch_bytes(M, K), dtype=torch.uint8, device=A.device)
    _check(L.moe_gemm_bf16(mode, _p(A), _p(B), _p(C), M, N, K, _p(scratch), _stream(stream)),
           "gemm_bf16")
    return C
