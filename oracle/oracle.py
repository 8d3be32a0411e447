"""ctypes wrapper around the plain C++ oracle (test infrastructure only).

bf16 tensors cross this interface as numpy ``uint16`` arrays holding raw bit
patterns; ids are ``int32``; scores and gradients ``float32``.
"""

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIBS = {
    "float": os.path.join(_HERE, "_build", "libmoe_oracle.so"),
    "double": os.path.join(_HERE, "_build", "libmoe_oracle_f64.so"),
}
_lock = threading.Lock()
_cache = {}


def build_oracle(force=False):
    """Compile both oracle builds (working type float, and double), with OpenMP
    where the compiler has it (the parallel loops keep every summation order, so
    the results do not depend on the thread count)."""
    os.makedirs(os.path.join(_HERE, "_build"), exist_ok=True)
    for kind, out in _LIBS.items():
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            continue
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", out + ".tmp", _SRC]
        if kind == "double":
            cmd.insert(1, "-DORC_DOUBLE")
        r = subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True, text=True)
        if r.returncode != 0:
            subprocess.check_call(cmd)
        os.replace(out + ".tmp", out)


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """Typed entry points of one oracle build."""

    def __init__(self, path):
        self.lib = ctypes.CDLL(path)
        L = self.lib
        vp, i32, f32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_long
        L.orc_real_bytes.restype = i32
        L.orc_float_to_bf16.argtypes = [vp, vp, i64]
        L.orc_dispatch.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.orc_dispatch.restype = i64
        L.orc_gather_rows.argtypes = [i32, i32, vp, vp, vp]
        L.orc_combine_rows.argtypes = [i32, i32, i32, vp, vp, vp]
        L.orc_forward.argtypes = [i32] * 5 + [f32] + [vp] * 5 + [i32, vp] + [vp] * 4
        L.orc_backward.argtypes = [i32] * 5 + [f32] + [vp] * 6 + [i32, vp] + [vp] * 6
        L.orc_wgrad_expert.argtypes = [i32] * 5 + [f32] + [vp] * 6 + [i32, vp, vp]
        L.orc_quant_mxfp8.argtypes = [i64, i32, vp, vp, vp]
        L.orc_e4m3_encode.argtypes = [vp, vp, i64]
        L.orc_e4m3_decode.argtypes = [vp, vp, i64]
        L.orc_forward_mxfp8.argtypes = [i32] * 5 + [f32] + [vp] * 7 + [i32, vp, vp, vp]
        L.orc_backward_mxfp8.argtypes = [i32] * 5 + [f32] + [vp] * 12 + [i32] + [vp] * 6
        L.orc_wgrad_expert_mxfp8.argtypes = [i32] * 5 + [f32] + [vp] * 12 + [i32, vp, vp]
        L.orc_e2m1_encode.argtypes = [vp, vp, i64]
        L.orc_e2m1_decode.argtypes = [vp, vp, i64]
        L.orc_quant_nvfp4.argtypes = [i64, i32, vp, f32, vp, vp]
        L.orc_prepare_nvfp4.argtypes = [i32, i64, i32, vp, vp, vp, vp]
        L.orc_forward_nvfp4.argtypes = ([i32] * 5 + [f32] + [vp] * 9 + [f32, f32, i32, vp]
                                        + [vp] * 3)
        L.orc_threads.restype = i32
        L.orc_set_threads.argtypes = [i32]
        L.orc_set_threads.restype = i32
        self.real_bytes = L.orc_real_bytes()

    def threads(self):
        """Host threads of the parallel loops (1 without OpenMP)."""
        return self.lib.orc_threads()

    def set_threads(self, n):
        """Use n host threads (results do not depend on n)."""
        return self.lib.orc_set_threads(int(n))

    # -- scalar helpers -------------------------------------------------------
    def float_to_bf16(self, f):
        f = np.ascontiguousarray(f, dtype=np.float32)
        out = np.empty(f.shape, np.uint16)
        self.lib.orc_float_to_bf16(_ptr(f), _ptr(out), f.size)
        return out

    # -- dispatch / gather / combine ------------------------------------------
    def dispatch(self, ids, E, BM):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, k = ids.shape
        counts = np.empty(E, np.int32)
        m_indptr = np.empty(E + 1, np.int32)
        off_pad = np.empty(E + 1, np.int32)
        rank_of = np.empty(T * k, np.int32)
        row_of = np.empty(T * k, np.int32)
        bad = self.lib.orc_dispatch(T, k, E, BM, _ptr(ids), _ptr(counts), _ptr(m_indptr),
                                    _ptr(off_pad), _ptr(rank_of), _ptr(row_of))
        return dict(counts=counts, m_indptr=m_indptr, off_pad=off_pad,
                    rank_of=rank_of.reshape(T, k), row_of=row_of.reshape(T, k), first_bad=bad)

    def gather_rows(self, x, token_of):
        x = np.ascontiguousarray(x, np.uint16)
        token_of = np.ascontiguousarray(token_of, np.int32)
        d = x.shape[1]
        out = np.empty((token_of.size, d), np.uint16)
        self.lib.orc_gather_rows(token_of.size, d, _ptr(x), _ptr(token_of), _ptr(out))
        return out

    def combine_rows(self, ys, row_of):
        ys = np.ascontiguousarray(ys, np.uint16)
        row_of = np.ascontiguousarray(row_of, np.int32)
        T, k = row_of.shape
        d = ys.shape[1]
        y = np.empty((T, d), np.uint16)
        self.lib.orc_combine_rows(T, k, d, _ptr(ys), _ptr(row_of), _ptr(y))
        return y

    # -- forward / backward ----------------------------------------------------
    @staticmethod
    def _dims(x, ids, w13):
        T, d = x.shape
        k = ids.shape[1]
        E, I2, _ = w13.shape
        return T, d, I2 // 2, E, k

    def forward(self, x, ids, scores, w13, w2, clamp=0.0, toks=None, intermediates=False):
        T, d, I, E, k = self._dims(x, ids, w13)
        toks_a = None if toks is None else np.ascontiguousarray(toks, np.int32)
        n = T if toks is None else toks_a.size
        y = np.empty((n, d), np.uint16)
        a = h = ys = None
        if intermediates:
            a = np.empty((n, k, 2 * I), np.uint16)
            h = np.empty((n, k, I), np.uint16)
            ys = np.empty((n, k, d), np.uint16)
        self.lib.orc_forward(T, d, I, E, k, float(clamp), _ptr(x), _ptr(ids), _ptr(scores),
                             _ptr(w13), _ptr(w2), n, _ptr(toks_a), _ptr(y), _ptr(a), _ptr(h), _ptr(ys))
        if intermediates:
            return y, dict(a=a, h=h, ys=ys)
        return y

    def backward(self, x, ids, scores, w13, w2, dy, clamp=0.0, toks=None, intermediates=False):
        T, d, I, E, k = self._dims(x, ids, w13)
        toks_a = None if toks is None else np.ascontiguousarray(toks, np.int32)
        n = T if toks is None else toks_a.size
        dx = np.empty((n, d), np.uint16)
        ds = np.empty((n, k), np.float32)
        dA = hs = g = dxe = None
        if intermediates:
            dA = np.empty((n, k, 2 * I), np.uint16)
            hs = np.empty((n, k, I), np.uint16)
            g = np.empty((n, k, I), np.float32)
            dxe = np.empty((n, k, d), np.uint16)
        self.lib.orc_backward(T, d, I, E, k, float(clamp), _ptr(x), _ptr(ids), _ptr(scores),
                              _ptr(w13), _ptr(w2), _ptr(dy), n, _ptr(toks_a), _ptr(dx), _ptr(ds),
                              _ptr(dA), _ptr(hs), _ptr(g), _ptr(dxe))
        if intermediates:
            return dx, ds, dict(dA=dA, hs=hs, g=g, dxe=dxe)
        return dx, ds

    def wgrad_expert(self, x, ids, scores, w13, w2, dy, e, clamp=0.0):
        T, d, I, E, k = self._dims(x, ids, w13)
        d13 = np.empty((2 * I, d), np.float32)
        d2 = np.empty((d, I), np.float32)
        rows = self.lib.orc_wgrad_expert(T, d, I, E, k, float(clamp), _ptr(x), _ptr(ids),
                                         _ptr(scores), _ptr(w13), _ptr(w2), _ptr(dy), int(e),
                                         _ptr(d13), _ptr(d2))
        return d13, d2, rows

    # -- MXFP8 -----------------------------------------------------------------
    def quant_mxfp8(self, m):
        m = np.ascontiguousarray(m, np.uint16)
        K = m.shape[-1]
        rows = m.size // K
        codes = np.empty(m.shape, np.uint8)
        scales = np.empty(m.shape[:-1] + (K // 32,), np.uint8)
        rc = self.lib.orc_quant_mxfp8(rows, K, _ptr(m), _ptr(codes), _ptr(scales))
        assert rc == 0
        return codes, scales

    def e4m3_encode(self, v):
        v = np.ascontiguousarray(v, np.float64)
        out = np.empty(v.shape, np.uint8)
        self.lib.orc_e4m3_encode(_ptr(v), _ptr(out), v.size)
        return out

    def e4m3_decode(self, c):
        c = np.ascontiguousarray(c, np.uint8)
        out = np.empty(c.shape, np.float64)
        self.lib.orc_e4m3_decode(_ptr(c), _ptr(out), c.size)
        return out

    def forward_mxfp8(self, x, ids, scores, w13q, w13s, w2q, w2s, clamp=0.0, toks=None,
                      return_h=False):
        T, d = x.shape
        k = ids.shape[1]
        E, I2, _ = w13q.shape
        I = I2 // 2
        toks_a = None if toks is None else np.ascontiguousarray(toks, np.int32)
        n = T if toks is None else toks_a.size
        y = np.empty((n, d), np.uint16)
        h = np.empty((n, k, I), np.uint16) if return_h else None
        self.lib.orc_forward_mxfp8(T, d, I, E, k, float(clamp), _ptr(x), _ptr(ids), _ptr(scores),
                                   _ptr(w13q), _ptr(w13s), _ptr(w2q), _ptr(w2s), n, _ptr(toks_a),
                                   _ptr(y), _ptr(h))
        return (y, h) if return_h else y

    def prepare_mxfp8_backward_weights(self, w13, w2):
        """Weights prepared for the MXFP8 backward GEMMs (quantised along their K):
        W2[e]^T [E, I, d] along d and W13[e]^T [E, d, 2I] along 2I."""
        w2t = np.ascontiguousarray(np.swapaxes(w2, 1, 2))
        w13t = np.ascontiguousarray(np.swapaxes(w13, 1, 2))
        w2tq, w2ts = self.quant_mxfp8(w2t)
        w13tq, w13ts = self.quant_mxfp8(w13t)
        return w13tq, w13ts, w2tq, w2ts

    def backward_mxfp8(self, x, ids, scores, fw, bw, dy, clamp=0.0, toks=None,
                       intermediates=False):
        """fw = (w13q, w13s, w2q, w2s) prepared along K of the forward GEMMs;
        bw = (w13tq, w13ts, w2tq, w2ts) from prepare_mxfp8_backward_weights."""
        T, d = x.shape
        k = ids.shape[1]
        E, I2, _ = fw[0].shape
        I = I2 // 2
        toks_a = None if toks is None else np.ascontiguousarray(toks, np.int32)
        n = T if toks is None else toks_a.size
        dx = np.empty((n, d), np.uint16)
        ds = np.empty((n, k), np.float32)
        dA = hs = dxe = None
        if intermediates:
            dA = np.empty((n, k, 2 * I), np.uint16)
            hs = np.empty((n, k, I), np.uint16)
            dxe = np.empty((n, k, d), np.uint16)
        self.lib.orc_backward_mxfp8(T, d, I, E, k, float(clamp), _ptr(x), _ptr(ids), _ptr(scores),
                                    *[_ptr(np.ascontiguousarray(w)) for w in fw],
                                    *[_ptr(np.ascontiguousarray(w)) for w in bw], _ptr(dy),
                                    n, _ptr(toks_a), _ptr(dx), _ptr(ds), _ptr(dA), _ptr(hs),
                                    _ptr(dxe))
        if intermediates:
            return dx, ds, dict(dA=dA, hs=hs, dxe=dxe)
        return dx, ds

    def wgrad_expert_mxfp8(self, x, ids, scores, fw, bw, dy, e, clamp=0.0):
        T, d = x.shape
        k = ids.shape[1]
        E, I2, _ = fw[0].shape
        I = I2 // 2
        d13 = np.empty((2 * I, d), np.float32)
        d2 = np.empty((d, I), np.float32)
        rows = self.lib.orc_wgrad_expert_mxfp8(T, d, I, E, k, float(clamp), _ptr(x), _ptr(ids),
                                               _ptr(scores),
                                               *[_ptr(np.ascontiguousarray(w)) for w in fw],
                                               *[_ptr(np.ascontiguousarray(w)) for w in bw],
                                               _ptr(dy), int(e), _ptr(d13), _ptr(d2))
        return d13, d2, rows


def _nvfp4_methods(cls):
    """NVFP4 entry points (E2M1 codes, E4M3 scales per 16 elements, per-tensor
    scale)."""

    def e2m1_encode(self, v):
        v = np.ascontiguousarray(v, np.float64)
        out = np.empty(v.shape, np.uint8)
        self.lib.orc_e2m1_encode(_ptr(v), _ptr(out), v.size)
        return out

    def e2m1_decode(self, c):
        c = np.ascontiguousarray(c, np.uint8)
        out = np.empty(c.shape, np.float64)
        self.lib.orc_e2m1_decode(_ptr(c), _ptr(out), c.size)
        return out

    def quant_nvfp4(self, m, g):
        """bf16 [..., K] with encode scale g -> (packed codes uint8 [..., K/2],
        E4M3 scales uint8 [..., K/16])."""
        m = np.ascontiguousarray(m, np.uint16)
        K = m.shape[-1]
        rows = m.size // K
        codes = np.empty(m.shape[:-1] + (K // 2,), np.uint8)
        scales = np.empty(m.shape[:-1] + (K // 16,), np.uint8)
        rc = self.lib.orc_quant_nvfp4(rows, K, _ptr(m), float(g), _ptr(codes), _ptr(scales))
        assert rc == 0
        return codes, scales

    def prepare_nvfp4(self, w):
        """bf16 [E, rows, K] -> (codes [E, rows, K/2], scales [E, rows, K/16],
        per-expert dequantisation scales float32 [E])."""
        w = np.ascontiguousarray(w, np.uint16)
        E, rows, K = w.shape
        codes = np.empty((E, rows, K // 2), np.uint8)
        scales = np.empty((E, rows, K // 16), np.uint8)
        sc = np.empty(E, np.float32)
        rc = self.lib.orc_prepare_nvfp4(E, rows, K, _ptr(w), _ptr(codes), _ptr(scales), _ptr(sc))
        assert rc == 0
        return codes, scales, sc

    def forward_nvfp4(self, x, ids, scores, w13p, w2p, x_scale, h_scale, clamp=0.0, toks=None,
                      intermediates=False):
        """w13p = prepare_nvfp4(W13), w2p = prepare_nvfp4(W2)."""
        T, d = x.shape
        k = ids.shape[1]
        E, I2, _ = w13p[0].shape
        I = I2 // 2
        toks_a = None if toks is None else np.ascontiguousarray(toks, np.int32)
        n = T if toks is None else toks_a.size
        y = np.empty((n, d), np.uint16)
        a = h = None
        if intermediates:
            a = np.empty((n, k, 2 * I), np.uint16)
            h = np.empty((n, k, I), np.uint16)
        c = lambda v: np.ascontiguousarray(v)
        self.lib.orc_forward_nvfp4(T, d, I, E, k, float(clamp), _ptr(c(x)), _ptr(c(ids)),
                                   _ptr(c(scores)), _ptr(c(w13p[0])), _ptr(c(w13p[1])),
                                   _ptr(c(np.asarray(w13p[2], np.float32))), _ptr(c(w2p[0])),
                                   _ptr(c(w2p[1])), _ptr(c(np.asarray(w2p[2], np.float32))),
                                   float(x_scale), float(h_scale), n, _ptr(toks_a), _ptr(y),
                                   _ptr(a), _ptr(h))
        if intermediates:
            return y, dict(a=a, h=h)
        return y

    for f in (e2m1_encode, e2m1_decode, quant_nvfp4, prepare_nvfp4, forward_nvfp4):
        setattr(cls, f.__name__, f)
    return cls


_nvfp4_methods(Oracle)


def load_oracle(kind="float"):
    """The oracle build whose working type is ``kind`` ("float" or "double")."""
    with _lock:
        if kind not in _cache:
            build_oracle()
            _cache[kind] = Oracle(_LIBS[kind])
        return _cache[kind]
