"""The C++ oracle (oracle/q4_oracle.cpp) behind the numpy oracle's API.

TEST INFRASTRUCTURE ONLY, like every module of this package: only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline legs use it.

This module only marshals arrays (shape checks, output allocation, dtype of
the returned arrays); every arithmetic step runs in the compiled C++ file,
which shares no code with the numpy oracle or the CUDA library.  The functions
take the same arguments and return the same dtypes as :mod:`oracle.q4_oracle`,
so the same pins run against both.  ``threads`` splits rows of a contraction
over host threads; results do not depend on it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "q4_oracle.cpp")
LIB = os.path.join(HERE, "libq4oracle.so")
CXXFLAGS = ["-O2", "-std=c++17", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-pthread"]

SOFTCAP = 30.0
E2B_LAYERS = 35
E2B_HIDDEN = 1536

_lib = None
_p = ctypes.c_void_p
_i = ctypes.c_int
_ll = ctypes.c_longlong
_d = ctypes.c_double
_f = ctypes.c_float


class _Mat(ctypes.Structure):
    _fields_ = [("codes", _p), ("scales", _p)]


_SIGS = {
    "q4o_version": (_i, []),
    "q4o_f16_from_f64": (None, [_p, _p, _ll]),
    "q4o_f64_from_f16": (None, [_p, _p, _ll]),
    "q4o_bf16_rne": (None, [_p, _p, _ll]),
    "q4o_quantize": (_i, [_p, _i, _i, _p, _p, _i]),
    "q4o_dequantize": (None, [_p, _p, _i, _i, _p]),
    "q4o_gemv": (None, [_p, _p, _p, _i, _i, _i, _p, _i]),
    "q4o_gemm_chunk": (None, [_p, _p, _p, _i, _i, _i, _p, _i]),
    "q4o_softcap": (None, [_p, _p, _ll, _d]),
    "q4o_lmhead": (None, [_p, _p, _p, _i, _i, _i, _d, _p, _p, _p, _p, _i]),
    "q4o_rmsnorm": (None, [_p, _p, _d, _ll, _i, _p]),
    "q4o_gelu_tanh": (None, [_p, _p, _ll]),
    "q4o_ple_embed_scale": (_d, []),
    "q4o_ple": (_i, [_p, _i, _p, _p, _i, _i, _i, _f, _p, _p, _i, _p, _d, _p, _p, _i]),
    "q4o_e2b_layer_dims": (None, [_i, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "q4o_e2b_layer": (None, [_p, _i, ctypes.POINTER(_Mat), _i, _i, _i, _d] + [_p] * 11 + [_i]),
    "q4o_e2b_pass": (None, [_p, _i, ctypes.POINTER(_Mat), _p, _i, _d, _p, _i]),
    "q4o_q2_gemv": (None, [_p, _p, _p, _i, _i, _i, _p, _i]),
    "q4o_q8_quantize": (_i, [_p, _i, _i, _p, _p]),
    "q4o_q8_dequantize": (None, [_p, _p, _i, _i, _p]),
    "q4o_ple_q8": (_i, [_p, _i, _p, _p, _i, _i, _i, _f, _p, _p, _p, _i, _p, _d, _p, _p, _i]),
    "q4o_a8_calibrate": (_f, [_p, _ll]),
    "q4o_a8_quantize": (None, [_p, _ll, _f, _p]),
    "q4o_gemv_a8": (None, [_p, _p, _p, _i, _i, _f, _p, _i]),
    "q4o_gemm_chunk_a8": (None, [_p, _p, _p, _i, _i, _i, _f, _p, _i]),
}


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile the C++ oracle with the system C++ compiler (g++), once."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["g++", *CXXFLAGS, "-o", out + ".tmp", src]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("C++ oracle build failed:\n" + r.stderr[-4000:])
    os.replace(out + ".tmp", out)
    return out


def load(path: str | None = None):
    """Load the compiled oracle (building it first if needed); ``path`` loads
    another build of the source (the mutant tests use that)."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(threads):
    return int(threads) if threads else 1


class Oracle:
    """One loaded build of the C++ oracle, with the numpy oracle's functions."""

    def __init__(self, lib):
        self.lib = lib
        self.PLE_EMBED_SCALE = float(lib.q4o_ple_embed_scale())
        self.E2B_FULL_LAYERS = tuple(l for l in range(E2B_LAYERS) if self.e2b_layer_dims(l)["q"] == 4096)
        self.SOFTCAP = SOFTCAP

    # number formats
    def to_f16(self, v):
        v = np.ascontiguousarray(v, dtype=np.float64)
        bits = np.empty(v.shape, dtype=np.uint16)
        self.lib.q4o_f16_from_f64(_ptr(v), _ptr(bits), v.size)
        return bits.view(np.float16)

    def f16_from_bits(self, bits):
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(bits.shape, dtype=np.float64)
        self.lib.q4o_f64_from_f16(_ptr(bits), _ptr(out), bits.size)
        return out

    def bf16_rne(self, v):
        v = np.ascontiguousarray(v, dtype=np.float32)
        out = np.empty_like(v)
        self.lib.q4o_bf16_rne(_ptr(v), _ptr(out), v.size)
        return out

    # a1
    def quantize_q4_0(self, W, threads=1):
        W = np.ascontiguousarray(W, dtype=np.float32)
        if W.ndim != 2 or W.shape[1] % 32:
            raise ValueError("W must be [N, K] with K a multiple of 32")
        N, K = W.shape
        codes = np.empty((N, K // 2), dtype=np.uint8)
        scales = np.empty((N, K // 32), dtype=np.uint16)
        st = self.lib.q4o_quantize(_ptr(W), N, K, _ptr(codes), _ptr(scales), _threads(threads))
        if st == 2:
            raise ValueError("non-finite weight")
        if st == 3:
            raise ValueError("block scale overflows fp16")
        if st != 0:
            raise ValueError(f"quantize failed ({st})")
        return codes, scales

    def dequantize_q4_0(self, codes, scales):
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        N, K = codes.shape[0], codes.shape[1] * 2
        out = np.empty((N, K), dtype=np.float64)
        self.lib.q4o_dequantize(_ptr(codes), _ptr(scales), N, K, _ptr(out))
        return out

    # a2
    def q4_gemv64(self, codes, scales, x_f16, threads=1):
        """The fp64 sums before the fp32 rounding of :meth:`q4_gemv`."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        x = np.ascontiguousarray(x_f16, dtype=np.float16)
        N, K = codes.shape[0], codes.shape[1] * 2
        B = 1 if x.ndim == 1 else x.shape[0]
        if x.size != B * K:
            raise ValueError("x must hold b rows of K values")
        y = np.empty((B, N), dtype=np.float64)
        self.lib.q4o_gemv(_ptr(codes), _ptr(scales), _ptr(x.view(np.uint16)), N, K, B, _ptr(y), _threads(threads))
        return y[0] if x.ndim == 1 else y

    def q4_gemv(self, codes, scales, x_f16, threads=1):
        return self.q4_gemv64(codes, scales, x_f16, threads).astype(np.float32)

    # a6
    def q4_gemm_chunk64(self, codes, scales, X_f16, threads=1):
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        X = np.ascontiguousarray(np.atleast_2d(X_f16), dtype=np.float16)
        N, K = codes.shape[0], codes.shape[1] * 2
        M = X.shape[0]
        if X.shape[1] != K:
            raise ValueError("X must be [M, K]")
        Y = np.empty((M, N), dtype=np.float64)
        self.lib.q4o_gemm_chunk(_ptr(codes), _ptr(scales), _ptr(X.view(np.uint16)), M, N, K, _ptr(Y),
                                _threads(threads))
        return Y

    def q4_gemm_chunk(self, codes, scales, X_f16, threads=1):
        return self.q4_gemm_chunk64(codes, scales, X_f16, threads).astype(np.float32)

    # a5
    def softcap(self, z, cap=SOFTCAP):
        z = np.ascontiguousarray(z, dtype=np.float64)
        s = np.empty_like(z)
        self.lib.q4o_softcap(_ptr(z), _ptr(s), z.size, float(cap))
        return s

    def lmhead64(self, codes, scales, h_f16, cap=SOFTCAP, threads=1, logits=True):
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        h = np.ascontiguousarray(np.atleast_2d(h_f16), dtype=np.float16)
        V, K = codes.shape[0], codes.shape[1] * 2
        B = h.shape[0]
        idx = np.empty(B, dtype=np.int32)
        t1 = np.empty(B, dtype=np.float64)
        t2 = np.empty(B, dtype=np.float64)
        s = np.empty((B, V), dtype=np.float64) if logits else None
        self.lib.q4o_lmhead(_ptr(codes), _ptr(scales), _ptr(h.view(np.uint16)), B, V, K, float(cap), _ptr(idx),
                            _ptr(t1), _ptr(t2), _ptr(s), _threads(threads))
        return idx, t1, t2, s

    def lmhead_softcap_argmax(self, codes, scales, h_f16, cap=SOFTCAP, threads=1):
        idx, t1, t2, s = self.lmhead64(codes, scales, h_f16, cap, threads)
        return idx, t1.astype(np.float32), t2.astype(np.float32), t1 - t2, s.astype(np.float32)

    # a4 and a7
    def rmsnorm(self, v, w=None, eps=1e-6, axis=-1):
        if axis not in (-1, np.ndim(v) - 1):
            raise ValueError("the C++ oracle normalises over the last axis")
        v = np.ascontiguousarray(v, dtype=np.float64)
        n = v.shape[-1]
        wv = None if w is None else np.ascontiguousarray(np.broadcast_to(w, (n,)), dtype=np.float64)
        out = np.empty_like(v)
        self.lib.q4o_rmsnorm(_ptr(v), _ptr(wv), float(eps), v.size // n, n, _ptr(out))
        return out

    def gelu_tanh(self, x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        y = np.empty_like(x)
        self.lib.q4o_gelu_tanh(_ptr(x), _ptr(y), x.size)
        return y

    def ple64(self, ids, table, row_scale, proj, hidden_f16, norm_w, L=35, ld=256, embed_scale=None, eps=1e-6,
              threads=1):
        ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
        table = np.ascontiguousarray(table, dtype=np.int8)
        V, PLD = table.shape
        if PLD != L * ld:
            raise ValueError("table width must be L*ld")
        row_scale = np.ascontiguousarray(row_scale, dtype=np.float32)
        proj = np.ascontiguousarray(proj, dtype=np.float32)
        hidden = np.ascontiguousarray(np.atleast_2d(hidden_f16), dtype=np.float16)
        norm_w = np.ascontiguousarray(norm_w, dtype=np.float32)
        S, D = ids.size, proj.shape[1]
        if proj.shape[0] != L * ld or hidden.shape != (S, D) or norm_w.size != ld or row_scale.size != V:
            raise ValueError("PLE operand shapes disagree")
        out = np.empty((S, L * ld), dtype=np.float64)
        gathered = np.empty((S, L * ld), dtype=np.int8)
        es = self.PLE_EMBED_SCALE if embed_scale is None else float(embed_scale)
        st = self.lib.q4o_ple(_ptr(ids), S, _ptr(table), _ptr(row_scale), V, L, ld, es, _ptr(proj),
                              _ptr(hidden.view(np.uint16)), D, _ptr(norm_w), float(eps), _ptr(out), _ptr(gathered),
                              _threads(threads))
        if st != 0:
            raise ValueError("token id out of range")
        return out, gathered

    def ple_gather_project(self, ids, table, row_scale, proj, hidden_f16, norm_w, L=35, ld=256, embed_scale=None,
                           eps=1e-6, threads=1):
        out, gathered = self.ple64(ids, table, row_scale, proj, hidden_f16, norm_w, L, ld, embed_scale, eps, threads)
        return out.astype(np.float32), gathered

    # NEXT-2: INT2 per-row symmetric GEMV (oracle.q2_oracle's API)
    def q2_gemv(self, codes, scales, x_f16, threads=1):
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.float32)
        x = np.ascontiguousarray(x_f16, dtype=np.float16)
        N, K = codes.shape[0], codes.shape[1] * 4
        B = 1 if x.ndim == 1 else x.shape[0]
        if x.size != B * K or scales.size != N:
            raise ValueError("INT2 operand shapes disagree")
        y = np.empty((B, N), dtype=np.float64)
        self.lib.q4o_q2_gemv(_ptr(codes), _ptr(scales), _ptr(x.view(np.uint16)), N, K, B, _ptr(y), _threads(threads))
        return y[0] if x.ndim == 1 else y

    # NEXT-4: int8 per-block-32 weights (oracle.q8_oracle's API)
    def quantize_q8_0(self, W):
        W = np.ascontiguousarray(W, dtype=np.float32)
        if W.ndim != 2 or W.shape[1] % 32:
            raise ValueError("W must be [N, K] with K a multiple of 32")
        N, K = W.shape
        codes = np.empty((N, K), dtype=np.int8)
        scales = np.empty((N, K // 32), dtype=np.uint16)
        st = self.lib.q4o_q8_quantize(_ptr(W), N, K, _ptr(codes), _ptr(scales))
        if st == 2:
            raise ValueError("non-finite weight")
        if st == 3:
            raise ValueError("block scale overflows fp16")
        if st != 0:
            raise ValueError(f"quantize failed ({st})")
        return codes, scales

    def dequantize_q8_0(self, codes, scales):
        codes = np.ascontiguousarray(codes, dtype=np.int8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        N, K = codes.shape
        out = np.empty((N, K), dtype=np.float64)
        self.lib.q4o_q8_dequantize(_ptr(codes), _ptr(scales), N, K, _ptr(out))
        return out

    def ple_gather_project_q8(self, ids, table, row_scale, codes, scales, hidden_f16, norm_w, L=35, ld=256,
                              embed_scale=None, eps=1e-6, threads=1):
        ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
        table = np.ascontiguousarray(table, dtype=np.int8)
        V, PLD = table.shape
        codes = np.ascontiguousarray(codes, dtype=np.int8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        row_scale = np.ascontiguousarray(row_scale, dtype=np.float32)
        hidden = np.ascontiguousarray(np.atleast_2d(hidden_f16), dtype=np.float16)
        norm_w = np.ascontiguousarray(norm_w, dtype=np.float32)
        S, D = ids.size, codes.shape[1]
        if (PLD != L * ld or codes.shape[0] != L * ld or scales.size != L * ld * D // 32 or hidden.shape != (S, D)
                or norm_w.size != ld or row_scale.size != V):
            raise ValueError("PLE operand shapes disagree")
        out = np.empty((S, L * ld), dtype=np.float64)
        gathered = np.empty((S, L * ld), dtype=np.int8)
        es = self.PLE_EMBED_SCALE if embed_scale is None else float(embed_scale)
        st = self.lib.q4o_ple_q8(_ptr(ids), S, _ptr(table), _ptr(row_scale), V, L, ld, es, _ptr(codes),
                                 _ptr(scales), _ptr(hidden.view(np.uint16)), D, _ptr(norm_w), float(eps), _ptr(out),
                                 _ptr(gathered), _threads(threads))
        if st != 0:
            raise ValueError("token id out of range")
        return out.astype(np.float32), gathered

    # NEXT-4: w4a8 activation quantize/dequantize (oracle.a8_oracle's API)
    def a8_calibrate(self, samples):
        x = np.ascontiguousarray(np.asarray(samples, dtype=np.float16)).reshape(-1)
        if not np.all(np.isfinite(x.astype(np.float32))):
            raise ValueError("non-finite calibration sample")
        return np.float32(self.lib.q4o_a8_calibrate(_ptr(x.view(np.uint16)), x.size))

    @staticmethod
    def _scale(s):
        s32 = np.float32(s)
        if not (np.isfinite(s32) and s32 > 0):
            raise ValueError("the activation scale must be finite and > 0")
        return float(s32)

    def a8_quantize(self, x_f16, s):
        x = np.ascontiguousarray(np.asarray(x_f16, dtype=np.float16))
        if not np.all(np.isfinite(x.astype(np.float32))):
            raise ValueError("non-finite activation")
        q = np.empty(x.shape, dtype=np.int32)
        self.lib.q4o_a8_quantize(_ptr(x.view(np.uint16)), x.size, self._scale(s), _ptr(q))
        return q.astype(np.int64)

    def a8_qdq(self, x_f16, s):
        return self.a8_quantize(x_f16, s).astype(np.float64) * float(np.float32(s))

    def q4_gemv_a8(self, codes, scales, x_f16, s, threads=1):
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        x = np.ascontiguousarray(x_f16, dtype=np.float16).reshape(-1)
        N, K = codes.shape[0], codes.shape[1] * 2
        if x.size != K:
            raise ValueError("x must hold K values")
        y = np.empty(N, dtype=np.float64)
        self.lib.q4o_gemv_a8(_ptr(codes), _ptr(scales), _ptr(x.view(np.uint16)), N, K, self._scale(s), _ptr(y),
                             _threads(threads))
        return y.astype(np.float32)

    def q4_gemm_chunk_a8(self, codes, scales, X_f16, s, threads=1):
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        X = np.ascontiguousarray(X_f16, dtype=np.float16)
        N, K = codes.shape[0], codes.shape[1] * 2
        M = X.shape[0]
        if X.shape != (M, K):
            raise ValueError("X must be [M, K]")
        Y = np.empty((M, N), dtype=np.float64)
        self.lib.q4o_gemm_chunk_a8(_ptr(codes), _ptr(scales), _ptr(X.view(np.uint16)), M, N, K, self._scale(s),
                                   _ptr(Y), _threads(threads))
        return Y.astype(np.float32)

    # a3
    def e2b_layer_dims(self, layer):
        q, kv, mlp = _i(), _i(), _i()
        self.lib.q4o_e2b_layer_dims(int(layer), ctypes.byref(q), ctypes.byref(kv), ctypes.byref(mlp))
        return {"q": q.value, "kv": kv.value, "mlp": mlp.value}

    @staticmethod
    def _mats(lw):
        keep = []
        mats = (_Mat * 7)()
        for i, key in enumerate(("q", "k", "v", "o", "g", "u", "d")):
            if key in lw:
                c = np.ascontiguousarray(lw[key][0], dtype=np.uint8)
                s = np.ascontiguousarray(lw[key][1], dtype=np.uint16)
                keep += [c, s]
                mats[i] = _Mat(c.ctypes.data, s.ctypes.data)
        return mats, keep

    def e2b_layer(self, h_f16, lw, eps=1e-6, threads=1):
        h = np.ascontiguousarray(h_f16, dtype=np.float16)
        H = h.size
        Q, I = lw["q"][0].shape[0], lw["g"][0].shape[0]
        KV = lw["k"][0].shape[0] if "k" in lw else 0
        if ("k" in lw) != ("v" in lw):
            raise ValueError("k and v go together")
        mats, keep = self._mats(lw)
        st = {"a": np.empty(H, np.float16), "q": np.empty(Q, np.float32), "k": np.empty(max(KV, 1), np.float32),
              "v": np.empty(max(KV, 1), np.float32), "o": np.empty(H, np.float32), "b": np.empty(H, np.float16),
              "g": np.empty(I, np.float32), "u": np.empty(I, np.float32), "m": np.empty(I, np.float16),
              "y": np.empty(H, np.float32), "h": np.empty(H, np.float16)}
        order = ("a", "q", "k", "v", "o", "b", "g", "u", "m", "y", "h")
        self.lib.q4o_e2b_layer(_ptr(h.view(np.uint16)), H, mats, Q, KV, I, float(eps),
                               *[_ptr(st[n].view(np.uint16) if st[n].dtype == np.float16 else st[n]) for n in order],
                               _threads(threads))
        del keep
        if KV == 0:
            del st["k"], st["v"]
        return st

    def e2b_pass(self, h0_f16, layers, eps=1e-6, threads=1):
        """The chain over ``layers`` (each a dict as for e2b_layer); final fp16 h."""
        h = np.ascontiguousarray(h0_f16, dtype=np.float16)
        H = h.size
        n = len(layers)
        mats = (_Mat * (7 * n))()
        dims = np.empty((n, 3), dtype=np.int32)
        keep = []
        for l, lw in enumerate(layers):
            m, k = self._mats(lw)
            keep += k
            for i in range(7):
                mats[7 * l + i] = m[i]
            dims[l] = (lw["q"][0].shape[0], lw["k"][0].shape[0] if "k" in lw else 0, lw["g"][0].shape[0])
        out = np.empty(H, dtype=np.float16)
        self.lib.q4o_e2b_pass(_ptr(h.view(np.uint16)), H, mats, _ptr(dims), n, float(eps), _ptr(out.view(np.uint16)),
                              _threads(threads))
        del keep
        return out


_default = None


def oracle() -> Oracle:
    """The C++ oracle built from oracle/q4_oracle.cpp."""
    global _default
    if _default is None:
        _default = Oracle(load())
    return _default
