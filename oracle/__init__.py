"""Plain CPU oracle for the I2_S x INT8 matmul and the I8_S fused ops.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are its only users. The GPU library never imports, links or
calls anything here, and nothing here imports the GPU library.

The arithmetic lives in ``oracle.cpp`` (plain C++, -O2 -ffp-contract=off, no
fast-math). This module builds it on demand with g++ and wraps it with ctypes
over numpy arrays. Every function cites the page section it follows in the C++
source.

Parity status of each function (what pins it, in tests/test_oracle_pins.py):
  i2s_pack / i2s_unpack   hand decode of crafted groups, hand-expected bytes,
                          independent round trip
  quantize_rows           hand-computed golden rows (tests/golden/), exhaustive
                          rounding check, amax floor closed form
  i2s_mul_mat             numpy int64 matmul in the power-of-two special case,
                          accumulator-headroom closed form, brute-force code
                          identity, degenerate scales, thread-count independence
  i8s_quantize            hand-computed golden, power-of-two closed form
  i8s_mul_mat_add         numpy int64 matmul in the power-of-two special case,
                          with and without ReLU and bias
  i8s_permute_cont        numpy transpose plus the carried scale bytes
  i8s_add_scaled          power-of-two scales (exact): numpy sum; swap symmetry
  i8s_rms_norm_scaled     constant-row closed form, power-of-two scale
                          invariance, unit RMS of the rows, zero rows, gamma
                          scaling
  i8s_im2col_asym         numpy pad + strided windows, causal geometry, the
                          carried scale bytes
  i8s_depthwise_mul_mat_add  numpy per-channel correlation in the power-of-two
                          special case
  w8a8_quantize_weights   hand-made ties (ties to even), amax floor
  w8a8_mul_mat            numpy int64 matmul with power-of-two scales
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17", "-fPIC", "-shared",
          "-pthread"]


def build(out_path: str = _LIB, plant: int = 0) -> str:
    """Compile the oracle into a shared library (plant != 0: a planted mistake)."""
    cmd = ["g++", *CFLAGS, f"-DORC_PLANT={int(plant)}", _SRC, "-o", out_path]
    subprocess.run(cmd, check=True)
    return out_path


def _stale(lib: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(_SRC)


_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_int = ctypes.c_int


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one build of oracle.cpp."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            lib_path = _LIB
            if _stale(lib_path):
                build(lib_path)
        self.path = lib_path
        L = ctypes.CDLL(lib_path)
        sig = {
            "orc_i2s_nbytes": (_i64, [_i64, _i64]),
            "orc_i2s_scale_offset": (_i64, [_i64, _i64]),
            "orc_i8s_nbytes": (_i64, [_i64]),
            "orc_i8s_scale_offset": (_i64, [_i64]),
            "orc_i2s_pack": (None, [_p, _i64, _i64, _f32, _p]),
            "orc_i2s_unpack": (None, [_p, _i64, _i64, _p, _p]),
            "orc_i2s_dequantize": (None, [_p, _i64, _i64, _p]),
            "orc_round": (_f32, [_f32]),
            "orc_round_array": (None, [_p, _i64, _p]),
            "orc_quantize_rows": (None, [_p, _i64, _i64, _p, _p, _p]),
            "orc_i2s_mul_mat": (None, [_p, _i64, _i64, _p, _i64, _p, _int, _p, _p, _p, _p]),
            "orc_i8s_pack": (None, [_p, _i64, _f32, _p]),
            "orc_i8s_unpack": (_f32, [_p, _i64, _p]),
            "orc_i8s_dequantize": (None, [_p, _i64, _p]),
            "orc_i8s_quantize": (None, [_p, _i64, _p]),
            "orc_i8s_mul_mat_add": (None, [_p, _i64, _i64, _p, _i64, _p, _int, _p, _p, _int]),
            "orc_i8s_permute_cont": (None, [_p, _i64, _i64, _p]),
            "orc_i8s_add_scaled": (None, [_p, _p, _i64, _p, _p]),
            "orc_i8s_rms_norm_scaled": (None, [_p, _i64, _i64, _f32, _p, _p, _p]),
            "orc_im2col_out_len": (_i64, [_i64, _i64, _i64, _i64, _i64]),
            "orc_i8s_im2col_asym": (None, [_p, _i64, _i64, _i64, _i64, _i64, _i64, _p]),
            "orc_i8s_depthwise_mul_mat_add": (None, [_p, _i64, _p, _i64, _i64, _i64, _i64, _i64, _p, _int,
                                                     _p, _p]),
            "orc_w8a8_quantize_weights": (None, [_p, _i64, _i64, _p, _p]),
            "orc_w8a8_quantize_rows": (None, [_p, _i64, _i64, _p, _p]),
            "orc_w8a8_mul_mat": (None, [_p, _p, _i64, _i64, _p, _i64, _p, _int, _p, _p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        self._L = L

    # -- layouts ------------------------------------------------------------
    def i2s_nbytes(self, N, K):
        return int(self._L.orc_i2s_nbytes(N, K))

    def i2s_scale_offset(self, N, K):
        return int(self._L.orc_i2s_scale_offset(N, K))

    def i8s_nbytes(self, n):
        return int(self._L.orc_i8s_nbytes(n))

    def i8s_scale_offset(self, n):
        return int(self._L.orc_i8s_scale_offset(n))

    # -- I2_S -----------------------------------------------------------------
    def i2s_pack(self, codes: np.ndarray, absmax: float) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        N, K = codes.shape
        dst = np.zeros(self.i2s_nbytes(N, K), dtype=np.uint8)
        self._L.orc_i2s_pack(_ptr(codes), N, K, float(absmax), _ptr(dst))
        return dst

    def i2s_unpack(self, packed: np.ndarray, N: int, K: int):
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        codes = np.zeros((N, K), dtype=np.uint8)
        a = np.zeros(1, dtype=np.float32)
        self._L.orc_i2s_unpack(_ptr(packed), N, K, _ptr(codes), _ptr(a))
        return codes, float(a[0])

    def i2s_dequantize(self, packed, N, K):
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        w = np.zeros((N, K), dtype=np.float32)
        self._L.orc_i2s_dequantize(_ptr(packed), N, K, _ptr(w))
        return w

    # -- quantizer ----------------------------------------------------------
    def round(self, v: float) -> float:
        return float(self._L.orc_round(float(v)))

    def round_array(self, v: np.ndarray) -> np.ndarray:
        v = np.ascontiguousarray(v, dtype=np.float32)
        out = np.empty_like(v)
        self._L.orc_round_array(_ptr(v), v.size, _ptr(out))
        return out

    def quantize_rows(self, x: np.ndarray):
        x = np.ascontiguousarray(x, dtype=np.float32)
        M, K = x.shape
        q = np.zeros((M, K), dtype=np.int8)
        s = np.zeros(M, dtype=np.float32)
        rs = np.zeros(M, dtype=np.int32)
        self._L.orc_quantize_rows(_ptr(x), M, K, _ptr(q), _ptr(s), _ptr(rs))
        return q, s, rs

    def i2s_mul_mat(self, w_packed, N, K, x, nth=1, want_sidecar=False):
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        x = np.ascontiguousarray(x, dtype=np.float32)
        M = x.shape[0]
        assert x.shape[1] == K
        y = np.zeros((M, N), dtype=np.float32)
        q = np.zeros((M, K), dtype=np.int8) if want_sidecar else None
        s = np.zeros(M, dtype=np.float32) if want_sidecar else None
        rs = np.zeros(M, dtype=np.int32) if want_sidecar else None
        dot = np.zeros((M, N), dtype=np.int32) if want_sidecar else None
        self._L.orc_i2s_mul_mat(_ptr(w_packed), N, K, _ptr(x), M, _ptr(y), int(nth),
                                _ptr(q), _ptr(s), _ptr(rs), _ptr(dot))
        if want_sidecar:
            return y, q, s, rs, dot
        return y

    # -- I8_S -----------------------------------------------------------------
    def i8s_pack(self, q: np.ndarray, scale: float) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.int8).reshape(-1)
        dst = np.zeros(self.i8s_nbytes(q.size), dtype=np.uint8)
        self._L.orc_i8s_pack(_ptr(q), q.size, float(scale), _ptr(dst))
        return dst

    def i8s_unpack(self, packed, n):
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        q = np.zeros(n, dtype=np.int8)
        s = self._L.orc_i8s_unpack(_ptr(packed), n, _ptr(q))
        return q, float(s)

    def i8s_dequantize(self, packed, n):
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        out = np.zeros(n, dtype=np.float32)
        self._L.orc_i8s_dequantize(_ptr(packed), n, _ptr(out))
        return out

    def i8s_quantize(self, y: np.ndarray) -> np.ndarray:
        y = np.ascontiguousarray(y, dtype=np.float32).reshape(-1)
        dst = np.zeros(self.i8s_nbytes(y.size), dtype=np.uint8)
        self._L.orc_i8s_quantize(_ptr(y), y.size, _ptr(dst))
        return dst

    def i8s_mul_mat_add(self, w_packed, N, K, x_packed, M, bias=None, relu=False, nth=1):
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        x_packed = np.ascontiguousarray(x_packed, dtype=np.uint8)
        if bias is not None:
            bias = np.ascontiguousarray(bias, dtype=np.float32)
        y8 = np.zeros(self.i8s_nbytes(M * N), dtype=np.uint8)
        yf = np.zeros((M, N), dtype=np.float32)
        self._L.orc_i8s_mul_mat_add(_ptr(w_packed), N, K, _ptr(x_packed), M, _ptr(bias),
                                    1 if relu else 0, _ptr(y8), _ptr(yf), int(nth))
        return y8, yf

    def i8s_permute_cont(self, packed, a, b):
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        dst = np.zeros(self.i8s_nbytes(a * b), dtype=np.uint8)
        self._L.orc_i8s_permute_cont(_ptr(packed), a, b, _ptr(dst))
        return dst

    # -- I8_S element-wise and conv pieces ---------------------------------
    def i8s_add_scaled(self, a_packed, b_packed, n):
        a_packed = np.ascontiguousarray(a_packed, dtype=np.uint8)
        b_packed = np.ascontiguousarray(b_packed, dtype=np.uint8)
        y8 = np.zeros(self.i8s_nbytes(n), dtype=np.uint8)
        yf = np.zeros(n, dtype=np.float32)
        self._L.orc_i8s_add_scaled(_ptr(a_packed), _ptr(b_packed), n, _ptr(y8), _ptr(yf))
        return y8, yf

    def i8s_rms_norm_scaled(self, x_packed, rows, ne0, eps=1e-5, gamma=None):
        x_packed = np.ascontiguousarray(x_packed, dtype=np.uint8)
        if gamma is not None:
            gamma = np.ascontiguousarray(gamma, dtype=np.float32)
        y8 = np.zeros(self.i8s_nbytes(rows * ne0), dtype=np.uint8)
        yf = np.zeros((rows, ne0), dtype=np.float32)
        self._L.orc_i8s_rms_norm_scaled(_ptr(x_packed), rows, ne0, float(eps), _ptr(gamma), _ptr(y8), _ptr(yf))
        return y8, yf

    def im2col_out_len(self, L, KW, stride, pad_l, pad_r):
        return int(self._L.orc_im2col_out_len(L, KW, stride, pad_l, pad_r))

    def i8s_im2col_asym(self, x_packed, C, L, KW, stride, pad_l, pad_r):
        x_packed = np.ascontiguousarray(x_packed, dtype=np.uint8)
        OL = self.im2col_out_len(L, KW, stride, pad_l, pad_r)
        dst = np.zeros(self.i8s_nbytes(OL * C * KW), dtype=np.uint8)
        self._L.orc_i8s_im2col_asym(_ptr(x_packed), C, L, KW, stride, pad_l, pad_r, _ptr(dst))
        return dst, OL

    def i8s_depthwise_mul_mat_add(self, w_packed, KW, x_packed, C, L, stride, pad_l, pad_r, bias=None,
                                  relu=False):
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        x_packed = np.ascontiguousarray(x_packed, dtype=np.uint8)
        if bias is not None:
            bias = np.ascontiguousarray(bias, dtype=np.float32)
        OL = self.im2col_out_len(L, KW, stride, pad_l, pad_r)
        y8 = np.zeros(self.i8s_nbytes(C * OL), dtype=np.uint8)
        yf = np.zeros((C, OL), dtype=np.float32)
        self._L.orc_i8s_depthwise_mul_mat_add(_ptr(w_packed), KW, _ptr(x_packed), C, L, stride, pad_l, pad_r,
                                              _ptr(bias), 1 if relu else 0, _ptr(y8), _ptr(yf))
        return y8, yf

    # -- W8A8 per-channel ---------------------------------------------------
    def w8a8_quantize_weights(self, w):
        w = np.ascontiguousarray(w, dtype=np.float32)
        N, K = w.shape
        wq = np.zeros((N, K), dtype=np.int8)
        bs = np.zeros(N, dtype=np.float32)
        self._L.orc_w8a8_quantize_weights(_ptr(w), N, K, _ptr(wq), _ptr(bs))
        return wq, bs

    def w8a8_quantize_rows(self, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        M, K = x.shape
        q = np.zeros((M, K), dtype=np.int8)
        s = np.zeros(M, dtype=np.float32)
        self._L.orc_w8a8_quantize_rows(_ptr(x), M, K, _ptr(q), _ptr(s))
        return q, s

    def w8a8_mul_mat(self, wq, bscale, x, nth=1, want_sidecar=False):
        wq = np.ascontiguousarray(wq, dtype=np.int8)
        bscale = np.ascontiguousarray(bscale, dtype=np.float32)
        x = np.ascontiguousarray(x, dtype=np.float32)
        N, K = wq.shape
        M = x.shape[0]
        d = np.zeros((M, N), dtype=np.float32)
        q = np.zeros((M, K), dtype=np.int8) if want_sidecar else None
        s = np.zeros(M, dtype=np.float32) if want_sidecar else None
        self._L.orc_w8a8_mul_mat(_ptr(wq), _ptr(bscale), N, K, _ptr(x), M, _ptr(d), int(nth), _ptr(q), _ptr(s))
        if want_sidecar:
            return d, q, s
        return d


_default: Oracle | None = None


def get() -> Oracle:
    """The shipped oracle build (compiled on first use if missing or stale)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
