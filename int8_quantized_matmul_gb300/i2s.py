"""Python binding of libi2s.so (include/i2s.h): argument marshalling only.

Every computation runs in the library's CUDA kernels. Torch is used for device
memory and streams: tensors are passed as raw device pointers, and calls are
queued on torch's current CUDA stream. Importing this module fails loudly if
the library has not been built (python -m int8_quantized_matmul_gb300.build).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libi2s.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libi2s.so is not built ({LIB_PATH} missing); run "
                      "`python -m int8_quantized_matmul_gb300.build` first")
_L = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_int = ctypes.c_int
_f32 = ctypes.c_float

MAX_GROUP = 256

STATUS = {0: "I2S_OK", -1: "I2S_E_BAD_SHAPE", -2: "I2S_E_NULL_PTR", -3: "I2S_E_MISALIGNED",
          -4: "I2S_E_WORKSPACE_TOO_SMALL", -5: "I2S_E_CUDA", -6: "I2S_E_DEVICE_TIMEOUT",
          -7: "I2S_E_UNSUPPORTED_DEVICE", -8: "I2S_E_BAD_ARG"}


class i2s_config(ctypes.Structure):
    _fields_ = [("path", _int), ("grid_ctas", _int), ("test_stall_cycles", _i64), ("w_layout", ctypes.c_uint)]


class i2s_problem(ctypes.Structure):
    _fields_ = [("w_i2s", _p), ("N", _i64), ("K", _i64), ("x", _p), ("y", _p), ("w_layout", ctypes.c_uint)]


class w8a8_problem(ctypes.Structure):
    _fields_ = [("packed", _p), ("bscale", _p), ("N", _i64), ("K", _i64), ("x", _p), ("d", _p)]


_SIGS = {
    "i2s_status_string": (ctypes.c_char_p, [_int]),
    "i2s_version": (_int, []),
    "i2s_device_supported": (_int, []),
    "i2s_nbytes": (_sz, [_i64, _i64]),
    "i2s_scale_offset": (_sz, [_i64, _i64]),
    "i2s_tiled_nbytes": (_sz, [_i64, _i64]),
    "i2s_tiled_scale_offset": (_sz, [_i64, _i64]),
    "i2s_tile_weights": (_int, [_p, _i64, _i64, _p, _p]),
    "i8s_nbytes": (_sz, [_i64]),
    "i8s_scale_offset": (_sz, [_i64]),
    "i2s_pack_host": (_int, [_p, _i64, _i64, _f32, _p]),
    "i8s_pack_host": (_int, [_p, _i64, _f32, _p]),
    "i2s_quantize_act": (_int, [_p, _i64, _i64, _p, _p, _p, _p]),
    "i2s_mul_mat_workspace": (_sz, [_i64, _i64, _i64]),
    "i2s_mul_mat": (_int, [_p, _i64, _i64, _p, _i64, _p, _p, _sz, _p]),
    "i2s_mul_mat_ex": (_int, [_p, _i64, _i64, _p, _i64, _p, _p, _sz, ctypes.POINTER(i2s_config), _p]),
    "i2s_mul_mat_noalloc": (_int, [_p, _i64, _i64, _p, _i64, _p, _p]),
    "i2s_noalloc_read_status": (_int, [_p]),
    "i2s_mul_mat_grouped_workspace": (_sz, [ctypes.POINTER(i2s_problem), _int, _i64]),
    "i2s_mul_mat_grouped": (_int, [ctypes.POINTER(i2s_problem), _int, _i64, _p, _sz, _p]),
    "i2s_mul_mat_grouped_quantize": (_int, [ctypes.POINTER(i2s_problem), _int, _i64, _p, _sz, _p]),
    "i2s_mul_mat_grouped_run": (_int, [ctypes.POINTER(i2s_problem), _int, _i64, _p, _sz, _p]),
    "i2s_mul_mat_grouped_host_workspace": (_sz, [ctypes.POINTER(i2s_problem), _int, _i64]),
    "i2s_mul_mat_grouped_host": (_int, [ctypes.POINTER(i2s_problem), _int, _i64, _p, _sz, _p]),
    "i2s_mul_mat_grouped_host_ex": (_int, [ctypes.POINTER(i2s_problem), _int, _i64, _p, _sz, ctypes.c_uint, _p]),
    "i2s_mul_mat_grouped_fused_workspace": (_sz, [ctypes.POINTER(i2s_problem), _int, _i64]),
    "i2s_mul_mat_grouped_fused_init": (_int, [_p, _sz, _p]),
    "i2s_mul_mat_grouped_fused": (_int, [ctypes.POINTER(i2s_problem), _int, _i64, _p, _sz, _p]),
    "i8s_mul_mat_workspace": (_sz, [_i64, _i64, _i64]),
    "i8s_ws_f32_offset": (_sz, []),
    "i8s_mul_mat_add_relu": (_int, [_p, _i64, _i64, _p, _i64, _p, _int, _p, _p, _sz, _p]),
    "i8s_requant_workspace": (_sz, [_i64]),
    "i8s_requant": (_int, [_p, _i64, _p, _p, _sz, _p]),
    "i2s_read_status": (_int, [_p, _p]),
    "i8s_packed_bytes": (_sz, [_i64, _i64]),
    "i8s_pack_weights": (_int, [_p, _i64, _i64, _p, _p]),
    "i8s_mul_mat_packed_workspace": (_sz, [_i64, _i64, _i64]),
    "i8s_mul_mat_add_relu_packed": (_int, [_p, _i64, _i64, _p, _i64, _p, _int, _p, _p, _sz, _p]),
    "i8s_eltwise_workspace": (_sz, [_i64]),
    "i8s_add_scaled": (_int, [_p, _p, _i64, _p, _p, _sz, _p]),
    "i8s_rms_norm_scaled": (_int, [_p, _i64, _i64, _f32, _p, _p, _p, _sz, _p]),
    "i8s_transpose": (_int, [_p, _i64, _i64, _p, _p]),
    "i8s_im2col_out_len": (_i64, [_i64, _i64, _i64, _i64, _i64]),
    "i8s_im2col_asym": (_int, [_p, _i64, _i64, _i64, _i64, _i64, _i64, _p, _p]),
    "i8s_depthwise_mul_mat_add": (_int, [_p, _i64, _p, _i64, _i64, _i64, _i64, _i64, _p, _int, _p, _p, _sz, _p]),
    "w8a8_quantize_weights": (_int, [_p, _i64, _i64, _p, _p, _p]),
    "w8a8_mul_mat_workspace": (_sz, [_i64, _i64, _i64]),
    "w8a8_mul_mat": (_int, [_p, _p, _i64, _i64, _p, _i64, _p, _p, _sz, _p]),
    "w8a8_packed_bytes": (_sz, [_i64, _i64]),
    "w8a8_pack_weights": (_int, [_p, _i64, _i64, _p, _p]),
    "w8a8_mul_mat_packed_workspace": (_sz, [_i64, _i64, _i64]),
    "w8a8_mul_mat_packed": (_int, [_p, _p, _i64, _i64, _p, _i64, _p, _p, _sz, _p]),
    "w8a8_mul_mat_grouped_workspace": (_sz, [ctypes.POINTER(w8a8_problem), _int, _i64]),
    "w8a8_mul_mat_grouped": (_int, [ctypes.POINTER(w8a8_problem), _int, _i64, _p, _sz, _p]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_L, _name)
    _fn.restype = _res
    _fn.argtypes = _args

lib = _L


class I2SError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} ({STATUS.get(status, status)})")


def status_string(status: int) -> str:
    return _L.i2s_status_string(int(status)).decode()


def _check(fn: str, rc: int):
    if rc != 0:
        raise I2SError(fn, rc)


def _torch():
    import torch
    return torch


def _stream():
    return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)


def _dptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _ws(nbytes: int, device):
    return _torch().empty(max(int(nbytes), 256), dtype=_torch().uint8, device=device)


# -- layouts and host packers -------------------------------------------------

def i2s_nbytes(N: int, K: int) -> int:
    return int(_L.i2s_nbytes(N, K))


def i2s_scale_offset(N: int, K: int) -> int:
    return int(_L.i2s_scale_offset(N, K))


def i8s_nbytes(n: int) -> int:
    return int(_L.i8s_nbytes(n))


def i8s_scale_offset(n: int) -> int:
    return int(_L.i8s_scale_offset(n))


def i2s_pack_host(codes: np.ndarray, w_scale: float) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = codes.shape
    out = np.zeros(i2s_nbytes(N, K) or 1, dtype=np.uint8)
    _check("i2s_pack_host", _L.i2s_pack_host(codes.ctypes.data, N, K, float(w_scale), out.ctypes.data))
    return out


def i8s_pack_host(q: np.ndarray, scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8).reshape(-1)
    out = np.zeros(i8s_nbytes(q.size), dtype=np.uint8)
    _check("i8s_pack_host", _L.i8s_pack_host(q.ctypes.data, q.size, float(scale), out.ctypes.data))
    return out


# -- device entry points --------------------------------------------------------

def i2s_quantize_act(x):
    """Per-row quantization of an M x K F32 CUDA tensor -> (q int8, scale, row_sum)."""
    torch = _torch()
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    s = torch.empty(M, dtype=torch.float32, device=x.device)
    rs = torch.empty(M, dtype=torch.int32, device=x.device)
    _check("i2s_quantize_act", _L.i2s_quantize_act(_dptr(x), M, K, _dptr(q), _dptr(s), _dptr(rs), _stream()))
    return q, s, rs


def i2s_mul_mat_workspace(M: int, N: int, K: int) -> int:
    return int(_L.i2s_mul_mat_workspace(M, N, K))


def i2s_mul_mat(w, N: int, K: int, x, y=None, ws=None, path: int = 0, grid_ctas: int = 0):
    """y (M x N F32) = I2_S weights w (N x K, device bytes, or their Tiled
    layout) times x (M x K F32). path / grid_ctas: the i2s_config overrides
    (0 = automatic)."""
    torch = _torch()
    wp, layout = _weight(w)
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = _ws(i2s_mul_mat_workspace(M, N, K), x.device)
    if path or grid_ctas or layout:
        cfg = i2s_config(path, grid_ctas, 0, layout)
        rc = _L.i2s_mul_mat_ex(wp, N, K, _dptr(x), M, _dptr(y), _dptr(ws), ws.numel(), ctypes.byref(cfg), _stream())
    else:
        rc = _L.i2s_mul_mat(wp, N, K, _dptr(x), M, _dptr(y), _dptr(ws), ws.numel(), _stream())
    _check("i2s_mul_mat", rc)
    return y


NOALLOC_SCRATCH_BYTES = 4194304   # I2S_NOALLOC_SCRATCH_BYTES


def i2s_mul_mat_noalloc(w, N: int, K: int, x, y):
    """y (M x N F32, caller-provided) = I2_S w times x, M <= 16, with the
    library's fixed per-device scratch instead of a workspace; nothing is
    allocated. Calls on one device must not overlap on the GPU."""
    M = x.shape[0]
    _check("i2s_mul_mat_noalloc", _L.i2s_mul_mat_noalloc(_dptr(w), N, K, _dptr(x), M, _dptr(y), _stream()))
    return y


LAYOUT_I2S = 0     # I2S_LAYOUT_I2S
LAYOUT_TILED = 1   # I2S_LAYOUT_TILED


class Tiled:
    """I2_S weights in the tiled layout written by i2s_tile_weights: `data` is
    a uint8 device tensor of i2s_tiled_nbytes(N, K) bytes. Give it as the
    weight of a grouped problem, in place of the I2_S bytes."""

    def __init__(self, data, N: int, K: int):
        self.data, self.N, self.K = data, N, K

    @property
    def device(self):
        return self.data.device


def i2s_tiled_nbytes(N: int, K: int) -> int:
    return int(_L.i2s_tiled_nbytes(N, K))


def i2s_tiled_scale_offset(N: int, K: int) -> int:
    return int(_L.i2s_tiled_scale_offset(N, K))


def tile_weights(w, N: int, K: int, out=None) -> Tiled:
    """The tiled layout of I2_S weights w (device), written once."""
    if out is None:
        out = _torch().empty(i2s_tiled_nbytes(N, K), dtype=_torch().uint8, device=w.device)
    _check("i2s_tile_weights", _L.i2s_tile_weights(_dptr(w), N, K, _dptr(out), _stream()))
    return Tiled(out, N, K)


def _weight(w):
    """(device pointer, I2S_LAYOUT_*) of a problem's weights."""
    if isinstance(w, Tiled):
        return _dptr(w.data), LAYOUT_TILED
    return _dptr(w), LAYOUT_I2S


def _problems(problems: Sequence):
    arr = (i2s_problem * len(problems))()
    for i, (w, N, K, x, y) in enumerate(problems):
        wp, layout = _weight(w)
        arr[i] = i2s_problem(wp, N, K, _dptr(x), _dptr(y), layout)
    return arr


def i2s_mul_mat_grouped_workspace(problems: Sequence, M: int) -> int:
    arr = _problems(problems)
    return int(_L.i2s_mul_mat_grouped_workspace(arr, len(problems), M))


def i2s_mul_mat_grouped_fused_workspace(problems: Sequence, M: int) -> int:
    arr = _problems(problems)
    return int(_L.i2s_mul_mat_grouped_fused_workspace(arr, len(problems), M))


def i2s_mul_mat_grouped_fused_init(ws):
    """Zeroes the flag area of a workspace before its first fused call."""
    _check("i2s_mul_mat_grouped_fused_init", _L.i2s_mul_mat_grouped_fused_init(_dptr(ws), ws.numel(), _stream()))
    return ws


def i2s_mul_mat_grouped_fused(problems: Sequence, M: int, ws=None):
    """The grouped decode matmul (M <= 16) as one launch that quantizes its own
    activations; ws must have been initialised (a new ws is)."""
    arr = _problems(problems)
    if ws is None:
        ws = _ws(_L.i2s_mul_mat_grouped_fused_workspace(arr, len(problems), M), problems[0][3].device)
        i2s_mul_mat_grouped_fused_init(ws)
    _check("i2s_mul_mat_grouped_fused",
           _L.i2s_mul_mat_grouped_fused(arr, len(problems), M, _dptr(ws), ws.numel(), _stream()))
    return ws


def i2s_mul_mat_grouped(problems: Sequence, M: int, ws=None):
    """Runs [(w, N, K, x, y), ...] (all with M activation rows) as one group."""
    arr = _problems(problems)
    if ws is None:
        ws = _ws(_L.i2s_mul_mat_grouped_workspace(arr, len(problems), M), problems[0][3].device)
    _check("i2s_mul_mat_grouped", _L.i2s_mul_mat_grouped(arr, len(problems), M, _dptr(ws), ws.numel(), _stream()))
    return ws


class Group:
    """A fixed list of projections [(w, N, K, x, y), ...] sharing M activation
    rows, marshalled once; quantize()/run() are the two phases and __call__
    runs both. The tensors must stay alive as long as the Group is used."""

    def __init__(self, problems: Sequence, M: int, ws=None):
        self.problems = list(problems)
        self.M = int(M)
        self.arr = _problems(self.problems)
        need = int(_L.i2s_mul_mat_grouped_workspace(self.arr, len(self.problems), self.M))
        if need == 0:
            raise I2SError("i2s_mul_mat_grouped_workspace", -1)
        self.ws = ws if ws is not None else _ws(need, self.problems[0][3].device)

    def quantize(self):
        _check("i2s_mul_mat_grouped_quantize",
               _L.i2s_mul_mat_grouped_quantize(self.arr, len(self.problems), self.M, _dptr(self.ws),
                                               self.ws.numel(), _stream()))

    def run(self):
        _check("i2s_mul_mat_grouped_run",
               _L.i2s_mul_mat_grouped_run(self.arr, len(self.problems), self.M, _dptr(self.ws), self.ws.numel(),
                                          _stream()))

    def __call__(self):
        _check("i2s_mul_mat_grouped",
               _L.i2s_mul_mat_grouped(self.arr, len(self.problems), self.M, _dptr(self.ws), self.ws.numel(),
                                      _stream()))


def _hptr(t) -> int:
    if t.is_cuda:
        raise ValueError("expected a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _host_problems(problems: Sequence):
    arr = (i2s_problem * len(problems))()
    for i, (w, N, K, x, y) in enumerate(problems):
        wp, layout = _weight(w)
        arr[i] = i2s_problem(wp, N, K, _hptr(x), _hptr(y), layout)
    return arr


HOST_MAPPED = 1     # I2S_HOST_MAPPED
HOST_MAPPED_Y = 2   # I2S_HOST_MAPPED_Y


class HostGroup:
    """A fixed list of projections [(w, N, K, x, y), ...] whose activations x
    and outputs y are host (CPU, ideally pinned) tensors and whose weights w
    are on the device; each call runs the grouped matmul on torch's current
    stream. By default x is copied up and y back around it
    (i2s_mul_mat_grouped_host); with mapped=True (every x and y in pinned,
    device-mapped memory, as torch's pin_memory() gives) the kernels read x
    and write y over the host link directly (I2S_HOST_MAPPED); with
    mapped="y" x is copied up and the epilogue writes y in place
    (I2S_HOST_MAPPED_Y)."""

    def __init__(self, problems: Sequence, M: int, device=None, ws=None, mapped=False):
        self.problems = list(problems)
        self.M = int(M)
        if mapped not in (False, True, "y"):
            raise ValueError("mapped is False, True or 'y'")
        self.flags = HOST_MAPPED_Y if mapped == "y" else (HOST_MAPPED if mapped else 0)
        self.arr = _host_problems(self.problems)
        need = int(_L.i2s_mul_mat_grouped_host_workspace(self.arr, len(self.problems), self.M))
        if need == 0:
            raise I2SError("i2s_mul_mat_grouped_host_workspace", -1)
        self.ws = ws if ws is not None else _ws(need, device if device is not None else self.problems[0][0].device)

    def __call__(self):
        _check("i2s_mul_mat_grouped_host_ex",
               _L.i2s_mul_mat_grouped_host_ex(self.arr, len(self.problems), self.M, _dptr(self.ws), self.ws.numel(),
                                              self.flags, _stream()))


def i2s_mul_mat_grouped_host(problems: Sequence, M: int, ws=None):
    """One call of HostGroup; returns the workspace (the outputs are valid
    once torch's current stream has finished)."""
    g = HostGroup(problems, M, ws=ws)
    g()
    return g.ws


class FusedGroup:
    """A fixed list of decode projections [(w, N, K, x, y), ...] with M <= 16
    rows, run as one fused launch (the GEMV quantizes its own activations);
    marshalled once, the workspace initialised once."""

    def __init__(self, problems: Sequence, M: int, ws=None):
        self.problems = list(problems)
        self.M = int(M)
        self.arr = _problems(self.problems)
        need = int(_L.i2s_mul_mat_grouped_fused_workspace(self.arr, len(self.problems), self.M))
        if need == 0:
            raise I2SError("i2s_mul_mat_grouped_fused_workspace", -1)
        self.ws = ws if ws is not None else _ws(need, self.problems[0][3].device)
        i2s_mul_mat_grouped_fused_init(self.ws)

    def __call__(self):
        _check("i2s_mul_mat_grouped_fused",
               _L.i2s_mul_mat_grouped_fused(self.arr, len(self.problems), self.M, _dptr(self.ws), self.ws.numel(),
                                            _stream()))


def i8s_mul_mat_workspace(M: int, N: int, K: int) -> int:
    return int(_L.i8s_mul_mat_workspace(M, N, K))


def i8s_ws_f32_offset() -> int:
    return int(_L.i8s_ws_f32_offset())


def i8s_mul_mat_add_relu(w, N: int, K: int, x, M: int, bias=None, relu: bool = False, y=None, ws=None):
    """I8_S y (M x N) = requant(W x^T + bias, ReLU optional); returns (y, ws)."""
    torch = _torch()
    if y is None:
        y = torch.empty(i8s_nbytes(M * N), dtype=torch.uint8, device=x.device)
    if ws is None:
        ws = _ws(i8s_mul_mat_workspace(M, N, K), x.device)
    _check("i8s_mul_mat_add_relu",
           _L.i8s_mul_mat_add_relu(_dptr(w), N, K, _dptr(x), M, _dptr(bias), 1 if relu else 0, _dptr(y), _dptr(ws),
                                   ws.numel(), _stream()))
    return y, ws


def i8s_pack_weights(w, N: int, K: int, packed=None):
    """f16 operand rows of an I8_S weight tensor plus its scale, written once."""
    if packed is None:
        packed = _torch().empty(int(_L.i8s_packed_bytes(N, K)), dtype=_torch().uint8, device=w.device)
    _check("i8s_pack_weights", _L.i8s_pack_weights(_dptr(w), N, K, _dptr(packed), _stream()))
    return packed


def i8s_mul_mat_add_relu_packed(packed, N: int, K: int, x, M: int, bias=None, relu: bool = False, y=None, ws=None):
    """i8s_mul_mat_add_relu over weights packed once by i8s_pack_weights; returns (y, ws)."""
    torch = _torch()
    if y is None:
        y = torch.empty(i8s_nbytes(M * N), dtype=torch.uint8, device=x.device)
    if ws is None:
        ws = _ws(int(_L.i8s_mul_mat_packed_workspace(M, N, K)), x.device)
    _check("i8s_mul_mat_add_relu_packed",
           _L.i8s_mul_mat_add_relu_packed(_dptr(packed), N, K, _dptr(x), M, _dptr(bias), 1 if relu else 0, _dptr(y),
                                          _dptr(ws), ws.numel(), _stream()))
    return y, ws


def i8s_ws_f32(ws, M: int, N: int):
    """View of the F32 output (before requantization) kept in an I8_S workspace."""
    off = i8s_ws_f32_offset()
    return ws[off:off + M * N * 4].view(_torch().float32).view(M, N)


def i8s_requant(y, dst=None, ws=None):
    torch = _torch()
    n = y.numel()
    if dst is None:
        dst = torch.empty(i8s_nbytes(n), dtype=torch.uint8, device=y.device)
    if ws is None:
        ws = _ws(_L.i8s_requant_workspace(n), y.device)
    _check("i8s_requant", _L.i8s_requant(_dptr(y), n, _dptr(dst), _dptr(ws), ws.numel(), _stream()))
    return dst


def i8s_eltwise_workspace(rows: int = 1) -> int:
    return int(_L.i8s_eltwise_workspace(rows))


def _u8(n: int, device):
    return _torch().empty(n, dtype=_torch().uint8, device=device)


def i8s_add_scaled(a, b, n: int, y=None, ws=None):
    """I8_S y = requant(a*a_scale + b*b_scale) over n elements."""
    if y is None:
        y = _u8(i8s_nbytes(n), a.device)
    if ws is None:
        ws = _ws(i8s_eltwise_workspace(1), a.device)
    _check("i8s_add_scaled", _L.i8s_add_scaled(_dptr(a), _dptr(b), n, _dptr(y), _dptr(ws), ws.numel(), _stream()))
    return y


def i8s_rms_norm_scaled(x, rows: int, ne0: int, eps: float = 1e-5, gamma=None, y=None, ws=None):
    """I8_S y = requant(RMSNorm of each of `rows` rows of ne0 values (* gamma))."""
    if y is None:
        y = _u8(i8s_nbytes(rows * ne0), x.device)
    if ws is None:
        ws = _ws(i8s_eltwise_workspace(rows), x.device)
    _check("i8s_rms_norm_scaled", _L.i8s_rms_norm_scaled(_dptr(x), rows, ne0, float(eps), _dptr(gamma), _dptr(y),
                                                         _dptr(ws), ws.numel(), _stream()))
    return y


def i8s_transpose(src, a: int, b: int, dst=None):
    """I8_S a x b -> b x a, the scale carried."""
    if dst is None:
        dst = _u8(i8s_nbytes(a * b), src.device)
    _check("i8s_transpose", _L.i8s_transpose(_dptr(src), a, b, _dptr(dst), _stream()))
    return dst


def i8s_im2col_out_len(L: int, KW: int, stride: int, pad_l: int, pad_r: int) -> int:
    return int(_L.i8s_im2col_out_len(L, KW, stride, pad_l, pad_r))


def i8s_im2col_asym(src, C: int, L: int, KW: int, stride: int, pad_l: int, pad_r: int, dst=None):
    """I8_S C x L -> OL x (C*KW) windows with independent left/right zero padding."""
    OL = i8s_im2col_out_len(L, KW, stride, pad_l, pad_r)
    if dst is None:
        dst = _u8(i8s_nbytes(OL * C * KW), src.device)
    _check("i8s_im2col_asym", _L.i8s_im2col_asym(_dptr(src), C, L, KW, stride, pad_l, pad_r, _dptr(dst), _stream()))
    return dst, OL


def i8s_depthwise_mul_mat_add(w, KW: int, x, C: int, L: int, stride: int, pad_l: int, pad_r: int, bias=None,
                              relu: bool = False, y=None, ws=None):
    """I8_S per-channel conv: y (C x OL) = requant(conv(x, w) * (w_scale*x_scale) + bias, ReLU optional)."""
    OL = i8s_im2col_out_len(L, KW, stride, pad_l, pad_r)
    if y is None:
        y = _u8(i8s_nbytes(C * OL), x.device)
    if ws is None:
        ws = _ws(i8s_eltwise_workspace(1), x.device)
    _check("i8s_depthwise_mul_mat_add",
           _L.i8s_depthwise_mul_mat_add(_dptr(w), KW, _dptr(x), C, L, stride, pad_l, pad_r, _dptr(bias),
                                        1 if relu else 0, _dptr(y), _dptr(ws), ws.numel(), _stream()))
    return y, OL


def w8a8_quantize_weights(w, wq=None, bscale=None):
    """Per-channel int8 weights of an N x K F32 tensor: (wq N x K int8, bscale N F32)."""
    torch = _torch()
    N, K = w.shape
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.int8, device=w.device)
    if bscale is None:
        bscale = torch.empty(N, dtype=torch.float32, device=w.device)
    _check("w8a8_quantize_weights", _L.w8a8_quantize_weights(_dptr(w), N, K, _dptr(wq), _dptr(bscale), _stream()))
    return wq, bscale


def w8a8_mul_mat_workspace(M: int, N: int, K: int) -> int:
    return int(_L.w8a8_mul_mat_workspace(M, N, K))


def w8a8_mul_mat(wq, bscale, x, d=None, ws=None):
    """d (M x N F32) = aScale[m] * bScale[n] * (int32 dot of the per-row int8 activations and wq)."""
    torch = _torch()
    N, K = wq.shape
    M = x.shape[0]
    if d is None:
        d = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = _ws(w8a8_mul_mat_workspace(M, N, K), x.device)
    _check("w8a8_mul_mat", _L.w8a8_mul_mat(_dptr(wq), _dptr(bscale), N, K, _dptr(x), M, _dptr(d), _dptr(ws),
                                           ws.numel(), _stream()))
    return d, ws


def w8a8_pack_weights(wq, packed=None):
    """The f16 operand rows of per-channel int8 weights (N x K), written once."""
    N, K = wq.shape
    if packed is None:
        packed = _u8(int(_L.w8a8_packed_bytes(N, K)), wq.device)
    _check("w8a8_pack_weights", _L.w8a8_pack_weights(_dptr(wq), N, K, _dptr(packed), _stream()))
    return packed


def w8a8_mul_mat_packed_workspace(M: int, N: int, K: int) -> int:
    return int(_L.w8a8_mul_mat_packed_workspace(M, N, K))


def w8a8_mul_mat_packed(packed, bscale, N: int, K: int, x, d=None, ws=None):
    """w8a8_mul_mat over weights packed once by w8a8_pack_weights."""
    torch = _torch()
    M = x.shape[0]
    if d is None:
        d = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = _ws(w8a8_mul_mat_packed_workspace(M, N, K), x.device)
    _check("w8a8_mul_mat_packed", _L.w8a8_mul_mat_packed(_dptr(packed), _dptr(bscale), N, K, _dptr(x), M, _dptr(d),
                                                         _dptr(ws), ws.numel(), _stream()))
    return d, ws


def _w8a8_problems(problems):
    arr = (w8a8_problem * len(problems))()
    for i, (packed, bscale, N, K, x, d) in enumerate(problems):
        arr[i] = w8a8_problem(_dptr(packed), _dptr(bscale), N, K, _dptr(x), _dptr(d))
    return arr


def w8a8_mul_mat_grouped(problems, M: int, ws=None):
    """problems: (packed, bscale, N, K, x, d) tuples with the same M; one
    quantization launch and one GEMM launch for all. Returns ws."""
    arr = _w8a8_problems(problems)
    if ws is None:
        ws = _ws(int(_L.w8a8_mul_mat_grouped_workspace(arr, len(problems), M)), problems[0][4].device)
    _check("w8a8_mul_mat_grouped", _L.w8a8_mul_mat_grouped(arr, len(problems), M, _dptr(ws), ws.numel(), _stream()))
    return ws


class W8A8Group:
    """A fixed list of packed W8A8 matmuls (same M) with its workspace, for
    repeated calls (and CUDA graph capture)."""

    def __init__(self, problems, M: int, ws=None):
        self.problems = list(problems)
        self.M = M
        self._arr = _w8a8_problems(self.problems)
        need = int(_L.w8a8_mul_mat_grouped_workspace(self._arr, len(self.problems), M))
        if need == 0:
            raise I2SError("w8a8_mul_mat_grouped_workspace", -1)
        self.ws = ws if ws is not None else _ws(need, self.problems[0][4].device)

    def __call__(self):
        _check("w8a8_mul_mat_grouped", _L.w8a8_mul_mat_grouped(self._arr, len(self.problems), self.M,
                                                               _dptr(self.ws), self.ws.numel(), _stream()))


def read_status(ws) -> int:
    return int(_L.i2s_read_status(_dptr(ws), _stream()))


def noalloc_read_status() -> int:
    return int(_L.i2s_noalloc_read_status(_stream()))


def device_supported() -> int:
    return int(_L.i2s_device_supported())
