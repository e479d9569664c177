"""The C-ABI library on the host (no GPU): exports, layouts, packers, validation.

Nothing here launches a kernel. Validation errors are returned before any CUDA
call, so they are exercised with dummy (never dereferenced) pointers.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from int8_quantized_matmul_gb300 import build as libbuild
from int8_quantized_matmul_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "i2s.h")


@pytest.fixture(scope="module")
def i2s():
    libbuild.build()
    from int8_quantized_matmul_gb300 import i2s as mod
    return mod


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*\b((?:i2s|i8s|w8a8)_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_core_calls():
    names = header_functions()
    for must in ("i2s_quantize_act", "i2s_mul_mat", "i8s_mul_mat_add_relu", "i8s_requant"):
        assert must in names
    # the rows past the core: element-wise and conv ops, packed and grouped calls, W8A8
    for must in ("i8s_add_scaled", "i8s_rms_norm_scaled", "i8s_transpose", "i8s_im2col_asym",
                 "i8s_depthwise_mul_mat_add", "i8s_pack_weights", "i8s_mul_mat_add_relu_packed",
                 "w8a8_quantize_weights", "w8a8_mul_mat", "w8a8_pack_weights", "w8a8_mul_mat_packed",
                 "w8a8_mul_mat_grouped"):
        assert must in names, must


def test_library_exports_every_declared_symbol(i2s):
    lib = ctypes.CDLL(i2s.LIB_PATH)
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_layout_helpers_match_oracle(i2s):
    o = oracle.get()
    for N, K in ((1, 128), (70, 1152), (1536, 8960), (151936, 1536)):
        assert i2s.i2s_nbytes(N, K) == o.i2s_nbytes(N, K)
        assert i2s.i2s_scale_offset(N, K) == o.i2s_scale_offset(N, K)
    for n in (1, 31, 32, 33, 900 * 8192 + 5):
        assert i2s.i8s_nbytes(n) == o.i8s_nbytes(n)
        assert i2s.i8s_scale_offset(n) == o.i8s_scale_offset(n)
    assert i2s.i2s_nbytes(4, 100) == 0 and i2s.i8s_nbytes(0) == 0


@pytest.mark.parametrize("N,K", [(1, 128), (70, 1152), (256, 1024), (3, 8960)])
def test_i2s_pack_host_matches_oracle_packer(i2s, N, K):
    c = synth.codes(N, K, seed=N + K)
    assert np.array_equal(i2s.i2s_pack_host(c, 0.0625), oracle.get().i2s_pack(c, 0.0625))


def test_i8s_pack_host_matches_oracle_packer(i2s):
    for n in (1, 33, 1000):
        q = synth.int8_normal(n, seed=n)
        assert np.array_equal(i2s.i8s_pack_host(q, 0.01), oracle.get().i8s_pack(q, 0.01))


def test_status_strings(i2s):
    for code in i2s.STATUS:
        assert i2s.status_string(code)
    assert i2s.status_string(-99) == "unknown status"


FAKE = 0x10000   # 64 KiB-aligned dummy address, never dereferenced


def test_validation_errors_need_no_device(i2s):
    L = i2s.lib
    ws_big = 1 << 30
    # K not a multiple of 128
    assert L.i2s_mul_mat(FAKE, 64, 100, FAKE, 4, FAKE, FAKE, ws_big, None) == -1
    # non-positive sizes
    assert L.i2s_mul_mat(FAKE, 0, 128, FAKE, 4, FAKE, FAKE, ws_big, None) == -1
    assert L.i2s_mul_mat(FAKE, 64, 128, FAKE, 0, FAKE, FAKE, ws_big, None) == -1
    # null pointers
    assert L.i2s_mul_mat(None, 64, 128, FAKE, 4, FAKE, FAKE, ws_big, None) == -2
    assert L.i2s_mul_mat(FAKE, 64, 128, FAKE, 4, FAKE, None, ws_big, None) == -2
    # misaligned
    assert L.i2s_mul_mat(FAKE + 4, 64, 128, FAKE, 4, FAKE, FAKE, ws_big, None) == -3
    assert L.i2s_mul_mat(FAKE, 64, 128, FAKE, 4, FAKE, FAKE + 16, ws_big, None) == -3
    # workspace too small
    need = i2s.i2s_mul_mat_workspace(4, 64, 128)
    assert need > 0
    assert L.i2s_mul_mat(FAKE, 64, 128, FAKE, 4, FAKE, FAKE, need - 1, None) == -4
    # I8_S
    assert L.i8s_mul_mat_add_relu(FAKE, 64, 0, FAKE, 4, None, 0, FAKE, FAKE, ws_big, None) == -1
    assert L.i8s_mul_mat_add_relu(FAKE, 64, 65537, FAKE, 4, None, 0, FAKE, FAKE, ws_big, None) == -1
    # any K >= 1 is a valid shape (rows padded to 64 positions inside)
    assert i2s.i8s_mul_mat_workspace(4, 64, 7) == i2s.i8s_mul_mat_workspace(4, 64, 64)
    assert L.i8s_mul_mat_add_relu(FAKE, 64, 128, FAKE, 4, None, 0, None, FAKE, ws_big, None) == -2
    need = i2s.i8s_mul_mat_workspace(4, 64, 128)
    assert L.i8s_mul_mat_add_relu(FAKE, 64, 128, FAKE, 4, None, 0, FAKE, FAKE, need - 1, None) == -4
    assert L.i8s_requant(FAKE, 0, FAKE, FAKE, ws_big, None) == -1
    assert L.i8s_requant(FAKE + 8, 10, FAKE, FAKE, ws_big, None) == -3
    assert L.i2s_quantize_act(FAKE, 4, 6, FAKE, FAKE, FAKE, None) == -1
    # grouped: count out of range
    arr = (i2s.i2s_problem * 1)()
    assert L.i2s_mul_mat_grouped(arr, 0, 1, FAKE, ws_big, None) == -8
    assert L.i2s_mul_mat_grouped(arr, 1, 1, FAKE, ws_big, None) == -2


def test_workspace_sizes_monotone(i2s):
    a = i2s.i2s_mul_mat_workspace(1, 1536, 1536)
    b = i2s.i2s_mul_mat_workspace(8, 1536, 1536)
    c = i2s.i2s_mul_mat_workspace(512, 1536, 8960)
    assert 0 < a < b < c
    assert i2s.i2s_mul_mat_workspace(4, 10, 100) == 0


def test_eltwise_and_w8a8_validation_needs_no_device(i2s):
    L = i2s.lib
    A = 1 << 20
    vp = ctypes.c_void_p
    E = {v: k for k, v in i2s.STATUS.items()}
    # element-wise: null, shape, alignment and overlap checks
    assert L.i8s_add_scaled(None, vp(A), 100, vp(2 * A), vp(3 * A), 256, None) == E["I2S_E_NULL_PTR"]
    assert L.i8s_add_scaled(vp(A), vp(2 * A), 0, vp(3 * A), vp(4 * A), 256, None) == E["I2S_E_BAD_SHAPE"]
    assert L.i8s_add_scaled(vp(A + 4), vp(2 * A), 100, vp(3 * A), vp(4 * A), 256, None) == E["I2S_E_MISALIGNED"]
    assert L.i8s_add_scaled(vp(A), vp(2 * A), 100, vp(A + 16), vp(4 * A), 256, None) == E["I2S_E_BAD_ARG"]
    assert L.i8s_add_scaled(vp(A), vp(2 * A), 100, vp(3 * A), vp(4 * A), 16, None) == E["I2S_E_WORKSPACE_TOO_SMALL"]
    assert L.i8s_rms_norm_scaled(vp(A), 4, 0, 1e-5, None, vp(2 * A), vp(3 * A), 4096, None) == E["I2S_E_BAD_SHAPE"]
    assert L.i8s_rms_norm_scaled(vp(A), 4, 200000, 1e-5, None, vp(2 * A), vp(3 * A), 4096, None) == E["I2S_E_BAD_SHAPE"]
    assert L.i8s_rms_norm_scaled(vp(A), 4, 32, -1.0, None, vp(2 * A), vp(3 * A), 4096, None) == E["I2S_E_BAD_SHAPE"]
    assert L.i8s_rms_norm_scaled(vp(A), 4, 32, 1e-5, vp(5), vp(2 * A), vp(3 * A), 4096, None) == E["I2S_E_MISALIGNED"]
    assert L.i8s_rms_norm_scaled(vp(A), 1000, 32, 1e-5, None, vp(2 * A), vp(3 * A), 256, None) == \
        E["I2S_E_WORKSPACE_TOO_SMALL"]
    assert L.i8s_transpose(vp(A), 0, 5, vp(2 * A), None) == E["I2S_E_BAD_SHAPE"]
    assert L.i8s_transpose(vp(A), 64, 64, vp(A + 64), None) == E["I2S_E_BAD_ARG"]
    # conv geometry
    assert i2s.i8s_im2col_out_len(20, 4, 1, 3, 0) == 20
    assert i2s.i8s_im2col_out_len(5, 7, 1, 0, 0) == 0
    assert i2s.i8s_im2col_out_len(40, 8, 4, 4, 0) == 10
    assert L.i8s_im2col_asym(vp(A), 2, 5, 7, 1, 0, 0, vp(2 * A), None) == E["I2S_E_BAD_SHAPE"]
    assert L.i8s_im2col_asym(vp(A), 2, 40, 8, 0, 4, 0, vp(2 * A), None) == E["I2S_E_BAD_SHAPE"]
    assert L.i8s_im2col_asym(vp(A), 2, 40, 8, 4, 4, 0, vp(2 * A + 3), None) == E["I2S_E_MISALIGNED"]
    assert L.i8s_depthwise_mul_mat_add(vp(A), 7, vp(2 * A), 4, 100, 1, 6, 0, None, 0, vp(2 * A + 16), vp(4 * A), 256,
                                       None) == E["I2S_E_BAD_ARG"]
    # W8A8: shapes (any K from 1 to 65536), alignment, group size
    assert L.w8a8_mul_mat(vp(A), vp(2 * A), 64, 0, vp(3 * A), 8, vp(4 * A), vp(5 * A), 1 << 30, None) == \
        E["I2S_E_BAD_SHAPE"]
    assert L.w8a8_mul_mat(vp(A), vp(2 * A), 64, 65537, vp(3 * A), 8, vp(4 * A), vp(5 * A), 1 << 30, None) == \
        E["I2S_E_BAD_SHAPE"]
    assert L.w8a8_mul_mat(vp(A + 8), vp(2 * A), 64, 128, vp(3 * A), 8, vp(4 * A), vp(5 * A), 1 << 30, None) == \
        E["I2S_E_MISALIGNED"]
    assert L.w8a8_packed_bytes(64, 128) == 64 * 128 * 2 and L.w8a8_packed_bytes(64, 100) == 64 * 128 * 2
    assert L.w8a8_packed_bytes(64, 0) == 0
    assert L.i8s_packed_bytes(64, 128) == 64 * 128 * 2 + 16 and L.i8s_packed_bytes(64, 7) == 64 * 64 * 2 + 16
    probs = (i2s.w8a8_problem * 9)()
    for i in range(9):
        probs[i] = i2s.w8a8_problem(A, A, 64, 128, A, A)
    assert L.w8a8_mul_mat_grouped(probs, 9, 8, vp(2 * A), 1 << 30, None) == E["I2S_E_BAD_ARG"]
    assert L.w8a8_mul_mat_grouped(probs, 0, 8, vp(2 * A), 1 << 30, None) == E["I2S_E_BAD_ARG"]
    assert L.w8a8_mul_mat_grouped_workspace(probs, 9, 8) == 0
    # a group's workspace: q, k, v share one activation (quantized once)
    shared = (i2s.w8a8_problem * 3)()
    for i in range(3):
        shared[i] = i2s.w8a8_problem(A, A, 64, 128, A, A)
    distinct = (i2s.w8a8_problem * 3)()
    for i in range(3):
        distinct[i] = i2s.w8a8_problem(A, A, 64, 128, A + 4096 * i, A)
    assert L.w8a8_mul_mat_grouped_workspace(distinct, 3, 8) > L.w8a8_mul_mat_grouped_workspace(shared, 3, 8) > 0


def test_fused_decode_validation_needs_no_device(i2s):
    L = i2s.lib
    A = 1 << 20
    vp = ctypes.c_void_p
    E = {v: k for k, v in i2s.STATUS.items()}
    probs = (i2s.i2s_problem * 2)()
    probs[0] = i2s.i2s_problem(A, 64, 1536, 2 * A, 3 * A)
    probs[1] = i2s.i2s_problem(A, 300, 1536, 2 * A, 4 * A)   # shares the activation
    ws1 = L.i2s_mul_mat_grouped_fused_workspace(probs, 2, 1)
    ws16 = L.i2s_mul_mat_grouped_fused_workspace(probs, 2, 16)
    assert 0 < ws1 < ws16
    assert L.i2s_mul_mat_grouped_fused_workspace(probs, 2, 17) == 0      # M <= 16 only
    assert L.i2s_mul_mat_grouped_fused(probs, 2, 17, vp(8 * A), 1 << 30, None) == E["I2S_E_BAD_SHAPE"]
    assert L.i2s_mul_mat_grouped_fused(probs, 0, 1, vp(8 * A), 1 << 30, None) == E["I2S_E_BAD_ARG"]
    assert L.i2s_mul_mat_grouped_fused(probs, 2, 1, vp(8 * A + 16), 1 << 30, None) == E["I2S_E_MISALIGNED"]
    assert L.i2s_mul_mat_grouped_fused(probs, 2, 1, vp(8 * A), ws1 - 1, None) == E["I2S_E_WORKSPACE_TOO_SMALL"]
    assert L.i2s_mul_mat_grouped_fused_init(None, 4096, None) == E["I2S_E_NULL_PTR"]
    assert L.i2s_mul_mat_grouped_fused_init(vp(8 * A + 16), 4096, None) == E["I2S_E_MISALIGNED"]
    assert L.i2s_mul_mat_grouped_fused_init(vp(8 * A), 1024, None) == E["I2S_E_WORKSPACE_TOO_SMALL"]
    # nine distinct K values are more than one launch's operand maps hold
    nine = (i2s.i2s_problem * 9)()
    for i in range(9):
        nine[i] = i2s.i2s_problem(A, 64, 128 * (i + 1), 2 * A + 65536 * i, 3 * A)
    assert L.i2s_mul_mat_grouped_fused_workspace(nine, 8, 4) > 0
    assert L.i2s_mul_mat_grouped_fused_workspace(nine, 9, 4) == 0
    assert L.i2s_mul_mat_grouped_fused(nine, 9, 4, vp(8 * A), 1 << 30, None) == E["I2S_E_BAD_ARG"]


def test_host_buffer_call_validation_and_copy_plan(i2s):
    # i2s_mul_mat_grouped_host: activations and outputs on the host. The
    # workspace is the grouped one followed by one device copy per merged host
    # range, so slices of one buffer cost one range each way.
    L = i2s.lib
    A = 1 << 20
    vp = ctypes.c_void_p
    E = {v: k for k, v in i2s.STATUS.items()}
    M, K = 4, 1536
    xb, yb = 64 * A, 96 * A                     # host addresses (never dereferenced)

    def problems(xs, ys, Ns):
        arr = (i2s.i2s_problem * len(xs))()
        for i, (x, y, N) in enumerate(zip(xs, ys, Ns)):
            arr[i] = i2s.i2s_problem(A, N, K, x, y)
        return arr

    def up(v):
        return (v + 255) // 256 * 256
    Ns = [64, 320, 256]
    # x: one activation shared by the first two, the third right after it;
    # y: three outputs back to back
    xs = [xb, xb, xb + M * K * 4]
    ys = [yb, yb + M * 64 * 4, yb + M * (64 + 320) * 4]
    merged = problems(xs, ys, Ns)
    grouped = L.i2s_mul_mat_grouped_workspace(merged, 3, M)
    assert grouped > 0
    assert L.i2s_mul_mat_grouped_host_workspace(merged, 3, M) == grouped + up(2 * M * K * 4) + up(M * 640 * 4)
    # the same problems with gaps between the host buffers: one range each
    apart = problems([xb, xb, xb + 2 * A], [yb, yb + A, yb + 2 * A], Ns)
    assert L.i2s_mul_mat_grouped_host_workspace(apart, 3, M) == (
        grouped + 2 * up(M * K * 4) + sum(up(M * n * 4) for n in Ns))
    need = L.i2s_mul_mat_grouped_host_workspace(merged, 3, M)
    ws = vp(8 * A)
    assert L.i2s_mul_mat_grouped_host(merged, 3, M, ws, need - 1, None) == E["I2S_E_WORKSPACE_TOO_SMALL"]
    assert L.i2s_mul_mat_grouped_host(merged, 3, M, vp(8 * A + 16), need, None) == E["I2S_E_MISALIGNED"]
    assert L.i2s_mul_mat_grouped_host(merged, 3, M, None, need, None) == E["I2S_E_NULL_PTR"]
    assert L.i2s_mul_mat_grouped_host(merged, 0, M, ws, need, None) == E["I2S_E_BAD_ARG"]
    # overlapping outputs, and an output over an activation, are rejected
    clash = problems(xs, [yb, yb + 16, yb + A], Ns)
    assert L.i2s_mul_mat_grouped_host_workspace(clash, 3, M) == 0
    assert L.i2s_mul_mat_grouped_host(clash, 3, M, ws, 1 << 30, None) == E["I2S_E_BAD_ARG"]
    onto = problems(xs, [yb, yb + A, xb + 64], Ns)
    assert L.i2s_mul_mat_grouped_host(onto, 3, M, ws, 1 << 30, None) == E["I2S_E_BAD_ARG"]
    odd = problems([xb + 8, xb, xb], ys, Ns)
    assert L.i2s_mul_mat_grouped_host(odd, 3, M, ws, 1 << 30, None) == E["I2S_E_MISALIGNED"]
    bad_k = problems(xs, ys, Ns)
    bad_k[1].K = 100
    assert L.i2s_mul_mat_grouped_host(bad_k, 3, M, ws, 1 << 30, None) == E["I2S_E_BAD_SHAPE"]
    # flags: I2S_HOST_MAPPED (1) and I2S_HOST_MAPPED_Y (2) are defined
    assert L.i2s_mul_mat_grouped_host_ex(merged, 3, M, ws, need, 4, None) == E["I2S_E_BAD_ARG"]
    assert L.i2s_mul_mat_grouped_host_ex(merged, 3, M, ws, need, 8, None) == E["I2S_E_BAD_ARG"]
    assert L.i2s_mul_mat_grouped_host_ex(clash, 3, M, ws, 1 << 30, 1, None) == E["I2S_E_BAD_ARG"]
    assert L.i2s_mul_mat_grouped_host_ex(clash, 3, M, ws, 1 << 30, 2, None) == E["I2S_E_BAD_ARG"]
    # outputs-only mapping stages the activations: the staged call's workspace
    assert L.i2s_mul_mat_grouped_host_ex(merged, 3, M, ws, need - 1, 2, None) == E["I2S_E_WORKSPACE_TOO_SMALL"]
    # both mapped needs only the grouped workspace
    assert L.i2s_mul_mat_grouped_host_ex(merged, 3, M, ws, grouped - 1, 1, None) == E["I2S_E_WORKSPACE_TOO_SMALL"]
    assert L.i2s_mul_mat_grouped_host_ex(merged, 3, M, ws, grouped - 1, 3, None) == E["I2S_E_WORKSPACE_TOO_SMALL"]


def test_tiled_layout_sizes_and_validation(i2s):
    # sizes against the header's formula; validation before any CUDA call
    from tests import tiled_layout
    L = i2s.lib
    A = 1 << 20
    vp = ctypes.c_void_p
    E = {v: k for k, v in i2s.STATUS.items()}
    for N, K in ((1, 128), (300, 1152), (256, 1536), (257, 1536), (1536, 8960), (151936, 1536)):
        tn, tk = tiled_layout.blocks(N, K)
        assert i2s.i2s_tiled_scale_offset(N, K) == tn * tk * 16384
        assert i2s.i2s_tiled_nbytes(N, K) == tiled_layout.nbytes(N, K) >= i2s.i2s_nbytes(N, K)
    for N, K in ((0, 128), (4, 100), (4, 0)):
        assert i2s.i2s_tiled_nbytes(N, K) == 0 and i2s.i2s_tiled_scale_offset(N, K) == 0
    assert L.i2s_tile_weights(None, 4, 128, vp(8 * A), None) == E["I2S_E_NULL_PTR"]
    assert L.i2s_tile_weights(vp(A), 4, 100, vp(8 * A), None) == E["I2S_E_BAD_SHAPE"]
    assert L.i2s_tile_weights(vp(A + 8), 4, 128, vp(8 * A), None) == E["I2S_E_MISALIGNED"]
    assert L.i2s_tile_weights(vp(A), 4, 128, vp(8 * A + 8), None) == E["I2S_E_MISALIGNED"]
    assert L.i2s_tile_weights(vp(A), 300, 1152, vp(A + 4096), None) == E["I2S_E_BAD_ARG"]   # overlap
    # a w_layout other than I2S_LAYOUT_I2S / I2S_LAYOUT_TILED, in every grouped form
    probs = (i2s.i2s_problem * 2)()
    probs[0] = i2s.i2s_problem(A, 64, 1536, 2 * A, 3 * A, i2s.LAYOUT_TILED)
    probs[1] = i2s.i2s_problem(A, 300, 1536, 2 * A, 4 * A, 2)
    ws = vp(8 * A)
    assert L.i2s_mul_mat_grouped(probs, 2, 4, ws, 1 << 30, None) == E["I2S_E_BAD_ARG"]
    assert L.i2s_mul_mat_grouped(probs, 2, 64, ws, 1 << 30, None) == E["I2S_E_BAD_ARG"]
    assert L.i2s_mul_mat_grouped_fused(probs, 2, 4, ws, 1 << 30, None) == E["I2S_E_BAD_ARG"]
    assert L.i2s_mul_mat_grouped_host(probs, 2, 4, ws, 1 << 30, None) == E["I2S_E_BAD_ARG"]
    assert L.i2s_mul_mat_grouped_workspace(probs, 2, 4) == 0
    probs[1].w_layout = i2s.LAYOUT_TILED
    assert L.i2s_mul_mat_grouped_workspace(probs, 2, 4) > 0


def test_tiled_layout_restatement_by_enumeration():
    # the numpy restatement against the header's sentence, byte by byte, on
    # small shapes with ragged rows and row bytes
    from tests import tiled_layout
    for N, K in ((3, 128), (130, 640), (257, 1152)):
        rb = K // 4
        packed = np.random.default_rng(N + K).integers(0, 256, N * rb + 32, dtype=np.uint8)
        t = tiled_layout.tile(packed, N, K)
        tn, tk = tiled_layout.blocks(N, K)
        assert t.size == tn * tk * 16384 + 32
        want = np.zeros(tn * tk * 16384, np.uint8)
        for n in range(N):
            for b in range(rb):
                i, rr = divmod(n, 128)
                j, cb = divmod(b, 128)
                c, off = divmod(cb, 16)
                want[(i * tk + j) * 16384 + rr * 128 + (c ^ (rr % 8)) * 16 + off] = packed[n * rb + b]
        np.testing.assert_array_equal(t[:-32], want)
        np.testing.assert_array_equal(t[-32:], packed[N * rb:])


def test_single_call_config_validation_needs_no_device(i2s):
    # i2s_mul_mat_ex checks its configuration (path, weight layout, stall) on
    # the host before any CUDA call
    L = i2s.lib
    A = 1 << 20
    E = {v: k for k, v in i2s.STATUS.items()}
    ws_need = i2s.i2s_mul_mat_workspace(4, 64, 128)

    def call(cfg, M=4):
        return L.i2s_mul_mat_ex(A, 64, 128, A, M, A, A, i2s.i2s_mul_mat_workspace(M, 64, 128), ctypes.byref(cfg), None)
    assert call(i2s.i2s_config(1, 0)) == E["I2S_E_BAD_ARG"]                     # no such path
    assert call(i2s.i2s_config(3, 0), M=17) == E["I2S_E_BAD_ARG"]               # the GEMV takes M <= 16
    assert call(i2s.i2s_config(0, 0, -1)) == E["I2S_E_BAD_ARG"]                 # negative stall
    assert call(i2s.i2s_config(0, 0, 0, 2)) == E["I2S_E_BAD_ARG"]               # no such weight layout
    assert ws_need > 0
