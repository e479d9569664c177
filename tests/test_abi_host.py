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
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*\b((?:i2s|i8s)_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_north_star_calls():
    names = header_functions()
    for must in ("i2s_quantize_act", "i2s_mul_mat", "i8s_mul_mat_add_relu", "i8s_requant"):
        assert must in names


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
    assert L.i8s_mul_mat_add_relu(FAKE, 64, 100, FAKE, 4, None, 0, FAKE, FAKE, ws_big, None) == -1
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
