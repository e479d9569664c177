"""The device-timeout path, exercised without a fault or a hang.

Every wait in the tensor-core kernels is bounded; when one runs out the kernel
records a timeout in the workspace's status word, sets its abort flag so that
every role leaves its loop, drains the copies and MMAs it has in flight,
frees its tensor memory and returns. Here the GEMV's epilogue is made to wait
on a barrier that nothing signals (i2s_config.test_stall_cycles, about a
millisecond), so the launch takes exactly that path with MMAs and copies in
flight. The host then reads I2S_E_DEVICE_TIMEOUT from i2s_read_status, and the
next normal call on the same workspace must match the CPU oracle bit for bit.
"""

import ctypes

import numpy as np
import pytest

import oracle
from int8_quantized_matmul_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

I2S_E_DEVICE_TIMEOUT = -6


@pytest.fixture(scope="module")
def i2s():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_quantized_matmul_gb300 import build as libbuild
    libbuild.build()
    from int8_quantized_matmul_gb300 import i2s as mod
    assert mod.device_supported() == 1, "the library needs an sm_103 device"
    return mod


def bits(t):
    torch.cuda.synchronize()
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("M,N,K", [(1, 300, 1536), (8, 900, 4608), (16, 1536, 8960)])
def test_gemv_gives_up_a_wait_then_the_workspace_is_clean(i2s, M, N, K):
    o = oracle.get()
    packed = o.i2s_pack(synth.codes(N, K, seed=M + N), 0.07)
    x = synth.normal_f32((M, K), seed=M + K, outlier_p=0.01)
    want = o.i2s_mul_mat(packed, N, K, x, nth=8).view(np.uint32)
    wd = torch.from_numpy(packed).cuda()
    xd = torch.from_numpy(x).cuda()
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(i2s.i2s_mul_mat_workspace(M, N, K), dtype=torch.uint8, device="cuda")

    def call(stall):
        cfg = i2s.i2s_config(3, 0, stall)
        return i2s.lib.i2s_mul_mat_ex(wd.data_ptr(), N, K, xd.data_ptr(), M, y.data_ptr(), ws.data_ptr(),
                                      ws.numel(), ctypes.byref(cfg), i2s._stream())

    assert call(2_000_000) == 0                       # launched; gives up after ~1 ms
    assert i2s.read_status(ws) == I2S_E_DEVICE_TIMEOUT
    assert i2s.read_status(ws) == 0                   # reading clears the word
    for _ in range(2):                                # the same workspace, normal calls
        assert call(0) == 0
        assert np.array_equal(bits(y), want)
        assert i2s.read_status(ws) == 0
    # the context is still usable by other work
    assert torch.equal(torch.arange(5, device="cuda") * 2, torch.arange(0, 10, 2, device="cuda"))


def test_negative_stall_is_rejected(i2s):
    cfg = i2s.i2s_config(3, 0, -1)
    A = 1 << 20
    ws_need = i2s.i2s_mul_mat_workspace(4, 64, 128)
    rc = i2s.lib.i2s_mul_mat_ex(A, 64, 128, A, 4, A, A, ws_need, ctypes.byref(cfg), None)
    assert rc == -8   # I2S_E_BAD_ARG, before anything is enqueued
