"""i2s_mul_mat_grouped_host (activations and outputs in host memory, one call
copying them up and back around the grouped matmul) against the CPU oracle,
bit for bit: a decoder layer's projections at M = 1, 8 and 64 (the GEMV and
GEMM paths), pinned and pageable host buffers, and repeated calls on one
workspace.
"""

import numpy as np
import pytest

import oracle
from int8_quantized_matmul_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def i2s():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_quantized_matmul_gb300 import build as libbuild
    libbuild.build()
    from int8_quantized_matmul_gb300 import i2s as mod
    assert mod.device_supported() == 1, "the library needs an sm_103 device"
    return mod


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def same_bits(a, b):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    bad = np.nonzero(a.view(np.uint32).reshape(-1) != b.view(np.uint32).reshape(-1))[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}"


def layer(o, M, seed, pinned):
    """One Qwen2-1.5B decoder layer: q, k, v share an activation, gate and up
    another; all activations are slices of one host buffer, all outputs of
    another."""
    acts = {"attn": 1536, "o": 1536, "ffn": 1536, "down": 8960}
    which = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "ffn", "up": "ffn", "down": "down"}
    x_all = torch.from_numpy(synth.normal_f32(M * sum(acts.values()), seed=seed, outlier_p=0.01))
    n_out = sum(N for _, N, _ in synth.QWEN2_1P5B_LAYER)
    y_all = torch.full((M * n_out,), float("nan"), dtype=torch.float32)
    if pinned:
        x_all, y_all = x_all.pin_memory(), y_all.pin_memory()
    xs, off = {}, 0
    for name, K in acts.items():
        xs[name] = x_all[off:off + M * K].view(M, K)
        off += M * K
    probs, keep, yo = [], [], 0
    for i, (name, N, K) in enumerate(synth.QWEN2_1P5B_LAYER):
        packed = o.i2s_pack(synth.codes(N, K, seed=seed * 10 + i), 0.03 + 0.01 * i)
        y = y_all[yo:yo + M * N].view(M, N)
        yo += M * N
        probs.append((torch.from_numpy(packed).cuda(), N, K, xs[which[name]], y))
        keep.append((packed, N, K, xs[which[name]], y))
    return probs, keep


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M", [1, 8, 64])
def test_host_call_decoder_layer(i2s, o, M, pinned):
    probs, keep = layer(o, M, seed=M + 3, pinned=pinned)
    g = i2s.HostGroup(probs, M)
    g()
    torch.cuda.synchronize()
    assert i2s.read_status(g.ws) == 0
    for packed, N, K, x, y in keep:
        same_bits(y.numpy(), o.i2s_mul_mat(packed, N, K, x.numpy(), nth=8))


def test_host_call_repeated_with_new_inputs(i2s, o):
    # three calls on one workspace, the host activations rewritten between
    # calls: each call's outputs follow its own inputs
    M = 8
    probs, keep = layer(o, M, seed=21, pinned=True)
    g = i2s.HostGroup(probs, M)
    for it in range(3):
        for _, _, _, x, _ in keep:
            x.copy_(torch.from_numpy(synth.normal_f32(x.shape, seed=100 + it + x.shape[1])))
        g()
        torch.cuda.synchronize()
        for packed, N, K, x, y in keep:
            same_bits(y.numpy(), o.i2s_mul_mat(packed, N, K, x.numpy(), nth=8))
    assert i2s.read_status(g.ws) == 0


@pytest.mark.parametrize("mode", [True, "y"])
@pytest.mark.parametrize("M", [1, 8, 64])
def test_host_call_mapped_decoder_layer(i2s, o, M, mode):
    # I2S_HOST_MAPPED: pinned (device-mapped) host buffers read and written by
    # the kernels directly, no staging copies; I2S_HOST_MAPPED_Y: x copied up,
    # y written in place by the epilogue. Same bits as the oracle either way.
    probs, keep = layer(o, M, seed=M + 50, pinned=True)
    g = i2s.HostGroup(probs, M, mapped=mode)
    for _ in range(2):
        for _, _, _, _, y in keep:
            y.fill_(float("nan"))
        g()
        torch.cuda.synchronize()
        assert i2s.read_status(g.ws) == 0
        for packed, N, K, x, y in keep:
            same_bits(y.numpy(), o.i2s_mul_mat(packed, N, K, x.numpy(), nth=8))


@pytest.mark.parametrize("mode", [True, "y"])
def test_host_call_mapped_rejects_pageable_buffers(i2s, o, mode):
    # the mapped modes check their ranges before anything is enqueued:
    # pageable buffers are refused, and the outputs stay untouched
    probs, keep = layer(o, 8, seed=77, pinned=False)
    g = i2s.HostGroup(probs, 8, mapped=mode)
    with pytest.raises(i2s.I2SError) as e:
        g()
    assert e.value.status == -8   # I2S_E_BAD_ARG
    torch.cuda.synchronize()
    for _, _, _, _, y in keep:
        assert torch.isnan(y).all()
