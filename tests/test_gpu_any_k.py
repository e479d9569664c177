"""I8_S mul_mat_add(_relu) and the W8A8 matmul at reduction lengths K that are
not multiples of 64, through the C ABI, against the CPU oracle bit for bit.

A conv run as im2col_asym then mul_mat_add ("VibeASR in audio.cpp", section
Encoder) reduces over C*KW positions, 7 for a 7-tap stem on a mono waveform;
"ggml: additive INT8/ternary types, fused CPU ops, and kernels for VibeASR
(1/2)", section Tests, runs mul_mat_add over several input and output channel
counts. The GPU pads each f16 operand row to a multiple of 64 positions with
zeros, which adds nothing to the integer dot; these tests check that claim at
K in {1, 4, 7, 28, 100, 224, 1000} and with ragged M and N.
"""

import numpy as np
import pytest

import oracle
from int8_quantized_matmul_gb300 import synth
from tests import pins

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ANY_K = [1, 7, 28, 100, 224, 1000]


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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def same_bits(a, b):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.nonzero(a.reshape(-1) != b.reshape(-1))[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}"


def i8s_inputs(o, M, N, K, seed):
    wp = o.i8s_pack(synth.int8_normal((N, K), seed=seed), 0.01)
    xp = o.i8s_quantize(synth.normal_f32((M, K), seed=seed + 1))
    bias = synth.normal_f32(N, seed=seed + 2, std=0.1)
    return wp, xp, bias


@pytest.mark.parametrize("K", ANY_K)
@pytest.mark.parametrize("M,N", [(3, 5), (40, 300), (161, 257)])
def test_i8s_mul_mat_add_any_k(i2s, o, M, N, K):
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=M + N + K)
    for relu in (False, True):
        y8, ws = i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dev(xp), M, bias=dev(bias), relu=relu)
        assert i2s.read_status(ws) == 0
        oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=relu, nth=4)
        same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
        same_bits(host(y8), oy8)


@pytest.mark.parametrize("K", [7, 100, 1000])
def test_i8s_packed_any_k(i2s, o, K):
    M, N = 77, 300
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=K + 5)
    packed = i2s.i8s_pack_weights(dev(wp), N, K)
    # the packed rows hold K rounded up to 64 positions, then the scale trailer
    Kp = (K + 63) // 64 * 64
    ph = host(packed)
    assert ph.size == 2 * N * Kp + 16
    off = o.i8s_scale_offset(N * K)
    assert np.array_equal(ph[2 * N * Kp:2 * N * Kp + 4], wp[off:off + 4])
    y8, ws = i2s.i8s_mul_mat_add_relu_packed(packed, N, K, dev(xp), M, bias=dev(bias), relu=True)
    assert i2s.read_status(ws) == 0
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=True, nth=4)
    same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
    same_bits(host(y8), oy8)


def test_i8s_conv_stem_as_im2col_then_mul_mat_add(i2s, o):
    # a causal 7-tap conv with 64 output channels on one input channel:
    # im2col_asym (left pad KW - stride, right pad 0) gives OL x 7 windows,
    # mul_mat_add over K = 7 gives OL x 64, with bias and ReLU, requantized
    C, L, KW, stride, N = 1, 24000, 7, 1, 64
    x = o.i8s_pack(synth.int8_normal((C, L), seed=3), 0.02)
    cols, OL = o.i8s_im2col_asym(x, C, L, KW, stride, KW - stride, 0)
    K = C * KW
    wp = o.i8s_pack(synth.int8_normal((N, K), seed=4), 0.01)
    bias = synth.normal_f32(N, seed=5, std=0.1)
    dcols, _ = i2s.i8s_im2col_asym(dev(x), C, L, KW, stride, KW - stride, 0)
    same_bits(host(dcols), cols)
    y8, ws = i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dcols, OL, bias=dev(bias), relu=True)
    assert i2s.read_status(ws) == 0
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, cols, OL, bias=bias, relu=True, nth=8)
    same_bits(host(i2s.i8s_ws_f32(ws, OL, N)), oyf)
    same_bits(host(y8), oy8)


def w8a8_inputs(o, M, N, K, seed):
    wq, bs = o.w8a8_quantize_weights(synth.normal_f32((N, K), seed=seed, std=0.02))
    x = synth.normal_f32((M, K), seed=seed + 1, outlier_p=0.01)
    return wq, bs, x


@pytest.mark.parametrize("K", ANY_K)
@pytest.mark.parametrize("M,N", [(3, 5), (161, 257)])
def test_w8a8_any_k(i2s, o, M, N, K):
    wq, bs, x = w8a8_inputs(o, M, N, K, seed=M * 7 + N + K)
    want = o.w8a8_mul_mat(wq, bs, x, nth=4)
    d, ws = i2s.w8a8_mul_mat(dev(wq), dev(bs), dev(x))
    assert i2s.read_status(ws) == 0
    same_bits(host(d), want)
    packed = i2s.w8a8_pack_weights(dev(wq))
    d2, ws2 = i2s.w8a8_mul_mat_packed(packed, dev(bs), N, K, dev(x))
    assert i2s.read_status(ws2) == 0
    same_bits(host(d2), want)


def test_w8a8_grouped_mixed_k(i2s, o):
    # one grouped call over projections with K = 28, 100 and 1000 (two share
    # an activation), every output against the oracle
    M = 45
    specs = [(300, 100, 0), (70, 100, 0), (257, 28, 1), (64, 1000, 2)]
    xs = {a: synth.normal_f32((M, K), seed=500 + a) for (_, K, a) in specs}
    dxs = {a: dev(v) for a, v in xs.items()}
    problems, refs = [], []
    for i, (N, K, a) in enumerate(specs):
        wq, bs = o.w8a8_quantize_weights(synth.normal_f32((N, K), seed=600 + i, std=0.02))
        d = torch.empty((M, N), dtype=torch.float32, device="cuda")
        problems.append((i2s.w8a8_pack_weights(dev(wq)), dev(bs), N, K, dxs[a], d))
        refs.append(o.w8a8_mul_mat(wq, bs, xs[a], nth=4))
    ws = i2s.w8a8_mul_mat_grouped(problems, M)
    assert i2s.read_status(ws) == 0
    for p, ref in zip(problems, refs):
        same_bits(host(p[5]), ref)


def test_i8s_epilogue_association_golden(i2s, o):
    # the hand-derived I8_S case (K = 4, scales that are not powers of two):
    # the GPU's F32 outputs against the fixture's bits directly
    c = pins.epilogue_cases()["i8s_epilogue"]
    K = int(c["K"][0])
    X = np.array([int(v) for v in c["x"]], dtype=np.int8)[None, :]
    W = np.array([[int(v) for v in c[f"w{i}"]] for i in range(2)], dtype=np.int8)
    bias = np.array([pins._hex_f32(v) for v in c["bias"]], dtype=np.float32)
    wp = o.i8s_pack(W, float(pins._hex_f32(c["w_scale"][0])))
    xp = o.i8s_pack(X, float(pins._hex_f32(c["x_scale"][0])))
    want = np.array([int(v, 16) for v in c["y"]], dtype=np.uint32)
    for relu in (False, True):
        _, ws = i2s.i8s_mul_mat_add_relu(dev(wp), 2, K, dev(xp), 1, bias=dev(bias), relu=relu)
        assert np.array_equal(host(i2s.i8s_ws_f32(ws, 1, 2))[0].view(np.uint32), want)


def test_w8a8_epilogue_association_golden(i2s, o):
    c = pins.epilogue_cases()["w8a8_epilogue"]
    x = np.array([float(v) for v in c["x"]], dtype=np.float32)[None, :]
    wq = np.array([[int(v) for v in c[f"wq{i}"]] for i in range(2)], dtype=np.int8)
    bs = np.array([pins._hex_f32(v) for v in c["b_scale"]], dtype=np.float32)
    want = np.array([int(v, 16) for v in c["d"]], dtype=np.uint32)
    d, _ = i2s.w8a8_mul_mat(dev(wq), dev(bs), dev(x))
    assert np.array_equal(host(d)[0].view(np.uint32), want)


@pytest.mark.parametrize("K", [4, 8188, 8192, 8196, 8960])
def test_w8a8_packed_row_lengths(i2s, o, K):
    # the packed and grouped calls quantize each activation row straight into
    # f16 operand rows: rows of up to 8192 values whose length is a multiple
    # of 4 are read as float4 and kept in registers, other rows take the
    # plain loop; both sides of that boundary against the oracle
    M, N = 5, 70
    wq, bs, x = w8a8_inputs(o, M, N, K, seed=K)
    want = o.w8a8_mul_mat(wq, bs, x, nth=4)
    packed = i2s.w8a8_pack_weights(dev(wq))
    d, ws = i2s.w8a8_mul_mat_packed(packed, dev(bs), N, K, dev(x))
    assert i2s.read_status(ws) == 0
    same_bits(host(d), want)
