"""I8_S element-wise ops, the encoder conv pieces and the W8A8 matmul on the
GPU (through the C ABI) against the CPU oracle, byte for byte.

Every output is an I8_S tensor (int8 payload, padding, F32 scale and zero
bytes) or an F32 array, compared as raw bytes: both sides perform the same
IEEE binary32 operations in the same order. Sizes cover empty tails of the
vector paths (n % 16, rows that are not whole 32-bit words), single elements,
several tiles with ragged edges and the full-size encoder shapes that
bench.py times.
"""

import numpy as np
import pytest

import oracle
from int8_quantized_matmul_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# two minutes of 24 kHz audio after the 32-channel stem
ENC_C, ENC_L = 32, 2_880_000


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


def same_bytes(a, b):
    a = np.ascontiguousarray(a).reshape(-1)
    b = np.ascontiguousarray(b).reshape(-1)
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.nonzero(a != b)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}: {a[bad[:5]]} vs {b[bad[:5]]}"


def i8s_tensor(o, shape, seed, std=40.0, scale=None):
    q = synth.int8_normal(shape, seed=seed, std=std)
    s = scale if scale is not None else float(synth.rng(seed + 1).uniform(0.001, 0.1))
    return q, o.i8s_pack(q, s)


# ---------------------------------------------------------------------------
# add_scaled
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 15, 16, 17, 4096, 100003, (1 << 20) + 7])
def test_add_scaled(i2s, o, n):
    _, a = i8s_tensor(o, n, seed=n)
    _, b = i8s_tensor(o, n, seed=n + 7)
    got = host(i2s.i8s_add_scaled(dev(a), dev(b), n))
    same_bytes(got, o.i8s_add_scaled(a, b, n)[0])


def test_add_scaled_cancels_to_zero(i2s, o):
    # b = -a with the same scale: every sum is exactly zero, so the output is
    # all-zero codes with the floored scale 1e-5/127
    n = 5000
    q, a = i8s_tensor(o, n, seed=3, scale=0.25)
    b = o.i8s_pack((-q.astype(np.int16)).astype(np.int8), 0.25)
    got = host(i2s.i8s_add_scaled(dev(a), dev(b), n))
    same_bytes(got, o.i8s_add_scaled(a, b, n)[0])
    assert not got[:n].any()


def test_add_scaled_encoder_size(i2s, o):
    n = ENC_C * ENC_L
    _, a = i8s_tensor(o, n, seed=11)
    _, b = i8s_tensor(o, n, seed=12)
    got = host(i2s.i8s_add_scaled(dev(a), dev(b), n))
    same_bytes(got, o.i8s_add_scaled(a, b, n)[0])


# ---------------------------------------------------------------------------
# rms_norm_scaled
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,ne0", [(1, 1), (3, 5), (7, 32), (100, 64), (33, 2048), (5, 130), (257, 7), (2, 8192)])
@pytest.mark.parametrize("with_gamma", [False, True])
def test_rms_norm_scaled(i2s, o, rows, ne0, with_gamma):
    _, x = i8s_tensor(o, (rows, ne0), seed=rows * 31 + ne0)
    gamma = synth.normal_f32(ne0, seed=ne0, std=0.5) if with_gamma else None
    got = host(i2s.i8s_rms_norm_scaled(dev(x), rows, ne0, 1e-5, gamma=dev(gamma) if with_gamma else None))
    same_bytes(got, o.i8s_rms_norm_scaled(x, rows, ne0, 1e-5, gamma=gamma)[0])


def test_rms_norm_zero_rows_and_eps(i2s, o):
    rows, ne0 = 9, 48
    q = synth.int8_normal((rows, ne0), seed=5)
    q[::3] = 0   # all-zero rows: the factor is 1/sqrt(eps), the outputs 0
    x = o.i8s_pack(q, 0.02)
    for eps in (1e-5, 1e-3, 3.0):   # eps > 0: with eps = 0 an all-zero row would give 0 * inf
        got = host(i2s.i8s_rms_norm_scaled(dev(x), rows, ne0, eps))
        same_bytes(got, o.i8s_rms_norm_scaled(x, rows, ne0, eps)[0])


def test_rms_norm_encoder_size(i2s, o):
    # channel-last RMSNorm over the 32 channels of every time step
    rows, ne0 = ENC_L, ENC_C
    _, x = i8s_tensor(o, (rows, ne0), seed=13)
    got = host(i2s.i8s_rms_norm_scaled(dev(x), rows, ne0, 1e-5))
    same_bytes(got, o.i8s_rms_norm_scaled(x, rows, ne0, 1e-5)[0])


# ---------------------------------------------------------------------------
# transpose (cont of a permute): the scale travels with the values
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("a,b", [(1, 1), (1, 100), (5, 7), (64, 64), (65, 129), (300, 17), (1000, 2048), (77, 1000), (600, 40)])
def test_transpose(i2s, o, a, b):
    _, src = i8s_tensor(o, (a, b), seed=a * 7 + b)
    got = host(i2s.i8s_transpose(dev(src), a, b))
    same_bytes(got, o.i8s_permute_cont(src, a, b))


def test_transpose_encoder_size(i2s, o):
    _, src = i8s_tensor(o, (ENC_C, ENC_L), seed=14)
    got = host(i2s.i8s_transpose(dev(src), ENC_C, ENC_L))
    same_bytes(got, o.i8s_permute_cont(src, ENC_C, ENC_L))
    # and back: the round trip restores the input bytes exactly
    back = host(i2s.i8s_transpose(dev(got), ENC_L, ENC_C))
    same_bytes(back, src)


# ---------------------------------------------------------------------------
# im2col_asym and the depthwise op
# ---------------------------------------------------------------------------

GEOMS = [
    (3, 20, 4, 1, 3, 0),      # causal, stride 1
    (5, 37, 7, 2, 5, 0),      # causal strided, odd kernel
    (2, 16, 8, 4, 4, 0),      # kernel 2*stride, left pad K - stride
    (4, 29, 3, 3, 0, 2),      # right pad only
    (1, 5, 7, 1, 6, 1),       # input shorter than the kernel
    (6, 64, 5, 5, 0, 0),      # no padding
    (64, 1000, 7, 1, 6, 0),   # a depthwise block's geometry
    (33, 513, 10, 5, 5, 0),   # stride 5, ragged everything
]


@pytest.mark.parametrize("C,L,KW,stride,pad_l,pad_r", GEOMS)
def test_im2col_asym(i2s, o, C, L, KW, stride, pad_l, pad_r):
    _, x = i8s_tensor(o, (C, L), seed=C * L + KW)
    got, OL = i2s.i8s_im2col_asym(dev(x), C, L, KW, stride, pad_l, pad_r)
    ref, OL_ref = o.i8s_im2col_asym(x, C, L, KW, stride, pad_l, pad_r)
    assert OL == OL_ref
    same_bytes(host(got), ref)


# kernels a multiple of 4 wide: output rows go out as 16-byte words where a
# block's bytes are a multiple of 16 (C*KW*T), word by word otherwise; ragged
# last blocks, 1..3 words per (t, c) group, both paddings
GEOMS_WIDE = [
    (4, 1001, 4, 1, 3, 0),
    (3, 777, 8, 2, 6, 0),
    (5, 3000, 12, 3, 9, 0),
    (16, 4099, 8, 2, 0, 6),
    (32, 9001, 4, 2, 2, 0),
]


@pytest.mark.parametrize("C,L,KW,stride,pad_l,pad_r", GEOMS_WIDE)
def test_im2col_asym_wide_kernels(i2s, o, C, L, KW, stride, pad_l, pad_r):
    _, x = i8s_tensor(o, (C, L), seed=C + L + KW)
    got, OL = i2s.i8s_im2col_asym(dev(x), C, L, KW, stride, pad_l, pad_r)
    ref, OL_ref = o.i8s_im2col_asym(x, C, L, KW, stride, pad_l, pad_r)
    assert OL == OL_ref
    same_bytes(host(got), ref)


# kernel 4, stride 2, channels a multiple of 32, rows a multiple of 16 bytes:
# the path with one channel per lane and no staging, at every even left pad
# modulo 16 (each is its own instantiation), with right pads, ragged output
# lengths (not a multiple of 32) and inputs shorter than one run
GEOMS_K4S2 = [(32, 4096, p, 0) for p in (0, 2, 4, 6, 8, 10, 12, 14)] + [
    (32, 4096, 18, 5),
    (64, 1008, 2, 3),
    (96, 160, 2, 0),
    (32, 16, 2, 0),
    (32, 48, 30, 7),
    (64, 80, 16, 16),
]


@pytest.mark.parametrize("C,L,pad_l,pad_r", GEOMS_K4S2)
def test_im2col_k4_s2(i2s, o, C, L, pad_l, pad_r):
    _, x = i8s_tensor(o, (C, L), seed=C + L + pad_l)
    got, OL = i2s.i8s_im2col_asym(dev(x), C, L, 4, 2, pad_l, pad_r)
    ref, OL_ref = o.i8s_im2col_asym(x, C, L, 4, 2, pad_l, pad_r)
    assert OL == OL_ref
    same_bytes(host(got), ref)


def test_im2col_encoder_size(i2s, o):
    # the stage-1 downsampling conv: kernel 4 = 2*stride, causal left pad 2
    C, L, KW, stride = ENC_C, ENC_L, 4, 2
    _, x = i8s_tensor(o, (C, L), seed=15)
    got, OL = i2s.i8s_im2col_asym(dev(x), C, L, KW, stride, KW - stride, 0)
    ref, _ = o.i8s_im2col_asym(x, C, L, KW, stride, KW - stride, 0)
    same_bytes(host(got), ref)


@pytest.mark.parametrize("C,L,KW,stride,pad_l,pad_r", GEOMS)
@pytest.mark.parametrize("relu", [False, True])
def test_depthwise(i2s, o, C, L, KW, stride, pad_l, pad_r, relu):
    _, w = i8s_tensor(o, (C, KW), seed=C + KW, scale=0.01)
    _, x = i8s_tensor(o, (C, L), seed=C * L)
    bias = synth.normal_f32(C, seed=C, std=0.1)
    got, OL = i2s.i8s_depthwise_mul_mat_add(dev(w), KW, dev(x), C, L, stride, pad_l, pad_r, bias=dev(bias),
                                            relu=relu)
    ref, _ = o.i8s_depthwise_mul_mat_add(w, KW, x, C, L, stride, pad_l, pad_r, bias=bias, relu=relu)
    same_bytes(host(got), ref)


@pytest.mark.parametrize("with_bias,relu", [(False, False), (False, True), (True, False), (True, True)])
def test_depthwise_stride1_bias_relu_combinations(i2s, o, with_bias, relu):
    # the stride-1 kernel is built for each combination of bias and ReLU
    C, L, KW = 40, 5000, 7
    _, w = i8s_tensor(o, (C, KW), seed=17, scale=0.01)
    _, x = i8s_tensor(o, (C, L), seed=18)
    bias = synth.normal_f32(C, seed=19, std=0.1) if with_bias else None
    got, OL = i2s.i8s_depthwise_mul_mat_add(dev(w), KW, dev(x), C, L, 1, KW - 1, 0,
                                            bias=dev(bias) if with_bias else None, relu=relu)
    ref, _ = o.i8s_depthwise_mul_mat_add(w, KW, x, C, L, 1, KW - 1, 0, bias=bias, relu=relu)
    same_bytes(host(got), ref)


def test_depthwise_no_bias_and_headroom(i2s, o):
    # every tap and input at +127 (acc = 7 * 127^2), no bias
    C, L, KW = 16, 300, 7
    w = o.i8s_pack(np.full((C, KW), 127, np.int8), 0.5)
    x = o.i8s_pack(np.full((C, L), 127, np.int8), 0.25)
    got, _ = i2s.i8s_depthwise_mul_mat_add(dev(w), KW, dev(x), C, L, 1, KW - 1, 0)
    ref, _ = o.i8s_depthwise_mul_mat_add(w, KW, x, C, L, 1, KW - 1, 0)
    same_bytes(host(got), ref)


def test_depthwise_positions_past_the_end_stay_out_of_the_amax(i2s, o):
    # Every real output has a full window (no padding): acc = 7 * 100 and the bias cancels
    # s * 700 exactly, so y = 0 everywhere and the amax is its floor. Positions past the last
    # output (OL = 994 is not a multiple of the kernel's 8-output groups) see zero-filled
    # windows, smaller acc and y != 0: folding any of them would change the scale and every byte.
    C, L, KW = 4, 1000, 7
    w = o.i8s_pack(np.full((C, KW), 1, np.int8), 0.5)
    x = o.i8s_pack(np.full((C, L), 100, np.int8), 0.01)
    s = np.float32(0.5) * np.float32(0.01)
    bias = np.full(C, -(np.float32(700.0) * s), np.float32)
    got, OL = i2s.i8s_depthwise_mul_mat_add(dev(w), KW, dev(x), C, L, 1, 0, 0, bias=dev(bias))
    ref, y_ref = o.i8s_depthwise_mul_mat_add(w, KW, x, C, L, 1, 0, 0, bias=bias)
    assert OL == y_ref.shape[1] == L - KW + 1
    assert not y_ref.any() and not ref[: C * OL].any()
    same_bytes(host(got), ref)


def test_depthwise_encoder_size(i2s, o):
    # the 7-tap causal depthwise conv of a stage-0 block
    C, L, KW = ENC_C, ENC_L, 7
    _, w = i8s_tensor(o, (C, KW), seed=16, scale=0.01)
    _, x = i8s_tensor(o, (C, L), seed=17)
    bias = synth.normal_f32(C, seed=18, std=0.1)
    got, _ = i2s.i8s_depthwise_mul_mat_add(dev(w), KW, dev(x), C, L, 1, KW - 1, 0, bias=dev(bias))
    ref, _ = o.i8s_depthwise_mul_mat_add(w, KW, x, C, L, 1, KW - 1, 0, bias=bias)
    same_bytes(host(got), ref)


# ---------------------------------------------------------------------------
# W8A8 per-channel
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 1), (3, 100), (64, 2048), (300, 777)])
def test_w8a8_quantize_weights(i2s, o, N, K):
    w = synth.normal_f32((N, K), seed=N * K, std=0.02)
    if N > 1:
        w[1] = 0.0   # an all-zero channel: the 1e-9 floor
    if K > 10:       # exact halfway values: scale 1 from amax 127
        w[0, :10] = np.array([127.0, 2.5, -2.5, 3.5, 0.5, -0.5, 1.5, 126.5, -127.0, 4.4], np.float32)
    wq, bs = i2s.w8a8_quantize_weights(dev(w))
    owq, obs = o.w8a8_quantize_weights(w)
    same_bytes(host(wq), owq)
    same_bytes(host(bs), obs)


def w8a8_inputs(o, M, N, K, seed):
    w = synth.normal_f32((N, K), seed=seed, std=0.02)
    wq, bs = o.w8a8_quantize_weights(w)
    x = synth.normal_f32((M, K), seed=seed + 1, outlier_p=0.01)
    return wq, bs, x


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (3, 5, 64), (17, 70, 256), (130, 257, 1024), (300, 640, 2048)])
def test_w8a8_mul_mat(i2s, o, M, N, K):
    wq, bs, x = w8a8_inputs(o, M, N, K, seed=M + N + K)
    d, ws = i2s.w8a8_mul_mat(dev(wq), dev(bs), dev(x))
    assert i2s.read_status(ws) == 0
    same_bytes(host(d), o.w8a8_mul_mat(wq, bs, x, nth=4))


def test_w8a8_160_row_tiles(i2s, o):
    # The GEMM takes 128- or 160-row activation tiles, whichever leaves less work on its busiest
    # CTA pair. The small shapes above take 128-row tiles; here 150 rows are one 160-row tile
    # against two 128-row ones, and with 76 weight tiles that is one unit per pair against two,
    # so the call runs on 160-row tiles with ten zero rows at the tail. Every output is compared.
    M, N, K = 150, 19456, 1024
    wq, bs, x = w8a8_inputs(o, M, N, K, seed=7)
    d, ws = i2s.w8a8_mul_mat(dev(wq), dev(bs), dev(x))
    assert i2s.read_status(ws) == 0
    same_bytes(host(d), o.w8a8_mul_mat(wq, bs, x, nth=8))


def test_w8a8_headroom_and_zero_rows(i2s, o):
    # codes at +-127 over K = 8192 (|acc| = 127^2 * 8192 > 2^24) and an
    # all-zero activation row (scale 1e-9/127, outputs 0)
    M, N, K = 16, 64, 8192
    wq = np.full((N, K), 127, np.int8)
    wq[1::2] = -127
    bs = np.full(N, 0.003, np.float32)
    x = np.full((M, K), 2.0, np.float32)
    x[3] = 0.0
    d, ws = i2s.w8a8_mul_mat(dev(wq), dev(bs), dev(x))
    same_bytes(host(d), o.w8a8_mul_mat(wq, bs, x))


# Qwen3-1.7B projections at prefill M = 512 (pp512), sampled rows: the
# activation quantizer is per row, so the oracle on a row subset gives those
# rows of d exactly.
QWEN3_1P7B = [(2048, 2048), (1024, 2048), (6144, 2048), (2048, 6144)]


@pytest.mark.parametrize("N,K", QWEN3_1P7B)
def test_w8a8_prefill_projection_sampled(i2s, o, N, K):
    M = 512
    wq, bs, x = w8a8_inputs(o, M, N, K, seed=N + K)
    d, ws = i2s.w8a8_mul_mat(dev(wq), dev(bs), dev(x))
    assert i2s.read_status(ws) == 0
    got = host(d)
    for m0 in (0, 251, M - 8):
        same_bytes(got[m0:m0 + 8], o.w8a8_mul_mat(wq, bs, x[m0:m0 + 8], nth=8))


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (17, 70, 256), (300, 640, 2048), (161, 257, 1088)])
def test_w8a8_packed(i2s, o, M, N, K):
    # weights packed once, then two calls on the same packed weights
    wq, bs, x = w8a8_inputs(o, M, N, K, seed=M * 3 + N + K)
    packed = i2s.w8a8_pack_weights(dev(wq))
    ref = o.w8a8_mul_mat(wq, bs, x, nth=4)
    d, ws = i2s.w8a8_mul_mat_packed(packed, dev(bs), N, K, dev(x))
    assert i2s.read_status(ws) == 0
    same_bytes(host(d), ref)
    x2 = synth.normal_f32((M, K), seed=M + 99)
    d2, _ = i2s.w8a8_mul_mat_packed(packed, dev(bs), N, K, dev(x2), ws=ws)
    same_bytes(host(d2), o.w8a8_mul_mat(wq, bs, x2, nth=4))


def test_w8a8_packed_prefill_projection_sampled(i2s, o):
    M, N, K = 512, 6144, 2048
    wq, bs, x = w8a8_inputs(o, M, N, K, seed=7)
    packed = i2s.w8a8_pack_weights(dev(wq))
    d, ws = i2s.w8a8_mul_mat_packed(packed, dev(bs), N, K, dev(x))
    got = host(d)
    for m0 in (0, 333, M - 8):
        same_bytes(got[m0:m0 + 8], o.w8a8_mul_mat(wq, bs, x[m0:m0 + 8], nth=8))


def test_device_rounding_around_every_half_integer(i2s, o):
    # amax = 127 makes inv = 127/127 = 1 exactly, so each code is round(y)
    # itself: every float within 2000 ulps of k + 1/2 (k = 0..126), of the
    # integers, and their negatives, against the CPU reference (C roundf)
    pts = []
    for k in range(128):
        for centre in (k + 0.5, float(k)):
            c = np.float32(centre)
            lo, hi = c, c
            for _ in range(2000):
                lo = np.nextafter(lo, np.float32(-np.inf), dtype=np.float32)
                hi = np.nextafter(hi, np.float32(np.inf), dtype=np.float32)
                pts += [lo, hi]
            pts.append(c)
    y = np.array(pts, dtype=np.float32)
    y = y[np.abs(y) <= 127.0]
    y = np.concatenate([y, -y, np.array([127.0, -127.0], np.float32)])
    got = host(i2s.i8s_requant(dev(y)))
    ref = o.i8s_quantize(y)
    same_bytes(got, ref)


def test_w8a8_grouped_layer(i2s, o):
    # a Qwen3-1.7B-shaped layer at a ragged M: q, k, v share one activation,
    # gate and up another; every output equals the oracle's, bit for bit
    M = 77
    specs = [("q", 2048, 2048, 0), ("k", 1024, 2048, 0), ("v", 1024, 2048, 0), ("o", 2048, 2048, 1),
             ("gate", 640, 2048, 2), ("up", 640, 2048, 2), ("down", 2048, 1088, 3)]
    xs = {a: synth.normal_f32((M, K), seed=200 + a, outlier_p=0.01) for (_, _, K, a) in specs}
    dxs = {a: dev(x) for a, x in xs.items()}
    problems, refs = [], []
    for i, (name, N, K, a) in enumerate(specs):
        wq, bs = o.w8a8_quantize_weights(synth.normal_f32((N, K), seed=300 + i, std=0.02))
        d = torch.empty((M, N), dtype=torch.float32, device="cuda")
        problems.append((i2s.w8a8_pack_weights(dev(wq)), dev(bs), N, K, dxs[a], d))
        refs.append(o.w8a8_mul_mat(wq, bs, xs[a], nth=8))
    ws = i2s.w8a8_mul_mat_grouped(problems, M)
    assert i2s.read_status(ws) == 0
    for p, ref in zip(problems, refs):
        same_bytes(host(p[5]), ref)
    # a second call on the same workspace (counters cleared by the call)
    for p in problems:
        p[5].zero_()
    i2s.w8a8_mul_mat_grouped(problems, M, ws=ws)
    for p, ref in zip(problems, refs):
        same_bytes(host(p[5]), ref)
