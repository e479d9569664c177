"""The fused decode launch (i2s_mul_mat_grouped_fused: the GEMV whose prologue
quantizes the activation rows) against the CPU oracle, bit for bit.

Covers the page's K x N grid as single-problem groups, a decoder layer and the
full 28-layer projection set at M = 1, 8, 9 and 16, the accumulator headroom
case, many calls in a row on one workspace (the flags each launch leaves
cleared for the next), replays of a captured CUDA graph, and many distinct K.
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def same_bits(a, b):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    bad = np.nonzero(a.view(np.uint32).reshape(-1) != b.view(np.uint32).reshape(-1))[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}"


def packed_problem(N, K, seed, w_scale=None):
    payload = synth.packed_code_bytes(N * K // 4, seed=seed)
    ws = np.float32(w_scale if w_scale is not None else synth.uniform_f32(1, seed + 7, 0.01, 0.1)[0])
    return np.concatenate([payload, np.frombuffer(ws.tobytes(), np.uint8), np.zeros(28, np.uint8)])


def _row_slice(packed, N, K, n0, n1):
    rb = K // 4
    return np.concatenate([packed[n0 * rb:n1 * rb], packed[N * rb:N * rb + 32]])


@pytest.mark.parametrize("K", [128, 1024, 1152])
@pytest.mark.parametrize("N", [1, 2, 64, 70, 100])
@pytest.mark.parametrize("M", [1, 3, 8, 16])
def test_fused_page_grid(i2s, o, K, N, M):
    c = synth.codes(N, K, seed=K * 7 + N + M)
    packed = o.i2s_pack(c, 0.05)
    x = synth.normal_f32((M, K), seed=K + N + M, outlier_p=0.01)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    wd, xd = dev(packed), dev(x)
    ws = i2s.i2s_mul_mat_grouped_fused([(wd, N, K, xd, y)], M)
    assert i2s.read_status(ws) == 0
    same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=4))


def decoder_layer(seed, M):
    """One Qwen2-1.5B decoder layer's projections: q, k, v share an activation,
    gate and up another; o and down have their own."""
    xs = {"attn": synth.normal_f32((M, 1536), seed=seed), "o": synth.normal_f32((M, 1536), seed=seed + 1),
          "ffn": synth.normal_f32((M, 1536), seed=seed + 2), "down": synth.normal_f32((M, 8960), seed=seed + 3)}
    which = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "ffn", "up": "ffn", "down": "down"}
    probs = [(name, N, K, packed_problem(N, K, seed * 10 + i), which[name])
             for i, (name, N, K) in enumerate(synth.QWEN2_1P5B_LAYER)]
    return probs, xs


@pytest.mark.parametrize("M", [1, 8, 9, 16])
def test_fused_decoder_layer(i2s, o, M):
    probs, xs = decoder_layer(seed=M, M=M)
    dx = {k: dev(v) for k, v in xs.items()}
    ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _, N, _, _, _ in probs]
    dw = [dev(p[3]) for p in probs]
    group = [(w, p[1], p[2], dx[p[4]], y) for w, p, y in zip(dw, probs, ys)]
    ws = i2s.i2s_mul_mat_grouped_fused(group, M)
    assert i2s.read_status(ws) == 0
    for (name, N, K, packed, a), y in zip(probs, ys):
        same_bits(host(y), o.i2s_mul_mat(packed, N, K, xs[a], nth=8))


@pytest.mark.parametrize("M", [1, 8])
def test_fused_full_decode_set_sampled(i2s, o, M):
    """All 196 projections of the 28-layer set in one fused launch (112
    distinct activations), checked on sampled weight rows of layers 0, 13
    and 27 and every output of layer 27's k projection."""
    rng = synth.rng(11 + M)
    group, keep = [], []
    xs_all = {}
    for layer in range(28):
        xs = {1536: [synth.normal_f32((M, 1536), seed=1000 * M + 4 * layer + j) for j in range(3)],
              8960: [synth.normal_f32((M, 8960), seed=1000 * M + 4 * layer + 3)]}
        dx = {k: [dev(v) for v in vs] for k, vs in xs.items()}
        which = {"q": 0, "k": 0, "v": 0, "o": 1, "gate": 2, "up": 2, "down": 0}
        for i, (name, N, K) in enumerate(synth.QWEN2_1P5B_LAYER):
            packed = packed_problem(N, K, seed=layer * 10 + i)
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            j = which[name]
            group.append((dev(packed), N, K, dx[K][j], y))
            keep.append((layer, name, N, K, packed, y, xs[K][j]))
    ws = i2s.i2s_mul_mat_grouped_fused(group, M)
    assert i2s.read_status(ws) == 0
    for layer, name, N, K, packed, y, x in keep:
        yh = host(y)
        if layer == 27 and name == "k":
            same_bits(yh, o.i2s_mul_mat(packed, N, K, x, nth=8))
        elif layer in (0, 13, 27):
            for n0 in sorted(set([0, N - 16] + list(rng.integers(0, N - 16, size=2)))):
                same_bits(yh[:, n0:n0 + 16], o.i2s_mul_mat(_row_slice(packed, N, K, n0, n0 + 16), 16, K, x, nth=8))


@pytest.mark.parametrize("M", [1, 16])
def test_fused_headroom_k8960(i2s, o, M):
    # every code 2, every activation quantizing to +127: dot = 254 K over six
    # K chunks per tile, the split-K partials zeroed by the launch's prologue
    K, N = 8960, 1536
    packed = o.i2s_pack(np.full((N, K), 2, np.uint8), 0.05)
    x = np.ones((M, K), np.float32)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = i2s.i2s_mul_mat_grouped_fused([(dev(packed), N, K, dev(x), y)], M)
    assert i2s.read_status(ws) == 0
    small = o.i2s_mul_mat(o.i2s_pack(np.full((4, K), 2, np.uint8), 0.05), 4, K, x[:2])
    assert (host(y).view(np.uint32) == small[0, 0].view(np.uint32)).all()


def test_fused_back_to_back_on_one_workspace(i2s, o):
    # twelve launches with no synchronisation alternate two input sets and two
    # output sets; each launch waits for the one before it and leaves the flags
    # cleared, so every output matches the oracle
    M = 8
    probs, xa = decoder_layer(seed=31, M=M)
    _, xb = decoder_layer(seed=32, M=M)
    dA = {k: dev(v) for k, v in xa.items()}
    dB = {k: dev(v) for k, v in xb.items()}
    dw = [dev(p[3]) for p in probs]
    ys = [[torch.zeros((M, N), dtype=torch.float32, device="cuda") for _, N, _, _, _ in probs] for _ in range(2)]
    groups = [[(w, p[1], p[2], d[p[4]], y) for w, p, y in zip(dw, probs, ys[i])] for i, d in enumerate((dA, dB))]
    ws = torch.empty(i2s.i2s_mul_mat_grouped_fused_workspace(groups[0], M), dtype=torch.uint8, device="cuda")
    i2s.i2s_mul_mat_grouped_fused_init(ws)
    for it in range(12):
        i2s.i2s_mul_mat_grouped_fused(groups[it % 2], M, ws=ws)
    assert i2s.read_status(ws) == 0
    for xs, yset in ((xa, ys[0]), (xb, ys[1])):
        for (name, N, K, packed, a), y in zip(probs, yset):
            same_bits(host(y), o.i2s_mul_mat(packed, N, K, xs[a], nth=8))
    # the flag area is clear again after the launches
    flags = host(ws[256:256 + 4 * (7 + 4 + 1)].view(torch.int32))
    assert not flags.any()


def test_fused_under_cuda_graph(i2s, o):
    M = 8
    probs, xs = decoder_layer(seed=41, M=M)
    dx = {k: dev(v) for k, v in xs.items()}
    dw = [dev(p[3]) for p in probs]
    ys = [torch.zeros((M, N), dtype=torch.float32, device="cuda") for _, N, _, _, _ in probs]
    group = [(w, p[1], p[2], dx[p[4]], y) for w, p, y in zip(dw, probs, ys)]
    ws = i2s.i2s_mul_mat_grouped_fused(group, M)   # initialises ws; warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            i2s.i2s_mul_mat_grouped_fused(group, M, ws=ws)
    for _ in range(3):
        for y in ys:
            y.zero_()
        g.replay()
        for (name, N, K, packed, a), y in zip(probs, ys):
            same_bits(host(y), o.i2s_mul_mat(packed, N, K, xs[a], nth=8))
    assert i2s.read_status(ws) == 0


def test_fused_eight_distinct_k_and_shared_activations(i2s, o):
    # eight K classes (the most one launch takes), two problems per class
    # sharing an activation, ragged N
    M = 5
    Ks = [128, 256, 640, 1024, 1536, 1664, 3072, 4736]
    group, keep = [], []
    for i, K in enumerate(Ks):
        x = synth.normal_f32((M, K), seed=70 + i, outlier_p=0.01)
        xd = dev(x)
        for j, N in enumerate((130, 67)):
            packed = packed_problem(N, K, seed=80 + 2 * i + j)
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            group.append((dev(packed), N, K, xd, y))
            keep.append((N, K, packed, x, y))
    ws = i2s.i2s_mul_mat_grouped_fused(group, M)
    assert i2s.read_status(ws) == 0
    for N, K, packed, x, y in keep:
        same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=4))
    # a ninth K is rejected before anything is enqueued
    extra = (dev(packed_problem(64, 2048, seed=99)), 64, 2048, dev(synth.normal_f32((M, 2048), seed=98)),
             torch.empty((M, 64), dtype=torch.float32, device="cuda"))
    assert i2s.i2s_mul_mat_grouped_fused_workspace(group + [extra], M) == 0
