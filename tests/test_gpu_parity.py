"""GPU path (through the C ABI) against the CPU oracle, bit for bit.

Every float output is compared as raw bits (uint32), every integer output
exactly: the method is exact up to its final IEEE multiplies, and both sides
perform those in binary32 round-to-nearest. Shapes span several tiles with
ragged tails; the full-size workloads are checked on sampled output rows that
the oracle computes one by one, plus properties that hold at any size.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from int8_quantized_matmul_gb300 import synth
from tests import pins

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
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.nonzero(a.reshape(-1) != b.reshape(-1))[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}: {a.reshape(-1)[bad[:5]]} vs {b.reshape(-1)[bad[:5]]}"


# ---------------------------------------------------------------------------
# activation quantizer
# ---------------------------------------------------------------------------

def test_quantize_act_golden_rows(i2s, o):
    cases = pins.load_cases("quant_rows.txt")
    x = np.zeros((len(cases), 128), dtype=np.float32)
    for i, c in enumerate(cases):
        x[i, :len(c["x"])] = [float(Fraction(v)) for v in c["x"]]
    q, s, rs = i2s.i2s_quantize_act(dev(x))
    q, s, rs = host(q), host(s), host(rs)
    for i, c in enumerate(cases):
        n = len(c["q"])
        assert np.array_equal(q[i, :n], np.array([int(v) for v in c["q"]], np.int8)), c["name"]
        assert int(rs[i]) == int(c["sum"][0])
        assert pins.f32_bits(s[i]) == pins.f32_bits(pins.nearest_f32(pins.parse_rational(c["scale"][0])))
    oq, os_, ors = o.quantize_rows(x)
    same_bits(q, oq), same_bits(s, os_), same_bits(rs, ors)


@pytest.mark.parametrize("M,K", [(1, 128), (37, 1152), (8, 8960), (513, 1536)])
def test_quantize_act_random(i2s, o, M, K):
    x = synth.normal_f32((M, K), seed=M * 7 + K, outlier_p=0.01)
    x[M // 2] = 0.0
    q, s, rs = i2s.i2s_quantize_act(dev(x))
    oq, os_, ors = o.quantize_rows(x)
    same_bits(host(q), oq)
    same_bits(host(s), os_)
    same_bits(host(rs), ors)


# ---------------------------------------------------------------------------
# I2_S matmul
# ---------------------------------------------------------------------------

def run_i2s(i2s, o, N, K, M, seed, w_scale=0.05, x=None, **kw):
    c = synth.codes(N, K, seed=seed)
    packed = o.i2s_pack(c, w_scale)
    if x is None:
        x = synth.normal_f32((M, K), seed=seed + 1, outlier_p=0.01)
    y = i2s.i2s_mul_mat(dev(packed), N, K, dev(x), **kw)
    return host(y), o.i2s_mul_mat(packed, N, K, x, nth=4)


@pytest.mark.parametrize("K", [128, 1024, 1152])
@pytest.mark.parametrize("N", [1, 2, 64, 70, 100])
@pytest.mark.parametrize("M", [1, 3, 8, 16])
def test_i2s_page_grid(i2s, o, K, N, M):
    got, want = run_i2s(i2s, o, N, K, M, seed=K * 131 + N * 7 + M)
    same_bits(got, want)


def test_i2s_single_matmul_n256_k1024_m4(i2s, o):
    # codes P = (.3,.4,.3), w_scale 0.05, x ~ N(0,1), seed 0
    c = synth.codes(256, 1024, seed=0)
    packed = o.i2s_pack(c, 0.05)
    x = synth.normal_f32((4, 1024), seed=0)
    y = host(i2s.i2s_mul_mat(dev(packed), 256, 1024, dev(x)))
    same_bits(y, o.i2s_mul_mat(packed, 256, 1024, x))


@pytest.mark.parametrize("M", [1, 2, 8, 9, 16])
@pytest.mark.parametrize("grid", [1, 5, 7, 0])
@pytest.mark.parametrize("K", [1152, 4608, 8960])
def test_i2s_gemv_tc_grid_sizes(i2s, o, M, grid, K):
    # CTA counts that cut row tiles into K-chunk segments at different places
    # (split-K partials combined by integer atomics) give identical bits
    import ctypes
    N = 900
    c = synth.codes(N, K, seed=M + K)
    packed = o.i2s_pack(c, 0.07)
    x = synth.normal_f32((M, K), seed=M + 1, outlier_p=0.01)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(i2s.i2s_mul_mat_workspace(M, N, K), dtype=torch.uint8, device="cuda")
    cfg = i2s.i2s_config(3, grid)
    wd, xd = dev(packed), dev(x)   # keep the device buffers alive across the call
    for _ in range(2):   # twice: the partial buffers are re-zeroed by each call
        rc = i2s.lib.i2s_mul_mat_ex(wd.data_ptr(), N, K, xd.data_ptr(), M, y.data_ptr(), ws.data_ptr(),
                                    ws.numel(), ctypes.byref(cfg), i2s._stream())
        assert rc == 0
        same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=8))
        assert i2s.read_status(ws) == 0


@pytest.mark.parametrize("M", [1, 8, 16])
def test_i2s_gemv_paths_agree(i2s, o, M):
    # the tensor-core GEMV (path 3) and GEMM (path 2) give the same bits
    c = synth.codes(300, 1536, seed=60 + M)
    packed = o.i2s_pack(c, 0.02)
    x = synth.normal_f32((M, 1536), seed=61 + M)
    want = o.i2s_mul_mat(packed, 300, 1536, x)
    for path in (2, 3):
        same_bits(host(i2s.i2s_mul_mat(dev(packed), 300, 1536, dev(x), path=path)), want)


@pytest.mark.parametrize("grid", [1, 2, 3, 4, 8, 0])
def test_i2s_split_k_gives_identical_bits(i2s, o, grid):
    # the shipped GEMV splits each 128-row tile into 1536-position K chunks;
    # small grids give each CTA a range that starts or ends inside a tile, so
    # partial dots from several CTAs meet in the integer split-K buffer
    got, want = run_i2s(i2s, o, 1100, 8960, 8, seed=77, path=3, grid_ctas=grid)
    same_bits(got, want)


@pytest.mark.parametrize("M", [9, 17, 40])
def test_i2s_row_counts_around_the_gemv_limit(i2s, o, M):
    # 9 rows: the GEMV's 16-row operand; 17 and 40: the GEMM's ragged tiles
    got, want = run_i2s(i2s, o, 300, 1152, M, seed=M)
    same_bits(got, want)


@pytest.mark.parametrize("M", [1, 8, 16])
@pytest.mark.parametrize("grid", [0, 7])
def test_i2s_headroom_k8960(i2s, o, M, grid):
    # every code 2 and every activation quantizing to +127 (x = 1.0) on the
    # shipped decode path: q = 127 becomes the digits (-1, 0, 2) of the GEMV's
    # operand, and dot = 254 K = 2,275,840 comes from six K chunks per tile;
    # grid 7 cuts tiles between CTAs, so the split-K sums meet at the extreme
    K, N = 8960, 1536
    packed = o.i2s_pack(np.full((N, K), 2, np.uint8), 0.05)
    x = np.ones((M, K), np.float32)
    y = host(i2s.i2s_mul_mat(dev(packed), N, K, dev(x), path=3, grid_ctas=grid))
    small = o.i2s_mul_mat(o.i2s_pack(np.full((4, K), 2, np.uint8), 0.05), 4, K, x[:2])
    assert (small == small[0, 0]).all()
    assert (y.view(np.uint32) == small[0, 0].view(np.uint32)).all()
    act_scale = np.float32(1.0) / np.float32(127.0)
    assert small[0, 0] == np.float32(127 * K) * (np.float32(0.05) * act_scale)


@pytest.mark.parametrize("M", [1, 64])
def test_i2s_epilogue_association_golden(i2s, o, M):
    # the hand-derived epilogue case (scales that are not powers of two, so the
    # order of the scale product decides the last bit) on the GPU, compared
    # with the fixture's bits directly: M = 1 runs the GEMV, M = 64 the GEMM
    c = pins.epilogue_cases()["i2s_epilogue"]
    K = int(c["K"][0])
    codes = np.array([pins._rle(c[f"codes{i}"], int) for i in range(3)], dtype=np.uint8)
    x = np.repeat(np.array(pins._rle(c["x"]), dtype=np.float32)[None, :], M, axis=0)
    packed = o.i2s_pack(codes, float(pins._hex_f32(c["w_scale"][0])))
    y = host(i2s.i2s_mul_mat(dev(packed), 3, K, dev(x)))
    want = np.array([int(v, 16) for v in c["y"]], dtype=np.uint32)
    assert (y.view(np.uint32) == want[None, :]).all(), [hex(v) for v in y[0].view(np.uint32)]


def test_i2s_degenerate(i2s, o):
    K, N, M = 1024, 70, 4
    x = synth.normal_f32((M, K), seed=3)
    x[1] = 0.0
    got, want = run_i2s(i2s, o, N, K, M, seed=5, x=x)
    same_bits(got, want)
    assert (got[1] == 0).all() and not np.isnan(got).any()
    zero_w = o.i2s_pack(np.ones((N, K), np.uint8), 0.0)
    y = host(i2s.i2s_mul_mat(dev(zero_w), N, K, dev(x)))
    assert (y == 0).all() and not np.isnan(y).any()


@pytest.mark.parametrize("N", [1, 2, 64, 70, 100])
def test_i2s_single_group_k128(i2s, o, N):
    got, want = run_i2s(i2s, o, N, 128, 3, seed=N)
    same_bits(got, want)


def test_i2s_code3_behaves_like_oracle(i2s, o):
    c = synth.codes(70, 256, seed=9)
    c[::7, ::5] = 3
    packed = o.i2s_pack(c, 0.5)
    x = synth.normal_f32((5, 256), seed=10)
    same_bits(host(i2s.i2s_mul_mat(dev(packed), 70, 256, dev(x))), o.i2s_mul_mat(packed, 70, 256, x))


def layer_problems(o, K_h=1536, K_i=8960, M=1, seed=0, scale_div=1):
    """One decoder layer's projections with the activations a real layer shares."""
    shapes = [(n, N // scale_div, K) for n, N, K in synth.QWEN2_1P5B_LAYER]
    xs = {1536: None}
    acts = {"attn": synth.normal_f32((M, K_h), seed=seed + 100),
            "o": synth.normal_f32((M, K_h), seed=seed + 101),
            "ffn": synth.normal_f32((M, K_h), seed=seed + 102),
            "down": synth.normal_f32((M, K_i), seed=seed + 103)}
    which = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "ffn", "up": "ffn", "down": "down"}
    probs = []
    for i, (name, N, K) in enumerate(shapes):
        c = synth.codes(N, K, seed=seed + i)
        ws = float(synth.uniform_f32(1, seed + 50 + i, 0.01, 0.1)[0])
        probs.append((name, N, K, o.i2s_pack(c, ws), acts[which[name]], which[name]))
    del xs
    return probs, acts


@pytest.mark.parametrize("M", [1, 8, 16])
def test_i2s_grouped_decoder_layer(i2s, o, M):
    probs, acts = layer_problems(o, M=M, seed=M)
    dacts = {k: dev(v) for k, v in acts.items()}
    dys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _, N, _, _, _, _ in probs]
    group = [(dev(p[3]), p[1], p[2], dacts[p[5]], y) for p, y in zip(probs, dys)]
    i2s.i2s_mul_mat_grouped(group, M)
    for (name, N, K, packed, x, _), y in zip(probs, dys):
        same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=4))


def test_i2s_grouped_under_cuda_graph(i2s, o):
    probs, acts = layer_problems(o, M=8, seed=3, scale_div=4)
    dacts = {k: dev(v) for k, v in acts.items()}
    dys = [torch.zeros((8, N), dtype=torch.float32, device="cuda") for _, N, _, _, _, _ in probs]
    group = [(dev(p[3]), p[1], p[2], dacts[p[5]], y) for p, y in zip(probs, dys)]
    ws = torch.empty(i2s.i2s_mul_mat_grouped_workspace(group, 8), dtype=torch.uint8, device="cuda")
    i2s.i2s_mul_mat_grouped(group, 8, ws=ws)   # warm-up outside capture
    torch.cuda.synchronize()
    for y in dys:
        y.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            i2s.i2s_mul_mat_grouped(group, 8, ws=ws)
    g.replay()
    for (name, N, K, packed, x, _), y in zip(probs, dys):
        same_bits(host(y), o.i2s_mul_mat(packed, N, K, x))


def test_i2s_grouped_back_to_back_on_one_workspace(i2s, o):
    # The quantization and GEMV launches are programmatic dependents of the
    # launch before them: each waits for it before touching the workspace.
    # Twelve calls alternate two input sets and two output sets on one
    # workspace with no synchronisation; a launch that wrote the workspace
    # while the previous GEMV still read it would corrupt an output.
    M = 8
    probs, acts_a = layer_problems(o, M=M, seed=21)
    _, acts_b = layer_problems(o, M=M, seed=22)
    dA = {k: dev(v) for k, v in acts_a.items()}
    dB = {k: dev(v) for k, v in acts_b.items()}
    ys = [[torch.zeros((M, N), dtype=torch.float32, device="cuda") for _, N, _, _, _, _ in probs] for _ in range(2)]
    dw = [dev(p[3]) for p in probs]
    groups = [[(w, p[1], p[2], acts[p[5]], y) for w, p, y in zip(dw, probs, ys[i])] for i, acts in enumerate((dA, dB))]
    ws = torch.empty(i2s.i2s_mul_mat_grouped_workspace(groups[0], M), dtype=torch.uint8, device="cuda")
    for it in range(12):
        i2s.i2s_mul_mat_grouped(groups[it % 2], M, ws=ws)
    assert i2s.read_status(ws) == 0
    for acts, yset in ((acts_a, ys[0]), (acts_b, ys[1])):
        for (name, N, K, packed, _, act), y in zip(probs, yset):
            same_bits(host(y), o.i2s_mul_mat(packed, N, K, acts[act], nth=4))


@pytest.mark.parametrize("M", [1, 8, 16])
def test_i2s_grouped_run_repeated_after_one_quantize(i2s, o, M):
    # A completed run leaves the split-K sums and tile counters at zero, so a
    # run may be repeated after one quantization: three runs, the outputs
    # cleared between them, each compared with the oracle (the down
    # projection, K = 8960, is split over six K chunks per tile)
    probs, acts = layer_problems(o, M=M, seed=40 + M)
    dacts = {k: dev(v) for k, v in acts.items()}
    dys = [torch.zeros((M, N), dtype=torch.float32, device="cuda") for _, N, _, _, _, _ in probs]
    group = i2s.Group([(dev(p[3]), p[1], p[2], dacts[p[5]], y) for p, y in zip(probs, dys)], M)
    group.quantize()
    for _ in range(3):
        for y in dys:
            y.zero_()
        group.run()
        assert i2s.read_status(group.ws) == 0
        for (name, N, K, packed, x, _), y in zip(probs, dys):
            same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=4))


def _row_slice(packed, N, K, n0, n1):
    """I2_S bytes of weight rows n0..n1 (rows are contiguous, K/4 bytes each)."""
    rb = K // 4
    return np.concatenate([packed[n0 * rb:n1 * rb], packed[N * rb:N * rb + 32]])


def test_i2s_full_decode_set_sampled(i2s, o):
    """The 28-layer Qwen2-1.5B projection set at M = 8, one grouped launch per
    layer pair, checked on sampled weight rows of every projection."""
    M = 8
    rng = synth.rng(5)
    for layer in (0, 27):
        xs = {1536: synth.normal_f32((M, 1536), seed=layer), 8960: synth.normal_f32((M, 8960), seed=layer + 1)}
        dx = {k: dev(v) for k, v in xs.items()}
        group, keep = [], []
        for i, (name, N, K) in enumerate(synth.QWEN2_1P5B_LAYER):
            payload = synth.packed_code_bytes(N * K // 4, seed=layer * 10 + i)
            ws = np.float32(synth.uniform_f32(1, layer * 10 + i, 0.01, 0.1)[0])
            packed = np.concatenate([payload, np.frombuffer(ws.tobytes(), np.uint8), np.zeros(28, np.uint8)])
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            group.append((dev(packed), N, K, dx[K], y))
            keep.append((name, N, K, packed, y))
        i2s.i2s_mul_mat_grouped(group, M)
        for name, N, K, packed, y in keep:
            yh = host(y)
            for n0 in sorted(set([0, N - 16] + list(rng.integers(0, N - 16, size=2)))):
                sub = _row_slice(packed, N, K, n0, n0 + 16)
                same_bits(yh[:, n0:n0 + 16], o.i2s_mul_mat(sub, 16, K, xs[K]))


def test_i2s_lm_head_m1_sampled(i2s, o):
    N, K, M = 151936, 1536, 1
    payload = synth.packed_code_bytes(N * K // 4, seed=99)
    packed = np.concatenate([payload, np.frombuffer(np.float32(0.03).tobytes(), np.uint8), np.zeros(28, np.uint8)])
    x = synth.normal_f32((M, K), seed=98)
    y = host(i2s.i2s_mul_mat(dev(packed), N, K, dev(x)))
    for n0 in (0, 70000, N - 32):
        same_bits(y[:, n0:n0 + 32], o.i2s_mul_mat(_row_slice(packed, N, K, n0, n0 + 32), 32, K, x))


# ---------------------------------------------------------------------------
# I2_S prefill GEMM (tcgen05)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M", [17, 64, 130, 512])
@pytest.mark.parametrize("N,K", [(100, 1152), (300, 1536), (257, 128), (128, 8960)])
def test_i2s_gemm(i2s, o, M, N, K):
    got, want = run_i2s(i2s, o, N, K, M, seed=M * 3 + N + K)
    same_bits(got, want)


@pytest.mark.parametrize("K", [128, 384, 1152])
@pytest.mark.parametrize("N", [1, 2, 100, 129])
@pytest.mark.parametrize("M", [17, 100])
def test_i2s_gemm_page_grid(i2s, o, K, N, M):
    # the page's small K x N grid on the tensor-core GEMM: fewer weight rows
    # than one tile (the code ring's rows past N arrive as zeros), K of one,
    # three and nine 128-position groups (an odd count leaves half of the last
    # 256-position stage past K)
    got, want = run_i2s(i2s, o, N, K, M, seed=K * 17 + N * 3 + M)
    same_bits(got, want)


@pytest.mark.parametrize("M", [1, 5, 16])
def test_i2s_gemm_small_m(i2s, o, M):
    got, want = run_i2s(i2s, o, 300, 1152, M, seed=M + 11, path=2)
    same_bits(got, want)


@pytest.mark.parametrize("grid", [1, 3, 7, 0])
def test_i2s_gemm_grid_sizes_give_identical_bits(i2s, o, grid):
    c = synth.codes(700, 1536, seed=4)
    packed = o.i2s_pack(c, 0.07)
    x = synth.normal_f32((300, 1536), seed=5, outlier_p=0.01)
    y = torch.empty((300, 700), dtype=torch.float32, device="cuda")
    ws = torch.empty(i2s.i2s_mul_mat_workspace(300, 700, 1536), dtype=torch.uint8, device="cuda")
    cfg = i2s.i2s_config(2, grid)
    import ctypes
    wd, xd = dev(packed), dev(x)   # keep the device buffers alive across the call
    rc = i2s.lib.i2s_mul_mat_ex(wd.data_ptr(), 700, 1536, xd.data_ptr(), 300, y.data_ptr(), ws.data_ptr(),
                                ws.numel(), ctypes.byref(cfg), i2s._stream())
    assert rc == 0
    same_bits(host(y), o.i2s_mul_mat(packed, 700, 1536, x, nth=8))
    assert i2s.read_status(ws) == 0


def test_i2s_gemm_headroom_k8960_m64(i2s, o):
    K, N, M = 8960, 1536, 64
    packed = o.i2s_pack(np.full((N, K), 2, np.uint8), 0.05)
    x = np.ones((M, K), np.float32)
    y = host(i2s.i2s_mul_mat(dev(packed), N, K, dev(x)))   # M = 64 -> tensor-core GEMM
    small = o.i2s_mul_mat(o.i2s_pack(np.full((4, K), 2, np.uint8), 0.05), 4, K, x[:2])
    assert (y.view(np.uint32) == small[0, 0].view(np.uint32)).all()


@pytest.mark.parametrize("M", [20, 300])
def test_i2s_gemm_headroom_k65536(i2s, o, M):
    # the largest K the library takes, every code 2, every q = 127: the
    # accumulator reaches sum (c/2) q = 127 K = 8,323,072, just below 2^23,
    # where binary32 still resolves the halves the digit MMAs add
    K, N = 65536, 256
    packed = o.i2s_pack(np.full((N, K), 2, np.uint8), 0.05)
    x = np.ones((M, K), np.float32)
    y = host(i2s.i2s_mul_mat(dev(packed), N, K, dev(x), path=2))
    small = o.i2s_mul_mat(o.i2s_pack(np.full((4, K), 2, np.uint8), 0.05), 4, K, x[:2])
    assert (small == small[0, 0]).all()
    assert (y.view(np.uint32) == small[0, 0].view(np.uint32)).all()


def test_i2s_gemm_large_k_random(i2s, o):
    # K = 40960 with random codes and 1% outliers, ragged N and M
    K, N, M = 40960, 300, 37
    got, want = run_i2s(i2s, o, N, K, M, seed=123)
    same_bits(got, want)


def test_i2s_gemm_degenerate(i2s, o):
    K, N, M = 1024, 70, 40
    x = synth.normal_f32((M, K), seed=13)
    x[7] = 0.0
    got, want = run_i2s(i2s, o, N, K, M, seed=14, x=x)
    same_bits(got, want)
    assert (got[7] == 0).all()
    zero_w = o.i2s_pack(np.ones((N, K), np.uint8), 0.0)
    y = host(i2s.i2s_mul_mat(dev(zero_w), N, K, dev(x)))
    assert (y == 0).all() and not np.isnan(y).any()


def test_i2s_gemm_prefill_layer_and_lm_head_sampled(i2s, o):
    """One decoder layer plus the lm_head at M = 512 (pp512 shape, 1% outliers),
    grouped into one tensor-core launch; sampled weight rows of each projection
    against the oracle."""
    M = 512
    rng = synth.rng(8)
    xs = {k: synth.normal_f32((M, 1536), seed=20 + k, outlier_p=0.01) for k in range(3)}
    xs[3] = synth.normal_f32((M, 8960), seed=23, outlier_p=0.01)
    which = {"q": 0, "k": 0, "v": 0, "o": 1, "gate": 2, "up": 2, "down": 3}
    dx = {k: dev(v) for k, v in xs.items()}
    shapes = list(synth.QWEN2_1P5B_LAYER) + [synth.QWEN2_1P5B_LM_HEAD]
    group, keep = [], []
    for i, (name, N, K) in enumerate(shapes):
        payload = synth.packed_code_bytes(N * K // 4, seed=300 + i)
        ws_ = np.float32(synth.uniform_f32(1, 400 + i, 0.01, 0.1)[0])
        packed = np.concatenate([payload, np.frombuffer(ws_.tobytes(), np.uint8), np.zeros(28, np.uint8)])
        a = which.get(name, 2)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        group.append((dev(packed), N, K, dx[a], y))
        keep.append((name, N, K, packed, y, xs[a]))
    ws = i2s.i2s_mul_mat_grouped(group, M)
    assert i2s.read_status(ws) == 0
    for name, N, K, packed, y, x in keep:
        yh = host(y)
        for n0 in sorted(set([0, N - 16] + list(rng.integers(0, N - 16, size=2)))):
            same_bits(yh[:, n0:n0 + 16], o.i2s_mul_mat(_row_slice(packed, N, K, n0, n0 + 16), 16, K, x, nth=8))


# ---------------------------------------------------------------------------
# I8_S requant and fused mul_mat_add(_relu)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 31, 4096, 1000003])
def test_i8s_requant(i2s, o, n):
    y = synth.normal_f32(n, seed=n, outlier_p=0.01)
    got = host(i2s.i8s_requant(dev(y)))
    same_bits(got, o.i8s_quantize(y))
    z = host(i2s.i8s_requant(dev(np.zeros(n, np.float32))))
    same_bits(z, o.i8s_quantize(np.zeros(n, np.float32)))


def i8s_inputs(o, M, N, K, seed):
    W = synth.int8_normal((N, K), seed=seed)
    wp = o.i8s_pack(W, 0.01)
    xp = o.i8s_quantize(synth.normal_f32((M, K), seed=seed + 1))
    bias = synth.normal_f32(N, seed=seed + 2, std=0.1)
    return wp, xp, bias


@pytest.mark.parametrize("M,N,K", [(3, 5, 64), (100, 300, 256), (130, 257, 1024), (64, 128, 2048)])
@pytest.mark.parametrize("relu", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_i8s_mul_mat_add(i2s, o, M, N, K, relu, with_bias):
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=M + N + K)
    b = bias if with_bias else None
    y8, ws = i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dev(xp), M, bias=dev(b) if b is not None else None, relu=relu)
    yf = host(i2s.i8s_ws_f32(ws, M, N))
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=b, relu=relu, nth=4)
    same_bits(yf, oyf)
    same_bits(host(y8), oy8)


@pytest.mark.parametrize("relu", [False, True])
def test_i8s_split_tiles_ragged_chunk(i2s, o, relu):
    # 10 weight tiles x 9 K chunks (K % 1024 = 704 and K % 128 = 64: the last chunk is short
    # and its last stage half past K) over 74 or 76 CTA pairs: ranges of one or two chunks cut
    # most tiles between pairs, and the pair that completes a tile adds the others' slots.
    # Every output is compared.
    M, N, K = 40, 2560, 8896
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=11 + relu)
    y8, ws = i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dev(xp), M, bias=dev(bias), relu=relu)
    assert i2s.read_status(ws) == 0
    yf = host(i2s.i8s_ws_f32(ws, M, N))
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=relu, nth=8)
    same_bits(yf, oyf)
    same_bits(host(y8), oy8)


@pytest.mark.parametrize("K", [384, 640, 1088, 3072])
def test_i8s_stage_ring_wraps(i2s, o, K):
    # 3, 5, 9 and 24 stages of 128 positions: every stage slot of the
    # operand ring is reused, with a ragged N that leaves part of the second
    # CTA of a pair without weight rows
    M, N = 64, 300
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=K)
    y8, ws = i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dev(xp), M, bias=dev(bias), relu=True)
    assert i2s.read_status(ws) == 0
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=True, nth=4)
    same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
    same_bits(host(y8), oy8)


def test_i8s_repeated_calls_identical(i2s, o):
    # the same call twenty times: every run's bits equal the oracle's (the MMA
    # issuers, producers and split-tile completion race differently each time)
    M, N, K = 300, 640, 4096
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=5)
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, nth=8)
    dw, dx, db = dev(wp), dev(xp), dev(bias)
    y8, ws = i2s.i8s_mul_mat_add_relu(dw, N, K, dx, M, bias=db)
    for _ in range(20):
        i2s.i8s_mul_mat_add_relu(dw, N, K, dx, M, bias=db, y=y8, ws=ws)
        assert i2s.read_status(ws) == 0
        same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
        same_bits(host(y8), oy8)


def test_i8s_headroom(i2s, o):
    # every weight and activation at +127: acc = 127*127*K = 132,120,576 (> 2^24)
    M, N, K = 16, 64, 8192
    wp = o.i8s_pack(np.full((N, K), 127, np.int8), 0.01)
    xp = o.i8s_pack(np.full((M, K), 127, np.int8), 0.02)
    y8, ws = i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dev(xp), M)
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M)
    same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
    same_bits(host(y8), oy8)


@pytest.mark.parametrize("N,K,relu", [(8192, 2048, True), (2048, 8192, False)])
def test_i8s_encoder_fc_full(i2s, o, N, K, relu):
    """Encoder FC1 (2048 -> 8192, ReLU) / FC2 (8192 -> 2048) at L = 900 frames,
    every F32 output and every I8_S byte (values, padding and the in-band
    scale) against the oracle."""
    M = 900
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=N)
    y8, ws = i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dev(xp), M, bias=dev(bias), relu=relu)
    assert i2s.read_status(ws) == 0
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=relu, nth=16)
    same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
    same_bits(host(y8), oy8)


@pytest.mark.parametrize("M,N,K", [(3, 5, 64), (100, 300, 256), (130, 257, 1024), (300, 640, 4096)])
@pytest.mark.parametrize("relu", [False, True])
def test_i8s_packed_weights(i2s, o, M, N, K, relu):
    # weights packed once (f16 rows + scale trailer), two calls on them
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=M + 2 * N + K)
    packed = i2s.i8s_pack_weights(dev(wp), N, K)
    ph = host(packed)
    assert np.array_equal(ph[2 * N * K:2 * N * K + 16], wp[o.i8s_scale_offset(N * K):o.i8s_scale_offset(N * K) + 16])
    y8, ws = i2s.i8s_mul_mat_add_relu_packed(packed, N, K, dev(xp), M, bias=dev(bias), relu=relu)
    assert i2s.read_status(ws) == 0
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=relu, nth=4)
    same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
    same_bits(host(y8), oy8)
    xp2 = o.i8s_quantize(synth.normal_f32((M, K), seed=M + 5))
    y8b, _ = i2s.i8s_mul_mat_add_relu_packed(packed, N, K, dev(xp2), M, bias=dev(bias), relu=relu, ws=ws)
    same_bits(host(y8b), o.i8s_mul_mat_add(wp, N, K, xp2, M, bias=bias, relu=relu, nth=4)[0])


def test_i8s_packed_encoder_fc1_full(i2s, o):
    M, N, K = 900, 8192, 2048
    wp, xp, bias = i8s_inputs(o, M, N, K, seed=N + 1)
    packed = i2s.i8s_pack_weights(dev(wp), N, K)
    y8, ws = i2s.i8s_mul_mat_add_relu_packed(packed, N, K, dev(xp), M, bias=dev(bias), relu=True)
    assert i2s.read_status(ws) == 0
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=True, nth=16)
    same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
    same_bits(host(y8), oy8)
