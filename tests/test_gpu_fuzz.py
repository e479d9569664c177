"""Seeded random shapes through the shipped paths, every output against the
CPU oracle bit for bit: grouped I2_S calls on the GEMV (M <= 16) and GEMM
(M > 16) paths with shared activations and ragged N, I8_S mul_mat_add(_relu)
at any K, and grouped W8A8 calls. Sizes stay small enough for the oracle.
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
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.nonzero(a.reshape(-1) != b.reshape(-1))[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}"


@pytest.mark.parametrize("case", range(48))
def test_fuzz_i2s_grouped(i2s, o, case):
    rng = np.random.default_rng(1000 + case)
    M = int(rng.choice([1, 2, 5, 8, 9, 13, 16, 17, 33, 64, 100, 129, 200]))
    n_act = int(rng.integers(1, 4))
    Ks = [int(rng.integers(1, 17)) * 128 for _ in range(n_act)]
    xs = [synth.normal_f32((M, K), seed=10 * case + a, outlier_p=0.02) for a, K in enumerate(Ks)]
    dxs = [dev(x) for x in xs]
    group, keep = [], []
    for i in range(int(rng.integers(1, 6))):
        a = int(rng.integers(0, n_act))
        K, N = Ks[a], int(rng.integers(1, 500))
        packed = o.i2s_pack(synth.codes(N, K, seed=100 * case + i), float(rng.uniform(0.005, 0.2)))
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        group.append((dev(packed), N, K, dxs[a], y))
        keep.append((packed, N, K, xs[a], y))
    ws = i2s.i2s_mul_mat_grouped(group, M)
    assert i2s.read_status(ws) == 0
    for packed, N, K, x, y in keep:
        same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=8))


@pytest.mark.parametrize("M", [4, 40])
def test_grouped_many_problems(i2s, o, M):
    # up to the group limit of small projections in one launch (M = 4: the
    # GEMV, M = 40: the GEMM), every output against the oracle: the kernels'
    # problem tables and their per-tile problem lookup cross every boundary
    rng = np.random.default_rng(77 + M)
    n_act = 7
    Ks = [128 * int(rng.integers(1, 4)) for _ in range(n_act)]
    xs = [synth.normal_f32((M, K), seed=500 + a, outlier_p=0.02) for a, K in enumerate(Ks)]
    dxs = [dev(x) for x in xs]
    count = 256 if M <= 16 else 200
    group, keep = [], []
    for i in range(count):
        a = int(rng.integers(0, n_act))
        K, N = Ks[a], int(rng.integers(1, 300))
        packed = o.i2s_pack(synth.codes(N, K, seed=9000 + i), float(rng.uniform(0.005, 0.2)))
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        group.append((dev(packed), N, K, dxs[a], y))
        keep.append((packed, N, K, xs[a], y))
    ws = i2s.i2s_mul_mat_grouped(group, M)
    assert i2s.read_status(ws) == 0
    for packed, N, K, x, y in keep:
        same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=8))


@pytest.mark.parametrize("case", range(24))
def test_fuzz_i8s_mul_mat_add(i2s, o, case):
    rng = np.random.default_rng(2000 + case)
    M, N, K = int(rng.integers(1, 400)), int(rng.integers(1, 600)), int(rng.integers(1, 3000))
    wp = o.i8s_pack(synth.int8_normal((N, K), seed=case), float(rng.uniform(0.001, 0.05)))
    xp = o.i8s_quantize(synth.normal_f32((M, K), seed=case + 50))
    bias = synth.normal_f32(N, seed=case + 60, std=0.1) if case % 3 else None
    relu = bool(case % 2)
    y8, ws = i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dev(xp), M, bias=None if bias is None else dev(bias), relu=relu)
    assert i2s.read_status(ws) == 0
    oy8, oyf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=relu, nth=8)
    same_bits(host(i2s.i8s_ws_f32(ws, M, N)), oyf)
    same_bits(host(y8), oy8)


@pytest.mark.parametrize("case", range(16))
def test_fuzz_w8a8_grouped(i2s, o, case):
    rng = np.random.default_rng(3000 + case)
    M = int(rng.integers(1, 300))
    Ks = [int(rng.integers(1, 2500)) for _ in range(int(rng.integers(1, 3)))]
    xs = {a: synth.normal_f32((M, K), seed=700 + 10 * case + a, outlier_p=0.01) for a, K in enumerate(Ks)}
    dxs = {a: dev(v) for a, v in xs.items()}
    problems, refs = [], []
    for i in range(int(rng.integers(1, 6))):
        a = int(rng.integers(0, len(Ks)))
        K, N = Ks[a], int(rng.integers(1, 500))
        wq, bs = o.w8a8_quantize_weights(synth.normal_f32((N, K), seed=800 + 10 * case + i, std=0.02))
        d = torch.empty((M, N), dtype=torch.float32, device="cuda")
        problems.append((i2s.w8a8_pack_weights(dev(wq)), dev(bs), N, K, dxs[a], d))
        refs.append(o.w8a8_mul_mat(wq, bs, xs[a], nth=8))
    ws = i2s.w8a8_mul_mat_grouped(problems, M)
    assert i2s.read_status(ws) == 0
    for p, ref in zip(problems, refs):
        same_bits(host(p[5]), ref)
