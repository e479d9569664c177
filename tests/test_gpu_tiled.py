"""Tiled I2_S weights (i2s_tile_weights) on the GPU.

The tiling kernel's bytes against the layout's numpy restatement, and the
grouped matmul on tiled weights against the same call on the I2_S bytes and
against the CPU oracle, bit for bit: the decode GEMV (M <= 16, split-K and
ragged tiles), the prefill GEMM, groups that mix the two layouts, the fused
decode launch, the host-buffer call (staged and mapped), the quantize and run
phases with repeated runs, the single-matrix call, and the accumulator
headroom case.
"""

import numpy as np
import pytest

import oracle
from int8_quantized_matmul_gb300 import synth
from tests import tiled_layout

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


def weights(o, N, K, seed):
    return o.i2s_pack(synth.codes(N, K, seed=seed), float(synth.uniform_f32(1, seed + 7, 0.01, 0.1)[0]))


# ragged rows (N % 128, an odd count of 128-row blocks), row bytes that end
# inside a 512-position block (K % 512 = 128, 384), a split-K shape
SHAPES = [(1, 128), (70, 640), (300, 1152), (256, 1536), (257, 1920), (900, 4608), (1536, 8960)]


@pytest.mark.parametrize("N,K", SHAPES + [(8960, 1536)])
def test_tile_weights_bytes(i2s, o, N, K):
    packed = weights(o, N, K, seed=N + K)
    t = i2s.tile_weights(dev(packed), N, K)
    assert t.data.numel() == i2s.i2s_tiled_nbytes(N, K)
    np.testing.assert_array_equal(host(t.data), tiled_layout.tile(packed, N, K))


def run_group(i2s, specs, M, tiled, seed, host_call=False, fused=False):
    """specs: [(N, K, act)]; problems with the same act share x. tiled: one
    flag per problem. Returns the outputs and the weights' packed bytes."""
    o = oracle.get()
    xs, packs, probs, ys = {}, [], [], []
    for i, (N, K, act) in enumerate(specs):
        if act not in xs:
            xs[act] = synth.normal_f32((M, K), seed=seed + 100 * act, outlier_p=0.01)
        packed = weights(o, N, K, seed=seed + 7 * i)
        packs.append(packed)
        w = dev(packed)
        if tiled[i]:
            w = i2s.tile_weights(w, N, K)
        ys.append(torch.full((M, N), float("nan"), dtype=torch.float32, device="cpu" if host_call else "cuda"))
        probs.append([w, N, K, act])
    xd = {a: (torch.from_numpy(x) if host_call else dev(x)) for a, x in xs.items()}
    problems = [(w, N, K, xd[act], y) for (w, N, K, act), y in zip(probs, ys)]
    if host_call:
        i2s.i2s_mul_mat_grouped_host(problems, M)
    elif fused:
        ws = i2s.i2s_mul_mat_grouped_fused(problems, M)
        assert i2s.read_status(ws) == 0
    else:
        ws = i2s.i2s_mul_mat_grouped(problems, M)
        assert i2s.read_status(ws) == 0
    torch.cuda.synchronize()
    return [y.cpu().numpy() if y.is_cuda else y.numpy() for y in ys], packs, xs


GROUP = [(300, 1152, 0), (256, 1536, 1), (1536, 8960, 2), (70, 640, 3), (900, 4608, 4), (257, 1920, 5),
         (128, 1536, 1)]


@pytest.mark.parametrize("M", [1, 8, 9, 16, 64, 200])
def test_tiled_group_matches_i2s_and_oracle(i2s, o, M):
    n = len(GROUP)
    got, packs, xs = run_group(i2s, GROUP, M, [True] * n, seed=M)
    ref, _, _ = run_group(i2s, GROUP, M, [False] * n, seed=M)
    for (N, K, act), g, r, packed in zip(GROUP, got, ref, packs):
        same_bits(g, r)
        same_bits(g, o.i2s_mul_mat(packed, N, K, xs[act], nth=8))


@pytest.mark.parametrize("M", [8, 100])
def test_mixed_layouts_in_one_group(i2s, o, M):
    flags = [i % 2 == 0 for i in range(len(GROUP))]
    got, packs, xs = run_group(i2s, GROUP, M, flags, seed=3 * M)
    for (N, K, act), g, packed in zip(GROUP, got, packs):
        same_bits(g, o.i2s_mul_mat(packed, N, K, xs[act], nth=8))


@pytest.mark.parametrize("M", [1, 16])
def test_tiled_fused_launch(i2s, o, M):
    flags = [i != 2 for i in range(len(GROUP))]
    got, packs, xs = run_group(i2s, GROUP, M, flags, seed=5 * M, fused=True)
    for (N, K, act), g, packed in zip(GROUP, got, packs):
        same_bits(g, o.i2s_mul_mat(packed, N, K, xs[act], nth=8))


@pytest.mark.parametrize("M", [8, 64])
def test_tiled_host_call(i2s, o, M):
    specs = GROUP[:4]
    got, packs, xs = run_group(i2s, specs, M, [True] * len(specs), seed=11 * M, host_call=True)
    for (N, K, act), g, packed in zip(specs, got, packs):
        same_bits(g, o.i2s_mul_mat(packed, N, K, xs[act], nth=8))


@pytest.mark.parametrize("M", [1, 8, 16, 64])
def test_tiled_headroom_k8960(i2s, o, M):
    # every code 2 (+1) and every activation quantized to 127: the largest
    # dot products the format allows, on the decode GEMV and the GEMM
    N, K = 384, 8960
    packed = o.i2s_pack(np.full((N, K), 2, np.uint8), 0.03125)
    x = np.ones((M, K), np.float32)
    w = i2s.tile_weights(dev(packed), N, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = i2s.i2s_mul_mat_grouped([(w, N, K, dev(x), y)], M)
    assert i2s.read_status(ws) == 0
    same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=8))


@pytest.mark.parametrize("M", [1, 8, 64])
def test_tiled_group_phases_repeated(i2s, o, M):
    # the bench's form: one quantization, then the run phase several times,
    # each leaving the split-K state at zero for the next
    specs = GROUP
    xs, packs, problems = {}, [], []
    for i, (N, K, act) in enumerate(specs):
        if act not in xs:
            xs[act] = synth.normal_f32((M, K), seed=70 + act + M, outlier_p=0.01)
        packed = weights(o, N, K, seed=90 + i)
        packs.append(packed)
        problems.append((i2s.tile_weights(dev(packed), N, K), N, K, act))
    xd = {a: dev(x) for a, x in xs.items()}
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for N, _, _ in specs]
    g = i2s.Group([(w, N, K, xd[act], y) for (w, N, K, act), y in zip(problems, ys)], M)
    g.quantize()
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        g.run()
        assert i2s.read_status(g.ws) == 0
        for (N, K, act), y, packed in zip(specs, ys, packs):
            same_bits(host(y), o.i2s_mul_mat(packed, N, K, xs[act], nth=8))


@pytest.mark.parametrize("mapped", [True, "y"])
def test_tiled_host_call_mapped(i2s, o, mapped):
    # pinned host activations and outputs read and written in place by the kernels
    M = 8
    specs = GROUP[:4]
    xs, packs, problems, ys = {}, [], [], []
    for i, (N, K, act) in enumerate(specs):
        if act not in xs:
            xs[act] = torch.from_numpy(synth.normal_f32((M, K), seed=40 + act, outlier_p=0.01)).pin_memory()
        packed = weights(o, N, K, seed=60 + i)
        packs.append(packed)
        y = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
        ys.append(y)
        problems.append((i2s.tile_weights(dev(packed), N, K), N, K, xs[act], y))
    h = i2s.HostGroup(problems, M, mapped=mapped)
    h()
    torch.cuda.synchronize()
    assert i2s.read_status(h.ws) == 0
    for (N, K, act), y, packed in zip(specs, ys, packs):
        same_bits(y.numpy(), o.i2s_mul_mat(packed, N, K, xs[act].numpy(), nth=8))


@pytest.mark.parametrize("path,grid", [(0, 0), (3, 0), (2, 0), (3, 40)])
@pytest.mark.parametrize("M", [1, 9, 16, 64])
def test_tiled_single_call(i2s, o, path, grid, M):
    # i2s_mul_mat_ex with I2S_LAYOUT_TILED in its config: automatic, GEMV and
    # GEMM paths, and a GEMV grid smaller than the SMs
    if path == 3 and M > 16:
        pytest.skip("the GEMV takes M <= 16")
    N, K = 900, 4608
    packed = weights(o, N, K, seed=M + path)
    x = synth.normal_f32((M, K), seed=M * 3 + path, outlier_p=0.01)
    y = i2s.i2s_mul_mat(i2s.tile_weights(dev(packed), N, K), N, K, dev(x), path=path, grid_ctas=grid)
    same_bits(host(y), o.i2s_mul_mat(packed, N, K, x, nth=8))
