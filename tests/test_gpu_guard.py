"""Guard bands around every output and workspace buffer.

Each device buffer a call writes (its output and its workspace) is a slice of
a larger allocation whose margins hold a known byte pattern. After the call the
margins must be unchanged, so no kernel writes outside the buffers it was
given, and the output must match the CPU oracle bit for bit. The shapes have
ragged edges (N, M and K off the tile sizes) where an out-of-range store would
show. Host buffers of the host-memory call are guarded the same way.
"""

import numpy as np
import pytest

import oracle
from int8_quantized_matmul_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 4096      # bytes on each side; a multiple of 256 keeps the slice's alignment
PATTERN = 0xA5


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


class Guarded:
    """A byte buffer of `nbytes` inside margins of the pattern (device or pinned host)."""

    def __init__(self, nbytes, device="cuda", pinned=False):
        self.n = int(nbytes)
        big = torch.full((self.n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.big = big.pin_memory() if pinned else big
        self.buf = self.big[GUARD:GUARD + self.n]

    def f32(self, *shape):
        return self.buf.view(torch.float32).view(*shape)

    def check(self, what):
        torch.cuda.synchronize()
        h = self.big.cpu().numpy()
        lo, hi = h[:GUARD], h[GUARD + self.n:]
        bad_lo = np.nonzero(lo != PATTERN)[0]
        bad_hi = np.nonzero(hi != PATTERN)[0]
        assert bad_lo.size == 0, f"{what}: {bad_lo.size} bytes written before the buffer, first at -{GUARD - bad_lo[-1]}"
        assert bad_hi.size == 0, f"{what}: {bad_hi.size} bytes written after the buffer, first at +{bad_hi[0]}"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pack_slices(sizes):
    """Offsets of buffers of `sizes` bytes laid out in one allocation, each on a
    16-byte boundary (the outputs' alignment rule); returns (offsets, total)."""
    offs, off = [], 0
    for n in sizes:
        offs.append(off)
        off = (off + n + 15) // 16 * 16
    return offs, off


def check_gaps(g, offs, sizes, what):
    """The bytes between the slices (alignment padding) still hold the pattern."""
    torch.cuda.synchronize()
    h = g.buf.cpu().numpy()
    for o_, n in zip(offs, sizes):
        end = o_ + n
        nxt = min([x for x in offs if x > o_], default=g.n)
        assert (h[end:nxt] == PATTERN).all(), f"{what}: bytes written between slices after offset {end}"


def same_bits(a, b):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.nonzero(a.reshape(-1) != b.reshape(-1))[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}"


@pytest.mark.parametrize("M,N,K", [(1, 300, 1152), (8, 257, 1536), (13, 129, 4608), (40, 300, 1152), (130, 257, 384)])
def test_guard_i2s_mul_mat(i2s, o, M, N, K):
    # M <= 16 runs the GEMV (split-K from K > 1536), larger M the GEMM
    packed = o.i2s_pack(synth.codes(N, K, seed=M + N), 0.04)
    x = synth.normal_f32((M, K), seed=K + M, outlier_p=0.02)
    y = Guarded(4 * M * N)
    ws = Guarded(i2s.i2s_mul_mat_workspace(M, N, K))
    i2s.i2s_mul_mat(dev(packed), N, K, dev(x), y=y.f32(M, N), ws=ws.buf)
    y.check("y")
    ws.check("workspace")
    assert i2s.read_status(ws.buf) == 0
    same_bits(y.f32(M, N).cpu().numpy(), o.i2s_mul_mat(packed, N, K, x, nth=8))


@pytest.mark.parametrize("M", [3, 16, 33])
def test_guard_i2s_grouped(i2s, o, M):
    # five projections, two sharing an activation; every output a slice of one
    # guarded buffer, back to back
    shapes = [(100, 1152, 0), (257, 1152, 0), (33, 384, 1), (500, 768, 2), (1, 128, 3)]
    acts = {0: 1152, 1: 384, 2: 768, 3: 128}
    xs = {a: synth.normal_f32((M, K), seed=70 + a, outlier_p=0.01) for a, K in acts.items()}
    dxs = {a: dev(x) for a, x in xs.items()}
    sizes = [4 * M * N for N, _, _ in shapes]
    offs, total = pack_slices(sizes)
    out = Guarded(total)
    group, keep = [], []
    for i, (N, K, a) in enumerate(shapes):
        packed = o.i2s_pack(synth.codes(N, K, seed=80 + i), 0.02 + 0.01 * i)
        y = out.buf[offs[i]:offs[i] + sizes[i]].view(torch.float32).view(M, N)
        group.append((dev(packed), N, K, dxs[a], y))
        keep.append((packed, N, K, xs[a], y))
    need = i2s.i2s_mul_mat_grouped_workspace(group, M)
    ws = Guarded(need)
    i2s.i2s_mul_mat_grouped(group, M, ws=ws.buf)
    out.check("outputs")
    check_gaps(out, offs, sizes, "outputs")
    ws.check("workspace")
    assert i2s.read_status(ws.buf) == 0
    for packed, N, K, x, y in keep:
        same_bits(y.cpu().numpy(), o.i2s_mul_mat(packed, N, K, x, nth=8))


@pytest.mark.parametrize("M,N,K,relu", [(100, 300, 256, True), (37, 257, 100, False), (161, 513, 1024, True)])
def test_guard_i8s_mul_mat_add(i2s, o, M, N, K, relu):
    W = synth.int8_normal((N, K), seed=N + K)
    wp = o.i8s_pack(W, 0.01)
    xp = o.i8s_quantize(synth.normal_f32((M, K), seed=M + K))
    bias = synth.normal_f32(N, seed=N, std=0.1)
    y = Guarded(i2s.i8s_nbytes(M * N))
    ws = Guarded(i2s.i8s_mul_mat_workspace(M, N, K))
    i2s.i8s_mul_mat_add_relu(dev(wp), N, K, dev(xp), M, bias=dev(bias), relu=relu, y=y.buf, ws=ws.buf)
    y.check("y")
    ws.check("workspace")
    assert i2s.read_status(ws.buf) == 0
    same_bits(y.buf.cpu().numpy(), o.i8s_mul_mat_add(wp, N, K, xp, M, bias=bias, relu=relu, nth=8)[0])


def test_guard_i8s_requant_and_eltwise(i2s, o):
    n = 100003
    yv = synth.normal_f32(n, seed=5, outlier_p=0.01)
    dst = Guarded(i2s.i8s_nbytes(n))
    ws = Guarded(i2s.lib.i8s_requant_workspace(n))
    i2s.i8s_requant(dev(yv), dst=dst.buf, ws=ws.buf)
    dst.check("requant output")
    ws.check("requant workspace")
    same_bits(dst.buf.cpu().numpy(), o.i8s_quantize(yv))

    a = o.i8s_pack(synth.int8_normal(n, seed=6, std=40.0), 0.03)
    b = o.i8s_pack(synth.int8_normal(n, seed=7, std=40.0), 0.05)
    y = Guarded(i2s.i8s_nbytes(n))
    ws = Guarded(i2s.i8s_eltwise_workspace(1))
    i2s.i8s_add_scaled(dev(a), dev(b), n, y=y.buf, ws=ws.buf)
    y.check("add_scaled output")
    ws.check("add_scaled workspace")
    same_bits(y.buf.cpu().numpy(), o.i8s_add_scaled(a, b, n)[0])

    rows, ne0 = 3001, 32
    x = o.i8s_pack(synth.int8_normal(rows * ne0, seed=8, std=40.0), 0.02)
    y = Guarded(i2s.i8s_nbytes(rows * ne0))
    ws = Guarded(i2s.i8s_eltwise_workspace(rows))
    i2s.i8s_rms_norm_scaled(dev(x), rows, ne0, 1e-5, y=y.buf, ws=ws.buf)
    y.check("rms_norm output")
    ws.check("rms_norm workspace")
    same_bits(y.buf.cpu().numpy(), o.i8s_rms_norm_scaled(x, rows, ne0, 1e-5)[0])


def test_guard_layout_ops(i2s, o):
    C, L = 5, 3001
    x = o.i8s_pack(synth.int8_normal(C * L, seed=9, std=40.0), 0.02)
    t = Guarded(i2s.i8s_nbytes(C * L))
    i2s.i8s_transpose(dev(x), C, L, dst=t.buf)
    t.check("transpose output")
    same_bits(t.buf.cpu().numpy(), o.i8s_permute_cont(x, C, L))

    KW, stride, pad_l, pad_r = 4, 2, 2, 1
    OL = i2s.i8s_im2col_out_len(L, KW, stride, pad_l, pad_r)
    col = Guarded(i2s.i8s_nbytes(OL * C * KW))
    i2s.i8s_im2col_asym(dev(x), C, L, KW, stride, pad_l, pad_r, dst=col.buf)
    col.check("im2col output")
    same_bits(col.buf.cpu().numpy(), o.i8s_im2col_asym(x, C, L, KW, stride, pad_l, pad_r)[0])

    KW, stride, pad_l, pad_r = 7, 1, 6, 0
    w = o.i8s_pack(synth.int8_normal(C * KW, seed=10, std=40.0), 0.01)
    bias = synth.normal_f32(C, seed=11, std=0.1)
    OL = i2s.i8s_im2col_out_len(L, KW, stride, pad_l, pad_r)
    y = Guarded(i2s.i8s_nbytes(C * OL))
    ws = Guarded(i2s.i8s_eltwise_workspace(1))
    i2s.i8s_depthwise_mul_mat_add(dev(w), KW, dev(x), C, L, stride, pad_l, pad_r, bias=dev(bias), y=y.buf, ws=ws.buf)
    y.check("depthwise output")
    ws.check("depthwise workspace")
    same_bits(y.buf.cpu().numpy(),
              o.i8s_depthwise_mul_mat_add(w, KW, x, C, L, stride, pad_l, pad_r, bias=bias)[0])


def test_guard_w8a8_grouped(i2s, o):
    M = 37
    shapes = [(70, 256), (257, 1024), (33, 100)]
    problems, keep = [], []
    sizes = [4 * M * N for N, _ in shapes]
    offs, total = pack_slices(sizes)
    out = Guarded(total)
    for i, (N, K) in enumerate(shapes):
        w = synth.normal_f32((N, K), seed=20 + i, std=0.02)
        wq, bs = o.w8a8_quantize_weights(w)
        packed = i2s.w8a8_pack_weights(dev(wq))
        x = synth.normal_f32((M, K), seed=30 + i, outlier_p=0.01)
        d = out.buf[offs[i]:offs[i] + sizes[i]].view(torch.float32).view(M, N)
        problems.append((packed, dev(bs), N, K, dev(x), d))
        keep.append((wq, bs, x, d))
    arr = i2s._w8a8_problems(problems)
    ws = Guarded(int(i2s.lib.w8a8_mul_mat_grouped_workspace(arr, len(problems), M)))
    i2s.w8a8_mul_mat_grouped(problems, M, ws=ws.buf)
    out.check("outputs")
    check_gaps(out, offs, sizes, "outputs")
    ws.check("workspace")
    assert i2s.read_status(ws.buf) == 0
    for wq, bs, x, d in keep:
        same_bits(d.cpu().numpy(), o.w8a8_mul_mat(wq, bs, x, nth=8))


@pytest.mark.parametrize("mapped", [False, "y"])
def test_guard_host_call(i2s, o, mapped):
    # host activations and outputs in guarded pinned buffers, the staging
    # workspace guarded on the device
    M, N, K = 8, 300, 1536
    packed = o.i2s_pack(synth.codes(N, K, seed=41), 0.05)
    xh = Guarded(4 * M * K, device="cpu", pinned=True)
    xh.f32(M, K).copy_(torch.from_numpy(synth.normal_f32((M, K), seed=42, outlier_p=0.01)))
    yh = Guarded(4 * M * N, device="cpu", pinned=True)
    probs = [(dev(packed), N, K, xh.f32(M, K), yh.f32(M, N))]
    need = int(i2s.lib.i2s_mul_mat_grouped_host_workspace(i2s._host_problems(probs), 1, M))
    ws = Guarded(need)
    g = i2s.HostGroup(probs, M, ws=ws.buf, mapped=mapped)
    g()
    torch.cuda.synchronize()
    yh.check("host output")
    xh.check("host activations")
    ws.check("workspace")
    assert i2s.read_status(ws.buf) == 0
    same_bits(yh.f32(M, N).numpy(), o.i2s_mul_mat(packed, N, K, xh.f32(M, K).numpy(), nth=8))


@pytest.mark.parametrize("N,K", [(1, 128), (300, 1152), (257, 1920), (1536, 8960)])
def test_guard_tile_weights_and_tiled_group(i2s, o, N, K):
    # the tiling kernel and its trailer copy write exactly i2s_tiled_nbytes;
    # the grouped GEMV and GEMM on the tiled copy write only their outputs
    from tests import tiled_layout
    packed = o.i2s_pack(synth.codes(N, K, seed=N + K), 0.04)
    gt = Guarded(i2s.i2s_tiled_nbytes(N, K))
    wt = i2s.tile_weights(dev(packed), N, K, out=gt.buf)
    gt.check("i2s_tile_weights")
    np.testing.assert_array_equal(gt.buf.cpu().numpy(), tiled_layout.tile(packed, N, K))
    for M in (3, 40):
        x = synth.normal_f32((M, K), seed=M + N)
        gy = Guarded(M * N * 4)
        y = gy.f32(M, N)
        xd = dev(x)
        gw = Guarded(i2s.i2s_mul_mat_grouped_workspace([(wt, N, K, xd, y)], M))
        i2s.i2s_mul_mat_grouped([(wt, N, K, xd, y)], M, ws=gw.buf)
        assert i2s.read_status(gw.buf) == 0
        gy.check(f"tiled group y, M={M}")
        gw.check(f"tiled group workspace, M={M}")
        np.testing.assert_array_equal(y.cpu().numpy().view(np.uint32), o.i2s_mul_mat(packed, N, K, x, nth=8).view(np.uint32))
