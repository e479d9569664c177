"""i2s_mul_mat_noalloc (fixed library scratch, no workspace) against
i2s_mul_mat (caller workspace) on the same device buffers, and against the CPU
oracle on sampled weight rows of the large decode shapes.

Both GPU entry points run the same arithmetic, so the outputs must agree bit
for bit (the tolerance every I2_S parity test uses). Each case calls the
no-alloc entry point twice in a row, and one test alternates shapes, so every
call after the first starts from the scratch contents the previous call left
behind.
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


def make_problem(i2s, M, N, K, seed):
    """I2_S weights (codes drawn as packed bytes, in-band scale) and M x K
    activations, drawn on the device."""
    w = synth.packed_code_bytes_device(i2s.i2s_nbytes(N, K), seed, "cuda")
    off = i2s.i2s_scale_offset(N, K)
    w[off:] = 0
    scale = torch.tensor([0.05 + 0.01 * (seed % 7)], dtype=torch.float32, device="cuda")
    w[off:off + 4] = scale.view(torch.uint8)
    x = synth.normal_f32_device(M * K, seed + 1, "cuda", outlier_p=0.01).view(M, K)
    return w, x


def need_bytes(M, N, K):
    """Scratch the call needs, by the formula documented with the entry point."""
    up = lambda v: (v + 255) // 256 * 256
    rows = 32 if M <= 8 else 48
    n = 1024 + up(rows * K // 2)
    if K > 1536:
        n += up(4 * M * N) + up(4 * ((N + 127) // 128))
    return n


def bits(t):
    torch.cuda.synchronize()
    return t.cpu().numpy().view(np.uint32)


def noalloc(i2s, w, N, K, x):
    y = torch.full((x.shape[0], N), float("nan"), dtype=torch.float32, device="cuda")
    i2s.i2s_mul_mat_noalloc(w, N, K, x, y)
    # no bounded device wait of the call ran out
    assert i2s.noalloc_read_status() == 0
    return y


@pytest.mark.parametrize("M,N,K", [
    (1, 1536, 1536),     # one K chunk: no split-K partials
    (8, 900, 4608),      # ragged row tile, split-K
    (16, 1536, 8960),    # down-projection shape, split-K with a ragged chunk
    (3, 8960, 1536),     # gate/up shape
    (9, 257, 2048),      # Mp = 16 with M = 9, one row past a tile
])
def test_noalloc_matches_workspace_path(i2s, M, N, K):
    w, x = make_problem(i2s, M, N, K, seed=M * 31 + N + K)
    want = bits(i2s.i2s_mul_mat(w, N, K, x))
    for _ in range(2):
        np.testing.assert_array_equal(bits(noalloc(i2s, w, N, K, x)), want)


def test_noalloc_alternating_shapes(i2s):
    # each call starts from the previous call's partial sums and counters
    shapes = [(16, 2000, 8960), (1, 700, 4608), (4, 151936 // 8, 1536)]
    probs = [make_problem(i2s, M, N, K, seed=100 + i) for i, (M, N, K) in enumerate(shapes)]
    wants = [bits(i2s.i2s_mul_mat(w, N, K, x)) for (w, x), (M, N, K) in zip(probs, shapes)]
    for _ in range(2):
        for (w, x), (M, N, K), want in zip(probs, shapes, wants):
            np.testing.assert_array_equal(bits(noalloc(i2s, w, N, K, x)), want)


def test_noalloc_near_the_scratch_limit(i2s):
    M, N, K = 16, 60000, 8960
    assert need_bytes(M, N, K) <= i2s.NOALLOC_SCRATCH_BYTES
    w, x = make_problem(i2s, M, N, K, seed=7)
    want = bits(i2s.i2s_mul_mat(w, N, K, x))
    for _ in range(2):
        np.testing.assert_array_equal(bits(noalloc(i2s, w, N, K, x)), want)


def test_noalloc_rejects_what_does_not_fit(i2s):
    # rejected on the host before anything is enqueued: y keeps its contents
    M, N, K = 16, 65536, 8960
    assert need_bytes(M, N, K) > i2s.NOALLOC_SCRATCH_BYTES
    w, x = make_problem(i2s, M, N, K, seed=8)
    y = torch.full((M, N), 3.0, dtype=torch.float32, device="cuda")
    rc = i2s.lib.i2s_mul_mat_noalloc(w.data_ptr(), N, K, x.data_ptr(), M, y.data_ptr(), i2s._stream())
    assert rc == -4   # I2S_E_WORKSPACE_TOO_SMALL
    x17 = torch.zeros((17, K), dtype=torch.float32, device="cuda")
    rc = i2s.lib.i2s_mul_mat_noalloc(w.data_ptr(), N, K, x17.data_ptr(), 17, y.data_ptr(), i2s._stream())
    assert rc == -1   # I2S_E_BAD_SHAPE: the no-alloc call covers M <= 16 only
    assert bool((y == 3.0).all())


@pytest.mark.parametrize("M,N,K", [(1, 8960, 1536), (8, 1536, 8960), (16, 151936 // 8, 1536)])
def test_noalloc_against_the_oracle_sampled(i2s, M, N, K):
    # the gate/up, down and (an eighth of) the output-head shapes: 32-row
    # slices of the weights, first, last and two inside, computed by the oracle
    o = oracle.get()
    w, x = make_problem(i2s, M, N, K, seed=M + N + K)
    wh = w.cpu().numpy()
    xh = x.cpu().numpy()
    rb = K // 4
    for _ in range(2):
        y = bits(noalloc(i2s, w, N, K, x)).view(np.float32)
        for n0 in (0, N // 3, (2 * N) // 3, N - 32):
            sub = np.concatenate([wh[n0 * rb:(n0 + 32) * rb], wh[N * rb:N * rb + 32]])
            want = o.i2s_mul_mat(sub, 32, K, xh, nth=8)
            np.testing.assert_array_equal(y[:, n0:n0 + 32].view(np.uint32), want.view(np.uint32))
