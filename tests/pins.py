"""Pins of the CPU oracle against facts that do not come from the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError if
the oracle disagrees with the pages or with mathematics. The pins use:
  * hand-derived fixtures under tests/golden/ (each cites its page section);
  * closed forms (accumulator headroom, degenerate scales);
  * special cases that reduce to numpy's int64 matmul (power-of-two scales make
    every float step exact, so the I2_S/I8_S result must equal an integer
    matmul times a power of two);
  * brute force (the code identity on single-group rows; exhaustive rounding).
They are run against the shipped oracle (test_oracle_pins.py) and against
builds with one planted mistake each (test_oracle_mutations.py).
"""

from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

from int8_quantized_matmul_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

F32_1E5 = Fraction(float(np.float32(1e-5)))   # binary32 value nearest to 1e-5


# ---------------------------------------------------------------------------
# fixture helpers
# ---------------------------------------------------------------------------

def nearest_f32(fr: Fraction) -> np.float32:
    """The binary32 value nearest to an exact rational (ties to even)."""
    c = np.float32(float(fr))
    best = c
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        d_best = abs(Fraction(float(best)) - fr)
        d_cand = abs(Fraction(float(cand)) - fr)
        if d_cand < d_best:
            best = cand
    return np.float32(best)


def parse_rational(tok: str) -> Fraction:
    if tok.startswith("f32(1e-5)/"):
        return F32_1E5 / int(tok.split("/")[1])
    p, q = tok.split("/")
    return Fraction(int(p), int(q))


def load_cases(name: str):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            else:
                cur[key] = vals
    return cases


def load_group_fixture():
    out = {}
    with open(os.path.join(GOLDEN, "i2s_group_decode.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def f32_bits(x) -> int:
    return int(np.asarray(x, dtype=np.float32).view(np.uint32))


# ---------------------------------------------------------------------------
# I2_S layout
# ---------------------------------------------------------------------------

def _crafted_group(filler: int, gp: int, marker: int) -> np.ndarray:
    g = np.full(32, filler, dtype=np.uint8)
    g[gp] = marker
    return g


def pin_i2s_hand_decode(o):
    fx = load_group_fixture()
    filler = int(fx["filler"][0], 16)
    for mk, ck in (("marker", "marker_codes"), ("marker2", "marker2_codes")):
        marker = int(fx[mk][0], 16)
        mcodes = [int(v) for v in fx[ck]]
        for gp in range(32):
            packed = np.concatenate([_crafted_group(filler, gp, marker), np.zeros(32, np.uint8)])
            codes, _ = o.i2s_unpack(packed, 1, 128)
            want = np.ones(128, dtype=np.uint8)
            for slot in range(4):
                want[32 * slot + gp] = mcodes[slot]
            assert np.array_equal(codes[0], want), f"decode of marker at gp={gp}"


def pin_i2s_hand_pack(o):
    fx = load_group_fixture()
    filler = int(fx["filler"][0], 16)
    marker = int(fx["marker"][0], 16)
    mcodes = [int(v) for v in fx["marker_codes"]]
    for gp in range(32):
        codes = np.ones((1, 128), dtype=np.uint8)
        for slot in range(4):
            codes[0, 32 * slot + gp] = mcodes[slot]
        packed = o.i2s_pack(codes, 0.25)
        assert np.array_equal(packed[:32], _crafted_group(filler, gp, marker)), f"pack gp={gp}"


def pin_i2s_layout_sizes(o):
    # 2 bits per value, row stride K/4 bytes, then the 32-byte scale trailer.
    for N, K in ((1, 128), (3, 1024), (70, 1152), (256, 1536)):
        assert o.i2s_nbytes(N, K) == N * K // 4 + 32
        assert o.i2s_scale_offset(N, K) == N * K // 4
    # A 2-row tensor: the second row starts K/4 bytes in, and the scale sits
    # right after the payload followed by 28 zero bytes.
    K = 256
    codes = np.ones((2, K), dtype=np.uint8)
    codes[1, 0] = 2
    packed = o.i2s_pack(codes, 0.75)
    assert packed[K // 4] == 0x95 and packed[0] == 0x55
    assert np.frombuffer(packed[2 * K // 4: 2 * K // 4 + 4].tobytes(), np.float32)[0] == 0.75
    assert not packed[2 * K // 4 + 4:].any()


def pin_i2s_roundtrip(o):
    c = synth.codes(5, 1152, seed=11)
    packed = o.i2s_pack(c, 0.125)
    c2, a = o.i2s_unpack(packed, 5, 1152)
    assert np.array_equal(c, c2) and a == 0.125
    w = o.i2s_dequantize(packed, 5, 1152)
    assert np.array_equal(w, (c.astype(np.float32) - 1.0) * np.float32(0.125))


# ---------------------------------------------------------------------------
# quantizer
# ---------------------------------------------------------------------------

def pin_quant_golden(o):
    for case in load_cases("quant_rows.txt"):
        x = np.array([float(Fraction(v)) for v in case["x"]], dtype=np.float32)[None, :]
        q, s, rs = o.quantize_rows(x)
        want_q = np.array([int(v) for v in case["q"]], dtype=np.int8)
        assert np.array_equal(q[0], want_q), (case["name"], q[0], want_q)
        assert int(rs[0]) == int(case["sum"][0]), case["name"]
        want_s = nearest_f32(parse_rational(case["scale"][0]))
        assert f32_bits(s[0]) == f32_bits(want_s), (case["name"], s[0], want_s)


def pin_quant_rows_independent(o):
    # Rows are quantized independently: stacking the golden rows (zero padded
    # to one width) gives each row its own scale.
    cases = [c for c in load_cases("quant_rows.txt")]
    width = max(len(c["x"]) for c in cases)
    x = np.zeros((len(cases), width), dtype=np.float32)
    for i, c in enumerate(cases):
        x[i, :len(c["x"])] = [float(Fraction(v)) for v in c["x"]]
    q, s, rs = o.quantize_rows(x)
    for i, c in enumerate(cases):
        n = len(c["q"])
        assert np.array_equal(q[i, :n], np.array([int(v) for v in c["q"]], np.int8)), c["name"]
        assert f32_bits(s[i]) == f32_bits(nearest_f32(parse_rational(c["scale"][0])))


def pin_round_exhaustive(o):
    # Every binary32 in [0.25, 8) (all halfway points of small integers), both
    # signs, plus +-2048 ulps around every k + 0.5 for k < 128; compared with
    # the definition "nearest, halfway away from zero" evaluated exactly in
    # float64 (|v| + 0.5 is exact in float64 for binary32 v).
    lo = np.float32(0.25).view(np.uint32)
    hi = np.float32(8.0).view(np.uint32)
    bits = np.arange(lo, hi, dtype=np.uint32)
    halves = np.float32(np.arange(128) + 0.5).view(np.uint32).astype(np.int64)
    around = (halves[:, None] + np.arange(-2048, 2049)[None, :]).reshape(-1).astype(np.uint32)
    v = np.concatenate([bits, around]).view(np.float32)
    v = np.concatenate([v, -v, np.array([0.0, -0.0, 127.49999, 127.5, 126.5], np.float32)])
    got = o.round_array(v)
    ref = (np.floor(np.abs(v.astype(np.float64)) + 0.5) * np.sign(v)).astype(np.float32)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (v[bad[:5]], got[bad[:5]], ref[bad[:5]])


# ---------------------------------------------------------------------------
# I2_S matmul
# ---------------------------------------------------------------------------

def _pow2_activations(M, K, seed, exps):
    """x[m] = integers in [-127,127] times 2^e_m, with one entry at +-127*2^e_m.

    For such rows amax = 127*2^e, so scale = 2^e and inv = 2^-e are exact and
    the quantized row is exactly the integer row.
    """
    g = synth.rng(seed)
    qi = g.integers(-127, 128, size=(M, K)).astype(np.int64)
    j = g.integers(0, K, size=M)
    sgn = g.choice([-1, 1], size=M)
    qi[np.arange(M), j] = 127 * sgn
    x = (qi * (2.0 ** np.asarray(exps, dtype=np.float64))[:, None]).astype(np.float32)
    return x, qi


def pin_i2s_pow2_special_case(o):
    # With w_scale = 2^-1 and row scales 2^e_m every float step is exact, so
    #   y[m, n] = sum_k (code[n,k] - 1) * q[m,k] * 2^(e_m - 1)
    # must equal numpy's int64 matmul. Grid: the page's K x N test grid.
    for K in (128, 1024, 1152):
        for N in (1, 2, 64, 70, 100):
            M = 3
            exps = [-3, 0, 2]
            c = synth.codes(N, K, seed=K * 1000 + N)
            x, qi = _pow2_activations(M, K, seed=K + N, exps=exps)
            packed = o.i2s_pack(c, 0.5)
            ref = (qi @ (c.astype(np.int64) - 1).T).astype(np.float64)
            ref = (ref * (2.0 ** (np.asarray(exps, np.float64) - 1.0))[:, None]).astype(np.float32)
            for nth in (1, 4):
                y = o.i2s_mul_mat(packed, N, K, x, nth=nth)
                assert np.array_equal(y, ref), (K, N, nth)


def pin_i2s_batched_rows(o):
    # A 3-D activation (2 x 4 x K) flattened to 8 rows gives the same rows as
    # running each 4-row slice alone (rows are independent).
    K, N = 1024, 70
    c = synth.codes(N, K, seed=5)
    packed = o.i2s_pack(c, 0.05)
    x = synth.normal_f32((2, 4, K), seed=6)
    y_all = o.i2s_mul_mat(packed, N, K, x.reshape(8, K))
    for b in range(2):
        assert np.array_equal(y_all[4 * b:4 * b + 4], o.i2s_mul_mat(packed, N, K, x[b]))


def pin_i2s_code_identity(o):
    # sum(code*q) = sum(w*q) + sum(q) on single-group rows, by brute force.
    K, N, M = 128, 64, 16
    c = synth.codes(N, K, seed=21)
    x, qi = _pow2_activations(M, K, seed=22, exps=[0] * M)
    packed = o.i2s_pack(c, 1.0)
    y, q, s, rs, dot = o.i2s_mul_mat(packed, N, K, x, want_sidecar=True)
    assert np.array_equal(q.astype(np.int64), qi)
    assert np.array_equal(rs.astype(np.int64), qi.sum(axis=1))
    code_q = qi @ c.astype(np.int64).T
    w_q = qi @ (c.astype(np.int64) - 1).T
    assert np.array_equal(dot.astype(np.int64), code_q)
    assert np.array_equal(dot.astype(np.int64) - rs.astype(np.int64)[:, None], w_q)


def pin_i2s_headroom(o):
    # Every code 2 and every activation quantizing to +127 (x = 127, so
    # scale = 1): dot = 254 K, row_sum = 127 K, y = 127 K * w_scale exactly.
    K, N, M = 8960, 8, 2
    c = np.full((N, K), 2, dtype=np.uint8)
    x = np.full((M, K), 127.0, dtype=np.float32)
    for w_scale, want in ((1.0, 127.0 * K), (0.25, 127.0 * K / 4)):
        packed = o.i2s_pack(c, w_scale)
        y, q, s, rs, dot = o.i2s_mul_mat(packed, N, K, x, want_sidecar=True)
        assert (q == 127).all() and (s == 1.0).all()
        assert (dot == 254 * K).all() and (rs == 127 * K).all()
        assert (y == np.float32(want)).all(), (y[0, 0], want)


def pin_i2s_degenerate(o):
    # All-zero weight tensor (codes 1, scale 0) -> exact zeros; a zeroed
    # activation row -> an exact-zero output row; never NaN.
    K, N, M = 1024, 70, 4
    x = synth.normal_f32((M, K), seed=31)
    x[2] = 0.0
    zero_w = o.i2s_pack(np.ones((N, K), np.uint8), 0.0)
    y = o.i2s_mul_mat(zero_w, N, K, x)
    assert not np.isnan(y).any() and (y == 0).all()
    packed = o.i2s_pack(synth.codes(N, K, seed=32), 0.05)
    y, q, s, rs, _ = o.i2s_mul_mat(packed, N, K, x, want_sidecar=True)
    assert not np.isnan(y).any()
    assert (y[2] == 0).all() and (q[2] == 0).all() and rs[2] == 0
    assert f32_bits(s[2]) == f32_bits(nearest_f32(F32_1E5 / 127))
    assert (y[[0, 1, 3]] != 0).any()


def pin_thread_count_independence(o):
    K, N, M = 1152, 300, 7
    packed = o.i2s_pack(synth.codes(N, K, seed=41), 0.03)
    x = synth.normal_f32((M, K), seed=42, outlier_p=0.01)
    y1 = o.i2s_mul_mat(packed, N, K, x, nth=1)
    for nth in (2, 4, 7):
        assert np.array_equal(y1.view(np.uint32), o.i2s_mul_mat(packed, N, K, x, nth=nth).view(np.uint32))


# ---------------------------------------------------------------------------
# I8_S
# ---------------------------------------------------------------------------

def pin_i8s_layout(o):
    for n, want in ((1, 64), (32, 64), (33, 96), (900 * 2048, 900 * 2048 + 32)):
        assert o.i8s_nbytes(n) == want
        assert o.i8s_scale_offset(n) == want - 32
    q = np.arange(-20, 13, dtype=np.int8)            # 33 values
    packed = o.i8s_pack(q, 0.5)
    assert np.array_equal(packed[:33].view(np.int8), q)
    assert not packed[33:64].any()
    assert np.frombuffer(packed[64:68].tobytes(), np.float32)[0] == 0.5
    assert not packed[68:].any()
    q2, s2 = o.i8s_unpack(packed, 33)
    assert np.array_equal(q2, q) and s2 == 0.5
    assert np.array_equal(o.i8s_dequantize(packed, 33), q.astype(np.float32) * np.float32(0.5))


def pin_i8s_requant_golden(o):
    for case in load_cases("i8s_requant.txt"):
        y = np.array([float(Fraction(v)) for v in case["y"]], dtype=np.float32)
        packed = o.i8s_quantize(y)
        q, s = o.i8s_unpack(packed, y.size)
        assert np.array_equal(q, np.array([int(v) for v in case["q"]], np.int8)), case["name"]
        assert f32_bits(s) == f32_bits(nearest_f32(parse_rational(case["scale"][0]))), case["name"]
    z = o.i8s_quantize(np.zeros(100, np.float32))
    assert not np.isnan(o.i8s_dequantize(z, 100)).any()
    assert (o.i8s_dequantize(z, 100) == 0).all()


def pin_i8s_mul_mat_add_special_case(o):
    # w_scale = 2^-1, x_scale = 2^-2, bias on the 2^-3 grid, small integers:
    # every float step is exact, so y = (W X^T)^T / 8 + bias (then ReLU) must
    # equal numpy's int64 matmul exactly.
    g = synth.rng(51)
    for (M, N, K) in ((3, 5, 64), (17, 70, 200), (8, 33, 2048)):
        W = g.integers(-7, 8, size=(N, K)).astype(np.int8)
        X = g.integers(-7, 8, size=(M, K)).astype(np.int8)
        bias = (g.integers(-32, 33, size=N) / 8.0).astype(np.float32)
        wp = o.i8s_pack(W, 0.5)
        xp = o.i8s_pack(X, 0.25)
        acc = X.astype(np.int64) @ W.astype(np.int64).T
        for relu in (False, True):
            for b in (None, bias):
                ref = acc.astype(np.float64) / 8.0
                if b is not None:
                    ref = ref + b.astype(np.float64)[None, :]
                if relu:
                    ref = np.maximum(ref, 0.0)
                y8, yf = o.i8s_mul_mat_add(wp, N, K, xp, M, bias=b, relu=relu, nth=3)
                assert np.array_equal(yf, ref.astype(np.float32)), (M, N, K, relu, b is None)
                # the op requantizes its own F32 output, one scale per tensor
                assert np.array_equal(y8, o.i8s_quantize(yf))


def pin_i8s_permute_cont(o):
    a, b = 5, 7
    q = synth.int8_normal((a, b), seed=61)
    packed = o.i8s_pack(q, 0.37)
    t = o.i8s_permute_cont(packed, a, b)
    off_src, off_dst = o.i8s_scale_offset(a * b), o.i8s_scale_offset(a * b)
    assert np.array_equal(t[off_dst:off_dst + 32], packed[off_src:off_src + 32])
    deq = o.i8s_dequantize(packed, a * b).reshape(a, b)
    assert np.array_equal(o.i8s_dequantize(t, a * b).reshape(b, a), deq.T)


def pin_i8s_add_scaled_pow2(o):
    # scales 2^-1 and 2^-3: qa/2 + qb/8 is exact in float, so numpy's float64
    # sum rounded to float32 is the exact result; the op then requantizes it
    for n in (1, 33, 4096, 100003):
        qa = synth.int8_normal(n, seed=71)
        qb = synth.int8_normal(n, seed=72)
        a, b = o.i8s_pack(qa, 0.5), o.i8s_pack(qb, 0.125)
        y8, yf = o.i8s_add_scaled(a, b, n)
        ref = qa.astype(np.float64) / 2.0 + qb.astype(np.float64) / 8.0
        assert np.array_equal(yf, ref.astype(np.float32)), n
        assert np.array_equal(y8, o.i8s_quantize(yf)), n
        # addition is commutative, scales included
        assert np.array_equal(o.i8s_add_scaled(b, a, n)[0], y8), n


def pin_i8s_rms_norm_closed_forms(o):
    # (1) constant rows, eps = 0, power-of-two scale and |c|: x = c*s, the mean
    #     square is (c*s)^2 exactly, so every output is sign(c) * 1 exactly
    cs = np.array([1, -1, 2, -4, 64, -64, 8, 16], dtype=np.int8)
    ne0 = 48
    q = np.repeat(cs[:, None], ne0, axis=1)
    y8, yf = o.i8s_rms_norm_scaled(o.i8s_pack(q, 0.125), len(cs), ne0, eps=0.0)
    assert np.array_equal(yf, np.sign(q).astype(np.float32))
    # ... and the requantized tensor is +-127 with scale 1/127
    qq, sc = o.i8s_unpack(y8, q.size)
    assert np.array_equal(qq.reshape(q.shape), (127 * np.sign(q)).astype(np.int8))
    assert sc == np.float32(1.0) / np.float32(127.0)
    # (2) with eps = 0 the result does not depend on a power-of-two input scale
    g = synth.rng(73)
    q = g.integers(-127, 128, size=(9, 70)).astype(np.int8)
    q[:, 0] = 5   # no all-zero row
    ya = o.i8s_rms_norm_scaled(o.i8s_pack(q, 0.5), 9, 70, eps=0.0)[1]
    yb = o.i8s_rms_norm_scaled(o.i8s_pack(q, 4.0), 9, 70, eps=0.0)[1]
    assert np.array_equal(ya, yb)
    # (3) rows come out with unit RMS (eps far below the mean square)
    q = synth.int8_normal((16, 64), seed=74)
    q[:, 0] = 100
    yf = o.i8s_rms_norm_scaled(o.i8s_pack(q, 0.05), 16, 64, eps=1e-5)[1].astype(np.float64)
    rms = np.sqrt((yf * yf).mean(axis=1))
    assert np.all(np.abs(rms - 1.0) < 1e-5), rms
    # (4) an all-zero row stays zero (eps keeps the factor finite)
    q = np.zeros((3, 32), dtype=np.int8)
    q[1] = 9
    yf = o.i8s_rms_norm_scaled(o.i8s_pack(q, 0.3), 3, 32, eps=1e-5)[1]
    assert np.all(yf[0] == 0) and np.all(yf[2] == 0) and np.all(yf[1] > 0)
    # (5) a power-of-two weight per feature scales the outputs exactly
    q = synth.int8_normal((5, 40), seed=75)
    q[:, 0] = 50
    gamma = (2.0 ** synth.rng(76).integers(-3, 4, size=40)).astype(np.float32)
    y0 = o.i8s_rms_norm_scaled(o.i8s_pack(q, 0.07), 5, 40)[1]
    yg = o.i8s_rms_norm_scaled(o.i8s_pack(q, 0.07), 5, 40, gamma=gamma)[1]
    assert np.array_equal(yg, y0 * gamma[None, :])


def pin_i8s_im2col_asym(o):
    g = synth.rng(77)
    for (C, L, KW, stride, pad_l, pad_r) in ((3, 20, 4, 1, 3, 0), (5, 37, 7, 2, 5, 0), (2, 16, 8, 4, 4, 0),
                                             (4, 29, 3, 3, 0, 2), (1, 5, 7, 1, 6, 1), (6, 64, 5, 5, 0, 0)):
        X = g.integers(-127, 128, size=(C, L)).astype(np.int8)
        packed = o.i8s_pack(X, 0.0625)
        dst, OL = o.i8s_im2col_asym(packed, C, L, KW, stride, pad_l, pad_r)
        xp = np.pad(X, ((0, 0), (pad_l, pad_r)))
        starts = list(range(0, xp.shape[1] - KW + 1, stride))
        assert OL == len(starts), (OL, len(starts))
        ref = np.stack([xp[:, t:t + KW].reshape(-1) for t in starts]) if starts else np.zeros((0, C * KW), np.int8)
        n = OL * C * KW
        assert np.array_equal(dst[:n].view(np.int8), ref.reshape(-1))
        off_s, off_d = o.i8s_scale_offset(C * L), o.i8s_scale_offset(n)
        assert np.array_equal(dst[off_d:off_d + 32], packed[off_s:off_s + 32])
    # causal geometry (left pad KW - stride, right pad 0): one output per
    # stride step, and output t sees no input past t*stride + stride - 1
    C, L, KW, stride = 2, 40, 8, 4
    X = np.zeros((C, L), dtype=np.int8)
    X[:, 21] = 7
    dst, OL = o.i8s_im2col_asym(o.i8s_pack(X, 1.0), C, L, KW, stride, KW - stride, 0)
    assert OL == L // stride
    cols = dst[:OL * C * KW].view(np.int8).reshape(OL, C, KW)
    first = min(t for t in range(OL) if cols[t].any())
    assert first * stride + stride - 1 >= 21 and (first - 1) * stride + stride - 1 < 21


def pin_i8s_depthwise_pow2(o):
    # w_scale 2^-1, x_scale 2^-2, bias on the 2^-3 grid: y = acc/8 + bias
    # exactly; acc is numpy's per-channel correlation of the padded input
    g = synth.rng(78)
    for (C, L, KW, stride, pad_l, pad_r) in ((4, 30, 7, 1, 6, 0), (3, 41, 7, 2, 5, 0), (8, 64, 3, 1, 1, 1)):
        W = g.integers(-20, 21, size=(C, KW)).astype(np.int8)
        X = g.integers(-127, 128, size=(C, L)).astype(np.int8)
        bias = (g.integers(-64, 65, size=C) / 8.0).astype(np.float32)
        wp, xp8 = o.i8s_pack(W, 0.5), o.i8s_pack(X, 0.25)
        xp = np.pad(X.astype(np.int64), ((0, 0), (pad_l, pad_r)))
        acc = np.stack([np.correlate(xp[c], W[c].astype(np.int64), mode="valid")[::stride] for c in range(C)])
        for relu in (False, True):
            y8, yf = o.i8s_depthwise_mul_mat_add(wp, KW, xp8, C, L, stride, pad_l, pad_r, bias=bias, relu=relu)
            ref = acc.astype(np.float64) / 8.0 + bias.astype(np.float64)[:, None]
            if relu:
                ref = np.maximum(ref, 0.0)
            assert yf.shape == ref.shape
            assert np.array_equal(yf, ref.astype(np.float32)), (C, L, relu)
            assert np.array_equal(y8, o.i8s_quantize(yf))


def pin_w8a8_weight_quant(o):
    # amax 127 gives scale exactly 1: the page divides by the scale and rounds
    # with lrintf, so halfway values go to the even neighbour
    w = np.array([[127.0, 2.5, -2.5, 3.5, 0.5, -0.5, 1.5, 126.5, -127.0, 4.4]], dtype=np.float32)
    wq, bs = o.w8a8_quantize_weights(w)
    assert bs[0] == np.float32(1.0)
    assert wq[0].tolist() == [127, 2, -2, 4, 0, 0, 2, 126, -127, 4]
    # an all-zero channel: the 1e-9 floor keeps the scale finite, codes 0
    wq, bs = o.w8a8_quantize_weights(np.zeros((2, 8), dtype=np.float32))
    assert np.all(wq == 0) and np.all(bs == np.float32(1e-9) / np.float32(127.0))


def pin_w8a8_mul_mat_pow2(o):
    # activations q/16 with max |q| = 127 per row: amax = 127/16, so the row
    # scale is exactly 1/16 and the codes are exactly q; weight scales 2^-3:
    # d = C / 128 exactly (|C| < 2^24)
    g = synth.rng(79)
    for (M, N, K) in ((3, 5, 64), (17, 70, 256), (9, 33, 2048)):
        Q = g.integers(-127, 128, size=(M, K)).astype(np.int64)
        Q[:, 0] = 127
        x = (Q / 16.0).astype(np.float32)
        wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
        bs = np.full(N, 0.125, dtype=np.float32)
        d, q, s = o.w8a8_mul_mat(wq, bs, x, nth=2, want_sidecar=True)
        assert np.array_equal(q.astype(np.int64), Q)
        assert np.all(s == np.float32(1.0 / 16.0))
        ref = (Q @ wq.astype(np.int64).T).astype(np.float64) / 128.0
        assert np.array_equal(d, ref.astype(np.float32)), (M, N, K)
    # the page's 1e-9 floor (not the 1e-5 of the I2_S quantizer): a row with
    # amax 1e-7 still uses the full code range
    x = np.zeros((1, 8), dtype=np.float32)
    x[0, 3] = 1e-7
    q, s = o.w8a8_quantize_rows(x)
    assert q[0, 3] == 127 and s[0] == np.float32(1e-7) / np.float32(127.0)


# ---------------------------------------------------------------------------
# epilogue association (non-power-of-two scales)
# ---------------------------------------------------------------------------

def _rle(tokens, conv=float):
    out = []
    for t in tokens:
        v, _, n = t.partition("*")
        out.extend([conv(v)] * (int(n) if n else 1))
    return out


def _hex_f32(tok: str) -> np.float32:
    return np.array([int(tok, 16)], dtype=np.uint32).view(np.float32)[0]


def epilogue_cases():
    return {c["name"]: c for c in load_cases("epilogue_association.txt")}


def pin_i2s_epilogue_association(o):
    # tests/golden/epilogue_association.txt, case i2s_epilogue: the page's
    # (float)(dot - row_sum) * (w_scale * act_scale) worked out by hand for
    # scales where the product order decides the last bit.
    c = epilogue_cases()["i2s_epilogue"]
    K = int(c["K"][0])
    codes = np.array([_rle(c[f"codes{i}"], int) for i in range(3)], dtype=np.uint8)
    x = np.array(_rle(c["x"]), dtype=np.float32)[None, :]
    assert codes.shape == (3, K) and x.shape == (1, K)
    w_scale = _hex_f32(c["w_scale"][0])
    want = np.array([int(v, 16) for v in c["y"]], dtype=np.uint32)
    # the fixture discriminates: the left-to-right order gives other bits
    D = np.array([int(v) for v in c["dot_minus_row_sum"]], dtype=np.float32)
    act_scale = _hex_f32("0x3C010204")
    wrong = ((D * w_scale).astype(np.float32) * act_scale).astype(np.float32)
    assert not np.any(wrong.view(np.uint32) == want)
    packed = o.i2s_pack(codes, float(w_scale))
    y, q, s, rs, dot = o.i2s_mul_mat(packed, 3, K, x, want_sidecar=True)
    assert f32_bits(s[0]) == 0x3C010204 and int(rs[0]) == 8255
    assert np.array_equal(dot[0].astype(np.int64) - int(rs[0]), D.astype(np.int64))
    assert np.array_equal(y[0].view(np.uint32), want), [hex(v) for v in y[0].view(np.uint32)]


def pin_i8s_epilogue_association(o):
    # case i8s_epilogue: (float)acc * (w_scale * x_scale) + bias, by hand
    c = epilogue_cases()["i8s_epilogue"]
    K = int(c["K"][0])
    X = np.array([int(v) for v in c["x"]], dtype=np.int8)[None, :]
    W = np.array([[int(v) for v in c[f"w{i}"]] for i in range(2)], dtype=np.int8)
    bias = np.array([_hex_f32(v) for v in c["bias"]], dtype=np.float32)
    ws, xs = _hex_f32(c["w_scale"][0]), _hex_f32(c["x_scale"][0])
    want = np.array([int(v, 16) for v in c["y"]], dtype=np.uint32)
    acc = (X.astype(np.int64) @ W.astype(np.int64).T)[0]
    assert acc.tolist() == [int(v) for v in c["acc"]]
    wrong = (((acc.astype(np.float32) * ws).astype(np.float32) * xs).astype(np.float32) + bias).astype(np.float32)
    assert not np.any(wrong.view(np.uint32) == want)
    for relu in (False, True):
        _, yf = o.i8s_mul_mat_add(o.i8s_pack(W, float(ws)), 2, K, o.i8s_pack(X, float(xs)), 1, bias=bias,
                                  relu=relu)
        assert np.array_equal(yf[0].view(np.uint32), want), (relu, [hex(v) for v in yf[0].view(np.uint32)])


def pin_w8a8_epilogue_association(o):
    # case w8a8_epilogue: (aScale * bScale) * (float)C, by hand
    c = epilogue_cases()["w8a8_epilogue"]
    K = int(c["K"][0])
    x = np.array([float(v) for v in c["x"]], dtype=np.float32)[None, :]
    wq = np.array([[int(v) for v in c[f"wq{i}"]] for i in range(2)], dtype=np.int8)
    bs = np.array([_hex_f32(v) for v in c["b_scale"]], dtype=np.float32)
    want = np.array([int(v, 16) for v in c["d"]], dtype=np.uint32)
    d, q, s = o.w8a8_mul_mat(wq, bs, x, want_sidecar=True)
    assert q[0].tolist() == [int(v) for v in c["q"]] and f32_bits(s[0]) == 0x3C010204
    acc = (q.astype(np.int64) @ wq.astype(np.int64).T)[0]
    assert acc.tolist() == [int(v) for v in c["acc"]]
    wrong = (s[0] * (bs * acc.astype(np.float32)).astype(np.float32)).astype(np.float32)
    assert not np.any(wrong.view(np.uint32) == want)
    assert np.array_equal(d[0].view(np.uint32), want), [hex(v) for v in d[0].view(np.uint32)]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
