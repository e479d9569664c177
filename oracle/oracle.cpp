// Plain CPU oracle for the I2_S ternary x INT8 matmul and the I8_S fused
// mul_mat_add(_relu).
//
// TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct statement
// of what the GPU library computes. Only the test suite, the smoke check and
// the benchmark's CPU-baseline leg load it. It shares no code, header, table or
// helper with the CUDA library, and the library never calls it.
//
// Built with plain gcc/g++ at -O2 -ffp-contract=off and no fast-math, so every
// float operation below is one IEEE-754 binary32 operation, rounded to nearest,
// in the order written (no fused multiply-add).
//
// Sources (web pages; cited by title and section):
//   [P1] "ggml: additive INT8/ternary types, fused CPU ops, and kernels for
//        VibeASR (1/2)" (audio.cpp pull request 447)
//   [P2] "ggml-cpu: ternary I2_S matmul kernel (VibeASR, 3/4)" (audio.cpp pull
//        request 445)
//   [P3] "VibeASR in audio.cpp" (docs/models/vibeasr.md)
//   [P4] "Experiment - int8 W8A8 path" (ork-driver wiki)
//
// Readings where the pages are silent (each is also listed in the design notes):
//   R1 rounding: round to nearest, halfway cases away from zero (C roundf).
//   R2 quantizer arithmetic: amax floored at 1e-5; scale = amax/127 (stored,
//      a multiplier); inv = 127/amax; v = x*inv; q = clamp(round(v), -127, 127).
//   R3 "padded" F32 scale: the payload is padded with zero bytes to a multiple
//      of 32, then the F32 scale, then 28 zero bytes (32-byte trailer).
//   R4 I8_S mul_mat_add: y = (float)acc * (w_scale*x_scale), then + bias[n],
//      then ReLU (y > 0 ? y : +0), then per-tensor requantization (R2).
//   R5 add_scaled: y = (float)qa*sa + (float)qb*sb (two products, one sum),
//      then per-tensor requantization (R2).
//   R6 rms_norm_scaled: rows of ne0 contiguous values x = q*s; mean square
//      ((float)sum(q^2) * (s*s)) / ne0 and row factor r = 1 / sqrt(mean + eps),
//      each an IEEE binary32 operation (the integer sum is exact); y = (x*r)
//      (*gamma[i]); then per-tensor requantization (R2). No weight when gamma
//      is null.
//   R7 im2col_asym: input C x L (L contiguous), output OL x (C*KW) with
//      dst[t][c*KW + k] = src[c][t*stride + k - pad_l] (0 outside [0, L)),
//      OL = (L + pad_l + pad_r - KW) / stride + 1; the scale is carried.
//   R8 depthwise mul_mat_add: per channel, the im2col_asym geometry of R7 on
//      that channel alone, acc in int32, then R4's epilogue with bias[c];
//      output C x OL.
//   R9 W8A8 ([P4]): per-channel weights: amax floored at 1e-9, bscale =
//      amax/127, q = rint(w / bscale) (ties to even, as the page's lrintf)
//      clamped to +-127; per-row activations: amax floored at 1e-9, ascale =
//      amax/127, inv = 127/amax, q = round(x*inv) (R1) clamped; then
//      d = ascale[m] * bscale[n] * (float)C, left to right.
//
// Parity pins: every function here is pinned by tests that do not re-use its
// arithmetic (hand decode, closed forms, brute force, numpy integer matmul in
// special cases); see tests/test_oracle_pins.py.

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <stdio.h>

#include <thread>
#include <vector>

#define ORC_API extern "C" __attribute__((visibility("default")))

// ORC_PLANT selects one deliberate mistake for the mutation test that proves
// the pins can fail (tests/test_oracle_mutations.py builds one library per
// value). The shipped oracle is built with ORC_PLANT == 0: no mistake.
#ifndef ORC_PLANT
#define ORC_PLANT 0
#endif

// ---------------------------------------------------------------------------
// Byte layouts ([P1] "Two new types"; [P2] "Kernels"; [P3] "Decoder")
// ---------------------------------------------------------------------------

static int64_t round_up32(int64_t n) { return (n + 31) / 32 * 32; }

// I2_S: 2 bits per value, so N*K/4 payload bytes (K % 128 == 0 makes this a
// whole number of 32-byte groups), then the 32-byte scale trailer (R3).
ORC_API int64_t orc_i2s_nbytes(int64_t N, int64_t K) { return N * K / 4 + 32; }
ORC_API int64_t orc_i2s_scale_offset(int64_t N, int64_t K) { return N * K / 4; }

// I8_S: nelements int8 bytes, zero padded to 32, then the 32-byte trailer (R3).
ORC_API int64_t orc_i8s_nbytes(int64_t n) { return round_up32(n) + 32; }
ORC_API int64_t orc_i8s_scale_offset(int64_t n) { return round_up32(n); }

static void put_scale(uint8_t* dst, int64_t off, float s) {
    memcpy(dst + off, &s, 4);
    memset(dst + off + 4, 0, 28);
}

static float get_scale(const uint8_t* src, int64_t off) {
    float s;
    memcpy(&s, src + off, 4);
    return s;
}

// ---------------------------------------------------------------------------
// I2_S packing ([P1] "Kernels", [P2] "Kernels"):
// the flat tensor is cut into groups of 128 values, each stored in 32 bytes.
// Byte gp of a group holds the group-relative positions gp, 32+gp, 64+gp and
// 96+gp in its bit pairs at shifts 6, 4, 2 and 0. Codes are {0,1,2} for the
// ternary values {-1,0,+1}.
// ---------------------------------------------------------------------------

// Packer: walks the values in flat order and drops each code into its place.
ORC_API void orc_i2s_pack(const uint8_t* codes, int64_t N, int64_t K, float absmax,
                          uint8_t* dst) {
    const int64_t n_values = N * K;
    memset(dst, 0, (size_t)(n_values / 4));
    for (int64_t f = 0; f < n_values; ++f) {
        const int64_t group = f / 128;
        const int64_t pos = f % 128;            // group-relative position
        const int64_t byte = group * 32 + pos % 32;
#if ORC_PLANT == 2
        const int shift = 2 * (int)(pos / 32);
#else
        const int shift = 6 - 2 * (int)(pos / 32);
#endif
        dst[byte] |= (uint8_t)((codes[f] & 3u) << shift);
    }
    put_scale(dst, orc_i2s_scale_offset(N, K), absmax);
}

// Unpacker, written independently of the packer: walks the bytes of each group
// and the four bit pairs of each byte.
ORC_API void orc_i2s_unpack(const uint8_t* src, int64_t N, int64_t K, uint8_t* codes,
                            float* absmax) {
    const int64_t n_groups = N * K / 128;
    for (int64_t g = 0; g < n_groups; ++g) {
        const uint8_t* grp = src + g * 32;
        uint8_t* out = codes + g * 128;
        for (int gp = 0; gp < 32; ++gp) {
            const uint8_t b = grp[gp];
#if ORC_PLANT == 1
            out[gp] = b & 3;
            out[32 + gp] = (b >> 2) & 3;
            out[64 + gp] = (b >> 4) & 3;
            out[96 + gp] = (b >> 6) & 3;
#else
            out[gp] = (b >> 6) & 3;
            out[32 + gp] = (b >> 4) & 3;
            out[64 + gp] = (b >> 2) & 3;
            out[96 + gp] = b & 3;
#endif
        }
    }
    if (absmax) *absmax = get_scale(src, orc_i2s_scale_offset(N, K));
}

// Dequantizer: w = (code - 1) * absmax ([P3] "Decoder": ternary {-1,0,+1}
// stored as codes {0,1,2} with one F32 absmax after the payload).
ORC_API void orc_i2s_dequantize(const uint8_t* src, int64_t N, int64_t K, float* w) {
    std::vector<uint8_t> c((size_t)(N * K));
    float a;
    orc_i2s_unpack(src, N, K, c.data(), &a);
    for (int64_t i = 0; i < N * K; ++i) w[i] = (float)((int)c[i] - 1) * a;
}

// ---------------------------------------------------------------------------
// Quantization of an F32 block to int8 with one multiplier scale
// ([P1] "Two new types": scale = amax/127, dequantize by multiplying;
//  [P3] "Encoder": amax floored at 1e-5;
//  [P4] "Implementation": scale = amax/127, inv = 127/amax, q = round(x*inv)
//  clamped to +-127). Rounding is R1.
// ---------------------------------------------------------------------------

ORC_API float orc_round(float v) { return roundf(v); }

ORC_API void orc_round_array(const float* v, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = roundf(v[i]);
}

// Quantizes x[0..n) to q with scale; returns the int8 sum in *sum (may be null).
static void quantize_block(const float* x, int64_t n, int8_t* q, float* scale, int32_t* sum) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
#if ORC_PLANT != 6
    if (amax < 1e-5f) amax = 1e-5f;
#endif
#if ORC_PLANT == 4
    const float s = 127.0f / amax;
#else
    const float s = amax / 127.0f;
#endif
    const float inv = 127.0f / amax;
    int64_t acc = 0;
    for (int64_t i = 0; i < n; ++i) {
        const float v = x[i] * inv;
#if ORC_PLANT == 5
        float r = rintf(v);
#else
        float r = roundf(v);
#endif
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)(int)r;
        acc += q[i];
    }
    *scale = s;
    if (sum) *sum = (int32_t)acc;
}

// Per-row activation quantization for the I2_S matmul ([P2] "Arithmetic" and
// "Kernels" threading paragraph; [P1] "Arithmetic is exact where it can be":
// quantized rows, then per-row scale and per-row int8 sum as a sidecar).
ORC_API void orc_quantize_rows(const float* x, int64_t M, int64_t K, int8_t* q,
                               float* act_scale, int32_t* row_sum) {
    for (int64_t m = 0; m < M; ++m)
        quantize_block(x + m * K, K, q + m * K, &act_scale[m], &row_sum[m]);
}

// ---------------------------------------------------------------------------
// I2_S x F32 -> F32 matmul ([P2] "Interface", "Arithmetic", "Kernels").
// W is N x K (K contiguous, row stride K/4 bytes), X is M x K, Y is M x N.
// Phase 1 quantizes activation rows striped over threads; the join is the
// barrier; phase 2 splits the output features in chunks of 64 over threads and
// sweeps the whole batch for each weight row. The result does not depend on
// the thread count.
//
// dot = sum_k code*q (int32), and by the code identity
// sum(code*q) = sum(w*q) + sum(q), the epilogue is
//   y = (float)(dot - row_sum) * (w_scale * act_scale).
// The oracle also forms sum(w*q) directly and aborts if the identity fails.
// ---------------------------------------------------------------------------

struct I2SJob {
    const uint8_t* codes;
    const int8_t* q;
    const float* act_scale;
    const int32_t* row_sum;
    float w_scale;
    int64_t M, N, K;
    float* y;
    int32_t* dot_out;   // optional, M x N raw sum(code*q)
};

static void i2s_features(const I2SJob* j, int tid, int nth) {
    const int64_t chunk = 64;
    const int64_t n_chunks = (j->N + chunk - 1) / chunk;
    for (int64_t c = tid; c < n_chunks; c += nth) {
        const int64_t n_lo = c * chunk;
        const int64_t n_hi = n_lo + chunk < j->N ? n_lo + chunk : j->N;
        for (int64_t n = n_lo; n < n_hi; ++n) {
            const uint8_t* wrow = j->codes + n * j->K;
            for (int64_t m = 0; m < j->M; ++m) {
                const int8_t* qrow = j->q + m * j->K;
                int64_t dot = 0, wq = 0;
                for (int64_t k = 0; k < j->K; ++k) {
                    dot += (int64_t)wrow[k] * qrow[k];
                    wq += (int64_t)((int)wrow[k] - 1) * qrow[k];
                }
                if (dot != wq + j->row_sum[m] || dot > INT32_MAX || dot < INT32_MIN) {
                    fprintf(stderr, "oracle: code identity or int32 range violated\n");
                    abort();
                }
#if ORC_PLANT == 9
                const int32_t d = (int32_t)(int16_t)dot;
#else
                const int32_t d = (int32_t)dot;
#endif
                if (j->dot_out) j->dot_out[m * j->N + n] = d;
#if ORC_PLANT == 3
                const float r = (float)d * (j->w_scale * j->act_scale[m]);
#elif ORC_PLANT == 10
                const float r = (float)(d - j->row_sum[m]) * (j->w_scale * j->act_scale[0]);
#elif ORC_PLANT == 21
                const float r = (float)(d - j->row_sum[m]) * j->w_scale * j->act_scale[m];
#else
                const float r = (float)(d - j->row_sum[m]) * (j->w_scale * j->act_scale[m]);
#endif
#if ORC_PLANT == 7
                j->y[n * j->M + m] = r;
#else
                j->y[m * j->N + n] = r;
#endif
            }
        }
    }
}

ORC_API void orc_i2s_mul_mat(const uint8_t* w_i2s, int64_t N, int64_t K, const float* x,
                             int64_t M, float* y, int nth, int8_t* q_out, float* scale_out,
                             int32_t* row_sum_out, int32_t* dot_out) {
    if (nth < 1) nth = 1;
    std::vector<uint8_t> codes((size_t)(N * K));
    float w_scale;
    orc_i2s_unpack(w_i2s, N, K, codes.data(), &w_scale);
    std::vector<int8_t> q((size_t)(M * K));
    std::vector<float> s((size_t)M);
    std::vector<int32_t> rs((size_t)M);

    // Phase 1: rows striped across threads (a row-wide absmax cannot be split).
    {
        std::vector<std::thread> ts;
        for (int t = 0; t < nth; ++t)
            ts.emplace_back([&, t] {
                for (int64_t m = t; m < M; m += nth)
                    quantize_block(x + m * K, K, q.data() + m * K, &s[m], &rs[m]);
            });
        for (auto& th : ts) th.join();   // the barrier
    }
    // Phase 2: output features split over threads.
    I2SJob job{codes.data(), q.data(), s.data(), rs.data(), w_scale, M, N, K, y, dot_out};
    {
        std::vector<std::thread> ts;
        for (int t = 0; t < nth; ++t) ts.emplace_back([&, t] { i2s_features(&job, t, nth); });
        for (auto& th : ts) th.join();
    }
    if (q_out) memcpy(q_out, q.data(), (size_t)(M * K));
    if (scale_out) memcpy(scale_out, s.data(), (size_t)M * 4);
    if (row_sum_out) memcpy(row_sum_out, rs.data(), (size_t)M * 4);
}

// ---------------------------------------------------------------------------
// I8_S: per-tensor int8 with an in-band multiplier scale ([P1] "Two new types").
// ---------------------------------------------------------------------------

ORC_API void orc_i8s_pack(const int8_t* q, int64_t n, float scale, uint8_t* dst) {
    const int64_t off = orc_i8s_scale_offset(n);
    memset(dst, 0, (size_t)off);
    memcpy(dst, q, (size_t)n);
    put_scale(dst, off, scale);
}

ORC_API float orc_i8s_unpack(const uint8_t* src, int64_t n, int8_t* q) {
    if (q) memcpy(q, src, (size_t)n);
    return get_scale(src, orc_i8s_scale_offset(n));
}

ORC_API void orc_i8s_dequantize(const uint8_t* src, int64_t n, float* out) {
    const float s = get_scale(src, orc_i8s_scale_offset(n));
    const int8_t* q = (const int8_t*)src;
    for (int64_t i = 0; i < n; ++i) out[i] = (float)q[i] * s;
}

// F32 -> I8_S, one scale for the whole tensor ([P1] "Five fused INT8 ops":
// every op requantizes its output; [P3] "Encoder": whole-waveform scale, amax
// floored at 1e-5).
ORC_API void orc_i8s_quantize(const float* y, int64_t n, uint8_t* dst) {
    std::vector<int8_t> q((size_t)n);
    float s;
    quantize_block(y, n, q.data(), &s, nullptr);
    orc_i8s_pack(q.data(), n, s, dst);
}

// ggml_mul_mat_add / ggml_mul_mat_add_relu ([P1] "Five fused INT8 ops"):
// I8_S W (N x K) times I8_S X (M x K) -> I8_S Y (M x N); bias added, optional
// ReLU, output requantized in the op. Formula and order are reading R4.
// y_f32 (optional) receives the F32 values before requantization.
ORC_API void orc_i8s_mul_mat_add(const uint8_t* w_i8s, int64_t N, int64_t K,
                                 const uint8_t* x_i8s, int64_t M, const float* bias,
                                 int relu, uint8_t* y_i8s, float* y_f32, int nth) {
    if (nth < 1) nth = 1;
    const int8_t* w = (const int8_t*)w_i8s;
    const int8_t* xq = (const int8_t*)x_i8s;
    const float ws = get_scale(w_i8s, orc_i8s_scale_offset(N * K));
    const float xs = get_scale(x_i8s, orc_i8s_scale_offset(M * K));
    const float sc = ws * xs;
    std::vector<float> yv((size_t)(M * N));
    std::vector<std::thread> ts;
    for (int t = 0; t < nth; ++t)
        ts.emplace_back([&, t] {
            for (int64_t n = t; n < N; n += nth) {
                for (int64_t m = 0; m < M; ++m) {
                    int64_t acc = 0;
                    for (int64_t k = 0; k < K; ++k) acc += (int64_t)w[n * K + k] * xq[m * K + k];
                    if (acc > INT32_MAX || acc < INT32_MIN) {
                        fprintf(stderr, "oracle: int32 accumulator range violated\n");
                        abort();
                    }
#if ORC_PLANT == 11
                    float v = (float)(int32_t)acc;
                    if (bias) v = v + bias[n];
                    v = v * sc;
#elif ORC_PLANT == 13
                    float v = (float)(int32_t)acc * ws;
                    if (bias) v = v + bias[n];
#elif ORC_PLANT == 22
                    float v = (float)(int32_t)acc * ws * xs;
                    if (bias) v = v + bias[n];
#else
                    float v = (float)(int32_t)acc * sc;
                    if (bias) v = v + bias[n];
#endif
#if ORC_PLANT != 12
                    if (relu) v = v > 0.0f ? v : 0.0f;
#endif
                    yv[m * N + n] = v;
                }
            }
        });
    for (auto& th : ts) th.join();
    if (y_f32) memcpy(y_f32, yv.data(), (size_t)(M * N) * 4);
    orc_i8s_quantize(yv.data(), M * N, y_i8s);
}

// ggml_cont(ggml_permute(...)) of an I8_S tensor: the values move, and the
// in-band scale must travel with them ([P1] "Two new types", dup/cont note).
// src is a x b (row-major); dst is b x a.
ORC_API void orc_i8s_permute_cont(const uint8_t* src, int64_t a, int64_t b, uint8_t* dst) {
    const int64_t n = a * b;
    const int8_t* s = (const int8_t*)src;
    std::vector<int8_t> t((size_t)n);
    for (int64_t i = 0; i < a; ++i)
        for (int64_t j = 0; j < b; ++j) t[j * a + i] = s[i * b + j];
#if ORC_PLANT == 8
    orc_i8s_pack(t.data(), n, 1.0f, dst);
#else
    orc_i8s_pack(t.data(), n, get_scale(src, orc_i8s_scale_offset(n)), dst);
#endif
}

// ---------------------------------------------------------------------------
// ggml_add_scaled ([P1] "Five fused INT8 ops": I8_S + I8_S -> I8_S with the
// two input scales reconciled). Reading R5: both inputs are dequantized (one
// IEEE product each), added (one IEEE sum) and the sum is requantized with one
// scale for the whole tensor. y_f32 (optional) receives the sums.
// ---------------------------------------------------------------------------
ORC_API void orc_i8s_add_scaled(const uint8_t* a_i8s, const uint8_t* b_i8s, int64_t n, uint8_t* y_i8s,
                                float* y_f32) {
    const int8_t* qa = (const int8_t*)a_i8s;
    const int8_t* qb = (const int8_t*)b_i8s;
    const float sa = get_scale(a_i8s, orc_i8s_scale_offset(n));
#if ORC_PLANT == 14
    const float sb = sa;
#else
    const float sb = get_scale(b_i8s, orc_i8s_scale_offset(n));
#endif
    std::vector<float> y((size_t)n);
    for (int64_t i = 0; i < n; ++i) {
        const float va = (float)qa[i] * sa;
        const float vb = (float)qb[i] * sb;
        y[i] = va + vb;
    }
    if (y_f32) memcpy(y_f32, y.data(), (size_t)n * 4);
    orc_i8s_quantize(y.data(), n, y_i8s);
}

// ---------------------------------------------------------------------------
// ggml_rms_norm_scaled ([P1] "Five fused INT8 ops": RMSNorm straight from I8_S
// to I8_S; [P3] "Encoder": RMSNorm epsilon 1e-5 everywhere). Reading R6. The
// mean square of a row of dequantized values q*s is s^2 * sum(q^2) / ne0; the
// integer sum is exact, and the rest is a fixed sequence of correctly rounded
// binary32 operations, so the row factor does not depend on a summation order.
// ---------------------------------------------------------------------------
ORC_API void orc_i8s_rms_norm_scaled(const uint8_t* x_i8s, int64_t rows, int64_t ne0, float eps,
                                     const float* gamma, uint8_t* y_i8s, float* y_f32) {
    const int64_t n = rows * ne0;
    const int8_t* q = (const int8_t*)x_i8s;
    const float s = get_scale(x_i8s, orc_i8s_scale_offset(n));
    std::vector<float> y((size_t)n);
    for (int64_t r = 0; r < rows; ++r) {
        const int8_t* qr = q + r * ne0;
        int64_t ssq = 0;
        for (int64_t i = 0; i < ne0; ++i) ssq += (int64_t)qr[i] * qr[i];
        const float ss = s * s;
#if ORC_PLANT == 15
        const float mean = (float)ssq / (float)ne0;
#elif ORC_PLANT == 16
        const float mean = ((float)ssq * ss) / (float)(ne0 > 1 ? ne0 - 1 : 1);
#else
        const float mean = ((float)ssq * ss) / (float)ne0;
#endif
        const float rf = 1.0f / sqrtf(mean + eps);
        for (int64_t i = 0; i < ne0; ++i) {
            const float x = (float)qr[i] * s;
            float v = x * rf;
            if (gamma) v = v * gamma[i];
            y[r * ne0 + i] = v;
        }
    }
    if (y_f32) memcpy(y_f32, y.data(), (size_t)n * 4);
    orc_i8s_quantize(y.data(), n, y_i8s);
}

// ---------------------------------------------------------------------------
// ggml_im2col_asym ([P1] "Five fused INT8 ops": im2col with independent
// left/right padding, so a causal conv needs no separate pad node; [P3]
// "Encoder": each stage starts with a strided causal conv, left pad
// K - stride, right pad 0). Reading R7. The padding is the value 0, exact in
// any scale, so the I8_S scale is carried unchanged.
// ---------------------------------------------------------------------------
ORC_API int64_t orc_im2col_out_len(int64_t L, int64_t KW, int64_t stride, int64_t pad_l, int64_t pad_r) {
    const int64_t span = L + pad_l + pad_r - KW;
    return span < 0 ? 0 : span / stride + 1;
}

ORC_API void orc_i8s_im2col_asym(const uint8_t* src_i8s, int64_t C, int64_t L, int64_t KW, int64_t stride,
                                 int64_t pad_l, int64_t pad_r, uint8_t* dst_i8s) {
    const int64_t OL = orc_im2col_out_len(L, KW, stride, pad_l, pad_r);
    const int8_t* src = (const int8_t*)src_i8s;
    std::vector<int8_t> out((size_t)(OL * C * KW));
    for (int64_t t = 0; t < OL; ++t)
        for (int64_t c = 0; c < C; ++c)
            for (int64_t k = 0; k < KW; ++k) {
#if ORC_PLANT == 17
                const int64_t pos = t * stride + k - pad_r;
#else
                const int64_t pos = t * stride + k - pad_l;
#endif
                out[(t * C + c) * KW + k] = (pos >= 0 && pos < L) ? src[c * L + pos] : (int8_t)0;
            }
    orc_i8s_pack(out.data(), OL * C * KW, get_scale(src_i8s, orc_i8s_scale_offset(C * L)), dst_i8s);
}

// ---------------------------------------------------------------------------
// Depthwise mul_mat_add ([P1] "Tests": depthwise mul_mat_add among the fused
// ops' cases; [P3] "Encoder": RMSNorm -> depthwise conv -> ... in every
// block, causal). Reading R8: channel c of the I8_S input (C x L) is
// convolved with row c of the I8_S kernel (C x KW) over the R7 geometry,
// accumulated exactly, then y = (float)acc * (w_scale*x_scale) + bias[c]
// (ReLU optional) and one scale for the whole C x OL output.
// ---------------------------------------------------------------------------
ORC_API void orc_i8s_depthwise_mul_mat_add(const uint8_t* w_i8s, int64_t KW, const uint8_t* x_i8s, int64_t C,
                                           int64_t L, int64_t stride, int64_t pad_l, int64_t pad_r,
                                           const float* bias, int relu, uint8_t* y_i8s, float* y_f32) {
    const int64_t OL = orc_im2col_out_len(L, KW, stride, pad_l, pad_r);
    const int8_t* w = (const int8_t*)w_i8s;
    const int8_t* x = (const int8_t*)x_i8s;
    const float ws = get_scale(w_i8s, orc_i8s_scale_offset(C * KW));
    const float xs = get_scale(x_i8s, orc_i8s_scale_offset(C * L));
    const float sc = ws * xs;
    std::vector<float> y((size_t)(C * OL));
    for (int64_t c = 0; c < C; ++c)
        for (int64_t t = 0; t < OL; ++t) {
            int64_t acc = 0;
            for (int64_t k = 0; k < KW; ++k) {
                const int64_t pos = t * stride + k - pad_l;
#if ORC_PLANT == 18
                const int64_t kk = KW - 1 - k;
#else
                const int64_t kk = k;
#endif
                if (pos >= 0 && pos < L) acc += (int64_t)w[c * KW + kk] * x[c * L + pos];
            }
            float v = (float)(int32_t)acc * sc;
            if (bias) v = v + bias[c];
            if (relu) v = v > 0.0f ? v : 0.0f;
            y[c * OL + t] = v;
        }
    if (y_f32) memcpy(y_f32, y.data(), (size_t)(C * OL) * 4);
    orc_i8s_quantize(y.data(), C * OL, y_i8s);
}

// ---------------------------------------------------------------------------
// W8A8 per-channel matmul ([P4] "Hypothesis" and "Implementation"): int8
// weights with one scale per output channel, int8 activations with one scale
// per row, int32 accumulation, then d[m][n] = aScale[m] * bScale[n] * C[m][n].
// Reading R9 for the two quantizers.
// ---------------------------------------------------------------------------

// Per-channel weight quantization, done once per weight on the page's
// cache-miss path: w is N x K F32; wq is N x K int8 (row n = channel n).
ORC_API void orc_w8a8_quantize_weights(const float* w, int64_t N, int64_t K, int8_t* wq, float* bscale) {
    for (int64_t n = 0; n < N; ++n) {
        float mx = 1e-9f;
        for (int64_t k = 0; k < K; ++k) {
            const float v = fabsf(w[n * K + k]);
            if (v > mx) mx = v;
        }
        const float s = mx / 127.0f;
        bscale[n] = s;
        for (int64_t k = 0; k < K; ++k) {
#if ORC_PLANT == 20
            float r = roundf(w[n * K + k] / s);
#else
            float r = rintf(w[n * K + k] / s);   // ties to even under the default rounding mode
#endif
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            wq[n * K + k] = (int8_t)(int)r;
        }
    }
}

// Per-row activation quantization with the page's 1e-9 floor.
ORC_API void orc_w8a8_quantize_rows(const float* x, int64_t M, int64_t K, int8_t* q, float* ascale) {
    for (int64_t m = 0; m < M; ++m) {
        const float* xr = x + m * K;
        float mx = 1e-9f;
        for (int64_t k = 0; k < K; ++k) {
            const float v = fabsf(xr[k]);
            if (v > mx) mx = v;
        }
        ascale[m] = mx / 127.0f;
        const float inv = 127.0f / mx;
        for (int64_t k = 0; k < K; ++k) {
            float r = roundf(xr[k] * inv);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[m * K + k] = (int8_t)(int)r;
        }
    }
}

ORC_API void orc_w8a8_mul_mat(const int8_t* wq, const float* bscale, int64_t N, int64_t K, const float* x,
                              int64_t M, float* d, int nth, int8_t* q_out, float* ascale_out) {
    if (nth < 1) nth = 1;
    std::vector<int8_t> q((size_t)(M * K));
    std::vector<float> as((size_t)M);
    orc_w8a8_quantize_rows(x, M, K, q.data(), as.data());
    std::vector<std::thread> ts;
    for (int t = 0; t < nth; ++t)
        ts.emplace_back([&, t] {
            for (int64_t n = t; n < N; n += nth)
                for (int64_t m = 0; m < M; ++m) {
                    int64_t acc = 0;
                    for (int64_t k = 0; k < K; ++k) acc += (int64_t)wq[n * K + k] * q[m * K + k];
                    if (acc > INT32_MAX || acc < INT32_MIN) {
                        fprintf(stderr, "oracle: int32 accumulator range violated\n");
                        abort();
                    }
#if ORC_PLANT == 19
                    d[m * N + n] = bscale[n] * (float)(int32_t)acc;
#elif ORC_PLANT == 23
                    d[m * N + n] = as[m] * (bscale[n] * (float)(int32_t)acc);
#else
                    d[m * N + n] = as[m] * bscale[n] * (float)(int32_t)acc;
#endif
                }
        });
    for (auto& th : ts) th.join();
    if (q_out) memcpy(q_out, q.data(), (size_t)(M * K));
    if (ascale_out) memcpy(ascale_out, as.data(), (size_t)M * 4);
}
