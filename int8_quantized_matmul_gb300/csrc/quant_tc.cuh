// Device helpers of the tensor-core GEMV's activation operand (the e2m1
// digit rows) and of its per-matrix weight tensor maps, shared by the
// quantization kernel (quant.cu) and the GEMV's fused prologue (gemv_tc.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace i2s {

// ---------------------------------------------------------------------------
// Tensor-core GEMV operand (kQuantE2M1Tc). Each q in [-127, 127] is written as
// three digits q = d0 + 8*d1 + 64*d2 with d0, d1 in [-4, 3] and d2 in [-2, 2],
// every one exact in e2m1; digit j of activation row m goes to operand row
// j*M' + m. The operand rows of absent activation rows (m >= M) and the rows
// after 3M' are never written: each MMA output column depends only on its own
// operand row, every 4-bit pattern is a finite e2m1 value, and the GEMV reads
// only the columns of present rows. Within a 128-position
// group the K order is the one the GEMV's converters produce from the packed
// weight bytes: element 16w + 8t + 2i + h holds position 32s + 4w + i, where
// (t, h) = (0, 0), (0, 1), (1, 0), (1, 1) for bit-pair slices s = 3, 1, 2, 0.
// Elements are packed two per byte, the even one in the low nibble.
// ---------------------------------------------------------------------------

// e2m1 code of an integer digit d in [-4, 3] (magnitudes 0, 1, 2, 3, 4 encode
// as 0, 2, 4, 5, 6; bit 3 is the sign).
__device__ __forceinline__ uint32_t e2m1_digit(int d) {
    const int a = d < 0 ? -d : d;
    const uint32_t mag = a <= 2 ? 2u * (uint32_t)a : (uint32_t)a + 2u;
    return mag | (d < 0 ? 8u : 0u);
}

// Balanced base-8 digits: q = d[0] + 8*d[1] + 64*d[2].
__device__ __forceinline__ void base8_digits(int q, int (&d)[3]) {
    d[0] = ((q + 4) & 7) - 4;
    const int q1 = (q - d[0]) >> 3;   // exact: q - d0 is a multiple of 8
    d[1] = ((q1 + 4) & 7) - 4;
    d[2] = (q1 - d[1]) >> 3;
}

// A unit is (group g, word w): the 16 positions 32s + 4w + i (s, i in 0..3) of
// 128-group g, read as four float4 and written as one 8-byte word per digit row.
__device__ __forceinline__ void load_unit(const float4* x4, int u, float4 (&v)[4]) {
    const int base = 32 * (u >> 3) + (u & 7);
#pragma unroll
    for (int s = 0; s < 4; ++s) v[s] = x4[base + 8 * s];
}

__device__ __forceinline__ float unit_amax(const float4 (&v)[4]) {
    float m = 0.0f;
#pragma unroll
    for (int s = 0; s < 4; ++s) m = fmaxf(m, fmaxf(fmaxf(fabsf(v[s].x), fabsf(v[s].y)), fmaxf(fabsf(v[s].z), fabsf(v[s].w))));
    return m;
}

// The three e2m1 digit nibbles of q, at bits 0, 8 and 16 (shared-memory table
// indexed by q + 127, filled at kernel start from base8_digits/e2m1_digit).
__device__ __forceinline__ uint32_t digit_code(int q) {
    int d[3];
    base8_digits(q, d);
    return e2m1_digit(d[0]) | (e2m1_digit(d[1]) << 8) | (e2m1_digit(d[2]) << 16);
}

// Four codes (byte j of c[i] = nibble pair of digit j for word byte i) ->
// the word of digit rows 0, 1 and 2 (byte i of out[j] = byte j of c[i]).
__device__ __forceinline__ void transpose_codes(const uint32_t (&c)[4], uint32_t (&out)[3]) {
    const uint32_t lo01 = __byte_perm(c[0], c[1], 0x5140);   // c0.b0 c1.b0 c0.b1 c1.b1
    const uint32_t lo23 = __byte_perm(c[2], c[3], 0x5140);
    const uint32_t hi01 = __byte_perm(c[0], c[1], 0x0062);   // c0.b2 c1.b2
    const uint32_t hi23 = __byte_perm(c[2], c[3], 0x0062);
    out[0] = __byte_perm(lo01, lo23, 0x5410);
    out[1] = __byte_perm(lo01, lo23, 0x7632);
    out[2] = __byte_perm(hi01, hi23, 0x5410);
}

// Quantizes a unit, writes its three digit words, returns the sum of its q.
__device__ __forceinline__ int emit_unit(const float4 (&v)[4], float inv, int u, uint8_t* op, size_t row_bytes, int Mp,
                                         int m, const uint32_t* code) {
    int q[4][4];
    int sum = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        q[s][0] = quantize_one(v[s].x, inv);
        q[s][1] = quantize_one(v[s].y, inv);
        q[s][2] = quantize_one(v[s].z, inv);
        q[s][3] = quantize_one(v[s].w, inv);
        sum += q[s][0] + q[s][1] + q[s][2] + q[s][3];
    }
    // word t = 0: low nibble slice 3, high nibble slice 1; t = 1: slices 2 and 0
    uint32_t c0[4], c1[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        c0[i] = code[q[3][i] + 127] | (code[q[1][i] + 127] << 4);
        c1[i] = code[q[2][i] + 127] | (code[q[0][i] + 127] << 4);
    }
    uint32_t w0[3], w1[3];
    transpose_codes(c0, w0);
    transpose_codes(c1, w1);
#pragma unroll
    for (int j = 0; j < 3; ++j)
        reinterpret_cast<uint2*>(op + (size_t)(j * Mp + m) * row_bytes)[u] = make_uint2(w0[j], w1[j]);
    return sum;
}

// Writes the TMA tensor map of a weight matrix at dst: the template tmpl
// (uint8 2-D, box 128 bytes x 128 rows, 128-byte swizzle) with its address,
// extents (K/4 bytes by N rows) and row stride replaced, then releases it to
// the tensor-map proxy (the weight producer acquires it before first use).
__device__ __forceinline__ void write_weight_map(const CUtensorMap& tmpl, CUtensorMap* dst, const void* w, int N,
                                                 int K) {
    const uint4* src = reinterpret_cast<const uint4*>(&tmpl);
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(CUtensorMap) / 16); ++k) d[k] = src[k];
    const uint32_t row_bytes = (uint32_t)(K / 4);
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst), "l"(w) : "memory");
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 0, %1;" ::"l"(dst), "r"(row_bytes) : "memory");
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(dst), "r"((uint32_t)N) : "memory");
    asm volatile("tensormap.replace.tile.global_stride.global.b1024.b64 [%0], 0, %1;" ::"l"(dst),
                 "l"((uint64_t)row_bytes) : "memory");
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

}  // namespace i2s
