// Per-row activation quantization ("ggml-cpu: ternary I2_S matmul kernel",
// sections Arithmetic and Kernels; "VibeASR in audio.cpp", section Encoder for
// the 1e-5 amax floor; "Experiment - int8 W8A8 path", section Implementation
// for scale = amax/127, inv = 127/amax, round, clamp to +-127).
//
// One CTA per row: the row is read once into registers, a block reduction
// finds its absmax, and the quantized values and their int8 sum (reduced the
// same way) are written out. Besides the plain int8 layout of the public sidecar, the kernel can
// write the operand layouts of the two matmul kernels directly, so no separate
// repacking pass is needed:
//   kQuantF16Perm   the tensor-core GEMM's activation operand: q as f16 in the
//                   K order in which the GEMM expands the packed codes;
//   kQuantE2M1Tc    the tensor-core GEMV's operand: each q as three base-8
//                   digits in e2m1, one operand row per digit (k_quant_rows_tc4).

#include "common.cuh"
#include "internal.h"

namespace i2s {

// K position of the f16 element at index e of a 128-group in the tensor-core
// operand order. The GEMM expands one 32-bit word of packed codes (bytes
// gp..gp+3 of a group, gp = 4w) into 8 f16 pairs: for each bit-pair slice s
// (shift 6, 4, 2, 0) the pair (byte 0, byte 2) then (byte 1, byte 3). So
// index e = 16w + 4s + j holds byte offset {0, 2, 1, 3}[j] of that slice.
__device__ __forceinline__ int perm_index_of(int pos) {   // pos: group-relative 0..127
    const int s = pos >> 5;
    const int gp = pos & 31;
    const int w = gp >> 2;
    const int c = gp & 3;
    const int j = (c == 0) ? 0 : (c == 2) ? 1 : (c == 1) ? 2 : 3;
    return 16 * w + 4 * s + j;
}

// Writes the four quantized values of positions 4c..4c+3 of row m in the
// requested operand layout.
__device__ __forceinline__ void emit4(const QuantArgs& a, const QuantJob& J, int m, int c, const int (&q)[4]) {
    const int K = J.K;
    if (a.layout == kQuantI8Rows) {
        uint32_t* q4 = reinterpret_cast<uint32_t*>(static_cast<int8_t*>(J.out) + (size_t)m * K);
        q4[c] = (uint32_t)(q[0] & 0xff) | ((uint32_t)(q[1] & 0xff) << 8) | ((uint32_t)(q[2] & 0xff) << 16) |
                ((uint32_t)(q[3] & 0xff) << 24);
    } else {   // kQuantF16Perm
        __half* out = static_cast<__half*>(J.out) + (size_t)m * K;
        const int pos0 = 4 * c;
        const int group_base = pos0 & ~127;
#pragma unroll
        for (int e = 0; e < 4; ++e) out[group_base + perm_index_of((pos0 + e) & 127)] = __int2half_rn(q[e]);
    }
}

constexpr int kQThreads = 256;
constexpr int kQCache = 12;   // float4 per thread kept in registers (rows up to 12288 values)

// One CTA per row: the row is loaded once (kept in registers), its absmax and
// int8 sum are reduced across the block, and the quantized values are written
// in the requested layout.
__global__ void __launch_bounds__(kQThreads) k_quant_rows(const __grid_constant__ QuantArgs a) {
    __shared__ float s_red[kQThreads / 32];
    __shared__ int s_sum[kQThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (a.status && blockIdx.x == 0 && tid == 0) *a.status = 0u;
    for (unsigned long long i = blockIdx.x * (unsigned long long)kQThreads + tid; i < a.zero_16;
         i += (unsigned long long)gridDim.x * kQThreads)
        a.zero[i] = make_uint4(0u, 0u, 0u, 0u);
    const QuantJob& J = a.j[blockIdx.x / a.rows];
    const int m = blockIdx.x % a.rows;
    const int K = J.K, K4 = K / 4;
    const float4* x4 = reinterpret_cast<const float4*>(J.x + (size_t)m * K);

    float4 cache[kQCache];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kQCache; ++i) {
        const int c = tid + i * kQThreads;
        cache[i] = c < K4 ? x4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(cache[i].x), fabsf(cache[i].y)), fmaxf(fabsf(cache[i].z), fabsf(cache[i].w))));
    }
    for (int c = tid + kQCache * kQThreads; c < K4; c += kQThreads) {   // rows longer than the cache
        const float4 v = x4[c];
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    amax = warp_max(amax);
    if (lane == 0) s_red[warp] = amax;
    __syncthreads();
    amax = s_red[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_red[w]);
    float scale, inv;
    quant_params(amax, scale, inv);

    int sum = 0;
#pragma unroll
    for (int i = 0; i < kQCache; ++i) {
        const int c = tid + i * kQThreads;
        if (c < K4) {
            const int q[4] = {quantize_one(cache[i].x, inv), quantize_one(cache[i].y, inv),
                              quantize_one(cache[i].z, inv), quantize_one(cache[i].w, inv)};
            sum += q[0] + q[1] + q[2] + q[3];
            emit4(a, J, m, c, q);
        }
    }
    for (int c = tid + kQCache * kQThreads; c < K4; c += kQThreads) {
        const float4 v = x4[c];
        const int q[4] = {quantize_one(v.x, inv), quantize_one(v.y, inv), quantize_one(v.z, inv), quantize_one(v.w, inv)};
        sum += q[0] + q[1] + q[2] + q[3];
        emit4(a, J, m, c, q);
    }
    sum = warp_sum(sum);
    if (lane == 0) s_sum[warp] = sum;
    __syncthreads();
    if (tid == 0) {
        int total = 0;
#pragma unroll
        for (int w = 0; w < kQThreads / 32; ++w) total += s_sum[w];
        J.scale[m] = scale;
        J.sum[m] = total;
    }
}

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

constexpr int kQ4Cache = 3;   // 16-value units cached per thread (rows up to 12288 values)

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

// Writes the TMA tensor map of weight matrix i: the template (uint8 2-D, box
// 128 bytes x 128 rows, 128-byte swizzle) with its address, extents (K/4 bytes
// by N rows) and row stride replaced, then releases it to the tensor-map proxy
// for the GEMV launch that follows.
__device__ __forceinline__ void write_weight_map(const QuantArgs& a, int i) {
    CUtensorMap* dst = a.wmaps + i;
    const uint4* src = reinterpret_cast<const uint4*>(&a.wtmpl);
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(CUtensorMap) / 16); ++k) d[k] = src[k];
    const WMapJob& J = a.wj[i];
    const uint32_t row_bytes = (uint32_t)(J.K / 4);
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst), "l"(J.w) : "memory");
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 0, %1;" ::"l"(dst), "r"(row_bytes) : "memory");
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(dst), "r"((uint32_t)J.N) : "memory");
    asm volatile("tensormap.replace.tile.global_stride.global.b1024.b64 [%0], 0, %1;" ::"l"(dst),
                 "l"((uint64_t)row_bytes) : "memory");
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

__global__ void __launch_bounds__(kQThreads) k_quant_rows_tc4(const __grid_constant__ QuantArgs a) {
    __shared__ float s_red[kQThreads / 32];
    __shared__ int s_sum[kQThreads / 32];
    __shared__ uint32_t s_code[255];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // launched as a programmatic dependent of the kernel before it: wait for
    // that kernel (which may use the same workspace, or produce x) before
    // reading or writing global memory
    if (tid < 255) s_code[tid] = digit_code(tid - 127);
    pdl_wait();
    if (a.status && blockIdx.x == 0 && tid == 0) *a.status = 0u;
    // map i is written by thread i / gridDim.x of CTA i % gridDim.x: one or two
    // maps per CTA instead of all of them in the first CTA, whose row work
    // would otherwise wait behind them
    for (int i = blockIdx.x + (int)gridDim.x * tid; i < a.n_wmaps; i += (int)gridDim.x * kQThreads) write_weight_map(a, i);
    for (unsigned long long i = blockIdx.x * (unsigned long long)kQThreads + tid; i < a.zero_16;
         i += (unsigned long long)gridDim.x * kQThreads)
        a.zero[i] = make_uint4(0u, 0u, 0u, 0u);
    const QuantJob& J = a.j[blockIdx.x / a.M];   // one CTA per present activation row
    const int m = blockIdx.x % a.M;
    const int Mp = a.rows;
    const int K = J.K, U = K / 16;
    const size_t row_bytes = (size_t)K / 2;
    uint8_t* op = static_cast<uint8_t*>(J.out);
    const float4* x4 = reinterpret_cast<const float4*>(J.x + (size_t)m * K);

    float4 cache[kQ4Cache][4];
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < kQ4Cache; ++c) {
        const int u = tid + c * kQThreads;
        if (u < U) {
            load_unit(x4, u, cache[c]);
            amax = fmaxf(amax, unit_amax(cache[c]));
        }
    }
    for (int u = tid + kQ4Cache * kQThreads; u < U; u += kQThreads) {   // rows longer than the cache
        float4 v[4];
        load_unit(x4, u, v);
        amax = fmaxf(amax, unit_amax(v));
    }
    amax = warp_max(amax);
    if (lane == 0) s_red[warp] = amax;
    __syncthreads();
    amax = s_red[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_red[w]);
    float scale, inv;
    quant_params(amax, scale, inv);

    int sum = 0;
#pragma unroll
    for (int c = 0; c < kQ4Cache; ++c) {
        const int u = tid + c * kQThreads;
        if (u < U) sum += emit_unit(cache[c], inv, u, op, row_bytes, Mp, m, s_code);
    }
    for (int u = tid + kQ4Cache * kQThreads; u < U; u += kQThreads) {
        float4 v[4];
        load_unit(x4, u, v);
        sum += emit_unit(v, inv, u, op, row_bytes, Mp, m, s_code);
    }
    sum = warp_sum(sum);
    if (lane == 0) s_sum[warp] = sum;
    __syncthreads();
    if (tid == 0) {
        int total = 0;
#pragma unroll
        for (int w = 0; w < kQThreads / 32; ++w) total += s_sum[w];
        J.scale[m] = scale;
        J.sum[m] = total;
    }
}

cudaError_t launch_quant(const QuantArgs& a, cudaStream_t s) {
    if (a.layout == kQuantE2M1Tc) {
        // the decode path: a programmatic dependent of the kernel before it
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(a.count * a.M), 1, 1);
        cfg.blockDim = dim3(kQThreads, 1, 1);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, k_quant_rows_tc4, a);
    } else
        k_quant_rows<<<a.count * a.rows, kQThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace i2s
