// I8_S element-wise and convolution pieces, and the W8A8 row quantizer
// ("ggml: additive INT8/ternary types, fused CPU ops, and kernels for VibeASR
// (1/2)", sections "Two new types", "Five fused INT8 ops" and "Tests";
// "VibeASR in audio.cpp", section "Encoder"; "Experiment - int8 W8A8 path",
// section "Implementation").
//
//   add_scaled       y = (float)qa*sa + (float)qb*sb, requantized per tensor
//   rms_norm_scaled  per row of ne0 values x = q*s: r = 1/sqrt(mean(x^2) + eps)
//                    with mean(x^2) = ((float)sum(q^2) * (s*s)) / ne0, each a
//                    correctly rounded binary32 operation; y = x*r (*gamma[i]),
//                    requantized per tensor
//   transpose        a x b -> b x a; the in-band scale travels with the values
//   im2col_asym      C x L -> OL x (C*KW), independent left/right padding
//   depthwise        per-channel causal conv, R4's epilogue with bias[c],
//                    requantized per tensor
//   w8a8 rows        per-row int8 activations, amax floored at 1e-9
//   w8a8 weights     per-channel int8 weights: rint(w / (amax/127)), amax
//                    floored at 1e-9; packed once into f16 operand rows
//   w8a8 rows (f16)  the packed call's row quantizer, straight into the GEMM's
//                    f16 operand rows
//
// Every op here moves bytes: each is bound by HBM bandwidth. An op whose output
// scale depends on the whole output runs two passes over its inputs: the first
// folds max|y| into one word (atomicMax on the float bits, valid because
// |y| >= 0), the second recomputes y and quantizes it. Recomputing costs fewer
// bytes than writing and re-reading an F32 intermediate.

#include "common.cuh"
#include "internal.h"

namespace i2s {

namespace {

constexpr int kEltThreads = 256;

__device__ __forceinline__ int64_t pad32(int64_t n) { return (n + 31) / 32 * 32; }

__device__ __forceinline__ float i8s_scale_of(const uint8_t* t, int64_t n) {
    return *reinterpret_cast<const float*>(t + pad32(n));
}

// Block-wide max folded into *amax_bits.
__device__ __forceinline__ void fold_max(float mx, unsigned int* amax_bits) {
    __shared__ float s_max[kEltThreads / 32];
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < kEltThreads / 32; ++i) mx = fmaxf(mx, s_max[i]);
        atomicMax(amax_bits, __float_as_uint(fmaxf(mx, s_max[0])));
    }
}

// The I8_S trailer of an n-element output: zero padding up to the next
// multiple of 32, the F32 scale, 28 zero bytes. Called by one block.
__device__ __forceinline__ void write_trailer(uint8_t* dst, int64_t n, float scale) {
    const int64_t padded = pad32(n);
    for (int64_t i = n + threadIdx.x; i < padded + 32; i += blockDim.x) {
        uint8_t b = 0;
        if (i >= padded && i < padded + 4) b = (uint8_t)(__float_as_uint(scale) >> (8 * (i - padded)));
        dst[i] = b;
    }
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
    return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) |
           ((uint32_t)(d & 0xff) << 24);
}

__device__ __forceinline__ int8_t byte_of(uint32_t w, int i) { return (int8_t)(w >> (8 * i)); }

// Stages bytes [pos0, pos0 + nbytes) of a row of L bytes (zeros outside
// [0, L)) in shared memory as 32-bit words read at aligned addresses: word i
// holds the row bytes from pos0 - sh + 4i, where sh = the misalignment of
// row + pos0. Words that reach outside the row take byte loads. Returns sh.
__device__ __forceinline__ int stage_window(const uint8_t* row, int64_t L, int64_t pos0, int nbytes, uint32_t* win32,
                                            int tid, int nthreads) {
    const int sh = (int)(((uintptr_t)row + (uintptr_t)pos0) & 3u);
    const int nw = (sh + nbytes + 3) >> 2;
    auto word = [&](int i) {
        const int64_t g = pos0 - sh + 4 * (int64_t)i;   // row position of the word's first byte
        if (g >= 0 && g + 4 <= L) return *reinterpret_cast<const uint32_t*>(row + g);
        uint32_t w = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (g + e >= 0 && g + e < L) w |= (uint32_t)row[g + e] << (8 * e);
        return w;
    };
    // four independent loads in flight per thread before any store: one load
    // at a time left the staging latency-bound
    for (int i0 = tid; i0 < nw; i0 += 4 * nthreads) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = i0 + e * nthreads < nw ? word(i0 + e * nthreads) : 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (i0 + e * nthreads < nw) win32[i0 + e * nthreads] = w[e];
    }
    return sh;
}

// As stage_window, with 16-byte loads: word i of win (16-byte aligned) holds
// the row bytes from pos0 - sh + 4i, where sh = the misalignment of row + pos0
// modulo 16. Every thread has its loads in flight before any store. Returns sh.
__device__ __forceinline__ int stage_window16(const uint8_t* row, int64_t L, int64_t pos0, int nbytes, uint32_t* win,
                                              int tid, int nthreads) {
    const int sh = (int)(((uintptr_t)row + (uintptr_t)pos0) & 15u);
    const int nq = (sh + nbytes + 15) >> 4;
    auto quad = [&](int i) {
        const int64_t g = pos0 - sh + 16 * (int64_t)i;   // row position of the quad's first byte
        if (g >= 0 && g + 16 <= L) return *reinterpret_cast<const uint4*>(row + g);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        for (int e = 0; e < 16; ++e)
            if (g + e >= 0 && g + e < L) w[e >> 2] |= (uint32_t)row[g + e] << (8 * (e & 3));
        return make_uint4(w[0], w[1], w[2], w[3]);
    };
    for (int i0 = tid; i0 < nq; i0 += 4 * nthreads) {
        uint4 v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = i0 + e * nthreads < nq ? quad(i0 + e * nthreads) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (i0 + e * nthreads < nq) reinterpret_cast<uint4*>(win)[i0 + e * nthreads] = v[e];
    }
    return sh;
}

// quantize_one without its clamp, for a value bounded by the amax its scale came
// from. Every caller in this file quantizes values whose largest magnitude is
// that amax (or lies below its floor): the second passes recompute exactly the
// values their first pass folded, and the W8A8 rows quantize the row they took
// the maximum of. With |x| <= amax and inv = fl(127 / amax) <=
// (127 / amax)(1 + 2^-24), fl(x * inv) is at most 127 + 2^-17 in magnitude,
// below 127.5, so the clamp of quantize_one never acts and both give the same
// integer.
__device__ __forceinline__ int quantize_bounded(float x, float inv) {
    const float v = __fmul_rn(x, inv);
    const float a = __fadd_rn(fabsf(v), 0x1.fffffep-2f);
    const int m = (int)(__float_as_uint(__fadd_rz(a, 12582912.0f)) - 0x4B400000u);
    return v < 0.0f ? -m : m;
}

// ---------------------------------------------------------------- add_scaled

__device__ __forceinline__ float add_one(int8_t qa, int8_t qb, float sa, float sb) {
    return __fadd_rn(__fmul_rn(i8_to_float(qa), sa), __fmul_rn(i8_to_float(qb), sb));
}

// Byte e of a word whose bytes were XORed with 0x80 (each int8 as q + 128),
// read as a float exactly: the byte placed in the low mantissa bits of 2^23 by
// one byte permute, minus 2^23 + 128 (the same value and rounding as
// i8_to_float, with the XOR done once per word).
__device__ __forceinline__ float i8x_to_float(uint32_t wx, int e) {
    return __fsub_rn(__uint_as_float(__byte_perm(wx, 0x4Bu, 0x4550u + (uint32_t)e)), 8388736.0f);
}

__device__ __forceinline__ float add_one_x(uint32_t wax, uint32_t wbx, int e, float sa, float sb) {
    return __fadd_rn(__fmul_rn(i8x_to_float(wax, e), sa), __fmul_rn(i8x_to_float(wbx, e), sb));
}

// Pass 1: max |y| over the tensor. 16 bytes of each input per thread and step.
__global__ void __launch_bounds__(kEltThreads) k_add_amax(const uint8_t* __restrict__ a, const uint8_t* __restrict__ b,
                                                          int64_t n, unsigned int* amax_bits) {
    const float sa = i8s_scale_of(a, n), sb = i8s_scale_of(b, n);
    const int64_t n16 = n / 16, stride = (int64_t)gridDim.x * blockDim.x;
    float mx = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint4 va = ldg_stream(a + 16 * i), vb = ldg_stream(b + 16 * i);
        const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int w = 0; w < 4; ++w)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                mx = fmaxf(mx, fabsf(add_one_x(wa[w] ^ 0x80808080u, wb[w] ^ 0x80808080u, e, sa, sb)));
    }
    if (blockIdx.x == 0)
        for (int64_t i = n16 * 16 + threadIdx.x; i < n; i += blockDim.x)
            mx = fmaxf(mx, fabsf(add_one((int8_t)a[i], (int8_t)b[i], sa, sb)));
    fold_max(mx, amax_bits);
}

// Pass 2: recompute y and quantize it with the folded amax.
__global__ void __launch_bounds__(kEltThreads) k_add_quant(const uint8_t* __restrict__ a, const uint8_t* __restrict__ b,
                                                           int64_t n, const unsigned int* __restrict__ amax_bits,
                                                           uint8_t* __restrict__ dst) {
    pdl_wait();   // the first pass's amax
    const float sa = i8s_scale_of(a, n), sb = i8s_scale_of(b, n);
    float scale, inv;
    quant_params(__uint_as_float(*amax_bits), scale, inv);
    const int64_t n16 = n / 16, stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint4 va = ldg_stream(a + 16 * i), vb = ldg_stream(b + 16 * i);
        const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
        uint32_t o[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            int q[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                q[e] = quantize_bounded(add_one_x(wa[w] ^ 0x80808080u, wb[w] ^ 0x80808080u, e, sa, sb), inv);
            o[w] = pack4(q[0], q[1], q[2], q[3]);
        }
        *reinterpret_cast<uint4*>(dst + 16 * i) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (blockIdx.x == 0) {
        for (int64_t i = n16 * 16 + threadIdx.x; i < n; i += blockDim.x)
            dst[i] = (uint8_t)(quantize_bounded(add_one((int8_t)a[i], (int8_t)b[i], sa, sb), inv) & 0xff);
        write_trailer(dst, n, scale);
    }
}

// ------------------------------------------------------------ rms_norm_scaled
// One warp per row (grid-stride over rows), lanes striding over the row.

__device__ __forceinline__ float rms_factor(int ssq, int64_t ne0, float s, float eps) {
    const float mean = __fdiv_rn(__fmul_rn((float)ssq, __fmul_rn(s, s)), (float)ne0);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

__device__ __forceinline__ float rms_one(int8_t q, float s, float r, const float* gamma, int64_t i) {
    float v = __fmul_rn(__fmul_rn(i8_to_float(q), s), r);
    if (gamma) v = __fmul_rn(v, gamma[i]);
    return v;
}

// Pass 1: the row factors (kept in the workspace) and max |y|.
__global__ void __launch_bounds__(kEltThreads) k_rms_rows(const uint8_t* __restrict__ x, int64_t rows, int64_t ne0,
                                                          float eps, const float* __restrict__ gamma,
                                                          float* __restrict__ rfac, unsigned int* amax_bits) {
    const int64_t n = rows * ne0;
    const float s = i8s_scale_of(x, n);
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int8_t* q = reinterpret_cast<const int8_t*>(x);
    float mx = 0.0f;
    for (int64_t row = warp0; row < rows; row += warps) {
        const int8_t* qr = q + row * ne0;
        int ssq = 0, qmax = 0;   // ne0 * 127^2 < 2^31 for ne0 < 133,000 (checked by the host)
        if ((ne0 & 3) == 0) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(qr);
            for (int64_t w = lane; w < ne0 / 4; w += 32) {
                const uint32_t v = src[w];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int b = byte_of(v, e);
                    ssq += b * b;
                    qmax = max(qmax, abs(b));
                }
            }
        } else {
            for (int64_t i = lane; i < ne0; i += 32) {
                const int v = qr[i];
                ssq += v * v;
                qmax = max(qmax, abs(v));
            }
        }
        ssq = warp_sum(ssq);
        const float r = rms_factor(ssq, ne0, s, eps);
        if (lane == 0) rfac[row] = r;
        if (gamma) {   // the weight varies along the row: every element
            for (int64_t i = lane; i < ne0; i += 32) mx = fmaxf(mx, fabsf(rms_one(qr[i], s, r, gamma, i)));
        } else {       // x*r is monotonic in |q|: the row's largest |q| gives its max
            qmax = (int)warp_max((float)qmax);
            mx = fmaxf(mx, fabsf(rms_one((int8_t)qmax, s, r, nullptr, 0)));
        }
    }
    fold_max(mx, amax_bits);
}

// Pass 2: y = x*r (*gamma), quantized with the folded amax; one warp per row
// again, four values per lane and step when rows are whole 32-bit words.
__global__ void __launch_bounds__(kEltThreads) k_rms_quant(const uint8_t* __restrict__ x, int64_t rows, int64_t ne0,
                                                           const float* __restrict__ gamma,
                                                           const float* __restrict__ rfac,
                                                           const unsigned int* __restrict__ amax_bits,
                                                           uint8_t* __restrict__ dst) {
    pdl_wait();   // the first pass's row factors and amax
    const int64_t n = rows * ne0;
    const float s = i8s_scale_of(x, n);
    float scale, inv;
    quant_params(__uint_as_float(*amax_bits), scale, inv);
    const int8_t* q = reinterpret_cast<const int8_t*>(x);
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const bool words = (ne0 & 3) == 0;
    for (int64_t row = warp0; row < rows; row += warps) {
        const float r = rfac[row];
        if (words) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(q + row * ne0);
            uint32_t* out = reinterpret_cast<uint32_t*>(dst + row * ne0);
            for (int64_t w = lane; w < ne0 / 4; w += 32) {
                const uint32_t v = src[w];
                int o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = quantize_bounded(rms_one(byte_of(v, e), s, r, gamma, 4 * w + e), inv);
                out[w] = pack4(o[0], o[1], o[2], o[3]);
            }
        } else {
            for (int64_t i = lane; i < ne0; i += 32)
                dst[row * ne0 + i] = (uint8_t)(quantize_bounded(rms_one(q[row * ne0 + i], s, r, gamma, i), inv) & 0xff);
        }
    }
    if (blockIdx.x == 0) write_trailer(dst, n, scale);
}

// Short rows (ne0 = 16*V bytes, V <= 4): one thread per row, V 16-byte loads.
// Pass 2 recomputes the row factor from the same bytes (cheaper than storing
// and re-reading it).
template <int V>
__device__ __forceinline__ void load_row16(const uint8_t* p, uint32_t (&w)[4 * V]) {
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const uint4 u = *reinterpret_cast<const uint4*>(p + 16 * v);
        w[4 * v] = u.x;
        w[4 * v + 1] = u.y;
        w[4 * v + 2] = u.z;
        w[4 * v + 3] = u.w;
    }
}

// The row's sum of squares (one 4-way int8 dot product per word, exact) and
// its largest |q|.
template <int V>
__device__ __forceinline__ float row_factor16(const uint32_t (&w)[4 * V], float s, float eps, int& qmax) {
    int ssq = 0;
    qmax = 0;
#pragma unroll
    for (int i = 0; i < 4 * V; ++i) {
        ssq = __dp4a((int)w[i], (int)w[i], ssq);
#pragma unroll
        for (int e = 0; e < 4; ++e) qmax = max(qmax, abs((int)byte_of(w[i], e)));
    }
    return rms_factor(ssq, 16 * V, s, eps);
}

template <int V, bool kGamma>
__global__ void __launch_bounds__(kEltThreads) k_rms_rows_t(const uint8_t* __restrict__ x, int64_t rows, float eps,
                                                            const float* __restrict__ gamma_arg,
                                                            unsigned int* amax_bits) {
    const float* gamma = kGamma ? gamma_arg : nullptr;   // known at compile time
    const float s = i8s_scale_of(x, rows * 16 * V);
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    float mx = 0.0f;
    for (int64_t row = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; row < rows; row += step) {
        uint32_t w[4 * V];
        load_row16<V>(x + row * 16 * V, w);
        int qmax;
        const float r = row_factor16<V>(w, s, eps, qmax);
        if (gamma) {
#pragma unroll
            for (int i = 0; i < 4 * V; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(rms_one(byte_of(w[i], e), s, r, gamma, 4 * i + e)));
        } else {
            mx = fmaxf(mx, fabsf(rms_one((int8_t)qmax, s, r, nullptr, 0)));
        }
    }
    fold_max(mx, amax_bits);
}

template <int V, bool kGamma>
__global__ void __launch_bounds__(kEltThreads) k_rms_quant_t(const uint8_t* __restrict__ x, int64_t rows, float eps,
                                                             const float* __restrict__ gamma_arg,
                                                             const unsigned int* __restrict__ amax_bits,
                                                             uint8_t* __restrict__ dst) {
    const float* gamma = kGamma ? gamma_arg : nullptr;   // known at compile time
    pdl_wait();   // the first pass's amax
    const float s = i8s_scale_of(x, rows * 16 * V);
    float scale, inv;
    quant_params(__uint_as_float(*amax_bits), scale, inv);
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t row = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; row < rows; row += step) {
        uint32_t w[4 * V];
        load_row16<V>(x + row * 16 * V, w);
        int qmax;
        const float r = row_factor16<V>(w, s, eps, qmax);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int wi = 4 * v + i;
                o[i] = pack4(quantize_bounded(rms_one(byte_of(w[wi], 0), s, r, gamma, 4 * wi), inv),
                             quantize_bounded(rms_one(byte_of(w[wi], 1), s, r, gamma, 4 * wi + 1), inv),
                             quantize_bounded(rms_one(byte_of(w[wi], 2), s, r, gamma, 4 * wi + 2), inv),
                             quantize_bounded(rms_one(byte_of(w[wi], 3), s, r, gamma, 4 * wi + 3), inv));
            }
            *reinterpret_cast<uint4*>(dst + row * 16 * V + 16 * v) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    if (blockIdx.x == 0) write_trailer(dst, rows * 16 * V, scale);
}

// ------------------------------------------------------------------ transpose
// Tiles of TR source rows x TC source columns through shared memory: 32 x 128
// for wide source rows, 128 x 32 for narrow ones (b < 128), so that loads and
// stores both move whole 128-byte segments per warp instruction. Loads: 32-bit
// words of source rows; stores: 32-bit words of destination rows (TR/4 words
// per destination segment). Edge tiles and rows that are not whole words take
// byte accesses.

template <int TR, int TC>
__global__ void __launch_bounds__(kEltThreads) k_transpose(const uint8_t* __restrict__ src, int64_t a, int64_t b,
                                                           uint8_t* __restrict__ dst, int64_t tiles_b) {
    __shared__ __align__(16) uint8_t tile[TR][TC + 4];
    constexpr int kRowWords = TC / 4, kColWords = TR / 4;
    const int64_t ti = blockIdx.x / tiles_b, tj = blockIdx.x - ti * tiles_b;
    const int64_t i0 = ti * TR, j0 = tj * TC;
    const bool full = i0 + TR <= a && j0 + TC <= b;
    if (full && (b & 3) == 0) {
#pragma unroll
        for (int w = threadIdx.x; w < TR * kRowWords; w += kEltThreads) {
            const int r = w / kRowWords, cw = w - r * kRowWords;
            *reinterpret_cast<uint32_t*>(&tile[r][4 * cw]) =
                *reinterpret_cast<const uint32_t*>(src + (i0 + r) * b + j0 + 4 * cw);
        }
    } else {
        for (int w = threadIdx.x; w < TR * kRowWords; w += kEltThreads) {
            const int r = w / kRowWords, cw = w - r * kRowWords;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t i = i0 + r, j = j0 + 4 * cw + e;
                tile[r][4 * cw + e] = (i < a && j < b) ? src[i * b + j] : (uint8_t)0;
            }
        }
    }
    __syncthreads();
    // destination row j0 + jr holds source rows i0 .. i0+TR-1 at column jr. A
    // thread reads one word from each of source rows 4k .. 4k+3 (columns
    // 4jq .. 4jq+3) and transposes the 4 x 4 bytes in registers: four output
    // words, one in each of destination rows 4jq .. 4jq+3
    for (int w = threadIdx.x; w < (TC / 4) * kColWords; w += kEltThreads) {
        const int jq = w / kColWords, k = w - jq * kColWords;
        const uint32_t r0 = *reinterpret_cast<const uint32_t*>(&tile[4 * k][4 * jq]);
        const uint32_t r1 = *reinterpret_cast<const uint32_t*>(&tile[4 * k + 1][4 * jq]);
        const uint32_t r2 = *reinterpret_cast<const uint32_t*>(&tile[4 * k + 2][4 * jq]);
        const uint32_t r3 = *reinterpret_cast<const uint32_t*>(&tile[4 * k + 3][4 * jq]);
        const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r0, r1, 0x7362);   // bytes 0,1 / 2,3
        const uint32_t t2 = __byte_perm(r2, r3, 0x5140), t3 = __byte_perm(r2, r3, 0x7362);
        const uint32_t v[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                               __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632)};
        const int64_t i = i0 + 4 * k;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int64_t j = j0 + 4 * jq + c;
            if (full && (a & 3) == 0) {
                *reinterpret_cast<uint32_t*>(dst + j * a + i) = v[c];
            } else if (j < b) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (i + e < a) dst[j * a + i + e] = (uint8_t)(v[c] >> (8 * e));
            }
        }
    }
    if (blockIdx.x == 0) {
        __syncthreads();
        write_trailer(dst, a * b, i8s_scale_of(src, a * b));
    }
}

// ---------------------------------------------------------------- im2col_asym

// KW = 4, stride 2, C a multiple of 32, L a multiple of 16 and a 16-byte
// aligned source (the encoder's stage-1 conv input): no staging. A warp takes
// 32 output positions t0 .. t0+31 of 32 channels, one channel per lane. Output
// row t holds, for channel c, the 4 bytes at positions 2t - pad_l .. +3 of the
// channel's row; the 32 windows of a lane span 66 bytes starting at
// s = 2 t0 - pad_l, which sits R bytes into a 16-byte chunk for every t0 (t0 is
// a multiple of 32), so the lane loads five 16-byte chunks (a chunk lies wholly
// inside [0, L) or wholly outside, where it reads as the zero padding) and
// forms each window as one funnel shift of two of their words, at offsets known
// at compile time. The warp's 32 lanes write word c of row t: 128 contiguous
// bytes per store.
template <int R>
__global__ void __launch_bounds__(kEltThreads) k_im2col_k4s2(const uint8_t* __restrict__ src, int C, int64_t L,
                                                             int pad_l, int64_t OL, uint8_t* __restrict__ dst) {
    const int64_t warp = (blockIdx.x * (int64_t)kEltThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int groups = C >> 5;
    const int64_t runs = (OL + 31) >> 5;
    if (warp < groups * runs) {
        const int64_t run = warp / groups;
        const int c = (int)(warp - run * groups) * 32 + lane;
        const int64_t t0 = run * 32;
        const int64_t base = 2 * t0 - pad_l - R;   // 16-byte aligned
        const uint8_t* row = src + (int64_t)c * L;
        uint32_t w[20];
#pragma unroll
        for (int ch = 0; ch < 5; ++ch) {
            const int64_t off = base + 16 * ch;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (off >= 0 && off < L) v = *reinterpret_cast<const uint4*>(row + off);
            w[4 * ch] = v.x, w[4 * ch + 1] = v.y, w[4 * ch + 2] = v.z, w[4 * ch + 3] = v.w;
        }
        const int64_t row_bytes = 4 * (int64_t)C;
        uint32_t* out = reinterpret_cast<uint32_t*>(dst + t0 * row_bytes) + c;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int o = R + 2 * i;   // window i's first byte within the loaded chunks
            const int q = o >> 2, sh = (o & 3) * 8;
            const uint32_t win = sh ? __funnelshift_r(w[q], w[q + 1], sh) : w[q];
            if (t0 + i < OL) out[(int64_t)i * C] = win;
        }
    }
    if (blockIdx.x == 0) write_trailer(dst, OL * C * 4, i8s_scale_of(src, (int64_t)C * L));
}



// Output and input sizes below 2^31 (checked by the host): 32-bit index math.
__global__ void __launch_bounds__(kEltThreads) k_im2col(const uint8_t* __restrict__ src, int C, int L, int KW,
                                                        int stride, int pad_l, int OL, uint8_t* __restrict__ dst) {
    const int n = OL * C * KW;
    const int8_t* x = reinterpret_cast<const int8_t*>(src);
    auto value = [&](int f) -> int {
        const int row = f / KW, k = f - row * KW;   // row = t*C + c
        const int t = row / C, c = row - t * C;
        const int pos = t * stride + k - pad_l;
        return (pos >= 0 && pos < L) ? (int)x[c * L + pos] : 0;
    };
    const int n4 = n / 4, step = gridDim.x * blockDim.x;
    for (int i4 = blockIdx.x * blockDim.x + threadIdx.x; i4 < n4; i4 += step)
        *reinterpret_cast<uint32_t*>(dst + 4 * i4) =
            pack4(value(4 * i4), value(4 * i4 + 1), value(4 * i4 + 2), value(4 * i4 + 3));
    if (blockIdx.x == 0) {
        for (int i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) dst[i] = (uint8_t)(value(i) & 0xff);
        write_trailer(dst, n, i8s_scale_of(src, (int64_t)C * L));
    }
}

// Windowed im2col: a block covers T output positions (t0 .. t0+T-1) of every
// channel. It stages each channel's input window (W = (T-1)*stride + KW bytes
// from position t0*stride - pad_l, zeros outside [0, L)) in shared memory with
// coalesced loads, then writes its T*C*KW contiguous output bytes as 32-bit
// words, one per thread and step, reading the window. T is a multiple of 4, so
// every block's output starts on a word. Sizes below 2^31 (checked by the host).
__global__ void __launch_bounds__(kEltThreads) k_im2col_win(const uint8_t* __restrict__ src, int C, int L, int KW,
                                                            int stride, int pad_l, int OL, int T, int W,
                                                            uint8_t* __restrict__ dst) {
    // per channel: Wc words of staged window (the row bytes from p0 - sh[c])
    extern __shared__ uint32_t wsm[];
    const int Wc = (W + 3 + 3) / 4 + 1;
    int* shs = reinterpret_cast<int*>(wsm + (size_t)C * Wc);
    const int t0 = blockIdx.x * T;
    const int p0 = t0 * stride - pad_l;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int c = warp; c < C; c += kEltThreads / 32) {
        const int sh = stage_window(src + (int64_t)c * L, L, p0, W, wsm + (size_t)c * Wc, lane, 32);
        if (lane == 0) shs[c] = sh;
    }
    __syncthreads();
    const uint8_t* win = reinterpret_cast<const uint8_t*>(wsm);
    const int Tn = min(T, OL - t0);
    const int nloc = Tn * C * KW;
    uint8_t* out = dst + (int64_t)t0 * C * KW;
    if ((KW & 3) == 0 && (nloc & 15) == 0 && ((uintptr_t)out & 15) == 0) {
        // four output words per thread and step, stored as one 16-byte word:
        // word w = (tl*C + c)*wpg + j, each from two aligned window words and
        // a funnel shift; (tl, c, j) advance with carries (no division)
        const int wpg = KW >> 2;   // words per (t, c) group
        constexpr int kStep = 4 * kEltThreads;   // words per block step
        const int dg = kStep / wpg, dj = kStep - dg * wpg;
        const int dtl = dg / C, dc = dg - dtl * C;
        int j, c, tl;
        {
            const int w0 = 4 * (int)threadIdx.x;
            const int g0 = w0 / wpg;
            j = w0 - g0 * wpg;
            tl = g0 / C;
            c = g0 - tl * C;
        }
        for (int q = threadIdx.x; 16 * q < nloc; q += kEltThreads) {
            uint32_t v[4];
            int jj = j, cc = c, tt = tl;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int off = cc * 4 * Wc + shs[cc] + tt * stride + 4 * jj;   // byte offset in the staged words
                v[e] = __funnelshift_r(wsm[off >> 2], wsm[(off >> 2) + 1], 8 * (off & 3));
                if (++jj == wpg) {
                    jj = 0;
                    if (++cc == C) { cc = 0; ++tt; }
                }
            }
            *reinterpret_cast<uint4*>(out + 16 * q) = make_uint4(v[0], v[1], v[2], v[3]);
            j += dj;
            if (j >= wpg) { j -= wpg; ++c; }
            c += dc;
            if (c >= C) { c -= C; ++tl; }
            tl += dtl;
        }
        if (blockIdx.x == 0) write_trailer(dst, (int64_t)OL * C * KW, i8s_scale_of(src, (int64_t)C * L));
        return;
    }
    if ((KW & 3) == 0) {
        // every output word lies inside one (t, c) group: two aligned window
        // words and a funnel shift (the window buffer has 4 spare bytes)
        const int wpg = KW >> 2;   // words per group
        // word w = (tl*C + c)*wpg + j; each step advances w by the block size,
        // so (tl, c, j) advance by fixed amounts with carries (no division)
        const int dg = kEltThreads / wpg, dj = kEltThreads - dg * wpg;
        const int dtl = dg / C, dc = dg - dtl * C;
        int j, c, tl;
        {
            const int g0 = threadIdx.x / wpg;
            j = threadIdx.x - g0 * wpg;
            tl = g0 / C;
            c = g0 - tl * C;
        }
        for (int w = threadIdx.x; 4 * w < nloc; w += kEltThreads) {
            const int off = c * 4 * Wc + shs[c] + tl * stride + 4 * j;   // byte offset in the staged words
            const uint32_t lo = wsm[off >> 2], hi = wsm[(off >> 2) + 1];
            *reinterpret_cast<uint32_t*>(out + 4 * w) = __funnelshift_r(lo, hi, 8 * (off & 3));
            j += dj;
            if (j >= wpg) { j -= wpg; ++c; }
            c += dc;
            if (c >= C) { c -= C; ++tl; }
            tl += dtl;
        }
        if (blockIdx.x == 0) write_trailer(dst, (int64_t)OL * C * KW, i8s_scale_of(src, (int64_t)C * L));
        return;
    }
    for (int w = threadIdx.x; 4 * w < nloc; w += kEltThreads) {
        const int f = 4 * w;
        const int g = f / KW;
        int k = f - g * KW, tl = g / C, c = g - tl * C;
        uint32_t v = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (f + e < nloc) v |= (uint32_t)win[c * 4 * Wc + shs[c] + tl * stride + k] << (8 * e);
            if (++k == KW) {
                k = 0;
                if (++c == C) { c = 0; ++tl; }
            }
        }
        if (f + 3 < nloc) {
            *reinterpret_cast<uint32_t*>(out + f) = v;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (f + e < nloc) out[f + e] = (uint8_t)(v >> (8 * e));
        }
    }
    if (blockIdx.x == 0) write_trailer(dst, (int64_t)OL * C * KW, i8s_scale_of(src, (int64_t)C * L));
}

// ------------------------------------------------------------------ depthwise

// Sizes below 2^31 (checked by the host): 32-bit index math.
struct DwArgs {
    const uint8_t* w;   // I8_S C x KW
    const uint8_t* x;   // I8_S C x L
    const float* bias;  // C or null
    int C, L, OL, KW, stride, pad_l, relu;
};

__device__ __forceinline__ float dw_one(const DwArgs& d, float sc, int f) {
    const int c = f / d.OL, t = f - c * d.OL;
    const int8_t* w = reinterpret_cast<const int8_t*>(d.w) + (int64_t)c * d.KW;
    const int8_t* x = reinterpret_cast<const int8_t*>(d.x) + (int64_t)c * d.L;
    int acc = 0;
    const int p0 = t * d.stride - d.pad_l;
    for (int k = 0; k < d.KW; ++k) {
        const int pos = p0 + k;
        if (pos >= 0 && pos < d.L) acc += (int)w[k] * (int)x[pos];
    }
    float v = __fmul_rn(__int2float_rn(acc), sc);
    if (d.bias) v = __fadd_rn(v, d.bias[c]);
    if (d.relu) v = v > 0.0f ? v : 0.0f;
    return v;
}

__global__ void __launch_bounds__(kEltThreads) k_dw_amax(const DwArgs d, unsigned int* amax_bits) {
    const float sc = __fmul_rn(i8s_scale_of(d.w, (int64_t)d.C * d.KW), i8s_scale_of(d.x, (int64_t)d.C * d.L));
    const int n = d.C * d.OL, step = gridDim.x * blockDim.x;
    float mx = 0.0f;
    for (int f = blockIdx.x * blockDim.x + threadIdx.x; f < n; f += step) mx = fmaxf(mx, fabsf(dw_one(d, sc, f)));
    fold_max(mx, amax_bits);
}

__global__ void __launch_bounds__(kEltThreads) k_dw_quant(const DwArgs d, const unsigned int* __restrict__ amax_bits,
                                                          uint8_t* __restrict__ dst) {
    const float sc = __fmul_rn(i8s_scale_of(d.w, (int64_t)d.C * d.KW), i8s_scale_of(d.x, (int64_t)d.C * d.L));
    float scale, inv;
    quant_params(__uint_as_float(*amax_bits), scale, inv);
    const int n = d.C * d.OL, n4 = n / 4, step = gridDim.x * blockDim.x;
    for (int i4 = blockIdx.x * blockDim.x + threadIdx.x; i4 < n4; i4 += step)
        *reinterpret_cast<uint32_t*>(dst + 4 * i4) =
            pack4(quantize_bounded(dw_one(d, sc, 4 * i4), inv), quantize_bounded(dw_one(d, sc, 4 * i4 + 1), inv),
                  quantize_bounded(dw_one(d, sc, 4 * i4 + 2), inv), quantize_bounded(dw_one(d, sc, 4 * i4 + 3), inv));
    if (blockIdx.x == 0) {
        for (int i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) dst[i] = (uint8_t)(quantize_bounded(dw_one(d, sc, i), inv) & 0xff);
        write_trailer(dst, n, scale);
    }
}

// Windowed depthwise: block (x, c) covers outputs t0 .. t0+1023 of channel c.
// It stages the channel's input window (1023*stride + KW bytes) and the KW
// taps in shared memory, then each thread forms four consecutive outputs.
// kQuant = false folds max|y|; kQuant = true quantizes and stores. Needs
// C <= 65535 (grid y), KW <= 64 and a window within 48 KB (host-checked).
constexpr int kDwT = 4 * kEltThreads;

template <bool kQuant>
__global__ void __launch_bounds__(kEltThreads) k_dw_win(const DwArgs d, int W, unsigned int* amax_bits,
                                                        uint8_t* __restrict__ dst) {
    extern __shared__ uint8_t dsm[];   // window (W bytes) then the taps
    int8_t* win = reinterpret_cast<int8_t*>(dsm);
    int8_t* taps = reinterpret_cast<int8_t*>(dsm + W);
    const int c = blockIdx.y;
    const int t0 = blockIdx.x * kDwT;
    const int p0 = t0 * d.stride - d.pad_l;
    const int8_t* row = reinterpret_cast<const int8_t*>(d.x) + (int64_t)c * d.L;
    for (int xo = threadIdx.x; xo < W; xo += kEltThreads) {
        const int pos = p0 + xo;
        win[xo] = (pos >= 0 && pos < d.L) ? row[pos] : (int8_t)0;
    }
    if (threadIdx.x < d.KW) taps[threadIdx.x] = reinterpret_cast<const int8_t*>(d.w)[(int64_t)c * d.KW + threadIdx.x];
    __syncthreads();
    const float sc = __fmul_rn(i8s_scale_of(d.w, (int64_t)d.C * d.KW), i8s_scale_of(d.x, (int64_t)d.C * d.L));
    const float bc = d.bias ? d.bias[c] : 0.0f;
    float scale = 0.0f, inv = 0.0f;
    if (kQuant) {
        pdl_wait();   // the first pass's amax
        quant_params(__uint_as_float(*amax_bits), scale, inv);
    }
    float mx = 0.0f;
    const int tl0 = 4 * threadIdx.x;
    uint8_t* out = dst + (int64_t)c * d.OL + t0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int t = t0 + tl0 + e;
        if (t < d.OL) {
            const int8_t* xw = win + (tl0 + e) * d.stride;
            int acc = 0;
            for (int k = 0; k < d.KW; ++k) acc += (int)taps[k] * (int)xw[k];
            float v = __fmul_rn(small_int_to_float(acc), sc);   // |acc| <= 64 * 128^2 < 2^22
            if (d.bias) v = __fadd_rn(v, bc);
            if (d.relu) v = v > 0.0f ? v : 0.0f;
            if (kQuant) out[tl0 + e] = (uint8_t)(quantize_bounded(v, inv) & 0xff);
            else mx = fmaxf(mx, fabsf(v));
        }
    }
    if (kQuant) {
        if (blockIdx.x == 0 && blockIdx.y == 0) write_trailer(dst, (int64_t)d.C * d.OL, scale);
    } else {
        fold_max(mx, amax_bits);
    }
}

// Stride-1 depthwise with at most 8 taps (the encoder blocks' 7-tap causal
// conv): eight consecutive outputs per thread from four window words; each
// output is two 4-way int8 dot products (__dp4a) of funnel-shifted window
// words with the taps packed into two words (zero past KW).
constexpr int kDw1Out = 8;
constexpr int kDw1Chunks = 4;                               // chunks of 2048 outputs per block
constexpr int kDw1T = kDw1Out * kEltThreads * kDw1Chunks;   // outputs per block

template <bool kQuant, bool kBias, bool kRelu>
__global__ void __launch_bounds__(kEltThreads) k_dw_s1(const DwArgs d, unsigned int* amax_bits,
                                                       uint8_t* __restrict__ dst) {
    constexpr int kWinBytes = kDw1T + 16;   // the block's outputs plus up to 8 taps, rounded
    __shared__ __align__(16) uint32_t win32[(kWinBytes + 15 + 15) / 16 * 4 + 4];
    const int c = blockIdx.y;
    const int t0 = blockIdx.x * kDw1T;
    const int p0 = t0 - d.pad_l;
    const uint8_t* row = d.x + (int64_t)c * d.L;
    // window byte b sits at byte b + sh16 of the staged words
    const int sh16 = stage_window16(row, d.L, p0, kWinBytes, win32, threadIdx.x, kEltThreads);
    const int sh = sh16 & 3, qsh = sh16 >> 2;
    const int8_t* wt = reinterpret_cast<const int8_t*>(d.w) + (int64_t)c * d.KW;
    uint32_t tw[2] = {0u, 0u};
    for (int k = 0; k < d.KW; ++k) tw[k >> 2] |= (uint32_t)(uint8_t)wt[k] << (8 * (k & 3));
    __syncthreads();
    const float sc = __fmul_rn(i8s_scale_of(d.w, (int64_t)d.C * d.KW), i8s_scale_of(d.x, (int64_t)d.C * d.L));
    const float bc = kBias ? d.bias[c] : 0.0f;
    float scale = 0.0f, inv = 0.0f;
    if (kQuant) {
        pdl_wait();   // the first pass's amax
        quant_params(__uint_as_float(*amax_bits), scale, inv);
    }
    // y of one accumulator, the same arithmetic in both passes
    auto y_of = [&](int acc) {
        float v = __fmul_rn(small_int_to_float(acc), sc);   // |acc| <= 64 * 128^2 < 2^22
        if (kBias) v = __fadd_rn(v, bc);
        if (kRelu) v = v > 0.0f ? v : 0.0f;
        return v;
    };
    // Pass 1 keeps the extremes of the live accumulators only. y_of is monotone in acc (an exact
    // int-to-float, then a multiply by one factor, an add and a ReLU, each rounded to nearest, and
    // rounding to nearest is monotone), so over any set of accumulators max |y| is reached at the
    // smallest or the largest one: the folded amax is the one every |y| would give.
    int lo = INT_MAX, hi = INT_MIN;
    const bool aligned = ((((int64_t)c * d.OL) & 3) == 0);
#pragma unroll 1
    for (int chunk = 0; chunk < kDw1Chunks; ++chunk) {
        const int tl0 = kDw1Out * (threadIdx.x + chunk * kEltThreads);
        // window bytes tl0 .. tl0+15: five staged words shifted by sh
        const int q0 = (tl0 >> 2) + qsh;
        uint32_t xw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) xw[i] = __funnelshift_r(win32[q0 + i], win32[q0 + i + 1], 8 * sh);
        int acc[kDw1Out];
#pragma unroll
        for (int e = 0; e < kDw1Out; ++e) {
            const int q = e >> 2, r = e & 3;
            const int x0 = (int)__funnelshift_r(xw[q], xw[q + 1], 8 * r);
            const int x1 = (int)__funnelshift_r(xw[q + 1], xw[q + 2], 8 * r);
            acc[e] = __dp4a(x1, (int)tw[1], __dp4a(x0, (int)tw[0], 0));
        }
        if (!kQuant) {
            const int nlive = d.OL - t0 - tl0;   // outputs of this group inside the row
            if (nlive >= kDw1Out) {
#pragma unroll
                for (int e = 0; e < kDw1Out; ++e) lo = min(lo, acc[e]), hi = max(hi, acc[e]);
            } else {
#pragma unroll
                for (int e = 0; e < kDw1Out; ++e)
                    if (e < nlive) lo = min(lo, acc[e]), hi = max(hi, acc[e]);
            }
            continue;
        }
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < kDw1Out; ++e)
            packed[e >> 2] |= (uint32_t)(quantize_bounded(y_of(acc[e]), inv) & 0xff) << (8 * (e & 3));
        {
            uint8_t* out = dst + (int64_t)c * d.OL + t0 + tl0;
            if (aligned && t0 + tl0 + kDw1Out <= d.OL) {
                reinterpret_cast<uint32_t*>(out)[0] = packed[0];
                reinterpret_cast<uint32_t*>(out)[1] = packed[1];
            } else {
#pragma unroll
                for (int e = 0; e < kDw1Out; ++e)
                    if (t0 + tl0 + e < d.OL) out[e] = (uint8_t)(packed[e >> 2] >> (8 * (e & 3)));
            }
        }
    }
    if (kQuant) {
        if (blockIdx.x == 0 && blockIdx.y == 0) write_trailer(dst, (int64_t)d.C * d.OL, scale);
    } else {
        const float mx = lo <= hi ? fmaxf(fabsf(y_of(lo)), fabsf(y_of(hi))) : 0.0f;
        fold_max(mx, amax_bits);
    }
}

// ------------------------------------------------------------ W8A8 row quant
// One CTA per activation row: the row's absmax (floored at 1e-9), then
// q = clamp(round(x * inv)) with inv = 127/amax and the stored scale amax/127.

__global__ void __launch_bounds__(kEltThreads) k_w8a8_rows(const float* __restrict__ x, int64_t K,
                                                           int8_t* __restrict__ q, float* __restrict__ ascale) {
    __shared__ float s_max[kEltThreads / 32];
    const int64_t m = blockIdx.x;
    const float* xr = x + m * K;
    float mx = 0.0f;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) mx = fmaxf(mx, fabsf(xr[k]));
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = s_max[0];
    for (int i = 1; i < kEltThreads / 32; ++i) mx = fmaxf(mx, s_max[i]);
    mx = fmaxf(mx, 1e-9f);
    const float inv = __fdiv_rn(127.0f, mx);
    if (threadIdx.x == 0) ascale[m] = __fdiv_rn(mx, 127.0f);
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) q[m * K + k] = (int8_t)quantize_bounded(xr[k], inv);
}

// W8A8 per-channel weights, one CTA per output channel: amax floored at 1e-9,
// bscale = amax/127, q = clamp(rint(w / bscale)) (division, ties to even).
__global__ void __launch_bounds__(kEltThreads) k_w8a8_weights(const float* __restrict__ w, int64_t K,
                                                              int8_t* __restrict__ wq, float* __restrict__ bscale) {
    __shared__ float s_max[kEltThreads / 32];
    const int64_t n = blockIdx.x;
    const float* wr = w + n * K;
    float mx = 0.0f;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) mx = fmaxf(mx, fabsf(wr[k]));
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = s_max[0];
    for (int i = 1; i < kEltThreads / 32; ++i) mx = fmaxf(mx, s_max[i]);
    mx = fmaxf(mx, 1e-9f);
    const float sc = __fdiv_rn(mx, 127.0f);
    if (threadIdx.x == 0) bscale[n] = sc;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
        const float r = fminf(fmaxf(rintf(__fdiv_rn(wr[k], sc)), -127.0f), 127.0f);
        wq[n * K + k] = (int8_t)(int)r;
    }
}

// The packed W8A8 calls' row quantizer: one block per operand row of each
// distinct activation (rows_pad rows each); a block with m < M quantizes row m
// (1e-9 floor) straight into the GEMM's f16 operand row (exact integers; the
// row holds K rounded up to 64 positions, the tail zero) and its scale, a
// block with m >= M writes a zero row. The same launch clears the
// status word, the amax word and the GEMM's split-tile counters.
constexpr int kW8Cache = 8;   // float4 per thread kept in registers (rows up to 8192 values)

__global__ void __launch_bounds__(kEltThreads) k_w8a8_rows_f16(const __grid_constant__ W8a8RowJobs J) {
    __shared__ float s_max[kEltThreads / 32];
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *J.status = 0u;
        *J.amax_bits = 0u;
    }
    for (unsigned long long i = blockIdx.x * (unsigned long long)kEltThreads + threadIdx.x; i < J.zero_16;
         i += (unsigned long long)gridDim.x * kEltThreads)
        J.zero[i] = make_uint4(0u, 0u, 0u, 0u);
    int j = 0;
    while (j + 1 < J.count && (int)blockIdx.x >= (j + 1) * J.rows_pad) ++j;
    const int64_t m = (int64_t)blockIdx.x - (int64_t)j * J.rows_pad;
    const int64_t K = J.K[j];
    const int64_t Kp = (K + 63) / 64 * 64;   // operand row length, the tail zero
    __half* out = J.xf[j] + m * Kp;
    if (m >= J.M) {   // Kp halves are Kp / 8 16-byte words
        for (int64_t k = threadIdx.x; k < Kp / 8; k += blockDim.x) reinterpret_cast<uint4*>(out)[k] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    for (int64_t k = K + threadIdx.x; k < Kp; k += blockDim.x) out[k] = __float2half_rn(0.0f);
    const float* xr = J.x[j] + m * K;
    // rows whose length is a multiple of 4 start 16-byte aligned: read as
    // float4, kept in registers, written four halves at a time
    const int K4 = (int)(K / 4);
    const bool vec = (K % 4) == 0 && K4 <= kW8Cache * kEltThreads;
    float4 c[kW8Cache];
    float mx = 0.0f;
    if (vec) {
        const float4* x4 = reinterpret_cast<const float4*>(xr);
#pragma unroll
        for (int i = 0; i < kW8Cache; ++i) {
            const int k4 = (int)threadIdx.x + i * kEltThreads;
            c[i] = k4 < K4 ? x4[k4] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(c[i].x), fabsf(c[i].y)), fmaxf(fabsf(c[i].z), fabsf(c[i].w))));
        }
    } else {
        for (int64_t k = threadIdx.x; k < K; k += blockDim.x) mx = fmaxf(mx, fabsf(xr[k]));
    }
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = s_max[0];
    for (int i = 1; i < kEltThreads / 32; ++i) mx = fmaxf(mx, s_max[i]);
    mx = fmaxf(mx, 1e-9f);
    const float inv = __fdiv_rn(127.0f, mx);
    if (threadIdx.x == 0) J.ascale[j][m] = __fdiv_rn(mx, 127.0f);
    if (vec) {
        uint2* o2 = reinterpret_cast<uint2*>(out);
#pragma unroll
        for (int i = 0; i < kW8Cache; ++i) {
            const int k4 = (int)threadIdx.x + i * kEltThreads;
            if (k4 < K4) {
                const __half2 lo = __halves2half2(__int2half_rn(quantize_bounded(c[i].x, inv)),
                                                  __int2half_rn(quantize_bounded(c[i].y, inv)));
                const __half2 hi = __halves2half2(__int2half_rn(quantize_bounded(c[i].z, inv)),
                                                  __int2half_rn(quantize_bounded(c[i].w, inv)));
                o2[k4] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
            }
        }
    } else {
        for (int64_t k = threadIdx.x; k < K; k += blockDim.x) out[k] = __int2half_rn(quantize_bounded(xr[k], inv));
    }
}

// int8 -> f16 (exact), 16 values per thread and step.
__global__ void __launch_bounds__(kEltThreads) k_i8_to_f16(const int8_t* __restrict__ src, int64_t n16,
                                                           __half* __restrict__ dst) {
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += step) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        __align__(16) __half h[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) h[j] = __int2half_rn(byte_of(w[j >> 2], j & 3));
        uint4* o = reinterpret_cast<uint4*>(dst + 16 * i);
        o[0] = *reinterpret_cast<const uint4*>(&h[0]);
        o[1] = *reinterpret_cast<const uint4*>(&h[8]);
    }
}

int elt_grid(int64_t work) {
    const int64_t want = (work + kEltThreads - 1) / kEltThreads;
    const int cap = device_sm_count() * 8;
    return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_add_scaled(const uint8_t* a, const uint8_t* b, int64_t n, unsigned int* amax_bits, uint8_t* dst,
                              cudaStream_t s) {
    const int grid = elt_grid(n / 16 + 1);
    k_add_amax<<<grid, kEltThreads, 0, s>>>(a, b, n, amax_bits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pdl(k_add_quant, dim3(grid), dim3(kEltThreads), 0, s, a, b, n, (const unsigned int*)amax_bits, dst);
}

// the two passes of the short-row rms_norm (the second a programmatic dependent)
template <int V, bool kGamma>
cudaError_t run_rms_t(int grid, const uint8_t* x, int64_t rows, float eps, const float* gamma, unsigned int* amax_bits,
                      uint8_t* dst, cudaStream_t s) {
    k_rms_rows_t<V, kGamma><<<grid, kEltThreads, 0, s>>>(x, rows, eps, gamma, amax_bits);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pdl(k_rms_quant_t<V, kGamma>, dim3(grid), dim3(kEltThreads), 0, s, x, rows, eps, gamma,
                      (const unsigned int*)amax_bits, dst);
}

cudaError_t launch_rms_norm_scaled(const uint8_t* x, int64_t rows, int64_t ne0, float eps, const float* gamma,
                                   float* rfac, unsigned int* amax_bits, uint8_t* dst, cudaStream_t s) {
    if (ne0 % 16 == 0 && ne0 <= 64) {   // short rows: one thread per row
        const int grid = elt_grid(rows);
        cudaError_t e = cudaSuccess;
        switch (ne0 / 16) {
            case 1: e = gamma ? run_rms_t<1, true>(grid, x, rows, eps, gamma, amax_bits, dst, s)
                              : run_rms_t<1, false>(grid, x, rows, eps, gamma, amax_bits, dst, s); break;
            case 2: e = gamma ? run_rms_t<2, true>(grid, x, rows, eps, gamma, amax_bits, dst, s)
                              : run_rms_t<2, false>(grid, x, rows, eps, gamma, amax_bits, dst, s); break;
            case 3: e = gamma ? run_rms_t<3, true>(grid, x, rows, eps, gamma, amax_bits, dst, s)
                              : run_rms_t<3, false>(grid, x, rows, eps, gamma, amax_bits, dst, s); break;
            default: e = gamma ? run_rms_t<4, true>(grid, x, rows, eps, gamma, amax_bits, dst, s)
                               : run_rms_t<4, false>(grid, x, rows, eps, gamma, amax_bits, dst, s); break;
        }
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    k_rms_rows<<<elt_grid(rows * 32), kEltThreads, 0, s>>>(x, rows, ne0, eps, gamma, rfac, amax_bits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pdl(k_rms_quant, dim3(elt_grid(rows * 32)), dim3(kEltThreads), 0, s, x, rows, ne0, gamma,
                      (const float*)rfac, (const unsigned int*)amax_bits, dst);
}

cudaError_t launch_i8s_transpose(const uint8_t* src, int64_t a, int64_t b, uint8_t* dst, cudaStream_t s) {
    // 16 KB tiles (sixteen 4-byte loads per thread in flight) where the rows
    // are wide or narrow enough to fill them, then 8 KB, 4 KB in between
    if (b >= 512) {
        const int64_t ta = (a + 31) / 32, tb = (b + 511) / 512;
        k_transpose<32, 512><<<(unsigned)(ta * tb), kEltThreads, 0, s>>>(src, a, b, dst, tb);
    } else if (b >= 256) {
        const int64_t ta = (a + 31) / 32, tb = (b + 255) / 256;
        k_transpose<32, 256><<<(unsigned)(ta * tb), kEltThreads, 0, s>>>(src, a, b, dst, tb);
    } else if (b >= 128) {
        const int64_t ta = (a + 31) / 32, tb = (b + 127) / 128;
        k_transpose<32, 128><<<(unsigned)(ta * tb), kEltThreads, 0, s>>>(src, a, b, dst, tb);
    } else if (a >= 512) {
        const int64_t ta = (a + 511) / 512, tb = (b + 31) / 32;
        k_transpose<512, 32><<<(unsigned)(ta * tb), kEltThreads, 0, s>>>(src, a, b, dst, tb);
    } else {
        const int64_t ta = (a + 255) / 256, tb = (b + 31) / 32;
        k_transpose<256, 32><<<(unsigned)(ta * tb), kEltThreads, 0, s>>>(src, a, b, dst, tb);
    }
    return cudaGetLastError();
}

cudaError_t launch_im2col_asym(const uint8_t* src, int64_t C, int64_t L, int KW, int stride, int pad_l, int64_t OL,
                               uint8_t* dst, cudaStream_t s) {
    // windowed kernel: T output positions per block (a multiple of 4, at most
    // 256) whose C windows fit in 48 KB of shared memory
    // per channel 4*Wc bytes of staged words (W window bytes, up to 3 bytes of
    // alignment shift, one spare word) and one shift word
    if (KW == 4 && stride == 2 && C % 32 == 0 && L % 16 == 0 && (pad_l & 1) == 0 &&
        ((uintptr_t)src & 15u) == 0 && ((uintptr_t)dst & 15u) == 0) {
        const int64_t warps = (C / 32) * ((OL + 31) / 32);
        const unsigned blocks = (unsigned)((warps * 32 + kEltThreads - 1) / kEltThreads);
        switch (((16 - pad_l % 16) % 16) / 2) {   // the window start's offset in its 16-byte chunk, halved
            case 0: k_im2col_k4s2<0><<<blocks, kEltThreads, 0, s>>>(src, (int)C, L, pad_l, OL, dst); break;
            case 1: k_im2col_k4s2<2><<<blocks, kEltThreads, 0, s>>>(src, (int)C, L, pad_l, OL, dst); break;
            case 2: k_im2col_k4s2<4><<<blocks, kEltThreads, 0, s>>>(src, (int)C, L, pad_l, OL, dst); break;
            case 3: k_im2col_k4s2<6><<<blocks, kEltThreads, 0, s>>>(src, (int)C, L, pad_l, OL, dst); break;
            case 4: k_im2col_k4s2<8><<<blocks, kEltThreads, 0, s>>>(src, (int)C, L, pad_l, OL, dst); break;
            case 5: k_im2col_k4s2<10><<<blocks, kEltThreads, 0, s>>>(src, (int)C, L, pad_l, OL, dst); break;
            case 6: k_im2col_k4s2<12><<<blocks, kEltThreads, 0, s>>>(src, (int)C, L, pad_l, OL, dst); break;
            default: k_im2col_k4s2<14><<<blocks, kEltThreads, 0, s>>>(src, (int)C, L, pad_l, OL, dst); break;
        }
        return cudaGetLastError();
    }
    constexpr int64_t kWinBytes = 48 * 1024;
    auto smem_for = [&](int64_t T_) {
        const int64_t W_ = (T_ - 1) * stride + KW;
        return C * (4 * ((W_ + 6) / 4 + 1) + 4);
    };
    int64_t T = 256;   // more blocks per SM overlap one block's staging with another's stores
    while (T >= 4 && smem_for(T) > kWinBytes) T -= 4;
    if (T >= 4) {
        const int64_t W = (T - 1) * stride + KW;
        const int64_t blocks = (OL + T - 1) / T;
        k_im2col_win<<<(unsigned)blocks, kEltThreads, (size_t)smem_for(T), s>>>(src, (int)C, (int)L, KW, stride,
                                                                                pad_l, (int)OL, (int)T, (int)W, dst);
        return cudaGetLastError();
    }
    k_im2col<<<elt_grid(OL * C * KW / 4 + 1), kEltThreads, 0, s>>>(src, (int)C, (int)L, KW, stride, pad_l, (int)OL,
                                                                   dst);
    return cudaGetLastError();
}

cudaError_t launch_depthwise(const uint8_t* w, const uint8_t* x, const float* bias, int64_t C, int64_t L, int KW,
                             int stride, int pad_l, int64_t OL, int relu, unsigned int* amax_bits, uint8_t* dst,
                             cudaStream_t s) {
    const DwArgs d{w, x, bias, (int)C, (int)L, (int)OL, KW, stride, pad_l, relu};
    if (stride == 1 && KW <= 8 && C <= 65535) {   // the 7-tap causal blocks: dp4a
        const dim3 g((unsigned)((OL + kDw1T - 1) / kDw1T), (unsigned)C);
        // bias and ReLU as template parameters: no per-output test of either
        auto run = [&](auto pass1, auto pass2) {
            pass1<<<g, kEltThreads, 0, s>>>(d, amax_bits, dst);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
            return launch_pdl(pass2, g, dim3(kEltThreads), 0, s, d, amax_bits, dst);
        };
        if (d.bias && d.relu) return run(k_dw_s1<false, true, true>, k_dw_s1<true, true, true>);
        if (d.bias) return run(k_dw_s1<false, true, false>, k_dw_s1<true, true, false>);
        if (d.relu) return run(k_dw_s1<false, false, true>, k_dw_s1<true, false, true>);
        return run(k_dw_s1<false, false, false>, k_dw_s1<true, false, false>);
    }
    const int64_t W = (int64_t)(kDwT - 1) * stride + KW;
    if (C <= 65535 && KW <= 64 && W + KW <= 48 * 1024) {   // windowed kernel
        const dim3 g((unsigned)((OL + kDwT - 1) / kDwT), (unsigned)C);
        const size_t sm = (size_t)(W + KW);
        k_dw_win<false><<<g, kEltThreads, sm, s>>>(d, (int)W, amax_bits, dst);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_pdl(k_dw_win<true>, g, dim3(kEltThreads), sm, s, d, (int)W, amax_bits, dst);
    }
    const int grid = elt_grid(C * OL / 4 + 1);
    k_dw_amax<<<grid, kEltThreads, 0, s>>>(d, amax_bits);
    k_dw_quant<<<grid, kEltThreads, 0, s>>>(d, amax_bits, dst);
    return cudaGetLastError();
}

cudaError_t launch_w8a8_rows(const float* x, int64_t M, int64_t K, int8_t* q, float* ascale, cudaStream_t s) {
    k_w8a8_rows<<<(unsigned)M, kEltThreads, 0, s>>>(x, K, q, ascale);
    return cudaGetLastError();
}

cudaError_t launch_w8a8_rows_f16(const W8a8RowJobs& J, cudaStream_t s) {
    k_w8a8_rows_f16<<<(unsigned)(J.count * J.rows_pad), kEltThreads, 0, s>>>(J);
    return cudaGetLastError();
}

cudaError_t launch_i8_to_f16(const int8_t* src, int64_t n, __half* dst, cudaStream_t s) {
    k_i8_to_f16<<<elt_grid(n / 16), kEltThreads, 0, s>>>(src, n / 16, dst);
    return cudaGetLastError();
}

cudaError_t launch_w8a8_weights(const float* w, int64_t N, int64_t K, int8_t* wq, float* bscale, cudaStream_t s) {
    k_w8a8_weights<<<(unsigned)N, kEltThreads, 0, s>>>(w, K, wq, bscale);
    return cudaGetLastError();
}

}  // namespace i2s
