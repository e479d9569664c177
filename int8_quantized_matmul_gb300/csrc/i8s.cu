// I8_S x I8_S fused mul_mat_add(_relu) and the per-tensor requantization
// ("ggml: additive INT8/ternary types, fused CPU ops, and kernels for VibeASR
// (1/2)", sections "Two new types" and "Five fused INT8 ops").
//
// The matmul epilogue forms y = (float)acc * (w_scale * x_scale) + bias[n],
// applies ReLU if asked, writes y (F32) to the workspace and folds max|y| into
// one word with atomicMax on the float bits (valid because |y| >= 0, where the
// IEEE order equals the unsigned order). The requant pass then turns the F32
// tensor into I8_S with one scale, as the op's output must be self-describing.
// Two passes are needed because the scale depends on the whole output.
//
// This file holds the requantization kernels and the pre-pass that writes the
// matmul's f16 operand rows; the matmul with its fused epilogue is the
// tensor-core kernel in i8s_tc.cu.

#include "common.cuh"
#include "internal.h"

namespace i2s {

namespace {

__global__ void __launch_bounds__(256) k_absmax(const float* __restrict__ y, int64_t n, unsigned int* amax_bits) {
    __shared__ float s_max[8];
    float mx = 0.0f;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) mx = fmaxf(mx, fabsf(y[i]));
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < 8; ++i) mx = fmaxf(mx, s_max[i]);
        atomicMax(amax_bits, __float_as_uint(fmaxf(mx, s_max[0])));
    }
}

// y (F32, n) -> I8_S bytes at dst: int8 payload, zero padding to 32 bytes, the
// F32 scale and 28 zero bytes. Each thread keeps U float4 loads in flight (a
// warp's loads cover 512 contiguous bytes per step); the host picks U so that
// one wave of resident CTAs covers the tensor.
template <int U>
__global__ void __launch_bounds__(256) k_requant(const float* __restrict__ y, int64_t n,
                                                 const unsigned int* __restrict__ amax_bits, uint8_t* dst) {
    pdl_wait();   // y and the folded amax come from the launch before
    float scale, inv;
    quant_params(__uint_as_float(*amax_bits), scale, inv);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t n4 = n / 4;
    const float4* y4 = reinterpret_cast<const float4*>(y);
    uint32_t* d4 = reinterpret_cast<uint32_t*>(dst);
    for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i0 < n4; i0 += U * stride) {
        float4 v[U];
#pragma unroll
        for (int e = 0; e < U; ++e) {
            const int64_t i = i0 + e * stride;
            v[e] = i < n4 ? y4[i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int e = 0; e < U; ++e) {
            const int64_t i = i0 + e * stride;
            if (i < n4)
                d4[i] = (uint32_t)(quantize_one(v[e].x, inv) & 0xff) | ((uint32_t)(quantize_one(v[e].y, inv) & 0xff) << 8) |
                        ((uint32_t)(quantize_one(v[e].z, inv) & 0xff) << 16) |
                        ((uint32_t)(quantize_one(v[e].w, inv) & 0xff) << 24);
        }
    }
    if (blockIdx.x == 0) {
        const int64_t padded = (n + 31) / 32 * 32;
        for (int64_t i = n4 * 4 + threadIdx.x; i < padded + 32; i += blockDim.x) {
            uint8_t b = 0;
            if (i < n) b = (uint8_t)(quantize_one(y[i], inv) & 0xff);
            else if (i >= padded && i < padded + 4) b = (uint8_t)(__float_as_uint(scale) >> (8 * (i - padded)));
            dst[i] = b;
        }
    }
}

// Four int8 (one 32-bit word) -> two f16x2 words, exactly: byte b becomes the
// f16 bit pattern 0x6400 | (b ^ 0x80) = 1152 + x (f16 integers are exact up to
// 2048), and one f16 subtraction of 1152 leaves x.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t t0 = __byte_perm(w, 0x64u, 0x4140) ^ 0x00800080u;   // bytes 0, 1
    const uint32_t t1 = __byte_perm(w, 0x64u, 0x4342) ^ 0x00800080u;   // bytes 2, 3
    const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480),
                                        __ushort_as_half((unsigned short)0x6480));   // 1152
    const __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&t0), bias);
    const __half2 h1 = __hsub2(*reinterpret_cast<const __half2*>(&t1), bias);
    lo = *reinterpret_cast<const uint32_t*>(&h0);
    hi = *reinterpret_cast<const uint32_t*>(&h1);
}

// int8 -> f16 rows of the weights (N x K) and activations (M x K, zero rows up
// to rows_pad); also clears the status and amax words and the split-tile
// tickets and masks. One unit is 8 values: 8 bytes in, 16 bytes out, so a
// warp's loads cover 256 contiguous bytes and its stores 512. Units [0, nw)
// are the weights, [nw, nw + nx_pad) the activations, those past nw + nx the
// zero rows (a zero byte converts to +0). Each thread keeps U units' loads in
// flight; the host picks U so that one wave of resident CTAs covers the call.
__device__ __forceinline__ void i8x8_to_f16(const uint2 v, uint4& o) {
    i8x4_to_f16x4(v.x, o.x, o.y);
    i8x4_to_f16x4(v.y, o.z, o.w);
}

template <int U>
__global__ void __launch_bounds__(256) k_i8s_to_f16(const uint2* __restrict__ w, unsigned long long nw,
                                                    uint4* __restrict__ wf, const uint2* __restrict__ x,
                                                    unsigned long long nx, unsigned long long nx_pad,
                                                    uint4* __restrict__ xf, uint4* zero, unsigned long long zero_16,
                                                    uint32_t* status, unsigned int* amax_bits) {
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    const unsigned long long t0 = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
    pdl_wait();   // the launch before may still use this workspace (or produce x)
    if (t0 == 0) {
        *status = 0u;
        *amax_bits = 0u;
    }
    for (unsigned long long i = t0; i < zero_16; i += stride) zero[i] = make_uint4(0u, 0u, 0u, 0u);
    const unsigned long long total = nw + nx_pad;
    for (unsigned long long i0 = t0; i0 < total; i0 += U * stride) {
        uint2 v[U];
#pragma unroll
        for (int e = 0; e < U; ++e) {
            const unsigned long long i = i0 + e * stride;
            v[e] = make_uint2(0u, 0u);
            if (i < nw) v[e] = __ldg(w + i);
            else if (i - nw < nx) v[e] = __ldg(x + (i - nw));
        }
#pragma unroll
        for (int e = 0; e < U; ++e) {
            const unsigned long long i = i0 + e * stride;
            if (i >= total) break;
            uint4 o;
            i8x8_to_f16(v[e], o);
            if (i < nw) wf[i] = o;
            else xf[i - nw] = o;
        }
    }
}

// K that is not a multiple of 64: src rows of K int8 (not 16-byte aligned)
// -> dst rows of Kp f16, positions K..Kp-1 and rows rows_in..rows_out-1 zero.
// Zero products add nothing, so the padded contraction is the same integer
// sum. One 16-byte output word (8 values) per thread and step, byte loads.
__device__ __forceinline__ void convert_rows_ragged(const int8_t* __restrict__ src, int rows_in, int rows_out, int K,
                                                    int Kp, uint4* __restrict__ dst, unsigned long long t0,
                                                    unsigned long long stride) {
    const unsigned long long words_per_row = (unsigned long long)(Kp / 8);
    const unsigned long long n = (unsigned long long)rows_out * words_per_row;
    for (unsigned long long i = t0; i < n; i += stride) {
        const int r = (int)(i / words_per_row);
        const int k0 = (int)(i - (unsigned long long)r * words_per_row) * 8;
        __align__(16) __half h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int k = k0 + j;
            const int v = (r < rows_in && k < K) ? (int)src[(size_t)r * K + k] : 0;
            h[j] = __int2half_rn(v);
        }
        dst[i] = *reinterpret_cast<const uint4*>(h);
    }
}

__global__ void __launch_bounds__(256) k_i8s_to_f16_ragged(const int8_t* __restrict__ w, int N, __half* __restrict__ wf,
                                                           const int8_t* __restrict__ x, int M, int rows_pad,
                                                           __half* __restrict__ xf, int K, int Kp, uint4* zero,
                                                           unsigned long long zero_16, uint32_t* status,
                                                           unsigned int* amax_bits) {
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    const unsigned long long t0 = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
    pdl_wait();   // the launch before may still use this workspace (or produce x)
    if (t0 == 0) {
        *status = 0u;
        *amax_bits = 0u;
    }
    for (unsigned long long i = t0; i < zero_16; i += stride) zero[i] = make_uint4(0u, 0u, 0u, 0u);
    if (w) convert_rows_ragged(w, N, N, K, Kp, reinterpret_cast<uint4*>(wf), t0, stride);
    convert_rows_ragged(x, M, rows_pad, K, Kp, reinterpret_cast<uint4*>(xf), t0, stride);
}

__global__ void __launch_bounds__(256) k_i8_to_f16_rows(const int8_t* __restrict__ src, int rows, int K, int Kp,
                                                        __half* __restrict__ dst) {
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    convert_rows_ragged(src, rows, rows, K, Kp, reinterpret_cast<uint4*>(dst),
                        blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x, stride);
}

int prepass_grid(unsigned long long n16) {
    const unsigned long long want = (n16 + 1023) / 1024;
    const int cap = device_sm_count() * 8;
    return (int)(want < (unsigned long long)cap ? (want < 1 ? 1 : want) : cap);
}

// Units in flight per thread for `units` conversion units: the fewest that let
// one wave of CTAs (eight of 256 threads per SM) cover the call, at most 16.
int prepass_units(unsigned long long units, int& grid) {
    const unsigned long long wave = (unsigned long long)device_sm_count() * 8 * 256;
    int u = 1;
    while (u < 16 && units > wave * (unsigned long long)u) u *= 2;
    unsigned long long g = (units + 256ull * u - 1) / (256ull * u);
    const unsigned long long cap = wave / 256;
    grid = (int)(g < 1 ? 1 : (g > cap ? cap : g));
    return u;
}

int grid_for(int64_t n4) {
    const int64_t want = (n4 + 255) / 256;
    const int cap = device_sm_count() * 8;
    return (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace


cudaError_t launch_i8s_to_f16(const int8_t* w, int N, __half* wf, const int8_t* x, int M, int rows_pad, int K,
                              __half* xf, void* zero, size_t zero_bytes, uint32_t* status, unsigned int* amax_bits,
                              cudaStream_t s) {
    const int Kp = (int)i8s_kpad(K);
    if (Kp != K) {
        const unsigned long long n8 = (unsigned long long)(N > rows_pad ? N : rows_pad) * (unsigned long long)(Kp / 8);
        return launch_pdl(k_i8s_to_f16_ragged, dim3(prepass_grid(n8 / 4)), dim3(256), 0, s, w, N, wf, x, M, rows_pad,
                          xf, K, Kp, static_cast<uint4*>(zero), (unsigned long long)(zero_bytes / 16), status,
                          amax_bits);
    }
    const unsigned long long nw = w ? (unsigned long long)N * K / 8 : 0ull;
    const unsigned long long nx = (unsigned long long)M * K / 8, nxp = (unsigned long long)rows_pad * K / 8;
    int grid = 1;
    const int u = prepass_units(nw + nxp, grid);
    auto go = [&](auto kern) {
        return launch_pdl(kern, dim3(grid), dim3(256), 0, s, reinterpret_cast<const uint2*>(w), nw,
                          reinterpret_cast<uint4*>(wf), reinterpret_cast<const uint2*>(x), nx, nxp,
                          reinterpret_cast<uint4*>(xf), static_cast<uint4*>(zero),
                          (unsigned long long)(zero_bytes / 16), status, amax_bits);
    };
    switch (u) {
        case 1: return go(k_i8s_to_f16<1>);
        case 2: return go(k_i8s_to_f16<2>);
        case 4: return go(k_i8s_to_f16<4>);
        case 8: return go(k_i8s_to_f16<8>);
        default: return go(k_i8s_to_f16<16>);
    }
}

cudaError_t launch_i8_to_f16_rows(const int8_t* src, int64_t rows, int64_t K, __half* dst, cudaStream_t s) {
    const int Kp = (int)i8s_kpad(K);
    k_i8_to_f16_rows<<<prepass_grid((unsigned long long)rows * (Kp / 8) / 4), 256, 0, s>>>(src, (int)rows, (int)K, Kp,
                                                                                          dst);
    return cudaGetLastError();
}

cudaError_t launch_absmax(const float* y, int64_t n, unsigned int* amax_bits, cudaStream_t s) {
    k_absmax<<<grid_for(n), 256, 0, s>>>(y, n, amax_bits);
    return cudaGetLastError();
}

cudaError_t launch_requant(const float* y, int64_t n, const unsigned int* amax_bits, uint8_t* dst, cudaStream_t s) {
    // the fewest float4 loads in flight per thread (at most 8) that let one
    // wave of CTAs (eight of 256 threads per SM) cover the tensor; a
    // programmatic dependent of the launch before
    const int64_t n4 = n / 4, wave = (int64_t)device_sm_count() * 8 * 256;
    int u = 1;
    while (u < 8 && n4 > wave * u) u *= 2;
    const int64_t g = (n4 + 256 * u - 1) / (256 * u), cap = wave / 256;
    const dim3 grid((unsigned)(g < 1 ? 1 : (g > cap ? cap : g)));
    switch (u) {
        case 1: return launch_pdl(k_requant<1>, grid, dim3(256), 0, s, y, n, amax_bits, dst);
        case 2: return launch_pdl(k_requant<2>, grid, dim3(256), 0, s, y, n, amax_bits, dst);
        case 4: return launch_pdl(k_requant<4>, grid, dim3(256), 0, s, y, n, amax_bits, dst);
        default: return launch_pdl(k_requant<8>, grid, dim3(256), 0, s, y, n, amax_bits, dst);
    }
}

}  // namespace i2s
