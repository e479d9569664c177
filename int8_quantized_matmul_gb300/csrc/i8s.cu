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
// This file holds the requantization kernels; the matmul with its fused
// epilogue is the tensor-core kernel in i8s_tc.cu.

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

int grid_for(int64_t n4) {
    const int64_t want = (n4 + 255) / 256;
    const int cap = device_sm_count() * 8;
    return (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace


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
