// Per-row activation quantization ("ggml-cpu: ternary I2_S matmul kernel",
// sections Arithmetic and Kernels; "VibeASR in audio.cpp", section Encoder for
// the 1e-5 amax floor; "Experiment - int8 W8A8 path", section Implementation
// for scale = amax/127, inv = 127/amax, round, clamp to +-127).
//
// One CTA per row: the row is read once into registers, a block reduction
// finds its absmax, and the quantized values and their int8 sum (reduced the
// same way) are written out: as plain int8 rows (the public sidecar,
// k_quant_rows), or straight into the operand layout of the two tensor-core
// matmuls, so no separate repacking pass is needed (kQuantE2M1Tc: each q as
// three base-8 digits in e2m1, one operand row per digit, k_quant_rows_tc4).

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "quant_tc.cuh"

namespace i2s {

// Writes the four quantized values of positions 4c..4c+3 of row m as plain
// int8 (the public sidecar layout).
__device__ __forceinline__ void emit4(const QuantJob& J, int m, int c, const int (&q)[4]) {
    uint32_t* q4 = reinterpret_cast<uint32_t*>(static_cast<int8_t*>(J.out) + (size_t)m * J.K);
    q4[c] = (uint32_t)(q[0] & 0xff) | ((uint32_t)(q[1] & 0xff) << 8) | ((uint32_t)(q[2] & 0xff) << 16) |
            ((uint32_t)(q[3] & 0xff) << 24);
}

constexpr int kQThreads = 256;
constexpr int kQ4Cache = 3;   // 16-value digit units cached per thread (rows up to 12288 values)
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
            emit4(J, m, c, q);
        }
    }
    for (int c = tid + kQCache * kQThreads; c < K4; c += kQThreads) {
        const float4 v = x4[c];
        const int q[4] = {quantize_one(v.x, inv), quantize_one(v.y, inv), quantize_one(v.z, inv), quantize_one(v.w, inv)};
        sum += q[0] + q[1] + q[2] + q[3];
        emit4(J, m, c, q);
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

// The e2m1 digit operand (kQuantE2M1Tc). Rows of at most kQuantWarpRowK
// positions (the first n_short jobs) are quantized one per warp, eight rows
// per CTA, with warp-level reductions only; longer rows take a whole CTA.
__global__ void __launch_bounds__(kQThreads) k_quant_rows_tc4(const __grid_constant__ QuantArgs a) {
    __shared__ float s_red[kQThreads / 32];
    __shared__ int s_sum[kQThreads / 32];
    __shared__ uint32_t s_code[255];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 255) s_code[tid] = digit_code(tid - 127);
    __syncthreads();
    // launched as a programmatic dependent of the kernel before it: wait for
    // that kernel (which may use the same workspace, or produce x) before
    // reading or writing global memory
    pdl_wait();
    if (a.status && blockIdx.x == 0 && tid == 0) *a.status = 0u;
    // map i is written by thread i / gridDim.x of CTA i % gridDim.x: one or two
    // maps per CTA instead of all of them in the first CTA, whose row work
    // would otherwise wait behind them
    for (int i = blockIdx.x + (int)gridDim.x * tid; i < a.n_wmaps; i += (int)gridDim.x * kQThreads)
        write_weight_map(a.wtmpl, a.wmaps + i, a.wj[i].w, a.wj[i].N, a.wj[i].K);
    for (unsigned long long i = blockIdx.x * (unsigned long long)kQThreads + tid; i < a.zero_16;
         i += (unsigned long long)gridDim.x * kQThreads)
        a.zero[i] = make_uint4(0u, 0u, 0u, 0u);
    const int Mp = a.rows;
    const int short_blocks = a.n_short * a.short_ctas;
    if ((int)blockIdx.x < short_blocks) {   // one warp per row
        const QuantJob& J = a.j[blockIdx.x / a.short_ctas];
        const int m = (blockIdx.x % a.short_ctas) * (kQThreads / 32) + warp;
        if (m >= a.M) return;
        const int K = J.K, U = K / 16;   // U <= 32 * kQ4Cache
        const float4* x4 = reinterpret_cast<const float4*>(J.x + (size_t)m * K);
        float4 cache[kQ4Cache][4];
        float amax = 0.0f;
#pragma unroll
        for (int c = 0; c < kQ4Cache; ++c) {
            const int u = lane + 32 * c;
            if (u < U) {
                load_unit(x4, u, cache[c]);
                amax = fmaxf(amax, unit_amax(cache[c]));
            }
        }
        amax = warp_max(amax);
        float scale, inv;
        quant_params(amax, scale, inv);
        int sum = 0;
#pragma unroll
        for (int c = 0; c < kQ4Cache; ++c) {
            const int u = lane + 32 * c;
            if (u < U) sum += emit_unit(cache[c], inv, u, static_cast<uint8_t*>(J.out), (size_t)K / 2, Mp, m, s_code);
        }
        sum = warp_sum(sum);
        if (lane == 0) {
            J.scale[m] = scale;
            J.sum[m] = sum;
        }
        return;
    }
    const int b = (int)blockIdx.x - short_blocks;   // one CTA per row
    const QuantJob& J = a.j[a.n_short + b / a.M];
    const int m = b % a.M;
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

static_assert(kQuantWarpRowK / 16 <= 32 * kQ4Cache, "a short row fits one warp's registers");

// Tiled I2_S weights: one thread per 16-byte piece of the output. Piece p of
// row rr in block (bi, bj) holds bytes 128 bj + 16 (p ^ (rr % 8)) .. +15 of
// payload row 128 bi + rr (the 128-byte swizzle of a TMA tile of 128 rows x
// 128 bytes), or zeros past N or past the row's bytes.
__global__ void __launch_bounds__(256) k_i2s_tile(const uint8_t* __restrict__ w, int64_t N, int row_bytes, int tk,
                                                  int64_t pieces, uint4* __restrict__ out) {
    constexpr int kPiecesPerRow = kTiledRowBytes / 16;
    constexpr int kPiecesPerBlock = kTiledBlockBytes / 16;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < pieces; t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = t / kPiecesPerBlock;
        const int in = (int)(t - blk * kPiecesPerBlock);
        const int rr = in / kPiecesPerRow, p = in % kPiecesPerRow;
        const int64_t bi = blk / tk;
        const int bj = (int)(blk - bi * tk);
        const int64_t row = bi * kTiledRows + rr;
        const int byte = bj * kTiledRowBytes + ((p ^ (rr & 7)) << 4);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < N && byte < row_bytes) v = __ldg(reinterpret_cast<const uint4*>(w + row * row_bytes + byte));
        out[t] = v;
    }
}

cudaError_t launch_i2s_tile(const uint8_t* w, int64_t N, int64_t K, uint8_t* tiled, cudaStream_t s) {
    const int64_t pieces = (int64_t)(tiled_scale_offset(N, K) / 16);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t want = (pieces + 255) / 256;
    const int grid = (int)(want < 8LL * sms ? want : 8LL * sms);
    k_i2s_tile<<<grid, 256, 0, s>>>(w, N, (int)(K / 4), (int)tiled_col_blocks(K), pieces, reinterpret_cast<uint4*>(tiled));
    return cudaGetLastError();
}

cudaError_t launch_quant(QuantArgs& a, cudaStream_t s) {
    if (a.layout == kQuantE2M1Tc) {
        // short rows first (stable), eight rows per CTA; then one CTA per long row
        std::stable_partition(a.j, a.j + a.count, [](const QuantJob& q) { return q.K <= kQuantWarpRowK; });
        a.n_short = 0;
        while (a.n_short < a.count && a.j[a.n_short].K <= kQuantWarpRowK) ++a.n_short;
        a.short_ctas = (a.M + kQThreads / 32 - 1) / (kQThreads / 32);
        // the decode path: a programmatic dependent of the kernel before it
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(a.n_short * a.short_ctas + (a.count - a.n_short) * a.M), 1, 1);
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
