// Per-row activation quantization ("ggml-cpu: ternary I2_S matmul kernel",
// sections Arithmetic and Kernels; "VibeASR in audio.cpp", section Encoder for
// the 1e-5 amax floor; "Experiment - int8 W8A8 path", section Implementation
// for scale = amax/127, inv = 127/amax, round, clamp to +-127).
//
// One warp per row: a shuffle reduction finds the row's absmax, then the row
// is read again (L1/L2 hit) and quantized. The int8 row sum is reduced the same
// way. Besides the plain int8 layout of the public sidecar, the kernel can
// write the operand layouts of the two matmul kernels directly, so no separate
// repacking pass is needed:
//   kQuantE4M3Frag  the decode GEMV's B operand: each q is split exactly into
//                   16*(q>>4) and (q&15), both exact in e4m3, stored in the
//                   warp-MMA fragment order (see gemv.cu);
//   kQuantF16Perm   the tensor-core GEMM's activation operand: q as f16 in the
//                   K order in which the GEMM expands the packed codes.

#include "common.cuh"
#include "internal.h"

namespace i2s {

// Word index, inside one row's GEMV operand records, of the e4m3 byte quad that
// holds positions p..p+3 (p % 4 == 0). A record covers 256 positions (64 bytes
// of codes per weight row) for one lane quad t; see gemv.cu for the matching
// fragment layout. Returns the index of the "high" word; the "low" word is +2.
__device__ __forceinline__ int frag_word(int p) {
    const int kb = p >> 8;          // 256-position block
    const int r = p & 255;
    const int half = r >> 7;        // which 32-byte group of the block
    const int p2 = r & 127;         // group-relative position
    const int slice = p2 >> 5;      // bit-pair slice: shift 6, 4, 2, 0
    const int gp = p2 & 31;         // byte within the group
    const int t = 2 * half + (gp >> 4);
    const int i = (gp >> 2) & 3;    // 32-bit word within the lane's 16 bytes
    const int h = slice >> 1;       // MMA pair: shifts (6,4) or (2,0)
    const int b = slice & 1;        // first or second k-half of the MMA
    return (kb * 4 + t) * 32 + 4 * (2 * i + h) + b;
}

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

__global__ void __launch_bounds__(256) k_quant_rows(const __grid_constant__ QuantArgs a) {
    const int gw = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (a.status && blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
    if (gw >= a.count * a.M) return;
    const QuantJob& J = a.j[gw / a.M];
    const int m = gw % a.M;
    const int K = J.K;
    const float4* x4 = reinterpret_cast<const float4*>(J.x + (size_t)m * K);

    float amax = 0.0f;
    for (int c = lane; c < K / 4; c += 32) {
        const float4 v = x4[c];
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    amax = warp_max(amax);
    float scale, inv;
    quant_params(amax, scale, inv);

    int sum = 0;
    if (a.layout == kQuantI8Rows) {
        uint32_t* q4 = reinterpret_cast<uint32_t*>(static_cast<int8_t*>(J.out) + (size_t)m * K);
        for (int c = lane; c < K / 4; c += 32) {
            const float4 v = x4[c];
            const int q0 = quantize_one(v.x, inv), q1 = quantize_one(v.y, inv);
            const int q2 = quantize_one(v.z, inv), q3 = quantize_one(v.w, inv);
            sum += q0 + q1 + q2 + q3;
            q4[c] = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8) | ((uint32_t)(q2 & 0xff) << 16) |
                    ((uint32_t)(q3 & 0xff) << 24);
        }
    } else if (a.layout == kQuantE4M3Frag) {
        uint32_t* rec = static_cast<uint32_t*>(J.out) + (size_t)m * (J.Kp / 2);
        for (int c = lane; c < J.Kp / 4; c += 32) {
            int q[4] = {0, 0, 0, 0};
            if (4 * c < K) {
                const float4 v = x4[c];
                q[0] = quantize_one(v.x, inv); q[1] = quantize_one(v.y, inv);
                q[2] = quantize_one(v.z, inv); q[3] = quantize_one(v.w, inv);
            }
            uint32_t hi = 0, lo = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sum += q[e];
                hi |= (uint32_t)e4m3_times16(q[e] >> 4) << (8 * e);
                lo |= (uint32_t)e4m3_small_int(q[e] & 15) << (8 * e);
            }
            const int wi = frag_word(4 * c);
            rec[wi] = hi;
            rec[wi + 2] = lo;
        }
    } else {   // kQuantF16Perm
        __half* out = static_cast<__half*>(J.out) + (size_t)m * K;
        for (int c = lane; c < K / 4; c += 32) {
            const float4 v = x4[c];
            const float vv[4] = {v.x, v.y, v.z, v.w};
            const int pos0 = 4 * c;
            const int group_base = pos0 & ~127;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int q = quantize_one(vv[e], inv);
                sum += q;
                out[group_base + perm_index_of((pos0 + e) & 127)] = __int2half_rn(q);
            }
        }
    }
    sum = warp_sum(sum);
    if (lane == 0) {
        J.scale[m] = scale;
        J.sum[m] = sum;
    }
}

cudaError_t launch_quant(const QuantArgs& a, cudaStream_t s) {
    const int warps = a.count * a.M;
    const int blocks = (warps + 7) / 8;
    k_quant_rows<<<blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace i2s
