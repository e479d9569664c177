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

// Position (within its 128-group) of the e4m3 element at index e of the
// tensor-core GEMV operand: TMEM column 4w + i of a K block holds the codes of
// group bytes 4w..4w+3 at bit-pair slice i, i.e. positions 32i + 4w + 0..3.
// Returns the element index of group-relative position p (p % 4 == 0 keeps
// the four elements of a word together).
__device__ __forceinline__ int e4m3_tc_index(int p) {
    return 16 * ((p & 31) >> 2) + 4 * (p >> 5) + (p & 3);
}

// Writes the four quantized values of positions 4c..4c+3 of row m in the
// requested operand layout.
__device__ __forceinline__ void emit4(const QuantArgs& a, const QuantJob& J, int m, int c, const int (&q)[4]) {
    const int K = J.K;
    if (a.layout == kQuantI8Rows) {
        uint32_t* q4 = reinterpret_cast<uint32_t*>(static_cast<int8_t*>(J.out) + (size_t)m * K);
        q4[c] = (uint32_t)(q[0] & 0xff) | ((uint32_t)(q[1] & 0xff) << 8) | ((uint32_t)(q[2] & 0xff) << 16) |
                ((uint32_t)(q[3] & 0xff) << 24);
    } else if (a.layout == kQuantE4M3Frag) {
        uint32_t* rec = static_cast<uint32_t*>(J.out) + (size_t)m * (J.Kp / 2);
        uint32_t hi = 0, lo = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            hi |= (uint32_t)e4m3_times16(q[e] >> 4) << (8 * e);
            lo |= (uint32_t)e4m3_small_int(q[e] & 15) << (8 * e);
        }
        const int wi = frag_word(4 * c);
        rec[wi] = hi;
        rec[wi + 2] = lo;
    } else if (a.layout == kQuantE4M3Tc) {
        uint32_t* hi = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(J.out) + (size_t)m * K);
        uint32_t* lo = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(J.out) + (size_t)(a.rows + m) * K);
        uint32_t h = 0, l = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            h |= (uint32_t)e4m3_times16(q[e] >> 4) << (8 * e);
            l |= (uint32_t)e4m3_small_int(q[e] & 15) << (8 * e);
        }
        const int p = 4 * c;
        const int word = ((p & ~127) + e4m3_tc_index(p & 127)) >> 2;
        hi[word] = h;
        lo[word] = l;
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
    if (m >= a.M) {
        // padding operand rows (kQuantE4M3Tc only): zero hi and lo rows
        uint32_t* hi = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(J.out) + (size_t)m * K);
        uint32_t* lo = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(J.out) + (size_t)(a.rows + m) * K);
        for (int c = tid; c < K4; c += kQThreads) { hi[c] = 0u; lo[c] = 0u; }
        return;
    }
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
    if (a.layout == kQuantE4M3Frag) {   // zero records of the padding positions K..Kp-1
        const int zero[4] = {0, 0, 0, 0};
        for (int c = K4 + tid; c < J.Kp / 4; c += kQThreads) emit4(a, J, m, c, zero);
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
    k_quant_rows<<<a.count * a.rows, kQThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace i2s
