// Decode GEMV for the I2_S ternary x INT8 matmul, M <= 16 activation rows
// ("ggml-cpu: ternary I2_S matmul kernel", sections Arithmetic and Kernels;
// "ggml: additive INT8/ternary types ...", section "Arithmetic is exact where
// it can be").
//
// The op is bound by weight bandwidth: every weight row is streamed from HBM
// once and reused for all M activation rows, as the pages' CPU kernel does.
//
// Arithmetic. The dot product sum_k code*q is formed on the legacy warp-level
// e4m3 tensor-core MMA (m16n8k32, fp32 accumulate), exactly:
//   * a code c in {0,1,2} read as an e4m3 bit pattern is the subnormal c*2^-9,
//     so the 2-bit fields need only a shift and a mask to become operands;
//   * q in [-127,127] is split as q = 16*(q>>4) + (q&15); both parts are exact
//     e4m3 values and feed two MMAs into the same accumulator;
//   * every product and partial sum is an integer multiple of 2^-9 below
//     2^24 * 2^-9 in magnitude (|dot| <= 254*K < 2^24 for K <= 66052), so
//     fp32 accumulation is exact and dot = acc * 2^9 exactly.
// The epilogue is the pages' y = (float)(dot - row_sum) * (w_scale*act_scale)
// with IEEE round-to-nearest multiplies.
//
// Fragment mapping. A lane (g = lane/4, t = lane%4) of a warp takes 16 bytes of
// codes for weight rows g and g+8 of a 16-row block, at byte 16t of each row's
// 64-byte K block (256 positions = groups 2kb and 2kb+1). Its four 32-bit
// words w_i (group bytes gp0+4i .. +3, gp0 = 16*(t%2)) yield, per bit-pair
// slice, four e4m3 codes for four consecutive positions. MMA (i, h) takes the
// slices (6,4) for h = 0 or (2,0) for h = 1 as its two k-halves. An MMA sums
// over its k index, so any bijection between k and K positions works as long
// as A and B use the same one; here the position of every A byte depends only
// on t, and the quantizer writes each activation byte at the B fragment slot
// of the same position (quant.cu, frag_word).
//
// Work split. A CTA of 8 warps owns 512 weight rows (64 per warp: four 16-row
// MMA blocks, four independent accumulator chains) and walks the K blocks of
// its share; all warps are on the same K block at a time, so the activation
// records of that block are staged once per CTA. Copies use cp.async into a
// three-stage ring: each thread copies (and alone reads) its own 128 weight
// bytes per K block; the 4 KB (8 KB for M > 8) of activation records are copied
// cooperatively, XOR-swizzled so the fragment reads are free of bank
// conflicts, and published with one block barrier per K block.

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace i2s {

namespace {

constexpr int kThreads = kGemvWarps * 32;
constexpr int kRB = kGemvRowsPerWarp / 16;   // 16-row MMA blocks per warp
constexpr int kWChunks = kRB * 2;            // 16-byte weight chunks per thread per K block
constexpr int kStages = 3;                   // cp.async ring depth (K blocks)

// Expands the codes of two weight words (rows g and g+8) for bit-pair slices
// S0 (first k-half) and S1 (second k-half) into e4m3 operands and issues the
// two MMAs of one (hi, lo) activation pair.
template <int S0, int S1>
__device__ __forceinline__ void mma_codes_pair(float (&c)[4], uint32_t wa, uint32_t wb, uint4 bw) {
    asm volatile(
        "{\n"
        ".reg .b32 a0, a1, a2, a3;\n"
        "shr.b32 a0, %4, %10;\n"
        "shr.b32 a2, %4, %11;\n"
        "shr.b32 a1, %5, %10;\n"
        "shr.b32 a3, %5, %11;\n"
        "and.b32 a0, a0, 0x03030303;\n"
        "and.b32 a1, a1, 0x03030303;\n"
        "and.b32 a2, a2, 0x03030303;\n"
        "and.b32 a3, a3, 0x03030303;\n"
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3}, {%6,%7}, {%0,%1,%2,%3};\n"
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3}, {%8,%9}, {%0,%1,%2,%3};\n"
        "}\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(wa), "r"(wb), "r"(bw.x), "r"(bw.y), "r"(bw.z), "r"(bw.w), "n"(S0), "n"(S1));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    const int n = valid ? 16 : 0;   // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Shared memory per stage: weight chunks [kWChunks][kThreads] then activation
// records [NB*32 records][8 chunks], each uint4.
template <int NB>
struct Layout {
    static constexpr int kW = kWChunks * kThreads;
    static constexpr int kB = NB * 32 * 8;
    static constexpr int kStage = kW + kB;
    static constexpr size_t kBytes = (size_t)kStages * kStage * sizeof(uint4);
};

template <int NB>
__global__ void __launch_bounds__(kThreads, NB == 1 ? 2 : 1) k_i2s_gemv(const __grid_constant__ GemvArgs a) {
    extern __shared__ uint4 smem[];
    using L = Layout<NB>;

    // Locate the problem owning this CTA (tile0 is increasing).
    const int bid = blockIdx.x;
    int lo = 0, hi = a.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.p[mid].tile0 <= bid) lo = mid; else hi = mid - 1;
    }
    const GemvProb& P = a.p[lo];
    const int S = a.split_k;
    const int local = bid - P.tile0;
    const int split = local % S;
    const int tile = local / S;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int N = P.N, K = P.K, M = a.M;
    const int row_bytes = K >> 2;
    const int KB = (K + 255) >> 8;
    const int kb_per = (KB + S - 1) / S;
    const int kb_lo = split * kb_per;
    const int kb_hi = min(KB, kb_lo + kb_per);
    const int row_base = tile * kGemvTileRows + warp * kGemvRowsPerWarp;
    const size_t rec_words_per_row = (size_t)KB * 128;   // 2*Kp bytes

    auto issue = [&](int kb, int stage) {
        uint4* sp = smem + stage * L::kStage;
        const int byte_in_row = kb * 64 + 16 * t;
        const bool col_ok = byte_in_row < row_bytes;
#pragma unroll
        for (int j = 0; j < kWChunks; ++j) {
            const int row = row_base + (j >> 1) * 16 + g + 8 * (j & 1);
            const bool ok = col_ok && row < N;
            cp_async16(sp + j * kThreads + tid, ok ? P.w + (size_t)row * row_bytes + byte_in_row : P.w, ok);
        }
#pragma unroll
        for (int e = 0; e < NB; ++e) {
            const int rec = e * 32 + (tid >> 3);   // record of activation row rec/4, lane quad rec%4
            const int u = tid & 7;
            const int col = rec >> 2, tt = rec & 3;
            const bool ok = col < M;
            const uint32_t* src = P.act + (size_t)col * rec_words_per_row + (size_t)(kb * 4 + tt) * 32 + u * 4;
            cp_async16(sp + L::kW + rec * 8 + (u ^ (rec & 7)), ok ? (const void*)src : (const void*)P.act, ok);
        }
    };

    float acc[NB][kRB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int rb = 0; rb < kRB; ++rb)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[nb][rb][c] = 0.0f;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (kb_lo + s < kb_hi) issue(kb_lo + s, s);
        cp_async_commit();
    }
    int st = 0;
#pragma unroll 1
    for (int kb = kb_lo; kb < kb_hi; ++kb) {
        cp_async_wait<kStages - 2>();   // this thread's copies of block kb have landed
        __syncthreads();                // everyone's copies of kb are visible; block kb-1 is consumed
        {
            int sa = st + kStages - 1;
            if (sa >= kStages) sa -= kStages;
            if (kb + kStages - 1 < kb_hi) issue(kb + kStages - 1, sa);
            cp_async_commit();
        }
        const uint4* sw = smem + st * L::kStage;
        const uint4* sb = sw + L::kW;
        if (++st == kStages) st = 0;

        // One 32-bit word per row block and k-pair at a time (a real loop, so
        // the code expansion cannot be hoisted into a large register set).
        const uint32_t* sw32 = reinterpret_cast<const uint32_t*>(sw);
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
            uint4 b0[NB], b1[NB];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int rec = nb * 32 + lane;   // lane = g*4 + t
                b0[nb] = sb[rec * 8 + ((2 * i) ^ (rec & 7))];
                b1[nb] = sb[rec * 8 + ((2 * i + 1) ^ (rec & 7))];
            }
            uint32_t wa[kRB], wb[kRB];
#pragma unroll
            for (int rb = 0; rb < kRB; ++rb) {
                wa[rb] = sw32[((2 * rb) * kThreads + tid) * 4 + i];
                wb[rb] = sw32[((2 * rb + 1) * kThreads + tid) * 4 + i];
            }
#pragma unroll
            for (int rb = 0; rb < kRB; ++rb)
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) mma_codes_pair<6, 4>(acc[nb][rb], wa[rb], wb[rb], b0[nb]);
#pragma unroll
            for (int rb = 0; rb < kRB; ++rb)
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) mma_codes_pair<2, 0>(acc[nb][rb], wa[rb], wb[rb], b1[nb]);
        }
    }

    // Epilogue. acc element c of block (nb, rb) is the dot of weight row
    // row_base + rb*16 + g + 8*(c>>1) with activation row nb*8 + 2t + (c&1).
    const float w_scale = *reinterpret_cast<const float*>(P.w + (size_t)N * row_bytes);
    if (S == 1) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int rb = 0; rb < kRB; ++rb)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int n = row_base + rb * 16 + g + 8 * (c >> 1);
                    const int m = nb * 8 + 2 * t + (c & 1);
                    if (n < N && m < M) {
                        const int dot = __float2int_rn(__fmul_rn(acc[nb][rb][c], 512.0f));
                        const float sc = __fmul_rn(w_scale, P.act_scale[m]);
                        P.y[(size_t)m * N + n] = __fmul_rn(__int2float_rn(dot - P.row_sum[m]), sc);
                    }
                }
        return;
    }

    // Split-K: exact integer partials, then the last CTA of the tile applies
    // the epilogue (integer addition is order-independent, so the result does
    // not depend on the split or on the arrival order).
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int rb = 0; rb < kRB; ++rb)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int n = row_base + rb * 16 + g + 8 * (c >> 1);
                const int m = nb * 8 + 2 * t + (c & 1);
                if (n < N && m < M)
                    atomicAdd(&P.dot_acc[(size_t)m * N + n], __float2int_rn(__fmul_rn(acc[nb][rb][c], 512.0f)));
            }
    __threadfence();
    __syncthreads();
    __shared__ unsigned int s_ticket;
    if (tid == 0) s_ticket = atomicAdd(&P.tickets[tile], 1u);
    __syncthreads();
    if (s_ticket != (unsigned)(S - 1)) return;
    __threadfence();
    const int n0 = tile * kGemvTileRows;
    for (int e = tid; e < kGemvTileRows * M; e += kThreads) {
        const int n = n0 + e % kGemvTileRows;
        const int m = e / kGemvTileRows;
        if (n < N) {
            const int dot = __ldcg(&P.dot_acc[(size_t)m * N + n]);
            const float sc = __fmul_rn(w_scale, P.act_scale[m]);
            P.y[(size_t)m * N + n] = __fmul_rn(__int2float_rn(dot - P.row_sum[m]), sc);
        }
    }
}

}  // namespace

int gemv_ctas_for(int N, int split_k) { return ((N + kGemvTileRows - 1) / kGemvTileRows) * split_k; }

cudaError_t launch_gemv(const GemvArgs& a, int total_ctas, cudaStream_t s) {
    // The shared-memory opt-in is a per-device function attribute.
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(k_i2s_gemv<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<1>::kBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_i2s_gemv<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<2>::kBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    if (a.M <= 8)
        k_i2s_gemv<1><<<total_ctas, kThreads, Layout<1>::kBytes, s>>>(a);
    else
        k_i2s_gemv<2><<<total_ctas, kThreads, Layout<2>::kBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace i2s
