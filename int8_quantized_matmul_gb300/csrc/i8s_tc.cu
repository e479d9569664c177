// I8_S x I8_S fused mul_mat_add(_relu) on the 5th-generation tensor cores
// ("ggml: additive INT8/ternary types, fused CPU ops, and kernels for VibeASR
// (1/2)", sections "Two new types" and "Five fused INT8 ops").
//
// acc[m][n] = sum_k W8[n][k] * X8[m][k] exactly in int32, then
// y = (float)acc * (w_scale * x_scale) (+ bias[n]) (ReLU), written as F32 with
// max|y| folded into one word for the requantization pass (i8s.cu).
//
// Arithmetic (exact): sm_103a has no integer tcgen05 MMA, so int8 values are
// carried as f16 integers (exact) through tcgen05.mma kind::f16 with f32
// accumulation. A product is at most 127^2 = 16129, so the partial sums of one
// 1024-position K chunk stay below 1024 * 16129 < 2^24 and are exact in f32.
// Every chunk gets a fresh accumulator, which the epilogue warps drain into an
// int32 running sum kept in tensor memory.
//
// Operands: the weights are the A operand (128 output features per tile).
// Converter threads (thread = weight row = TMEM lane) load each row's int8
// bytes, turn them into f16 pairs and tcgen05.st them into a TMEM ring, where
// the MMA reads them. The activations are the B operand: a pre-pass writes
// them once as f16 rows (k_i8s_x_to_f16), and TMA streams 128-row x 64-position
// tiles into a shared-memory ring.
//
// Work: units are (tile, K chunk) pairs, tile-major. Each CTA (one per SM)
// takes a contiguous range of units. A tile whose chunks are split between
// CTAs is completed through exact int32 atomics and a per-tile ticket; the CTA
// that brings the ticket to the chunk count applies the epilogue.
//
// Roles (448 threads): warps 0-3 drain and epilogue (TMEM lanes 32w..32w+31),
// warps 4-11 converters (two per TMEM lane quarter), warp 12 TMA producer,
// warp 13 TMEM allocation and MMA issue. Every wait is bounded (~1 s) and
// records a timeout in the status word.

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace i2s {

namespace {

constexpr int kThreads8 = 448;
constexpr int kEpiWarps8 = 4;
constexpr int kCvtWarp0 = 4;                 // warps 4-11: two converter warps per TMEM lane quarter
constexpr int kCvtWarps8 = 8;
constexpr int kTmaWarp8 = 12;
constexpr int kMmaWarp8 = 13;
constexpr int kKB8 = 64;                     // K positions per stage
constexpr int kStagesPerChunk = kI8sChunkK / kKB8;
constexpr int kAStages = 4;                  // TMEM A ring (32 columns per stage)
constexpr int kBStages8 = 6;                 // shared-memory B ring
constexpr int kBStage8Bytes = kI8sTile * kKB8 * 2;   // 128 rows x 128 bytes
constexpr uint32_t kTmemCols8 = 512;
constexpr uint32_t kDCol8a = 128, kDCol8b = 256;   // the two f32 accumulators
constexpr uint32_t kSCol8 = 384;             // int32 running sums
constexpr long long kWaitLimit8 = 2000000000LL;

struct Smem8 {
    uint64_t full_a[kAStages];
    uint64_t empty_a[kAStages];
    uint64_t full_b[kBStages8];
    uint64_t empty_b[kBStages8];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint64_t epi_sync;
    uint64_t epi_bcast;
    uint32_t tmem_base;
    int abort;
    int final_flag;
};

constexpr size_t kSmem8Used = 1024 + (size_t)kBStages8 * kBStage8Bytes + sizeof(Smem8);
// At least 120 KB so that one CTA runs per SM: it holds all 512 TMEM columns.
constexpr size_t kSmem8Bytes = kSmem8Used > 120 * 1024 ? kSmem8Used : 120 * 1024;

// The part of the unit range [u, u_hi) that lies in one tile.
struct Seg8 {
    int tile, wt, at, c_lo, c_hi, units;
    bool live;
};

__device__ __forceinline__ Seg8 seg8_at(const I8sTcArgs& a, int u, int u_hi) {
    Seg8 g;
    g.live = u < u_hi;
    if (!g.live) return g;
    g.tile = u / a.chunks;
    g.c_lo = u - g.tile * a.chunks;
    g.c_hi = min(a.chunks, g.c_lo + (u_hi - u));
    g.units = g.c_hi - g.c_lo;
    g.wt = g.tile / a.n_at;
    g.at = g.tile - g.wt * a.n_at;
    return g;
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

__global__ void __launch_bounds__(kThreads8, 1) k_i8s_gemm_tc(const __grid_constant__ I8sTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sB = smem;
    Smem8& S = *reinterpret_cast<Smem8*>(sB + (size_t)kBStages8 * kBStage8Bytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int u_begin = (int)(((long long)blockIdx.x * a.total_units) / gridDim.x);
    const int u_end = (int)(((long long)(blockIdx.x + 1) * a.total_units) / gridDim.x);
    const int KB = a.K / kKB8;

    if (tid == 0) {
        for (int s = 0; s < kAStages; ++s) {
            tc::mbar_init(&S.full_a[s], kCvtWarps8 * 32);
            tc::mbar_init(&S.empty_a[s], 1);
        }
        for (int s = 0; s < kBStages8; ++s) {
            tc::mbar_init(&S.full_b[s], 1);
            tc::mbar_init(&S.empty_b[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&S.tmem_full[b], 1);
            tc::mbar_init(&S.tmem_empty[b], kEpiWarps8 * 32);
        }
        tc::mbar_init(&S.mma_done, 1);
        tc::mbar_init(&S.epi_sync, kEpiWarps8 * 32);
        tc::mbar_init(&S.epi_bcast, 1);
        S.abort = 0;
        S.final_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kMmaWarp8) {
        tc::tmem_alloc(&S.tmem_base, kTmemCols8);
        tc::tmem_relinquish();
    }
    if (warp == kTmaWarp8 && lane == 0) tc::tma_prefetch_desc(&a.xmap);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = S.tmem_base;
    volatile int* abort_flag = &S.abort;
    auto fail = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(a.status, code);
    };

    int ucur = u_begin;
    auto next_seg = [&](const Seg8& g) { ucur += g.units; return seg8_at(a, ucur, u_end); };

    if (warp == kTmaWarp8) {
        // ---------------------------------------------- activation producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool pending[kBStages8] = {};
            uint32_t pending_phase[kBStages8] = {};
            bool ok = true;
            for (Seg8 g = seg8_at(a, ucur, u_end); ok && g.live; g = next_seg(g)) {
                const int kb_hi = min(KB, g.c_hi * kStagesPerChunk);
                for (int kb = g.c_lo * kStagesPerChunk; kb < kb_hi; ++kb) {
                    if (!tc::mbar_wait_idle(&S.empty_b[stage], phase ^ 1, abort_flag, kWaitLimit8)) { fail(1); ok = false; break; }
                    tc::mbar_arrive_expect_tx(&S.full_b[stage], kBStage8Bytes);
                    tc::tma_load_2d(sB + (size_t)stage * kBStage8Bytes, &a.xmap, kb * kKB8, g.at * kI8sTile,
                                    &S.full_b[stage]);
                    pending[stage] = true;
                    pending_phase[stage] = phase;
                    if (++stage == kBStages8) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok)
                for (int s = 0; s < kBStages8; ++s)
                    if (pending[s]) tc::mbar_wait(&S.full_b[s], pending_phase[s], abort_flag, kWaitLimit8 / 8);
        }
    } else if (warp >= kCvtWarp0 && warp < kCvtWarp0 + kCvtWarps8) {
        // ---------------------------------------------------------- converters
        // thread = weight row = TMEM lane, two threads per row: half hf turns
        // the row's bytes 32hf..32hf+31 of each 64-position stage into TMEM
        // columns 16hf..16hf+15; three stages of row bytes in flight.
        const int q = (warp - kCvtWarp0) & 3;   // TMEM lane quarter (warp % 4)
        const int hf = (warp - kCvtWarp0) >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(16 * hf);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (Seg8 g = seg8_at(a, ucur, u_end); ok && g.live; g = next_seg(g)) {
            const int n = g.wt * kI8sTile + r;
            const bool valid = n < a.N;
            const int8_t* row = a.w + (size_t)(valid ? n : 0) * a.K + 32 * hf;
            const int kb_lo = g.c_lo * kStagesPerChunk;
            const int kb_hi = min(KB, g.c_hi * kStagesPerChunk);
            uint4 buf[3][2];
            auto load = [&](uint4 (&b)[2], int kb) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    b[i] = valid ? ldg_stream(row + (size_t)kb * kKB8 + 16 * i) : make_uint4(0, 0, 0, 0);
            };
#pragma unroll
            for (int j = 0; j < 3; ++j)
                if (kb_lo + j < kb_hi) load(buf[j], kb_lo + j);
            for (int kb0 = kb_lo; ok && kb0 < kb_hi; kb0 += 3) {
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const int kb = kb0 + j;
                    if (kb >= kb_hi) break;
                    uint32_t v[16];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint32_t w4[4] = {buf[j][i].x, buf[j][i].y, buf[j][i].z, buf[j][i].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) i8x4_to_f16x4(w4[e], v[8 * i + 2 * e], v[8 * i + 2 * e + 1]);
                    }
                    if (kb + 3 < kb_hi) load(buf[j], kb + 3);
                    if (!tc::mbar_wait_idle(&S.empty_a[stage], phase ^ 1, abort_flag, kWaitLimit8)) { fail(2); ok = false; break; }
                    tc::tc_fence_after();
                    tc::tmem_st_32x32b_x16(lane_base + (uint32_t)(stage * 32), v);
                    tc::tmem_st_wait();
                    tc::tc_fence_before();
                    tc::mbar_arrive(&S.full_a[stage]);
                    if (++stage == kAStages) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == kMmaWarp8) {
        // ---------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(kI8sTile, kI8sTile);
            int stage = 0, bstage = 0;
            uint32_t phase = 0, bphase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            for (Seg8 g = seg8_at(a, ucur, u_end); ok && g.live; g = next_seg(g)) {
                for (int c = g.c_lo; ok && c < g.c_hi; ++c) {
                    if (!tc::mbar_wait_spin(&S.tmem_empty[buf], buf_phase ^ 1, abort_flag, kWaitLimit8)) { fail(4); ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (buf ? kDCol8b : kDCol8a);
                    const int kb_lo = c * kStagesPerChunk, kb_hi = min(KB, (c + 1) * kStagesPerChunk);
                    for (int kb = kb_lo; kb < kb_hi; ++kb) {
                        if (!tc::mbar_wait_spin(&S.full_a[stage], phase, abort_flag, kWaitLimit8) ||
                            !tc::mbar_wait_spin(&S.full_b[bstage], bphase, abort_flag, kWaitLimit8)) { fail(8); ok = false; break; }
                        tc::tc_fence_after();
                        const uint64_t bd = tc::sdesc_sw128_kmajor(tc::smem_u32(sB + (size_t)bstage * kBStage8Bytes));
                        const uint32_t a0 = tmem_base + (uint32_t)(stage * 32);
                        const uint32_t first = kb != kb_lo;
#pragma unroll
                        for (int k = 0; k < kKB8 / 16; ++k)   // 16 positions = 8 A columns = 32 B bytes per MMA
                            tc::umma_f16_tmem_a(d_tmem, a0 + 8u * k, bd + 2 * k, idesc, k == 0 ? first : 1u);
                        tc::umma_commit(&S.empty_a[stage]);
                        tc::umma_commit(&S.empty_b[bstage]);
                        if (++stage == kAStages) { stage = 0; phase ^= 1; }
                        if (++bstage == kBStages8) { bstage = 0; bphase ^= 1; }
                    }
                    if (!ok) break;
                    tc::umma_commit(&S.tmem_full[buf]);
                    if (++buf == 2) { buf = 0; buf_phase ^= 1; }
                }
            }
            tc::umma_commit(&S.mma_done);
            tc::mbar_wait(&S.mma_done, 0, abort_flag, kWaitLimit8 / 8);
        }
    } else if (warp < kEpiWarps8) {
        // ------------------------------------------------- drain and epilogue
        const int r = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        int buf = 0;
        uint32_t buf_phase = 0, sync_phase = 0;
        const float sc = __fmul_rn(*a.w_scale_ptr, *a.x_scale_ptr);
        float local_max = 0.0f;
        bool ok = true;
        for (Seg8 g = seg8_at(a, ucur, u_end); ok && g.live; g = next_seg(g)) {
            // drain each chunk's f32 accumulator (exact integers) into the int32 sums
            for (int c = g.c_lo; c < g.c_hi; ++c) {
                if (!tc::mbar_wait_idle(&S.tmem_full[buf], buf_phase, abort_flag, kWaitLimit8)) { fail(16); ok = false; break; }
                tc::tc_fence_after();
                const uint32_t dcol = tmem_base + lane_off + (buf ? kDCol8b : kDCol8a);
                const uint32_t scol = tmem_base + lane_off + kSCol8;
#pragma unroll 1
                for (int h = 0; h < kI8sTile / 32; ++h) {
                    uint32_t d[32], s[32];
                    tc::tmem_ld_32x32b_x32(dcol + 32u * h, d);
                    if (c != g.c_lo) tc::tmem_ld_32x32b_x32(scol + 32u * h, s);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int x = __float2int_rn(__uint_as_float(d[j]));
                        s[j] = (uint32_t)((c != g.c_lo ? (int)s[j] : 0) + x);
                    }
                    tc::tmem_st_32x32b_x32(scol + 32u * h, s);
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                tc::mbar_arrive(&S.tmem_empty[buf]);
                if (++buf == 2) { buf = 0; buf_phase ^= 1; }
            }
            if (!ok) break;
            const int n = g.wt * kI8sTile + r;
            const int m0 = g.at * kI8sTile;
            const uint32_t scol = tmem_base + lane_off + kSCol8;
            int32_t* part = a.part + (size_t)g.tile * kI8sTile * kI8sTile;
            bool write = g.c_lo == 0 && g.c_hi == a.chunks;
            if (!write) {
                // this CTA holds only some chunks of the tile: add them to the
                // tile's exact int32 sums; the CTA completing the count finishes
#pragma unroll 1
                for (int h = 0; h < kI8sTile / 32; ++h) {
                    uint32_t s[32];
                    tc::tmem_ld_32x32b_x32(scol + 32u * h, s);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) atomicAdd(&part[(size_t)(32 * h + j) * kI8sTile + r], (int)s[j]);
                }
                __threadfence();
                tc::mbar_arrive(&S.epi_sync);
                if (!tc::mbar_wait_idle(&S.epi_sync, sync_phase, abort_flag, kWaitLimit8)) { fail(32); break; }
                if (r == 0) {
                    __threadfence();
                    const unsigned prev = atomicAdd(&a.tickets[g.tile], (unsigned)g.units);
                    S.final_flag = prev + (unsigned)g.units == (unsigned)a.chunks;
                    tc::mbar_arrive(&S.epi_bcast);
                }
                if (!tc::mbar_wait_idle(&S.epi_bcast, sync_phase, abort_flag, kWaitLimit8)) { fail(32); break; }
                sync_phase ^= 1;
                write = S.final_flag != 0;
                if (write) __threadfence();
            }
            if (write) {
                const bool full = g.c_lo == 0 && g.c_hi == a.chunks;
                const float bn = (a.bias && n < a.N) ? a.bias[n] : 0.0f;
#pragma unroll 1
                for (int h = 0; h < kI8sTile / 32; ++h) {
                    uint32_t s[32];
                    if (full) {
                        tc::tmem_ld_32x32b_x32(scol + 32u * h, s);
                        tc::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) s[j] = (uint32_t)__ldcg(&part[(size_t)(32 * h + j) * kI8sTile + r]);
                    }
                    if (n < a.N) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int m = m0 + 32 * h + j;
                            if (m < a.M) {
                                float v = __fmul_rn(__int2float_rn((int)s[j]), sc);
                                if (a.bias) v = __fadd_rn(v, bn);
                                if (a.relu) v = v > 0.0f ? v : 0.0f;
                                a.y[(size_t)m * a.N + n] = v;
                                local_max = fmaxf(local_max, fabsf(v));
                            }
                        }
                    }
                }
            }
        }
        local_max = warp_max(local_max);
        if (lane == 0) atomicMax(a.amax_bits, __float_as_uint(local_max));
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp8) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, kTmemCols8);
    }
}

// int8 activations -> f16 rows (zero rows up to rows_pad); also clears the
// status and amax words and the split-tile sums and tickets.
__global__ void __launch_bounds__(256) k_i8s_x_to_f16(const int8_t* __restrict__ x, int M, int K, int rows_pad,
                                                      __half* __restrict__ xf, uint4* zero, unsigned long long zero_16,
                                                      uint32_t* status, unsigned int* amax_bits) {
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    const unsigned long long t0 = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
    if (t0 == 0) {
        *status = 0u;
        *amax_bits = 0u;
    }
    for (unsigned long long i = t0; i < zero_16; i += stride) zero[i] = make_uint4(0u, 0u, 0u, 0u);
    const unsigned long long n16 = (unsigned long long)rows_pad * K / 16;   // 16 values per step
    const unsigned long long valid16 = (unsigned long long)M * K / 16;
    for (unsigned long long i = t0; i < n16; i += stride) {
        uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
        if (i < valid16) {
            const uint4 v = reinterpret_cast<const uint4*>(x)[i];
            i8x4_to_f16x4(v.x, o0.x, o0.y);
            i8x4_to_f16x4(v.y, o0.z, o0.w);
            i8x4_to_f16x4(v.z, o1.x, o1.y);
            i8x4_to_f16x4(v.w, o1.z, o1.w);
        }
        reinterpret_cast<uint4*>(xf)[2 * i] = o0;
        reinterpret_cast<uint4*>(xf)[2 * i + 1] = o1;
    }
}

}  // namespace

cudaError_t launch_i8s_x_to_f16(const int8_t* x, int M, int K, int rows_pad, __half* xf, void* zero, size_t zero_bytes,
                                uint32_t* status, unsigned int* amax_bits, cudaStream_t s) {
    const unsigned long long n = (unsigned long long)rows_pad * K / 16;
    const unsigned long long want = (n + 255) / 256;
    const int cap = device_sm_count() * 8;
    const int grid = (int)(want < (unsigned long long)cap ? (want < 1 ? 1 : want) : cap);
    k_i8s_x_to_f16<<<grid, 256, 0, s>>>(x, M, K, rows_pad, xf, static_cast<uint4*>(zero), zero_bytes / 16, status,
                                        amax_bits);
    return cudaGetLastError();
}

cudaError_t launch_i8s_gemm_tc(const I8sTcArgs& a, int grid, cudaStream_t s) {
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(k_i8s_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem8Bytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    k_i8s_gemm_tc<<<grid, kThreads8, kSmem8Bytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace i2s
