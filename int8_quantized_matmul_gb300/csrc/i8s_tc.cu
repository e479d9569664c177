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
// Operands: a pre-pass (k_i8s_to_f16, i8s.cu) converts the int8 weights and
// activations to f16 rows once per call. The kernel runs on CTA pairs (clusters
// of two CTAs on two SMs) driving cta_group::2 MMAs: a tile is 256 output
// features (the A operand; 128 rows in each CTA's shared memory and TMEM) x 160
// activation rows (the B operand; 80 rows in each CTA's shared memory). Each
// CTA streams its halves through TMA into its own 4-stage ring, every load
// counted on the leader's (rank 0) barrier. One stage covers 128 K positions:
// two swizzle atoms of A and of B, eight 256 x 160 x 16 MMAs issued by the
// leader. Splitting B halves each CTA's shared-memory stage (52 KB instead of
// 72 KB for a 128 x 160 tile), so one more stage is in flight, and one MMA
// instruction does the work of two SMs.
//
// Work: units are (tile, K chunk) pairs, tile-major. Each CTA pair takes a
// contiguous range of units; each CTA owns its 128 rows of every tile. A tile whose chunks are split between
// CTAs is completed exactly: every segment but the last stores its int32 sums
// in a slot of its own and marks it in the tile's mask; the CTA that brings
// the tile's ticket to the chunk count adds the marked slots to its sums and
// applies the epilogue (plain stores instead of contended atomics).
//
// MMA issue: one thread needs well over 100 SM cycles to issue a tcgen05.mma,
// more than the tensor time of a 128 x 160 x 16 MMA per SM, so four warps of
// the leader issue, taking the stages of the stream in turn (each always the
// same ring slot), all into the same accumulator.
// Every MMA accumulates (the drain zeroes the accumulator after reading it);
// the partial sums are exact integers, so the order in which the four
// streams land does not matter.
//
// Roles (416 threads per CTA): warps 0-7 drain and epilogue (warp w: TMEM
// lanes 32(w%4)..+31 of the CTA's own TMEM, accumulator columns 80(w/4)..+79),
// warp 8 TMA producer, warps 9-12 MMA issue (the leader's; warp 9 of each CTA
// also allocates TMEM, collectively for the pair). Every wait is bounded (~1 s) and records a timeout in the status word.
//
// Barriers: full[s] (leader) counts the leader's expect_tx and both CTAs'
// bytes of stage s; empty[s] (both CTAs) and tmem_full[b] (both) get the
// leader's multicast commits; tmem_empty[b] (leader) counts both CTAs' 256
// epilogue threads, the peer's by remote arrive.

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace i2s {

namespace {

constexpr int kThreads8 = 416;
constexpr int kEpiWarps8 = 8;                // two per TMEM lane quarter, one per half of the columns
constexpr int kTmaWarp8 = 8;
constexpr int kMmaWarp8 = 9;                // warps 9-12
constexpr int kIssuers8 = 4;
constexpr int kKB8 = 128;                    // K positions per stage (two 64-position swizzle atoms)
constexpr int kStagesPerChunk = kI8sChunkK / kKB8;
constexpr int kStages8 = 4;
constexpr int kAAtomBytes = kI8sTileN * 128;          // 128 rows x 64 f16
constexpr int kAStage8 = 2 * kAAtomBytes;
constexpr uint32_t kTmemCols8 = 512;
constexpr long long kWaitLimit8 = 2000000000LL;

// What depends on BM, the activation rows of a tile (the MMA N): kI8sTileM
// (160) or kI8sTileMSmall (128).
template <int BM>
struct Tile8 {
    static constexpr int kBRows = BM / 2;                  // activation rows of a tile in each CTA
    static constexpr int kBAtomBytes = kBRows * 128;       // BM/2 rows x 64 f16 (a multiple of 1024)
    static constexpr int kBStage = 2 * kBAtomBytes;
    static constexpr uint32_t kDColA = 0, kDColB = BM;     // the two f32 accumulators
    static constexpr uint32_t kSCol = 2 * BM;              // int32 running sums
    static constexpr int kEpiCols = BM / 2;                // accumulator columns each epilogue warp owns
    static constexpr int kESlices = kEpiCols / 16;         // 16-column TMEM slices of them
    static_assert(kEpiCols % 16 == 0, "epilogue slices");
    static_assert(kSCol + BM <= kTmemCols8, "TMEM budget");
    static_assert(kBAtomBytes % 1024 == 0 && BM % 32 == 0, "swizzle atoms of the B half");
    static_assert(BM % 16 == 0 && BM <= 256, "MMA N");
};
// Issuer i takes the stages s with s % kIssuers8 == i. Each ring slot must
// always be served by the same issuer: a parity wait cannot tell the phase it
// wants from the one two phases later, so an issuer must never wait on a slot
// whose previous phase another issuer has not consumed yet.
static_assert(kStages8 % kIssuers8 == 0, "ring slots per issuer");

struct Smem8 {
    uint64_t full[kStages8];
    uint64_t empty[kStages8];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done[kIssuers8];
    uint64_t epi_sync;
    uint64_t epi_bcast;
    unsigned long long final_mask;
    uint32_t tmem_base;
    int abort;
    int final_flag;
};

template <int BM>
constexpr size_t smem8_bytes() {
    return 1024 + (size_t)kStages8 * (kAStage8 + Tile8<BM>::kBStage) + sizeof(Smem8);
}

// The part of the unit range [u, u_hi) that lies in one tile of matmul p.
// Units are numbered matmul by matmul, tile-major within each.
struct Seg8 {
    int p, tile, wt, at, c_lo, c_hi, units;
    bool live;
};

__device__ __forceinline__ Seg8 seg8_at(const I8sTcArgs& a, int u, int u_hi) {
    Seg8 g;
    g.live = u < u_hi;
    if (!g.live) return g;
    g.p = 0;
    while (g.p + 1 < a.count && a.p[g.p + 1].unit0 <= u) ++g.p;
    const int chunks = a.p[g.p].chunks;
    const int local = u - a.p[g.p].unit0;
    g.tile = local / chunks;
    g.c_lo = local - g.tile * chunks;
    g.c_hi = min(chunks, g.c_lo + (u_hi - u));
    g.units = g.c_hi - g.c_lo;
    g.wt = g.tile / a.n_at;
    g.at = g.tile - g.wt * a.n_at;
    return g;
}

// Arrive on a barrier of the cluster without release semantics. The drain
// releases an accumulator with it: what the MMAs must not overtake are its
// TMEM loads and stores, complete at tcgen05.wait::ld / ::st before it, not
// the global stores of an earlier tile's epilogue, which a release arrive
// would wait for.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

template <int BM>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads8, 1) k_i8s_gemm_tc(const __grid_constant__ I8sTcArgs a) {
    using T = Tile8<BM>;
    constexpr int kBRows8 = T::kBRows;
    constexpr int kBAtomBytes = T::kBAtomBytes;
    constexpr int kBStage8 = T::kBStage;
    constexpr uint32_t kDCol8a = T::kDColA, kDCol8b = T::kDColB;
    constexpr uint32_t kSCol8 = T::kSCol;
    constexpr int kEpiCols8 = T::kEpiCols;
    constexpr int kESlices8 = T::kESlices;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = sA + (size_t)kStages8 * kAStage8;
    Smem8& S = *reinterpret_cast<Smem8*>(sB + (size_t)kStages8 * kBStage8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = tc::cluster_rank();   // 0: the leader, which issues the MMAs
    const int pair = blockIdx.x >> 1;
    const int u_begin = a.bounds[pair];   // this pair's units, planned on the host
    const int u_end = a.bounds[pair + 1];
    // stages of 128 positions; with K % 128 == 64 the last stage's second atom
    // lies past K, where the TMA box is zero-filled, which adds nothing to the
    // dot products
    auto stages_of = [&](int p) { return (a.p[p].K + kKB8 - 1) / kKB8; };

    if (tid == 0) {
        for (int s = 0; s < kStages8; ++s) {
            tc::mbar_init(&S.full[s], 1);
            tc::mbar_init(&S.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&S.tmem_full[b], kIssuers8);
            tc::mbar_init(&S.tmem_empty[b], 2 * kEpiWarps8 * 32);   // both CTAs' epilogue threads
        }
        for (int i = 0; i < kIssuers8; ++i) tc::mbar_init(&S.mma_done[i], 1);
        tc::mbar_init(&S.epi_sync, kEpiWarps8 * 32);
        tc::mbar_init(&S.epi_bcast, 1);
        S.abort = 0;
        S.final_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kMmaWarp8) {   // one warp of each CTA, collectively for the pair
        tc::pair_tmem_alloc(&S.tmem_base, kTmemCols8);
        tc::pair_tmem_relinquish();
    }
    if (warp == kTmaWarp8 && lane == 0) {
        for (int i = 0; i < a.count; ++i) {
            tc::tma_prefetch_desc(&a.p[i].xmap);
            tc::tma_prefetch_desc(&a.p[i].wmap);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = S.tmem_base;
    if (warp < kEpiWarps8) {
        // both accumulators start at zero (every MMA accumulates): each warp
        // its lane quarter and its half of the columns
        const uint32_t base = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)((warp >> 2) * kEpiCols8);
#pragma unroll
        for (int h = 0; h < kESlices8; ++h) {
            tc::tmem_st_zero_32x32b_x16(base + kDCol8a + 16u * h);
            tc::tmem_st_zero_32x32b_x16(base + kDCol8b + 16u * h);
        }
        tc::tmem_st_wait();
    }
    // both CTAs' barriers initialised and accumulators zeroed before any
    // remote arrive, multicast commit or MMA
    tc::tc_fence_before();
    tc::cluster_sync();
    tc::tc_fence_after();
    // everything above touched only parameters, shared memory and TMEM; the
    // operands, counters and outputs are used from here on, after the launch
    // before this one (the pre-pass or the row quantizer) has completed
    pdl_wait();
    volatile int* abort_flag = &S.abort;
    auto fail = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(a.status, code);
    };

    int ucur = u_begin;
    auto next_seg = [&](const Seg8& g) { ucur += g.units; return seg8_at(a, ucur, u_end); };

    if (warp == kTmaWarp8) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool pending[kStages8] = {};
            uint32_t pending_phase[kStages8] = {};
            bool ok = true;
            for (Seg8 g = seg8_at(a, ucur, u_end); ok && g.live; g = next_seg(g)) {
                const CUtensorMap* wmap = &a.p[g.p].wmap;
                const CUtensorMap* xmap = &a.p[g.p].xmap;
                const int kb_hi = min(stages_of(g.p), g.c_hi * kStagesPerChunk);
                const int wrow = g.wt * (2 * kI8sTileN) + (int)rank * kI8sTileN;   // this CTA's weight rows
                const int xrow = g.at * BM + (int)rank * kBRows8;           // this CTA's activation rows
                for (int kb = g.c_lo * kStagesPerChunk; kb < kb_hi; ++kb) {
                    if (!tc::mbar_wait_idle(&S.empty[stage], phase ^ 1, abort_flag, kWaitLimit8)) { fail(1); ok = false; break; }
                    // the leader expects both CTAs' bytes; a peer's bytes may land first
                    if (rank == 0) tc::mbar_arrive_expect_tx(&S.full[stage], 2 * (kAStage8 + kBStage8));
                    const uint32_t full_bar = tc::smem_in_rank(&S.full[stage], 0);
                    uint8_t* da = sA + (size_t)stage * kAStage8;
                    uint8_t* db = sB + (size_t)stage * kBStage8;
                    const int x0 = kb * kKB8;
                    tc::pair_tma_load_2d(da, wmap, x0, wrow, full_bar);
                    tc::pair_tma_load_2d(da + kAAtomBytes, wmap, x0 + 64, wrow, full_bar);
                    tc::pair_tma_load_2d(db, xmap, x0, xrow, full_bar);
                    tc::pair_tma_load_2d(db + kBAtomBytes, xmap, x0 + 64, xrow, full_bar);
                    pending[stage] = true;
                    pending_phase[stage] = phase;
                    if (++stage == kStages8) { stage = 0; phase ^= 1; }
                }
            }
            // on a failure, let this CTA's copies in flight land before it exits
            // (the leader's own full barriers count them; the peer's copies land
            // within the bounded waits of the final cluster barrier's wait)
            if (!ok && rank == 0)
                for (int s = 0; s < kStages8; ++s)
                    if (pending[s]) tc::mbar_wait_drain(&S.full[s], pending_phase[s], kWaitLimit8 / 8);
        }
    } else if (warp >= kMmaWarp8 && warp < kMmaWarp8 + kIssuers8 && rank == 0) {
        // ---------------------------------------------------------- MMA issue
        // issuer `me` takes the stages whose position in this CTA's stage
        // stream is me modulo kIssuers8; the ring index advances over all
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(2 * kI8sTileN, BM);   // 256 x 160 over the pair
            const int me = warp - kMmaWarp8;
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            int seq = 0;
            bool ok = true;
            for (Seg8 g = seg8_at(a, ucur, u_end); ok && g.live; g = next_seg(g)) {
                const int KB = stages_of(g.p);
                for (int c = g.c_lo; ok && c < g.c_hi; ++c) {
                    if (!tc::mbar_wait_spin(&S.tmem_empty[buf], buf_phase ^ 1, abort_flag, kWaitLimit8)) { fail(4); ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (buf ? kDCol8b : kDCol8a);
                    const int kb_lo = c * kStagesPerChunk, kb_hi = min(KB, (c + 1) * kStagesPerChunk);
                    for (int kb = kb_lo; kb < kb_hi; ++kb, ++seq) {
                        if (seq % kIssuers8 == me) {
                            if (!tc::mbar_wait_spin(&S.full[stage], phase, abort_flag, kWaitLimit8)) { fail(8); ok = false; break; }
                            tc::tc_fence_after();
                            const uint64_t ad = tc::sdesc_sw128_kmajor(tc::smem_u32(sA + (size_t)stage * kAStage8));
                            const uint64_t bd = tc::sdesc_sw128_kmajor(tc::smem_u32(sB + (size_t)stage * kBStage8));
#pragma unroll
                            for (int k = 0; k < kKB8 / 16; ++k) {   // atom k/4, +32 bytes per 16 positions
                                const uint64_t ak = ad + (uint64_t)((k >> 2) * (kAAtomBytes >> 4)) + 2 * (k & 3);
                                const uint64_t bk = bd + (uint64_t)((k >> 2) * (kBAtomBytes >> 4)) + 2 * (k & 3);
                                tc::pair_umma_f16(d_tmem, ak, bk, idesc, 1u);
                            }
                            tc::pair_commit(&S.empty[stage], 0x3);   // both CTAs' stage slots are free
                        }
                        if (++stage == kStages8) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    // the chunk is complete (in both CTAs' TMEM) once every issuer's MMAs are
                    tc::pair_commit(&S.tmem_full[buf], 0x3);
                    if (++buf == 2) { buf = 0; buf_phase ^= 1; }
                }
            }
            tc::pair_commit(&S.mma_done[me], 0x1);
            tc::mbar_wait_drain(&S.mma_done[me], 0, kWaitLimit8 / 8);
        }
    } else if (warp < kEpiWarps8) {
        // ------------------------------------------------- drain and epilogue
        const int q = warp & 3;                        // TMEM lane quarter
        const int c0 = (warp >> 2) * kEpiCols8;        // first accumulator column (activation row) of this warp
        const int r = q * 32 + lane;                   // TMEM lane = weight row of this CTA's half
        const uint32_t lane_off = ((uint32_t)(q * 32) << 16) + (uint32_t)c0;
        int buf = 0;
        uint32_t buf_phase = 0, sync_phase = 0;
        const int M = a.M;
        const bool relu = a.relu != 0;
        float local_max = 0.0f;
        bool ok = true;
        for (Seg8 g = seg8_at(a, ucur, u_end); ok && g.live; g = next_seg(g)) {
            const I8sProb& P = a.p[g.p];
            const float sc = __fmul_rn(*P.w_scale_ptr, *P.x_scale_ptr);
            float* const yb = P.y;
            const int N = P.N, chunks = P.chunks;
            const bool has_bias = P.bias != nullptr;
            const bool w8a8 = P.col_scale != nullptr;   // per-row / per-channel scales, no bias or ReLU
            // drain each chunk's f32 accumulator (exact integers) into the int32 sums
            for (int c = g.c_lo; c < g.c_hi; ++c) {
                if (!tc::mbar_wait_idle(&S.tmem_full[buf], buf_phase, abort_flag, kWaitLimit8)) { fail(16); ok = false; break; }
                tc::tc_fence_after();
                const uint32_t dcol = tmem_base + lane_off + (buf ? kDCol8b : kDCol8a);
                const uint32_t scol = tmem_base + lane_off + kSCol8;
#pragma unroll 1
                for (int h = 0; h < kESlices8; ++h) {
                    uint32_t d[16], s[16];
                    tc::tmem_ld_32x32b_x16(dcol + 16u * h, d);
                    if (c != g.c_lo) tc::tmem_ld_32x32b_x16(scol + 16u * h, s);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int x = __float2int_rn(__uint_as_float(d[j]));
                        s[j] = (uint32_t)((c != g.c_lo ? (int)s[j] : 0) + x);
                    }
                    tc::tmem_st_32x32b_x16(scol + 16u * h, s);
                    tc::tmem_st_zero_32x32b_x16(dcol + 16u * h);   // the next chunk accumulates from zero
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                mbar_arrive_cluster_relaxed(tc::smem_in_rank(&S.tmem_empty[buf], 0));   // the leader's barrier
                if (++buf == 2) { buf = 0; buf_phase ^= 1; }
            }
            if (!ok) break;
            const int n = g.wt * (2 * kI8sTileN) + (int)rank * kI8sTileN + r;
            const int ht = P.ht0 + 2 * g.tile + (int)rank;   // this CTA's half of the tile: its ticket and mask
            const int m0 = g.at * BM + c0;     // first activation row of this warp's columns
            const uint32_t scol = tmem_base + lane_off + kSCol8;
            constexpr size_t kSlot = (size_t)BM * kI8sTileN;   // one segment's int32 sums
            int32_t* slots = a.part + ((size_t)P.slot0 + (size_t)(2 * g.tile + (int)rank) * chunks) * kSlot +
                             (size_t)c0 * kI8sTileN;
            bool write = g.c_lo == 0 && g.c_hi == chunks;
            unsigned long long others = 0;   // slots of the tile's other segments (final CTA)
            if (!write) {
                // this CTA holds only some chunks of the tile: store its exact
                // int32 sums in the slot of its first chunk (plain coalesced
                // stores), mark the slot, then count its chunks; the CTA that
                // completes the count adds the marked slots to its own sums
                int32_t* mine = slots + (size_t)g.c_lo * kSlot;
#pragma unroll 1
                for (int h = 0; h < kESlices8; ++h) {
                    uint32_t s[16];
                    tc::tmem_ld_32x32b_x16(scol + 16u * h, s);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) __stcg(&mine[(size_t)(16 * h + j) * kI8sTileN + r], (int)s[j]);
                }
                __threadfence();
                tc::mbar_arrive(&S.epi_sync);
                if (!tc::mbar_wait_idle(&S.epi_sync, sync_phase, abort_flag, kWaitLimit8)) { fail(32); break; }
                if (warp == 0 && lane == 0) {
                    const unsigned long long bit = 1ull << g.c_lo;
                    const unsigned long long seen = atomicOr(&a.slot_masks[ht], bit) | bit;
                    __threadfence();
                    const unsigned prev = atomicAdd(&a.tickets[ht], (unsigned)g.units);
                    const bool last = prev + (unsigned)g.units == (unsigned)chunks;
                    // every other segment set its bit before adding to the ticket
                    S.final_mask = last ? (atomicOr(&a.slot_masks[ht], 0ull) | seen) & ~bit : 0ull;
                    S.final_flag = last;
                    tc::mbar_arrive(&S.epi_bcast);
                }
                if (!tc::mbar_wait_idle(&S.epi_bcast, sync_phase, abort_flag, kWaitLimit8)) { fail(32); break; }
                sync_phase ^= 1;
                write = S.final_flag != 0;
                others = S.final_mask;
                if (write) __threadfence();
            }
            if (write) {
                const float bn = (has_bias && n < N) ? P.bias[n] : 0.0f;
                const float bs_n = (w8a8 && n < N) ? P.col_scale[n] : 0.0f;
#pragma unroll 1
                for (int h = 0; h < kESlices8; ++h) {
                    uint32_t s[16];
                    tc::tmem_ld_32x32b_x16(scol + 16u * h, s);
                    tc::tmem_ld_wait();
                    for (unsigned long long mk = others; mk; mk &= mk - 1) {
                        const int32_t* src = slots + (size_t)__ffsll((long long)mk) * kSlot - kSlot;
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            s[j] = (uint32_t)((int)s[j] + __ldcg(&src[(size_t)(16 * h + j) * kI8sTileN + r]));
                    }
                    // all 16 values first (no per-element branch, so the
                    // conversions and products overlap), then the stores
                    float v[16];
                    if (w8a8) {
                        // per-row activation and per-channel weight scales:
                        // d = (as[m] * bs[n]) * (float)acc
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float as = P.row_scale[min(m0 + 16 * h + j, M - 1)];
                            v[j] = __fmul_rn(__fmul_rn(as, bs_n), __int2float_rn((int)s[j]));
                        }
                    } else if (has_bias) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = __fadd_rn(__fmul_rn(__int2float_rn((int)s[j]), sc), bn);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(__int2float_rn((int)s[j]), sc);
                    }
                    if (relu) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = v[j] > 0.0f ? v[j] : 0.0f;
                    }
                    if (n < N) {
                        float* yp = yb + (size_t)(m0 + 16 * h) * N + n;
                        const int rows = M - (m0 + 16 * h);
                        if (rows >= 16) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                yp[(size_t)j * N] = v[j];
                                local_max = fmaxf(local_max, fabsf(v[j]));
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (j < rows) {
                                    yp[(size_t)j * N] = v[j];
                                    local_max = fmaxf(local_max, fabsf(v[j]));
                                }
                        }
                    }
                }
            }
        }
        local_max = warp_max(local_max);
        if (lane == 0) atomicMax(a.amax_bits, __float_as_uint(local_max));
    }

    // every MMA of the pair has completed (the epilogues waited for the last
    // tmem_full) and neither CTA's shared memory is read any more
    __syncwarp();
    tc::tc_fence_before();
    tc::cluster_sync();
    if (warp == kMmaWarp8) {
        tc::tc_fence_after();
        tc::pair_tmem_dealloc(tmem_base, kTmemCols8);
    }
}

}  // namespace

// Per device: 1 + the number of CTA pairs that can be resident at once (0:
// not yet configured). Clusters must fit inside a GPC, so on a part whose
// GPCs have odd SM counts this is below half the SM count, and a persistent
// grid of more pairs would run its surplus as a second wave.
static std::atomic<int> g_pairs[64];

static cudaError_t configure(int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    *dev_out = dev;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_pairs[dev].load() > 0) return cudaSuccess;
    e = cudaFuncSetAttribute(k_i8s_gemm_tc<kI8sTileM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem8_bytes<kI8sTileM>());
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_i8s_gemm_tc<kI8sTileMSmall>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem8_bytes<kI8sTileMSmall>());
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms & ~1), 1, 1);
    cfg.blockDim = dim3(kThreads8, 1, 1);
    cfg.dynamicSmemBytes = smem8_bytes<kI8sTileM>();   // the larger of the two: pairs that fit either
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, (void*)k_i8s_gemm_tc<kI8sTileM>, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    g_pairs[dev].store(1 + clusters);
    return cudaSuccess;
}

int i8s_gemm_tc_max_pairs() {
    int dev = 0;
    if (configure(&dev) != cudaSuccess) return 1;
    return g_pairs[dev].load() - 1;
}

cudaError_t launch_i8s_gemm_tc(const I8sTcArgs& a, int grid, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = configure(&dev);
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the launch before it
    if (a.tile_m == kI8sTileMSmall)
        return launch_pdl(k_i8s_gemm_tc<kI8sTileMSmall>, dim3(grid), dim3(kThreads8), smem8_bytes<kI8sTileMSmall>(), s, a);
    if (a.tile_m != kI8sTileM) return cudaErrorInvalidValue;
    return launch_pdl(k_i8s_gemm_tc<kI8sTileM>, dim3(grid), dim3(kThreads8), smem8_bytes<kI8sTileM>(), s, a);
}

}  // namespace i2s
