// Decode GEMV for the I2_S ternary x INT8 matmul (M <= 16 activation rows) on
// the 5th-generation tensor cores ("ggml-cpu: ternary I2_S matmul kernel",
// sections Arithmetic and Kernels; "ggml: additive INT8/ternary types ...",
// "Arithmetic is exact where it can be").
//
// The op is bound by weight bandwidth: each 2-bit weight is read from HBM
// once and used for all M activation rows. What limits a tensor-core GEMV here
// is the expansion of the codes into MMA operands, so it is kept off shared
// memory: converter threads expand each weight row's codes in registers and
// write them straight into tensor memory (tcgen05.st), and the MMA reads its A
// operand from there.
//
// Arithmetic (exact): tcgen05.mma kind::f8f6f4 with e4m3 operands and f32
// accumulation.
//   * A: a code c in {0,1,2} read as an e4m3 bit pattern is the subnormal
//     c * 2^-9, so (packed >> s) & 0x03030303 yields four operands.
//   * B: each quantized activation q in [-127,127] is split exactly into
//     16*(q>>4) and (q&15), both exact e4m3 values, stored as two operand rows
//     ("hi" rows 0..M'-1 and "lo" rows M'..2M'-1 with M' = 8 or 16), so
//     MMA N = 2M'.
//   * D columns m and M'+m hold sum_k c*16*(q>>4) * 2^-9 and sum_k c*(q&15) *
//     2^-9: integer multiples of 2^-9 below 2^24 * 2^-9 in magnitude, held
//     exactly in f32. dot = (D_hi + D_lo) * 2^9, as two exact conversions.
// The epilogue is the pages' y = (float)(dot - row_sum) * (w_scale*act_scale).
//
// K order: a K block is one 128-position group (32 packed bytes per weight
// row). TMEM column 4w + i of the block holds the four codes of word w (group
// bytes 4w..4w+3) at shift (6, 4, 2, 0)[i], i.e. positions 32i + 4w + 0..3;
// the quantizer writes the B rows in the same order (quant.cu,
// e4m3_tc_index), and the dot product does not depend on the order.
//
// Roles (persistent CTAs, static tile schedule, 128 weight rows per tile):
//   warp 8     weight producer: per 4 K blocks, each row's contiguous 128
//              packed bytes, copied with cp.async by 8 consecutive lanes (a warp
//              instruction moves 4 whole rows) into a 4-stage shared ring (rows
//              padded to 144 bytes so the 16-byte reads are free of bank
//              conflicts), completion signalled on an mbarrier;
//   warps 0-3  converters: thread = weight row = TMEM lane reads its row's 32
//              bytes of a K block, expands them and tcgen05.st's them into a
//              4-stage TMEM ring of A operands;
//   warp 10    TMA producer of the B rows of each K block;
//   warp 9     TMEM allocation and the MMA issuer;
//   warps 4-7  epilogue (TMEM lanes 32(w-4) .. +31 = weight rows).
// Every wait is bounded (~1 s) and reports a timeout in the status word.

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace i2s {

namespace {

constexpr int kThreadsGv = 352;
constexpr int kCvtWarpsGv = 4;
constexpr int kEpiWarp0 = 4;
constexpr int kWProdWarp = 8;
constexpr int kMmaWarpGv = 9;
constexpr int kBProdWarp = 10;
constexpr int kKB = 256;               // K positions per pipeline stage (64 packed bytes per row)
constexpr int kSbK = 2;                // stages per weight super-block (128 bytes per row)
constexpr int kWStages = 3;            // weight ring depth (super-blocks)
constexpr int kWPitch = 144;           // padded bytes per row in the weight ring
constexpr int kStagesGv = 3;           // TMEM A ring depth (stages of 64 columns)
constexpr int kBRingBytes = 32 * 1024; // activation ring: 8 stages of 4 KB (M' = 8) or 4 of 8 KB (M' = 16)
constexpr int kBStagesMax = 16;
constexpr int kTileRows = 128;
constexpr int kWStageBytes = kTileRows * kWPitch;
constexpr uint32_t kTmemColsGv = 256;  // A ring 3 x 64 columns, D 2 x 32 columns
constexpr uint32_t kDCol0 = 192;
constexpr long long kWaitLimitGv = 2000000000LL;

struct SmemGv {
    uint64_t full_w[kWStages];          // a weight super-block stage is in shared memory
    uint64_t empty_w[kWStages];         // every converter is done with a stage
    uint64_t full_a[kStagesGv];
    uint64_t empty[kStagesGv];          // TMEM A stage free (MMA done)
    uint64_t full_b[kBStagesMax];
    uint64_t empty_b[kBStagesMax];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint64_t epi_sync;                  // the 4 epilogue warps finished their partial-dot atomics
    uint64_t epi_bcast;                 // the split-K finalize decision is published
    uint32_t tmem_base;
    int abort;
    int final_flag;
};

constexpr size_t kSProbBytes = 64;      // shared copy of one problem-table entry (SProb)
constexpr size_t kSmemGvUsed = 1024 + (size_t)kBRingBytes + (size_t)kWStages * kWStageBytes + sizeof(SmemGv) + 16 +
                               (size_t)kMaxGroup * kSProbBytes;
// At least 80 KB so that at most two CTAs share an SM: each holds 256 of the
// 512 TMEM columns for its whole life.
constexpr size_t kSmemGvBytes = kSmemGvUsed > 80 * 1024 ? kSmemGvUsed : 80 * 1024;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    const int n = valid ? 16 : 0;   // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrives on `bar` once every cp.async this thread issued so far has completed
// (the arrival is counted in the barrier's expected count: .noinc).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Problem table copied into shared memory at kernel start (parameter-space
// reads through a generic pointer are slow once the table misses the constant
// cache, and every role resolves a problem at each segment).
struct SProb {
    const uint8_t* w;
    const float* act_scale;
    const int32_t* row_sum;
    float* y;
    int N, K, map, unit0, chunks, dot_off, ticket_off, pad;
};

constexpr int kChunkStages = kGemvChunkPositions / kKB;   // 6 stages per work unit

// A segment: the consecutive K chunks of one row tile that fall inside this
// CTA's contiguous range of work units [u, u_hi). Every role walks the same
// segments in the same order.
struct Seg {
    const uint8_t* w;
    const float* act_scale;
    const int32_t* row_sum;
    float* y;
    int N, K, map, n0, tile, st_lo, st_hi, c_lo, c_hi, chunks, dot_off, ticket_off, units;
    bool live;
};

static_assert(sizeof(SProb) == kSProbBytes, "SProb size");

// sp holds the n_sp problem-table entries this CTA's unit range touches.
__device__ __forceinline__ Seg seg_at(const SProb* sp, int n_sp, int u, int u_hi) {
    Seg g;
    g.live = u < u_hi;
    if (!g.live) return g;
    int lo = 0, hi = n_sp - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sp[mid].unit0 <= u) lo = mid; else hi = mid - 1;
    }
    const SProb& P = sp[lo];
    const int local = u - P.unit0;
    g.w = P.w;
    g.act_scale = P.act_scale;
    g.row_sum = P.row_sum;
    g.y = P.y;
    g.N = P.N;
    g.K = P.K;
    g.map = P.map;
    g.chunks = P.chunks;
    g.dot_off = P.dot_off;
    g.ticket_off = P.ticket_off;
    g.tile = local / P.chunks;
    g.c_lo = local - g.tile * P.chunks;
    g.c_hi = min(P.chunks, g.c_lo + (u_hi - u));
    g.units = g.c_hi - g.c_lo;
    g.n0 = g.tile * kTileRows;
    const int KB = (P.K + kKB - 1) / kKB;
    g.st_lo = g.c_lo * kChunkStages;
    g.st_hi = min(KB, g.c_hi * kChunkStages);
    return g;
}

__global__ void __launch_bounds__(kThreadsGv, 2) k_i2s_gemv_tc(const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sB = smem;
    uint8_t* sW = sB + (size_t)kBRingBytes;
    SmemGv& S = *reinterpret_cast<SmemGv*>(sW + (size_t)kWStages * kWStageBytes);
    SProb* sp = reinterpret_cast<SProb*>(reinterpret_cast<uint8_t*>(&S) + ((sizeof(SmemGv) + 15) & ~(size_t)15));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Mp = a.BN;                                     // operand rows per half (8 or 16); MMA N = 2*Mp
    const uint32_t b_sub = (uint32_t)(2 * Mp) * 128u;        // one 128-position operand sub-tile (1024-aligned)
    const uint32_t b_stage_bytes = 2 * b_sub;                // a stage holds two sub-tiles
    const int b_stages = kBRingBytes / (int)b_stage_bytes;
    // this CTA's contiguous share of the work units
    const int u_begin = (int)(((long long)blockIdx.x * a.total_tiles) / gridDim.x);
    const int u_end = (int)(((long long)(blockIdx.x + 1) * a.total_tiles) / gridDim.x);

    // Copy the (few) problem-table entries this CTA's unit range touches.
    __shared__ int s_prange[2];
    if (tid == 0) {
        auto find = [&](int u) {
            int lo = 0, hi = a.count - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (a.p[mid].tile0 <= u) lo = mid; else hi = mid - 1;
            }
            return lo;
        };
        s_prange[0] = find(u_begin);
        s_prange[1] = u_end > u_begin ? find(u_end - 1) : s_prange[0];
    }
    __syncthreads();
    const int p_first = s_prange[0];
    const int n_sp = s_prange[1] - p_first + 1;
    for (int i = tid; i < n_sp; i += kThreadsGv) {
        const TcProb& P = a.p[p_first + i];
        sp[i] = SProb{P.w, P.act_scale, P.row_sum, P.y, P.N, P.K, P.map, P.tile0, P.chunks, P.dot_off, P.ticket_off, 0};
    }
    if (tid == 0) {
        for (int s = 0; s < kWStages; ++s) {
            tc::mbar_init(&S.full_w[s], 32);                  // one cp.async-completion arrival per producer lane
            tc::mbar_init(&S.empty_w[s], kCvtWarpsGv * 32);
        }
        for (int s = 0; s < kStagesGv; ++s) {
            tc::mbar_init(&S.full_a[s], kCvtWarpsGv * 32);
            tc::mbar_init(&S.empty[s], 1);
        }
        for (int s = 0; s < kBStagesMax; ++s) {
            tc::mbar_init(&S.full_b[s], 1);
            tc::mbar_init(&S.empty_b[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&S.tmem_full[b], 1);
            tc::mbar_init(&S.tmem_empty[b], 4 * 32);
        }
        tc::mbar_init(&S.mma_done, 1);
        tc::mbar_init(&S.epi_sync, 4 * 32);
        tc::mbar_init(&S.epi_bcast, 1);
        S.abort = 0;
        S.final_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kMmaWarpGv) {
        tc::tmem_alloc(&S.tmem_base, kTmemColsGv);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = S.tmem_base;
    volatile int* abort_flag = &S.abort;
    auto fail = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(a.status, code);
    };

    int ucur = u_begin;   // each role advances its own copy of the unit cursor
    auto next_seg = [&](const Seg& g) { ucur += g.units; return seg_at(sp, n_sp, ucur, u_end); };

    if (warp == kWProdWarp) {
        // --------------------------------------------------- weight producer
        // Per super-block (two stages, 512 positions), each row's contiguous
        // packed bytes (up to 128) are copied with cp.async, 8 consecutive lanes
        // per row (a warp instruction moves 4 whole rows), into a 3-stage ring;
        // completion is signalled on the stage's mbarrier by every lane.
        int ws = 0;
        uint32_t wphase = 0;
        bool ok = true;
        for (Seg g = seg_at(sp, n_sp, ucur, u_end); ok && g.live; g = next_seg(g)) {
            const int row_bytes = g.K / 4;
            const int end = min(g.st_hi * 64, row_bytes);
            for (int off = g.st_lo * 64; off < end; off += 128) {
                const int bytes = min(128, end - off);   // 32, 64, 96 or 128
                if (!tc::mbar_wait_spin(&S.empty_w[ws], wphase ^ 1, abort_flag, kWaitLimitGv)) { fail(1024); ok = false; break; }
                const uint8_t* base = g.w + (size_t)g.n0 * row_bytes + off;
                uint8_t* dst = sW + (size_t)ws * kWStageBytes;
                if (bytes == 128) {
                    const int col = lane & 7;
                    for (int row = lane >> 3; row < kTileRows; row += 4) {
                        const bool v = g.n0 + row < g.N;
                        cp_async16(dst + row * kWPitch + col * 16, v ? base + (size_t)row * row_bytes + col * 16 : g.w, v);
                    }
                } else {
                    const int cpr = bytes / 16;   // 16-byte chunks per row
                    for (int ch = lane; ch < kTileRows * cpr; ch += 32) {
                        const int row = ch / cpr, col = ch - row * cpr;
                        const bool v = g.n0 + row < g.N;
                        cp_async16(dst + row * kWPitch + col * 16, v ? base + (size_t)row * row_bytes + col * 16 : g.w, v);
                    }
                }
                cp_async_arrive(&S.full_w[ws]);
                if (++ws == kWStages) { ws = 0; wphase ^= 1; }
            }
        }
        cp_async_wait<0>();
    } else if (warp < kCvtWarpsGv) {
        // ---------------------------------------------------------- converters
        // thread = weight row = TMEM lane: per stage, read the row's 64 (or 32)
        // bytes from the weight ring, expand, tcgen05.st into the TMEM ring;
        // then wait for the stage's activation operand to land and publish the
        // stage, so that one barrier tells the MMA thread both are ready.
        const int r = tid;
        const uint32_t lane_base = tmem_base + ((uint32_t)(warp * 32) << 16);
        int ws = 0, stage = 0, bstage = 0;
        uint32_t wphase = 0, phase = 0, bphase = 0;
        bool ok = true;
        for (Seg g = seg_at(sp, n_sp, ucur, u_end); ok && g.live; g = next_seg(g)) {
            const bool valid = g.n0 + r < g.N;
            const int row_bytes = g.K / 4;
            const int end = min(g.st_hi * 64, row_bytes);
            for (int off = g.st_lo * 64; ok && off < end; off += 128) {
                const int bytes = min(128, end - off);
                if (!tc::mbar_wait_spin(&S.full_w[ws], wphase, abort_flag, kWaitLimitGv)) { fail(32); ok = false; break; }
                const uint8_t* row = sW + (size_t)ws * kWStageBytes + r * kWPitch;
                for (int so = 0; so < bytes; so += 64) {            // one pipeline stage: 64 (or 32) bytes
                    const bool two = bytes - so >= 64;              // 256 positions, else 128
                    uint4 c[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) c[i] = make_uint4(0, 0, 0, 0);
                    if (valid) {
                        c[0] = *reinterpret_cast<const uint4*>(row + so);
                        c[1] = *reinterpret_cast<const uint4*>(row + so + 16);
                        if (two) {
                            c[2] = *reinterpret_cast<const uint4*>(row + so + 32);
                            c[3] = *reinterpret_cast<const uint4*>(row + so + 48);
                        }
                    }
                    if (so + 64 >= bytes) tc::mbar_arrive(&S.empty_w[ws]);   // this row's bytes of the ring stage are read
                    uint32_t v[64];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t w4[4] = {c[i].x, c[i].y, c[i].z, c[i].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int w = 4 * i + j;   // word of the 64 bytes (group = w / 8)
                            v[4 * w + 0] = (w4[j] >> 6) & 0x03030303u;
                            v[4 * w + 1] = (w4[j] >> 4) & 0x03030303u;
                            v[4 * w + 2] = (w4[j] >> 2) & 0x03030303u;
                            v[4 * w + 3] = w4[j] & 0x03030303u;
                        }
                    }
                    if (!tc::mbar_wait_spin(&S.empty[stage], phase ^ 1, abort_flag, kWaitLimitGv)) { fail(32); ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t col0 = lane_base + (uint32_t)(stage * 64);
                    uint32_t (&v0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[0]);
                    uint32_t (&v1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[32]);
                    tc::tmem_st_32x32b_x32(col0, v0);
                    if (two) tc::tmem_st_32x32b_x32(col0 + 32, v1);
                    tc::tmem_st_wait();
                    // the stage's activation operand must have landed before publishing
                    if (!tc::mbar_wait_spin(&S.full_b[bstage], bphase, abort_flag, kWaitLimitGv)) { fail(32); ok = false; break; }
                    tc::tc_fence_before();
                    tc::mbar_arrive(&S.full_a[stage]);
                    if (++stage == kStagesGv) { stage = 0; phase ^= 1; }
                    if (++bstage == b_stages) { bstage = 0; bphase ^= 1; }
                }
                if (++ws == kWStages) { ws = 0; wphase ^= 1; }
            }
        }
    } else if (warp == kBProdWarp) {
        // ---------------------------------------------- activation producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool pending[kBStagesMax] = {};
            uint32_t pending_phase[kBStagesMax] = {};
            bool ok = true;
            {
                const Seg g0 = seg_at(sp, n_sp, ucur, u_end);
                if (g0.live) tc::tma_prefetch_desc(&a.maps[g0.map]);
            }
            for (Seg g = seg_at(sp, n_sp, ucur, u_end); ok && g.live; g = next_seg(g)) {
                const CUtensorMap* map = &a.maps[g.map];
                {   // fetch the next segment's descriptor while this one streams
                    const Seg gn = seg_at(sp, n_sp, ucur + g.units, u_end);
                    if (gn.live && gn.map != g.map) tc::tma_prefetch_desc(&a.maps[gn.map]);
                }
                for (int kb = g.st_lo; kb < g.st_hi; ++kb) {
                    const bool two = (kb + 1) * kKB <= g.K;
                    if (!tc::mbar_wait_spin(&S.empty_b[stage], phase ^ 1, abort_flag, kWaitLimitGv)) { fail(64); ok = false; break; }
                    tc::mbar_arrive_expect_tx(&S.full_b[stage], two ? b_stage_bytes : b_sub);
                    uint8_t* dst = sB + (size_t)stage * b_stage_bytes;
                    tc::tma_load_2d(dst, map, kb * kKB, 0, &S.full_b[stage]);
                    if (two) tc::tma_load_2d(dst + b_sub, map, kb * kKB + 128, 0, &S.full_b[stage]);
                    pending[stage] = true;
                    pending_phase[stage] = phase;
                    if (++stage == b_stages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok)
                for (int s = 0; s < b_stages; ++s)
                    if (pending[s]) tc::mbar_wait(&S.full_b[s], pending_phase[s], abort_flag, kWaitLimitGv / 8);
        }
    } else if (warp == kMmaWarpGv) {
        // ---------------------------------------------------------------- MMA
        // One wait per stage: a complete full_a implies the activation operand
        // has landed too (the converters waited for it before arriving).
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_e4m3_f32(kTileRows, 2 * Mp);
            int stage = 0, bstage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (Seg g = seg_at(sp, n_sp, ucur, u_end); ok && g.live; g = next_seg(g)) {
                if (!tc::mbar_wait_spin(&S.tmem_empty[acc], acc_phase ^ 1, abort_flag, kWaitLimitGv)) { fail(128); break; }
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem_base + kDCol0 + (uint32_t)(acc * 32);
                for (int kb = g.st_lo; kb < g.st_hi; ++kb) {
                    const int steps = (kb + 1) * kKB <= g.K ? 8 : 4;   // 32 positions per MMA
                    if (!tc::mbar_wait_spin(&S.full_a[stage], phase, abort_flag, kWaitLimitGv)) { fail(256); ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t b0 = tc::smem_u32(sB + (size_t)bstage * b_stage_bytes);
                    const uint64_t bd0 = tc::sdesc_sw128_kmajor(b0);
                    const uint64_t bd1 = tc::sdesc_sw128_kmajor(b0 + b_sub);
                    for (int k = 0; k < steps; ++k)
                        tc::umma_f8f6f4_tmem_a(d_tmem, tmem_base + (uint32_t)(stage * 64 + k * 8),
                                               (k < 4 ? bd0 : bd1) + 2 * (k & 3), idesc, (kb != g.st_lo) || k != 0);
                    tc::umma_commit(&S.empty[stage]);
                    tc::umma_commit(&S.empty_b[bstage]);
                    if (++stage == kStagesGv) { stage = 0; phase ^= 1; }
                    if (++bstage == b_stages) bstage = 0;
                }
                if (!ok) break;
                tc::umma_commit(&S.tmem_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            tc::umma_commit(&S.mma_done);
            tc::mbar_wait(&S.mma_done, 0, abort_flag, kWaitLimitGv / 8);
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ------------------------------------------------------------ epilogue
        // A segment that covers all K chunks of its tile writes y directly.
        // Otherwise its exact int32 partial dots are added to the workspace;
        // the segment whose chunks complete the tile's count applies the
        // epilogue to the summed dots (integer addition is order-independent).
        const int q = warp - kEpiWarp0;   // TMEM lane quarter
        const int r = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0, sync_phase = 0;
        for (Seg g = seg_at(sp, n_sp, ucur, u_end); g.live; g = next_seg(g)) {
            const int n = g.n0 + r;
            if (!tc::mbar_wait(&S.tmem_full[acc], acc_phase, abort_flag, kWaitLimitGv)) { fail(512); break; }
            tc::tc_fence_after();
            uint32_t v[32];
            tc::tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + kDCol0 + (uint32_t)(acc * 32), v);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            tc::mbar_arrive(&S.tmem_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            int dot[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                // "lo" operand rows start at column Mp (8 or 16); indices stay static
                const float d_hi = __uint_as_float(v[m]);
                const float d_lo = __uint_as_float(Mp == 8 ? v[(8 + m) & 31] : v[(16 + m) & 31]);
                dot[m] = __float2int_rn(__fmul_rn(d_hi, 512.0f)) + __float2int_rn(__fmul_rn(d_lo, 512.0f));
            }
            bool write = g.c_lo == 0 && g.c_hi == g.chunks;
            if (!write) {
                int32_t* part = a.dot_base + g.dot_off;
                if (n < g.N) {
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        if (m < a.M) atomicAdd(&part[(size_t)m * g.N + n], dot[m]);
                }
                __threadfence();
                tc::mbar_arrive(&S.epi_sync);
                if (!tc::mbar_wait_spin(&S.epi_sync, sync_phase, abort_flag, kWaitLimitGv)) { fail(2048); break; }
                if (r == 0) {
                    __threadfence();
                    const unsigned prev = atomicAdd(&a.ticket_base[g.ticket_off + g.tile], (unsigned)g.units);
                    S.final_flag = prev + (unsigned)g.units == (unsigned)g.chunks;
                    tc::mbar_arrive(&S.epi_bcast);
                }
                if (!tc::mbar_wait_spin(&S.epi_bcast, sync_phase, abort_flag, kWaitLimitGv)) { fail(2048); break; }
                sync_phase ^= 1;
                write = S.final_flag != 0;
                if (write) {
                    __threadfence();
                    if (n < g.N) {
#pragma unroll
                        for (int m = 0; m < 16; ++m)
                            if (m < a.M) dot[m] = __ldcg(&part[(size_t)m * g.N + n]);
                    }
                }
            }
            if (write && n < g.N) {
                const float w_scale = *reinterpret_cast<const float*>(g.w + (size_t)g.N * (g.K / 4));
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    if (m < a.M) {
                        const float sc = __fmul_rn(w_scale, g.act_scale[m]);
                        g.y[(size_t)m * g.N + n] = __fmul_rn(__int2float_rn(dot[m] - g.row_sum[m]), sc);
                    }
                }
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpGv) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, kTmemColsGv);
    }
}

}  // namespace

cudaError_t launch_gemv_tc(const TcArgs& a, int grid, cudaStream_t s) {
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(k_i2s_gemv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemGvBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    k_i2s_gemv_tc<<<grid, kThreadsGv, kSmemGvBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace i2s
