// Prefill GEMM for the I2_S ternary x INT8 matmul (M > 16 activation rows) on
// the 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA)
// ("ggml-cpu: ternary I2_S matmul kernel", sections Arithmetic and Kernels;
// "ggml: additive INT8/ternary types ...", "Arithmetic is exact where it can
// be").
//
// sm_103a has no integer tcgen05 MMA, so the exact int32 dot sum_k code*q is
// formed with kind::f16 and f32 accumulation, exactly:
//   * a code c in {0,1,2} placed in the low bits of an f16 is the subnormal
//     c*2^-24, so a shift and a mask turn two packed codes into an f16 pair;
//   * q in [-127,127] is an exact f16 integer (the quantizer writes it so);
//   * every product and partial sum is an integer multiple of 2^-24 of
//     magnitude <= 254*K*2^-24 < 1 for K <= 66052, which binary32 holds
//     exactly, so dot = D * 2^24 exactly.
//
// Roles (one CTA per SM, persistent over a static tile schedule):
//   warps 0-3  epilogue: TMEM -> registers, y = (float)(dot - row_sum) *
//              (w_scale * act_scale), coalesced F32 stores (warp w reads
//              TMEM lanes 32w..32w+31 = weight rows of the tile);
//   warps 4-11 converters: two threads per weight row of the 128-row tile,
//              each loading 8 of the row's 16 packed bytes per K block (64
//              positions) and expanding them to 32 f16 in the 128B-swizzled
//              K-major layout, then fencing the writes into the async proxy;
//   warp 12    TMA producer of the activation tile (f16, 128B swizzle);
//   warps 13-14 MMA issue (one lane each; warp 13 also allocates TMEM).
// CTA pairs: the kernel runs on clusters of two CTAs on two SMs driving
// cta_group::2 MMAs. A tile is 256 weight rows (the "swapped" A operand; 128
// converted in each CTA's shared memory, 128 accumulator rows in each CTA's
// TMEM) x up to 256 activation rows (the B operand; half of them TMA'd into
// each CTA's shared memory). The leader (rank 0) issues M = 256 x N x K = 16
// MMAs, 4 per K block; both CTAs' converters and TMA loads report to the
// leader's stage barriers, its commits multicast to both CTAs, and each CTA's
// epilogue releases the leader's accumulator barrier by a remote arrive. Two
// TMEM accumulators of 256 columns let the epilogue of one tile overlap the
// MMAs of the next. One thread needs well over 100 SM cycles to issue a
// tcgen05.mma, so two warps issue, taking the K blocks of the stream in turn,
// both into the tile's accumulator: every MMA accumulates, the epilogue zeroes
// an accumulator after reading it, and since every partial sum is exact the
// order in which the two streams land does not matter.
//
// K order: the converters emit a K block's 64 positions in the order in which
// the packed bytes yield them (per 32-bit word: for each bit-pair slice, bytes
// (0,2) then (1,3)); the quantizer writes the activation operand in the same
// order (quant.cu, perm_index_of), and a dot product does not depend on the
// order of its terms.
//
// Every wait is bounded: after ~1 s without progress the kernel records a
// timeout in the status word, lets its own TMA copies land (bounded), waits
// for its issued MMAs (bounded), frees TMEM and returns.

#include <atomic>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace i2s {

namespace {

constexpr int kEpiWarps = 4;
constexpr int kCvtWarps = 8;               // two threads per weight row, 8 packed bytes each
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;                // warps 13-14
constexpr int kIssuersTc = 2;
constexpr int kThreadsTc = 480;
constexpr int kStagesTc = 6;
constexpr int kCvtPrefetch = 8;             // K blocks of packed codes each converter keeps in flight
constexpr int kBlockK = 64;                 // K positions per stage (one 128-byte f16 row)
constexpr int kTileW = 128;                 // weight rows per tile (MMA M)
constexpr int kATileBytes = kTileW * 128;   // 16 KB
constexpr int kBTileBytesMax = 128 * 128;   // 16 KB: this CTA's half of up to 256 activation rows
constexpr int kTmemCols = 512;
constexpr long long kWaitLimit = 2000000000LL;   // ~1 s of SM clocks
// Issuer i takes the K blocks s with s % kIssuersTc == i; each stage slot must
// always be served by the same issuer (a parity wait cannot tell the phase it
// wants from the one two phases later).
static_assert(kStagesTc % kIssuersTc == 0, "ring slots per issuer");
static_assert(kCvtPrefetch % 2 == 0, "converters take K blocks in pairs");

struct SmemTc {
    float sc_col[2][256];   // epilogue: w_scale * act_scale[m] per tile column, by accumulator
    float rs_col[2][256];   // epilogue: row_sum[m] per tile column (exact as a float), by accumulator
    uint64_t full_a[kStagesTc];
    uint64_t full_b[kStagesTc];
    uint64_t empty[kStagesTc];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done[kIssuersTc];
    uint64_t stage_bar;     // the epilogue threads have staged a tile's column factors
    alignas(16) uint8_t signal[16];   // source (peer) and destination (leader) of the stage-ready copies
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemTcBytes = 1024 + (size_t)kStagesTc * (kATileBytes + kBTileBytesMax) + sizeof(SmemTc);

__device__ __forceinline__ int find_problem(const TcArgs& a, int tile) {
    int lo = 0, hi = a.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.p[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Expands one 32-bit word of packed codes into 8 f16 pairs (two 16-byte
// chunks): for slices s = 6, 4, 2, 0: (byte0, byte2) then (byte1, byte3).
__device__ __forceinline__ void expand_word_f16(uint32_t w, uint4& c0, uint4& c1) {
    constexpr uint32_t m = 0x00030003u;
    c0.x = (w >> 6) & m;  c0.y = (w >> 14) & m;
    c0.z = (w >> 4) & m;  c0.w = (w >> 12) & m;
    c1.x = (w >> 2) & m;  c1.y = (w >> 10) & m;
    c1.z = w & m;         c1.w = (w >> 8) & m;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsTc, 1) k_i2s_gemm_tc(const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + (size_t)kStagesTc * kATileBytes;
    SmemTc& S = *reinterpret_cast<SmemTc*>(sB + (size_t)kStagesTc * kBTileBytesMax);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int BN = a.BN;
    const int BH = BN / 2;                                  // activation rows of a tile in each CTA
    const uint32_t b_half_bytes = (uint32_t)BH * 128u;
    const uint32_t rank = tc::cluster_rank();               // 0: the leader, which issues the MMAs
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

    if (tid == 0) {
        for (int s = 0; s < kStagesTc; ++s) {
            // one arrive per converter warp; the leader's also counts the
            // 16 bytes of the peer's stage-ready copy
            tc::mbar_init(&S.full_a[s], kCvtWarps);
            tc::mbar_init(&S.full_b[s], 1);
            tc::mbar_init(&S.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&S.tmem_full[b], kIssuersTc);
            tc::mbar_init(&S.tmem_empty[b], 2 * kEpiWarps);   // one arrive per epilogue warp of both CTAs
        }
        for (int i = 0; i < kIssuersTc; ++i) tc::mbar_init(&S.mma_done[i], 1);
        tc::mbar_init(&S.stage_bar, kEpiWarps * 32);
        S.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == kMmaWarp) {   // one warp of each CTA, collectively for the pair
        tc::pair_tmem_alloc(&S.tmem_base, kTmemCols);
        tc::pair_tmem_relinquish();
    }
    if (warp == kTmaWarp && lane == 0)
        for (int i = 0; i < a.n_maps; ++i) tc::tma_prefetch_desc(&a.maps[i]);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = S.tmem_base;
    volatile int* abort_flag = &S.abort;
    if (warp < kEpiWarps) {
        // both accumulators start at zero (every MMA accumulates)
        for (uint32_t col = 0; col < (uint32_t)kTmemCols; col += 32)
            tc::tmem_st_zero_32x32b_x32(tmem_base + ((uint32_t)(warp * 32) << 16) + col);
        tc::tmem_st_wait();
    }
    // both CTAs' barriers initialised and accumulators zeroed before any
    // remote arrive, multicast commit or MMA
    tc::tc_fence_before();
    tc::cluster_sync();
    tc::tc_fence_after();

    auto fail = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(a.status, code);
    };

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool pending[kStagesTc] = {};
            uint32_t pending_phase[kStagesTc] = {};
            bool ok = true;
            for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
                const TcProb& P = a.p[find_problem(a, tile)];
                const int at = (tile - P.tile0) % P.n_act_tiles;
                const int KB = P.K / kBlockK;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&S.empty[stage], phase ^ 1, abort_flag, kWaitLimit)) { fail(1); ok = false; break; }
                    // the leader expects both CTAs' halves; a peer's bytes may land first
                    if (rank == 0) tc::mbar_arrive_expect_tx(&S.full_b[stage], 2 * b_half_bytes);
                    tc::pair_tma_load_2d(sB + (size_t)stage * kBTileBytesMax, &a.maps[P.map], kb * kBlockK,
                                         at * BN + (int)rank * BH, tc::smem_in_rank(&S.full_b[stage], 0));
                    pending[stage] = true;
                    pending_phase[stage] = phase;
                    if (++stage == kStagesTc) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && rank == 0) {
                // let the copies in flight land before the CTA exits (they are
                // counted on the leader's barriers)
                for (int s = 0; s < kStagesTc; ++s)
                    if (pending[s]) tc::mbar_wait(&S.full_b[s], pending_phase[s], abort_flag, kWaitLimit / 8);
            }
        }
    } else if (warp >= kEpiWarps && warp < kEpiWarps + kCvtWarps) {
        // ---------------------------------------------------------- converters
        // two threads per weight row: thread half hf expands the row's packed
        // bytes 8hf..8hf+7 of each K block (32 positions) into 4 f16 chunks
        const int ct = tid - kEpiWarps * 32;
        const int r = ct & (kTileW - 1);   // weight row within the tile
        const int hf = ct >> 7;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
            const TcProb& P = a.p[find_problem(a, tile)];
            const int wt = (tile - P.tile0) / P.n_act_tiles;
            const int n = wt * (2 * kTileW) + (int)rank * kTileW + r;   // this CTA's half of the 256 rows
            const int KB = P.K / kBlockK;
            const bool valid = n < P.N;
            const uint8_t* src = P.w + (size_t)(valid ? n : 0) * (P.K / 4) + 8 * hf;
            auto load = [&](int kb) {
                return (valid && kb < KB) ? __ldg(reinterpret_cast<const uint2*>(src + (size_t)kb * 16))
                                          : make_uint2(0u, 0u);
            };
            // the row's packed bytes, kCvtPrefetch K blocks ahead
            uint2 buf[kCvtPrefetch];
#pragma unroll
            for (int j = 0; j < kCvtPrefetch; ++j) buf[j] = load(j);
            for (int kb0 = 0; ok && kb0 < KB; kb0 += kCvtPrefetch) {
                // two K blocks (stage slots) per pass: one proxy fence and one
                // warp sync for both halve the per-stage latency of the loop
#pragma unroll
                for (int j = 0; j < kCvtPrefetch; j += 2) {
                    const int kb = kb0 + j;
                    if (kb >= KB) break;
                    const bool two = kb + 1 < KB;
                    const int stage1 = stage + 1 == kStagesTc ? 0 : stage + 1;
                    const uint32_t phase1 = stage + 1 == kStagesTc ? phase ^ 1 : phase;
                    // warp-uniform outcome: the warp arrives as one
                    bool got = tc::mbar_wait(&S.empty[stage], phase ^ 1, abort_flag, kWaitLimit);
                    if (got && two) got = tc::mbar_wait(&S.empty[stage1], phase1 ^ 1, abort_flag, kWaitLimit);
                    if (!__all_sync(0xffffffffu, got)) { fail(2); ok = false; break; }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h == 1 && !two) break;
                        uint8_t* dst = sA + (size_t)(h ? stage1 : stage) * kATileBytes;
                        const uint32_t words[2] = {buf[j + h].x, buf[j + h].y};
                        buf[j + h] = load(kb + h + kCvtPrefetch);
#pragma unroll
                        for (int w = 0; w < 2; ++w) {
                            const int word = 2 * hf + w;   // 32-bit word of the row's 16 bytes
                            uint4 c0, c1;
                            expand_word_f16(words[w], c0, c1);
                            *reinterpret_cast<uint4*>(dst + tc::sw128_offset(r, 2 * word)) = c0;
                            *reinterpret_cast<uint4*>(dst + tc::sw128_offset(r, 2 * word + 1)) = c1;
                        }
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    // CTA-scope arrives: a cluster-scope release here would
                    // also wait for this thread's prefetched loads to land
                    if (lane == 0) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (h == 1 && !two) break;
                            uint64_t* bar = &S.full_a[h ? stage1 : stage];
                            if (rank == 0 && warp == kEpiWarps) tc::mbar_arrive_expect_tx(bar, 16);
                            else tc::mbar_arrive(bar);
                        }
                    }
                    stage = stage1;
                    phase = phase1;
                    if (two && ++stage == kStagesTc) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp >= kMmaWarp && warp < kMmaWarp + kIssuersTc && rank == 0) {
        // ---------------------------------------------------------- MMA issue
        // issuer `me` takes the K blocks whose position in this CTA's stream
        // is me modulo kIssuersTc; the ring index advances over all of them
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16_f32(2 * kTileW, BN);   // 256 x BN over the pair
            const int me = warp - kMmaWarp;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int seq = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
                const TcProb& P = a.p[find_problem(a, tile)];
                const int KB = P.K / kBlockK;
                if (!tc::mbar_wait(&S.tmem_empty[acc], acc_phase ^ 1, abort_flag, kWaitLimit)) { fail(4); break; }
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
                for (int kb = 0; kb < KB; ++kb, ++seq) {
                    if (seq % kIssuersTc == me) {
                        if (!tc::mbar_wait(&S.full_a[stage], phase, abort_flag, kWaitLimit) ||
                            !tc::mbar_wait(&S.full_b[stage], phase, abort_flag, kWaitLimit)) { fail(8); ok = false; break; }
                        tc::tc_fence_after();
                        const uint64_t ad = tc::sdesc_sw128_kmajor(tc::smem_u32(sA + (size_t)stage * kATileBytes));
                        const uint64_t bd = tc::sdesc_sw128_kmajor(tc::smem_u32(sB + (size_t)stage * kBTileBytesMax));
#pragma unroll
                        for (int k = 0; k < kBlockK / 16; ++k)   // +32 bytes per 16-element K step
                            tc::pair_umma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, 1u);
                        tc::pair_commit(&S.empty[stage], 0x3);   // both CTAs' stage slots are free
                    }
                    if (++stage == kStagesTc) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                // the tile is complete (in both CTAs' TMEM) once every issuer's MMAs are
                tc::pair_commit(&S.tmem_full[acc], 0x3);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            // every MMA this thread issued has completed before TMEM is freed
            tc::pair_commit(&S.mma_done[me], 0x1);
            tc::mbar_wait(&S.mma_done[me], 0, abort_flag, kWaitLimit / 8);
        }
    } else if (warp == kMmaWarp && rank == 1) {
        // ---------------------------------------------------------- forwarder
        // the peer's converted stages, each signalled to the leader's barrier
        // by a 16-byte copy, in the order the MMAs consume them (a remote
        // release arrive costs over a thousand cycles, serialising the ring)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
                const int KB = a.p[find_problem(a, tile)].K / kBlockK;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&S.full_a[stage], phase, abort_flag, kWaitLimit)) { fail(8); ok = false; break; }
                    tc::dsmem_copy_signal(tc::smem_in_rank(S.signal, 0), S.signal, 16,
                                          tc::smem_in_rank(&S.full_a[stage], 0));
                    if (++stage == kStagesTc) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp < kEpiWarps) {
        // ------------------------------------------------------------ epilogue
        const int r = warp * 32 + lane;   // TMEM lane = weight row within the tile
        int acc = 0;
        uint32_t acc_phase = 0, stage_phase = 0;
        for (int tile = pair; tile < a.total_tiles; tile += n_pairs) {
            const TcProb& P = a.p[find_problem(a, tile)];
            const int local = tile - P.tile0;
            const int wt = local / P.n_act_tiles, at = local % P.n_act_tiles;
            const int n = wt * (2 * kTileW) + (int)rank * kTileW + r;
            // stage the tile's per-column factors (w_scale * act_scale[m] and
            // row_sum[m]) in shared memory while the accumulator fills
            const int m_base = at * BN;
            {
                const float w_scale = *reinterpret_cast<const float*>(P.w + (size_t)P.N * (P.K / 4));
                float* sc_col = S.sc_col[acc];
                float* rs_col = S.rs_col[acc];
                for (int j = r; j < BN; j += kEpiWarps * 32) {
                    const int m = m_base + j;
                    sc_col[j] = m < a.M ? __fmul_rn(w_scale, P.act_scale[m]) : 0.0f;
                    rs_col[j] = m < a.M ? (float)P.row_sum[m] : 0.0f;   // |row_sum| <= 127 K < 2^24
                }
                // every epilogue thread has staged its columns (bounded wait)
                tc::mbar_arrive(&S.stage_bar);
                if (!__all_sync(0xffffffffu, tc::mbar_wait(&S.stage_bar, stage_phase, abort_flag, kWaitLimit))) {
                    fail(16);
                    break;
                }
                stage_phase ^= 1;
            }
            if (!__all_sync(0xffffffffu, tc::mbar_wait(&S.tmem_full[acc], acc_phase, abort_flag, kWaitLimit))) {
                fail(16);
                break;
            }
            tc::tc_fence_after();
            const float* sc_col = S.sc_col[acc];
            const float* rs_col = S.rs_col[acc];
            const int N = P.N, M = a.M;
            float* y_col = P.y + n;   // this thread's output column
            // TMEM -> registers 32 columns at a time, the load of the next slice
            // overlapping the stores of this one; the accumulator is released as
            // soon as its last slice is in registers
            const uint32_t d_addr = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * 256);
            const int C = (BN + 31) / 32;
            auto store_slice = [&](int c, uint32_t (&v)[32]) {
                if (n >= N) return;
                // 16 outputs at a time, computed in place with no per-element
                // branch so that the conversions overlap, then stored (static
                // indices keep v[] in registers; jj < C * 32 <= 256 stays
                // inside the per-column tables)
                const int rows = min(BN - c * 32, M - (m_base + c * 32));
                float* yp = y_col + (size_t)(m_base + c * 32) * N;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                    for (int j = 16 * hh; j < 16 * hh + 16; ++j) {
                        const int jj = c * 32 + j;
                        // D * 2^24 is the integer dot, exact; so is dot - row_sum
                        // (|.| < 2^24): the float of (dot - row_sum) without any
                        // conversion instruction
                        const float dr = __fsub_rn(__fmul_rn(__uint_as_float(v[j]), 16777216.0f), rs_col[jj]);
                        v[j] = __float_as_uint(__fmul_rn(dr, sc_col[jj]));
                    }
                    if (rows >= 32) {
#pragma unroll
                        for (int j = 16 * hh; j < 16 * hh + 16; ++j) yp[(size_t)j * N] = __uint_as_float(v[j]);
                    } else {
#pragma unroll
                        for (int j = 16 * hh; j < 16 * hh + 16; ++j)
                            if (j < rows) yp[(size_t)j * N] = __uint_as_float(v[j]);
                    }
                }
            };
            auto release = [&]() {
                // every slice is in registers: zero the accumulator for the
                // tile after next, then hand it back
                for (int c2 = 0; c2 < C; ++c2) tc::tmem_st_zero_32x32b_x32(d_addr + 32u * c2);
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_cluster(tc::smem_in_rank(&S.tmem_empty[acc], 0));   // the leader's barrier
            };
            uint32_t va[32], vb[32];
            tc::tmem_ld_32x32b_x32(d_addr, va);
            tc::tmem_ld_wait();
            if (C == 1) release();
            for (int c = 0; c < C; c += 2) {
                if (c + 1 < C) tc::tmem_ld_32x32b_x32(d_addr + 32u * (c + 1), vb);
                store_slice(c, va);
                if (c + 1 < C) {
                    tc::tmem_ld_wait();
                    if (c + 2 == C) release();
                    if (c + 2 < C) tc::tmem_ld_32x32b_x32(d_addr + 32u * (c + 2), va);
                    store_slice(c + 1, vb);
                    if (c + 2 < C) {
                        tc::tmem_ld_wait();
                        if (c + 3 == C) release();
                    }
                }
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    // every MMA of the pair has completed (the epilogues waited for the last
    // tmem_full) and neither CTA's shared memory is read any more
    __syncwarp();
    tc::tc_fence_before();
    tc::cluster_sync();
    if (warp == kMmaWarp) {
        tc::tc_fence_after();
        tc::pair_tmem_dealloc(tmem_base, kTmemCols);
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load();
    if (f) return f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f);
    return f;
}

}  // namespace

size_t gemm_tc_smem_bytes() { return kSmemTcBytes; }

// 2-D tensor map of an f16 operand of `rows` x `K` (K contiguous), box 64 x box_rows,
// 128-byte swizzle, zero fill beyond the extents.
bool make_f16_operand_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    std::memset(map, 0, sizeof(*map));
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBlockK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map of a uint8 matrix of `rows` x `row_bytes` (row-major), box
// 128 bytes x box_rows, 128-byte swizzle, zero fill beyond the extents: the
// GEMV's activation operand and the template of its weight maps.
bool make_u8_operand_map(CUtensorMap* map, const void* base, int rows, int row_bytes, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    std::memset(map, 0, sizeof(*map));
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
    e = cudaFuncSetAttribute(k_i2s_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTcBytes);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms & ~1), 1, 1);
    cfg.blockDim = dim3(kThreadsTc, 1, 1);
    cfg.dynamicSmemBytes = kSmemTcBytes;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, (void*)k_i2s_gemm_tc, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    g_pairs[dev].store(1 + clusters);
    return cudaSuccess;
}

int gemm_tc_max_pairs() {
    int dev = 0;
    if (configure(&dev) != cudaSuccess) return 1;
    return g_pairs[dev].load() - 1;
}

cudaError_t launch_gemm_tc(const TcArgs& a, int grid, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = configure(&dev);
    if (e != cudaSuccess) return e;
    k_i2s_gemm_tc<<<grid, kThreadsTc, kSmemTcBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace i2s
