// Prefill GEMM for the I2_S ternary x INT8 matmul (M > 16 activation rows) on
// the 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA)
// ("ggml-cpu: ternary I2_S matmul kernel", sections Arithmetic and Kernels;
// "ggml: additive INT8/ternary types ...", "Arithmetic is exact where it can
// be").
//
// sm_103a has no integer tcgen05 MMA. The exact int32 dot sum_k code*q is
// formed with tcgen05.mma kind::mxf4 (packed e2m1 operands, ue8m0 block
// scales, f32 accumulation), exactly:
//   * A: a code c in {0,1,2} read as an e2m1 nibble is c/2, so
//     packed & 0x33333333 and (packed >> 2) & 0x33333333 turn a 32-bit word
//     of packed codes into sixteen operands (as in the decode GEMV);
//   * B: each quantized activation q is three balanced base-8 digits
//     q = d0 + 8*d1 + 64*d2 (d0, d1 in [-4,3], d2 in [-2,2]), each exact in
//     e2m1, stored as three digit planes (the GEMV's operand layout, one plane
//     per digit). The MMAs of plane j use the block scale 2^(3j) (ue8m0 127,
//     130, 133), so the three MMAs of a 64-position step, which share the A
//     descriptor, add (c/2)*q into ONE accumulator;
//   * every product is a multiple of 1/2 and every partial sum stays below
//     2^23: the completed steps contribute at most 127 per position, and the
//     step each of the three issue streams has in flight at most
//     (4 + 8*4 + 64*2) * 64, so 127*65536 + 3*164*64 < 2^23 and binary32
//     holds every partial sum exactly. dot = 2*D.
// Each 256-position stage holds 16 KB of A (converted, in TMEM) and
// 3 * BN/2 * 128 bytes of B (shared memory) per CTA, and the tensor time of a
// step is that of three fp4 MMAs.
//
// Roles (one CTA per SM, persistent over a static tile schedule):
//   warps 0-7  epilogue: TMEM -> registers, y = (float)(dot - row_sum) *
//              (w_scale * act_scale), coalesced F32 stores (warp w reads
//              TMEM lanes 32(w%4)..+31 = weight rows of the tile, columns
//              (w/4)*BN/2..+BN/2-1 = activation rows);
//   warps 8-11 converters: one thread per weight row of the 128-row tile =
//              TMEM lane, reading the row's 64 packed bytes of a stage from
//              the code ring and storing its 128 bytes of e2m1 operands
//              (32 columns) into the stage's slot of a six-stage A ring in
//              TMEM (tcgen05.st), which the MMAs read as their A operand;
//   warp 12    TMA producer of the three digit planes of the activation tile;
//   warps 13-15 MMA issue (one lane each; warp 13 also allocates TMEM): one
//              thread needs about a hundred cycles to issue an MMA, more than
//              the MMA's tensor time, so three take the stages in turn;
//   warp 16    producer of the packed codes: a three-stage ring of 128 rows
//              x 128 bytes (two operand stages, 128-byte swizzle) that runs
//              ahead of the operand ring, so the converters never wait on
//              global loads; one TMA tile per stage, or on tiled weights one
//              bulk copy of a block that is already in the ring's layout.
// CTA pairs: the kernel runs on clusters of two CTAs on two SMs driving
// cta_group::2 MMAs. A tile is 256 weight rows (128 converted into each CTA's
// TMEM, 128 accumulator rows in each CTA's TMEM) x BN <= 128 activation rows
// (half of each plane TMA'd into each CTA's shared memory).
// The leader (rank 0) issues M = 256 x N = BN x K = 64 MMAs, 12 per stage;
// both CTAs' converters and TMA loads report to the leader's stage barriers,
// its commits multicast to both CTAs, and each CTA's epilogue releases the
// leader's accumulator barrier by a remote arrive. TMEM per CTA: two
// accumulators of 128 columns (the epilogue of one tile overlaps the MMAs of
// the next), the block scales (64 columns) and the A ring (6 x 32 columns).
// The issuers all accumulate into the tile's accumulator.
//
// K order: within a 128-position group, element 16w + 8t + 2i + h of the A
// and B rows holds position 32s + 4w + i, where (t, h) = (0,0), (0,1), (1,0),
// (1,1) for bit-pair slices s = 3, 1, 2, 0: the order in which the masks
// yield the packed codes. The quantizer writes the digit planes in the same
// order (quant.cu, kQuantE2M1Tc), and a dot product does not depend on the
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

constexpr int kEpiWarps = 8;               // two per TMEM lane quarter, each half of the columns
constexpr int kCvtWarps = 4;               // one thread per weight row
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;                // warps 13-15
constexpr int kCodeWarp = 16;               // TMA producer of the packed codes
constexpr int kIssuersTc = 3;
constexpr int kThreadsTc = 544;
constexpr int kStagesTc = 6;
constexpr int kCodeStages = 3;              // ring of packed-code stages, ahead of the operand ring
constexpr int kCodeStageBytes = 128 * 128;  // 128 weight rows x 128 packed bytes (512 positions: two operand stages)
static_assert(kCodeStageBytes == kTiledBlockBytes, "a code stage is one block of tiled weights");
constexpr int kBlockK = 256;                // K positions per stage (one 128-byte row of e2m1)
constexpr int kTileW = 128;                 // weight rows per CTA (half of the pair's MMA M)
constexpr int kBPlaneMax = 64 * 128;        // one digit plane of this CTA's half of up to 128 activation rows
constexpr int kBStageMax = 3 * kBPlaneMax;  // 24 KB
constexpr int kTmemCols = 512;
constexpr uint32_t kAccCols = 128;          // two accumulators of BN <= 128 columns
constexpr uint32_t kSfaCol = 256;           // block scales: A (all 1), then B for digits 0, 1, 2 (1, 8, 64)
constexpr uint32_t kSfbCol0 = 272;
constexpr uint32_t kSfCols = 16;
constexpr uint32_t kACol0 = 320;            // the A ring in TMEM: one stage of 256 e2m1 per lane
constexpr uint32_t kAStageCols = 32;        //   (eight per 32-bit column) per kAStageCols columns
constexpr long long kWaitLimit = 2000000000LL;   // ~1 s of SM clocks
static_assert(kStagesTc % kIssuersTc == 0, "ring slots per issuer");
static_assert(kSfbCol0 + 3 * kSfCols <= kACol0, "TMEM budget: scales below the A ring");
static_assert(kACol0 + kStagesTc * kAStageCols <= (uint32_t)kTmemCols, "TMEM budget: the A ring");

struct SmemTc {
    TcProb prob[kMaxGroup];   // the launch's problem table, copied from the parameters
    float sc_col[2][128];   // epilogue: w_scale * act_scale[m] per tile column, by accumulator
    float rs_col[2][128];   // epilogue: row_sum[m] per tile column (exact as a float), by accumulator
    uint64_t full_a[kStagesTc];
    uint64_t full_b[kStagesTc];
    uint64_t empty[kStagesTc];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done[kIssuersTc];
    uint64_t code_full[kCodeStages];    // a stage of packed codes has landed
    uint64_t code_empty[kCodeStages];   // every converter warp has read it
    uint64_t stage_bar;     // the epilogue threads have staged a tile's column factors
    alignas(16) uint8_t signal[16];   // source (peer) and destination (leader) of the stage-ready copies
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemTcBytes =
    1024 + (size_t)kStagesTc * kBStageMax + (size_t)kCodeStages * kCodeStageBytes + sizeof(SmemTc);

// The problem holding `tile`, from the problem before: each role visits its
// tiles in increasing order, and the problems' tile ranges are in order, so
// the search only moves forward (over the shared-memory copy of the table).
__device__ __forceinline__ int next_problem(const TcProb* sp, int count, int pi, int tile) {
    while (pi + 1 < count && sp[pi + 1].tile0 <= tile) ++pi;
    return pi;
}

// Two 32-bit words of packed codes -> one 16-byte chunk of e2m1 operands:
// for each word, the codes at shifts 0 and 4 (slices 3 and 1), then those at
// shifts 2 and 6 (slices 2 and 0), one nibble each (c/2 in e2m1).
__device__ __forceinline__ uint4 expand_words_e2m1(uint32_t w0, uint32_t w1) {
    constexpr uint32_t m = 0x33333333u;
    return make_uint4(w0 & m, (w0 >> 2) & m, w1 & m, (w1 >> 2) & m);
}

// Arrive on a barrier of the cluster without release semantics. The epilogue
// releases an accumulator with it: what the MMAs must not overtake are its
// TMEM loads and zeroing stores, complete at tcgen05.wait::ld / ::st before
// it, not its global stores of y, which a release arrive would wait for (over
// a thousand cycles per warp and tile).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Leader only: D (+)= A * B^T over the pair, kind::mxf4 with block scaling, A
// read from both CTAs' TMEM (each CTA's 128 lanes, eight e2m1 per 32-bit
// column, element 8c + i in bits 4i..4i+3 of column c), B in shared memory.
__device__ __forceinline__ void pair_umma_mxf4_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                      uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                      uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], [%1], %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsTc, 1) k_i2s_gemm_tc(const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sB = smem;
    uint8_t* sC = sB + (size_t)kStagesTc * kBStageMax;   // packed codes (1024-aligned)
    SmemTc& S = *reinterpret_cast<SmemTc*>(sC + (size_t)kCodeStages * kCodeStageBytes);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int BN = a.BN;                                    // activation rows per tile (<= 128)
    const int BH = BN / 2;                                  // of them in each CTA
    const uint32_t plane_bytes = (uint32_t)BH * 128u;       // one digit plane of this CTA's half
    const int rows_pad = a.n_act_rows;                      // rows of one digit plane of the operand
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
        for (int s = 0; s < kCodeStages; ++s) {
            tc::mbar_init(&S.code_full[s], 1);
            tc::mbar_init(&S.code_empty[s], kCvtWarps);
        }
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
    static_assert(sizeof(TcProb) % 16 == 0, "problem entries copy as 16-byte words");
    for (int i = tid; i < a.count * (int)(sizeof(TcProb) / 16); i += kThreadsTc)
        reinterpret_cast<uint4*>(S.prob)[i] = reinterpret_cast<const uint4*>(a.p)[i];
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = S.tmem_base;
    volatile int* abort_flag = &S.abort;
    if (warp < 4) {
        // both accumulators start at zero (every MMA accumulates); the block
        // scales: 1.0 for A, 2^(3j) for digit plane j, in every lane and byte
        // (warps 0-3 cover the four lane quarters)
        const uint32_t lane_base = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
        for (uint32_t col = 0; col < 2 * kAccCols; col += 32) tc::tmem_st_zero_32x32b_x32(lane_base + col);
        uint32_t sf[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) sf[i] = 0x7F7F7F7Fu;
        tc::tmem_st_32x32b_x16(lane_base + kSfaCol, sf);
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const uint32_t e = 127u + 3u * (uint32_t)j;
#pragma unroll
            for (int i = 0; i < 16; ++i) sf[i] = e * 0x01010101u;
            tc::tmem_st_32x32b_x16(lane_base + kSfbCol0 + kSfCols * (uint32_t)j, sf);
        }
        tc::tmem_st_wait();
    }
    // both CTAs' barriers initialised, accumulators zeroed and scales written
    // before any remote arrive, multicast commit or MMA
    tc::tc_fence_before();
    tc::cluster_sync();
    tc::tc_fence_after();

    auto fail = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(a.status, code);
    };

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        // per stage: this CTA's half of the tile's rows in each digit plane
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool pending[kStagesTc] = {};
            uint32_t pending_phase[kStagesTc] = {};
            bool ok = true;
            int pi = 0;
            for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
                pi = next_problem(S.prob, a.count, pi, tile);
                const TcProb& P = S.prob[pi];
                const int at = (tile - P.tile0) % P.n_act_tiles;
                const int KB = P.K / kBlockK + (P.K % kBlockK ? 1 : 0);
                const int row = at * BN + (int)rank * BH;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&S.empty[stage], phase ^ 1, abort_flag, kWaitLimit)) { fail(1); ok = false; break; }
                    // the leader expects both CTAs' planes; a peer's bytes may land first
                    if (rank == 0) tc::mbar_arrive_expect_tx(&S.full_b[stage], 6 * plane_bytes);
                    uint8_t* dst = sB + (size_t)stage * kBStageMax;
                    const uint32_t bar = tc::smem_in_rank(&S.full_b[stage], 0);
#pragma unroll
                    for (int j = 0; j < 3; ++j)
                        tc::pair_tma_load_2d(dst + (size_t)j * plane_bytes, &a.maps[P.map], kb * (kBlockK / 2),
                                             j * rows_pad + row, bar);
                    pending[stage] = true;
                    pending_phase[stage] = phase;
                    if (++stage == kStagesTc) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && rank == 0) {
                // let the copies in flight land before the CTA exits (they are
                // counted on the leader's barriers)
                for (int s = 0; s < kStagesTc; ++s)
                    if (pending[s]) tc::mbar_wait_drain(&S.full_b[s], pending_phase[s], kWaitLimit / 8);
            }
        }
    } else if (warp == kCodeWarp) {
        // ------------------------------------------------------- code producer
        // per stage: this CTA's 128 weight rows x 128 packed bytes of the
        // tile (rows past N and bytes past K/4 are zero-filled), from the
        // problem's map (written by the quantization launch), into a ring that
        // runs ahead of the operand stages; on tiled weights the stage is one
        // 16 KB block, already in the ring's layout: one bulk copy
        if (lane == 0) {
            int cs = 0;
            uint32_t cphase = 0;
            bool pending[kCodeStages] = {};
            uint32_t pending_phase[kCodeStages] = {};
            bool ok = true;
            int cur_p = -1, pi = 0;
            for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
                pi = next_problem(S.prob, a.count, pi, tile);
                const TcProb& P = S.prob[pi];
                const CUtensorMap* map = a.wmaps + pi;
                if (pi != cur_p) {   // first use of this map: order it after the writer's release
                    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
                    cur_p = pi;
                }
                const int wt = (tile - P.tile0) / P.n_act_tiles;
                const int n0 = wt * (2 * kTileW) + (int)rank * kTileW;
                const int KB = P.K / kBlockK + (P.K % kBlockK ? 1 : 0);
                const bool tiled = (a.tiled[pi >> 5] >> (pi & 31)) & 1u;
                // tiled: this CTA's row block; its column blocks follow one another
                const uint8_t* blk = P.w + (size_t)(n0 / kTiledRows) * tiled_col_blocks(P.K) * kTiledBlockBytes;
                for (int kb = 0; kb < KB; kb += 2) {   // one code stage per two operand stages
                    if (!tc::mbar_wait(&S.code_empty[cs], cphase ^ 1, abort_flag, kWaitLimit)) { fail(32); ok = false; break; }
                    tc::mbar_arrive_expect_tx(&S.code_full[cs], kCodeStageBytes);
                    if (tiled)
                        tc::bulk_load(sC + (size_t)cs * kCodeStageBytes, blk + (size_t)(kb / 2) * kTiledBlockBytes,
                                      kCodeStageBytes, &S.code_full[cs]);
                    else
                        tc::tma_load_2d(sC + (size_t)cs * kCodeStageBytes, map, kb * 64, n0, &S.code_full[cs]);
                    pending[cs] = true;
                    pending_phase[cs] = cphase;
                    if (++cs == kCodeStages) { cs = 0; cphase ^= 1; }
                }
            }
            if (!ok)
                for (int s2 = 0; s2 < kCodeStages; ++s2)
                    if (pending[s2]) tc::mbar_wait_drain(&S.code_full[s2], pending_phase[s2], kWaitLimit / 8);
        }
    } else if (warp >= kEpiWarps && warp < kEpiWarps + kCvtWarps) {
        // ---------------------------------------------------------- converters
        // one thread per weight row: per operand stage the row's 64 packed
        // bytes (two 128-position groups), read from a code stage (128-byte
        // swizzle; one code stage holds two operand stages), become the 128
        // bytes of e2m1 operands of the stage row
        const int r = tid - kEpiWarps * 32;   // weight row within the CTA's half of the tile
        // = TMEM lane: converter warp w reaches lane quarter w % 4
        const uint32_t lane_a = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + kACol0;
        int stage = 0, cs = 0;
        uint32_t phase = 0, cphase = 0;
        bool ok = true;
        int pi = 0;
        for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
            pi = next_problem(S.prob, a.count, pi, tile);
            const TcProb& P = S.prob[pi];
            const int KB = P.K / kBlockK + (P.K % kBlockK ? 1 : 0);
            for (int kb = 0; ok && kb < KB; kb += 2) {
                // two stages per pass: one proxy fence and one warp sync for both
                const bool two = kb + 1 < KB;
                const int stage1 = stage + 1 == kStagesTc ? 0 : stage + 1;
                const uint32_t phase1 = stage + 1 == kStagesTc ? phase ^ 1 : phase;
                // the codes first (their slots free as soon as they are in
                // registers), then the operand slots; warp-uniform outcomes
                bool got = tc::mbar_wait(&S.code_full[cs], cphase, abort_flag, kWaitLimit);
                if (!__all_sync(0xffffffffu, got)) { fail(2); ok = false; break; }
                uint4 v[2][4];
                {
                    const uint8_t* src = sC + (size_t)cs * kCodeStageBytes;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int c = 0; c < 4; ++c)   // operand stage h: 16-byte pieces 4h..4h+3 of the row
                            v[h][c] = (h == 1 && !two) ? make_uint4(0u, 0u, 0u, 0u)
                                                       : *reinterpret_cast<const uint4*>(src + tc::sw128_offset(r, 4 * h + c));
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&S.code_empty[cs]);
                got = tc::mbar_wait(&S.empty[stage], phase ^ 1, abort_flag, kWaitLimit);
                if (got && two) got = tc::mbar_wait(&S.empty[stage1], phase1 ^ 1, abort_flag, kWaitLimit);
                if (!__all_sync(0xffffffffu, got)) { fail(2); ok = false; break; }
                // the MMAs that read these A stages have completed (their
                // commit released the empty barriers): TMEM stores after them
                tc::tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && !two) break;
                    // code word j -> e2m1 columns 2j and 2j + 1 of the lane's stage
                    uint32_t e[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 c4 = expand_words_e2m1(v[h][i].x, v[h][i].y);
                        const uint4 d4 = expand_words_e2m1(v[h][i].z, v[h][i].w);
                        e[8 * i] = c4.x, e[8 * i + 1] = c4.y, e[8 * i + 2] = c4.z, e[8 * i + 3] = c4.w;
                        e[8 * i + 4] = d4.x, e[8 * i + 5] = d4.y, e[8 * i + 6] = d4.z, e[8 * i + 7] = d4.w;
                    }
                    tc::tmem_st_32x32b_x32(lane_a + (uint32_t)(h ? stage1 : stage) * kAStageCols, e);
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                // CTA-scope arrives: a cluster-scope release here would
                // also wait for this thread's earlier memory operations
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
                if (++cs == kCodeStages) { cs = 0; cphase ^= 1; }
            }
        }
    } else if (warp >= kMmaWarp && warp < kMmaWarp + kIssuersTc && rank == 0) {
        // ---------------------------------------------------------- MMA issue
        // issuer `me` takes the stages whose position in this CTA's stream is
        // me modulo kIssuersTc; the ring index advances over all of them. Per
        // 64-position step the three digit MMAs are issued back to back (the
        // exactness bound above relies on it).
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_mxf4_f32(2 * kTileW, BN);   // 256 x BN over the pair
            const uint32_t sfa = tmem_base + kSfaCol;
            const int me = warp - kMmaWarp;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int seq = 0;
            bool ok = true;
            int pi = 0;
            for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
                pi = next_problem(S.prob, a.count, pi, tile);
                const TcProb& P = S.prob[pi];
                const int KB = P.K / kBlockK + (P.K % kBlockK ? 1 : 0);
                if (!tc::mbar_wait(&S.tmem_empty[acc], acc_phase ^ 1, abort_flag, kWaitLimit)) { fail(4); break; }
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccCols;
                for (int kb = 0; kb < KB; ++kb, ++seq) {
                    if (seq % kIssuersTc == me) {
                        if (!tc::mbar_wait(&S.full_a[stage], phase, abort_flag, kWaitLimit) ||
                            !tc::mbar_wait(&S.full_b[stage], phase, abort_flag, kWaitLimit)) { fail(8); ok = false; break; }
                        tc::tc_fence_after();
                        const uint32_t a_tm = tmem_base + kACol0 + (uint32_t)stage * kAStageCols;
                        const uint32_t b0 = tc::smem_u32(sB + (size_t)stage * kBStageMax);
                        const uint64_t bd0 = tc::sdesc_sw128_kmajor(b0);
                        const uint64_t bd1 = tc::sdesc_sw128_kmajor(b0 + plane_bytes);
                        const uint64_t bd2 = tc::sdesc_sw128_kmajor(b0 + 2 * plane_bytes);
                        // a stage past K/128 groups holds zero codes in its second half
                        const int steps = (kb * kBlockK + kBlockK <= P.K) ? 4 : 2;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {   // +32 bytes (64 e2m1) per step
                            if (k >= steps) break;
                            const uint32_t ak = a_tm + 8u * (uint32_t)k;   // 64 e2m1 per step
                            pair_umma_mxf4_tmem_a(d_tmem, ak, bd0 + 2 * k, idesc, sfa, tmem_base + kSfbCol0, 1u);
                            pair_umma_mxf4_tmem_a(d_tmem, ak, bd1 + 2 * k, idesc, sfa,
                                                  tmem_base + kSfbCol0 + kSfCols, 1u);
                            pair_umma_mxf4_tmem_a(d_tmem, ak, bd2 + 2 * k, idesc, sfa,
                                                  tmem_base + kSfbCol0 + 2 * kSfCols, 1u);
                        }
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
            tc::mbar_wait_drain(&S.mma_done[me], 0, kWaitLimit / 8);
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
            int pi = 0;
            for (int tile = pair; ok && tile < a.total_tiles; tile += n_pairs) {
                pi = next_problem(S.prob, a.count, pi, tile);
                const TcProb& P = S.prob[pi];
                const int KB = P.K / kBlockK + (P.K % kBlockK ? 1 : 0);
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
        const int q = warp & 3;                // TMEM lane quarter
        const int r = q * 32 + lane;           // TMEM lane = weight row within the tile
        const int half = warp >> 2;            // which half of the accumulator's columns
        int acc = 0;
        uint32_t acc_phase = 0, stage_phase = 0;
        int pi = 0;
        for (int tile = pair; tile < a.total_tiles; tile += n_pairs) {
            pi = next_problem(S.prob, a.count, pi, tile);
            const TcProb& P = S.prob[pi];
            const int local = tile - P.tile0;
            const int wt = local / P.n_act_tiles, at = local % P.n_act_tiles;
            const int n = wt * (2 * kTileW) + (int)rank * kTileW + r;
            // stage the tile's per-column factors (w_scale * act_scale[m] and
            // row_sum[m]) in shared memory while the accumulator fills
            const int m_base = at * BN;
            {
                const bool tiled = (a.tiled[pi >> 5] >> (pi & 31)) & 1u;
                const float w_scale = *reinterpret_cast<const float*>(
                    P.w + (tiled ? tiled_scale_offset(P.N, P.K) : (size_t)P.N * (P.K / 4)));
                float* sc_col = S.sc_col[acc];
                float* rs_col = S.rs_col[acc];
                for (int j = tid; j < BN; j += kEpiWarps * 32) {
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
            // this warp's BN/2 columns, 16 at a time: the load of the next
            // slice overlaps the stores of this one; the accumulator is released
            // as soon as its last slice is in registers
            const int c_base = half * (BN / 2);
            const uint32_t d_addr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * kAccCols + (uint32_t)c_base;
            const int H = BN / 32;   // 16-column slices per warp
            auto store_slice = [&](int h, const uint32_t (&v)[16]) {
                if (n >= N) return;
                const int m0 = c_base + 16 * h;   // first tile column of the slice
                const int rows = min(16, M - (m_base + m0));
                float* yp = y_col + (size_t)(m_base + m0) * N;
                float o[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    // 2 * D is the integer dot, exact; so is dot - row_sum
                    // (|.| < 2^24): the float of (dot - row_sum) without any
                    // conversion instruction
                    const float dr = __fsub_rn(__fmul_rn(__uint_as_float(v[j]), 2.0f), rs_col[m0 + j]);
                    o[j] = __fmul_rn(dr, sc_col[m0 + j]);
                }
                if (rows >= 16) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) yp[(size_t)j * N] = o[j];
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < rows) yp[(size_t)j * N] = o[j];
                }
            };
            auto release = [&]() {
                // every slice is in registers: zero this warp's columns of the
                // accumulator for the tile after next, then hand them back
                for (int h2 = 0; h2 < H; ++h2) tc::tmem_st_zero_32x32b_x16(d_addr + 16u * h2);
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(tc::smem_in_rank(&S.tmem_empty[acc], 0));   // the leader's barrier
            };
            uint32_t va[16], vb[16];
            tc::tmem_ld_32x32b_x16(d_addr, va);
            tc::tmem_ld_wait();
            if (H == 1) release();
            for (int h = 0; h < H; h += 2) {
                if (h + 1 < H) tc::tmem_ld_32x32b_x16(d_addr + 16u * (h + 1), vb);
                store_slice(h, va);
                if (h + 1 < H) {
                    tc::tmem_ld_wait();
                    if (h + 2 == H) release();
                    if (h + 2 < H) tc::tmem_ld_32x32b_x16(d_addr + 16u * (h + 2), va);
                    store_slice(h + 1, vb);
                    if (h + 2 < H) {
                        tc::tmem_ld_wait();
                        if (h + 3 == H) release();
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
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};   // 64 f16 = one 128-byte swizzle row
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
