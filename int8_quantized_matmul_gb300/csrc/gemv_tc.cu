// Decode GEMV for the I2_S ternary x INT8 matmul (M <= 16 activation rows) on
// the 5th-generation tensor cores ("ggml-cpu: ternary I2_S matmul kernel",
// sections Arithmetic and Kernels; "ggml: additive INT8/ternary types ...",
// "Arithmetic is exact where it can be").
//
// The op is bound by weight bandwidth: each 2-bit weight is read from HBM
// once and used for all M activation rows. What limits a tensor-core GEMV here
// is turning the codes into MMA operands and issuing the MMAs, so the codes
// are expanded in registers and written straight into tensor memory
// (tcgen05.st), where the MMA reads its A operand, and each MMA covers as many
// codes as the hardware allows.
//
// Arithmetic (exact): tcgen05.mma kind::mxf4 (packed e2m1 operands, K = 64 per
// instruction) with every block scale equal to 1 and f32 accumulation.
//   * A: a code c in {0,1,2} read as an e2m1 nibble is c/2, so
//     packed & 0x33333333 and (packed >> 2) & 0x33333333 yield eight operands
//     each.
//   * B: each quantized activation q in [-127,127] is written as three digits
//     q = d0 + 8*d1 + 64*d2 (d0, d1 in [-4,3], d2 in [-2,2]), each an exact
//     e2m1 value, one operand row per digit: row j*M' + m (M' = 8 or 16), so
//     MMA N = 32 (M' = 8, with 8 unused rows) or 48. Rows of absent
//     activation rows hold stale values; their D columns are never read.
//   * D column j*M' + m holds sum_k (c/2)*d_j: a multiple of 1/2 below 2^23,
//     exact in f32. dot = 2*D_0 + 16*D_1 + 128*D_2, formed in integers.
// The epilogue is the pages' y = (float)(dot - row_sum) * (w_scale*act_scale).
//
// K order: TMEM column 16g + 2w + t of a stage holds, for 128-group g, the
// eight codes of group word w (bytes 4w..4w+3) at shifts (0,4) (t = 0) or
// (2,6) (t = 1), in that nibble order per byte; the quantizer writes the B
// rows in the same order (quant.cu, k_quant_rows_tc4), and the dot product
// does not depend on the order.
//
// Roles (persistent CTAs, contiguous ranges of work units, 128 weight rows per
// tile, 512 K positions per pipeline stage):
//   warp 8     weight producer: one TMA box per stage (128 rows x 128 packed
//              bytes, 128-byte swizzle, so the converters' 16-byte row reads
//              are free of bank conflicts) into a 3-stage shared ring. Each
//              weight matrix has its own tensor map, written into the
//              workspace by the quantization launch from a template;
//   warps 0-3  converters: thread = weight row = TMEM lane reads its row's 128
//              bytes, expands them and tcgen05.st's them into a 2-stage TMEM
//              ring of A operands (64 columns per stage);
//   warp 10    TMA producer of the B rows of each stage;
//   warp 9     TMEM allocation and the MMA issuer (8 MMAs per stage);
//   warps 4-7  epilogue (TMEM lanes 32(w-4) .. +31 = weight rows).
// Every wait is bounded (~1 s) and reports a timeout in the status word. The
// MMA thread spins on its barriers; the other roles suspend while they wait,
// leaving the issue slots to the converters and the MMA thread.

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "quant_tc.cuh"
#include "tc.cuh"

namespace i2s {

namespace {

constexpr int kThreadsGv = 384;
constexpr int kCvtWarpsGv = 4;
constexpr int kEpiWarp0 = 4;
constexpr int kWProdWarp = 8;
constexpr int kMmaWarpGv = 9;
constexpr int kBProdWarp = 10;
constexpr int kMmaWarpGv2 = 11;        // the second MMA issuer
constexpr int kIssuersGv = 2;
constexpr int kKB = 512;               // K positions per pipeline stage (128 packed bytes per row)
constexpr int kStageBytes = kKB / 4;
constexpr int kWStages = 3;            // weight ring depth (16 KB stages, 128-byte swizzle)
constexpr int kStagesGv = 2;           // TMEM A ring depth (stages of 64 columns)
constexpr int kBRingBytes = 36 * 1024; // activation ring: 4 stages of 8 KB (M' = 8) or 3 of 12 KB (M' = 16)
constexpr int kBStagesMax = 8;
constexpr int kTileRows = 128;
constexpr int kWStageBytes = kTileRows * kStageBytes;
static_assert(kWStageBytes == kTiledBlockBytes && kStageBytes == kTiledRowBytes, "a weight stage is one block of tiled weights");
constexpr uint32_t kTmemColsGv = 256;
// TMEM columns: A stages 0..127, accumulator 0 at 128 (up to 48 columns),
// block scales 176..191, accumulator 1 at 192.
constexpr uint32_t kDCol0 = 128, kDCol1 = 192;
constexpr uint32_t kSfCol = 176;
constexpr uint32_t kSfOnes = 0x7F7F7F7Fu;   // ue8m0 1.0 in every byte
constexpr long long kWaitLimitGv = 2000000000LL;

struct SmemGv {
    uint64_t full_w[kWStages];          // a weight stage is in shared memory
    uint64_t empty_w[kWStages];         // every converter is done with a stage
    uint64_t full_a[kStagesGv];
    uint64_t empty[kStagesGv];          // TMEM A stage free (MMA done)
    uint64_t full_b[kBStagesMax];
    uint64_t empty_b[kBStagesMax];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done[kIssuersGv];
    uint64_t epi_sync;                  // the 4 epilogue warps finished their partial-dot atomics
    uint64_t epi_bcast;                 // the split-K finalize decision is published
    uint64_t never;                     // test only: a barrier nothing arrives on
    uint32_t tmem_base;
    int abort;
    int final_flag;
};

constexpr size_t kSProbBytes = 80;      // shared copy of one problem-table entry (SProb)
constexpr size_t kSmemGvUsed = 1024 + (size_t)kBRingBytes + (size_t)kWStages * kWStageBytes + sizeof(SmemGv) + 16 +
                               (size_t)kMaxGroup * kSProbBytes;
// At least 80 KB so that at most two CTAs share an SM: each holds 256 of the
// 512 TMEM columns for its whole life.
constexpr size_t kSmemGvBytes = kSmemGvUsed > 80 * 1024 ? kSmemGvUsed : 80 * 1024;

// Problem table copied into shared memory at kernel start (parameter-space
// reads through a generic pointer are slow once the table misses the constant
// cache, and every role resolves a problem at each segment).
struct SProb {
    const uint8_t* w;
    const float* act_scale;
    const int32_t* row_sum;
    float* y;
    int N, K, map, unit0, chunks, dot_off, ticket_off, pidx;
    int row0;   // first row of the activation operand in its map (fused launch: stacked operands)
    int act;    // activation index (fused launch: its ready counter)
    int tiled;  // the weights are in the tiled layout (i2s_tile_weights)
};

constexpr int kChunkStages = kGemvChunkPositions / kKB;   // 3 stages per work unit

// A segment: the consecutive K chunks of one row tile that fall inside this
// CTA's contiguous range of work units [u, u_hi). Every role walks the same
// segments in the same order.
struct Seg {
    const uint8_t* w;
    const float* act_scale;
    const int32_t* row_sum;
    float* y;
    int N, K, map, pidx, sidx, n0, tile, st_lo, st_hi, c_lo, c_hi, chunks, dot_off, ticket_off, units, row0, act, tiled;
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
    g.sidx = lo;
    g.w = P.w;
    g.act_scale = P.act_scale;
    g.row_sum = P.row_sum;
    g.y = P.y;
    g.N = P.N;
    g.K = P.K;
    g.map = P.map;
    g.pidx = P.pidx;
    g.row0 = P.row0;
    g.act = P.act;
    g.tiled = P.tiled;
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

// The segment after g, starting at unit u (< u_hi when live). A segment that
// does not reach u_hi ends at its tile's last chunk, so the next one starts at
// chunk 0 of the following tile (or of the next problem's first tile): a step
// with no search and no division, unlike seg_at.
__device__ __forceinline__ Seg seg_next(const SProb* sp, const Seg& g, int u, int u_hi) {
    Seg n;
    n.live = u < u_hi;
    if (!n.live) return n;
    n.sidx = g.sidx;
    n.tile = g.tile + 1;
    if (n.tile >= (sp[n.sidx].N + kTileRows - 1) / kTileRows) {
        ++n.sidx;
        n.tile = 0;
    }
    const SProb& P = sp[n.sidx];
    n.w = P.w;
    n.act_scale = P.act_scale;
    n.row_sum = P.row_sum;
    n.y = P.y;
    n.N = P.N;
    n.K = P.K;
    n.map = P.map;
    n.pidx = P.pidx;
    n.row0 = P.row0;
    n.act = P.act;
    n.tiled = P.tiled;
    n.chunks = P.chunks;
    n.dot_off = P.dot_off;
    n.ticket_off = P.ticket_off;
    n.c_lo = 0;
    n.c_hi = min(P.chunks, u_hi - u);
    n.units = n.c_hi;
    n.n0 = n.tile * kTileRows;
    n.st_lo = 0;
    n.st_hi = min((P.K + kKB - 1) / kKB, n.c_hi * kChunkStages);
    return n;
}

// --------------------------------------------------------------------------
// Fused launch: helpers of the prologue and of the waits on it.
// --------------------------------------------------------------------------

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits (bounded, suspending between polls) until *p reaches want.
__device__ __forceinline__ bool wait_flag(const uint32_t* p, uint32_t want, volatile int* abort_flag, long long limit) {
    const long long t0 = clock64();
    while (ld_acquire_u32(p) < want) {
        if (*abort_flag || clock64() - t0 > limit) return false;
        __nanosleep(64);
    }
    return true;
}

// The prologue's quantizer team: every warp but the weight producer (352
// threads), synchronised by named barrier 1.
constexpr int kTeamThreads = kThreadsGv - 32;
__device__ __forceinline__ void team_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kTeamThreads) : "memory"); }

constexpr int kTeamRows = 64;      // rows of one batch (shared-memory slots)
constexpr int kTeamUnits = 2;      // 16-value units per thread kept in registers in the one-pass case

// Shared state of the prologue's quantizer: one batch of up to kTeamRows rows.
struct TeamRows {
    uint32_t amax_bits[kTeamRows];   // max |x| of each row, as float bits (non-negative, so integer max works)
    float inv[kTeamRows];
    int sum[kTeamRows];
    int act[kTeamRows], m[kTeamRows];
    int u0[kTeamRows + 1];           // first 16-value unit of each row in the batch's flattened order
};

// Row of flattened unit j of a batch of n rows (binary search over u0).
__device__ __forceinline__ int team_row_of(const TeamRows& R, int n, int j) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (R.u0[mid] <= j) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void team_load(const GvFusedArgs& a, const TeamRows& R, int r, int j, float4 (&v)[4]) {
    const GvAct& A = a.acts[R.act[r]];
    load_unit(reinterpret_cast<const float4*>(A.x + (size_t)R.m[r] * A.K), j - R.u0[r], v);
}

__device__ __forceinline__ int team_emit(const GvFusedArgs& a, const TeamRows& R, int r, int j, const float4 (&v)[4],
                                         int Mp, const uint32_t* code) {
    const GvAct& A = a.acts[R.act[r]];
    return emit_unit(v, R.inv[r], j - R.u0[r], A.op, (size_t)A.K / 2, Mp, R.m[r], code);
}

// The prologue's share of the row quantization, done by the team (thread t).
// The rows of all activations are laid end to end, each costing K positions;
// this CTA takes the rows whose first position falls in its equal share
// [lo, hi) of the total. Rows are handled in batches, every row of a batch at
// once: each thread loads its 16-value units, folds each row's max |x| into
// shared memory, and after a barrier quantizes with the row's 127/amax,
// writes the e2m1 digit rows and folds the int8 sums. A batch whose units fit
// in registers (kTeamUnits per thread) is read once; a longer row is read
// twice (the second pass from L2). Each row is then published with its scale
// and sum through its activation's ready counter (a release). The CTA that
// owns row 0 of an activation first zeroes the split-K partial dots and
// chunk counters of the problems that read it, so every add to them comes
// after the zeroing.
template <int Mp>
__device__ void fused_quantize(const GvFusedArgs& a, int t, const uint32_t* code, TeamRows& R) {
    const long long C = a.cost_total, G = gridDim.x, b = blockIdx.x;
    const long long lo = (b * C + G - 1) / G, hi = ((b + 1) * C + G - 1) / G;
    if (lo >= hi) return;
    constexpr int kCap = kTeamUnits * kTeamThreads;
    // the last activation starting at or before lo (activations are laid out
    // in order of cost0), and its first row starting at or after lo
    int ai = 0;
    {
        int last = a.n_acts - 1;
        while (ai < last) {
            const int mid = (ai + last + 1) >> 1;
            if (a.acts[mid].cost0 <= lo) ai = mid; else last = mid - 1;
        }
    }
    int m = 0;
    {
        const GvAct& A = a.acts[ai];
        if (lo > A.cost0) m = (int)((lo - A.cost0 + A.K - 1) / A.K);
    }
    while (true) {
        // gather the next batch (the same walk in every team thread): rows
        // starting in [lo, hi), while they fit the registers (a longer row
        // goes alone)
        int n = 0, units = 0;
        while (n < kTeamRows && ai < a.n_acts) {
            const GvAct& A = a.acts[ai];
            if (m >= a.M) { ++ai; m = 0; continue; }
            if (A.cost0 + (long long)m * A.K >= hi) break;
            const int u = A.K / 16;
            if (n > 0 && units + u > kCap) break;
            if (t == 0) {
                R.act[n] = ai;
                R.m[n] = m;
                R.u0[n] = units;
                R.amax_bits[n] = 0u;
                R.sum[n] = 0;
            }
            units += u;
            ++n;
            ++m;
        }
        if (n == 0) break;
        if (t == 0) R.u0[n] = units;
        team_sync();
        // zero the split-K areas of activations whose row 0 is in the batch
        for (int i = 0; i < n; ++i) {
            if (R.m[i] != 0) continue;
            const GvAct& A = a.acts[R.act[i]];
            for (int e = t; e < A.dot_n; e += kTeamThreads) a.dot_base[A.dot_lo + e] = 0;
            for (int e = t; e < A.tk_n; e += kTeamThreads) a.ticket_base[A.tk_lo + e] = 0u;
        }
        if (units <= kCap) {
            // one pass: every load in flight at once, the units kept in registers
            float4 v[kTeamUnits][4];
            int rr[kTeamUnits];
#pragma unroll
            for (int c = 0; c < kTeamUnits; ++c) {
                const int j = t + c * kTeamThreads;
                rr[c] = j < units ? team_row_of(R, n, j) : -1;
                if (rr[c] >= 0) team_load(a, R, rr[c], j, v[c]);
            }
#pragma unroll
            for (int c = 0; c < kTeamUnits; ++c)
                if (rr[c] >= 0) atomicMax(&R.amax_bits[rr[c]], __float_as_uint(unit_amax(v[c])));
            team_sync();
            for (int i = t; i < n; i += kTeamThreads) {
                float scale, inv;
                quant_params(__uint_as_float(R.amax_bits[i]), scale, inv);
                R.inv[i] = inv;
            }
            team_sync();
#pragma unroll
            for (int c = 0; c < kTeamUnits; ++c)
                if (rr[c] >= 0) atomicAdd(&R.sum[rr[c]], team_emit(a, R, rr[c], t + c * kTeamThreads, v[c], Mp, code));
        } else {
            // one row longer than the registers hold: two passes
            for (int j = t; j < units; j += kTeamThreads) {
                float4 v[4];
                team_load(a, R, 0, j, v);
                atomicMax(&R.amax_bits[0], __float_as_uint(unit_amax(v)));
            }
            team_sync();
            if (t == 0) {
                float scale, inv;
                quant_params(__uint_as_float(R.amax_bits[0]), scale, inv);
                R.inv[0] = inv;
            }
            team_sync();
            for (int j = t; j < units; j += kTeamThreads) {
                float4 v[4];
                team_load(a, R, 0, j, v);
                atomicAdd(&R.sum[0], team_emit(a, R, 0, j, v, Mp, code));
            }
        }
        // the digit rows are read by other CTAs' TMA loads (the async proxy)
        asm volatile("fence.proxy.async.global;" ::: "memory");
        team_sync();
        // a fence of the counting thread after the barrier orders every team
        // thread's stores (digit rows, zeroed areas) and its own scale and sum
        // before the count
        for (int i = t; i < n; i += kTeamThreads) {
            const GvAct& A = a.acts[R.act[i]];
            float scale, inv;
            quant_params(__uint_as_float(R.amax_bits[i]), scale, inv);
            A.scale[R.m[i]] = scale;
            A.sum[R.m[i]] = R.sum[i];
            __threadfence();
            atomicAdd(&a.flags[a.count + R.act[i]], 1u);
        }
        team_sync();   // the batch's shared slots are reused by the next batch
    }
}

template <bool kFused, typename Args>
__device__ __forceinline__ const CUtensorMap* act_map(const Args& a, int i) {
    if constexpr (kFused) return &a.kmaps[i];
    else return &a.maps[i];
}

template <int Mp, bool kFused, typename Args>
__global__ void __launch_bounds__(kThreadsGv, 2) k_i2s_gemv_tc(const __grid_constant__ Args a) {
    constexpr int kN = gemv_tc_op_rows(Mp);                 // MMA N: three digit rows per activation row, padded
    constexpr uint32_t kBSub = (uint32_t)kN * 128u;          // one 256-position operand sub-tile (1024-aligned)
    constexpr uint32_t kBStageBytes = 2 * kBSub;             // a stage holds two sub-tiles
    constexpr int kBStages = kBRingBytes / (int)kBStageBytes;
    static_assert(kBStages >= 2 && kBStages <= kBStagesMax, "activation ring depth");
    static_assert(kN % 16 == 0 && kN <= 48, "MMA N");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sB = smem;
    uint8_t* sW = sB + (size_t)kBRingBytes;
    SmemGv& S = *reinterpret_cast<SmemGv*>(sW + (size_t)kWStages * kWStageBytes);
    SProb* sp = reinterpret_cast<SProb*>(reinterpret_cast<uint8_t*>(&S) + ((sizeof(SmemGv) + 15) & ~(size_t)15));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's contiguous share of the work units
    // This CTA's contiguous share of the work units. With two CTAs per SM the
    // first CTA placed on an SM (the first half of the grid) is issued ahead of
    // the second and runs faster, so the host may give it a larger share.
    const int h = (int)gridDim.x / 2;
    const long long w1 = a.share_first, w2 = a.share_second;
    const long long den = (long long)h * w1 + (long long)((int)gridDim.x - h) * w2;
    auto bound = [&](int b) {
        const long long num = b <= h ? (long long)b * w1 : (long long)h * w1 + (long long)(b - h) * w2;
        return (int)(num * a.total_tiles / den);
    };
    const int u_begin = bound((int)blockIdx.x);
    const int u_end = bound((int)blockIdx.x + 1);

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
        int map = P.map, row0 = 0;
        if constexpr (kFused) {   // stacked operands: the activation's class map and first row
            map = a.acts[P.map].kclass;
            row0 = a.acts[P.map].row0;
        }
        const int pi = p_first + i;
        sp[i] = SProb{P.w, P.act_scale, P.row_sum, P.y, P.N, P.K, map, P.tile0, P.chunks, P.dot_off, P.ticket_off,
                      pi, row0, P.map, (int)((a.tiled[pi >> 5] >> (pi & 31)) & 1u)};
    }
    uint32_t* s_code = nullptr;
    TeamRows* s_rows = nullptr;
    if constexpr (kFused) {   // the digit table and row slots of the prologue's quantizer
        __shared__ uint32_t s_code_tab[255];
        __shared__ TeamRows s_rows_team;
        if (tid < 255) s_code_tab[tid] = digit_code(tid - 127);
        s_code = s_code_tab;
        s_rows = &s_rows_team;
    }
    if (tid == 0) {
        for (int s = 0; s < kWStages; ++s) {
            tc::mbar_init(&S.full_w[s], 1);                   // the producer's arrive.expect_tx (+ TMA bytes)
            tc::mbar_init(&S.empty_w[s], kCvtWarpsGv * 32);
        }
        for (int s = 0; s < kStagesGv; ++s) {
            tc::mbar_init(&S.full_a[s], kCvtWarpsGv * 32);
            tc::mbar_init(&S.empty[s], kIssuersGv);
        }
        for (int s = 0; s < kBStagesMax; ++s) {
            tc::mbar_init(&S.full_b[s], 1);
            tc::mbar_init(&S.empty_b[s], kIssuersGv);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&S.tmem_full[b], kIssuersGv);
            tc::mbar_init(&S.tmem_empty[b], 4 * 32);
        }
        for (int i = 0; i < kIssuersGv; ++i) tc::mbar_init(&S.mma_done[i], 1);
        tc::mbar_init(&S.epi_sync, 4 * 32);
        tc::mbar_init(&S.epi_bcast, 1);
        tc::mbar_init(&S.never, 1);
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
    if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // both accumulators start at zero (every MMA accumulates)
        const uint32_t lane_off = (uint32_t)((warp - kEpiWarp0) * 32) << 16;
        tc::tmem_st_zero_32x32b_x32(tmem_base + lane_off + kDCol0);
        tc::tmem_st_zero_32x32b_x32(tmem_base + lane_off + kDCol1);
        if (kN > 32) {
            tc::tmem_st_zero_32x32b_x16(tmem_base + lane_off + kDCol0 + 32);
            tc::tmem_st_zero_32x32b_x16(tmem_base + lane_off + kDCol1 + 32);
        }
        tc::tmem_st_wait();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    // everything above touched only parameters, shared memory and TMEM; the
    // workspace (operands, weight maps, partial sums) is read from here on,
    // after the quantization launch before this one has completed
    pdl_wait();
    if constexpr (kFused) {
        // Prologue of the fused launch: the activation producer's lanes write
        // the weight maps (map i by CTA i mod grid) and flag each; every warp
        // but the weight producer then quantizes this CTA's share of the
        // activation rows. The weight producer starts streaming at once,
        // waiting only for the flag of the map it needs; the activation
        // producer and the epilogue wait for the ready counter of their
        // activation.
        if (warp == kBProdWarp) {
            for (int i = (int)blockIdx.x + (int)gridDim.x * lane; i < a.count; i += (int)gridDim.x * 32) {
                const TcProb& P = a.p[i];
                write_weight_map(a.wtmpl, a.wmaps + i, P.w, P.N, P.K);
                st_release_u32(a.flags + i, 1u);
            }
        }
        if (warp != kWProdWarp)   // the team: thread index without the weight producer's warp
            fused_quantize<Mp>(a, warp < kWProdWarp ? tid : tid - 32, s_code, *s_rows);
    }

    int ucur = u_begin;   // each role advances its own copy of the unit cursor
    auto next_seg = [&](const Seg& g) { ucur += g.units; return seg_next(sp, g, ucur, u_end); };

    if (warp == kWProdWarp) {
        // --------------------------------------------------- weight producer
        // One TMA box per stage: 128 rows x 128 packed bytes of the tile, from
        // the problem's weight map (written by the quantization launch; rows
        // past N and bytes past K/4 are zero-filled), into a 3-stage ring. On
        // tiled weights the stage is one 16 KB block, already in the ring's
        // layout: one bulk copy.
        if (lane == 0) {
            int ws = 0;
            uint32_t wphase = 0;
            bool pending[kWStages] = {};
            uint32_t pending_phase[kWStages] = {};
            bool ok = true;
            int cur_p = -1;
            for (Seg g = seg_at(sp, n_sp, ucur, u_end); ok && g.live; g = next_seg(g)) {
                const CUtensorMap* map = a.wmaps + g.pidx;
                if (g.pidx != cur_p) {   // first use of this map: order it after the writer's release
                    if constexpr (kFused) {
                        if (!wait_flag(a.flags + g.pidx, 1u, abort_flag, kWaitLimitGv)) { fail(4096); ok = false; break; }
                    }
                    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
                    cur_p = g.pidx;
                }
                const int row_bytes = g.K / 4;
                const int end = min(g.st_hi * kStageBytes, row_bytes);
                for (int off = g.st_lo * kStageBytes; off < end; off += kStageBytes) {
                    if (!tc::mbar_wait_idle(&S.empty_w[ws], wphase ^ 1, abort_flag, kWaitLimitGv)) { fail(1024); ok = false; break; }
                    tc::mbar_arrive_expect_tx(&S.full_w[ws], kWStageBytes);
                    if (g.tiled) {   // block (tile, stage) of the tiled weights
                        const size_t blk = (size_t)(g.n0 / kTiledRows) * tiled_col_blocks(g.K) + off / kTiledRowBytes;
                        tc::bulk_load(sW + (size_t)ws * kWStageBytes, g.w + blk * kTiledBlockBytes, kWStageBytes,
                                      &S.full_w[ws]);
                    } else {
                        tc::tma_load_2d(sW + (size_t)ws * kWStageBytes, map, off, g.n0, &S.full_w[ws]);
                    }
                    pending[ws] = true;
                    pending_phase[ws] = wphase;
                    if (++ws == kWStages) { ws = 0; wphase ^= 1; }
                }
            }
            if (!ok)
                for (int s2 = 0; s2 < kWStages; ++s2)
                    if (pending[s2]) tc::mbar_wait_drain(&S.full_w[s2], pending_phase[s2], kWaitLimitGv / 8);
        }
    } else if (warp < kCvtWarpsGv) {
        // ---------------------------------------------------------- converters
        // thread = weight row = TMEM lane. First the block scales (all 1.0),
        // then per stage: read the row's 128 (or fewer) bytes from the weight
        // ring, expand, tcgen05.st into the TMEM ring; wait for the stage's
        // activation operand to land and publish the stage, so that one
        // barrier tells the MMA thread both are ready.
        const int r = tid;
        const uint32_t lane_base = tmem_base + ((uint32_t)(warp * 32) << 16);
        {
            uint32_t ones[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) ones[i] = kSfOnes;
            tc::tmem_st_32x32b_x16(lane_base + kSfCol, ones);
        }
        int ws = 0, stage = 0, bstage = 0;
        uint32_t wphase = 0, phase = 0, bphase = 0;
        bool ok = true;
        for (Seg g = seg_at(sp, n_sp, ucur, u_end); ok && g.live; g = next_seg(g)) {
            const int row_bytes = g.K / 4;
            const int end = min(g.st_hi * kStageBytes, row_bytes);
            for (int off = g.st_lo * kStageBytes; off < end; off += kStageBytes) {
                const int bytes = min(kStageBytes, end - off);
                if (!tc::mbar_wait_idle(&S.full_w[ws], wphase, abort_flag, kWaitLimitGv)) { fail(32); ok = false; break; }
                const uint8_t* wst = sW + (size_t)ws * kWStageBytes;
                uint4 c[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {   // rows past N and bytes past K/4 arrive as zeros
                    c[i] = make_uint4(0, 0, 0, 0);
                    if (16 * i < bytes) c[i] = *reinterpret_cast<const uint4*>(wst + tc::sw128_offset(r, i));
                }
                // the loads complete while this thread waits for its TMEM stage
                if (!tc::mbar_wait_idle(&S.empty[stage], phase ^ 1, abort_flag, kWaitLimitGv)) { fail(32); ok = false; break; }
                tc::mbar_arrive(&S.empty_w[ws]);   // this row's bytes of the ring stage are read
                if (++ws == kWStages) { ws = 0; wphase ^= 1; }
                tc::tc_fence_after();
                const uint32_t col0 = lane_base + (uint32_t)(stage * 64);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (half == 1 && bytes <= 64) break;
                    uint32_t v[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 q = c[4 * half + i];
                        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            v[8 * i + 2 * j] = w4[j] & 0x33333333u;
                            v[8 * i + 2 * j + 1] = (w4[j] >> 2) & 0x33333333u;
                        }
                    }
                    tc::tmem_st_32x32b_x32(col0 + 32u * half, v);
                }
                tc::tmem_st_wait();
                // the stage's activation operand must have landed before publishing
                if (!tc::mbar_wait_idle(&S.full_b[bstage], bphase, abort_flag, kWaitLimitGv)) { fail(32); ok = false; break; }
                tc::tc_fence_before();
                tc::mbar_arrive(&S.full_a[stage]);
                if (++stage == kStagesGv) { stage = 0; phase ^= 1; }
                if (++bstage == kBStages) { bstage = 0; bphase ^= 1; }
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
                if (g0.live) tc::tma_prefetch_desc(act_map<kFused>(a, g0.map));
            }
            int cur_act = -1;
            for (Seg g = seg_at(sp, n_sp, ucur, u_end); ok && g.live; g = next_seg(g)) {
                const CUtensorMap* map = act_map<kFused>(a, g.map);
                {   // fetch the next segment's descriptor while this one streams
                    const Seg gn = seg_next(sp, g, ucur + g.units, u_end);
                    if (gn.live && gn.map != g.map) tc::tma_prefetch_desc(act_map<kFused>(a, gn.map));
                }
                if constexpr (kFused) {   // the activation's rows are quantized by the prologue
                    if (g.act != cur_act) {
                        if (!wait_flag(a.flags + a.count + g.act, (uint32_t)a.M, abort_flag, kWaitLimitGv)) {
                            fail(8192);
                            ok = false;
                            break;
                        }
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        cur_act = g.act;
                    }
                }
                for (int kb = g.st_lo; kb < g.st_hi; ++kb) {
                    const bool two = kb * kKB + kKB / 2 < g.K;   // the stage reaches its second 256 positions
                    if (!tc::mbar_wait_idle(&S.empty_b[stage], phase ^ 1, abort_flag, kWaitLimitGv)) { fail(64); ok = false; break; }
                    tc::mbar_arrive_expect_tx(&S.full_b[stage], two ? kBStageBytes : kBSub);
                    uint8_t* dst = sB + (size_t)stage * kBStageBytes;
                    tc::tma_load_2d(dst, map, kb * (kKB / 2), g.row0, &S.full_b[stage]);
                    if (two) tc::tma_load_2d(dst + kBSub, map, kb * (kKB / 2) + 128, g.row0, &S.full_b[stage]);
                    pending[stage] = true;
                    pending_phase[stage] = phase;
                    if (++stage == kBStages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok)
                for (int s = 0; s < kBStages; ++s)
                    if (pending[s]) tc::mbar_wait_drain(&S.full_b[s], pending_phase[s], kWaitLimitGv / 8);
        }
    } else if (warp == kMmaWarpGv || warp == kMmaWarpGv2) {
        // ---------------------------------------------------------- MMA issue
        // One thread needs well over 100 SM cycles to issue a tcgen05.mma, so
        // two warps issue every stage, each the MMAs of one 256-position half,
        // both into the segment's accumulator. Every MMA accumulates; the
        // epilogue zeroes an accumulator after reading it, and the sums are
        // exact integers, so the order in which the two streams land does not
        // matter. A stage is free again once both issuers have committed.
        // One wait per stage: a complete full_a implies the activation operand
        // has landed too (the converters waited for it before arriving). The
        // stage's MMAs (two per 128-position group) are unrolled.
        if (lane == 0) {
            const int me = warp == kMmaWarpGv ? 0 : 1;
            constexpr uint32_t idesc = tc::idesc_mxf4_f32(kTileRows, kN);
            const uint32_t sfa = tmem_base + kSfCol, sfb = tmem_base + kSfCol + 4;
            int stage = 0, bstage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (Seg g = seg_at(sp, n_sp, ucur, u_end); ok && g.live; g = next_seg(g)) {
                if (!tc::mbar_wait_idle(&S.tmem_empty[acc], acc_phase ^ 1, abort_flag, kWaitLimitGv)) { fail(128); break; }
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (acc ? kDCol1 : kDCol0);
                for (int kb = g.st_lo; kb < g.st_hi; ++kb) {
                    const int n_mma = 2 * min(4, (g.K - kb * kKB) / 128);   // 64 positions per MMA
                    if (!tc::mbar_wait_idle(&S.full_a[stage], phase, abort_flag, kWaitLimitGv)) { fail(256); ok = false; break; }
                    tc::tc_fence_after();
                    // issuer `me` takes the stage's 256-position half `me`: MMAs 4me..4me+3
                    const uint32_t b0 = tc::smem_u32(sB + (size_t)bstage * kBStageBytes);
                    const uint64_t bd = tc::sdesc_sw128_kmajor(b0 + (me ? kBSub : 0u));
                    const uint32_t a0 = tmem_base + (uint32_t)(stage * 64) + 32u * (uint32_t)me;
                    if (n_mma == 8) {   // full stage: straight-line issue
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc::umma_mxf4_tmem_a(d_tmem, a0 + 8u * k, bd + 2 * k, idesc, sfa, sfb, 1u);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (4 * me + k < n_mma) tc::umma_mxf4_tmem_a(d_tmem, a0 + 8u * k, bd + 2 * k, idesc, sfa, sfb, 1u);
                    }
                    tc::umma_commit(&S.empty[stage]);      // one arrival from each issuer
                    tc::umma_commit(&S.empty_b[bstage]);
                    if (++stage == kStagesGv) { stage = 0; phase ^= 1; }
                    if (++bstage == kBStages) bstage = 0;
                }
                if (!ok) break;
                tc::umma_commit(&S.tmem_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            tc::umma_commit(&S.mma_done[me]);
            tc::mbar_wait_drain(&S.mma_done[me], 0, kWaitLimitGv / 8);
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ------------------------------------------------------------ epilogue
        // A segment that covers all K chunks of its tile writes y directly.
        // Otherwise its exact int32 partial dots are added to the workspace;
        // the segment whose chunks complete the tile's count applies the
        // epilogue to the summed dots (integer addition is order-independent)
        // and returns the tile's partial dots and ticket to zero, so a launch
        // leaves the split-K state as it found it (a run may be repeated
        // without a new quantization).
        const int q = warp - kEpiWarp0;   // TMEM lane quarter
        const int r = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0, sync_phase = 0;
        int cur_act = -1;
        for (Seg g = seg_at(sp, n_sp, ucur, u_end); g.live; g = next_seg(g)) {
            const int n = g.n0 + r;
            if constexpr (kFused) {   // row scales and sums, and the zeroed partials, come from the prologue
                if (g.act != cur_act) {
                    if (!wait_flag(a.flags + a.count + g.act, (uint32_t)a.M, abort_flag, kWaitLimitGv)) { fail(8192); break; }
                    cur_act = g.act;
                }
            }
            if constexpr (!kFused) {
                if (a.test_stall_cycles > 0) {
                    // test only: a bounded wait that nothing ends, so the
                    // launch takes its give-up path with its MMAs and copies in
                    // flight (the status word records the timeout)
                    tc::mbar_wait(&S.never, 0, abort_flag, a.test_stall_cycles);
                    fail(512);
                    break;
                }
            }
            if (!tc::mbar_wait(&S.tmem_full[acc], acc_phase, abort_flag, kWaitLimitGv)) { fail(512); break; }
            tc::tc_fence_after();
            const uint32_t dcol = tmem_base + ((uint32_t)(q * 32) << 16) + (acc ? kDCol1 : kDCol0);
            uint32_t v[48];
            tc::tmem_ld_32x32b_x32(dcol, *reinterpret_cast<uint32_t (*)[32]>(&v[0]));
            if (kN > 32) tc::tmem_ld_32x32b_x16(dcol + 32, *reinterpret_cast<uint32_t (*)[16]>(&v[32]));
            tc::tmem_ld_wait();
            // zero the accumulator for the segment after next, then hand it back
            tc::tmem_st_zero_32x32b_x32(dcol);
            if (kN > 32) tc::tmem_st_zero_32x32b_x16(dcol + 32);
            tc::tmem_st_wait();
            tc::tc_fence_before();
            tc::mbar_arrive(&S.tmem_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            int dot[Mp];
#pragma unroll
            for (int m = 0; m < Mp; ++m) {
                // 2*D_j is an exact integer; dot = sum_j 8^j * 2*D_j
                const int d0 = __float2int_rn(__fmul_rn(__uint_as_float(v[m]), 2.0f));
                const int d1 = __float2int_rn(__fmul_rn(__uint_as_float(v[Mp + m]), 2.0f));
                const int d2 = __float2int_rn(__fmul_rn(__uint_as_float(v[2 * Mp + m]), 2.0f));
                dot[m] = d0 + 8 * d1 + 64 * d2;
            }
            bool write = g.c_lo == 0 && g.c_hi == g.chunks;
            if (!write) {
                int32_t* part = a.dot_base + g.dot_off;
                if (n < g.N) {
#pragma unroll
                    for (int m = 0; m < Mp; ++m)
                        if (m < a.M) atomicAdd(&part[(size_t)m * g.N + n], dot[m]);
                }
                __threadfence();
                tc::mbar_arrive(&S.epi_sync);
                if (!tc::mbar_wait_idle(&S.epi_sync, sync_phase, abort_flag, kWaitLimitGv)) { fail(2048); break; }
                if (r == 0) {
                    __threadfence();
                    unsigned* ticket = &a.ticket_base[g.ticket_off + g.tile];
                    const unsigned prev = atomicAdd(ticket, (unsigned)g.units);
                    const bool last = prev + (unsigned)g.units == (unsigned)g.chunks;
                    // every other segment of the tile has counted itself: the
                    // ticket starts the next launch on this workspace at zero
                    if (last) *ticket = 0u;
                    S.final_flag = last;
                    tc::mbar_arrive(&S.epi_bcast);
                }
                if (!tc::mbar_wait_idle(&S.epi_bcast, sync_phase, abort_flag, kWaitLimitGv)) { fail(2048); break; }
                sync_phase ^= 1;
                write = S.final_flag != 0;
                if (write) {
                    __threadfence();
                    if (n < g.N) {   // read the summed dots and leave zeros for the next launch
#pragma unroll
                        for (int m = 0; m < Mp; ++m)
                            if (m < a.M) {
                                dot[m] = __ldcg(&part[(size_t)m * g.N + n]);
                                part[(size_t)m * g.N + n] = 0;
                            }
                    }
                }
            }
            if (write && n < g.N) {
                const float w_scale = *reinterpret_cast<const float*>(
                    g.w + (g.tiled ? tiled_scale_offset(g.N, g.K) : (size_t)g.N * (g.K / 4)));
#pragma unroll
                for (int m = 0; m < Mp; ++m) {
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
    if constexpr (kFused) {
        // The last CTA to finish clears the flags and counters for the next
        // launch on this workspace (every CTA has read its last flag by now).
        if (tid == 0) {
            __threadfence();
            uint32_t* done = a.flags + a.count + a.n_acts;
            if (atomicAdd(done, 1u) == gridDim.x - 1) {
                __threadfence();
                for (int i = 0; i < a.count + a.n_acts; ++i) a.flags[i] = 0u;
                __threadfence();
                *done = 0u;
            }
        }
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
        e = cudaFuncSetAttribute(k_i2s_gemv_tc<8, false, TcArgs>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemGvBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_i2s_gemv_tc<16, false, TcArgs>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemGvBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    // a programmatic dependent of the quantization launch before it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreadsGv, 1, 1);
    cfg.dynamicSmemBytes = kSmemGvBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.BN == 8) return cudaLaunchKernelEx(&cfg, k_i2s_gemv_tc<8, false, TcArgs>, a);
    return cudaLaunchKernelEx(&cfg, k_i2s_gemv_tc<16, false, TcArgs>, a);
}

cudaError_t launch_gemv_fused(const GvFusedArgs& a, int grid, cudaStream_t s) {
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(k_i2s_gemv_tc<8, true, GvFusedArgs>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemGvBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_i2s_gemv_tc<16, true, GvFusedArgs>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemGvBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    // a programmatic dependent of the launch before it (which may produce x
    // or use this workspace): the prologue starts after pdl_wait
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreadsGv, 1, 1);
    cfg.dynamicSmemBytes = kSmemGvBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.BN == 8) return cudaLaunchKernelEx(&cfg, k_i2s_gemv_tc<8, true, GvFusedArgs>, a);
    return cudaLaunchKernelEx(&cfg, k_i2s_gemv_tc<16, true, GvFusedArgs>, a);
}

}  // namespace i2s
