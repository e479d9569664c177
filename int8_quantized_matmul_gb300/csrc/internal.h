// Host-side declarations shared by the translation units of libi2s.so.
// Not part of the public ABI (include/i2s.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace i2s {

constexpr int kMaxGroup = 256;   // same value as I2S_MAX_GROUP

// Tiled I2_S weights (i2s_tile_weights): blocks of 128 rows x 128 bytes (512
// positions), each the shared-memory image of one 128-byte-swizzled TMA tile
// of the weights, row blocks padded to an even count (a CTA pair's 256 rows),
// the I2_S trailer after the blocks.
constexpr int kTiledRows = 128;
constexpr int kTiledRowBytes = 128;
constexpr int kTiledBlockBytes = kTiledRows * kTiledRowBytes;   // 16384
__host__ __device__ __forceinline__ long long tiled_row_blocks(long long N) { return 2 * ((N + 255) / 256); }
__host__ __device__ __forceinline__ long long tiled_col_blocks(long long K) { return (K + 511) / 512; }
__host__ __device__ __forceinline__ size_t tiled_scale_offset(long long N, long long K) {
    return (size_t)(tiled_row_blocks(N) * tiled_col_blocks(K)) * kTiledBlockBytes;
}
// Bit i of a launch's tiled mask: problem i's weights are in the tiled layout.
constexpr int kTiledMaskWords = kMaxGroup / 32;

// ---------------------------------------------------------------------------
// Row quantizer. One warp quantizes one row of one activation matrix.
// ---------------------------------------------------------------------------
enum QuantLayout : int {
    kQuantI8Rows = 0,    // plain int8, row-major M x K (the public sidecar)
    kQuantE2M1Tc = 3,    // tensor-core GEMV and GEMM operand: e2m1 digit rows, digit j of row m at row j*rows + m, K/2 bytes each
};

struct QuantJob {
    const float* x;   // M x K F32
    void* out;        // layout-dependent
    float* scale;     // M
    int32_t* sum;     // M
    int K;
    int Kp;           // row stride of the operand in elements (K for every layout in use)
};

// A weight matrix whose TMA tensor map the quantization launch writes for the
// tensor-core GEMV (kQuantE2M1Tc only).
struct WMapJob {
    const void* w;   // I2_S bytes (payload N x K/4)
    int N;
    int K;
};

struct QuantArgs {
    CUtensorMap wtmpl;  // template map: uint8 2-D, box 128 bytes x 128 rows, 128-byte swizzle
    CUtensorMap* wmaps; // if set, n_wmaps maps written here, wj[i] -> wmaps[i]
    uint32_t* status;   // if set, cleared by the launch (the matmul that follows reports into it)
    uint4* zero;        // if set, zero_16 16-byte words zeroed by the launch (split-K partials)
    unsigned long long zero_16;
    int count;
    int M;
    int rows;           // rows written per job: M, or M' (8 or 16) for kQuantE2M1Tc
    int layout;
    int n_short;        // kQuantE2M1Tc: jobs j < n_short have K <= kQuantWarpRowK (one warp per row),
    int short_ctas;     //   each over short_ctas CTAs; set by launch_quant, which orders the jobs
    int n_wmaps;
    WMapJob wj[kMaxGroup];
    QuantJob j[kMaxGroup];
};

// Rows of at most this many positions are quantized one per warp (kQuantE2M1Tc).
constexpr int kQuantWarpRowK = 1536;
// Orders a.j (short rows first), sets n_short and short_ctas, and launches.
cudaError_t launch_quant(QuantArgs& a, cudaStream_t s);
// Writes the tiled layout of an I2_S payload (N x row_bytes, row_bytes a
// multiple of 16) into tiled (tiled_scale_offset(N, K) bytes); no trailer.
cudaError_t launch_i2s_tile(const uint8_t* w, int64_t N, int64_t K, uint8_t* tiled, cudaStream_t s);

// ---------------------------------------------------------------------------
// Prefill GEMM (M > 16) on tcgen05 (gemm_tc.cu).
// ---------------------------------------------------------------------------
constexpr int kTcMaxMaps = 120;   // distinct activation operands per launch
constexpr int kTcTileW = 128;     // weight rows per tile

struct TcProb {
    const uint8_t* w;         // I2_S bytes
    const float* act_scale;   // M
    const int32_t* row_sum;   // M
    float* y;                 // M x N
    int N;
    int K;
    int map;                  // index into TcArgs::maps (the activation operand)
    int tile0;                // GEMM: first linear tile; GEMV: first linear work unit
    int n_act_tiles;          // GEMM: ceil(M / BN)
    int chunks;               // GEMV: K chunks per row tile (work units per tile)
    int dot_off;              // GEMV, chunks > 1: offset (elements) of this problem's M x N partial dots
    int ticket_off;           // GEMV, chunks > 1: offset of this problem's per-tile chunk counters
};

struct TcArgs {
    CUtensorMap maps[kTcMaxMaps];
    const CUtensorMap* wmaps; // per-problem weight maps in the workspace (written by the quantize launch)
    uint32_t* status;         // workspace status word (timeouts)
    int32_t* dot_base;        // GEMV split-K partial dots (zeroed by the quantize launch)
    uint32_t* ticket_base;    // GEMV split-K chunk counters (zeroed by the quantize launch)
    int n_maps;
    int count;
    int M;
    int BN;                   // GEMM: activation rows per tile (MMA N, multiple of 32, <= 128);
                              // GEMV: M' (8 or 16), MMA N = gemv_tc_op_rows(M')
    int n_act_rows;           // GEMM: rows of one digit plane of the activation operands (M rounded up to BN)

    int total_tiles;          // GEMM: tiles; GEMV: work units
    int share_first;          // GEMV: relative unit shares of the first and second half of the
    int share_second;         //   grid (the first and second CTA placed on each SM)
    long long test_stall_cycles;   // GEMV, test only: > 0 makes the epilogue give up a wait nothing ends
    uint32_t tiled[kTiledMaskWords];   // problems whose weights are in the tiled layout
    TcProb p[kMaxGroup];
};

constexpr int kGemvChunkPositions = 1536;   // K positions per GEMV work unit
// Relative unit shares of the first and second CTA placed on each SM when the
// GEMV grid is full (two CTAs per SM): the first is issued ahead of the second,
// and this split was measured to let both finish together.
constexpr int kGemvShareFirst = 23, kGemvShareSecond = 17;

// Tensor-core GEMM (M > 16): activation rows per tile and the rows of one digit
// plane of its operand.
__host__ __device__ constexpr int gemm_tc_bn(int64_t M) { return M >= 128 ? 128 : (int)((M + 31) / 32 * 32); }
__host__ __device__ constexpr int64_t gemm_tc_rows_pad(int64_t M) { return (M + gemm_tc_bn(M) - 1) / gemm_tc_bn(M) * gemm_tc_bn(M); }

// Tensor-core GEMV activation operand: M' = 8 (M <= 8) or 16 activation rows,
// each split into three base-8 digit rows (digit j of row m at row j*M' + m),
// padded to a multiple of 16 rows (the MMA N). Row-major, K/2 bytes per row.
__host__ __device__ constexpr int gemv_tc_mp(int64_t M) { return M <= 8 ? 8 : 16; }
__host__ __device__ constexpr int gemv_tc_op_rows(int Mp) { return Mp == 8 ? 32 : 48; }

// Fused decode launch (i2s_mul_mat_grouped_fused): the GEMV whose prologue
// quantizes the activations and writes the weight maps itself. The digit
// operands of all activations with the same K are stacked in one buffer (one
// tensor map per distinct K); activation a's rows start at row0.
constexpr int kGvMaxKClasses = 8;
struct GvAct {
    const float* x;      // M x K F32 (the caller's)
    float* scale;        // M row scales (workspace)
    int32_t* sum;        // M row sums (workspace)
    uint8_t* op;         // its gemv_tc_op_rows(M') digit rows of K/2 bytes (workspace)
    long long cost0;     // position of its first row in the launch's quantization order (K per row)
    int K;
    int kclass;          // index into kmaps
    int row0;            // first operand row in its class's stacked buffer
    int dot_lo, dot_n;   // split-K partial dots of the problems that read it (one contiguous range)
    int tk_lo, tk_n;     // their chunk counters (one contiguous range)
};
struct GvFusedArgs {
    CUtensorMap kmaps[kGvMaxKClasses];
    CUtensorMap wtmpl;          // uint8 2-D template, box 128 bytes x 128 rows, 128-byte swizzle
    GvAct acts[kTcMaxMaps];
    CUtensorMap* wmaps;         // one map per problem (workspace), written by the prologue
    uint32_t* flags;            // [count] map written, [n_acts] rows quantized, [1] CTAs done
    uint32_t* status;
    int32_t* dot_base;          // split-K partial dots, zeroed by the prologue
    uint32_t* ticket_base;      // split-K chunk counters, zeroed by the prologue
    long long cost_total;       // sum over activations of M * K
    int n_acts, count, M, BN, total_tiles, share_first, share_second;
    uint32_t tiled[kTiledMaskWords];   // problems whose weights are in the tiled layout
    TcProb p[kMaxGroup];        // TcProb::map = activation index (its class and row0 in acts[])
};
cudaError_t launch_gemv_fused(const GvFusedArgs& a, int grid, cudaStream_t s);

// Kernel parameters are limited to 32764 bytes.
static_assert(sizeof(TcArgs) <= 32764, "TcArgs exceeds the kernel parameter limit");
static_assert(sizeof(GvFusedArgs) <= 32764, "GvFusedArgs exceeds the kernel parameter limit");
static_assert(sizeof(QuantArgs) <= 32764, "QuantArgs exceeds the kernel parameter limit");

bool make_f16_operand_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows);
// rows x row_bytes uint8 matrix, box {128 bytes, box_rows}, 128-byte swizzle
bool make_u8_operand_map(CUtensorMap* map, const void* base, int rows, int row_bytes, int box_rows);
cudaError_t launch_gemm_tc(const TcArgs& a, int grid, cudaStream_t s);
int gemm_tc_max_pairs();   // CTA pairs of the GEMM that fit on the device at once
cudaError_t launch_gemv_tc(const TcArgs& a, int grid, cudaStream_t s);

// ---------------------------------------------------------------------------
// I8_S fused matmul on tcgen05 (i8s_tc.cu) and the per-tensor requant (i8s.cu).
// ---------------------------------------------------------------------------

// Tensor-core I8_S GEMM (i8s_tc.cu): 128 x 160 or 128 x 128 output tiles
// (output features x activation rows), K in chunks of kI8sChunkK positions
// whose f32 partial sums are exact (1024 * 127^2 < 2^24).
constexpr int kI8sTileN = 128;        // output features (weight rows) per tile: the MMA M
constexpr int kI8sTileM = 160;        // activation rows per tile: the MMA N
constexpr int kI8sTileMSmall = 128;   // the other tile height
constexpr int kI8sChunkK = 1024;
constexpr int kI8sMaxK = 64 * kI8sChunkK;   // at most 64 chunks (the slot mask of a split tile)

// The f16 operand rows of the I8_S / W8A8 GEMM hold K rounded up to a
// multiple of 64 positions (one 128-byte swizzle atom), the tail zero-filled:
// a zero product adds nothing, so any K gives the exact integer dot.
inline int64_t i8s_kpad(int64_t K) { return (K + 63) / 64 * 64; }

// A first estimate of the tile height of a launch whose matmuls have M rows,
// N[i] features and K[i] positions, run by `pairs` CTA pairs, counting units
// as if split evenly (the host refines it with the actual pair plan). The busiest pair takes
// ceil(units / pairs) work units (a 256-feature x tm-row tile over one K
// chunk) and each unit moves 256 weight rows and tm activation rows of
// operands through shared memory, the kernel's bound. The height with the
// smaller product wins, 160 on a tie (fewer, larger units): 128 when 160 would
// pad M with more zero rows (512 rows: 640 against 512), 160 when the extra
// units of 128 would lengthen the busiest pair (900 rows: 6 x 416 against
// 7 x 384 over 76 pairs).
inline int i8s_tile_m(int64_t M, const int64_t* N, const int64_t* K, int count, int pairs) {
    int64_t best_cost = -1;
    int best = kI8sTileM;
    for (int tm : {kI8sTileM, kI8sTileMSmall}) {
        int64_t units = 0;
        for (int i = 0; i < count; ++i)
            units += (N[i] + 2 * kI8sTileN - 1) / (2 * kI8sTileN) * ((M + tm - 1) / tm) *
                     ((K[i] + kI8sChunkK - 1) / kI8sChunkK);
        const int64_t p = pairs > 0 ? pairs : 1;
        const int64_t cost = (units + p - 1) / p * (2 * kI8sTileN + tm);
        if (best_cost < 0 || cost < best_cost) best_cost = cost, best = tm;
    }
    return best;
}

// One matmul of a launch: its operand maps, scales, output and offsets into
// the launch's split-tile areas.
constexpr int kI8sMaxGroup = 8;
constexpr int kI8sMaxPairs = 128;   // CTA pairs of one launch (a GB300 holds 76 at once)
struct I8sProb {
    CUtensorMap xmap;          // f16 activations, rows_pad x K, box 64 x tile_m / 2, 128-byte swizzle
    CUtensorMap wmap;          // f16 weights, N x K, box 64 x kI8sTileN, 128-byte swizzle
    const float* w_scale_ptr;  // I8_S: the weight and activation scales (W8A8: any valid floats)
    const float* x_scale_ptr;
    const float* bias;         // N or null
    float* y;                  // M x N F32
    const float* row_scale;    // W8A8 only (col_scale set): per-row activation scales, M
    const float* col_scale;    // W8A8 only: per-channel weight scales, N; null for I8_S
    long long slot0;           // first split-tile slot (tile_m x kI8sTileN int32 sums) of this matmul
    int N, K;
    int n_wt, chunks;          // n_wt: 256-feature tiles (a CTA pair each); chunks: ceil(K / kI8sChunkK)
    int unit0;                 // first work unit
    int ht0;                   // first half-tile (ticket and mask index)
};

struct I8sTcArgs {
    I8sProb p[kI8sMaxGroup];
    unsigned int* amax_bits;   // max |y| as float bits (cleared by the pre-pass); one word per launch
    int32_t* part;             // split tiles: slots of tile_m x kI8sTileN int32 sums
    uint32_t* tickets;         // half-tile chunk counters (cleared by the pre-pass)
    unsigned long long* slot_masks;   // half-tile masks of the slots written (cleared by the pre-pass)
    uint32_t* status;
    int count;                 // matmuls in the launch (1 .. kI8sMaxGroup), all with the same M
    int M, n_at, relu, total_units;
    int tile_m;                // activation rows per tile: kI8sTileM or kI8sTileMSmall
    int bounds[kI8sMaxPairs + 1];   // CTA pair q runs units [bounds[q], bounds[q + 1])
};
static_assert(sizeof(I8sTcArgs) <= 32764, "I8sTcArgs exceeds the kernel parameter limit");
cudaError_t launch_i8s_to_f16(const int8_t* w, int N, __half* wf, const int8_t* x, int M, int rows_pad, int K,
                              __half* xf, void* zero, size_t zero_bytes, uint32_t* status, unsigned int* amax_bits,
                              cudaStream_t s);
// N x K int8 rows (any K) -> N x i8s_kpad(K) f16 rows, the tail zero.
cudaError_t launch_i8_to_f16_rows(const int8_t* src, int64_t rows, int64_t K, __half* dst, cudaStream_t s);
cudaError_t launch_i8s_gemm_tc(const I8sTcArgs& a, int grid, cudaStream_t s);
int i8s_gemm_tc_max_pairs();   // CTA pairs of the I8_S GEMM that fit on the device at once

cudaError_t launch_absmax(const float* y, int64_t n, unsigned int* amax_bits, cudaStream_t s);

// I8_S element-wise ops, convolution pieces and the W8A8 quantizers (i8s_elt.cu).
cudaError_t launch_add_scaled(const uint8_t* a, const uint8_t* b, int64_t n, unsigned int* amax_bits, uint8_t* dst,
                              cudaStream_t s);
cudaError_t launch_rms_norm_scaled(const uint8_t* x, int64_t rows, int64_t ne0, float eps, const float* gamma,
                                   float* rfac, unsigned int* amax_bits, uint8_t* dst, cudaStream_t s);
cudaError_t launch_i8s_transpose(const uint8_t* src, int64_t a, int64_t b, uint8_t* dst, cudaStream_t s);
cudaError_t launch_im2col_asym(const uint8_t* src, int64_t C, int64_t L, int KW, int stride, int pad_l, int64_t OL,
                               uint8_t* dst, cudaStream_t s);
cudaError_t launch_depthwise(const uint8_t* w, const uint8_t* x, const float* bias, int64_t C, int64_t L, int KW,
                             int stride, int pad_l, int64_t OL, int relu, unsigned int* amax_bits, uint8_t* dst,
                             cudaStream_t s);
cudaError_t launch_w8a8_rows(const float* x, int64_t M, int64_t K, int8_t* q, float* ascale, cudaStream_t s);
cudaError_t launch_w8a8_weights(const float* w, int64_t N, int64_t K, int8_t* wq, float* bscale, cudaStream_t s);
// Row quantization of the packed W8A8 calls: one job per distinct activation.
struct W8a8RowJobs {
    const float* x[kI8sMaxGroup];   // M x K F32
    __half* xf[kI8sMaxGroup];       // rows_pad x i8s_kpad(K) f16 operand rows (tail zero)
    float* ascale[kI8sMaxGroup];    // M row scales
    int K[kI8sMaxGroup];
    int count, M, rows_pad;
    uint4* zero;                    // cleared by the launch (the GEMM's tickets and masks)
    unsigned long long zero_16;
    uint32_t* status;
    unsigned int* amax_bits;
};
cudaError_t launch_w8a8_rows_f16(const W8a8RowJobs& J, cudaStream_t s);
cudaError_t launch_i8_to_f16(const int8_t* src, int64_t n, __half* dst, cudaStream_t s);
cudaError_t launch_requant(const float* y, int64_t n, const unsigned int* amax_bits, uint8_t* dst,
                           cudaStream_t s);

int device_sm_count();

}  // namespace i2s
