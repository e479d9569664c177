// The C ABI of libi2s.so (declared and documented in include/i2s.h): argument
// validation, workspace layout, path choice and kernel launches. Every step of
// the computation runs in the kernels of quant.cu, gemv.cu, gemm_tc.cu and
// i8s.cu; this file only marshals.

#include <algorithm>
#include <atomic>
#include <cstring>
#include <vector>

#include "../../include/i2s.h"
#include "internal.h"

namespace i2s {

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeader = 256;             // status word at 0, amax word at 128
constexpr size_t kStatusOff = 0;
constexpr size_t kAmaxOff = 128;
constexpr int kMaxDevices = 64;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned256(const void* p) { return ((uintptr_t)p & 255u) == 0; }

struct DevInfo {
    std::atomic<int> state{0};   // 0 unknown, 1 supported, 2 unsupported
    int sms = 0;
};
DevInfo g_dev[kMaxDevices];

// Returns I2S_OK if the current device is sm_103, caching per device.
int check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return I2S_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return I2S_E_UNSUPPORTED_DEVICE;
    DevInfo& d = g_dev[dev];
    int st = d.state.load(std::memory_order_acquire);
    if (st == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return I2S_E_CUDA;
        d.sms = sms;
        st = (major == 10 && minor == 3) ? 1 : 2;
        d.state.store(st, std::memory_order_release);
    }
    return st == 1 ? I2S_OK : I2S_E_UNSUPPORTED_DEVICE;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? I2S_OK : I2S_E_CUDA; }

// ---------------------------------------------------------------------------
// I2_S workspace: [header][act_scale M][row_sum M][operand][dot_acc M*N][tickets]
// The operand is large enough for either matmul path: the GEMV's e2m1 digit
// rows or the GEMM's f16 rows (2 bytes per position, K rounded up to 256).
// ---------------------------------------------------------------------------
struct ActSlot {
    size_t scale_off, sum_off, op_off;
};

size_t act_slot_bytes(int64_t M, int64_t K) {
    size_t op = 3 * (size_t)gemm_tc_rows_pad(M) * (size_t)(K / 2);   // GEMM: three digit planes
    if (M <= 16) {
        const size_t tc = (size_t)gemv_tc_op_rows(gemv_tc_mp(M)) * (size_t)(K / 2);   // GEMV tensor-core operand
        if (tc > op) op = tc;
    }
    return align_up((size_t)M * 4) * 2 + align_up(op);
}

ActSlot act_slot_at(size_t base, int64_t M) {
    ActSlot s;
    s.scale_off = base;
    s.sum_off = base + align_up((size_t)M * 4);
    s.op_off = s.sum_off + align_up((size_t)M * 4);
    return s;
}

bool i2s_shape_ok(int64_t N, int64_t K, int64_t M) {
    if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return false;
    if (M * K >= ((int64_t)1 << 31) || N * (K / 4) >= ((int64_t)1 << 31) || M * N >= ((int64_t)1 << 31)) return false;
    if (K > 65536) return false;   // keeps |dot| = |sum code*q| <= 254*K below 2^24
    return true;
}


}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    if (g_dev[dev].state.load() == 0) check_device();
    return g_dev[dev].sms > 0 ? g_dev[dev].sms : 152;
}

}  // namespace i2s

using namespace i2s;

#pragma GCC visibility push(default)
extern "C" {

static int run_gemm_tc(const i2s_problem* probs, int count, int64_t M, void* ws, int grid_ctas,
                       i2s_stream_t stream, int phases);
static int run_gemv_tc(const i2s_problem* probs, int count, int64_t M, void* ws, int grid_ctas,
                       i2s_stream_t stream, int phases, long long test_stall_cycles = 0);

const char* i2s_status_string(int status) {
    switch (status) {
        case I2S_OK: return "ok";
        case I2S_E_BAD_SHAPE: return "bad shape";
        case I2S_E_NULL_PTR: return "null pointer";
        case I2S_E_MISALIGNED: return "misaligned pointer";
        case I2S_E_WORKSPACE_TOO_SMALL: return "workspace too small";
        case I2S_E_CUDA: return "CUDA error";
        case I2S_E_DEVICE_TIMEOUT: return "device wait timed out";
        case I2S_E_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
        case I2S_E_BAD_ARG: return "bad argument";
        default: return "unknown status";
    }
}

int i2s_version(void) { return 200; }

int i2s_device_supported(void) {
    const int r = check_device();
    if (r == I2S_OK) return 1;
    if (r == I2S_E_UNSUPPORTED_DEVICE) return 0;
    return r;
}

size_t i2s_nbytes(int64_t N, int64_t K) {
    if (N < 1 || K < 128 || K % 128) return 0;
    return (size_t)N * (size_t)K / 4 + 32;
}
size_t i2s_scale_offset(int64_t N, int64_t K) {
    if (N < 1 || K < 128 || K % 128) return 0;
    return (size_t)N * (size_t)K / 4;
}
size_t i2s_tiled_scale_offset(int64_t N, int64_t K) {
    if (N < 1 || K < 128 || K % 128) return 0;
    return tiled_scale_offset(N, K);
}
size_t i2s_tiled_nbytes(int64_t N, int64_t K) {
    const size_t off = i2s_tiled_scale_offset(N, K);
    return off ? off + 32 : 0;
}

int i2s_tile_weights(const void* w_i2s, int64_t N, int64_t K, void* tiled, i2s_stream_t stream) {
    if (!w_i2s || !tiled) return I2S_E_NULL_PTR;
    if (!i2s_shape_ok(N, K, 1)) return I2S_E_BAD_SHAPE;
    if (!aligned16(w_i2s) || !aligned16(tiled)) return I2S_E_MISALIGNED;
    const uintptr_t a0 = (uintptr_t)w_i2s, a1 = a0 + i2s_nbytes(N, K);
    const uintptr_t b0 = (uintptr_t)tiled, b1 = b0 + i2s_tiled_nbytes(N, K);
    if (a0 < b1 && b0 < a1) return I2S_E_BAD_ARG;   // the buffers overlap
    int r = check_device();
    if (r) return r;
    const uint8_t* w = static_cast<const uint8_t*>(w_i2s);
    uint8_t* t = static_cast<uint8_t*>(tiled);
    r = cuda_status(launch_i2s_tile(w, N, K, t, stream));
    if (r) return r;
    return cuda_status(cudaMemcpyAsync(t + tiled_scale_offset(N, K), w + i2s_scale_offset(N, K), 32,
                                       cudaMemcpyDeviceToDevice, stream));
}

size_t i8s_nbytes(int64_t n) { return n < 1 ? 0 : (size_t)round_up(n, 32) + 32; }
size_t i8s_scale_offset(int64_t n) { return n < 1 ? 0 : (size_t)round_up(n, 32); }

int i2s_pack_host(const uint8_t* codes, int64_t N, int64_t K, float w_scale, void* dst) {
    if (!codes || !dst) return I2S_E_NULL_PTR;
    if (N < 1 || K < 128 || K % 128) return I2S_E_BAD_SHAPE;
    uint8_t* out = static_cast<uint8_t*>(dst);
    const int64_t groups = N * K / 128;
    for (int64_t g = 0; g < groups; ++g) {
        const uint8_t* c = codes + g * 128;
        uint8_t* o = out + g * 32;
        for (int gp = 0; gp < 32; ++gp)
            o[gp] = (uint8_t)(((c[gp] & 3) << 6) | ((c[32 + gp] & 3) << 4) | ((c[64 + gp] & 3) << 2) | (c[96 + gp] & 3));
    }
    uint8_t* trailer = out + N * K / 4;
    std::memset(trailer, 0, 32);
    std::memcpy(trailer, &w_scale, 4);
    return I2S_OK;
}

int i8s_pack_host(const int8_t* q, int64_t n, float scale, void* dst) {
    if (!q || !dst) return I2S_E_NULL_PTR;
    if (n < 1) return I2S_E_BAD_SHAPE;
    uint8_t* out = static_cast<uint8_t*>(dst);
    const size_t off = i8s_scale_offset(n);
    std::memcpy(out, q, (size_t)n);
    std::memset(out + n, 0, off + 32 - (size_t)n);
    std::memcpy(out + off, &scale, 4);
    return I2S_OK;
}

int i2s_quantize_act(const float* x, int64_t M, int64_t K, int8_t* q, float* act_scale, int32_t* row_sum,
                     i2s_stream_t stream) {
    if (!x || !q || !act_scale || !row_sum) return I2S_E_NULL_PTR;
    if (M < 1 || K < 4 || K % 4 || M * K >= ((int64_t)1 << 31)) return I2S_E_BAD_SHAPE;
    if (!aligned16(x) || ((uintptr_t)q & 3u) || ((uintptr_t)act_scale & 3u) || ((uintptr_t)row_sum & 3u))
        return I2S_E_MISALIGNED;
    int r = check_device();
    if (r) return r;
    QuantArgs a;
    a.wmaps = nullptr;
    a.n_wmaps = 0;
    a.status = nullptr;
    a.zero = nullptr;
    a.zero_16 = 0;
    a.count = 1;
    a.M = (int)M;
    a.rows = (int)M;
    a.layout = kQuantI8Rows;
    a.j[0] = QuantJob{x, q, act_scale, row_sum, (int)K, (int)K};
    return cuda_status(launch_quant(a, stream));
}

// Split-K partial area of one problem: M x N int32 partial dots and one chunk
// counter per 128-row tile.
static size_t split_area_bytes(int64_t M, int64_t N) {
    const size_t tiles = (size_t)((N + kTcTileW - 1) / kTcTileW);
    return align_up((size_t)M * (size_t)N * 4) + align_up(tiles * 4);
}

// TMA tensor maps of the GEMV's weight matrices (one per problem), at the end.
static size_t wmap_area(int count) { return align_up((size_t)count * sizeof(CUtensorMap)); }

size_t i2s_mul_mat_workspace(int64_t M, int64_t N, int64_t K) {
    if (!i2s_shape_ok(N, K, M)) return 0;
    return kHeader + act_slot_bytes(M, K) + split_area_bytes(M, N) + wmap_area(1);
}

int i2s_mul_mat_ex(const void* w_i2s, int64_t N, int64_t K, const float* x, int64_t M, float* y, void* ws,
                   size_t ws_bytes, const i2s_config* config, i2s_stream_t stream) {
    if (!w_i2s || !x || !y || !ws) return I2S_E_NULL_PTR;
    if (!i2s_shape_ok(N, K, M)) return I2S_E_BAD_SHAPE;
    if (!aligned16(w_i2s) || !aligned16(x) || !aligned16(y) || !aligned256(ws)) return I2S_E_MISALIGNED;
    if (ws_bytes < i2s_mul_mat_workspace(M, N, K)) return I2S_E_WORKSPACE_TOO_SMALL;
    // the configuration, checked on the host before any CUDA call
    const int path = config ? config->path : 0;
    if (path != 0 && path != 2 && path != 3) return I2S_E_BAD_ARG;
    if (path == 3 && M > 16) return I2S_E_BAD_ARG;
    const unsigned layout = config ? config->w_layout : I2S_LAYOUT_I2S;
    if (layout != I2S_LAYOUT_I2S && layout != I2S_LAYOUT_TILED) return I2S_E_BAD_ARG;
    if (config && config->test_stall_cycles < 0) return I2S_E_BAD_ARG;
    int r = check_device();
    if (r) return r;

    i2s_problem p{w_i2s, N, K, x, y, layout};
    if (path == 2 || (path == 0 && M > 16)) return run_gemm_tc(&p, 1, M, ws, config ? config->grid_ctas : 0, stream, 3);
    return run_gemv_tc(&p, 1, M, ws, config ? config->grid_ctas : 0, stream, 3,
                       config ? (long long)config->test_stall_cycles : 0);
}

int i2s_mul_mat(const void* w_i2s, int64_t N, int64_t K, const float* x, int64_t M, float* y, void* ws,
                size_t ws_bytes, i2s_stream_t stream) {
    return i2s_mul_mat_ex(w_i2s, N, K, x, M, y, ws, ws_bytes, nullptr, stream);
}

// Distinct activations of a group, in first-use order.
// The checks every grouped entry point makes on each problem, in this order.
static int check_problem(const i2s_problem& p, int64_t M) {
    if (!p.w_i2s || !p.x || !p.y) return I2S_E_NULL_PTR;
    if (!i2s_shape_ok(p.N, p.K, M)) return I2S_E_BAD_SHAPE;
    if (!aligned16(p.w_i2s) || !aligned16(p.x) || !aligned16(p.y)) return I2S_E_MISALIGNED;
    if (p.w_layout != I2S_LAYOUT_I2S && p.w_layout != I2S_LAYOUT_TILED) return I2S_E_BAD_ARG;
    return I2S_OK;
}

// Bit i set: problem i's weights are in the tiled layout.
static void fill_tiled_mask(uint32_t* mask, const i2s_problem* probs, int count) {
    for (int w = 0; w < kTiledMaskWords; ++w) mask[w] = 0;
    for (int i = 0; i < count; ++i)
        if (probs[i].w_layout == I2S_LAYOUT_TILED) mask[i >> 5] |= 1u << (i & 31);
}

static int group_acts(const i2s_problem* probs, int count, std::vector<int>& act_of,
                      std::vector<int>& first) {
    act_of.assign(count, -1);
    first.clear();
    for (int i = 0; i < count; ++i) {
        for (size_t a = 0; a < first.size(); ++a) {
            const i2s_problem& f = probs[first[a]];
            if (f.x == probs[i].x && f.K == probs[i].K) { act_of[i] = (int)a; break; }
        }
        if (act_of[i] < 0) { act_of[i] = (int)first.size(); first.push_back(i); }
    }
    return (int)first.size();
}

// Tensor-core GEMM path (M > 16): phase 1 quantizes every distinct activation
// into the e2m1 digit planes, phase 2 runs one persistent GEMM launch over
// all problems. Arguments are validated by the callers.
static int run_gemm_tc(const i2s_problem* probs, int count, int64_t M, void* ws, int grid_ctas,
                       i2s_stream_t stream, int phases) {
    std::vector<int> act_of, first;
    const int n_act = group_acts(probs, count, act_of, first);
    if (n_act > kTcMaxMaps) return I2S_E_BAD_ARG;
    uint8_t* base = static_cast<uint8_t*>(ws);
    std::vector<ActSlot> slots(n_act);
    size_t off = kHeader;
    for (int a = 0; a < n_act; ++a) {
        slots[a] = act_slot_at(off, M);
        off += act_slot_bytes(M, probs[first[a]].K);
    }
    // one TMA map per weight matrix (its packed codes), written by the
    // quantization launch
    CUtensorMap* wmaps = reinterpret_cast<CUtensorMap*>(base + off);
    int r;
    if (phases & 1) {
        static thread_local QuantArgs qa;
        if (!make_u8_operand_map(&qa.wtmpl, wmaps, kTcTileW, 128, kTcTileW)) return I2S_E_CUDA;
        qa.wmaps = wmaps;
        qa.n_wmaps = count;
        for (int i = 0; i < count; ++i) qa.wj[i] = WMapJob{probs[i].w_i2s, (int)probs[i].N, (int)probs[i].K};
        qa.status = reinterpret_cast<uint32_t*>(base + kStatusOff);
        qa.zero = nullptr;
        qa.zero_16 = 0;
        qa.count = n_act;
        qa.M = (int)M;
        qa.rows = (int)gemm_tc_rows_pad(M);
        qa.layout = kQuantE2M1Tc;
        for (int a = 0; a < n_act; ++a) {
            const i2s_problem& p = probs[first[a]];
            qa.j[a] = QuantJob{p.x, base + slots[a].op_off, reinterpret_cast<float*>(base + slots[a].scale_off),
                               reinterpret_cast<int32_t*>(base + slots[a].sum_off), (int)p.K, (int)p.K};
        }
        r = cuda_status(launch_quant(qa, stream));
        if (r) return r;
    }
    if (phases & 2) {
        static thread_local TcArgs ta;
        const int BN = gemm_tc_bn(M);
        const int rows_pad = (int)gemm_tc_rows_pad(M);
        ta.n_maps = n_act;
        ta.count = count;
        ta.M = (int)M;
        ta.BN = BN;
        ta.n_act_rows = rows_pad;
        ta.test_stall_cycles = 0;
        ta.status = reinterpret_cast<uint32_t*>(base + kStatusOff);
        ta.wmaps = wmaps;
        // the three digit planes of each activation; each CTA of a pair loads
        // half of a tile's activation rows of a plane
        for (int a = 0; a < n_act; ++a)
            if (!make_u8_operand_map(&ta.maps[a], base + slots[a].op_off, 3 * rows_pad, (int)(probs[first[a]].K / 2),
                                     BN / 2))
                return I2S_E_CUDA;
        const int n_act_tiles = (int)((M + BN - 1) / BN);
        int tiles = 0;
        for (int i = 0; i < count; ++i) {
            const i2s_problem& q = probs[i];
            const ActSlot& s = slots[act_of[i]];
            TcProb& p = ta.p[i];
            p.w = static_cast<const uint8_t*>(q.w_i2s);
            p.act_scale = reinterpret_cast<const float*>(base + s.scale_off);
            p.row_sum = reinterpret_cast<const int32_t*>(base + s.sum_off);
            p.y = q.y;
            p.N = (int)q.N;
            p.K = (int)q.K;
            p.map = act_of[i];
            p.tile0 = tiles;
            p.n_act_tiles = n_act_tiles;
            tiles += (int)((q.N + 2 * kTcTileW - 1) / (2 * kTcTileW)) * n_act_tiles;   // 256-row tiles, one CTA pair each
        }
        ta.total_tiles = tiles;
        fill_tiled_mask(ta.tiled, probs, count);
        const int sms = device_sm_count();
        int pairs = (grid_ctas > 0 ? grid_ctas : sms) / 2;   // clusters of two CTAs
        const int resident = gemm_tc_max_pairs();   // a persistent grid: no second wave
        if (pairs > resident) pairs = resident;
        if (pairs > tiles) pairs = tiles;
        if (pairs < 1) pairs = 1;
        r = cuda_status(launch_gemm_tc(ta, 2 * pairs, stream));
        if (r) return r;
    }
    return I2S_OK;
}

// Tensor-core GEMV path (M <= 16): phase 1 quantizes every distinct activation
// into the e2m1 digit operand rows, phase 2 runs one persistent launch over all
// problems (two CTAs per SM). Arguments are validated by the callers.

static int run_gemv_tc(const i2s_problem* probs, int count, int64_t M, void* ws, int grid_ctas,
                       i2s_stream_t stream, int phases, long long test_stall_cycles) {
    std::vector<int> act_of, first;
    const int n_act = group_acts(probs, count, act_of, first);
    if (n_act > kTcMaxMaps) return I2S_E_BAD_ARG;
    const int Mp = gemv_tc_mp(M);
    uint8_t* base = static_cast<uint8_t*>(ws);
    std::vector<ActSlot> slots(n_act);
    size_t off = kHeader;
    for (int a = 0; a < n_act; ++a) {
        slots[a] = act_slot_at(off, M);
        off += act_slot_bytes(M, probs[first[a]].K);
    }
    int r;
    // split-K partial dots and chunk counters (problems with K above one chunk)
    size_t dots = 0, tickets = 0;
    for (int i = 0; i < count; ++i)
        if (probs[i].K > kGemvChunkPositions) {
            dots += (size_t)M * (size_t)probs[i].N;
            tickets += (size_t)((probs[i].N + kTcTileW - 1) / kTcTileW);
        }
    const size_t dot_off_bytes = off;
    const size_t ticket_off_bytes = off + align_up(dots * 4);
    const size_t split_bytes = align_up(dots * 4) + align_up(tickets * 4);
    // one TMA map per weight matrix, written by the quantization launch
    CUtensorMap* wmaps = reinterpret_cast<CUtensorMap*>(base + dot_off_bytes + split_bytes);
    if (phases & 1) {
        static thread_local QuantArgs qa;
        if (!make_u8_operand_map(&qa.wtmpl, wmaps, kTcTileW, 128, kTcTileW)) return I2S_E_CUDA;
        qa.wmaps = wmaps;
        qa.n_wmaps = count;
        for (int i = 0; i < count; ++i) qa.wj[i] = WMapJob{probs[i].w_i2s, (int)probs[i].N, (int)probs[i].K};
        qa.status = reinterpret_cast<uint32_t*>(base + kStatusOff);
        qa.zero = split_bytes ? reinterpret_cast<uint4*>(base + dot_off_bytes) : nullptr;
        qa.zero_16 = split_bytes / 16;
        qa.count = n_act;
        qa.M = (int)M;
        qa.rows = Mp;
        qa.layout = kQuantE2M1Tc;
        for (int a = 0; a < n_act; ++a) {
            const i2s_problem& p = probs[first[a]];
            qa.j[a] = QuantJob{p.x, base + slots[a].op_off, reinterpret_cast<float*>(base + slots[a].scale_off),
                               reinterpret_cast<int32_t*>(base + slots[a].sum_off), (int)p.K, (int)p.K};
        }
        r = cuda_status(launch_quant(qa, stream));
        if (r) return r;
    }
    if (phases & 2) {
        static thread_local TcArgs ta;
        ta.n_maps = n_act;
        ta.count = count;
        ta.M = (int)M;
        ta.BN = Mp;
        ta.status = reinterpret_cast<uint32_t*>(base + kStatusOff);
        for (int a = 0; a < n_act; ++a)
            if (!make_u8_operand_map(&ta.maps[a], base + slots[a].op_off, gemv_tc_op_rows(Mp),
                                     (int)(probs[first[a]].K / 2), gemv_tc_op_rows(Mp)))
                return I2S_E_CUDA;
        ta.dot_base = reinterpret_cast<int32_t*>(base + dot_off_bytes);
        ta.ticket_base = reinterpret_cast<uint32_t*>(base + ticket_off_bytes);
        ta.wmaps = wmaps;
        int units = 0, dot_elems = 0, ticket_elems = 0;
        for (int i = 0; i < count; ++i) {
            const i2s_problem& q = probs[i];
            const ActSlot& s = slots[act_of[i]];
            TcProb& p = ta.p[i];
            const int row_tiles = (int)((q.N + kTcTileW - 1) / kTcTileW);
            const int chunks = (int)((q.K + kGemvChunkPositions - 1) / kGemvChunkPositions);
            p.w = static_cast<const uint8_t*>(q.w_i2s);
            p.act_scale = reinterpret_cast<const float*>(base + s.scale_off);
            p.row_sum = reinterpret_cast<const int32_t*>(base + s.sum_off);
            p.y = q.y;
            p.N = (int)q.N;
            p.K = (int)q.K;
            p.map = act_of[i];
            p.tile0 = units;
            p.n_act_tiles = 1;
            p.chunks = chunks;
            p.dot_off = dot_elems;
            p.ticket_off = ticket_elems;
            if (chunks > 1) {
                dot_elems += (int)(M * q.N);
                ticket_elems += row_tiles;
            }
            units += row_tiles * chunks;
        }
        ta.total_tiles = units;
        fill_tiled_mask(ta.tiled, probs, count);
        const int tiles = units;
        const int cap = 2 * device_sm_count();
        int grid = grid_ctas > 0 ? grid_ctas : cap;
        if (grid > cap) grid = cap;
        if (grid > tiles) grid = tiles;
        // With a full grid (two CTAs per SM) the first CTA on each SM gets the
        // larger share measured to make both finish together.
        ta.share_first = grid == cap ? kGemvShareFirst : 1;
        ta.share_second = grid == cap ? kGemvShareSecond : 1;
        ta.test_stall_cycles = test_stall_cycles;
        r = cuda_status(launch_gemv_tc(ta, grid, stream));
        if (r) return r;
    }
    return I2S_OK;
}

// ---------------------------------------------------------------------------
// Fused decode launch: one GEMV launch whose prologue quantizes the
// activations. Workspace: [header: status][flags, a fixed area cleared by
// i2s_mul_mat_grouped_fused_init and left clear by every launch][row scales
// and sums, 16 per activation][per distinct K: the digit operands of its
// activations, stacked][split-K partial dots][chunk counters][weight maps].
// ---------------------------------------------------------------------------
static constexpr size_t kFusedFlagBytes = 2048;   // >= 4 * (I2S_MAX_GROUP + kTcMaxMaps + 1)
static_assert(kFusedFlagBytes >= 4 * (kMaxGroup + kTcMaxMaps + 1), "fused flag area");

struct FusedPlan {
    int n_act = 0, n_class = 0;
    std::vector<int> act_of, first, class_of_act, idx_in_class;
    int class_K[kGvMaxKClasses] = {};
    int class_n[kGvMaxKClasses] = {};
    size_t scale_off = 0, sum_off = 0, class_off[kGvMaxKClasses] = {}, dot_off = 0, ticket_off = 0, map_off = 0,
           end = 0;
};

// returns I2S_OK or BAD_ARG (too many activations or distinct K)
static int fused_plan(const i2s_problem* probs, int count, int64_t M, FusedPlan& pl) {
    pl.n_act = group_acts(probs, count, pl.act_of, pl.first);
    if (pl.n_act > kTcMaxMaps) return I2S_E_BAD_ARG;
    const int op_rows = gemv_tc_op_rows(gemv_tc_mp(M));
    pl.class_of_act.assign(pl.n_act, -1);
    pl.idx_in_class.assign(pl.n_act, 0);
    for (int a = 0; a < pl.n_act; ++a) {
        const int K = (int)probs[pl.first[a]].K;
        int c = 0;
        while (c < pl.n_class && pl.class_K[c] != K) ++c;
        if (c == pl.n_class) {
            if (pl.n_class == kGvMaxKClasses) return I2S_E_BAD_ARG;
            pl.class_K[pl.n_class++] = K;
        }
        pl.class_of_act[a] = c;
        pl.idx_in_class[a] = pl.class_n[c]++;
    }
    size_t off = kHeader + kFusedFlagBytes;
    pl.scale_off = off;
    off += align_up((size_t)pl.n_act * 16 * 4);
    pl.sum_off = off;
    off += align_up((size_t)pl.n_act * 16 * 4);
    for (int c = 0; c < pl.n_class; ++c) {
        pl.class_off[c] = off;
        off += align_up((size_t)pl.class_n[c] * op_rows * (size_t)(pl.class_K[c] / 2));
    }
    size_t dots = 0, tickets = 0;
    for (int i = 0; i < count; ++i)
        if (probs[i].K > kGemvChunkPositions) {
            dots += (size_t)M * (size_t)probs[i].N;
            tickets += (size_t)((probs[i].N + kTcTileW - 1) / kTcTileW);
        }
    pl.dot_off = off;
    off += align_up(dots * 4);
    pl.ticket_off = off;
    off += align_up(tickets * 4);
    pl.map_off = off;
    off += wmap_area(count);
    pl.end = off;
    return I2S_OK;
}

static int fused_check(const i2s_problem* probs, int count, int64_t M) {
    if (!probs) return I2S_E_NULL_PTR;
    if (count < 1 || count > I2S_MAX_GROUP) return I2S_E_BAD_ARG;
    if (M < 1 || M > 16) return I2S_E_BAD_SHAPE;
    for (int i = 0; i < count; ++i) {
        const i2s_problem& p = probs[i];
        if (const int r = check_problem(p, M)) return r;
    }
    return I2S_OK;
}

size_t i2s_mul_mat_grouped_fused_workspace(const i2s_problem* probs, int count, int64_t M) {
    if (fused_check(probs, count, M) != I2S_OK) return 0;
    FusedPlan pl;
    if (fused_plan(probs, count, M, pl) != I2S_OK) return 0;
    return pl.end;
}

int i2s_mul_mat_grouped_fused_init(void* ws, size_t ws_bytes, i2s_stream_t stream) {
    if (!ws) return I2S_E_NULL_PTR;
    if (!aligned256(ws)) return I2S_E_MISALIGNED;
    if (ws_bytes < kHeader + kFusedFlagBytes) return I2S_E_WORKSPACE_TOO_SMALL;
    int r = check_device();
    if (r) return r;
    return cuda_status(cudaMemsetAsync(ws, 0, kHeader + kFusedFlagBytes, stream));
}

int i2s_mul_mat_grouped_fused(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                              i2s_stream_t stream) {
    int r = fused_check(probs, count, M);
    if (r) return r;
    if (!ws) return I2S_E_NULL_PTR;
    if (!aligned256(ws)) return I2S_E_MISALIGNED;
    FusedPlan pl;
    r = fused_plan(probs, count, M, pl);
    if (r) return r;
    if (ws_bytes < pl.end) return I2S_E_WORKSPACE_TOO_SMALL;
    r = check_device();
    if (r) return r;
    const int Mp = gemv_tc_mp(M);
    const int op_rows = gemv_tc_op_rows(Mp);
    uint8_t* base = static_cast<uint8_t*>(ws);
    static thread_local GvFusedArgs fa;
    for (int c = 0; c < pl.n_class; ++c)
        if (!make_u8_operand_map(&fa.kmaps[c], base + pl.class_off[c], pl.class_n[c] * op_rows, pl.class_K[c] / 2,
                                 op_rows))
            return I2S_E_CUDA;
    CUtensorMap* wmaps = reinterpret_cast<CUtensorMap*>(base + pl.map_off);
    if (!make_u8_operand_map(&fa.wtmpl, wmaps, kTcTileW, 128, kTcTileW)) return I2S_E_CUDA;
    long long cost = 0;
    for (int a = 0; a < pl.n_act; ++a) {
        const i2s_problem& p = probs[pl.first[a]];
        GvAct& A = fa.acts[a];
        const int c = pl.class_of_act[a];
        A.x = p.x;
        A.scale = reinterpret_cast<float*>(base + pl.scale_off) + 16 * a;
        A.sum = reinterpret_cast<int32_t*>(base + pl.sum_off) + 16 * a;
        A.row0 = pl.idx_in_class[a] * op_rows;
        A.op = base + pl.class_off[c] + (size_t)A.row0 * (size_t)(p.K / 2);
        A.cost0 = cost;
        A.K = (int)p.K;
        A.kclass = c;
        A.dot_lo = A.dot_n = A.tk_lo = A.tk_n = 0;
        cost += M * p.K;
    }
    // split-K areas laid out activation by activation, so the prologue zeroes
    // one contiguous range per activation
    std::vector<int> dot_off(count, 0), ticket_off(count, 0);
    {
        int dot_elems = 0, ticket_elems = 0;
        for (int a = 0; a < pl.n_act; ++a) {
            GvAct& A = fa.acts[a];
            A.dot_lo = dot_elems;
            A.tk_lo = ticket_elems;
            for (int i = 0; i < count; ++i) {
                if (pl.act_of[i] != a || probs[i].K <= kGemvChunkPositions) continue;
                dot_off[i] = dot_elems;
                ticket_off[i] = ticket_elems;
                dot_elems += (int)(M * probs[i].N);
                ticket_elems += (int)((probs[i].N + kTcTileW - 1) / kTcTileW);
            }
            A.dot_n = dot_elems - A.dot_lo;
            A.tk_n = ticket_elems - A.tk_lo;
        }
    }
    fa.cost_total = cost;
    fa.wmaps = wmaps;
    fa.flags = reinterpret_cast<uint32_t*>(base + kHeader);
    fa.status = reinterpret_cast<uint32_t*>(base + kStatusOff);
    fa.dot_base = reinterpret_cast<int32_t*>(base + pl.dot_off);
    fa.ticket_base = reinterpret_cast<uint32_t*>(base + pl.ticket_off);
    fa.n_acts = pl.n_act;
    fa.count = count;
    fill_tiled_mask(fa.tiled, probs, count);
    fa.M = (int)M;
    fa.BN = Mp;
    int units = 0;
    for (int i = 0; i < count; ++i) {
        const i2s_problem& q = probs[i];
        const int act = pl.act_of[i];
        TcProb& P = fa.p[i];
        const int row_tiles = (int)((q.N + kTcTileW - 1) / kTcTileW);
        const int chunks = (int)((q.K + kGemvChunkPositions - 1) / kGemvChunkPositions);
        P.w = static_cast<const uint8_t*>(q.w_i2s);
        P.act_scale = fa.acts[act].scale;
        P.row_sum = fa.acts[act].sum;
        P.y = q.y;
        P.N = (int)q.N;
        P.K = (int)q.K;
        P.map = act;
        P.tile0 = units;
        P.n_act_tiles = 1;
        P.chunks = chunks;
        P.dot_off = dot_off[i];
        P.ticket_off = ticket_off[i];
        units += row_tiles * chunks;
    }
    fa.total_tiles = units;
    const int cap = 2 * device_sm_count();
    const int grid = units < cap ? units : cap;
    fa.share_first = grid == cap ? kGemvShareFirst : 1;
    fa.share_second = grid == cap ? kGemvShareSecond : 1;
    return cuda_status(launch_gemv_fused(fa, grid, stream));
}

size_t i2s_mul_mat_grouped_workspace(const i2s_problem* probs, int count, int64_t M) {
    if (!probs || count < 1 || count > I2S_MAX_GROUP) return 0;
    for (int i = 0; i < count; ++i)
        if (probs[i].w_layout != I2S_LAYOUT_I2S && probs[i].w_layout != I2S_LAYOUT_TILED) return 0;
    std::vector<int> act_of, first;
    group_acts(probs, count, act_of, first);
    size_t total = kHeader;
    for (int a : first) {
        if (!i2s_shape_ok(probs[a].N, probs[a].K, M)) return 0;
        total += act_slot_bytes(M, probs[a].K);
    }
    if (M > 16) {   // the GEMM's per-problem maps of the packed codes
        for (int i = 0; i < count; ++i)
            if (!i2s_shape_ok(probs[i].N, probs[i].K, M)) return 0;
        total += wmap_area(count);
    }
    if (M <= 16) {   // split-K partials of the tensor-core GEMV
        size_t dots = 0, tickets = 0;
        for (int i = 0; i < count; ++i) {
            if (!i2s_shape_ok(probs[i].N, probs[i].K, M)) return 0;
            if (probs[i].K > kGemvChunkPositions) {
                dots += (size_t)M * (size_t)probs[i].N;
                tickets += (size_t)((probs[i].N + kTcTileW - 1) / kTcTileW);
            }
        }
        total += align_up(dots * 4) + align_up(tickets * 4) + wmap_area(count);
    }
    return total;
}

// Phase bits of a grouped call: 1 = quantize the distinct activations into
// the workspace, 2 = run the matmuls from the workspace. M <= 16 runs the
// tensor-core GEMV, larger M the tensor-core GEMM.
static int grouped_impl(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                        i2s_stream_t stream, int phases) {
    if (!probs || !ws) return I2S_E_NULL_PTR;
    if (count < 1 || count > I2S_MAX_GROUP) return I2S_E_BAD_ARG;
    for (int i = 0; i < count; ++i) {
        const i2s_problem& p = probs[i];
        if (const int r = check_problem(p, M)) return r;
    }
    if (!aligned256(ws)) return I2S_E_MISALIGNED;
    if (ws_bytes < i2s_mul_mat_grouped_workspace(probs, count, M)) return I2S_E_WORKSPACE_TOO_SMALL;
    int r = check_device();
    if (r) return r;
    if (M > 16) return run_gemm_tc(probs, count, M, ws, 0, stream, phases);
    return run_gemv_tc(probs, count, M, ws, 0, stream, phases);
}

int i2s_mul_mat_grouped(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                        i2s_stream_t stream) {
    return grouped_impl(probs, count, M, ws, ws_bytes, stream, 3);
}

int i2s_mul_mat_grouped_quantize(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                                 i2s_stream_t stream) {
    return grouped_impl(probs, count, M, ws, ws_bytes, stream, 1);
}

int i2s_mul_mat_grouped_run(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                            i2s_stream_t stream) {
    return grouped_impl(probs, count, M, ws, ws_bytes, stream, 2);
}

// ---------------------------------------------------------------------------
// Grouped call on host activations and outputs. Workspace: [grouped
// workspace][device copies of the merged activation ranges][device copies of
// the merged output ranges], each copy 256-byte aligned.
// ---------------------------------------------------------------------------
struct HostSpan {
    uintptr_t lo, hi;   // host byte range
    size_t off;         // its device copy's offset in the workspace
};

// Merges the host byte ranges that touch or overlap into spans sorted by
// address and lays their device copies out from `base`. Returns the end offset.
static size_t host_spans(std::vector<std::pair<uintptr_t, uintptr_t>> r, size_t base, std::vector<HostSpan>& out) {
    std::sort(r.begin(), r.end());
    out.clear();
    for (const auto& e : r) {
        if (!out.empty() && e.first <= out.back().hi) {
            out.back().hi = std::max(out.back().hi, e.second);
        } else {
            out.push_back({e.first, e.second, 0});
        }
    }
    for (HostSpan& s : out) {
        s.off = base;
        base += align_up((size_t)(s.hi - s.lo));
    }
    return base;
}

// The span holding host address p (spans sorted, p inside one of them).
static const HostSpan& span_of(const std::vector<HostSpan>& spans, uintptr_t p) {
    size_t lo = 0, hi = spans.size();
    while (hi - lo > 1) {
        const size_t mid = (lo + hi) / 2;
        if (spans[mid].lo <= p) lo = mid; else hi = mid;
    }
    return spans[lo];
}

struct HostPlan {
    std::vector<HostSpan> xs, ys;
    size_t grouped = 0, total = 0;
};

// Validates the host problem list and lays out the workspace. Returns a status.
static int host_plan(const i2s_problem* probs, int count, int64_t M, HostPlan& pl) {
    if (!probs) return I2S_E_NULL_PTR;
    if (count < 1 || count > I2S_MAX_GROUP) return I2S_E_BAD_ARG;
    std::vector<std::pair<uintptr_t, uintptr_t>> xr, yr;
    for (int i = 0; i < count; ++i) {
        const i2s_problem& p = probs[i];
        if (const int r = check_problem(p, M)) return r;
        const uintptr_t x = (uintptr_t)p.x, y = (uintptr_t)p.y;
        xr.push_back({x, x + (uintptr_t)(M * p.K) * 4});
        yr.push_back({y, y + (uintptr_t)(M * p.N) * 4});
    }
    // outputs may overlap neither one another nor any activation
    std::vector<std::pair<uintptr_t, uintptr_t>> ys = yr;
    std::sort(ys.begin(), ys.end());
    for (size_t i = 1; i < ys.size(); ++i)
        if (ys[i].first < ys[i - 1].second) return I2S_E_BAD_ARG;
    for (const auto& y : ys)
        for (const auto& x : xr)
            if (y.first < x.second && x.first < y.second) return I2S_E_BAD_ARG;
    pl.grouped = i2s_mul_mat_grouped_workspace(probs, count, M);
    if (pl.grouped == 0) return I2S_E_BAD_SHAPE;
    const size_t after_x = host_spans(xr, pl.grouped, pl.xs);
    pl.total = host_spans(yr, after_x, pl.ys);
    return I2S_OK;
}

size_t i2s_mul_mat_grouped_host_workspace(const i2s_problem* probs, int count, int64_t M) {
    HostPlan pl;
    return host_plan(probs, count, M, pl) == I2S_OK ? pl.total : 0;
}

// True if host address p lies in page-locked memory that the current device
// reaches at the same address (cudaHostAlloc / cudaMallocHost memory, or
// memory registered as mapped, under unified addressing).
static bool mapped_host(uintptr_t p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, (const void*)p) != cudaSuccess) {
        cudaGetLastError();   // clear the error this query may leave
        return false;
    }
    return at.type == cudaMemoryTypeHost && at.devicePointer == (void*)p;
}

int i2s_mul_mat_grouped_host_ex(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                                unsigned flags, i2s_stream_t stream) {
    if (flags & ~(unsigned)(I2S_HOST_MAPPED | I2S_HOST_MAPPED_Y)) return I2S_E_BAD_ARG;
    const bool map_y = (flags & I2S_HOST_MAPPED_Y) != 0u;
    HostPlan pl;
    int r = host_plan(probs, count, M, pl);
    if (r) return r;
    if (!ws) return I2S_E_NULL_PTR;
    if (!aligned256(ws)) return I2S_E_MISALIGNED;
    // mapped: the kernels read x and write y where they are, so only the
    // grouped workspace is needed
    if (ws_bytes < ((flags & I2S_HOST_MAPPED) ? pl.grouped : pl.total)) return I2S_E_WORKSPACE_TOO_SMALL;
    r = check_device();
    if (r) return r;
    if (flags & I2S_HOST_MAPPED) {
        for (const HostSpan& sp : pl.xs)
            if (!mapped_host(sp.lo) || !mapped_host(sp.hi - 1)) return I2S_E_BAD_ARG;
        for (const HostSpan& sp : pl.ys)
            if (!mapped_host(sp.lo) || !mapped_host(sp.hi - 1)) return I2S_E_BAD_ARG;
        return grouped_impl(probs, count, M, ws, pl.grouped, stream, 3);
    }
    if (map_y)
        for (const HostSpan& sp : pl.ys)
            if (!mapped_host(sp.lo) || !mapped_host(sp.hi - 1)) return I2S_E_BAD_ARG;
    char* base = (char*)ws;
    std::vector<i2s_problem> dev(probs, probs + count);
    for (i2s_problem& p : dev) {
        const HostSpan& sx = span_of(pl.xs, (uintptr_t)p.x);
        p.x = (const float*)(base + sx.off + ((uintptr_t)p.x - sx.lo));
        if (!map_y) {
            const HostSpan& sy = span_of(pl.ys, (uintptr_t)p.y);
            p.y = (float*)(base + sy.off + ((uintptr_t)p.y - sy.lo));
        }
    }
    for (const HostSpan& s : pl.xs) {
        r = cuda_status(cudaMemcpyAsync(base + s.off, (const void*)s.lo, s.hi - s.lo, cudaMemcpyHostToDevice, stream));
        if (r) return r;
    }
    r = grouped_impl(dev.data(), count, M, ws, pl.grouped, stream, 3);
    if (r || map_y) return r;
    for (const HostSpan& s : pl.ys) {
        r = cuda_status(cudaMemcpyAsync((void*)s.lo, base + s.off, s.hi - s.lo, cudaMemcpyDeviceToHost, stream));
        if (r) return r;
    }
    return I2S_OK;
}

int i2s_mul_mat_grouped_host(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                             i2s_stream_t stream) {
    return i2s_mul_mat_grouped_host_ex(probs, count, M, ws, ws_bytes, 0u, stream);
}

size_t i8s_ws_f32_offset(void) { return kHeader; }

static bool overlaps(const void* a, size_t na, const void* b, size_t nb);

// I8_S workspace: [header: status, amax][y F32 M x N][activations f16,
// rows_pad x K][weights f16, N x K][split-tile int32 sums, half-tiles x chunks
// slots of tm x 128][half-tile tickets][half-tile slot masks]. A tile is 256
// output features x tm activation rows (tm = 160 or 128, chosen per call),
// computed by a CTA pair; each CTA owns one 128-feature half. The workspace
// sizes are the larger of the two layouts, so they need no device.
static int64_t i8s_rows_pad(int64_t M, int tm) { return (M + tm - 1) / tm * tm; }
static int64_t i8s_tiles(int64_t M, int64_t N, int tm) {   // half-tiles: 128 features x tm rows
    return 2 * ((N + 2 * kI8sTileN - 1) / (2 * kI8sTileN)) * ((M + tm - 1) / tm);
}

static int64_t i8s_chunks(int64_t K) { return (K + kI8sChunkK - 1) / kI8sChunkK; }

// Ranges of whole tiles, in order, of at most L units each (a tile of matmul
// i is chunks_i units): the number of ranges, their bounds in `bounds`, or -1
// when a tile is larger than L or more than `max_ranges` ranges are needed.
static int pack_whole_tiles(const I8sTcArgs& a, int64_t L, int64_t max_ranges, int* bounds) {
    int ranges = 0;
    int64_t cur = 0, u = 0;
    bounds[0] = 0;
    for (int i = 0; i < a.count; ++i) {
        const int64_t c = a.p[i].chunks, n = (int64_t)a.p[i].n_wt * a.n_at;
        if (c > L) return -1;
        for (int64_t t = 0; t < n; ++t) {
            if (cur + c > L) {   // close the range before this tile
                if (++ranges >= max_ranges) return -1;
                bounds[ranges] = (int)u;
                cur = 0;
            }
            cur += c;
            u += c;
        }
    }
    bounds[++ranges] = (int)u;
    return ranges;
}

// The CTA pairs of a launch and their unit ranges (a.bounds; a.total_units
// and the matmuls' tiles set). An even split over the resident pairs gives the
// busiest pair L0 = ceil(units / resident) units. Whole tiles are packed into
// ranges of at most L units for the smallest L in [L0, 4 L0 / 3] that needs
// no more than the resident pairs, so that no tile is cut between pairs: a
// cut tile stores and reloads an 80 KB slot of int32 sums per CTA, while the
// pairs share L2 bandwidth and the ones left idle cost little. The encoder's
// FC1 (tiles of 2 units) runs as 64 pairs of 3 tiles, FC2 (8 units) as 48
// pairs of one tile. Without such an L, the units are split evenly over the
// fewest pairs that keep L0.
static int i8s_plan_pairs(I8sTcArgs& a) {
    const int64_t units = a.total_units;
    int64_t resident = i8s_gemm_tc_max_pairs();
    resident = std::max<int64_t>(1, std::min<int64_t>(resident, kI8sMaxPairs));
    const int64_t L0 = (units + resident - 1) / resident;
    int64_t tiles = 0;
    for (int i = 0; i < a.count; ++i) tiles += (int64_t)a.p[i].n_wt * a.n_at;
    if (tiles <= 65536)   // bounds the host work of the search
        for (int64_t L = L0; 3 * L <= 4 * L0; ++L) {
            const int pairs = pack_whole_tiles(a, L, resident, a.bounds);
            if (pairs > 0) return pairs;
        }
    const int pairs = (int)((units + L0 - 1) / L0);
    for (int q = 0; q <= pairs; ++q) a.bounds[q] = (int)(((int64_t)q * units) / pairs);
    return pairs;
}

// the tile height of a launch over these matmuls (the resident pairs decide)
// The tile height of a launch. The busiest CTA pair's work bounds the
// kernel, and a unit moves 256 weight rows and tm activation rows of operands
// through shared memory per K position. For each height the pair ranges are
// planned as the launch plans them (whole tiles where it can), and the height
// whose busiest pair moves fewer operand rows wins, 160 on a tie. (Counting
// units as if they were split evenly would favour 160 for the encoder's FC2,
// whose whole tiles then run on 48 pairs of 8 x 416 rows, against 64 pairs of
// 8 x 384 rows with 128-row tiles.)
static int i8s_pick_tile(int64_t M, const int64_t* N, const int64_t* K, int count) {
    static thread_local I8sTcArgs t;
    int best = kI8sTileM;
    int64_t best_cost = -1;
    for (int tm : {kI8sTileM, kI8sTileMSmall}) {
        t.count = count;
        t.n_at = (int)((M + tm - 1) / tm);
        int64_t units = 0;
        for (int i = 0; i < count; ++i) {
            t.p[i].n_wt = (int)((N[i] + 2 * kI8sTileN - 1) / (2 * kI8sTileN));
            t.p[i].chunks = (int)i8s_chunks(K[i]);
            units += (int64_t)t.p[i].n_wt * t.n_at * t.p[i].chunks;
        }
        if (units >= ((int64_t)1 << 30)) return i8s_tile_m(M, N, K, count, i8s_gemm_tc_max_pairs());
        t.total_units = (int)units;
        const int pairs = i8s_plan_pairs(t);
        int64_t busiest = 0;
        for (int q = 0; q < pairs; ++q) busiest = std::max<int64_t>(busiest, t.bounds[q + 1] - t.bounds[q]);
        const int64_t cost = busiest * (2 * kI8sTileN + tm);
        if (best_cost < 0 || cost < best_cost) best_cost = cost, best = tm;
    }
    return best;
}

// K is the operand row length i8s_kpad(K) wherever f16 rows are sized.
static size_t i8s_ws_for(int64_t M, int64_t N, int64_t K, int tm) {
    K = i8s_kpad(K);
    const size_t tiles = (size_t)i8s_tiles(M, N, tm);
    return kHeader + align_up((size_t)M * (size_t)N * 4) + align_up((size_t)i8s_rows_pad(M, tm) * (size_t)K * 2) +
           align_up((size_t)N * (size_t)K * 2) + align_up(tiles * (size_t)i8s_chunks(K) * kI8sTileN * tm * 4) +
           align_up(tiles * 4) + align_up(tiles * 8);
}

size_t i8s_mul_mat_workspace(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1 || i8s_kpad(K) > kI8sMaxK) return 0;
    return std::max(i8s_ws_for(M, N, K, kI8sTileM), i8s_ws_for(M, N, K, kI8sTileMSmall));
}

// The I8_S call over f16 weight rows wf: either converted from w_i8s into the
// workspace by this call's pre-pass (w_i8s set), or packed earlier (w_i8s
// null, wf the caller's packed rows). w_scale points at the weight scale.
static int i8s_run(const int8_t* w_i8s, const __half* wf_packed, const float* w_scale, int64_t N, int64_t K,
                   const void* x_i8s, int64_t M, const float* bias, int relu, void* y_i8s, void* ws,
                   i2s_stream_t stream) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    unsigned int* amax = reinterpret_cast<unsigned int*>(base + kAmaxOff);
    uint32_t* status = reinterpret_cast<uint32_t*>(base + kStatusOff);
    float* yf = reinterpret_cast<float*>(base + kHeader);
    const int64_t Kx = K;         // the activation's own K (its scale trailer follows M*Kx bytes)
    K = i8s_kpad(K);              // operand row length from here on
    const int tm = i8s_pick_tile(M, &N, &K, 1);
    const int64_t rows_pad = i8s_rows_pad(M, tm);
    const size_t tiles = (size_t)i8s_tiles(M, N, tm);
    const size_t xf_off = kHeader + align_up((size_t)M * (size_t)N * 4);
    const size_t wf_off = xf_off + align_up((size_t)rows_pad * (size_t)K * 2);
    const size_t part_off = wf_off + (w_i8s ? align_up((size_t)N * (size_t)K * 2) : 0);
    const size_t tick_off = part_off + align_up(tiles * (size_t)i8s_chunks(K) * kI8sTileN * tm * 4);
    const size_t mask_off = tick_off + align_up(tiles * 4);
    const size_t zero_bytes = mask_off + align_up(tiles * 8) - tick_off;   // tickets and masks (slots need no clearing)
    __half* xf = reinterpret_cast<__half*>(base + xf_off);
    const __half* wf = w_i8s ? reinterpret_cast<__half*>(base + wf_off) : wf_packed;
    // pre-pass: weights (unless packed) and activations to f16 rows, once per
    // call; clears the status and amax words and the split-tile tickets
    int r = cuda_status(launch_i8s_to_f16(w_i8s, w_i8s ? (int)N : 0, reinterpret_cast<__half*>(base + wf_off),
                                          static_cast<const int8_t*>(x_i8s), (int)M, (int)rows_pad, (int)Kx, xf,
                                          base + tick_off, zero_bytes, status, amax, stream));
    if (r) return r;
    static thread_local I8sTcArgs a;
    I8sProb& P = a.p[0];
    if (!make_f16_operand_map(&P.xmap, xf, (int)rows_pad, (int)K, tm / 2)) return I2S_E_CUDA;
    if (!make_f16_operand_map(&P.wmap, wf, (int)N, (int)K, kI8sTileN)) return I2S_E_CUDA;
    P.w_scale_ptr = w_scale;
    P.x_scale_ptr = reinterpret_cast<const float*>(static_cast<const uint8_t*>(x_i8s) + i8s_scale_offset(M * Kx));
    P.bias = bias;
    P.row_scale = nullptr;
    P.col_scale = nullptr;
    P.y = yf;
    P.slot0 = 0;
    P.N = (int)N;
    P.K = (int)K;
    P.n_wt = (int)((N + 2 * kI8sTileN - 1) / (2 * kI8sTileN));   // 256-feature tiles
    P.chunks = (int)i8s_chunks(K);
    P.unit0 = 0;
    P.ht0 = 0;
    a.count = 1;
    a.amax_bits = amax;
    a.part = reinterpret_cast<int32_t*>(base + part_off);
    a.tickets = reinterpret_cast<uint32_t*>(base + tick_off);
    a.slot_masks = reinterpret_cast<unsigned long long*>(base + mask_off);
    a.status = status;
    a.M = (int)M;
    a.relu = relu ? 1 : 0;
    a.tile_m = tm;
    a.n_at = (int)(rows_pad / tm);
    a.total_units = (int)(tiles / 2) * P.chunks;   // units of whole (256-feature) tiles
    const int grid = 2 * i8s_plan_pairs(a);   // at most the resident pairs, clusters of two CTAs
    r = cuda_status(launch_i8s_gemm_tc(a, grid, stream));
    if (r) return r;
    return cuda_status(launch_requant(yf, M * N, amax, static_cast<uint8_t*>(y_i8s), stream));
}

static int i8s_check(const void* w, int64_t N, int64_t K, const void* x_i8s, int64_t M, const float* bias,
                     const void* y_i8s, const void* ws) {
    if (!w || !x_i8s || !y_i8s || !ws) return I2S_E_NULL_PTR;
    if (M < 1 || N < 1 || K < 1 || i8s_kpad(K) > kI8sMaxK) return I2S_E_BAD_SHAPE;
    if (M * K >= ((int64_t)1 << 31) || N * K >= ((int64_t)1 << 31) || M * N >= ((int64_t)1 << 31))
        return I2S_E_BAD_SHAPE;
    if (!aligned16(w) || !aligned16(x_i8s) || !aligned16(y_i8s) || !aligned256(ws) || (bias && ((uintptr_t)bias & 3u)))
        return I2S_E_MISALIGNED;
    return I2S_OK;
}

int i8s_mul_mat_add_relu(const void* w_i8s, int64_t N, int64_t K, const void* x_i8s, int64_t M, const float* bias,
                         int relu, void* y_i8s, void* ws, size_t ws_bytes, i2s_stream_t stream) {
    int r = i8s_check(w_i8s, N, K, x_i8s, M, bias, y_i8s, ws);
    if (r) return r;
    if (ws_bytes < i8s_mul_mat_workspace(M, N, K)) return I2S_E_WORKSPACE_TOO_SMALL;
    r = check_device();
    if (r) return r;
    const float* w_scale =
        reinterpret_cast<const float*>(static_cast<const uint8_t*>(w_i8s) + i8s_scale_offset(N * K));
    return i8s_run(static_cast<const int8_t*>(w_i8s), nullptr, w_scale, N, K, x_i8s, M, bias, relu, y_i8s, ws, stream);
}

size_t i8s_packed_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1 || i8s_kpad(K) > kI8sMaxK || N * i8s_kpad(K) >= ((int64_t)1 << 31)) return 0;
    return (size_t)N * (size_t)i8s_kpad(K) * 2 + 16;
}

int i8s_pack_weights(const void* w_i8s, int64_t N, int64_t K, void* packed, i2s_stream_t stream) {
    if (!w_i8s || !packed) return I2S_E_NULL_PTR;
    if (i8s_packed_bytes(N, K) == 0) return I2S_E_BAD_SHAPE;
    if (!aligned16(w_i8s) || !aligned16(packed)) return I2S_E_MISALIGNED;
    if (overlaps(w_i8s, i8s_nbytes(N * K), packed, i8s_packed_bytes(N, K))) return I2S_E_BAD_ARG;
    int r = check_device();
    if (r) return r;
    uint8_t* dst = static_cast<uint8_t*>(packed);
    const int64_t Kp = i8s_kpad(K);
    r = cuda_status(K == Kp ? launch_i8_to_f16(static_cast<const int8_t*>(w_i8s), N * K, reinterpret_cast<__half*>(dst), stream)
                            : launch_i8_to_f16_rows(static_cast<const int8_t*>(w_i8s), N, K, reinterpret_cast<__half*>(dst),
                                                    stream));
    if (r) return r;
    // the 16-byte trailer: the weight scale, then zeros
    r = cuda_status(cudaMemsetAsync(dst + (size_t)N * Kp * 2, 0, 16, stream));
    if (r) return r;
    return cuda_status(cudaMemcpyAsync(dst + (size_t)N * Kp * 2, static_cast<const uint8_t*>(w_i8s) + i8s_scale_offset(N * K),
                                       4, cudaMemcpyDeviceToDevice, stream));
}

size_t i8s_mul_mat_packed_workspace(int64_t M, int64_t N, int64_t K) {
    const size_t full = i8s_mul_mat_workspace(M, N, K);
    return full == 0 ? 0 : full - align_up((size_t)N * (size_t)i8s_kpad(K) * 2);
}

int i8s_mul_mat_add_relu_packed(const void* packed, int64_t N, int64_t K, const void* x_i8s, int64_t M,
                                const float* bias, int relu, void* y_i8s, void* ws, size_t ws_bytes,
                                i2s_stream_t stream) {
    int r = i8s_check(packed, N, K, x_i8s, M, bias, y_i8s, ws);
    if (r) return r;
    if (ws_bytes < i8s_mul_mat_packed_workspace(M, N, K)) return I2S_E_WORKSPACE_TOO_SMALL;
    r = check_device();
    if (r) return r;
    const uint8_t* p = static_cast<const uint8_t*>(packed);
    return i8s_run(nullptr, reinterpret_cast<const __half*>(p),
                   reinterpret_cast<const float*>(p + (size_t)N * i8s_kpad(K) * 2), N, K, x_i8s, M, bias, relu, y_i8s, ws,
                   stream);
}

size_t i8s_requant_workspace(int64_t n) { return n < 1 ? 0 : kHeader; }

int i8s_requant(const float* y, int64_t n, void* dst_i8s, void* ws, size_t ws_bytes, i2s_stream_t stream) {
    if (!y || !dst_i8s || !ws) return I2S_E_NULL_PTR;
    if (n < 1 || n >= ((int64_t)1 << 40)) return I2S_E_BAD_SHAPE;
    if (!aligned16(y) || !aligned16(dst_i8s) || !aligned256(ws)) return I2S_E_MISALIGNED;
    if (ws_bytes < i8s_requant_workspace(n)) return I2S_E_WORKSPACE_TOO_SMALL;
    int r = check_device();
    if (r) return r;
    unsigned int* amax = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + kAmaxOff);
    r = cuda_status(cudaMemsetAsync(amax, 0, 4, stream));
    if (r) return r;
    r = cuda_status(launch_absmax(y, n, amax, stream));
    if (r) return r;
    return cuda_status(launch_requant(y, n, amax, static_cast<uint8_t*>(dst_i8s), stream));
}

// ---------------------------------------------------------------------------
// I8_S element-wise ops, convolution pieces and W8A8. Workspace of the
// element-wise ops: [header: status, amax][row factors, rows F32].
// ---------------------------------------------------------------------------

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

size_t i8s_eltwise_workspace(int64_t rows) {
    return rows < 1 ? 0 : kHeader + align_up((size_t)rows * 4);
}

int i8s_add_scaled(const void* a_i8s, const void* b_i8s, int64_t n, void* y_i8s, void* ws, size_t ws_bytes,
                   i2s_stream_t stream) {
    if (!a_i8s || !b_i8s || !y_i8s || !ws) return I2S_E_NULL_PTR;
    if (n < 1 || n >= ((int64_t)1 << 40)) return I2S_E_BAD_SHAPE;
    if (!aligned16(a_i8s) || !aligned16(b_i8s) || !aligned16(y_i8s) || !aligned256(ws)) return I2S_E_MISALIGNED;
    const size_t nb = i8s_nbytes(n);
    if (overlaps(y_i8s, nb, a_i8s, nb) || overlaps(y_i8s, nb, b_i8s, nb)) return I2S_E_BAD_ARG;
    if (ws_bytes < i8s_eltwise_workspace(1)) return I2S_E_WORKSPACE_TOO_SMALL;
    int r = check_device();
    if (r) return r;
    unsigned int* amax = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + kAmaxOff);
    r = cuda_status(cudaMemsetAsync(amax, 0, 4, stream));
    if (r) return r;
    return cuda_status(launch_add_scaled(static_cast<const uint8_t*>(a_i8s), static_cast<const uint8_t*>(b_i8s), n,
                                         amax, static_cast<uint8_t*>(y_i8s), stream));
}

int i8s_rms_norm_scaled(const void* x_i8s, int64_t rows, int64_t ne0, float eps, const float* gamma, void* y_i8s,
                        void* ws, size_t ws_bytes, i2s_stream_t stream) {
    if (!x_i8s || !y_i8s || !ws) return I2S_E_NULL_PTR;
    if (rows < 1 || ne0 < 1 || ne0 > 131072 || rows * ne0 >= ((int64_t)1 << 40) || !(eps >= 0.0f))
        return I2S_E_BAD_SHAPE;
    if (!aligned16(x_i8s) || !aligned16(y_i8s) || !aligned256(ws) || (gamma && ((uintptr_t)gamma & 3u)))
        return I2S_E_MISALIGNED;
    const size_t nb = i8s_nbytes(rows * ne0);
    if (overlaps(y_i8s, nb, x_i8s, nb)) return I2S_E_BAD_ARG;
    if (ws_bytes < i8s_eltwise_workspace(rows)) return I2S_E_WORKSPACE_TOO_SMALL;
    int r = check_device();
    if (r) return r;
    uint8_t* base = static_cast<uint8_t*>(ws);
    unsigned int* amax = reinterpret_cast<unsigned int*>(base + kAmaxOff);
    r = cuda_status(cudaMemsetAsync(amax, 0, 4, stream));
    if (r) return r;
    return cuda_status(launch_rms_norm_scaled(static_cast<const uint8_t*>(x_i8s), rows, ne0, eps, gamma,
                                              reinterpret_cast<float*>(base + kHeader), amax,
                                              static_cast<uint8_t*>(y_i8s), stream));
}

int i8s_transpose(const void* src_i8s, int64_t a, int64_t b, void* dst_i8s, i2s_stream_t stream) {
    if (!src_i8s || !dst_i8s) return I2S_E_NULL_PTR;
    if (a < 1 || b < 1 || a * b >= ((int64_t)1 << 40) || ((a + 31) / 32) * ((b + 31) / 32) >= ((int64_t)1 << 31))
        return I2S_E_BAD_SHAPE;
    const size_t nb = i8s_nbytes(a * b);
    if (overlaps(dst_i8s, nb, src_i8s, nb)) return I2S_E_BAD_ARG;
    int r = check_device();
    if (r) return r;
    return cuda_status(launch_i8s_transpose(static_cast<const uint8_t*>(src_i8s), a, b,
                                            static_cast<uint8_t*>(dst_i8s), stream));
}

int64_t i8s_im2col_out_len(int64_t L, int64_t KW, int64_t stride, int64_t pad_l, int64_t pad_r) {
    if (L < 1 || KW < 1 || stride < 1 || pad_l < 0 || pad_r < 0) return 0;
    const int64_t span = L + pad_l + pad_r - KW;
    return span < 0 ? 0 : span / stride + 1;
}

static bool conv_shape_ok(int64_t C, int64_t L, int64_t KW, int64_t stride, int64_t pad_l, int64_t pad_r) {
    if (C < 1 || L < 1 || KW < 1 || stride < 1 || pad_l < 0 || pad_r < 0) return false;
    if (KW > 65536 || stride > 65536 || pad_l > 65536 || pad_r > 65536) return false;
    const int64_t OL = i8s_im2col_out_len(L, KW, stride, pad_l, pad_r);
    const int64_t lim = (int64_t)1 << 31;
    return OL >= 1 && C * L < lim && OL * C * KW < lim && C * OL < lim && L + pad_l + pad_r < lim;
}

int i8s_im2col_asym(const void* src_i8s, int64_t C, int64_t L, int64_t KW, int64_t stride, int64_t pad_l,
                    int64_t pad_r, void* dst_i8s, i2s_stream_t stream) {
    if (!src_i8s || !dst_i8s) return I2S_E_NULL_PTR;
    if (!conv_shape_ok(C, L, KW, stride, pad_l, pad_r)) return I2S_E_BAD_SHAPE;
    if (!aligned16(dst_i8s)) return I2S_E_MISALIGNED;
    const int64_t OL = i8s_im2col_out_len(L, KW, stride, pad_l, pad_r);
    if (overlaps(dst_i8s, i8s_nbytes(OL * C * KW), src_i8s, i8s_nbytes(C * L))) return I2S_E_BAD_ARG;
    int r = check_device();
    if (r) return r;
    return cuda_status(launch_im2col_asym(static_cast<const uint8_t*>(src_i8s), C, L, (int)KW, (int)stride,
                                          (int)pad_l, OL, static_cast<uint8_t*>(dst_i8s), stream));
}

int i8s_depthwise_mul_mat_add(const void* w_i8s, int64_t KW, const void* x_i8s, int64_t C, int64_t L,
                              int64_t stride, int64_t pad_l, int64_t pad_r, const float* bias, int relu,
                              void* y_i8s, void* ws, size_t ws_bytes, i2s_stream_t stream) {
    if (!w_i8s || !x_i8s || !y_i8s || !ws) return I2S_E_NULL_PTR;
    if (!conv_shape_ok(C, L, KW, stride, pad_l, pad_r)) return I2S_E_BAD_SHAPE;
    if (!aligned16(y_i8s) || !aligned256(ws) || (bias && ((uintptr_t)bias & 3u))) return I2S_E_MISALIGNED;
    const int64_t OL = i8s_im2col_out_len(L, KW, stride, pad_l, pad_r);
    const size_t ny = i8s_nbytes(C * OL);
    if (overlaps(y_i8s, ny, x_i8s, i8s_nbytes(C * L)) || overlaps(y_i8s, ny, w_i8s, i8s_nbytes(C * KW)))
        return I2S_E_BAD_ARG;
    if (ws_bytes < i8s_eltwise_workspace(1)) return I2S_E_WORKSPACE_TOO_SMALL;
    int r = check_device();
    if (r) return r;
    unsigned int* amax = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + kAmaxOff);
    r = cuda_status(cudaMemsetAsync(amax, 0, 4, stream));
    if (r) return r;
    return cuda_status(launch_depthwise(static_cast<const uint8_t*>(w_i8s), static_cast<const uint8_t*>(x_i8s), bias,
                                        C, L, (int)KW, (int)stride, (int)pad_l, OL, relu ? 1 : 0, amax,
                                        static_cast<uint8_t*>(y_i8s), stream));
}

int w8a8_quantize_weights(const float* w, int64_t N, int64_t K, int8_t* wq, float* bscale, i2s_stream_t stream) {
    if (!w || !wq || !bscale) return I2S_E_NULL_PTR;
    if (N < 1 || K < 1 || N * K >= ((int64_t)1 << 40) || N >= ((int64_t)1 << 31)) return I2S_E_BAD_SHAPE;
    if (((uintptr_t)w & 3u) || ((uintptr_t)bscale & 3u)) return I2S_E_MISALIGNED;
    int r = check_device();
    if (r) return r;
    return cuda_status(launch_w8a8_weights(w, N, K, wq, bscale, stream));
}

// The I8_S tensor-core GEMM with the W8A8 epilogue over f16 operands already
// in place (xf: rows_pad x K, wf: N x K); the split-tile areas of the
// workspace start at part_off and were cleared by the launch before.
static int launch_w8a8_gemm(const __half* wf, const float* bscale, const float* ascale, const __half* xf, int64_t N,
                            int64_t K, int64_t M, int tm, float* d, uint8_t* base, size_t part_off,
                            i2s_stream_t stream) {
    const int64_t rows_pad = i8s_rows_pad(M, tm);
    const size_t tiles = (size_t)i8s_tiles(M, N, tm);
    const size_t tick_off = part_off + align_up(tiles * (size_t)i8s_chunks(K) * kI8sTileN * tm * 4);
    const size_t mask_off = tick_off + align_up(tiles * 4);
    static thread_local I8sTcArgs a;
    I8sProb& P = a.p[0];
    if (!make_f16_operand_map(&P.xmap, xf, (int)rows_pad, (int)K, tm / 2)) return I2S_E_CUDA;
    if (!make_f16_operand_map(&P.wmap, wf, (int)N, (int)K, kI8sTileN)) return I2S_E_CUDA;
    P.w_scale_ptr = bscale;   // read by the kernel's I8_S path; the W8A8 epilogue uses the arrays
    P.x_scale_ptr = ascale;
    P.bias = nullptr;
    P.row_scale = ascale;
    P.col_scale = bscale;
    P.y = d;
    P.slot0 = 0;
    P.N = (int)N;
    P.K = (int)K;
    P.n_wt = (int)((N + 2 * kI8sTileN - 1) / (2 * kI8sTileN));
    P.chunks = (int)i8s_chunks(K);
    P.unit0 = 0;
    P.ht0 = 0;
    a.count = 1;
    a.amax_bits = reinterpret_cast<unsigned int*>(base + kAmaxOff);
    a.part = reinterpret_cast<int32_t*>(base + part_off);
    a.tickets = reinterpret_cast<uint32_t*>(base + tick_off);
    a.slot_masks = reinterpret_cast<unsigned long long*>(base + mask_off);
    a.status = reinterpret_cast<uint32_t*>(base + kStatusOff);
    a.M = (int)M;
    a.relu = 0;
    a.tile_m = tm;
    a.n_at = (int)(rows_pad / tm);
    a.total_units = (int)(tiles / 2) * P.chunks;
    return cuda_status(launch_i8s_gemm_tc(a, 2 * i8s_plan_pairs(a), stream));
}

// bytes of the GEMM's split-tile areas (slots, tickets, masks)
static size_t w8a8_split_bytes(int64_t M, int64_t N, int64_t K, int tm) {
    const size_t tiles = (size_t)i8s_tiles(M, N, tm);
    return align_up(tiles * (size_t)i8s_chunks(K) * kI8sTileN * tm * 4) + align_up(tiles * 4) + align_up(tiles * 8);
}

static bool w8a8_shape_ok(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1 || i8s_kpad(K) > kI8sMaxK) return false;
    const int64_t Kp = i8s_kpad(K);
    return M * Kp < ((int64_t)1 << 31) && N * Kp < ((int64_t)1 << 31) && M * N < ((int64_t)1 << 31);
}

// W8A8 workspace (int8 weights): [header: status, amax][activations int8,
// M x K][row scales, M F32][activations f16, rows_pad x Kp][weights f16,
// N x Kp][split-tile slots, tickets, masks], Kp = i8s_kpad(K).
static size_t w8a8_front(int64_t M, int64_t K) { return kHeader + align_up((size_t)M * K) + align_up((size_t)M * 4); }

static size_t w8a8_ws_for(int64_t M, int64_t N, int64_t K, int tm) {
    const int64_t Kp = i8s_kpad(K);
    return w8a8_front(M, K) + align_up((size_t)i8s_rows_pad(M, tm) * (size_t)Kp * 2) +
           align_up((size_t)N * (size_t)Kp * 2) + w8a8_split_bytes(M, N, Kp, tm);
}

size_t w8a8_mul_mat_workspace(int64_t M, int64_t N, int64_t K) {
    if (!w8a8_shape_ok(M, N, K)) return 0;
    return std::max(w8a8_ws_for(M, N, K, kI8sTileM), w8a8_ws_for(M, N, K, kI8sTileMSmall));
}

int w8a8_mul_mat(const int8_t* wq, const float* bscale, int64_t N, int64_t K, const float* x, int64_t M, float* d,
                 void* ws, size_t ws_bytes, i2s_stream_t stream) {
    if (!wq || !bscale || !x || !d || !ws) return I2S_E_NULL_PTR;
    if (!w8a8_shape_ok(M, N, K)) return I2S_E_BAD_SHAPE;
    if (!aligned16(wq) || !aligned16(x) || !aligned16(d) || !aligned256(ws) || ((uintptr_t)bscale & 3u))
        return I2S_E_MISALIGNED;
    if (ws_bytes < w8a8_mul_mat_workspace(M, N, K)) return I2S_E_WORKSPACE_TOO_SMALL;
    int r = check_device();
    if (r) return r;
    uint8_t* base = static_cast<uint8_t*>(ws);
    unsigned int* amax = reinterpret_cast<unsigned int*>(base + kAmaxOff);
    uint32_t* status = reinterpret_cast<uint32_t*>(base + kStatusOff);
    int8_t* xq = reinterpret_cast<int8_t*>(base + kHeader);
    float* ascale = reinterpret_cast<float*>(base + kHeader + align_up((size_t)M * K));
    int64_t Kp = i8s_kpad(K);   // operand row length (the tail zero-filled by the pre-pass)
    const int tm = i8s_pick_tile(M, &N, &Kp, 1);
    const int64_t rows_pad = i8s_rows_pad(M, tm);
    const size_t xf_off = w8a8_front(M, K);
    const size_t wf_off = xf_off + align_up((size_t)rows_pad * (size_t)Kp * 2);
    const size_t part_off = wf_off + align_up((size_t)N * (size_t)Kp * 2);
    const size_t tiles = (size_t)i8s_tiles(M, N, tm);
    const size_t tick_off = part_off + align_up(tiles * (size_t)i8s_chunks(Kp) * kI8sTileN * tm * 4);
    const size_t zero_bytes = w8a8_split_bytes(M, N, Kp, tm) - (tick_off - part_off);   // tickets and masks
    __half* xf = reinterpret_cast<__half*>(base + xf_off);
    __half* wf = reinterpret_cast<__half*>(base + wf_off);
    // per-row activation quantization (1e-9 floor), then the int8 rows and
    // weights to f16 (the pre-pass also clears the status word and the
    // split-tile tickets), then the tensor-core GEMM with the W8A8 epilogue
    r = cuda_status(launch_w8a8_rows(x, M, K, xq, ascale, stream));
    if (r) return r;
    r = cuda_status(launch_i8s_to_f16(wq, (int)N, wf, xq, (int)M, (int)rows_pad, (int)K, xf, base + tick_off, zero_bytes,
                                      status, amax, stream));
    if (r) return r;
    return launch_w8a8_gemm(wf, bscale, ascale, xf, N, Kp, M, tm, d, base, part_off, stream);
}

size_t w8a8_packed_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1 || i8s_kpad(K) > kI8sMaxK || N * i8s_kpad(K) >= ((int64_t)1 << 31)) return 0;
    return (size_t)N * (size_t)i8s_kpad(K) * 2;
}

int w8a8_pack_weights(const int8_t* wq, int64_t N, int64_t K, void* packed, i2s_stream_t stream) {
    if (!wq || !packed) return I2S_E_NULL_PTR;
    if (w8a8_packed_bytes(N, K) == 0) return I2S_E_BAD_SHAPE;
    if (!aligned16(wq) || !aligned16(packed)) return I2S_E_MISALIGNED;
    if (overlaps(wq, (size_t)N * K, packed, w8a8_packed_bytes(N, K))) return I2S_E_BAD_ARG;
    int r = check_device();
    if (r) return r;
    if (K % 64 == 0) return cuda_status(launch_i8_to_f16(wq, N * K, static_cast<__half*>(packed), stream));
    return cuda_status(launch_i8_to_f16_rows(wq, N, K, static_cast<__half*>(packed), stream));
}

// Packed W8A8 calls, one matmul or a group of them with the same M. Workspace:
// [header: status, amax][per distinct activation (x, K): row scales, M F32;
// f16 operand rows, rows_pad x K][split-tile slots of every matmul][half-tile
// tickets][half-tile slot masks]. Matmuls whose x pointer and K are equal
// share one quantized activation.
namespace {
struct W8a8Plan {
    int n_act = 0;
    int act_of[kI8sMaxGroup];
    size_t act_off[kI8sMaxGroup];   // row scales; the f16 rows follow at align_up(M * 4)
    size_t slots = 0, tiles = 0;    // slots (tm x kI8sTileN int32 each), half-tiles
    size_t part_off = 0, tick_off = 0, mask_off = 0, end = 0;
};
}  // namespace

static_assert(kI8sMaxGroup == W8A8_MAX_GROUP, "one GEMM launch holds every matmul of a group");

static W8a8Plan w8a8_plan(const w8a8_problem* probs, int count, int64_t M, int tm) {
    W8a8Plan pl;
    const int64_t rows_pad = i8s_rows_pad(M, tm);
    size_t off = kHeader;
    for (int i = 0; i < count; ++i) {
        int a = -1;
        for (int j = 0; j < i; ++j)
            if (probs[j].x == probs[i].x && probs[j].K == probs[i].K) { a = pl.act_of[j]; break; }
        if (a < 0) {
            a = pl.n_act++;
            pl.act_off[a] = off;
            off += align_up((size_t)M * 4) + align_up((size_t)rows_pad * (size_t)i8s_kpad(probs[i].K) * 2);
        }
        pl.act_of[i] = a;
        const size_t ht = (size_t)i8s_tiles(M, probs[i].N, tm);
        pl.tiles += ht;
        pl.slots += ht * (size_t)i8s_chunks(i8s_kpad(probs[i].K));
    }
    pl.part_off = off;
    pl.tick_off = pl.part_off + align_up(pl.slots * kI8sTileN * tm * 4);
    pl.mask_off = pl.tick_off + align_up(pl.tiles * 4);
    pl.end = pl.mask_off + align_up(pl.tiles * 8);
    return pl;
}

static int w8a8_group_ok(const w8a8_problem* probs, int count, int64_t M) {
    if (!probs) return I2S_E_NULL_PTR;
    if (count < 1 || count > W8A8_MAX_GROUP) return I2S_E_BAD_ARG;
    int64_t units = 0;
    for (int i = 0; i < count; ++i) {
        const w8a8_problem& q = probs[i];
        if (!q.packed || !q.bscale || !q.x || !q.d) return I2S_E_NULL_PTR;
        if (!w8a8_shape_ok(M, q.N, q.K)) return I2S_E_BAD_SHAPE;
        if (!aligned16(q.packed) || !aligned16(q.x) || !aligned16(q.d) || ((uintptr_t)q.bscale & 3u))
            return I2S_E_MISALIGNED;
        units += (int64_t)i8s_tiles(M, q.N, kI8sTileMSmall) / 2 * i8s_chunks(i8s_kpad(q.K));   // the more numerous
    }
    return units < ((int64_t)1 << 30) ? I2S_OK : I2S_E_BAD_SHAPE;
}

size_t w8a8_mul_mat_grouped_workspace(const w8a8_problem* probs, int count, int64_t M) {
    if (w8a8_group_ok(probs, count, M) != I2S_OK) return 0;
    return std::max(w8a8_plan(probs, count, M, kI8sTileM).end, w8a8_plan(probs, count, M, kI8sTileMSmall).end);
}

int w8a8_mul_mat_grouped(const w8a8_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                         i2s_stream_t stream) {
    int r = w8a8_group_ok(probs, count, M);
    if (r) return r;
    if (!ws) return I2S_E_NULL_PTR;
    if (!aligned256(ws)) return I2S_E_MISALIGNED;
    if (ws_bytes < w8a8_mul_mat_grouped_workspace(probs, count, M)) return I2S_E_WORKSPACE_TOO_SMALL;
    r = check_device();
    if (r) return r;
    int64_t Ns[kI8sMaxGroup], Ks[kI8sMaxGroup];
    for (int i = 0; i < count; ++i) Ns[i] = probs[i].N, Ks[i] = i8s_kpad(probs[i].K);
    const int tm = i8s_pick_tile(M, Ns, Ks, count);
    const W8a8Plan pl = w8a8_plan(probs, count, M, tm);
    uint8_t* base = static_cast<uint8_t*>(ws);
    const int64_t rows_pad = i8s_rows_pad(M, tm);
    // one launch quantizes every distinct activation into its f16 operand
    // rows (and clears the status, amax and split-tile counters)
    static thread_local W8a8RowJobs J;
    J.count = pl.n_act;
    J.M = (int)M;
    J.rows_pad = (int)rows_pad;
    for (int i = 0; i < count; ++i) {
        const int a = pl.act_of[i];
        J.x[a] = probs[i].x;
        J.K[a] = (int)probs[i].K;
        J.ascale[a] = reinterpret_cast<float*>(base + pl.act_off[a]);
        J.xf[a] = reinterpret_cast<__half*>(base + pl.act_off[a] + align_up((size_t)M * 4));
    }
    J.zero = reinterpret_cast<uint4*>(base + pl.tick_off);
    J.zero_16 = (pl.end - pl.tick_off) / 16;
    J.status = reinterpret_cast<uint32_t*>(base + kStatusOff);
    J.amax_bits = reinterpret_cast<unsigned int*>(base + kAmaxOff);
    r = cuda_status(launch_w8a8_rows_f16(J, stream));
    if (r) return r;
    // one tensor-core GEMM over every matmul, units numbered matmul by matmul
    static thread_local I8sTcArgs a;
    int units = 0, ht = 0;
    long long slot = 0;
    for (int i = 0; i < count; ++i) {
        const w8a8_problem& q = probs[i];
        I8sProb& P = a.p[i];
        const int act = pl.act_of[i];
        const int Kp = (int)i8s_kpad(q.K);   // operand row length
        if (!make_f16_operand_map(&P.xmap, J.xf[act], (int)rows_pad, Kp, tm / 2)) return I2S_E_CUDA;
        if (!make_f16_operand_map(&P.wmap, q.packed, (int)q.N, Kp, kI8sTileN)) return I2S_E_CUDA;
        P.w_scale_ptr = q.bscale;   // read by the kernel's I8_S path; the W8A8 epilogue uses the arrays
        P.x_scale_ptr = J.ascale[act];
        P.bias = nullptr;
        P.row_scale = J.ascale[act];
        P.col_scale = q.bscale;
        P.y = q.d;
        P.N = (int)q.N;
        P.K = Kp;
        P.n_wt = (int)((q.N + 2 * kI8sTileN - 1) / (2 * kI8sTileN));
        P.chunks = (int)i8s_chunks(Kp);
        P.unit0 = units;
        P.ht0 = ht;
        P.slot0 = slot;
        const int tiles_i = (int)i8s_tiles(M, q.N, tm);   // half-tiles
        units += tiles_i / 2 * P.chunks;
        ht += tiles_i;
        slot += (long long)tiles_i * P.chunks;
    }
    a.count = count;
    a.amax_bits = J.amax_bits;
    a.part = reinterpret_cast<int32_t*>(base + pl.part_off);
    a.tickets = reinterpret_cast<uint32_t*>(base + pl.tick_off);
    a.slot_masks = reinterpret_cast<unsigned long long*>(base + pl.mask_off);
    a.status = J.status;
    a.M = (int)M;
    a.relu = 0;
    a.tile_m = tm;
    a.n_at = (int)(rows_pad / tm);
    a.total_units = units;
    return cuda_status(launch_i8s_gemm_tc(a, 2 * i8s_plan_pairs(a), stream));
}

size_t w8a8_mul_mat_packed_workspace(int64_t M, int64_t N, int64_t K) {
    if (!w8a8_shape_ok(M, N, K)) return 0;
    const w8a8_problem q{reinterpret_cast<const void*>(16), reinterpret_cast<const float*>(16), N, K,
                         reinterpret_cast<const float*>(16), reinterpret_cast<float*>(16)};
    return w8a8_mul_mat_grouped_workspace(&q, 1, M);
}

int w8a8_mul_mat_packed(const void* packed, const float* bscale, int64_t N, int64_t K, const float* x, int64_t M,
                        float* d, void* ws, size_t ws_bytes, i2s_stream_t stream) {
    const w8a8_problem q{packed, bscale, N, K, x, d};
    return w8a8_mul_mat_grouped(&q, 1, M, ws, ws_bytes, stream);
}

int i2s_read_status(void* ws, i2s_stream_t stream) {
    if (!ws) return I2S_E_NULL_PTR;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return I2S_E_CUDA;
    uint32_t word = 0;
    uint8_t* p = static_cast<uint8_t*>(ws) + kStatusOff;
    if (cudaMemcpy(&word, p, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return I2S_E_CUDA;
    if (word == 0) return I2S_OK;
    if (cudaMemset(p, 0, 4) != cudaSuccess) return I2S_E_CUDA;
    return I2S_E_DEVICE_TIMEOUT;
}

}  // extern "C"
#pragma GCC visibility pop
