// i2s_mul_mat_noalloc: the decode I2_S matmul (M <= 16) with its scratch in a
// fixed device array owned by the library, for callers that cannot hand the
// library a workspace (declared and documented in include/i2s.h).
//
// It runs the same two launches as i2s_mul_mat's tensor-core GEMV path -- the
// per-row quantization into the e2m1 digit operand, then the tcgen05 GEMV --
// for a single problem, with the workspace replaced by g_scratch below. The
// scratch layout:
//   [0, 256)          status word (cleared by the quantization launch)
//   [256, 512)        the weight matrix's TMA map (written by the quantization launch)
//   [512, 768)        act_scale, M F32
//   [768, 1024)       row_sum, M int32
//   [1024, op_end)    e2m1 operand: gemv_tc_op_rows(Mp) digit rows of K/2 bytes
//   [op_end, ...)     K > 1536 only: M x N int32 split-K partials, then one
//                     uint32 chunk counter per 128-row tile; both zeroed by
//                     the quantization launch of every call.
// Nothing in this file allocates: the array is part of the library's device
// image, its address is looked up once per device, and the launch arguments
// live on the calling thread's stack.

#include <atomic>

#include "../../include/i2s.h"
#include "internal.h"

namespace i2s {
namespace {

constexpr size_t kScratchBytes = I2S_NOALLOC_SCRATCH_BYTES;
constexpr size_t kSlotAlign = 256;
constexpr int kMaxDev = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

size_t up256(size_t v) { return (v + kSlotAlign - 1) / kSlotAlign * kSlotAlign; }

// Per-device set-up, done by the first call made with that device current:
// the architecture check, the SM count and the address of g_scratch.
struct NoAllocDev {
    std::atomic<int> state{0};   // 0 not set up, 1 ready, negative: an I2S_E_* status
    unsigned char* scratch = nullptr;
    int sms = 0;
};
NoAllocDev g_na[kMaxDev];

int noalloc_setup(NoAllocDev*& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return I2S_E_CUDA;
    if (dev < 0 || dev >= kMaxDev) return I2S_E_UNSUPPORTED_DEVICE;
    NoAllocDev& d = g_na[dev];
    int st = d.state.load(std::memory_order_acquire);
    if (st == 0) {
        // Two threads may race through here; both compute the same values.
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return I2S_E_CUDA;
        if (!(major == 10 && minor == 3)) {
            d.state.store(I2S_E_UNSUPPORTED_DEVICE, std::memory_order_release);
            return I2S_E_UNSUPPORTED_DEVICE;
        }
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return I2S_E_CUDA;
        d.scratch = static_cast<unsigned char*>(p);
        d.sms = sms;
        d.state.store(1, std::memory_order_release);
        st = 1;
    }
    if (st != 1) return st;
    out = &d;
    return I2S_OK;
}

}  // namespace
}  // namespace i2s

using namespace i2s;

#pragma GCC visibility push(default)
extern "C" {

int i2s_mul_mat_noalloc(const void* w_i2s, int64_t N, int64_t K, const float* x, int64_t M, float* y,
                        i2s_stream_t stream) {
    if (!w_i2s || !x || !y) return I2S_E_NULL_PTR;
    if (M < 1 || M > 16 || N < 1 || K < 128 || K % 128 != 0 || K > 65536) return I2S_E_BAD_SHAPE;
    if (N * (K / 4) >= ((int64_t)1 << 31)) return I2S_E_BAD_SHAPE;
    if (((uintptr_t)w_i2s & 15u) || ((uintptr_t)x & 15u) || ((uintptr_t)y & 15u)) return I2S_E_MISALIGNED;

    const int Mp = gemv_tc_mp(M);
    const int op_rows = gemv_tc_op_rows(Mp);
    const bool split = K > kGemvChunkPositions;
    const size_t map_off = kSlotAlign;
    const size_t scale_off = map_off + kSlotAlign;
    const size_t sum_off = scale_off + up256((size_t)M * 4);
    const size_t op_off = sum_off + up256((size_t)M * 4);
    const size_t dot_off = op_off + up256((size_t)op_rows * (size_t)(K / 2));
    const int row_tiles = (int)((N + kTcTileW - 1) / kTcTileW);
    const size_t ticket_off = dot_off + (split ? up256((size_t)M * (size_t)N * 4) : 0);
    const size_t end = ticket_off + (split ? up256((size_t)row_tiles * 4) : 0);
    if (end > kScratchBytes) return I2S_E_WORKSPACE_TOO_SMALL;

    NoAllocDev* d = nullptr;
    int r = noalloc_setup(d);
    if (r) return r;
    unsigned char* base = d->scratch;
    uint32_t* status = reinterpret_cast<uint32_t*>(base);
    float* act_scale = reinterpret_cast<float*>(base + scale_off);
    int32_t* row_sum = reinterpret_cast<int32_t*>(base + sum_off);

    // Phase 1: quantize x into the operand; the same launch clears the status
    // word and the split-K partials and counters left by the previous call.
    QuantArgs qa;
    CUtensorMap* wmap = reinterpret_cast<CUtensorMap*>(base + map_off);
    if (!make_u8_operand_map(&qa.wtmpl, wmap, kTcTileW, 128, kTcTileW)) return I2S_E_CUDA;
    qa.wmaps = wmap;
    qa.n_wmaps = 1;
    qa.wj[0] = WMapJob{w_i2s, (int)N, (int)K};
    qa.status = status;
    qa.zero = split ? reinterpret_cast<uint4*>(base + dot_off) : nullptr;
    qa.zero_16 = split ? (end - dot_off) / 16 : 0;
    qa.count = 1;
    qa.M = (int)M;
    qa.rows = Mp;
    qa.layout = kQuantE2M1Tc;
    qa.j[0] = QuantJob{x, base + op_off, act_scale, row_sum, (int)K, (int)K};
    if (launch_quant(qa, stream) != cudaSuccess) return I2S_E_CUDA;

    // Phase 2: the tensor-core GEMV over the row tiles (x K chunks).
    TcArgs ta;
    ta.n_maps = 1;
    ta.count = 1;
    ta.M = (int)M;
    ta.BN = Mp;
    ta.status = status;
    if (!make_u8_operand_map(&ta.maps[0], base + op_off, op_rows, (int)(K / 2), op_rows)) return I2S_E_CUDA;
    ta.wmaps = wmap;
    ta.test_stall_cycles = 0;
    for (int w = 0; w < kTiledMaskWords; ++w) ta.tiled[w] = 0;   // I2_S bytes
    ta.dot_base = reinterpret_cast<int32_t*>(base + dot_off);
    ta.ticket_base = reinterpret_cast<uint32_t*>(base + ticket_off);
    const int chunks = (int)((K + kGemvChunkPositions - 1) / kGemvChunkPositions);
    TcProb& p = ta.p[0];
    p.w = static_cast<const uint8_t*>(w_i2s);
    p.act_scale = act_scale;
    p.row_sum = row_sum;
    p.y = y;
    p.N = (int)N;
    p.K = (int)K;
    p.map = 0;
    p.tile0 = 0;
    p.n_act_tiles = 1;
    p.chunks = chunks;
    p.dot_off = 0;
    p.ticket_off = 0;
    ta.total_tiles = row_tiles * chunks;
    const int cap = 2 * (d->sms > 0 ? d->sms : 152);
    const int grid = ta.total_tiles < cap ? ta.total_tiles : cap;
    // the same split of units between the two CTAs of an SM as the workspace path
    ta.share_first = grid == cap ? kGemvShareFirst : 1;
    ta.share_second = grid == cap ? kGemvShareSecond : 1;
    if (launch_gemv_tc(ta, grid, stream) != cudaSuccess) return I2S_E_CUDA;
    return I2S_OK;
}

int i2s_noalloc_read_status(i2s_stream_t stream) {
    NoAllocDev* d = nullptr;
    int r = noalloc_setup(d);
    if (r) return r;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return I2S_E_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, d->scratch, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return I2S_E_CUDA;
    if (word == 0) return I2S_OK;
    if (cudaMemset(d->scratch, 0, 4) != cudaSuccess) return I2S_E_CUDA;
    return I2S_E_DEVICE_TIMEOUT;
}

}  // extern "C"
#pragma GCC visibility pop
