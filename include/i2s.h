/*
 * i2s.h - C ABI of libi2s.so: the I2_S ternary-weight x INT8-activation
 * matmul and the I8_S x I8_S fused mul_mat_add(_relu), on NVIDIA GB300
 * (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [P1] "ggml: additive INT8/ternary types, fused CPU ops, and kernels for
 *        VibeASR (1/2)" (audio.cpp pull request 447)
 *   [P2] "ggml-cpu: ternary I2_S matmul kernel (VibeASR, 3/4)" (audio.cpp
 *        pull request 445)
 *   [P3] "VibeASR in audio.cpp"
 *   [P4] "Experiment - int8 W8A8 path" (ork-driver wiki)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Shapes follow ggml: a weight W is N x K (K contiguous), activations X are
 * M x K (K contiguous), outputs Y are M x N (N contiguous). All sizes are
 * element counts.
 *
 * Pointers documented as "device" must point to memory the current CUDA device
 * can read or write (cudaMalloc, torch CUDA tensors, managed memory). Pointers
 * documented as "host" are ordinary CPU memory. The library never allocates,
 * frees or retains any caller buffer; the caller owns every buffer and must
 * keep it alive until the work queued on `stream` has finished.
 *
 * Device entry points are asynchronous and stream-ordered: they validate their
 * arguments on the host, enqueue kernels on `stream` (NULL = legacy default
 * stream) and return without synchronizing. A non-zero return means nothing
 * was enqueued (argument errors) or the launch failed (I2S_E_CUDA).
 *
 * Scales live in band, after the payload ([P1] "Two new types"), so a weight
 * or I8_S activation is fully described by its bytes and its shape.
 *
 * Byte layouts
 * ------------
 * I2_S (N x K, K % 128 == 0): N*K/4 payload bytes. The flat tensor is cut
 *   into groups of 128 values stored in 32 bytes; byte gp of a group holds the
 *   group-relative positions gp, 32+gp, 64+gp, 96+gp in its bit pairs at
 *   shifts 6, 4, 2, 0 ([P1] Kernels; [P2] Kernels). Codes {0,1,2} stand for
 *   the ternary values {-1,0,+1}. Then the F32 absmax (a multiplier:
 *   w = (code-1)*absmax) at byte offset N*K/4, then 28 zero bytes.
 * I8_S (n elements): n int8 bytes, zero padded to a multiple of 32, then the
 *   F32 scale (a multiplier: x = q*scale, scale = amax/127), then 28 zero
 *   bytes ([P1] "Two new types"). The pages call the scale "padded" without
 *   saying how; the 32-byte trailer is this library's reading.
 *
 * Arithmetic ([P2] Arithmetic; [P1] "Arithmetic is exact where it can be")
 * ----------
 * Every result is bit-identical to the plain definition:
 *   row quantization: amax = max(max_k |x|, 1e-5); scale = amax/127;
 *     inv = 127/amax; q = clamp(round(x*inv), -127, 127), halfway cases
 *     rounded away from zero; row_sum = sum_k q.
 *   I2_S: dot = sum_k code*q (int32, exact);
 *     y = (float)(dot - row_sum) * (w_scale * act_scale).
 *   I8_S: acc = sum_k w*x (int32, exact);
 *     y = (float)acc * (w_scale * x_scale) + bias[n]; ReLU: y > 0 ? y : +0;
 *     the output is requantized with one scale for the whole tensor.
 * Every float step is one IEEE-754 binary32 operation rounded to nearest
 * (no fused multiply-add).
 */
#ifndef I2S_H
#define I2S_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* i2s_stream_t;

/* Status codes (0 = success). */
enum {
    I2S_OK = 0,
    I2S_E_BAD_SHAPE = -1,          /* non-positive size, K % 128 != 0, too large */
    I2S_E_NULL_PTR = -2,           /* a required pointer is NULL */
    I2S_E_MISALIGNED = -3,         /* a device pointer is not 16-byte aligned */
    I2S_E_WORKSPACE_TOO_SMALL = -4,/* ws_bytes below the *_workspace() size */
    I2S_E_CUDA = -5,               /* a CUDA runtime call or launch failed */
    I2S_E_DEVICE_TIMEOUT = -6,     /* a kernel gave up a bounded wait (see i2s_read_status) */
    I2S_E_UNSUPPORTED_DEVICE = -7, /* current device is not sm_103 */
    I2S_E_BAD_ARG = -8             /* any other invalid argument */
};

/* Human-readable name of a status code. Never NULL; the string is static. */
const char* i2s_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int i2s_version(void);

/* 1 if the current CUDA device can run this library (compute capability
 * 10.3), 0 if not, a negative status if the CUDA runtime fails. */
int i2s_device_supported(void);

/* ---------------------------------------------------------------------------
 * Layout helpers (host only, no CUDA calls). Return 0 for invalid shapes.
 * ------------------------------------------------------------------------- */
size_t i2s_nbytes(int64_t N, int64_t K);        /* N*K/4 + 32 */
size_t i2s_scale_offset(int64_t N, int64_t K);  /* N*K/4 */
size_t i8s_nbytes(int64_t n);                   /* align32(n) + 32 */
size_t i8s_scale_offset(int64_t n);             /* align32(n) */

/* Packs N x K ternary codes (host, one code in {0,1,2} per byte, row-major)
 * and the F32 absmax into I2_S bytes at dst (host, i2s_nbytes(N,K) bytes).
 * Codes above 3 are masked to their low 2 bits. Errors: BAD_SHAPE, NULL_PTR. */
int i2s_pack_host(const uint8_t* codes, int64_t N, int64_t K, float w_scale, void* dst);

/* Packs n int8 values (host) and an F32 scale into I8_S bytes at dst (host,
 * i8s_nbytes(n) bytes). Errors: BAD_SHAPE, NULL_PTR. */
int i8s_pack_host(const int8_t* q, int64_t n, float scale, void* dst);

/* ---------------------------------------------------------------------------
 * Tiled I2_S weights: the bytes of an I2_S tensor rearranged once, at load
 * time, into contiguous 16 KB blocks. The GEMV and GEMM kernels read each
 * block with one bulk copy instead of a strided tile of 128 row pieces, and
 * give the same results, bit for bit, as on the I2_S bytes.
 *
 * Layout: the rows are split into Tn = 2*ceil(N/256) blocks of 128 rows, each
 * row's K/4 bytes into Tk = ceil(K/512) blocks of 128 bytes. Block (i, j)
 * holds bytes 128j..128j+127 of rows 128i..128i+127 and starts at byte
 * (i*Tk + j)*16384. Row rr of a block starts at byte rr*128 of it, and the
 * row's 16-byte piece c (its bytes 16c..16c+15 of the block) is stored as
 * piece c ^ (rr % 8). Bytes of rows past N or past K/4 are zero. The I2_S
 * tensor's 32-byte trailer (the F32 weight scale first) follows at
 * Tn*Tk*16384.
 * ------------------------------------------------------------------------- */
#define I2S_LAYOUT_I2S 0u     /* i2s_problem::w_layout: w_i2s holds I2_S bytes */
#define I2S_LAYOUT_TILED 1u   /* w_i2s holds the tiled layout (i2s_tile_weights) */
size_t i2s_tiled_nbytes(int64_t N, int64_t K);        /* Tn*Tk*16384 + 32 */
size_t i2s_tiled_scale_offset(int64_t N, int64_t K);  /* Tn*Tk*16384 */

/* Writes the tiled layout of the I2_S weights w_i2s (device,
 * i2s_nbytes(N, K) bytes) into tiled (device, i2s_tiled_nbytes(N, K) bytes),
 * enqueued on stream. N and K as for i2s_mul_mat. Errors: BAD_SHAPE,
 * NULL_PTR, MISALIGNED (a pointer not 16-byte aligned), BAD_ARG (the buffers
 * overlap), CUDA. */
int i2s_tile_weights(const void* w_i2s, int64_t N, int64_t K, void* tiled, i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * Activation quantization, per row ([P2] Arithmetic and the threading
 * paragraph of Kernels; [P3] Encoder for the 1e-5 floor; [P4] Implementation
 * for scale = amax/127, inv = 127/amax, round, clamp +-127).
 *
 * x        device, M x K F32, 16-byte aligned.
 * q        device, M x K int8 (row-major, same order as x).
 * act_scale device, M F32: amax/127 of each row.
 * row_sum  device, M int32: sum of each quantized row (the sidecar that the
 *          I2_S epilogue subtracts, [P1] "Arithmetic is exact where it can be").
 * K % 4 == 0 is required (K % 128 == 0 for use with I2_S weights).
 * Errors: BAD_SHAPE, NULL_PTR, MISALIGNED, CUDA.
 * ------------------------------------------------------------------------- */
int i2s_quantize_act(const float* x, int64_t M, int64_t K, int8_t* q, float* act_scale,
                     int32_t* row_sum, i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * I2_S x F32 -> F32 matmul: ggml_mul_mat with an I2_S src0 and an F32 src1
 * ([P2] Interface, Arithmetic; [P1] "Five fused INT8 ops", last paragraph).
 *
 * w_i2s  device, i2s_nbytes(N,K) bytes of I2_S weights (scale read in band).
 * x      device, M x K F32 activations (a batched 3-D src1 is passed flattened
 *        into M rows), 16-byte aligned.
 * y      device, M x N F32 output, 16-byte aligned.
 * ws     device workspace of at least i2s_mul_mat_workspace(M,N,K) bytes,
 *        256-byte aligned; holds the quantized rows, per-row scale and sum
 *        (the counterpart of the sidecar the CPU mul_mat keeps in its work
 *        buffer, [P2] Kernels, threading paragraph), the
 *        TMA descriptors of the weight matrix, the integer partial sums of a
 *        K-split launch and a status word. Not preserved between calls; calls
 *        sharing one ws must be ordered on one stream.
 * Requirements: K % 128 == 0, M >= 1, N >= 1, M*K < 2^31, N*K/4 < 2^31.
 * M <= 16 runs the decode GEMV (weight-bandwidth bound); larger M runs the
 * GEMM. Both run on the tcgen05 tensor cores and give identical bits.
 * Errors: BAD_SHAPE, NULL_PTR, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA.
 * ------------------------------------------------------------------------- */
size_t i2s_mul_mat_workspace(int64_t M, int64_t N, int64_t K);
int i2s_mul_mat(const void* w_i2s, int64_t N, int64_t K, const float* x, int64_t M, float* y,
                void* ws, size_t ws_bytes, i2s_stream_t stream);

/* Launch-shape overrides for testing and tuning. Every setting gives the same
 * bits; zero fields mean "choose automatically". */
enum {
    I2S_PATH_AUTO = 0,   /* M <= 16: the GEMV, else the GEMM */
    I2S_PATH_GEMM = 2,   /* tensor-core GEMM, any M */
    I2S_PATH_GEMV = 3    /* tensor-core GEMV, M <= 16 (BAD_ARG above) */
};
typedef struct i2s_config {
    int path;        /* I2S_PATH_*; any other value is BAD_ARG */
    int grid_ctas;   /* persistent CTA count: GEMV at most 2 per SM; GEMM runs CTA pairs
                        (rounded down to an even count, at least 2, at most the pairs that
                        fit at once) */
    int64_t test_stall_cycles;   /* tests only, GEMV path: > 0 makes the GEMV's epilogue
                        wait this many SM cycles on a barrier nothing signals, then give
                        up, so that the launch leaves through its device-timeout path
                        (copies and MMAs in flight drained, TMEM freed) and
                        i2s_read_status reports I2S_E_DEVICE_TIMEOUT. The output is then
                        incomplete. 0 for normal use; negative is BAD_ARG. */
    unsigned w_layout;   /* I2S_LAYOUT_I2S (0) or I2S_LAYOUT_TILED (w_i2s then holds the
                        output of i2s_tile_weights); other values are BAD_ARG */
} i2s_config;

int i2s_mul_mat_ex(const void* w_i2s, int64_t N, int64_t K, const float* x, int64_t M, float* y,
                   void* ws, size_t ws_bytes, const i2s_config* config, i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * Decode I2_S matmul without a workspace. It exists for callers that cannot
 * provide device scratch memory: a plain C or
 * ctypes host with no device allocator of its own, or a serving loop that
 * must not allocate once it runs, because cudaMalloc and cudaFree can
 * synchronize the device and a fixed memory budget leaves no room for
 * per-call buffers. Such a caller passes only the weights, the activations
 * and the output; the call itself allocates no memory.
 *
 * Same operation, arguments, requirements and bits as i2s_mul_mat on the
 * tensor-core GEMV path, limited to 1 <= M <= 16 (BAD_SHAPE otherwise). The
 * scratch is a fixed array of I2S_NOALLOC_SCRATCH_BYTES inside the library's
 * device code, one per device. A problem needs 1024 + up256(R*K/2) bytes of
 * it (R = 32 for M <= 8, else 48) plus, when K > 1536, up256(4*M*N) +
 * up256(4*ceil(N/128)), where up256 rounds up to a multiple of 256. A problem
 * that needs more is rejected with WORKSPACE_TOO_SMALL before anything is
 * enqueued. Every decode projection of a 1.5B-parameter decoder (K, N up to
 * 8960, a 151936-row output head at K = 1536) fits.
 *
 * Set-up: the first call made with a device current loads the array on that
 * device and looks up its address, which later calls on that device reuse.
 * Make that first call (for example one warm-up call) before capturing any
 * stream, and before the point from which the caller cannot tolerate set-up
 * work. A device reset (cudaDeviceReset) unloads the array and invalidates
 * that address: a process that resets a device must not call this entry
 * point on that device again.
 * Races: every call on a device uses the same array, so calls whose work can
 * overlap on the GPU race and give wrong results. Order all calls on one
 * device, for example on a single stream.
 * Contents: the array keeps what the previous call left in it. Each call
 * clears what must start at zero (the status word, the split-K partial sums
 * and their counters) in its first launch, so callers never clear it.
 * Device waits that run out are recorded in the array's status word, which
 * this call cannot return (its return value reports validation and launch
 * errors only); i2s_noalloc_read_status below reads it.
 * Errors: BAD_SHAPE, NULL_PTR, MISALIGNED, WORKSPACE_TOO_SMALL,
 * UNSUPPORTED_DEVICE, CUDA.
 * ------------------------------------------------------------------------- */
#define I2S_NOALLOC_SCRATCH_BYTES 4194304
int i2s_mul_mat_noalloc(const void* w_i2s, int64_t N, int64_t K, const float* x, int64_t M, float* y,
                        i2s_stream_t stream);

/* The no-alloc counterpart of i2s_read_status, for the current device:
 * synchronizes `stream`, reads the status word of the library's scratch array,
 * clears it, and returns I2S_OK or I2S_E_DEVICE_TIMEOUT. It sets the device up
 * as a first i2s_mul_mat_noalloc call would (so it may run before any).
 * Errors: UNSUPPORTED_DEVICE, CUDA. */
int i2s_noalloc_read_status(i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped I2_S matmul: several independent projections with the same number of
 * activation rows M, run as one quantization launch plus one GEMV/GEMM launch
 * (the per-layer q/k/v/o/gate/up/down set of a decoder, or many layers).
 * Projections whose x pointers (and K) are equal share one quantization.
 *
 * probs  host array of `count` problems; read during the call only.
 * count  1 .. I2S_MAX_GROUP.
 * ws     device workspace of at least i2s_mul_mat_grouped_workspace() bytes.
 * Requirements per problem as for i2s_mul_mat.
 * Errors: as i2s_mul_mat, plus BAD_ARG for count out of range or a w_layout
 * other than I2S_LAYOUT_I2S and I2S_LAYOUT_TILED.
 * ------------------------------------------------------------------------- */
#define I2S_MAX_GROUP 256

typedef struct i2s_problem {
    const void* w_i2s; /* device, I2_S N x K (or its tiled layout, below) */
    int64_t N;
    int64_t K;
    const float* x;    /* device, M x K F32 */
    float* y;          /* device, M x N F32 */
    unsigned w_layout; /* I2S_LAYOUT_I2S (0) or I2S_LAYOUT_TILED; other values BAD_ARG.
                          A group may mix the two. */
} i2s_problem;

size_t i2s_mul_mat_grouped_workspace(const i2s_problem* probs, int count, int64_t M);
int i2s_mul_mat_grouped(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                        i2s_stream_t stream);

/* The two phases of i2s_mul_mat_grouped as separate calls, as the pages'
 * mul_mat runs them ([P2] Kernels, threading paragraph: quantize the rows,
 * one barrier, then the output features). _quantize writes every distinct
 * activation's quantized rows, scale and row sum into ws; _run computes all
 * the projections from ws. A _run call must use the same problem list, M and
 * workspace as the _quantize call before it on the stream. Splitting lets a
 * caller quantize once and run the projections later or several times: a
 * completed _run leaves the workspace's split-K sums and counters at zero, as
 * _quantize leaves them.
 * Errors: as i2s_mul_mat_grouped. */
int i2s_mul_mat_grouped_quantize(const i2s_problem* probs, int count, int64_t M, void* ws,
                                 size_t ws_bytes, i2s_stream_t stream);
int i2s_mul_mat_grouped_run(const i2s_problem* probs, int count, int64_t M, void* ws,
                            size_t ws_bytes, i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * The grouped I2_S matmul on HOST activations and outputs: one call enqueues
 * the activations' copy to the device, the grouped matmul (same kernels and
 * results as i2s_mul_mat_grouped) and the outputs' copy back, all on
 * `stream`. This is the whole mul_mat of [P2] Kernels for a caller whose
 * src1 rows and results live in CPU memory; the weights stay on the device.
 *
 * probs  host array of `count` problems as for i2s_mul_mat_grouped, except
 *        that x (M x K F32) and y (M x N F32) are HOST pointers, 16-byte
 *        aligned. With page-locked memory (cudaHostAlloc, cudaHostRegister)
 *        the copies are asynchronous; with pageable memory the runtime
 *        stages them and the call may return only after they are done.
 * ws     device workspace of at least i2s_mul_mat_grouped_host_workspace()
 *        bytes, 256-byte aligned: the grouped workspace (so i2s_read_status
 *        reads the same status word), then device copies of the activations
 *        and outputs.
 * Copies: host ranges of the activations that touch or overlap are merged,
 * and each merged range moves up with one cudaMemcpyAsync; the outputs come
 * back the same way. Activations and outputs that are slices of one buffer
 * each take one copy each way. y holds the results once the stream's work is
 * done; x and y must stay valid until then.
 * Errors: as i2s_mul_mat_grouped, plus BAD_ARG if two outputs overlap or an
 * output overlaps an activation. The workspace query returns 0 for a list the
 * call would reject.
 * ------------------------------------------------------------------------- */
size_t i2s_mul_mat_grouped_host_workspace(const i2s_problem* probs, int count, int64_t M);
int i2s_mul_mat_grouped_host(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                             i2s_stream_t stream);

/* As i2s_mul_mat_grouped_host, with flags:
 *   0                 the staged copies above;
 *   I2S_HOST_MAPPED   every x and y lies in page-locked host memory that the
 *                     device reaches at the same address (cudaHostAlloc or
 *                     cudaMallocHost memory, or memory registered with
 *                     cudaHostRegisterMapped, under unified addressing): the
 *                     quantization kernel reads x and the matmul's epilogue
 *                     writes y over the host link directly, with no staging
 *                     copies and no staging area (a workspace of
 *                     i2s_mul_mat_grouped_workspace() bytes is enough). Every
 *                     byte of every x and y must be so mapped; the call checks
 *                     the ends of each merged range (cudaPointerGetAttributes)
 *                     and returns BAD_ARG, with nothing enqueued, if one is not.
 *   I2S_HOST_MAPPED_Y only the outputs are so mapped and written in place by
 *                     the epilogue; the activations are staged (one copy up
 *                     per merged range, as with flags 0), so their transfer
 *                     runs on a copy engine and can overlap kernels of other
 *                     streams. The workspace is the staged call's. Every byte
 *                     of every y must be mapped (checked as above).
 * I2S_HOST_MAPPED with I2S_HOST_MAPPED_Y is I2S_HOST_MAPPED. Same results, bit
 * for bit, in every mode. Errors: as i2s_mul_mat_grouped_host, plus BAD_ARG
 * for unknown flag bits. */
#define I2S_HOST_MAPPED 1u
#define I2S_HOST_MAPPED_Y 2u
int i2s_mul_mat_grouped_host_ex(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                                unsigned flags, i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * Fused decode step: the grouped I2_S matmul for M <= 16 as ONE launch whose
 * prologue quantizes the activations, as the pages' mul_mat quantizes its
 * src1 rows before the dot products in the same op ([P2] Kernels, threading
 * paragraph; [P1] "Five fused INT8 ops", last paragraph). The rows of every
 * distinct activation are spread over the launch's CTAs by cost; each row's
 * e2m1 digit operand, scale and sum are published through a per-activation
 * ready counter, and the weight stream starts before the activations are
 * ready. Same results, bit for bit, as i2s_mul_mat_grouped.
 *
 * The workspace (i2s_mul_mat_grouped_fused_workspace bytes, 256-byte aligned)
 * carries state between calls: a fixed area of flags at its start that every
 * launch leaves cleared for the next one. Zero that area once with
 * i2s_mul_mat_grouped_fused_init before the first fused call on a workspace
 * (and again if the workspace was used for anything else in between). Calls
 * sharing a workspace must be ordered on one stream. A device wait that runs
 * out is recorded in the status word (i2s_read_status), which these calls do
 * not clear.
 * Requirements: 1 <= M <= 16; per problem as i2s_mul_mat; at most
 * 8 distinct K among the problems and 120 distinct activations (BAD_ARG).
 * Errors: as i2s_mul_mat_grouped.
 * ------------------------------------------------------------------------- */
size_t i2s_mul_mat_grouped_fused_workspace(const i2s_problem* probs, int count, int64_t M);
int i2s_mul_mat_grouped_fused_init(void* ws, size_t ws_bytes, i2s_stream_t stream);
int i2s_mul_mat_grouped_fused(const i2s_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                              i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * I8_S x I8_S -> I8_S fused matmul + bias (+ ReLU) with requantization in the
 * op: ggml_mul_mat_add (relu = 0) and ggml_mul_mat_add_relu (relu != 0)
 * ([P1] "Five fused INT8 ops").
 *
 * w_i8s  device, i8s_nbytes(N*K) bytes: N x K int8 weights + in-band scale.
 * x_i8s  device, i8s_nbytes(M*K) bytes: M x K int8 activations + scale.
 * bias   device, N F32, or NULL for no bias.
 * y_i8s  device, i8s_nbytes(M*N) bytes: M x N int8 output + in-band scale.
 * ws     device workspace of at least i8s_mul_mat_workspace(M,N,K) bytes,
 *        256-byte aligned. After the call it holds the F32 output before
 *        requantization (M x N, row-major) at offset 256 (i8s_ws_f32_offset).
 * Requirements: K >= 1 with Kp <= 65536, Kp = K rounded up to a multiple of
 * 64 (at most 64 accumulation chunks of 1024 positions); M*Kp, N*Kp, M*N <
 * 2^31; all pointers 16-byte aligned. Any K is allowed: a conv run as
 * im2col_asym then mul_mat_add has K = C*KW ([P3] Encoder), for example 7
 * for a mono waveform stem. The operand rows hold Kp positions, the tail
 * zero, which adds nothing to the integer dot.
 * Errors: BAD_SHAPE, NULL_PTR, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA.
 * ------------------------------------------------------------------------- */
size_t i8s_mul_mat_workspace(int64_t M, int64_t N, int64_t K);
size_t i8s_ws_f32_offset(void);
int i8s_mul_mat_add_relu(const void* w_i8s, int64_t N, int64_t K, const void* x_i8s, int64_t M,
                         const float* bias, int relu, void* y_i8s, void* ws, size_t ws_bytes,
                         i2s_stream_t stream);

/* Weights packed once (a load-time repack, as ggml's CPU backends repack weights
 * for their kernels): i8s_pack_weights writes the f16 operand rows of an I8_S
 * weight tensor (exact integers, N x Kp, Kp = K rounded up to 64, the tail
 * zero) followed by a 16-byte trailer holding its F32 scale:
 * i8s_packed_bytes(N,K) bytes, 16-byte aligned, caller-owned.
 * i8s_mul_mat_add_relu_packed then computes the same result as
 * i8s_mul_mat_add_relu without converting the weights on every call; its
 * workspace is i8s_mul_mat_packed_workspace(M,N,K) bytes (the F32 output
 * before requantization is at the same offset). Requirements and errors as
 * i8s_mul_mat_add_relu (BAD_ARG: the packed buffer overlaps the weights). */
size_t i8s_packed_bytes(int64_t N, int64_t K);
int i8s_pack_weights(const void* w_i8s, int64_t N, int64_t K, void* packed, i2s_stream_t stream);
size_t i8s_mul_mat_packed_workspace(int64_t M, int64_t N, int64_t K);
int i8s_mul_mat_add_relu_packed(const void* packed, int64_t N, int64_t K, const void* x_i8s, int64_t M,
                                const float* bias, int relu, void* y_i8s, void* ws, size_t ws_bytes,
                                i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * F32 -> I8_S requantization with one scale for the whole tensor ([P1] "Two
 * new types", "Five fused INT8 ops"; [P3] Encoder): amax = max(max|y|, 1e-5),
 * scale = amax/127, q = clamp(round(y*127/amax), -127, 127).
 *
 * y      device, n F32, 16-byte aligned.
 * dst    device, i8s_nbytes(n) bytes.
 * ws     device workspace of at least i8s_requant_workspace(n) bytes.
 * Errors: BAD_SHAPE, NULL_PTR, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA.
 * ------------------------------------------------------------------------- */
size_t i8s_requant_workspace(int64_t n);
int i8s_requant(const float* y, int64_t n, void* dst_i8s, void* ws, size_t ws_bytes,
                i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * I8_S element-wise ops ([P1] "Five fused INT8 ops": ggml_add_scaled and
 * ggml_rms_norm_scaled; "Two new types", the dup/cont note: a permuted copy
 * carries the in-band scale). Each output is a self-describing I8_S tensor:
 * where its scale depends on the values, the op requantizes per tensor as
 * i8s_requant does (amax floored at 1e-5, scale = amax/127, round half away
 * from zero, clamp to +-127). Two passes over the inputs: the first folds
 * max|y|, the second recomputes y and quantizes it.
 *
 * i8s_add_scaled:      y = (float)a*a_scale + (float)b*b_scale (two IEEE
 *                      products, one IEEE sum), n elements.
 * i8s_rms_norm_scaled: rows x ne0 (ne0 contiguous), each row normalised:
 *                      x = q*scale; mean = ((float)sum(q^2) * (scale*scale))
 *                      / ne0; r = 1/sqrt(mean + eps), each a correctly
 *                      rounded binary32 operation; y = (x*r) (* gamma[i]).
 *                      eps >= 0: 1e-5 in the encoder ([P3] "Encoder"); with
 *                      eps = 0 an all-zero row is undefined (0 * inf). gamma:
 *                      device F32 [ne0] or NULL for none. ne0 <= 131072.
 * i8s_transpose:       src a x b (row-major) -> dst b x a, scale copied
 *                      (ggml_cont(ggml_permute(...))). No workspace.
 *
 * Inputs and outputs are device I8_S buffers of i8s_nbytes(n) bytes; an
 * output must not overlap an input. add_scaled and rms_norm_scaled need
 * 16-byte aligned buffers and a 256-byte aligned workspace of at least
 * i8s_eltwise_workspace(rows) bytes (rows = 1 for add_scaled).
 * Errors: BAD_SHAPE, NULL_PTR, MISALIGNED, WORKSPACE_TOO_SMALL, BAD_ARG (an
 * output overlapping an input), CUDA.
 * ------------------------------------------------------------------------- */
size_t i8s_eltwise_workspace(int64_t rows);
int i8s_add_scaled(const void* a_i8s, const void* b_i8s, int64_t n, void* y_i8s, void* ws,
                   size_t ws_bytes, i2s_stream_t stream);
int i8s_rms_norm_scaled(const void* x_i8s, int64_t rows, int64_t ne0, float eps, const float* gamma,
                        void* y_i8s, void* ws, size_t ws_bytes, i2s_stream_t stream);
int i8s_transpose(const void* src_i8s, int64_t a, int64_t b, void* dst_i8s, i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * Encoder convolution pieces on I8_S ([P1] "Five fused INT8 ops":
 * ggml_im2col_asym, im2col with independent left/right padding so that a
 * causal conv needs no pad node; "Tests": depthwise mul_mat_add; [P3]
 * "Encoder": strided causal convs with left pad K - stride, right pad 0, and
 * a depthwise conv in every block).
 *
 * Geometry: input C x L (L contiguous, one channel per row); kernel width KW,
 * stride, left pad pad_l, right pad pad_r (zeros); output length
 * OL = (L + pad_l + pad_r - KW) / stride + 1 (i8s_im2col_out_len; 0 if the
 * padded input is shorter than KW).
 *
 * i8s_im2col_asym:  dst is OL x (C*KW), dst[t][c*KW + k] =
 *                   src[c][t*stride + k - pad_l] (0 outside the input), with
 *                   the input's scale. No workspace.
 * i8s_depthwise_mul_mat_add: w_i8s is C x KW (one kernel row per channel);
 *                   y[c][t] = (float)acc * (w_scale*x_scale) + bias[c], ReLU
 *                   if relu != 0, acc = sum_k w[c][k] * x[c][t*stride + k -
 *                   pad_l] in int32; y is C x OL, requantized per tensor.
 *                   bias: device F32 [C] or NULL. Workspace as
 *                   i8s_eltwise_workspace(1).
 * Requirements: C, L, KW, stride >= 1; pad_l, pad_r >= 0; C*L, OL*C*KW and
 * C*OL < 2^31; dst/y 16-byte aligned; no overlap of output and inputs.
 * Errors: BAD_SHAPE, NULL_PTR, MISALIGNED, WORKSPACE_TOO_SMALL, BAD_ARG (an
 * output overlapping an input), CUDA.
 * ------------------------------------------------------------------------- */
int64_t i8s_im2col_out_len(int64_t L, int64_t KW, int64_t stride, int64_t pad_l, int64_t pad_r);
int i8s_im2col_asym(const void* src_i8s, int64_t C, int64_t L, int64_t KW, int64_t stride, int64_t pad_l,
                    int64_t pad_r, void* dst_i8s, i2s_stream_t stream);
int i8s_depthwise_mul_mat_add(const void* w_i8s, int64_t KW, const void* x_i8s, int64_t C, int64_t L,
                              int64_t stride, int64_t pad_l, int64_t pad_r, const float* bias, int relu,
                              void* y_i8s, void* ws, size_t ws_bytes, i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * W8A8 per-channel matmul ([P4] "Experiment - int8 W8A8 path", sections
 * "Hypothesis" and "Implementation"): int8 weights with one scale per output
 * channel, int8 activations with one scale per row, int32 accumulation, then
 * d[m][n] = aScale[m] * bScale[n] * (float)C[m][n] (left to right).
 *
 * w8a8_quantize_weights: w is N x K F32 (device); per channel n: amax =
 *   max(max_k |w|, 1e-9), bscale[n] = amax/127, wq = clamp(rint(w /
 *   bscale[n]), -127, 127) (an IEEE division, ties to even), N x K int8.
 * w8a8_mul_mat: x is M x K F32 (device); per row: amax = max(max_k |x|,
 *   1e-9), aScale[m] = amax/127, q = clamp(round(x * (127/amax))) (half away
 *   from zero); d is M x N F32. The exact int32 dot runs on the I8_S
 *   tensor-core path (f16 operands, f32 chunk sums of at most 1024
 *   positions, drained into int32).
 * Requirements: K >= 1 with Kp <= 65536 (Kp = K rounded up to a multiple of
 * 64; the operand rows hold Kp positions, the tail zero); M*Kp, N*Kp, M*N <
 * 2^31; 16-byte aligned pointers; ws 256-byte aligned, at least
 * w8a8_mul_mat_workspace.
 * Errors: BAD_SHAPE, NULL_PTR, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA.
 * ------------------------------------------------------------------------- */
int w8a8_quantize_weights(const float* w, int64_t N, int64_t K, int8_t* wq, float* bscale,
                          i2s_stream_t stream);
size_t w8a8_mul_mat_workspace(int64_t M, int64_t N, int64_t K);
int w8a8_mul_mat(const int8_t* wq, const float* bscale, int64_t N, int64_t K, const float* x, int64_t M,
                 float* d, void* ws, size_t ws_bytes, i2s_stream_t stream);

/* Packed weights ([P4] Implementation: the weights are quantized and packed
 * for the matrix unit once, on the cache-miss path, and reused by every call).
 * w8a8_pack_weights writes the f16 operand rows of wq (exact integers, N x Kp,
 * Kp = K rounded up to 64, the tail zero; w8a8_packed_bytes(N,K) bytes,
 * 16-byte aligned, caller-owned) once;
 * w8a8_mul_mat_packed then runs each call as two launches (rows quantized
 * straight into f16 operand rows, then the GEMM) with no per-call weight
 * conversion. Same requirements and results as w8a8_mul_mat; workspace at least
 * w8a8_mul_mat_packed_workspace(M,N,K) bytes. */
size_t w8a8_packed_bytes(int64_t N, int64_t K);
int w8a8_pack_weights(const int8_t* wq, int64_t N, int64_t K, void* packed, i2s_stream_t stream);
size_t w8a8_mul_mat_packed_workspace(int64_t M, int64_t N, int64_t K);
int w8a8_mul_mat_packed(const void* packed, const float* bscale, int64_t N, int64_t K, const float* x,
                        int64_t M, float* d, void* ws, size_t ws_bytes, i2s_stream_t stream);

/* Several packed W8A8 matmuls with the same M in two launches: one quantizes
 * every distinct activation (problems whose x pointer and K are equal share
 * it, as q, k and v do), one tensor-core GEMM covers every matmul, so small
 * projections share the GPU instead of each leaving most SMs idle. Results are
 * those of w8a8_mul_mat_packed for each problem, bit for bit.
 * probs  host array of `count` problems (1 .. W8A8_MAX_GROUP); read during the
 *        call only. Per problem as w8a8_mul_mat_packed.
 * ws     device workspace of at least w8a8_mul_mat_grouped_workspace() bytes,
 *        256-byte aligned.
 * Errors: as w8a8_mul_mat_packed, plus BAD_ARG for count out of range. */
#define W8A8_MAX_GROUP 8

typedef struct w8a8_problem {
    const void* packed;   /* device, w8a8_pack_weights output (N x K) */
    const float* bscale;  /* device, N per-channel weight scales */
    int64_t N;
    int64_t K;
    const float* x;       /* device, M x K F32 activations */
    float* d;             /* device, M x N F32 output */
} w8a8_problem;

size_t w8a8_mul_mat_grouped_workspace(const w8a8_problem* probs, int count, int64_t M);
int w8a8_mul_mat_grouped(const w8a8_problem* probs, int count, int64_t M, void* ws, size_t ws_bytes,
                         i2s_stream_t stream);

/* ---------------------------------------------------------------------------
 * Device status. Kernels with bounded waits (the tensor-core pipelines) never
 * trap: when a wait runs out they record a code in the status word at the
 * start of the workspace and exit. Every i2s_mul_mat* call clears the word in
 * its first (quantization) launch, so it reflects the latest call on that
 * workspace. This call synchronizes `stream`, reads and clears that word, and
 * returns I2S_OK or I2S_E_DEVICE_TIMEOUT (or I2S_E_CUDA if the stream reports
 * an error).
 * ------------------------------------------------------------------------- */
int i2s_read_status(void* ws, i2s_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* I2S_H */
