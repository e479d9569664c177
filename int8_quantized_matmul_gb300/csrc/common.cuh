// Device helpers shared by the libi2s kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace i2s {

// The quantizer step shared by the row quantizer and the per-tensor
// requantizer: q = clamp(round(x * inv), -127, 127), rounding halfway cases
// away from zero, in full-rate operations (the conversion instructions run at
// an eighth of the FP32 rate). Clamping first gives the same result. Then
// round(|v|) = floor(a) with a = |v| + h, h = 0.5 - 2^-25 (the largest float
// below one half), the sum rounded to nearest: for |v| just below k + 1/2 the
// sum stays below k + 1, at exactly k + 1/2 it is the midpoint k + 1 - 2^-25,
// which rounds (ties to even) to k + 1, and for |v| >= 2^22 it cannot reach
// the next integer. floor(a) (a < 128) is read from the low bits of
// a + 1.5*2^23 added with rounding toward zero, and the sign is put back on
// the integer. Checked on the GPU around every half integer against the CPU
// reference (C roundf).
__device__ __forceinline__ int quantize_one(float x, float inv) {
    const float v = fminf(fmaxf(__fmul_rn(x, inv), -127.0f), 127.0f);
    const float a = __fadd_rn(fabsf(v), 0x1.fffffep-2f);
    const int m = (int)(__float_as_uint(__fadd_rz(a, 12582912.0f)) - 0x4B400000u);
    return v < 0.0f ? -m : m;
}

// int -> float exactly for |v| < 2^22 in two full-rate operations: v added to
// the bit pattern of 1.5*2^23 (where the float step is 1), minus 1.5*2^23.
__device__ __forceinline__ float small_int_to_float(int v) {
    return __fsub_rn(__int_as_float(0x4B400000 + v), 12582912.0f);
}

// int8 -> float exactly in two full-rate operations: the byte b + 128 placed
// in the mantissa of 2^23 (XOR with 0x4B000080), minus 2^23 + 128.
__device__ __forceinline__ float i8_to_float(int8_t b) {
    return __fsub_rn(__uint_as_float((uint32_t)(uint8_t)b ^ 0x4B000080u), 8388736.0f);
}

// amax floor and the two divisions of the quantizer: scale = amax/127 is
// stored (a multiplier), inv = 127/amax multiplies each element.
__device__ __forceinline__ void quant_params(float amax, float& scale, float& inv) {
    amax = fmaxf(amax, 1e-5f);
    scale = __fdiv_rn(amax, 127.0f);
    inv = __fdiv_rn(127.0f, amax);
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization is scheduled as the CTAs of the kernel before it on the
// stream retire, instead of after that kernel's completion is processed;
// pdl_wait blocks until the previous kernel has completed and its memory is
// visible. A no-op in a kernel launched without the attribute. (An explicit
// early trigger, griddepcontrol.launch_dependents, made the decode step
// slower: the GEMV's CTAs then took SM resources while the quantization
// kernel was still running.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches a kernel as a programmatic dependent of the launch before it on
// the stream (the kernel must call pdl_wait before touching what that launch
// wrote, or what it may still read).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace i2s
