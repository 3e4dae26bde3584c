// Device helpers shared by the kernels of the Qwen3 decoder forward (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q3 {

typedef __nv_bfloat16 bf16;

// Bits of the device error word.
enum : uint32_t {
    ERR_TOKEN_RANGE = 1u,   // a token id outside [0, vocab) was clamped
    ERR_POSITION = 2u,      // a position at or beyond max_ctx was skipped
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Eight bf16 packed in a uint4 -> eight floats.
__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(p[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// Dot product of 8 bf16 weights (uint4) with 8 bf16 activations (uint4), fp32 accumulate.
__device__ __forceinline__ float dot8(const uint4 &w, const uint4 &x, float acc) {
    const __nv_bfloat162 *pw = reinterpret_cast<const __nv_bfloat162 *>(&w);
    const __nv_bfloat162 *px = reinterpret_cast<const __nv_bfloat162 *>(&x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 a = __bfloat1622float2(pw[i]);
        float2 b = __bfloat1622float2(px[i]);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
    }
    return acc;
}

// Streaming 16-byte load that does not allocate in L1 (weights are read once per launch).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Programmatic dependent launch: wait until the preceding kernel in the stream has
// completed and flushed its writes (a no-op when launched without the attribute) ...
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// ... and allow the next kernel in the stream to begin launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ float silu(float x) { return x / (1.0f + __expf(-x)); }

}  // namespace q3
