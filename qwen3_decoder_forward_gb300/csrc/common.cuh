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
    ERR_TIMEOUT = 4u,       // a bounded wait on an asynchronous copy gave up
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

// ---- mbarrier + bulk asynchronous copies (TMA engine, untiled) ---------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cta(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completing on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Asks L2 to fetch [src, src + bytes) (16-byte aligned, multiple of 16); no completion.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// Default limit of a bounded wait: 2^31 SM cycles, about a second at 2 GHz.
constexpr long long WAIT_LIMIT_DEFAULT = 1ll << 31;

// Waits for phase `phase` of `bar` for at most WAIT_LIMIT_DEFAULT SM cycles; on timeout
// sets ERR_TIMEOUT in *err and returns false instead of spinning forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t phase, uint32_t *err) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, phase)) {
        if (clock64() - t0 > WAIT_LIMIT_DEFAULT) {
            if (err) atomicOr(err, ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// The device status block of a context is err[0] = error bits, err[1] = the wait limit of
// the decode kernels in SM cycles (0: WAIT_LIMIT_DEFAULT), set by the host between calls.
// Kernels read it once, at their start, with their other constant inputs.
__device__ __forceinline__ long long wait_limit(const uint32_t *err) {
    if (!err) return WAIT_LIMIT_DEFAULT;
    const uint32_t l = __ldcg(err + 1);
    return l ? (long long)l : WAIT_LIMIT_DEFAULT;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// mbar_wait_bounded with the limit `lim` from wait_limit (the decode kernels: weight and KV
// streams).  The default limit waits as mbar_wait_bounded does; a limit set by the host polls
// without suspending, so that a wait on a copy issued just before gives up deterministically
// when the limit is a few cycles.  A caller that gives up must still let its issued copies land
// (mbar_wait_bounded with a null err, the default limit) before the CTA exits.
__device__ __forceinline__ bool mbar_wait_ctx(uint64_t *bar, uint32_t phase, uint32_t *err, long long lim) {
    if (lim == WAIT_LIMIT_DEFAULT) return mbar_wait_bounded(bar, phase, err);
    const long long t0 = clock64();
    while (!mbar_test_wait(bar, phase)) {
        if (clock64() - t0 > lim) {
            if (err) atomicOr(err, ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

}  // namespace q3
