// RMSNorm kernels: embedding gather + norm (layer 0), norm of the residual stream, and the
// final norm of each sequence's last row.
//
// RMSNorm(x; g)_i = x_i / sqrt(mean_j x_j^2 + eps) * g_i with eps inside the root
// ("手写Qwen3-0.6B推理", Qwen3RMSNorm; "古法手撕简易LLM推理器", 工具函数).  The residual
// stream stays fp32; the normed row is stored bf16 because it is the next GEMM's operand.
// One CTA of C/4 threads per row, four consecutive elements per thread.

#include "kernels.h"

namespace q3 {

namespace {

// Sum over the CTA (blockDim.x a multiple of 32, at most 1024).
__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    const int nw = blockDim.x >> 5;
    float t = lane < nw ? red[lane] : 0.0f;
    t = warp_sum(t);
    return t;
}

__device__ __forceinline__ void norm_store(float4 x, const float *gamma, bf16 *dst, int C,
                                          float eps, float *red) {
    const float ss = block_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w, red);
    const float inv = rsqrtf(ss / (float)C + eps);
    const float4 g = reinterpret_cast<const float4 *>(gamma)[threadIdx.x];
    uint2 o;
    o.x = pack_bf16x2(x.x * inv * g.x, x.y * inv * g.y);
    o.y = pack_bf16x2(x.z * inv * g.z, x.w * inv * g.w);
    reinterpret_cast<uint2 *>(dst)[threadIdx.x] = o;
}

__global__ void k_embed_rmsnorm(const int32_t *__restrict__ tokens, Rows r,
                                const bf16 *__restrict__ embed, const float *__restrict__ gamma,
                                float *__restrict__ resid, bf16 *__restrict__ xn, int C, int V,
                                float eps, uint32_t *err, float *__restrict__ zero_buf) {
    __shared__ float red[32];
    pdl_wait();
    const int row = blockIdx.x;
    if (zero_buf)  // this row of a buffer the next kernel accumulates into
        reinterpret_cast<float4 *>(zero_buf + (size_t)row * C)[threadIdx.x] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int id = tokens[row];
    if (id < 0 || id >= V) {
        if (threadIdx.x == 0) atomicOr(err, ERR_TOKEN_RANGE);
        id = id < 0 ? 0 : V - 1;
    }
    if (threadIdx.x == 0) {
        int slot, pos;
        if (r.cu_seqlens) {  // packed prefill: find the sequence holding this row
            int lo = 0, hi = r.B - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (r.cu_seqlens[mid] <= row) lo = mid; else hi = mid - 1;
            }
            slot = r.slots[lo];
            pos = row - r.cu_seqlens[lo] + (r.append ? r.ctx_len[slot] : 0);
        } else {  // decode: one row per sequence, appended after the cached tokens
            slot = r.slots[row];
            pos = r.ctx_len[slot];
        }
        r.row_slot[row] = slot;
        r.row_pos[row] = pos;
    }
    const uint2 e = reinterpret_cast<const uint2 *>(embed + (size_t)id * C)[threadIdx.x];
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&e.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&e.y));
    const float4 x = make_float4(a.x, a.y, b.x, b.y);
    reinterpret_cast<float4 *>(resid + (size_t)row * C)[threadIdx.x] = x;
    pdl_trigger();
    norm_store(x, gamma, xn + (size_t)row * C, C, eps, red);
}

__global__ void k_rmsnorm(const float *__restrict__ resid, const float *__restrict__ gamma,
                          bf16 *__restrict__ xn, int C, float eps) {
    __shared__ float red[32];
    pdl_wait();
    const int row = blockIdx.x;
    const float4 x = reinterpret_cast<const float4 *>(resid + (size_t)row * C)[threadIdx.x];
    pdl_trigger();
    norm_store(x, gamma, xn + (size_t)row * C, C, eps, red);
}

__global__ void k_final_norm(const float *__restrict__ resid, const int32_t *__restrict__ cu,
                             const float *__restrict__ gamma, bf16 *__restrict__ out, int C,
                             float eps) {
    __shared__ float red[32];
    pdl_wait();
    const int b = blockIdx.x;
    const int row = cu ? cu[b + 1] - 1 : b;
    const float4 x = reinterpret_cast<const float4 *>(resid + (size_t)row * C)[threadIdx.x];
    pdl_trigger();
    norm_store(x, gamma, out + (size_t)b * C, C, eps, red);
}

__global__ void k_bf16_to_f32(const bf16 *__restrict__ src, float *__restrict__ dst, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = __bfloat162float(src[i]);
}

}  // namespace

cudaError_t launch_embed_rmsnorm(const Launch &lc, const int32_t *tokens, const Rows &r,
                                 const bf16 *embed, const float *gamma, float *resid, bf16 *xn,
                                 int C, int V, float eps, uint32_t *err, float *zero_buf) {
    return launch(lc, k_embed_rmsnorm, dim3(r.rows), dim3(C / 4), 0, tokens, r, embed, gamma,
                  resid, xn, C, V, eps, err, zero_buf);
}

cudaError_t launch_rmsnorm(const Launch &lc, const float *resid, int rows, const float *gamma,
                           bf16 *xn, int C, float eps) {
    return launch(lc, k_rmsnorm, dim3(rows), dim3(C / 4), 0, resid, gamma, xn, C, eps);
}

cudaError_t launch_final_norm(const Launch &lc, const float *resid, const int32_t *cu_seqlens,
                              int B, const float *gamma, bf16 *out, int C, float eps) {
    return launch(lc, k_final_norm, dim3(B), dim3(C / 4), 0, resid, cu_seqlens, gamma, out, C,
                  eps);
}

cudaError_t launch_bf16_to_f32(const Launch &lc, const bf16 *src, float *dst, int n) {
    return launch(lc, k_bf16_to_f32, dim3((n + 255) / 256), dim3(256), 0, src, dst, n);
}

}  // namespace q3
