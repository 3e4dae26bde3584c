// Split-KV decode attention: one new query row per sequence against its cached keys 0..p.
//
// A decode query at absolute position p sees every cached key 0..p, its own included
// ("从零开始写Qwen3", Attn: no causal flag for a length-1 query; "古法手撕简易LLM推理器",
// 核心计算函数与Transformer层: no mask once offset > 0, the new key appended first).  The
// Hq/Hkv query heads of one KV head are served by the same CTA so each K/V row is read
// from HBM once ("手写Qwen3-0.6B推理", Attention: K/V shared by a group of query heads).
//
// Pass 1, grid (split, kv head, sequence): 8 lanes per key (16 dims each), 4 keys per warp
// and step; dot products reduced with 3 warp shuffles; an online softmax (m, l, acc) per
// 8-lane group, merged across groups with shuffles and across the 4 warps in shared
// memory.  Writes (m, l) and the unnormalised acc of its key range to a workspace.
// Pass 2, grid (query head, sequence): the log-sum-exp merge of the splits.
// Scores are pre-scaled by log2(e)/sqrt(128) so exp2 is used throughout.

#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int WARPS = 4;

template <int G>
__global__ void __launch_bounds__(WARPS * 32) k_attn_decode_split(
    const bf16 *__restrict__ q, const bf16 *__restrict__ k_layer, const bf16 *__restrict__ v_layer,
    Rows r, int kps, float *__restrict__ ws_ml, float *__restrict__ ws_o, int Hq, int Hkv,
    int max_ctx, float scale_log2) {
    __shared__ float red_ml[WARPS][G][2];
    __shared__ float red_o[WARPS][G][D];
    pdl_wait();
    pdl_trigger();
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int n_split = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane & 7, kg = lane >> 3;
    const int slot = r.row_slot[b];
    const int ctx = min(r.row_pos[b] + 1, max_ctx);
    const int k_begin = split * kps;
    const int k_end = min(ctx, k_begin + kps);

    float qv[G][16];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        const bf16 *qp = q + ((size_t)b * Hq + g * G + gi) * D + sub * 16;
        float t[8];
        unpack8(*reinterpret_cast<const uint4 *>(qp), t);
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[gi][e] = t[e] * scale_log2;
        unpack8(*reinterpret_cast<const uint4 *>(qp + 8), t);
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[gi][8 + e] = t[e] * scale_log2;
    }
    float m[G], l[G], acc[G][16];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        m[gi] = -INFINITY;
        l[gi] = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[gi][e] = 0.0f;
    }

    const bf16 *kb = k_layer + ((size_t)slot * Hkv + g) * max_ctx * D + sub * 16;
    const bf16 *vb = v_layer + ((size_t)slot * Hkv + g) * max_ctx * D + sub * 16;
    for (int j0 = k_begin; j0 < k_end; j0 += WARPS * 4) {
        const int j = j0 + warp * 4 + kg;
        const bool valid = j < k_end;
        uint4 k0, k1, v0, v1;
        if (valid) {
            k0 = ld_stream(kb + (size_t)j * D);
            k1 = ld_stream(kb + (size_t)j * D + 8);
            v0 = ld_stream(vb + (size_t)j * D);
            v1 = ld_stream(vb + (size_t)j * D + 8);
        } else {
            k0 = k1 = v0 = v1 = make_uint4(0, 0, 0, 0);
        }
        float kf[16], vf[16];
        unpack8(k0, kf);
        unpack8(k1, kf + 8);
        unpack8(v0, vf);
        unpack8(v1, vf + 8);
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            float s = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) s = fmaf(qv[gi][e], kf[e], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            if (valid) {
                const float mn = fmaxf(m[gi], s);
                const float c = exp2f(m[gi] - mn);
                const float p = exp2f(s - mn);
                l[gi] = l[gi] * c + p;
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[gi][e] = fmaf(p, vf[e], acc[gi][e] * c);
                m[gi] = mn;
            }
        }
    }
    // Merge the four 8-lane key groups of the warp.
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[gi], off);
            const float lo = __shfl_xor_sync(0xffffffffu, l[gi], off);
            const float mn = fmaxf(m[gi], mo);
            const float c1 = mn == -INFINITY ? 0.0f : exp2f(m[gi] - mn);
            const float c2 = mn == -INFINITY ? 0.0f : exp2f(mo - mn);
            l[gi] = l[gi] * c1 + lo * c2;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float ao = __shfl_xor_sync(0xffffffffu, acc[gi][e], off);
                acc[gi][e] = acc[gi][e] * c1 + ao * c2;
            }
            m[gi] = mn;
        }
    }
    if (kg == 0) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            if (sub == 0) {
                red_ml[warp][gi][0] = m[gi];
                red_ml[warp][gi][1] = l[gi];
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) red_o[warp][gi][sub * 16 + e] = acc[gi][e];
        }
    }
    __syncthreads();
    // Merge the warps: thread t handles dims t (and t+128*k) of every head of the group.
    for (int idx = threadIdx.x; idx < G * D; idx += WARPS * 32) {
        const int gi = idx / D, d = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) mx = fmaxf(mx, red_ml[w][gi][0]);
        float lsum = 0.0f, o = 0.0f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const float c = mx == -INFINITY ? 0.0f : exp2f(red_ml[w][gi][0] - mx);
            lsum += red_ml[w][gi][1] * c;
            o += red_o[w][gi][d] * c;
        }
        const size_t part = ((size_t)b * Hq + g * G + gi) * n_split + split;
        ws_o[part * D + d] = o;
        if (d == 0) {
            ws_ml[part * 2] = mx;
            ws_ml[part * 2 + 1] = lsum;
        }
    }
}

__global__ void __launch_bounds__(D) k_attn_decode_combine(const float *__restrict__ ws_ml,
                                                           const float *__restrict__ ws_o,
                                                           int n_split, bf16 *__restrict__ out,
                                                           int Hq) {
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const size_t base = ((size_t)b * Hq + h) * n_split;
    float mx = -INFINITY;
    for (int s = 0; s < n_split; ++s) mx = fmaxf(mx, ws_ml[(base + s) * 2]);
    float lsum = 0.0f, o = 0.0f;
    for (int s = 0; s < n_split; ++s) {
        const float ms = ws_ml[(base + s) * 2];
        if (ms == -INFINITY) continue;
        const float c = exp2f(ms - mx);
        lsum += ws_ml[(base + s) * 2 + 1] * c;
        o += ws_o[(base + s) * D + d] * c;
    }
    out[((size_t)b * Hq + h) * D + d] = __float2bfloat16(o / lsum);
}

template <int G>
cudaError_t run(const Launch &lc, const bf16 *q, const bf16 *k_layer, const bf16 *v_layer,
                const Rows &r, int n_split, int kps, float *ws_ml, float *ws_o, bf16 *out, int Hq,
                int Hkv, int max_ctx) {
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    cudaError_t e = launch(lc, k_attn_decode_split<G>, dim3(n_split, Hkv, r.B), dim3(WARPS * 32), 0,
                           q, k_layer, v_layer, r, kps, ws_ml, ws_o, Hq, Hkv, max_ctx, scale_log2);
    if (e != cudaSuccess) return e;
    return launch(lc, k_attn_decode_combine, dim3(Hq, r.B), dim3(D), 0, (const float *)ws_ml,
                  (const float *)ws_o, n_split, out, Hq);
}

}  // namespace

cudaError_t launch_attn_decode(const Launch &lc, const bf16 *q, const bf16 *k_layer,
                               const bf16 *v_layer, const Rows &r, int n_split,
                               int keys_per_split, float *ws_ml, float *ws_o, bf16 *out, int Hq,
                               int Hkv, int max_ctx) {
    switch (Hq / Hkv) {
        case 1: return run<1>(lc, q, k_layer, v_layer, r, n_split, keys_per_split, ws_ml, ws_o, out, Hq, Hkv, max_ctx);
        case 2: return run<2>(lc, q, k_layer, v_layer, r, n_split, keys_per_split, ws_ml, ws_o, out, Hq, Hkv, max_ctx);
        case 4: return run<4>(lc, q, k_layer, v_layer, r, n_split, keys_per_split, ws_ml, ws_o, out, Hq, Hkv, max_ctx);
        case 8: return run<8>(lc, q, k_layer, v_layer, r, n_split, keys_per_split, ws_ml, ws_o, out, Hq, Hkv, max_ctx);
    }
    return cudaErrorInvalidValue;
}

}  // namespace q3
