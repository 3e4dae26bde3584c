// Tied lm_head fused with greedy argmax: next[b] = argmax_v E[v] . x[b], lowest index on ties.
//
// The head reuses the embedding table ("手写Qwen3-0.6B推理", Qwen3Model: lm_head.weight =
// embed_tokens.weight) and is applied only to each sequence's last row ("第 3 章", 4.1);
// the greedy choice is torch.argmax's ("第 3 章", 4.3 Sampler: argmax when no temperature),
// which returns the first maximal index.
//
// Pass 1: a grid-stride sweep over vocabulary rows, two rows per warp, E rows streamed once
// from HBM and dotted with every x[b] (staged in shared memory).  Lane b keeps the running
// best (value, index) of batch row b; each CTA writes one partial per b.  Logits are
// stored too when asked for.  Pass 2: one CTA per b reduces the partials, writes the token
// and records the slot's new length (position of its last row + 1).

#include "kernels.h"

namespace q3 {

namespace {

constexpr int WARPS = 4, RPW = 2, MAX_B = 32;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

template <int KV>
__global__ void __launch_bounds__(WARPS * 32) k_lmhead(const bf16 *__restrict__ X, int B,
                                                      const bf16 *__restrict__ E, int V,
                                                      float *__restrict__ logits,
                                                      float *__restrict__ part_val,
                                                      int32_t *__restrict__ part_idx, int b_off,
                                                      int B_total) {
    extern __shared__ __align__(16) uint4 xs[];  // [B][C/8]
    __shared__ float red_v[WARPS][MAX_B];
    __shared__ int red_i[WARPS][MAX_B];
    constexpr int C = KV * 256;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const uint4 *xg = reinterpret_cast<const uint4 *>(X);
    for (int i = threadIdx.x; i < B * (C / 8); i += WARPS * 32) xs[i] = xg[i];
    __syncthreads();

    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    const int stride = gridDim.x * WARPS * RPW;
    for (int row0 = (blockIdx.x * WARPS + warp) * RPW; row0 < V; row0 += stride) {
        uint4 w[RPW][KV];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int row = min(row0 + r, V - 1);
#pragma unroll
            for (int i = 0; i < KV; ++i) w[r][i] = ld_stream(E + (size_t)row * C + (i * 32 + lane) * 8);
        }
        for (int b = 0; b < B; ++b) {
            float acc[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) acc[r] = 0.0f;
#pragma unroll
            for (int i = 0; i < KV; ++i) {
                const uint4 x = xs[b * (C / 8) + i * 32 + lane];
#pragma unroll
                for (int r = 0; r < RPW; ++r) acc[r] = dot8(w[r][i], x, acc[r]);
            }
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const float v = warp_sum(acc[r]);
                const int row = row0 + r;
                if (row < V) {
                    if (lane == b && better(v, row, best_v, best_i)) {
                        best_v = v;
                        best_i = row;
                    }
                    if (logits && lane == 0) logits[(size_t)(b_off + b) * V + row] = v;
                }
            }
        }
    }
    if (lane < B) {
        red_v[warp][lane] = best_v;
        red_i[warp][lane] = best_i;
    }
    __syncthreads();
    if (warp == 0 && lane < B) {
        float bv = red_v[0][lane];
        int bi = red_i[0][lane];
#pragma unroll
        for (int w = 1; w < WARPS; ++w)
            if (better(red_v[w][lane], red_i[w][lane], bv, bi)) {
                bv = red_v[w][lane];
                bi = red_i[w][lane];
            }
        part_val[(size_t)(b_off + lane) * gridDim.x + blockIdx.x] = bv;
        part_idx[(size_t)(b_off + lane) * gridDim.x + blockIdx.x] = bi;
    }
}

__global__ void __launch_bounds__(256) k_argmax_reduce(const float *__restrict__ part_val,
                                                       const int32_t *__restrict__ part_idx,
                                                       int n_parts, int32_t *__restrict__ next_tok,
                                                       Rows r) {
    __shared__ float sv[256];
    __shared__ int si[256];
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int p = threadIdx.x; p < n_parts; p += 256) {
        const float v = part_val[(size_t)b * n_parts + p];
        const int i = part_idx[(size_t)b * n_parts + p];
        if (better(v, i, bv, bi)) {
            bv = v;
            bi = i;
        }
    }
    sv[threadIdx.x] = bv;
    si[threadIdx.x] = bi;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (threadIdx.x < s && better(sv[threadIdx.x + s], si[threadIdx.x + s], sv[threadIdx.x], si[threadIdx.x])) {
            sv[threadIdx.x] = sv[threadIdx.x + s];
            si[threadIdx.x] = si[threadIdx.x + s];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        next_tok[b] = si[0];
        if (r.ctx_len) {
            const int row = r.cu_seqlens ? r.cu_seqlens[b + 1] - 1 : b;
            r.ctx_len[r.row_slot[row]] = r.row_pos[row] + 1;
        }
    }
}

template <int KV>
cudaError_t run(const Launch &lc, const bf16 *X, int B, const bf16 *E, int V, float *logits,
                float *part_val, int32_t *part_idx, int n_parts, int32_t *next_tok, const Rows &r, uint32_t *err) {
    cudaError_t e;
    constexpr int C = KV * 256;
    if (B > 8 && C == 1024) {
        // 9..32 rows per pass on the tensor cores (the SIMT pass is compute-bound there), one
        // wave of CTAs: one partial per SM and row
        n_parts = n_parts < lmhead_mma_parts(lc.num_sms) ? n_parts : lmhead_mma_parts(lc.num_sms);
        for (int b0 = 0; b0 < B; b0 += MAX_B) {
            const int bc = B - b0 < MAX_B ? B - b0 : MAX_B;
            e = launch_lmhead_mma(lc, X + (size_t)b0 * C, bc, C, E, V, logits ? logits + (size_t)b0 * V : nullptr,
                                  part_val + (size_t)b0 * n_parts, part_idx + (size_t)b0 * n_parts, n_parts, err);
            if (e != cudaSuccess) return e;
        }
    } else {
        e = cudaFuncSetAttribute(k_lmhead<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 MAX_B * KV * 256 * (int)sizeof(bf16));
        if (e != cudaSuccess) return e;
        for (int b0 = 0; b0 < B; b0 += MAX_B) {
            const int bc = B - b0 < MAX_B ? B - b0 : MAX_B;
            e = launch(lc, k_lmhead<KV>, dim3(n_parts), dim3(WARPS * 32), (size_t)bc * C * sizeof(bf16),
                       X + (size_t)b0 * C, bc, E, V, logits, part_val, part_idx, b0, B);
            if (e != cudaSuccess) return e;
        }
    }
    return launch(lc, k_argmax_reduce, dim3(B), dim3(256), 0, (const float *)part_val,
                  (const int32_t *)part_idx, n_parts, next_tok, r);
}

}  // namespace

int lmhead_parts(int num_sms) { return num_sms * 4; }

cudaError_t launch_lmhead_argmax(const Launch &lc, const bf16 *X, int B, int C, const bf16 *E,
                                 int V, float *logits, float *part_val, int32_t *part_idx,
                                 int n_parts, int32_t *next_tok, const Rows &r, uint32_t *err) {
    switch (C) {
        case 256: return run<1>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
        case 512: return run<2>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
        case 768: return run<3>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
        case 1024: return run<4>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
        case 1536: return run<6>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
        case 2048: return run<8>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
        case 2560: return run<10>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
        case 3072: return run<12>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
        case 4096: return run<16>(lc, X, B, E, V, logits, part_val, part_idx, n_parts, next_tok, r, err);
    }
    return cudaErrorInvalidValue;
}

}  // namespace q3
