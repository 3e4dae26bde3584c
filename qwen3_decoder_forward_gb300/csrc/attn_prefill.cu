// Causal GQA prefill attention over packed, ragged sequences (flash-style, online softmax).
//
//   o_h[i] = sum_{j<=i} softmax_j(q_h[i] . k_g[j] / sqrt(128)) v_g[j],  g = h / (Hq/Hkv)
// ("手写Qwen3-0.6B推理", Attention; "第 3 章", 3.3: lower-triangular mask, K/V shared by
// Hq/Hkv query heads; "从零开始写Qwen3", Attn: scale 1/sqrt(D)).  Scores and the softmax
// are fp32; probabilities are rounded to bf16 for the P.V product.  Keys come from the
// layer's KV cache (already normalised and rotated), so prefill and decode read the same
// bytes.
//
// CTA = (64-query tile, query head, sequence), 4 warps of 16 query rows.  K/V tiles of 64
// keys are double-buffered in shared memory with cp.async; S = QK^T and O += PV use
// mma.sync m16n8k16, P stays in registers.  Tiles above the diagonal are skipped, the
// diagonal tile is masked.

#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int BQ = 64, BKV = 64, THREADS = 128;
constexpr int KV_TILE_BYTES = BKV * D * 2;          // 16 KB
constexpr int SMEM_BYTES = 2 * 2 * KV_TILE_BYTES;  // K and V, double-buffered

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N));
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t *r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_t(uint32_t *r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float *c, const uint32_t *a, const uint32_t *b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Byte offset of 16-byte chunk ch (0..15) of row `row` in a [64][128] bf16 tile.
__device__ __forceinline__ int swz(int row, int ch) { return row * 256 + ((ch ^ (row & 7)) << 4); }

__global__ void __launch_bounds__(THREADS) k_attn_prefill(
    const bf16 *__restrict__ q, const bf16 *__restrict__ k_layer, const bf16 *__restrict__ v_layer,
    const int32_t *__restrict__ cu, const int32_t *__restrict__ slots, bf16 *__restrict__ out,
    int Hq, int Hkv, int max_ctx, float scale_log2) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_wait();
    // longest tiles first: query tile index counts down with blockIdx.x
    const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int start = cu[b], len = cu[b + 1] - start;
    const int q0 = qt * BQ;
    if (q0 >= len) return;
    const int g = h / (Hq / Hkv);
    const int slot = slots[b];
    const bf16 *kbase = k_layer + ((size_t)slot * Hkv + g) * max_ctx * D;
    const bf16 *vbase = v_layer + ((size_t)slot * Hkv + g) * max_ctx * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Q fragments of this warp's 16 rows (A operand of m16n8k16, 8 k-steps over D).
    // Staged through the first K buffer, which is then reused.
    uint32_t qf[8][4];
    {
        uint8_t *sq = smem;
        for (int c = tid; c < BQ * 16; c += THREADS) {
            const int row = c >> 4, ch = c & 15;
            const int qi = min(q0 + row, len - 1);
            cp_async16(smem_u32(sq + swz(row, ch)), q + ((size_t)(start + qi) * Hq + h) * D + ch * 8);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int row = warp * 16 + (lane & 15);
            ldmatrix_x4(qf[kk], smem_u32(sq + swz(row, kk * 2 + (lane >> 4))));
        }
        __syncthreads();
    }

    const int kv_end = min(len, q0 + BQ);  // keys needed by this tile: 0 .. kv_end-1
    const int n_tiles = (kv_end + BKV - 1) / BKV;

    auto load_kv = [&](int buf, int t) {
        uint8_t *sk = smem + buf * 2 * KV_TILE_BYTES;
        uint8_t *sv = sk + KV_TILE_BYTES;
        const int j0 = t * BKV;
        for (int c = tid; c < BKV * 16; c += THREADS) {
            const int row = c >> 4, ch = c & 15;
            const int j = j0 + row;
            const bool ok = j < kv_end;
            const int jj = ok ? j : 0;
            cp_async16_zfill(smem_u32(sk + swz(row, ch)), kbase + (size_t)jj * D + ch * 8, ok);
            cp_async16_zfill(smem_u32(sv + swz(row, ch)), vbase + (size_t)jj * D + ch * 8, ok);
        }
    };

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.0f, 0.0f};
    const int gq = lane >> 2, tq = lane & 3;
    const int qrow0 = q0 + warp * 16 + gq;  // this thread's query rows: qrow0 and qrow0 + 8

    load_kv(0, 0);
    cp_async_commit();
    for (int t = 0; t < n_tiles; ++t) {
        if (t + 1 < n_tiles) load_kv((t + 1) & 1, t + 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const uint8_t *sk = smem + (t & 1) * 2 * KV_TILE_BYTES;
        const uint8_t *sv = sk + KV_TILE_BYTES;

        // S = Q K^T for 16 rows x 64 keys (8 n-tiles of 8 keys).
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int nj = 0; nj < 4; ++nj) {
                const int row = nj * 16 + (lane & 7) + ((lane >> 4) << 3);
                uint32_t r[4];
                ldmatrix_x4(r, smem_u32(sk + swz(row, kk * 2 + ((lane >> 3) & 1))));
                const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
                mma_bf16(s[nj * 2], qf[kk], b0);
                mma_bf16(s[nj * 2 + 1], qf[kk], b1);
            }
        }
        // Causal mask (only tiles that reach past the first query row need it).
        const int j0 = t * BKV;
        if (j0 + BKV - 1 > q0) {
#pragma unroll
            for (int ni = 0; ni < 8; ++ni)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = j0 + ni * 8 + 2 * tq + (e & 1);
                    const int i = qrow0 + (e >> 1) * 8;
                    if (j > i || j >= kv_end) s[ni][e] = -INFINITY;
                }
        }
        // Online softmax per row (rows gq and gq+8 of the warp tile; 4 lanes share a row).
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float mx = -INFINITY;
#pragma unroll
            for (int ni = 0; ni < 8; ++ni) mx = fmaxf(mx, fmaxf(s[ni][hr * 2], s[ni][hr * 2 + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_r[hr], mx);
            const float corr = m_new == -INFINITY ? 1.0f : exp2f((m_r[hr] - m_new) * scale_log2);
            const float mb = m_new == -INFINITY ? 0.0f : m_new * scale_log2;
            float sum = 0.0f;
#pragma unroll
            for (int ni = 0; ni < 8; ++ni) {
                const float p0 = exp2f(s[ni][hr * 2] * scale_log2 - mb);
                const float p1 = exp2f(s[ni][hr * 2 + 1] * scale_log2 - mb);
                s[ni][hr * 2] = p0;
                s[ni][hr * 2 + 1] = p1;
                sum += p0 + p1;
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            l_r[hr] = l_r[hr] * corr + sum;
            m_r[hr] = m_new;
#pragma unroll
            for (int di = 0; di < 16; ++di) {
                o[di][hr * 2] *= corr;
                o[di][hr * 2 + 1] *= corr;
            }
        }
        // O += P V: P (16 x 64) as A fragments, V (64 keys x 128) via ldmatrix.trans.
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 16 keys per step
            uint32_t pa[4];
            pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int dj = 0; dj < 8; ++dj) {  // 16 output columns per ldmatrix.x4
                const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = dj * 2 + (lane >> 4);
                uint32_t r[4];
                ldmatrix_x4_t(r, smem_u32(sv + swz(row, ch)));
                const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
                mma_bf16(o[dj * 2], pa, b0);
                mma_bf16(o[dj * 2 + 1], pa, b1);
            }
        }
        __syncthreads();
    }
    pdl_trigger();

#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int i = qrow0 + hr * 8;
        if (i >= len) continue;
        const float inv = 1.0f / l_r[hr];
        bf16 *dst = out + ((size_t)(start + i) * Hq + h) * D;
#pragma unroll
        for (int di = 0; di < 16; ++di) {
            const int col = di * 8 + 2 * tq;
            *reinterpret_cast<uint32_t *>(dst + col) =
                pack_bf16x2(o[di][hr * 2] * inv, o[di][hr * 2 + 1] * inv);
        }
    }
}

}  // namespace

cudaError_t launch_attn_prefill(const Launch &lc, const bf16 *q, const bf16 *k_layer,
                                const bf16 *v_layer, const int32_t *cu_seqlens,
                                const int32_t *slots, int B, int max_len, bf16 *out, int Hq,
                                int Hkv, int max_ctx) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    const dim3 grid((max_len + BQ - 1) / BQ, Hq, B);
    return launch(lc, k_attn_prefill, grid, dim3(THREADS), SMEM_BYTES, q, k_layer, v_layer,
                  cu_seqlens, slots, out, Hq, Hkv, max_ctx, scale_log2);
}

}  // namespace q3
