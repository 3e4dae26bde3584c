// Prefill projection GEMM, out[M,N] = A[M,K] . W[N,K]^T with bf16 operands and fp32
// accumulation, for the QKV, o, gate_up and down projections ("手写Qwen3-0.6B推理",
// Attention and MLP: nn.Linear without bias; "第 3 章", 3.3/3.4: merged qkv_proj and
// gate_up_proj).
//
// Warp-level mma.sync (m16n8k16) kernel: 128x128x32 CTA tiles, 8 warps of 64x32, a
// 4-stage cp.async ring with an XOR-swizzled shared layout read by ldmatrix.  Rows of A
// beyond M are clamped on load and dropped on store (ragged token counts).  Epilogues:
//   EPI_F32        store fp32
//   EPI_RESID_ADD  add into the fp32 residual stream (o_proj and down_proj: "h <- h + ...")
//   EPI_SWIGLU     W rows interleaved (gate_j, up_j): store bf16 silu(gate)*up
//                  ("手写Qwen3-0.6B推理", MLP; "第 3 章", 3.4 act_fn on the merged output)

#include "kernels.h"

namespace q3 {

namespace {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 4, THREADS = 256;
constexpr int TILE_BYTES = BM * BK * 2;  // one operand tile of one stage
constexpr int SMEM_BYTES = STAGES * 2 * TILE_BYTES;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
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
__device__ __forceinline__ void mma_bf16(float *c, const uint32_t *a, const uint32_t *b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Byte offset of 16-byte chunk `ch` (0..3) of tile row `row` (64-byte rows).
__device__ __forceinline__ int swz(int row, int ch) { return row * 64 + ((ch ^ ((row >> 1) & 3)) << 4); }

template <int EPI>
__global__ void __launch_bounds__(THREADS) k_gemm(const bf16 *__restrict__ A, int M, int K,
                                                  const bf16 *__restrict__ W, int N, void *out) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_wait();
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;

    auto load_stage = [&](int stage, int kt) {
        uint8_t *sA = smem + stage * 2 * TILE_BYTES;
        uint8_t *sB = sA + TILE_BYTES;
        const int k0 = kt * BK;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = tid + i * THREADS;
            const int row = c >> 2, ch = c & 3;
            const int ar = min(m0 + row, M - 1);
            cp_async16(smem_u32(sA + swz(row, ch)), A + (size_t)ar * K + k0 + ch * 8);
            cp_async16(smem_u32(sB + swz(row, ch)), W + (size_t)(n0 + row) * K + k0 + ch * 8);
        }
    };

    float acc[4][4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.0f;

    const int KT = K / BK;
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < KT) load_stage(s, s);
        cp_async_commit();
    }
    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        const int nk = kt + STAGES - 1;
        if (nk < KT) load_stage(nk % STAGES, nk);
        cp_async_commit();
        const uint8_t *sA = smem + (kt % STAGES) * 2 * TILE_BYTES;
        const uint8_t *sB = sA + TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t af[4][4], bfr[4][2];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi) {
                const int row = wm * 64 + mi * 16 + (lane & 15);
                ldmatrix_x4(af[mi], smem_u32(sA + swz(row, kk * 2 + (lane >> 4))));
            }
#pragma unroll
            for (int nj = 0; nj < 2; ++nj) {
                const int row = wn * 32 + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
                uint32_t r[4];
                ldmatrix_x4(r, smem_u32(sB + swz(row, kk * 2 + ((lane >> 3) & 1))));
                bfr[nj * 2][0] = r[0];
                bfr[nj * 2][1] = r[1];
                bfr[nj * 2 + 1][0] = r[2];
                bfr[nj * 2 + 1][1] = r[3];
            }
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) mma_bf16(acc[mi][ni], af[mi], bfr[ni]);
        }
    }
    cp_async_wait<0>();
    pdl_trigger();

    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int row = m0 + wm * 64 + mi * 16 + g + half * 8;
            if (row >= M) continue;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int col = n0 + wn * 32 + ni * 8 + 2 * t;
                const float v0 = acc[mi][ni][half * 2], v1 = acc[mi][ni][half * 2 + 1];
                if (EPI == EPI_F32) {
                    *reinterpret_cast<float2 *>((float *)out + (size_t)row * N + col) = make_float2(v0, v1);
                } else if (EPI == EPI_RESID_ADD) {
                    float2 *p = reinterpret_cast<float2 *>((float *)out + (size_t)row * N + col);
                    float2 r = *p;
                    r.x += v0;
                    r.y += v1;
                    *p = r;
                } else {
                    ((bf16 *)out)[(size_t)row * (N / 2) + (col >> 1)] = __float2bfloat16(silu(v0) * v1);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemm(const Launch &lc, const bf16 *A, int M, int K, const bf16 *W, int N,
                        int epi, void *out) {
    if (M <= 0) return cudaSuccess;
    if (N % BN != 0 || K % BK != 0) return cudaErrorInvalidValue;
    const dim3 grid(N / BN, (M + BM - 1) / BM);
    switch (epi) {
        case EPI_F32:
            cudaFuncSetAttribute(k_gemm<EPI_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            return launch(lc, k_gemm<EPI_F32>, grid, dim3(THREADS), SMEM_BYTES, A, M, K, W, N, out);
        case EPI_RESID_ADD:
            cudaFuncSetAttribute(k_gemm<EPI_RESID_ADD>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            return launch(lc, k_gemm<EPI_RESID_ADD>, grid, dim3(THREADS), SMEM_BYTES, A, M, K, W, N, out);
        case EPI_SWIGLU:
            cudaFuncSetAttribute(k_gemm<EPI_SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            return launch(lc, k_gemm<EPI_SWIGLU>, grid, dim3(THREADS), SMEM_BYTES, A, M, K, W, N, out);
    }
    return cudaErrorInvalidValue;
}

}  // namespace q3
