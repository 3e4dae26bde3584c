// Decode projections: out[M,N] = X[M,K] . W[N,K]^T for a handful of rows (M <= 32 per
// launch), bound by streaming W from HBM.  Same epilogues as the prefill GEMM.
//
// Each warp owns RPW consecutive weight rows and holds them in registers (K/256 16-byte
// loads per lane per row, issued before the kernel waits on its predecessor, so the
// weight stream of one kernel overlaps the tail of the previous one under programmatic
// dependent launch).  The M activation rows are staged in shared memory once per CTA and
// every weight row is dotted with all of them: weights are read from HBM exactly once.

#include "kernels.h"

namespace q3 {

namespace {

constexpr int WARPS = 4;
constexpr int MAX_M = 32;

template <int EPI, int KV, int RPW>
__global__ void __launch_bounds__(WARPS * 32) k_gemv(const bf16 *__restrict__ X, int M,
                                                    const bf16 *__restrict__ W, int N,
                                                    void *out) {
    extern __shared__ __align__(16) uint4 xs[];  // [M][K/8]
    constexpr int K = KV * 256;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * WARPS + warp) * RPW;
    const bool active = row0 < N;

    uint4 w[RPW][KV];
    if (active) {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int i = 0; i < KV; ++i)
                w[r][i] = ld_stream(W + (size_t)(row0 + r) * K + (i * 32 + lane) * 8);
    }
    pdl_wait();
    pdl_trigger();
    const uint4 *xg = reinterpret_cast<const uint4 *>(X);
    for (int i = threadIdx.x; i < M * (K / 8); i += WARPS * 32) xs[i] = xg[i];
    __syncthreads();
    if (!active) return;

    for (int b = 0; b < M; ++b) {
        float acc[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) acc[r] = 0.0f;
#pragma unroll
        for (int i = 0; i < KV; ++i) {
            const uint4 x = xs[b * (K / 8) + i * 32 + lane];
#pragma unroll
            for (int r = 0; r < RPW; ++r) acc[r] = dot8(w[r][i], x, acc[r]);
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) acc[r] = warp_sum(acc[r]);
        if (lane == 0) {
            if (EPI == EPI_F32) {
#pragma unroll
                for (int r = 0; r < RPW; ++r) ((float *)out)[(size_t)b * N + row0 + r] = acc[r];
            } else if (EPI == EPI_RESID_ADD) {
#pragma unroll
                for (int r = 0; r < RPW; ++r) ((float *)out)[(size_t)b * N + row0 + r] += acc[r];
            } else {
#pragma unroll
                for (int r = 0; r < RPW; r += 2)
                    ((bf16 *)out)[(size_t)b * (N / 2) + ((row0 + r) >> 1)] =
                        __float2bfloat16(silu(acc[r]) * acc[r + 1]);
            }
        }
    }
}

template <int EPI, int KV, int RPW>
cudaError_t run(const Launch &lc, const bf16 *X, int M, const bf16 *W, int N, void *out) {
    const size_t smem = (size_t)M * KV * 256 * sizeof(bf16);
    cudaError_t e = cudaFuncSetAttribute(k_gemv<EPI, KV, RPW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         MAX_M * KV * 256 * (int)sizeof(bf16));
    if (e != cudaSuccess) return e;
    const int rows_per_cta = WARPS * RPW;
    return launch(lc, k_gemv<EPI, KV, RPW>, dim3((N + rows_per_cta - 1) / rows_per_cta),
                  dim3(WARPS * 32), smem, X, M, W, N, out);
}

template <int EPI>
cudaError_t dispatch(const Launch &lc, const bf16 *X, int M, int K, const bf16 *W, int N, void *out) {
    // Two rows per warp where K is small (and always for the paired SwiGLU rows).
    switch (K) {
        case 1024: return run<EPI, 4, 2>(lc, X, M, W, N, out);
        case 2048: return EPI == EPI_SWIGLU ? run<EPI, 8, 2>(lc, X, M, W, N, out)
                                            : run<EPI, 8, 1>(lc, X, M, W, N, out);
        case 3072: return EPI == EPI_SWIGLU ? run<EPI, 12, 2>(lc, X, M, W, N, out)
                                            : run<EPI, 12, 1>(lc, X, M, W, N, out);
        case 4096: return EPI == EPI_SWIGLU ? run<EPI, 16, 2>(lc, X, M, W, N, out)
                                            : run<EPI, 16, 1>(lc, X, M, W, N, out);
        case 256: return run<EPI, 1, 2>(lc, X, M, W, N, out);
        case 512: return run<EPI, 2, 2>(lc, X, M, W, N, out);
        case 768: return run<EPI, 3, 2>(lc, X, M, W, N, out);
        case 1536: return run<EPI, 6, 2>(lc, X, M, W, N, out);
        case 2560: return run<EPI, 10, 2>(lc, X, M, W, N, out);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemv(const Launch &lc, const bf16 *X, int M, int K, const bf16 *W, int N,
                        int epi, void *out) {
    for (int m0 = 0; m0 < M; m0 += MAX_M) {
        const int mc = M - m0 < MAX_M ? M - m0 : MAX_M;
        const bf16 *Xc = X + (size_t)m0 * K;
        cudaError_t e;
        if (epi == EPI_F32)
            e = dispatch<EPI_F32>(lc, Xc, mc, K, W, N, (float *)out + (size_t)m0 * N);
        else if (epi == EPI_RESID_ADD)
            e = dispatch<EPI_RESID_ADD>(lc, Xc, mc, K, W, N, (float *)out + (size_t)m0 * N);
        else
            e = dispatch<EPI_SWIGLU>(lc, Xc, mc, K, W, N, (bf16 *)out + (size_t)m0 * (N / 2));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace q3
