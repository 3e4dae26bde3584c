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

// ---- v2: one weight block per CTA, fetched by a bulk copy before the dependency wait -------
//
// For M <= 8 rows.  CTA i owns weight rows [i*R, i*R + R): thread 0 starts one bulk
// asynchronous copy of that contiguous block into shared memory, then the CTA waits for the
// preceding kernel (programmatic dependent launch), so the block streams in while the
// previous kernel is still running.  With NORM the inputs are fp32 residual rows that are
// RMS-normalised on the way into shared memory ("手写Qwen3-0.6B推理", Qwen3RMSNorm; the norm
// of "第 3 章" 3.2 folded into its consumer); otherwise they are bf16 rows.
constexpr int V2_WARPS = 8;
constexpr int V2_MAX_M = 8;

template <int EPI, bool NORM, int KV>
__global__ void __launch_bounds__(V2_WARPS * 32) k_gemv_bulk(const void *__restrict__ Xin, int M,
                                                            const bf16 *__restrict__ W, int N, int R,
                                                            void *out, const float *__restrict__ gain,
                                                            float eps, uint32_t *err,
                                                            const bf16 *__restrict__ W_ahead) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int K = KV * 256;
    constexpr int RPW = EPI == EPI_SWIGLU ? 2 : 1;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint4 *ws = reinterpret_cast<uint4 *>(smem + 128);  // [R][K/8]
    uint4 *xs = ws + (size_t)R * (K / 8);                 // [M][K/8]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * R;
    const int nrows = min(R, N - row0);
    // One bulk copy per weight row, issued by the 32 lanes of warp 0: many copies in flight
    // per SM (a single large copy per CTA keeps too few bytes in flight to fill HBM).
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(bar, 1);
            mbar_expect_tx(bar, (uint32_t)nrows * K * 2);
        }
        __syncwarp();
        for (int rr = lane; rr < nrows; rr += 32)
            bulk_g2s(ws + (size_t)rr * (K / 8), W + (size_t)(row0 + rr) * K, K * 2, bar);
    } else if (warp == 1 && lane == 0 && W_ahead) {
        // The same block of a projection that runs later (the next layer's): bring it into L2
        // now, so HBM keeps streaming while the dependency chain runs from L2.
        prefetch_l2(W_ahead + (size_t)row0 * K, (uint32_t)nrows * K * 2);
    }
    float4 gv[NORM ? 2 * KV : 1];  // static gains: loaded before the dependency wait
    if (NORM) {
#pragma unroll
        for (int i = 0; i < 2 * KV; ++i) gv[i] = reinterpret_cast<const float4 *>(gain)[i * 32 + lane];
    }
    pdl_wait();
    pdl_trigger();
    if (NORM) {
        const float *res = static_cast<const float *>(Xin);
        for (int b = warp; b < M; b += V2_WARPS) {
            const float4 *rp = reinterpret_cast<const float4 *>(res + (size_t)b * K);
            float4 v[2 * KV];
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < 2 * KV; ++i) {
                v[i] = rp[i * 32 + lane];
                ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
            }
            const float inv = rsqrtf(warp_sum(ss) / (float)K + eps);
            uint2 *dst = reinterpret_cast<uint2 *>(xs + (size_t)b * (K / 8));
#pragma unroll
            for (int i = 0; i < 2 * KV; ++i) {
                const float4 g = gv[i];
                uint2 o;
                o.x = pack_bf16x2(v[i].x * inv * g.x, v[i].y * inv * g.y);
                o.y = pack_bf16x2(v[i].z * inv * g.z, v[i].w * inv * g.w);
                dst[i * 32 + lane] = o;
            }
        }
    } else {
        const uint4 *xg = static_cast<const uint4 *>(Xin);
        for (int i = threadIdx.x; i < M * (K / 8); i += V2_WARPS * 32) xs[i] = xg[i];
    }
    __syncthreads();
    if (!mbar_wait_bounded(bar, 0, err)) {
        mbar_wait_bounded(bar, 0, nullptr);  // let the copy land before the CTA exits
        return;
    }
    for (int grp = warp; grp * RPW < nrows; grp += V2_WARPS) {
        const int lr = grp * RPW;  // local row
        for (int b = 0; b < M; ++b) {
            float acc[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) acc[r] = 0.0f;
#pragma unroll
            for (int i = 0; i < KV; ++i) {
                const uint4 x = xs[b * (K / 8) + i * 32 + lane];
#pragma unroll
                for (int r = 0; r < RPW; ++r) acc[r] = dot8(ws[(lr + r) * (K / 8) + i * 32 + lane], x, acc[r]);
            }
#pragma unroll
            for (int r = 0; r < RPW; ++r) acc[r] = warp_sum(acc[r]);
            if (lane == 0) {
                const int row = row0 + lr;
                if (EPI == EPI_F32) {
                    ((float *)out)[(size_t)b * N + row] = acc[0];
                } else if (EPI == EPI_RESID_ADD) {
                    ((float *)out)[(size_t)b * N + row] += acc[0];
                } else {
                    ((bf16 *)out)[(size_t)b * (N / 2) + (row >> 1)] = __float2bfloat16(silu(acc[0]) * acc[RPW - 1]);
                }
            }
        }
    }
}

template <int EPI, bool NORM, int KV>
cudaError_t run_bulk(const Launch &lc, const void *X, int M, const bf16 *W, int N, void *out,
                     const float *gain, float eps, uint32_t *err, const bf16 *W_ahead) {
    constexpr int K = KV * 256;
    int R = (N + lc.num_sms - 1) / lc.num_sms;
    R = (R + 1) & ~1;  // even: SwiGLU rows come in (gate, up) pairs
    const size_t smem = 128 + (size_t)R * K * 2 + (size_t)M * K * 2;
    cudaError_t e = cudaFuncSetAttribute(k_gemv_bulk<EPI, NORM, KV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch(lc, k_gemv_bulk<EPI, NORM, KV>, dim3((N + R - 1) / R), dim3(V2_WARPS * 32), smem, X, M,
                  W, N, R, out, gain, eps, err, W_ahead);
}

template <int EPI, bool NORM>
cudaError_t dispatch_bulk(const Launch &lc, const void *X, int M, int K, const bf16 *W, int N,
                          void *out, const float *gain, float eps, uint32_t *err, const bf16 *W_ahead) {
    switch (K) {
        case 1024: return run_bulk<EPI, NORM, 4>(lc, X, M, W, N, out, gain, eps, err, W_ahead);
        case 2048: return run_bulk<EPI, NORM, 8>(lc, X, M, W, N, out, gain, eps, err, W_ahead);
        case 3072: return run_bulk<EPI, NORM, 12>(lc, X, M, W, N, out, gain, eps, err, W_ahead);
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

bool gemv_fused_supported(int M, int K) {
    return M >= 1 && M <= V2_MAX_M && (K == 1024 || K == 2048 || K == 3072);
}

cudaError_t launch_gemv_fused(const Launch &lc, const void *X, int M, int K, const bf16 *W, int N,
                              int epi, void *out, const float *norm_gain, float eps, uint32_t *err,
                              const bf16 *W_ahead) {
    if (!gemv_fused_supported(M, K) || N % 2) return cudaErrorInvalidValue;
    const bool norm = norm_gain != nullptr;
    if (epi == EPI_F32)
        return norm ? dispatch_bulk<EPI_F32, true>(lc, X, M, K, W, N, out, norm_gain, eps, err, W_ahead)
                    : dispatch_bulk<EPI_F32, false>(lc, X, M, K, W, N, out, norm_gain, eps, err, W_ahead);
    if (epi == EPI_RESID_ADD)
        return norm ? dispatch_bulk<EPI_RESID_ADD, true>(lc, X, M, K, W, N, out, norm_gain, eps, err, W_ahead)
                    : dispatch_bulk<EPI_RESID_ADD, false>(lc, X, M, K, W, N, out, norm_gain, eps, err, W_ahead);
    return norm ? dispatch_bulk<EPI_SWIGLU, true>(lc, X, M, K, W, N, out, norm_gain, eps, err, W_ahead)
                : dispatch_bulk<EPI_SWIGLU, false>(lc, X, M, K, W, N, out, norm_gain, eps, err, W_ahead);
}

}  // namespace q3
