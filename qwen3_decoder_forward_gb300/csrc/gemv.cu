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
                                                            const bf16 *__restrict__ W_ahead, float *zero_buf,
                                                            int zero_n) {
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
    const long long lim = wait_limit(err);
    float4 gv[NORM ? 2 * KV : 1];  // static gains: loaded before the dependency wait
    if (NORM) {
#pragma unroll
        for (int i = 0; i < 2 * KV; ++i) gv[i] = reinterpret_cast<const float4 *>(gain)[i * 32 + lane];
    }
    pdl_wait();
    pdl_trigger();
    if (zero_buf) {  // clear this CTA's share of a buffer a later kernel accumulates into
        const int per = (zero_n + gridDim.x - 1) / gridDim.x;
        for (int i = blockIdx.x * per + threadIdx.x; i < min(zero_n, (blockIdx.x + 1) * per); i += blockDim.x)
            zero_buf[i] = 0.0f;
    }
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
    if (!mbar_wait_ctx(bar, 0, err, lim)) {
        mbar_wait_bounded(bar, 0, nullptr);  // let the copy land before the CTA exits
        return;
    }
    // Each warp works on up to RB rows at once (rows warp, warp + 8, ...; SwiGLU pairs stay
    // together) with two accumulators per row, so the loads and the reductions of several rows
    // overlap instead of running one row after another.
    constexpr int RB = 4;
    const int n_grp = (nrows + RPW - 1) / RPW;
    for (int g0 = warp; g0 < n_grp; g0 += V2_WARPS * (RB / RPW)) {
        // groups of this warp in this pass (warp-uniform)
        const int ng = min(RB / RPW, (n_grp - g0 + V2_WARPS - 1) / V2_WARPS);
        for (int b = 0; b < M; ++b) {
            float prev[RB];  // residual values for RESID_ADD, loaded before the dot products
            if (EPI == EPI_RESID_ADD && lane == 0) {
#pragma unroll
                for (int r = 0; r < RB; ++r)
                    if (r < ng) prev[r] = ((const float *)out)[(size_t)b * N + row0 + g0 + r * V2_WARPS];
            }
            float acc[RB][2];
#pragma unroll
            for (int r = 0; r < RB; ++r) acc[r][0] = acc[r][1] = 0.0f;
#pragma unroll
            for (int i = 0; i < KV; ++i) {
                const uint4 x = xs[b * (K / 8) + i * 32 + lane];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const int grp = g0 + (r / RPW) * V2_WARPS;
                    const int lr = grp * RPW + (r % RPW);
                    if (r / RPW < ng) acc[r][i & 1] = dot8(ws[(size_t)lr * (K / 8) + i * 32 + lane], x, acc[r][i & 1]);
                }
            }
            float sum[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r)
                if (r / RPW < ng) sum[r] = warp_sum(acc[r][0] + acc[r][1]);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < RB; r += RPW) {
                    if (r / RPW >= ng) continue;
                    const int grp = g0 + (r / RPW) * V2_WARPS;
                    const int row = row0 + grp * RPW;
                    if (EPI == EPI_F32) {
                        ((float *)out)[(size_t)b * N + row] = sum[r];
                    } else if (EPI == EPI_RESID_ADD) {
                        ((float *)out)[(size_t)b * N + row] = prev[r] + sum[r];
                    } else {
                        ((bf16 *)out)[(size_t)b * (N / 2) + (row >> 1)] = __float2bfloat16(silu(sum[r]) * sum[r + 1]);
                    }
                }
            }
        }
    }
}

template <int EPI, bool NORM, int KV>
cudaError_t run_bulk(const Launch &lc, const void *X, int M, const bf16 *W, int N, void *out,
                     const float *gain, float eps, uint32_t *err, const bf16 *W_ahead, float *zero_buf,
                     int zero_n) {
    constexpr int K = KV * 256;
    int R = (N + lc.num_sms - 1) / lc.num_sms;
    R = (R + 1) & ~1;  // even: SwiGLU rows come in (gate, up) pairs
    const size_t smem = 128 + (size_t)R * K * 2 + (size_t)M * K * 2;
    cudaError_t e = cudaFuncSetAttribute(k_gemv_bulk<EPI, NORM, KV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch(lc, k_gemv_bulk<EPI, NORM, KV>, dim3((N + R - 1) / R), dim3(V2_WARPS * 32), smem, X, M,
                  W, N, R, out, gain, eps, err, W_ahead, zero_buf, zero_n);
}

template <int EPI, bool NORM>
cudaError_t dispatch_bulk(const Launch &lc, const void *X, int M, int K, const bf16 *W, int N,
                          void *out, const float *gain, float eps, uint32_t *err, const bf16 *W_ahead,
                          float *zero_buf, int zero_n) {
    switch (K) {
        case 1024: return run_bulk<EPI, NORM, 4>(lc, X, M, W, N, out, gain, eps, err, W_ahead, zero_buf, zero_n);
        case 2048: return run_bulk<EPI, NORM, 8>(lc, X, M, W, N, out, gain, eps, err, W_ahead, zero_buf, zero_n);
        case 3072: return run_bulk<EPI, NORM, 12>(lc, X, M, W, N, out, gain, eps, err, W_ahead, zero_buf, zero_n);
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
                              const bf16 *W_ahead, float *zero_buf, int zero_n) {
    if (!gemv_fused_supported(M, K) || N % 2) return cudaErrorInvalidValue;
    const bool norm = norm_gain != nullptr;
#define Q3_BULK(E, Nm) dispatch_bulk<E, Nm>(lc, X, M, K, W, N, out, norm_gain, eps, err, W_ahead, zero_buf, zero_n)
    if (epi == EPI_F32) return norm ? Q3_BULK(EPI_F32, true) : Q3_BULK(EPI_F32, false);
    if (epi == EPI_RESID_ADD) return norm ? Q3_BULK(EPI_RESID_ADD, true) : Q3_BULK(EPI_RESID_ADD, false);
    return norm ? Q3_BULK(EPI_SWIGLU, true) : Q3_BULK(EPI_SWIGLU, false);
#undef Q3_BULK
}

// ---- the whole MLP of a decode step in one kernel ------------------------------------------
//
//   out[b] += h[b] (this CTA's slice) + sum_j act[b][j] WdT[j]   over this CTA's act indices j
//   act[b][j] = silu(gate_j . m[b]) * (up_j . m[b]),  m[b] = RMSNorm(h[b]; gain)
// ("手写Qwen3-0.6B推理", MLP: down(silu(gate(x)) * up(x)); the residual add of
// Qwen3DecoderLayer).  CTA c owns act indices [c*NA, c*NA + NA): it bulk-copies their
// interleaved gate/up weight rows and the matching rows of the transposed down weight (WdT
// [I, C]) into shared memory before the dependency wait, so the down projection is split over
// the CTAs along its reduction dimension and each CTA adds its partial sums (and its slice of
// the residual h) into `out`, which must be zero on entry.  The fp32 additions of the CTAs
// land in an unspecified order (vector atomics), so results may differ between runs in the
// last bits.
constexpr int MLP_WARPS = 8;

template <int KV>
__global__ void __launch_bounds__(MLP_WARPS * 32) k_mlp_fused(const float *__restrict__ h, int M,
                                                             const float *__restrict__ gain, float eps,
                                                             const bf16 *__restrict__ Wgu, const bf16 *__restrict__ WdT,
                                                             int I, int NA, float *out, uint32_t *err,
                                                             const bf16 *__restrict__ Wgu_ahead,
                                                             const bf16 *__restrict__ WdT_ahead) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int C = KV * 256;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint4 *wgu = reinterpret_cast<uint4 *>(smem + 128);  // [2*NA][C/8]
    uint4 *wd = wgu + (size_t)2 * NA * (C / 8);           // [NA][C/8]
    uint4 *xs = wd + (size_t)NA * (C / 8);                // [M][C/8]
    float *act = reinterpret_cast<float *>(xs + (size_t)M * (C / 8));  // [M][NA]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int a0 = blockIdx.x * NA;
    const int na = min(NA, I - a0);
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(bar, 1);
            mbar_expect_tx(bar, (uint32_t)na * 3 * C * 2);
        }
        __syncwarp();
        for (int rr = lane; rr < 2 * na; rr += 32)
            bulk_g2s(wgu + (size_t)rr * (C / 8), Wgu + (size_t)(2 * a0 + rr) * C, C * 2, bar);
        for (int rr = lane; rr < na; rr += 32)
            bulk_g2s(wd + (size_t)rr * (C / 8), WdT + (size_t)(a0 + rr) * C, C * 2, bar);
    } else if (warp == 1 && lane == 0 && Wgu_ahead) {
        prefetch_l2(Wgu_ahead + (size_t)2 * a0 * C, (uint32_t)na * 2 * C * 2);
        prefetch_l2(WdT_ahead + (size_t)a0 * C, (uint32_t)na * C * 2);
    }
    const long long lim = wait_limit(err);
    float4 gv[2 * KV];
#pragma unroll
    for (int i = 0; i < 2 * KV; ++i) gv[i] = reinterpret_cast<const float4 *>(gain)[i * 32 + lane];
    pdl_wait();
    pdl_trigger();
    // residual slice of this CTA into out (other CTAs add their partials to the same rows)
    {
        const int per = (C + gridDim.x - 1) / gridDim.x;
        const int e0 = blockIdx.x * per, e1 = min(C, e0 + per);
        for (int i = threadIdx.x; i < M * per; i += blockDim.x) {
            const int b = i / per, e = e0 + i % per;
            if (e < e1) atomicAdd(out + (size_t)b * C + e, h[(size_t)b * C + e]);
        }
    }
    for (int b = warp; b < M; b += MLP_WARPS) {  // m[b] = RMSNorm(h[b]) into shared memory
        const float4 *rp = reinterpret_cast<const float4 *>(h + (size_t)b * C);
        float4 v[2 * KV];
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < 2 * KV; ++i) {
            v[i] = rp[i * 32 + lane];
            ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        }
        const float inv = rsqrtf(warp_sum(ss) / (float)C + eps);
        uint2 *dst = reinterpret_cast<uint2 *>(xs + (size_t)b * (C / 8));
#pragma unroll
        for (int i = 0; i < 2 * KV; ++i) {
            uint2 o;
            o.x = pack_bf16x2(v[i].x * inv * gv[i].x, v[i].y * inv * gv[i].y);
            o.y = pack_bf16x2(v[i].z * inv * gv[i].z, v[i].w * inv * gv[i].w);
            dst[i * 32 + lane] = o;
        }
    }
    __syncthreads();
    const bool ok = __syncthreads_and(mbar_wait_ctx(bar, 0, err, lim));
    if (!ok) {
        mbar_wait_bounded(bar, 0, nullptr);
        return;
    }
    // gate/up pairs -> act
    for (int j = warp; j < na; j += MLP_WARPS) {
        for (int b = 0; b < M; ++b) {
            float g = 0.0f, u = 0.0f;
#pragma unroll
            for (int i = 0; i < KV; ++i) {
                const uint4 x = xs[b * (C / 8) + i * 32 + lane];
                g = dot8(wgu[(size_t)(2 * j) * (C / 8) + i * 32 + lane], x, g);
                u = dot8(wgu[(size_t)(2 * j + 1) * (C / 8) + i * 32 + lane], x, u);
            }
            g = warp_sum(g);
            u = warp_sum(u);
            if (lane == 0) act[b * NA + j] = __bfloat162float(__float2bfloat16(silu(g) * u));
        }
    }
    __syncthreads();
    // down projection, split along its reduction dimension: this CTA's act indices only
    for (int b = 0; b < M; ++b) {
        for (int n0 = threadIdx.x * 4; n0 < C; n0 += blockDim.x * 4) {
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int j = 0; j < na; ++j) {
                const float a = act[b * NA + j];
                const uint2 w = *reinterpret_cast<const uint2 *>(reinterpret_cast<const bf16 *>(wd) + (size_t)j * C + n0);
                const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
                const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
                acc.x = fmaf(a, w01.x, acc.x);
                acc.y = fmaf(a, w01.y, acc.y);
                acc.z = fmaf(a, w23.x, acc.z);
                acc.w = fmaf(a, w23.y, acc.w);
            }
            atomicAdd(reinterpret_cast<float4 *>(out + (size_t)b * C + n0), acc);
        }
    }
}

template <int KV>
cudaError_t run_mlp(const Launch &lc, const float *h, int M, const float *gain, float eps, const bf16 *Wgu,
                    const bf16 *WdT, int I, float *out, uint32_t *err, const bf16 *Wgu_ahead, const bf16 *WdT_ahead) {
    constexpr int C = KV * 256;
    const int NA = (I + lc.num_sms - 1) / lc.num_sms;
    const size_t smem = 128 + (size_t)NA * 3 * C * 2 + (size_t)M * C * 2 + (size_t)M * NA * 4;
    cudaError_t e = cudaFuncSetAttribute(k_mlp_fused<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch(lc, k_mlp_fused<KV>, dim3((I + NA - 1) / NA), dim3(MLP_WARPS * 32), smem, h, M, gain, eps, Wgu,
                  WdT, I, NA, out, err, Wgu_ahead, WdT_ahead);
}

bool mlp_fused_supported(int M, int C, int I, int num_sms) {
    const int NA = (I + num_sms - 1) / num_sms;
    const size_t smem = 128 + (size_t)NA * 3 * C * 2 + (size_t)M * C * 2 + (size_t)M * NA * 4;
    return M >= 1 && M <= 4 && C == 1024 && smem <= 200 * 1024;
}

cudaError_t launch_mlp_fused(const Launch &lc, const float *h, int M, int C, const float *gain, float eps,
                             const bf16 *Wgu, const bf16 *WdT, int I, float *out, uint32_t *err,
                             const bf16 *Wgu_ahead, const bf16 *WdT_ahead) {
    if (!mlp_fused_supported(M, C, I, lc.num_sms)) return cudaErrorInvalidValue;
    return run_mlp<4>(lc, h, M, gain, eps, Wgu, WdT, I, out, err, Wgu_ahead, WdT_ahead);
}

// ---- tensor-core decode projection for 9..32 rows -------------------------------------------
//
// out[M,N] = X[M,K] . W[N,K]^T with the weights as the M side of mma.sync m16n8k16 and the
// batch rows as the N side.  CTA = 16 weight rows x one K slice (K/KS): the rows are bulk-
// copied into padded shared memory before the dependency wait, X (zero-padded to 32 rows) is
// loaded after it, the 4 warps split the K slice, and their partial tiles are summed through
// shared memory.  With KS > 1 (RESID_ADD only) the slices add into the output with atomics.
constexpr int MMA_ROWS = 16, MMA_MPAD = 32, MMA_WARPS = 4;

__device__ __forceinline__ void ldsm_x4(uint32_t *r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int EPI, int KS, int MP>  // MP: batch rows padded to 16 or 32
__global__ void __launch_bounds__(MMA_WARPS * 32) k_gemv_mma(const bf16 *__restrict__ X, int M, int K,
                                                             const bf16 *__restrict__ W, int N, void *out,
                                                             uint32_t *err) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int Kc = K / KS;
    const int stride = Kc * 2 + 16;  // padded row stride (bytes): conflict-free ldmatrix
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint8_t *ws = smem + 128;                      // [16][stride]
    uint8_t *xs = ws + MMA_ROWS * stride;          // [32][stride]
    float *red = reinterpret_cast<float *>(xs + MP * stride);  // [warps][16][MP]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * MMA_ROWS, ks = blockIdx.y, k0 = ks * Kc;
    uint64_t *xbar = bar + 1;
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(bar, 1);
            mbar_init(xbar, 1);
            mbar_expect_tx(bar, (uint32_t)MMA_ROWS * Kc * 2);
        }
        __syncwarp();
        if (lane < MMA_ROWS) bulk_g2s(ws + lane * stride, W + (size_t)(row0 + lane) * K + k0, Kc * 2, bar);
    }
    const long long lim = wait_limit(err);
    // rows of X beyond M are zero
    for (int i = threadIdx.x; i < (MP - M) * (Kc / 8); i += MMA_WARPS * 32)
        *reinterpret_cast<uint4 *>(xs + (M + i / (Kc / 8)) * stride + (i % (Kc / 8)) * 16) = make_uint4(0, 0, 0, 0);
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    // X rows by bulk copies: one round trip for the whole operand
    if (warp == 1) {
        if (lane == 0) mbar_expect_tx(xbar, (uint32_t)M * Kc * 2);
        __syncwarp();
        if (lane < M) bulk_g2s(xs + lane * stride, X + (size_t)lane * K + k0, Kc * 2, xbar);
    }
    const bool ok = __syncthreads_and(mbar_wait_ctx(bar, 0, err, lim) && mbar_wait_ctx(xbar, 0, err, lim));
    if (!ok) {
        mbar_wait_bounded(bar, 0, nullptr);
        mbar_wait_bounded(xbar, 0, nullptr);
        return;
    }
    float acc[MP / 8][4];
#pragma unroll
    for (int j = 0; j < MP / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    const int kq = Kc / MMA_WARPS;  // this warp's quarter of the slice
    const uint32_t wsa = smem_addr(ws), xsa = smem_addr(xs);
    for (int kk = warp * kq; kk < (warp + 1) * kq; kk += 16) {
        uint32_t a[4];
        ldsm_x4(a, wsa + (lane & 15) * stride + (kk + (lane >> 4) * 8) * 2);
#pragma unroll
        for (int nb = 0; nb < MP / 16; ++nb) {  // an ldmatrix.x4 per 16 padded batch rows
            uint32_t b[4];
            const int n = nb * 16 + (lane & 7) + ((lane >> 4) << 3);
            ldsm_x4(b, xsa + n * stride + (kk + ((lane >> 3) & 1) * 8) * 2);
            mma16816(acc[nb * 2], a, b[0], b[1]);
            mma16816(acc[nb * 2 + 1], a, b[2], b[3]);
        }
    }
    // partial tiles of the 4 warps -> shared memory, then sum
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < MP / 8; ++j) {
        float *rw = red + warp * MMA_ROWS * MP;
        rw[g * MP + j * 8 + 2 * t] = acc[j][0];
        rw[g * MP + j * 8 + 2 * t + 1] = acc[j][1];
        rw[(g + 8) * MP + j * 8 + 2 * t] = acc[j][2];
        rw[(g + 8) * MP + j * 8 + 2 * t + 1] = acc[j][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < MMA_ROWS * MP; i += MMA_WARPS * 32) {
        const int r = i / MP, b = i % MP;  // r: weight row, b: batch row
        if (b >= M) continue;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < MMA_WARPS; ++w) v += red[w * MMA_ROWS * MP + i];
        const int n = row0 + r;
        if (EPI == EPI_F32) {
            ((float *)out)[(size_t)b * N + n] = v;
        } else if (EPI == EPI_RESID_ADD) {
            if (KS == 1) ((float *)out)[(size_t)b * N + n] += v;
            else atomicAdd((float *)out + (size_t)b * N + n, v);
        } else if ((r & 1) == 0) {  // SwiGLU: rows (2j, 2j+1) = (gate_j, up_j)
            float up = 0.0f;
#pragma unroll
            for (int w = 0; w < MMA_WARPS; ++w) up += red[w * MMA_ROWS * MP + i + MP];
            ((bf16 *)out)[(size_t)b * (N / 2) + (n >> 1)] = __float2bfloat16(silu(v) * up);
        }
    }
}

// ---- tensor-core lm_head + argmax for 9..32 rows -----------------------------------------
//
// One CTA per SM walks 32-row tiles of the (tied) embedding table, tiles s, s + grid, ...: a
// producer warp keeps a two-stage ring of them filled with bulk copies (one 2 KB row a lane),
// and four MMA warps each multiply 16 of the tile's rows with 16 of the 32 (zero-padded) rows
// of x over the whole K (mma.sync m16n8k16, four independent accumulator chains per n-tile),
// store the logits when asked, and keep the running best (value, index) of their batch
// columns in registers -- lowest index on ties.  A warp frees a stage with an mbarrier
// arrival; nothing is reduced across warps until the end.  One partial per CTA and row goes
// to part_val/part_idx for the reduction kernel.
constexpr int LM_ROWS = 32, LM_STAGES = 2, LM_WARPS = 4, LM_BAR = 1;

__device__ __forceinline__ bool lm_better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

template <int KV>
__global__ void __launch_bounds__((LM_WARPS + 1) * 32) k_lmhead_mma(const bf16 *__restrict__ X, int M,
                                                                     const bf16 *__restrict__ E, int V,
                                                                     float *__restrict__ logits,
                                                                     float *__restrict__ part_val,
                                                                     int32_t *__restrict__ part_idx, uint32_t *err) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int C = KV * 256;
    constexpr int stride = C * 2 + 16;                 // padded row (bytes): conflict-free ldmatrix
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [LM_STAGES]
    uint64_t *empty = full + LM_STAGES;                   // [LM_STAGES]
    uint64_t *xbar = empty + LM_STAGES;
    uint8_t *ring = smem + 128;                                    // [LM_STAGES][LM_ROWS][stride]
    uint8_t *xs = ring + (size_t)LM_STAGES * LM_ROWS * stride;    // [32][stride]
    __shared__ float fin_v[2][MMA_MPAD];
    __shared__ int fin_i[2][MMA_MPAD];
    __shared__ volatile int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (V + LM_ROWS - 1) / LM_ROWS;
    const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const long long lim = wait_limit(err);
    if (threadIdx.x == 0) {
        for (int st = 0; st < LM_STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], LM_WARPS);
        }
        mbar_init(xbar, 1);
        s_abort = 0;
    }
    for (int i = threadIdx.x; i < (MMA_MPAD - M) * (C / 8); i += blockDim.x)  // rows of x beyond M are zero
        *reinterpret_cast<uint4 *>(xs + (M + i / (C / 8)) * stride + (i % (C / 8)) * 16) = make_uint4(0, 0, 0, 0);
    if (V % LM_ROWS)  // rows past V in a partial last tile must be finite: zero the stages once
        for (int i = threadIdx.x; i < LM_STAGES * LM_ROWS * (C / 8); i += blockDim.x)
            *reinterpret_cast<uint4 *>(ring + (i / (C / 8)) * stride + (i % (C / 8)) * 16) = make_uint4(0, 0, 0, 0);
    __syncthreads();

    if (warp == LM_WARPS) {
        // ---- producer: tiles into the ring, x after the dependency wait ----
        auto issue = [&](int i) {
            const int st = i % LM_STAGES, r0 = (blockIdx.x + i * gridDim.x) * LM_ROWS;
            const int nr = min(LM_ROWS, V - r0);
            if (lane == 0) mbar_expect_tx(&full[st], (uint32_t)nr * C * 2);
            __syncwarp();
            if (lane < nr)
                bulk_g2s(ring + ((size_t)st * LM_ROWS + lane) * stride, E + (size_t)(r0 + lane) * C, C * 2, &full[st]);
        };
        int issued = min(LM_STAGES, my_tiles);
        for (int i = 0; i < issued; ++i) issue(i);
        pdl_wait();
        pdl_trigger();
        if (lane == 0) mbar_expect_tx(xbar, (uint32_t)M * C * 2);
        __syncwarp();
        if (lane < M) bulk_g2s(xs + lane * stride, X + (size_t)lane * C, C * 2, xbar);
        for (int i = LM_STAGES; i < my_tiles; ++i) {
            // the stage is free once the MMA warps are done with tile i - LM_STAGES
            bool ok = true;
            if (lane == 0) {
                const long long t0 = clock64();
                while (!mbar_try_wait(&empty[i % LM_STAGES], (uint32_t)((i / LM_STAGES - 1) & 1))) {
                    if (s_abort) { ok = false; break; }
                    if (clock64() - t0 > lim) {
                        if (err) atomicOr(err, ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            issue(i);
            issued = i + 1;
        }
        // the copies in flight land before the CTA may exit (the MMA warps took them all
        // unless a wait gave up)
        if (lane == 0) {
            for (int j = max(0, issued - LM_STAGES); j < issued; ++j)
                mbar_wait_bounded(&full[j % LM_STAGES], (uint32_t)((j / LM_STAGES) & 1), nullptr);
            mbar_wait_bounded(xbar, 0, nullptr);
        }
        return;
    }

    // ---- MMA warps: rows 16 mt .. of each tile, batch columns 16 nh .. 16 nh + 15 ----
    const int mt = warp & 1, nh = warp >> 1;
    const bool active = 16 * nh < M;
    const int g = lane >> 2, t = lane & 3;
    float bv[2][2];
    int bi[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            bv[nt][j] = -INFINITY;
            bi[nt][j] = 0x7fffffff;
        }
    bool ok = !__any_sync(0xffffffffu, !mbar_wait_ctx(xbar, 0, err, lim));
    const uint32_t xsa = smem_addr(xs) + (16 * nh + (lane & 7) + ((lane >> 4) << 3)) * stride + ((lane >> 3) & 1) * 16;
    for (int i = 0; ok && i < my_tiles; ++i) {
        const int st = i % LM_STAGES;
        if (__any_sync(0xffffffffu, !mbar_wait_ctx(&full[st], (uint32_t)((i / LM_STAGES) & 1), err, lim))) {
            ok = false;
            break;
        }
        if (active) {
            const uint32_t wsa =
                smem_addr(ring + ((size_t)st * LM_ROWS + mt * 16 + (lane & 15)) * stride) + (lane >> 4) * 16;
            float acc[2][4][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) acc[nt][ch][0] = acc[nt][ch][1] = acc[nt][ch][2] = acc[nt][ch][3] = 0.0f;
#pragma unroll 2
            for (int kk = 0; kk < C; kk += 64) {
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const int k = kk + ch * 16;
                    uint32_t a[4], b[4];
                    ldsm_x4(a, wsa + k * 2);
                    ldsm_x4(b, xsa + k * 2);
                    mma16816(acc[0][ch], a, b[0], b[1]);
                    mma16816(acc[1][ch], a, b[2], b[3]);
                }
            }
            const int r0 = (blockIdx.x + i * gridDim.x) * LM_ROWS + mt * 16;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int e = 2 * h + j;
                        const float v = acc[nt][0][e] + acc[nt][1][e] + acc[nt][2][e] + acc[nt][3][e];
                        const int row = r0 + g + 8 * h, b = 16 * nh + 8 * nt + 2 * t + j;
                        if (row < V && b < M) {
                            if (logits) logits[(size_t)b * V + row] = v;
                            if (lm_better(v, row, bv[nt][j], bi[nt][j])) {
                                bv[nt][j] = v;
                                bi[nt][j] = row;
                            }
                        }
                    }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cta(&empty[st]);
    }
    if (!ok && lane == 0) s_abort = 1;  // the producer stops issuing
    // best of each batch column over the warp's rows (lanes with the same t), then the two halves
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv[nt][j], o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi[nt][j], o);
                if (lm_better(ov, oi, bv[nt][j], bi[nt][j])) {
                    bv[nt][j] = ov;
                    bi[nt][j] = oi;
                }
            }
    if (active && lane < 4)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int b = 16 * nh + 8 * nt + 2 * t + j;
                if (b < M) {
                    fin_v[mt][b] = bv[nt][j];
                    fin_i[mt][b] = bi[nt][j];
                }
            }
    uint32_t any_fail;
    asm volatile("{ .reg .pred a, b; setp.eq.u32 a, %1, 0; bar.red.or.pred b, %2, %3, a; selp.u32 %0, 1, 0, b; }"
                 : "=r"(any_fail)
                 : "r"((uint32_t)ok), "n"(LM_BAR), "n"(LM_WARPS * 32)
                 : "memory");
    if (threadIdx.x < M) {
        const int b = threadIdx.x;
        float v = fin_v[0][b];
        int ix = fin_i[0][b];
        if (lm_better(fin_v[1][b], fin_i[1][b], v, ix)) {
            v = fin_v[1][b];
            ix = fin_i[1][b];
        }
        if (any_fail) {  // (+inf, -1) wins the reduction: the row's token is -1
            v = INFINITY;
            ix = -1;
        }
        part_val[(size_t)b * gridDim.x + blockIdx.x] = v;
        part_idx[(size_t)b * gridDim.x + blockIdx.x] = ix;
    }
}

cudaError_t launch_lmhead_mma(const Launch &lc, const bf16 *X, int M, int C, const bf16 *E, int V, float *logits,
                              float *part_val, int32_t *part_idx, int n_parts, uint32_t *err) {
    if (C != 1024 || M < 1 || M > MMA_MPAD) return cudaErrorInvalidValue;
    constexpr int KV = 4;
    const size_t smem = 128 + (size_t)(LM_STAGES * LM_ROWS + MMA_MPAD) * (KV * 256 * 2 + 16);
    cudaError_t e = cudaFuncSetAttribute(k_lmhead_mma<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch(lc, k_lmhead_mma<KV>, dim3(n_parts), dim3((LM_WARPS + 1) * 32), smem, X, M, E, V, logits, part_val,
                  part_idx, err);
}

int lmhead_mma_parts(int num_sms) { return num_sms; }

template <int EPI, int KS, int MP>
cudaError_t run_mma_p(const Launch &lc, const bf16 *X, int M, int K, const bf16 *W, int N, void *out, uint32_t *err) {
    const int Kc = K / KS;
    const size_t smem = 128 + (size_t)(MMA_ROWS + MP) * (Kc * 2 + 16) + MMA_WARPS * MMA_ROWS * MP * 4;
    cudaError_t e = cudaFuncSetAttribute(k_gemv_mma<EPI, KS, MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch(lc, k_gemv_mma<EPI, KS, MP>, dim3(N / MMA_ROWS, KS), dim3(MMA_WARPS * 32), smem, X, M, K, W, N,
                  out, err);
}

// up to 16 rows: half the shared memory (more CTAs an SM) and half the B fragments
template <int EPI, int KS>
cudaError_t run_mma(const Launch &lc, const bf16 *X, int M, int K, const bf16 *W, int N, void *out, uint32_t *err) {
    return M <= 16 ? run_mma_p<EPI, KS, 16>(lc, X, M, K, W, N, out, err)
                   : run_mma_p<EPI, KS, 32>(lc, X, M, K, W, N, out, err);
}

bool gemv_mma_supported(int M, int K, int N) {
    return M >= 1 && M <= MMA_MPAD && N % MMA_ROWS == 0 && K % 256 == 0 && K <= 3072;
}

cudaError_t launch_gemv_mma(const Launch &lc, const bf16 *X, int M, int K, const bf16 *W, int N, int epi,
                            void *out, uint32_t *err) {
    if (!gemv_mma_supported(M, K, N)) return cudaErrorInvalidValue;
    // Residual adds split K over 2 or 4 CTAs (fp32 atomics; order unspecified): o_proj and down
    // have only N/16 = 64 weight-row tiles, and K above 2048 with 32 rows would not fit shared
    // memory in one slice.  The other epilogues need whole sums and keep K in one slice.
    if (epi == EPI_RESID_ADD) {
        if (K >= 2048 && (K / 4) % 256 == 0) return run_mma<EPI_RESID_ADD, 4>(lc, X, M, K, W, N, out, err);
        if ((K / 2) % 256 == 0) return run_mma<EPI_RESID_ADD, 2>(lc, X, M, K, W, N, out, err);
        if (K <= 2048) return run_mma<EPI_RESID_ADD, 1>(lc, X, M, K, W, N, out, err);
        return cudaErrorInvalidValue;
    }
    if (K > 2048) return cudaErrorInvalidValue;
    if (epi == EPI_F32) return run_mma<EPI_F32, 1>(lc, X, M, K, W, N, out, err);
    return run_mma<EPI_SWIGLU, 1>(lc, X, M, K, W, N, out, err);
}

// WdT[j][n] = Wd[n][j]: the down projection stored transposed for the split-K MLP kernel.
__global__ void k_transpose_bf16(const bf16 *__restrict__ src, bf16 *__restrict__ dst, int rows, int cols) {
    __shared__ bf16 tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = src[(size_t)r * cols + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols) dst[(size_t)c * rows + r] = tile[threadIdx.x][i];
    }
}

cudaError_t launch_transpose_bf16(const Launch &lc, const bf16 *src, bf16 *dst, int rows, int cols) {
    return launch(lc, k_transpose_bf16, dim3((cols + 31) / 32, (rows + 31) / 32), dim3(32, 8), 0, src, dst, rows,
                  cols);
}

}  // namespace q3
