// Prefill projection GEMM on the 5th-generation tensor cores: out[M,N] = A[M,K] . W[N,K]^T,
// bf16 operands, fp32 accumulation in tensor memory.  Same contract and epilogues as the
// mma.sync GEMM (QKV, o, gate_up + SwiGLU, down: "手写Qwen3-0.6B推理", Attention and MLP;
// "第 3 章", 3.3/3.4 merged projections).
//
// Tiles of 128 x 256 outputs, 4 roles:
//   warp 0, one thread : TMA producer -- A and W tiles (64 K-columns, 128-byte swizzle) into a
//                        4-stage shared-memory ring, completion counted on mbarriers;
//   warp 1, one thread : MMA issuer -- tcgen05.mma (M=128, N=256, K=16) per stage, the stage
//                        released back to the producer by tcgen05.commit;
//   warps 2-9          : epilogue -- tcgen05.ld of TMEM lanes 32(w%4)..+31 (one output row per
//                        thread), then the fp32 / residual-add / SwiGLU / QKV store.  The
//                        residual add moves h through shared memory by TMA: 32 rows x 32
//                        columns of fp32 per warp in, the sums out, so that the rows (4 KB
//                        apart) travel as tiles rather than one 16-byte piece of 32 rows per
//                        instruction.
// Rows of A beyond M are zero-filled by TMA and dropped on store (ragged token counts).
// Every mbarrier wait is bounded: on timeout the CTA flags ERR_TIMEOUT, drains, frees its
// tensor memory and returns.

#include <cuda.h>

#include <mutex>

#include "kernels.h"

namespace q3 {

namespace {

constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64, TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;                  // 16 KB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;                  // 32 KB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;        // 48 KB
constexpr int TC_SMEM = TC_STAGES * TC_STAGE_BYTES + 256 + 1024;  // ring + barriers + alignment
// The residual-add epilogue's tiles of h: one per epilogue warp, 32 rows x 32 fp32 columns
// (128-byte rows, 128-byte swizzle), 1024-aligned after the barriers.
constexpr int TC_H_BOX = 32;
constexpr int TC_H_BYTES = TC_H_BOX * TC_H_BOX * 4;  // 4 KB
constexpr int TC_H_OFF = TC_STAGES * TC_STAGE_BYTES + 1024;
constexpr int TC_SMEM_RESID = TC_H_OFF + 8 * TC_H_BYTES + 1024;
static_assert(TC_SMEM_RESID <= 227 * 1024, "residual epilogue tiles exceed shared memory");

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with the 128-byte
// swizzle: rows of 128 bytes (64 elements), 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)(16 >> 4) << 16;            // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                    // descriptor version
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}

// Shared -> global tile store through the tensor map (rows past the tensor's end are not written).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_addr(src)), "r"(x), "r"(y)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The stores issued by this thread have read their shared memory.
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The stores issued by this thread are complete.
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Persistent form: each CTA walks tiles blockIdx.x, blockIdx.x + gridDim.x, ... (row-block
// major, so CTAs running together share A rows).  Two TMEM accumulators of 256 columns: the
// MMA thread fills one while the epilogue warps drain the other.
//   warp 0 (1 thread) TMA producer; warp 1 (1 thread) MMA issuer and TMEM owner;
//   warps 2-9 epilogue, warp w reading TMEM lanes 32*(w%4) .. 32*(w%4)+31 and the columns
//   128*((w-2)/4) .. +127 of the tile (for QKV: one head of the tile's two).
constexpr int TCP_THREADS = 320, TCP_EPI_WARPS = 8;
constexpr uint32_t TCP_TMEM_COLS = 512;

struct EpiArgs {
    void *out;
    // EPI_QKV: per-head RMSNorm + rotate-half RoPE of q and k, V as projected; q to q_out
    // [rows, Hq, 128], k and v into the layer's cache at (row_slot, row_pos).
    const int32_t *row_slot, *row_pos;
    const float *q_gain, *k_gain;
    // (cos, sin) of frequencies 2k and 2k+1 at position pos: rope_t[k * max_ctx + pos], k < 32
    const float4 *rope_t;
    bf16 *q_out, *k_layer, *v_layer;
    int Hq, Hkv, max_ctx;
    KvMap kv;  // where the cache row of (slot, head, pos) lives
    float eps;
    // RMSNorm folded into the GEMMs around it (RowNorm in kernels.h): scale rows by
    // rsqrt(sum(ss_in[row][*]) / norm_c + eps) (QKV, SwiGLU), or, with xn_out (residual add),
    // also write bf16(h * gamma_out) and the sum of squares of each 128-column half of h.
    const float *ss_in;
    float *ss_out;
    bf16 *xn_out;
    const float *gamma_out;
    int norm_c;
};

// rsqrt(mean of squares + eps) of a row from its per-128-column partial sums (fixed order).
__device__ __forceinline__ float row_scale(const EpiArgs &ea, int row) {
    const int np = ea.norm_c / 128;
    const float *p = ea.ss_in + (size_t)row * np;
    float s = 0.0f;
    for (int i = 0; i < np; ++i) s += p[i];
    return rsqrtf(s / (float)ea.norm_c + ea.eps);
}

// SwiGLU of row-scaled gate/up pairs: silu(rs * g) * (rs * u), bf16.
__device__ __forceinline__ void store_swiglu_scaled(const uint32_t *v, float rs, int row, int col, int N, void *out) {
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float a0 = silu(rs * __uint_as_float(v[4 * j])) * (rs * __uint_as_float(v[4 * j + 1]));
        const float a1 = silu(rs * __uint_as_float(v[4 * j + 2])) * (rs * __uint_as_float(v[4 * j + 3]));
        o[j] = pack_bf16x2(a0, a1);
    }
    uint4 *dst = reinterpret_cast<uint4 *>((bf16 *)out + (size_t)row * (N / 2) + col / 2);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void store_chunk(int EPI_, const uint32_t *v, int row, int col, int N, void *out) {
    if (EPI_ == EPI_F32) {
        float4 *dst = reinterpret_cast<float4 *>((float *)out + (size_t)row * N + col);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                                 __uint_as_float(v[4 * j + 3]));
    } else {  // SwiGLU: columns (2j, 2j+1) are (gate_j, up_j)
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float a0 = silu(__uint_as_float(v[4 * j])) * __uint_as_float(v[4 * j + 1]);
            const float a1 = silu(__uint_as_float(v[4 * j + 2])) * __uint_as_float(v[4 * j + 3]);
            o[j] = pack_bf16x2(a0, a1);
        }
        uint4 *dst = reinterpret_cast<uint4 *>((bf16 *)out + (size_t)row * (N / 2) + col / 2);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

template <int EPI>
__global__ void __launch_bounds__(TCP_THREADS, 1) k_gemm_tcp(const __grid_constant__ CUtensorMap tmA,
                                                             const __grid_constant__ CUtensorMap tmB,
                                                             const __grid_constant__ CUtensorMap tmH, int M, int N,
                                                             int K, EpiArgs ea, uint32_t *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + TC_STAGES * TC_STAGE_BYTES);
    uint64_t *empty = full + TC_STAGES;
    uint64_t *tm_full = empty + TC_STAGES;  // [2]
    uint64_t *tm_empty = tm_full + 2;       // [2]
    uint64_t *hbar = tm_empty + 2;          // [8] residual tiles of the epilogue warps
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(hbar + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = K / TC_BK;
    const int tiles_n = N / TC_BN, tiles = ((M + TC_BM - 1) / TC_BM) * tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tm_full[a], 1);
            mbar_init(&tm_empty[a], TCP_EPI_WARPS);  // one arrival per epilogue warp
        }
        for (int w = 0; w < TCP_EPI_WARPS; ++w) mbar_init(&hbar[w], 1);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(TCP_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // A is the previous kernel's output

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;  // k-blocks issued so far (ring position)
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int m0 = (t / tiles_n) * TC_BM, n0 = (t % tiles_n) * TC_BN;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % TC_STAGES;
                    if (it >= TC_STAGES && !mbar_wait_bounded(&empty[s], ((it / TC_STAGES) & 1) ^ 1, err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + s * TC_STAGE_BYTES;
                    mbar_expect_tx(&full[s], TC_STAGE_BYTES);
                    tma_load_2d(sa, &tmA, kb * TC_BK, m0, &full[s]);
                    tma_load_2d(sa + TC_A_BYTES, &tmB, kb * TC_BK, n0, &full[s]);
                }
            }
            if (!ok)  // let the copies in flight land before the CTA can leave
                for (int j = (it > TC_STAGES ? it - TC_STAGES : 0); j < it; ++j)
                    mbar_wait_bounded(&full[j % TC_STAGES], (j / TC_STAGES) & 1, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(TC_BM, TC_BN);
            int it = 0, local = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++local) {
                const int a = local & 1;
                if (local >= 2 && !mbar_wait_bounded(&tm_empty[a], ((local >> 1) & 1) ^ 1, err)) break;
                tc_fence_after();
                const uint32_t acc = tmem + a * TC_BN;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % TC_STAGES;
                    if (!mbar_wait_bounded(&full[s], (it / TC_STAGES) & 1, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + s * TC_STAGE_BYTES), sb = sa + TC_A_BYTES;
#pragma unroll
                    for (int k = 0; k < TC_BK / 16; ++k)
                        tc_mma(acc, sdesc_k_sw128(sa + k * 32), sdesc_k_sw128(sb + k * 32), idesc, (kb | k) != 0);
                    tc_commit(&empty[s]);
                }
                if (ok) tc_commit(&tm_full[a]);
            }
        }
    } else {
        // epilogue warps 2..9
        const int q = warp & 3;         // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;  // 128-column half of the tile
        const int ew = warp - 2;
        uint8_t *hbuf = smem + TC_H_OFF + ew * TC_H_BYTES;  // this warp's residual tile
        uint32_t hph = 0;                                   // phase of hbar[ew]
        bool failed = false;
        int local = 0;
        for (int t = blockIdx.x; t < tiles && !failed; t += gridDim.x, ++local) {
            const int a = local & 1;
            const int m0 = (t / tiles_n) * TC_BM, n0 = (t % tiles_n) * TC_BN;
            const int row = m0 + q * 32 + lane;
            // residual add: the warp's 32 rows (none of them past M for `live`), 32 columns at a
            // time; the first tile of h is requested before the accumulator is ready
            const bool rows_live = m0 + q * 32 < M;
            const bool live = EPI == EPI_RESID_ADD && rows_live;
            const int hy = m0 + q * 32;
            if (live && lane == 0) {
                mbar_expect_tx(&hbar[ew], TC_H_BYTES);
                tma_load_2d(hbuf, &tmH, n0 + half * 128, hy, &hbar[ew]);
            }
            // what a row's epilogue needs besides the accumulator, read while the MMAs run: the
            // folded input norm's row scale, and for QKV the row's cache slot and position
            float rs = 1.0f;
            int slot = 0, pos = 0;
            if ((EPI == EPI_SWIGLU || EPI == EPI_QKV) && ea.ss_in && row < M) rs = row_scale(ea, row);
            if (EPI == EPI_QKV && row < M) {
                slot = ea.row_slot[row];
                pos = ea.row_pos[row];
            }
            const bool ready = __all_sync(0xffffffffu, mbar_wait_bounded(&tm_full[a], (local >> 1) & 1, err));
            if (!ready) {
                if (live) mbar_wait_bounded(&hbar[ew], hph, nullptr);  // let the copy land
                break;
            }
            tc_fence_after();
            const uint32_t t_row = tmem + a * TC_BN + ((uint32_t)(q * 32) << 16);
            if (EPI == EPI_RESID_ADD) {
                // The thread's row sits at hbuf + 128 lane, its 16-byte piece j at piece
                // j ^ (lane % 8) of the row (the 128-byte swizzle): 8 lanes reading piece j of
                // 8 rows touch 8 different bank groups.
                float4 *hr = reinterpret_cast<float4 *>(hbuf + lane * 128);
                float ss = 0.0f;
#pragma unroll 1
                for (int c = half * 4; c < half * 4 + 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(t_row + c * 32, v);
                    if (!live) continue;
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&hbar[ew], hph, err))) {
                        mbar_wait_bounded(&hbar[ew], hph, nullptr);  // let the copy land
                        failed = true;
                        break;
                    }
                    hph ^= 1;
                    const int col = n0 + c * 32;
                    const float4 *g4 = reinterpret_cast<const float4 *>(ea.gamma_out + col);
                    uint32_t o[16];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int u = j ^ (lane & 7);
                        float4 r = hr[u];
                        r.x += __uint_as_float(v[4 * j]);
                        r.y += __uint_as_float(v[4 * j + 1]);
                        r.z += __uint_as_float(v[4 * j + 2]);
                        r.w += __uint_as_float(v[4 * j + 3]);
                        hr[u] = r;
                        if (ea.xn_out) {
                            ss += r.x * r.x + r.y * r.y + r.z * r.z + r.w * r.w;
                            const float4 g = g4[j];
                            o[2 * j] = pack_bf16x2(r.x * g.x, r.y * g.y);
                            o[2 * j + 1] = pack_bf16x2(r.z * g.z, r.w * g.w);
                        }
                    }
                    if (ea.xn_out && row < M) {
                        uint4 *xd = reinterpret_cast<uint4 *>(ea.xn_out + (size_t)row * N + col);
#pragma unroll
                        for (int j = 0; j < 4; ++j) xd[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
                    }
                    // the sums go out as a tile; the buffer then takes the next 32 columns
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmH, hbuf, col, hy);
                        tma_store_wait_read();
                        if (c + 1 < half * 4 + 4) {
                            mbar_expect_tx(&hbar[ew], TC_H_BYTES);
                            tma_load_2d(hbuf, &tmH, col + 32, hy, &hbar[ew]);
                        }
                    }
                    __syncwarp();
                }
                if (failed) break;
                if (ea.xn_out && live && row < M) ea.ss_out[(size_t)row * (N / 128) + n0 / 128 + half] = ss;
            } else if (EPI == EPI_SWIGLU && ea.ss_in) {
#pragma unroll 1
                for (int c = half * 4; c < half * 4 + 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(t_row + c * 32, v);
                    if (row < M) store_swiglu_scaled(v, rs, row, n0 + c * 32, N, ea.out);
                }
            } else if (EPI != EPI_QKV) {
#pragma unroll 1
                for (int c = half * 4; c < half * 4 + 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(t_row + c * 32, v);
                    if (row < M) store_chunk(EPI, v, row, n0 + c * 32, N, ea.out);
                }
            } else {
                // two heads of 128 columns per tile: head index within [q | k | v]
                // rs: the input RMSNorm's row scale (1 when the operand came normalised)
                {
                    const int hh = half;
                    const int head = n0 / 128 + hh;
                    const uint32_t th = t_row + hh * 128;
                    const bool is_v = head >= ea.Hq + ea.Hkv;
                    float inv = rs;  // V: the row scale alone
                    if (!is_v) {  // pass 1: sum of squares over the head's 128 columns
                        float ss = 0.0f;
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            uint32_t v[32];
                            tmem_ld32(th + c * 32, v);
#pragma unroll
                            for (int j = 0; j < 32; ++j) ss += __uint_as_float(v[j]) * __uint_as_float(v[j]);
                        }
                        // head RMSNorm of the row-scaled values rs * v
                        inv = rs * rsqrtf(ss * (rs * rs) * (1.0f / 128.0f) + ea.eps);
                    }
                    const float *gain = head < ea.Hq ? ea.q_gain : ea.k_gain;
                    bf16 *dst;
                    if (head < ea.Hq)
                        dst = ea.q_out + ((size_t)row * ea.Hq + head) * 128;
                    else {
                        const int g = is_v ? head - ea.Hq - ea.Hkv : head - ea.Hq;
                        // (pos is checked against max_ctx before the store; keep the table index in range)
                        dst = (is_v ? ea.v_layer : ea.k_layer) +
                              kv_row(ea.kv, slot, ea.Hkv, g, ea.max_ctx, pos < ea.max_ctx ? pos : 0) * 128;
                    }
                    // q leaves as TMA tiles of 32 rows x 32 columns (two a pass); k and v go
                    // to their cache rows, which need not be contiguous across the warp's rows
                    const bool q_tma = head < ea.Hq && rows_live;
                    // pass 2: elements i (chunk c) and i+64 (chunk c+2) rotate together
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t lo[32], hi[32];
                        tmem_ld32(th + c * 32, lo);
                        tmem_ld32(th + (c + 2) * 32, hi);
                        const bool valid = row < M && pos < ea.max_ctx;
                        // the results as bf16 pairs, packed as soon as they are computed
                        uint32_t pl[16], ph[16];
                        if (valid) {
                            if (is_v) {
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    pl[j] = pack_bf16x2(__uint_as_float(lo[2 * j]) * inv, __uint_as_float(lo[2 * j + 1]) * inv);
                                    ph[j] = pack_bf16x2(__uint_as_float(hi[2 * j]) * inv, __uint_as_float(hi[2 * j + 1]) * inv);
                                }
                            } else {
                                // frequency-pair-major table: the 32 lanes (rows at mostly
                                // consecutive positions) read neighbouring 16-byte entries;
                                // gains and table in 16-byte loads (four columns per step)
                                const float4 *cs = ea.rope_t + (size_t)(c * 16) * ea.max_ctx + pos;
                                const float4 *gl4 = reinterpret_cast<const float4 *>(gain + c * 32);
                                const float4 *gh4 = reinterpret_cast<const float4 *>(gain + 64 + c * 32);
#pragma unroll
                                for (int qd = 0; qd < 8; ++qd) {
                                    const float4 ga = gl4[qd], gb = gh4[qd];
                                    const float4 r0 = cs[(size_t)(2 * qd) * ea.max_ctx];      // i = 4 qd, 4 qd + 1
                                    const float4 r1 = cs[(size_t)(2 * qd + 1) * ea.max_ctx];  // i = 4 qd + 2, 4 qd + 3
                                    const float gav[4] = {ga.x, ga.y, ga.z, ga.w}, gbv[4] = {gb.x, gb.y, gb.z, gb.w};
                                    const float cv[4] = {r0.x, r0.z, r1.x, r1.z}, sv[4] = {r0.y, r0.w, r1.y, r1.w};
                                    float xl[4], xh[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int j = 4 * qd + e;
                                        const float a0 = __uint_as_float(lo[j]) * inv * gav[e];
                                        const float b0 = __uint_as_float(hi[j]) * inv * gbv[e];
                                        xl[e] = a0 * cv[e] - b0 * sv[e];  // x_i cos - x_{i+64} sin
                                        xh[e] = b0 * cv[e] + a0 * sv[e];  // x_{i+64} cos + x_i sin
                                    }
                                    pl[2 * qd] = pack_bf16x2(xl[0], xl[1]);
                                    pl[2 * qd + 1] = pack_bf16x2(xl[2], xl[3]);
                                    ph[2 * qd] = pack_bf16x2(xh[0], xh[1]);
                                    ph[2 * qd + 1] = pack_bf16x2(xh[2], xh[3]);
                                }
                            }
                        }
                        if (q_tma) {
                            // the two boxes of this pass, 64-byte rows with the 64-byte swizzle:
                            // 16-byte piece u of row r sits at piece u ^ ((r / 2) % 4), so 8
                            // lanes storing piece u of 8 rows touch 8 different bank groups
                            uint8_t *bl = hbuf, *bh = hbuf + TC_H_BYTES / 2;
                            const int sw = (lane >> 1) & 3;
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                uint4 va = make_uint4(0, 0, 0, 0), vb = va;  // rows past M or max_ctx: zeros
                                if (valid) {
                                    va = make_uint4(pl[4 * u], pl[4 * u + 1], pl[4 * u + 2], pl[4 * u + 3]);
                                    vb = make_uint4(ph[4 * u], ph[4 * u + 1], ph[4 * u + 2], ph[4 * u + 3]);
                                }
                                *reinterpret_cast<uint4 *>(bl + lane * 64 + ((u ^ sw) << 4)) = va;
                                *reinterpret_cast<uint4 *>(bh + lane * 64 + ((u ^ sw) << 4)) = vb;
                            }
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&tmH, bl, head * 128 + c * 32, hy);
                                tma_store_2d(&tmH, bh, head * 128 + 64 + c * 32, hy);
                                tma_store_wait_read();  // the buffer is free for the next pass
                            }
                            __syncwarp();
                        } else if (valid) {
                            uint4 *dl = reinterpret_cast<uint4 *>(dst + c * 32), *dh = reinterpret_cast<uint4 *>(dst + 64 + c * 32);
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                dl[u] = make_uint4(pl[4 * u], pl[4 * u + 1], pl[4 * u + 2], pl[4 * u + 3]);
                                dh[u] = make_uint4(ph[4 * u], ph[4 * u + 1], ph[4 * u + 2], ph[4 * u + 3]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&tm_empty[a])) : "memory");
        }
        if ((EPI == EPI_RESID_ADD || EPI == EPI_QKV) && lane == 0) tma_store_wait_all();  // tiles are in global memory
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TCP_TMEM_COLS));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D map of a row-major bf16 matrix [rows, cols] read as boxes of 64 columns x box_rows rows.
bool make_map(CUtensorMap *map, const bf16 *base, int rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16 *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map of the fp32 residual [rows, cols] as boxes of 32 x 32 (128-byte rows, 128-byte swizzle).
bool make_map_h(CUtensorMap *map, const float *base, int rows, int cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    const cuuint32_t box[2] = {(cuuint32_t)TC_H_BOX, (cuuint32_t)TC_H_BOX};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map of q [rows, Hq * 128] bf16 as boxes of 32 columns x 32 rows (64-byte rows, 64-byte swizzle).
bool make_map_q(CUtensorMap *map, const bf16 *base, int rows, int cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)TC_H_BOX, (cuuint32_t)TC_H_BOX};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16 *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI>
cudaError_t run_tcp(const Launch &lc, const CUtensorMap &ma, const CUtensorMap &mb, int M, int N, int K,
                    const EpiArgs &ea, uint32_t *err) {
    CUtensorMap mh = {};
    if (EPI == EPI_RESID_ADD && !make_map_h(&mh, static_cast<const float *>(ea.out), M, N)) return cudaErrorInvalidValue;
    if (EPI == EPI_QKV && !make_map_q(&mh, ea.q_out, M, ea.Hq * 128)) return cudaErrorInvalidValue;
    const int smem = EPI == EPI_RESID_ADD || EPI == EPI_QKV ? TC_SMEM_RESID : TC_SMEM;
    cudaError_t e = cudaFuncSetAttribute(k_gemm_tcp<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int tiles = ((M + TC_BM - 1) / TC_BM) * (N / TC_BN);
    const int grid = tiles < lc.num_sms ? tiles : lc.num_sms;
    return launch(lc, k_gemm_tcp<EPI>, dim3(grid), dim3(TCP_THREADS), smem, ma, mb, mh, M, N, K, ea, err);
}

}  // namespace

bool gemm_tc_supported(int M, int K, int N) {
    return M >= 1 && K >= TC_BK && K % TC_BK == 0 && N >= TC_BN && N % TC_BN == 0 && encode_fn() != nullptr;
}

cudaError_t launch_gemm_tc(const Launch &lc, const bf16 *A, int M, int K, const bf16 *W, int N, int epi,
                           void *out, uint32_t *err, const RowNorm &rn) {
    if (!gemm_tc_supported(M, K, N) || epi == EPI_QKV) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(W)) & 15) return cudaErrorInvalidValue;
    // the residual travels by TMA: 16-byte aligned base (N % 256 == 0 gives the row pitch)
    if (epi == EPI_RESID_ADD && (reinterpret_cast<uintptr_t>(out) & 15)) return cudaErrorInvalidValue;
    if (rn.xn_out && (epi != EPI_RESID_ADD || !rn.ss_out || !rn.gamma_out || N % 128)) return cudaErrorInvalidValue;
    if (rn.ss_in && (epi != EPI_SWIGLU || rn.norm_c != K || K % 128)) return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, M, K, TC_BM) || !make_map(&mb, W, N, K, TC_BN)) return cudaErrorInvalidValue;
    EpiArgs ea = {};
    ea.out = out;
    ea.ss_in = rn.ss_in;
    ea.ss_out = rn.ss_out;
    ea.xn_out = rn.xn_out;
    ea.gamma_out = rn.gamma_out;
    ea.norm_c = rn.norm_c;
    ea.eps = rn.eps;
    switch (epi) {
        case EPI_F32: return run_tcp<EPI_F32>(lc, ma, mb, M, N, K, ea, err);
        case EPI_RESID_ADD: return run_tcp<EPI_RESID_ADD>(lc, ma, mb, M, N, K, ea, err);
        case EPI_SWIGLU: return run_tcp<EPI_SWIGLU>(lc, ma, mb, M, N, K, ea, err);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc_qkv(const Launch &lc, const bf16 *A, int M, int K, const bf16 *W, int N, const Rows &r,
                               const float *q_gain, const float *k_gain, const float4 *rope_t, bf16 *q_out,
                               bf16 *k_layer, bf16 *v_layer, int Hq, int Hkv, int max_ctx, float eps,
                               uint32_t *err, const float *ss_in) {
    if (!gemm_tc_supported(M, K, N) || N != (Hq + 2 * Hkv) * 128 || (ss_in && K % 128)) return cudaErrorInvalidValue;
    if (reinterpret_cast<uintptr_t>(q_out) & 15) return cudaErrorInvalidValue;  // q leaves by TMA
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, M, K, TC_BM) || !make_map(&mb, W, N, K, TC_BN)) return cudaErrorInvalidValue;
    EpiArgs ea = {};
    ea.row_slot = r.row_slot;
    ea.row_pos = r.row_pos;
    ea.q_gain = q_gain;
    ea.k_gain = k_gain;
    ea.rope_t = rope_t;
    ea.q_out = q_out;
    ea.k_layer = k_layer;
    ea.v_layer = v_layer;
    ea.Hq = Hq;
    ea.Hkv = Hkv;
    ea.max_ctx = max_ctx;
    ea.kv = r.kv;
    ea.eps = eps;
    ea.ss_in = ss_in;
    ea.norm_c = K;
    return run_tcp<EPI_QKV>(lc, ma, mb, M, N, K, ea, err);
}

}  // namespace q3
