// Causal GQA prefill attention on the 5th-generation tensor cores (flash-style, online softmax).
//
//   o_h[i] = sum_{j<=i} softmax_j(q_h[i] . k_g[j] / sqrt(128)) v_g[j],  g = h / (Hq/Hkv)
// ("手写Qwen3-0.6B推理", Attention; "第 3 章", 3.3: lower-triangular mask, K/V shared by Hq/Hkv
// query heads; "从零开始写Qwen3", Attn: scale 1/sqrt(D)).  Same contract as the mma.sync kernel
// in attn_prefill.cu: q bf16 [N, Hq, 128] packed by cu_seqlens, K/V read from the layer's cache
// [slot][Hkv][max_ctx][128], out bf16 [N, Hq*128].
//
// CTA = 128 queries x the 2 query heads of one KV head (the GQA pair shares every K/V tile);
// 18 warps:
//   warp 16 (1 thread): TMA -- both Q tiles once, then each K tile (two-stage ring) and V tile
//                      of 128 keys (128-byte swizzle, two 64-column halves per tile);
//   warp 17 (1 thread): MMA -- S_h = Q_h K^T (M=128, N=128, K=128) into TMEM and, as each head's
//                      P is ready, O_h += P_h V (V read MN-major), issued per head in the order
//                      P_0 V(j), S_0(j+1), P_1 V(j), S_1(j+1): the scores of one head's next tile
//                      are computed while the other head's softmax runs;
//   warps 0-7 / 8-15:  eight softmax warps per head -- warps w and w+4 of a head read the same
//                      32 TMEM lanes (query rows) and split the 128 columns (keys) in halves:
//                      each thread takes 64 scores of its row (tcgen05.ld), the two halves
//                      exchange their row maxima through shared memory (a named barrier per
//                      tile and pair of warps), apply the causal mask and the online softmax in fp32,
//                      write P (bf16) into tensor memory over the first 64 columns of S_h
//                      (the P V MMA reads its A operand from there, not from shared memory)
//                      and rescale their half of the row of the TMEM accumulator O_h when the
//                      reference maximum moves; the two partial row sums meet at the end.
// The two warpgroups work on their heads at the same time while the tensor core alternates
// between them, so the exponentials of one head overlap the MMAs of the other.
// Every mbarrier wait is bounded; on timeout the CTA flags ERR_TIMEOUT and skips to the end.

#include <cuda.h>

#include <mutex>

#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128, BQ = 128, BK = 128, THREADS = 576;
constexpr int TMA_WARP = 16, MMA_WARP = 17;  // warps 0-15 run the softmax
constexpr int TILE_BYTES = 128 * D * 2;  // a [128][128] bf16 tile as two 64-column halves
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr uint32_t TMEM_COLS = 512;  // S0: 0-127, S1: 128-255, O0: 256-383, O1: 384-511

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, A K-major, B K-major
// (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t idesc(int m, int n, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
// O += A B with A (M x K, bf16, two elements per 32-bit column, row = TMEM lane) in tensor memory.
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 columns of this thread's TMEM lane (no wait: the caller issues tcgen05.wait::st).
__device__ __forceinline__ void st16_nowait(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void st32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
        "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
        "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
        "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

struct Bars {
    uint64_t q_full, kfull[2], kempty[2], vfull, vempty;
    uint64_t s_full[2], p_full[2], o_full[2];
    uint32_t tmem;
    float xmax[2][2][2][BQ];  // [tile parity][head][column half][row]: partial row maxima
    float xsum[2][2][BQ];     // [head][column half][row]: partial row sums at the end
    int xfail[2][2][2][4];    // [tile parity][head][column half][row quarter]: this warp's wait gave up
};
// 1024 bytes of alignment slack, Q0, Q1, the K ring (2), V, the barriers
constexpr int SMEM_BYTES = 1024 + TILE_BYTES * 5 + (int)sizeof(Bars);

__global__ void __launch_bounds__(THREADS, 1) k_attn_prefill_tc(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, const int32_t *__restrict__ cu, const int32_t *__restrict__ slots,
    const int32_t *__restrict__ row_pos, bf16 *__restrict__ out, int Hq, int Hkv, int max_ctx, float scale_log2,
    uint32_t *err, KvMap kv) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = smem;                    // [2] tiles
    uint8_t *k_s = q_s + 2 * TILE_BYTES;    // [2] tiles: K ring
    uint8_t *v_s = k_s + 2 * TILE_BYTES;
    Bars *bars = reinterpret_cast<Bars *>(v_s + TILE_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = gridDim.x - 1 - blockIdx.x, g = blockIdx.y, b = blockIdx.z;  // longest tiles first
    pdl_wait();
    const int start = cu[b], len = cu[b + 1] - start;
    const int q0 = qt * BQ;
    if (q0 >= len) return;  // uniform: no barrier or TMEM touched yet
    const int h0 = g * 2;    // the pair of query heads of KV head g (Hq == 2 Hkv)
    const int slot = slots[b];  // cache rows of key tile j: kv_row(kv, slot, Hkv, g, max_ctx, j * BK) + 0..127
    // The sequence's rows are positions off .. off+len-1 of its slot (off > 0 when the call
    // continues a slot that already holds off tokens): query off+i sees keys 0 .. off+i, the
    // bottom-right alignment of the causal mask.
    const int off = row_pos[start];
    const int n_tiles = (off + min(len, q0 + BQ) + BK - 1) / BK;
    // tiles j >= first_masked hold a key above this CTA's first query and need the mask
    const int first_masked = (off + q0 + 1) / BK;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int st = 0; st < 2; ++st) {
            mbar_init(&bars->kfull[st], 1);
            mbar_init(&bars->kempty[st], 1);
        }
        mbar_init(&bars->vfull, 1);
        mbar_init(&bars->vempty, 1);
        for (int hh = 0; hh < 2; ++hh) {
            mbar_init(&bars->s_full[hh], 1);
            mbar_init(&bars->p_full[hh], 8 * 32);
            mbar_init(&bars->o_full[hh], 1);
        }
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&bars->tmem)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = bars->tmem;

    bool ok = true;
    if (warp == TMA_WARP) {
        if (lane == 0) {
            mbar_expect_tx(&bars->q_full, 2 * TILE_BYTES);
            for (int hh = 0; hh < 2; ++hh) {
                tma2d(q_s + hh * TILE_BYTES, &tmQ, (h0 + hh) * D, start + q0, &bars->q_full);
                tma2d(q_s + hh * TILE_BYTES + HALF_BYTES, &tmQ, (h0 + hh) * D + 64, start + q0, &bars->q_full);
            }
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int st = j & 1;  // K tile j into ring stage j % 2, once tile j - 2 has been used
                if (j >= 2 && !mbar_wait_bounded(&bars->kempty[st], ((j - 2) >> 1) & 1, err)) { ok = false; break; }
                // a paged cache keeps whole 128-key tiles inside one block (block size % 128 == 0)
                const int row_j = (int)kv_row(kv, slot, Hkv, g, max_ctx, j * BK);
                mbar_expect_tx(&bars->kfull[st], TILE_BYTES);
                tma2d(k_s + st * TILE_BYTES, &tmK, 0, row_j, &bars->kfull[st]);
                tma2d(k_s + st * TILE_BYTES + HALF_BYTES, &tmK, 64, row_j, &bars->kfull[st]);
                if (j > 0 && !mbar_wait_bounded(&bars->vempty, (j - 1) & 1, err)) { ok = false; break; }
                mbar_expect_tx(&bars->vfull, TILE_BYTES);
                tma2d(v_s, &tmV, 0, row_j, &bars->vfull);
                tma2d(v_s + HALF_BYTES, &tmV, 64, row_j, &bars->vfull);
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            constexpr uint32_t id_s = idesc(BQ, BK, 0), id_o = idesc(BQ, D, 1);
            ok = mbar_wait_bounded(&bars->q_full, 0, err);
            // Descriptors built once; a byte offset o moves the start-address field by o >> 4
            // (shared-memory addresses stay below 2^18, so the 14-bit field never carries).
            const uint64_t dq[2] = {sdesc(smem_addr(q_s), 16, 1024), sdesc(smem_addr(q_s + TILE_BYTES), 16, 1024)};
            const uint64_t dk[2] = {sdesc(smem_addr(k_s), 16, 1024), sdesc(smem_addr(k_s + TILE_BYTES), 16, 1024)};
            const uint64_t dv = sdesc(smem_addr(v_s), HALF_BYTES, 1024);
            auto issue_s = [&](int hh, int j) {  // S_hh = Q_hh K(j)^T
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4);
                    mma(tmem + hh * 128, dq[hh] + off, dk[j & 1] + off, id_s, kk != 0);
                }
                commit(&bars->s_full[hh]);
                if (hh == 1) commit(&bars->kempty[j & 1]);  // both heads have read K(j)
            };
            if (ok && mbar_wait_bounded(&bars->kfull[0], 0, err)) {
                fence_after();
                issue_s(0, 0);
                issue_s(1, 0);
            } else {
                ok = false;
            }
            for (int j = 0; j < n_tiles && ok; ++j) {
                if (!mbar_wait_bounded(&bars->vfull, j & 1, err)) { ok = false; break; }
                for (int hh = 0; hh < 2 && ok; ++hh) {
                    // P_hh(j) is written (and S_hh(j) read): O_hh += P_hh V(j), then S_hh(j+1)
                    if (!mbar_wait_bounded(&bars->p_full[hh], j & 1, err)) { ok = false; break; }
                    fence_after();
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // P from TMEM (16 keys = 8 columns, over S_hh); V: MN-major, 16 keys = 2048 bytes
                        mma_ts(tmem + 256 + hh * 128, tmem + hh * 128 + kk * 8, dv + (uint64_t)(kk * 2048 >> 4), id_o,
                               (j | kk) != 0);
                    }
                    commit(&bars->o_full[hh]);
                    if (hh == 1) commit(&bars->vempty);  // both heads have read V(j)
                    if (j + 1 < n_tiles) {
                        if (hh == 0 && !mbar_wait_bounded(&bars->kfull[(j + 1) & 1], ((j + 1) >> 1) & 1, err)) {
                            ok = false;
                            break;
                        }
                        fence_after();
                        issue_s(hh, j + 1);
                    }
                }
            }
        }
    } else {
        // softmax: head hh = warp / 8; warps w and w + 4 of the head share query rows
        // r = 32 (w % 4) + lane and take the column halves ch = (w % 8) / 4
        const int hh = warp >> 3, wl = warp & 7, ch = wl >> 2;
        const int r = (wl & 3) * 32 + lane;
        const int qi = q0 + r;        // row within this call's part of the sequence
        const int qa = off + qi;      // its position (keys 0..qa are visible)
        const int kend = off + len;   // keys at or beyond kend do not exist yet
        const uint32_t lane_base = (uint32_t)((wl & 3) * 32) << 16;
        const uint32_t t_s = tmem + hh * 128 + ch * 64 + lane_base, t_o = tmem + 256 + hh * 128 + ch * 64 + lane_base;
        // the two warps that share these query rows meet at their own named barrier
        auto head_sync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(1 + hh * 4 + (wl & 3)), "r"(2 * 32) : "memory"); };
        float m_run = -INFINITY, l_run = 0.0f;
        bool gave_up = false;  // warp-uniform
        // P (bf16, two keys per column) overwrites the first 64 columns of S_hh: keys
        // ch*64 + c*32 .. +31 of this row go to columns ch*32 + c*16 .. +15 of its lane.  Both
        // halves of the row hold their scores in registers past the pair's barrier, so no
        // score is overwritten before it is read.
        const uint32_t t_p = tmem + hh * 128 + ch * 32 + lane_base;
        for (int j = 0; j < n_tiles; ++j) {
            // A wait that gives up is posted with the row maxima and acted on after the pair's
            // barrier: both warps of the pair see both flags of this tile and leave the loop
            // together.  The flags alternate with the tile parity, so a partner cannot post the
            // next tile's flag before this warp has read this one.
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars->s_full[hh], j & 1, err))) gave_up = true;
            fence_after();
            const int k0 = j * BK + ch * 64;  // first key of this thread's half
            // Only tiles reaching above the CTA's first query mask: every key of an earlier
            // tile is below it, hence visible and inside the sequence.
            const bool diag = j >= first_masked;
            float v[2][32];
            ld32(t_s, v[0]);
            ld32(t_s + 32, v[1]);
            // pass 1: maximum of the visible scores of this half (eight partial maxima)
            float mxp[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mxp[i] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (diag) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int kj = k0 + c * 32 + i;
                        if (kj <= qa && kj < kend) mxp[i & 7] = fmaxf(mxp[i & 7], v[c][i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) mxp[i & 7] = fmaxf(mxp[i & 7], v[c][i]);
                }
            }
            const float mh = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                   fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
            bars->xmax[j & 1][hh][ch][r] = mh;
            if (lane == 0) bars->xfail[j & 1][hh][ch][wl & 3] = gave_up;
            head_sync();
            const float mx = fmaxf(mh, bars->xmax[j & 1][hh][ch ^ 1][r]);
            if (gave_up || bars->xfail[j & 1][hh][ch ^ 1][wl & 3]) {
                ok = false;
                break;
            }
            // The reference maximum moves only when the tile's maximum exceeds it by more than
            // 2^8: softmax does not depend on the reference, P stays below 256 (exact enough in
            // bf16, far from overflow) and the rescale of O through TMEM becomes rare.  Both
            // halves of a row see the same maximum, so they take the same decision.
            const float m_tile = mx * scale_log2;
            float m_new = m_run, corr = 1.0f;
            if (m_run == -INFINITY || m_tile > m_run + 8.0f) {
                m_new = m_tile;
                corr = m_run == -INFINITY ? 0.0f : exp2f(m_run - m_tile);
            }
            // pass 2: probabilities, partial row sum, P (bf16) into tensor memory.
            // The tensor core finished the previous P V (it precedes this tile's S in issue order).
            float sp[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) sp[i] = 0.0f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t pk[16];
                if (diag) {
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const int kj = k0 + c * 32 + i;
                        const float p0 = (kj <= qa && kj < kend) ? exp2f(fmaf(v[c][i], scale_log2, -m_new)) : 0.0f;
                        const float p1 =
                            (kj + 1 <= qa && kj + 1 < kend) ? exp2f(fmaf(v[c][i + 1], scale_log2, -m_new)) : 0.0f;
                        sp[(i >> 1) & 7] += p0 + p1;
                        pk[i / 2] = pack_bf16x2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float p0 = exp2f(fmaf(v[c][i], scale_log2, -m_new));
                        const float p1 = exp2f(fmaf(v[c][i + 1], scale_log2, -m_new));
                        sp[(i >> 1) & 7] += p0 + p1;
                        pk[i / 2] = pack_bf16x2(p0, p1);
                    }
                }
                st16_nowait(t_p + c * 16, pk);
            }
            const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
            l_run = l_run * corr + sum;
            m_run = m_new;
            // O_h holds tiles < j (implied by s_full; waited so that o_full's phases stay in step)
            bool o_ok = true;
            if (j > 0 && !__all_sync(0xffffffffu, mbar_wait_bounded(&bars->o_full[hh], (j - 1) & 1, err))) {
                o_ok = false;
                gave_up = true;  // the loop ends at the next barrier
            }
            if (o_ok && j > 0 && __any_sync(0xffffffffu, corr != 1.0f)) {  // rescale this half-row of O_h
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    float o[32];
                    ld32(t_o + c * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= corr;
                    st32(t_o + c * 32, o);
                }
            }
            // P is in tensor memory: complete the stores, then hand over
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            fence_before();
            arrive(&bars->p_full[hh]);
        }
        if (gave_up) ok = false;
        // the two halves' row sums; the output row is then written in two halves
        bars->xsum[hh][ch][r] = l_run;
        head_sync();
        const float l_tot = l_run + bars->xsum[hh][ch ^ 1][r];
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->o_full[hh], (n_tiles - 1) & 1, err));
        if (ok) {
            fence_after();
            const float inv = 1.0f / l_tot;
            uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)(start + qi) * Hq + h0 + hh) * D + ch * 64);
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                float v[32];
                ld32(t_o + c * 32, v);
                if (qi < len) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[c * 4 + i] = make_uint4(pack_bf16x2(v[8 * i] * inv, v[8 * i + 1] * inv),
                                                    pack_bf16x2(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                                    pack_bf16x2(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                                    pack_bf16x2(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
                }
            }
        }
    }
    pdl_trigger();
    fence_before();
    __syncthreads();
    if (warp == MMA_WARP) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode() {
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

// [rows, cols] bf16 row-major, boxes of 64 columns x 128 rows, 128-byte swizzle
bool map2d(CUtensorMap *m, const bf16 *base, uint64_t rows, uint64_t cols) {
    EncodeTiledFn fn = encode();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16 *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool kv_tile_map(CUtensorMap *m, const bf16 *base, uint64_t rows) {
    EncodeTiledFn fn = encode();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16 *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool attn_prefill_tc_supported(int Hq, int Hkv) { return Hq == 2 * Hkv && encode() != nullptr; }

cudaError_t launch_attn_prefill_tc(const Launch &lc, const bf16 *q, int N, const bf16 *k_layer,
                                   const bf16 *v_layer, const int32_t *cu_seqlens, const int32_t *slots,
                                   const int32_t *row_pos, int B, int max_len, int max_seqs, bf16 *out, int Hq,
                                   int Hkv, int max_ctx, uint32_t *err, const KvMap &kv, size_t kv_rows_paged) {
    CUtensorMap mq, mk, mv;
    if (kv.table && (kv.bs % BK || kv_rows_paged == 0)) return cudaErrorInvalidValue;
    const uint64_t kv_rows = kv.table ? (uint64_t)kv_rows_paged : (uint64_t)max_seqs * Hkv * max_ctx;
    if (!map2d(&mq, q, (uint64_t)N, (uint64_t)Hq * D) || !map2d(&mk, k_layer, kv_rows, D) ||
        !map2d(&mv, v_layer, kv_rows, D))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    return launch(lc, k_attn_prefill_tc, dim3((max_len + BQ - 1) / BQ, Hkv, B), dim3(THREADS), SMEM_BYTES, mq, mk, mv,
                  cu_seqlens, slots, row_pos, out, Hq, Hkv, max_ctx, scale_log2, err, kv);
}

}  // namespace q3
