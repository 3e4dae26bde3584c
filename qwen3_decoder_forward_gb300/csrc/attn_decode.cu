// Split-KV decode attention: one new query row per sequence against its cached keys 0..p.
//
// A decode query at absolute position p sees every cached key 0..p, its own included
// ("从零开始写Qwen3", Attn: no causal flag for a length-1 query; "古法手撕简易LLM推理器",
// 核心计算函数与Transformer层: no mask once offset > 0, the new key appended first).  The
// Hq/Hkv query heads of one KV head are served by the same CTA so each K/V row is read
// from HBM once ("手写Qwen3-0.6B推理", Attention: K/V shared by a group of query heads).
//
// Grid (split, KV head, sequence).  The scores and the weighted sum run on the tensor cores
// (mma.sync m16n8k16) in transposed form: S^T = K Q^T with the keys as the M side (16 per warp
// and chunk), the G <= 8 query heads of the KV head as the N side and the 128 dimensions as the
// reduction; then O^T += V^T P^T with the dimensions as the M side (8 tiles), the heads as N and
// the 16 keys as the reduction.  The online softmax (m, l per head) works on the score
// fragments: a maximum over the 8 lanes holding a head's 16 scores, exp2 of the scores, the
// rescale of the O^T fragments only when a maximum moves.  P^T reaches the B-operand layout
// with 8 shuffles.  The four warps' partials are merged in shared memory; each split writes
// (m, l) and the unnormalised output of its key range to a workspace and the last CTA of a
// (sequence, KV head) takes the log-sum-exp merge of the splits.  Scores are pre-scaled by
// log2(e)/sqrt(128) (folded into bf16 q) so exp2 is used throughout; P is bf16, as in the
// prefill attention.
//
// K/V chunks of 64 keys arrive by tensor-map copies (four 64 x 64 boxes, 128-byte swizzle, so
// that ldmatrix reads 8 keys of one 16-byte column without bank conflicts) into a three-stage
// ring.  Split ranges are whole chunks, so a chunk of a paged cache never crosses a block.
// The last chunk of a range may reach past its keys: those rows (finite, from the zeroed cache
// or other positions) are masked.
//
// QK-norm + RoPE + KV write in the prologue: each CTA normalises and rotates its query heads
// and the new key from the QKV projection's fp32 row (lane `sub` of each 8-lane group holds
// elements sub*16 .. sub*16+15, so the RoPE partner i+64 of element i sits in lane sub^4).
// The new K (rounded to bf16, as the cache stores it) and V are written to the cache by split 0
// and, as a one-key 16-row tile, taken by warp 0 of the split that covers the new position.
//
// Every kernel of the decode chain passes its own dependency wait before it lets the next
// kernel launch, so when this kernel starts, every kernel before the QKV projection has
// completed: the cached rows 0..pos-1, the row positions, the gains and the RoPE table are
// final, and the first stages are requested before the wait.  Only q/k/v of the new row come
// from the immediately preceding kernel.
//
// Split s of n covers keys [s*per, min((s+1)*per, p+1)) with per = ceil((p+1)/n) rounded up to
// whole chunks, from the sequence's own position on the device: the ranges stay balanced for
// every length that a recorded launch (a fixed n) serves.  The CTA that finishes last for a
// (sequence, KV head) merges all splits (a counter per pair, incremented after a memory fence
// and reset by that CTA): no second kernel and no waiting on other CTAs.

#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int STAGES = 3;
constexpr int NW = 4;                         // warps per CTA: 16 keys of each chunk each
constexpr int CHUNK = NW * 16;                // keys per ring stage
constexpr int BOX_BYTES = 64 * 64 * 2;        // [64 keys][64 dims] bf16, 128-byte swizzle
constexpr int STAGE_BYTES = 4 * BOX_BYTES;    // K dims 0-63, 64-127, then V
constexpr int NEW_HALF = 16 * 128;            // the new row's tile: 16 rows of one 64-dim half
constexpr int NEW_BYTES = 4 * NEW_HALF;       // K halves, then V halves
constexpr int MAX_G = 8;

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16(x)); }

// byte offset of 16-byte unit u of row `row` in a box whose rows are 128 bytes, 128-byte swizzle
__device__ __forceinline__ uint32_t swz(int row, int u) { return (uint32_t)(row * 128 + ((u ^ (row & 7)) << 4)); }

__device__ __forceinline__ void ldsm_x4(uint32_t *r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t *r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
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
__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}

template <int G, bool PAGED>
__global__ void __launch_bounds__(NW * 32, 2) k_attn_decode_fused(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const float *__restrict__ qkv,
    Rows r, const float *__restrict__ q_gain, const float *__restrict__ k_gain, const float2 *__restrict__ rope,
    bf16 *__restrict__ k_layer, bf16 *__restrict__ v_layer, float *__restrict__ ws_ml, float *__restrict__ ws_o,
    int *__restrict__ counters, bf16 *__restrict__ out, int Hq, int Hkv, int max_ctx, float eps, float scale_log2,
    uint32_t *err) {
    extern __shared__ uint8_t smem_raw[];
    // the swizzle pattern of a box repeats every 1024 bytes: the ring starts on such a boundary
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *s_new = ring + (size_t)STAGES * STAGE_BYTES;        // [K half 0, 1 | V half 0, 1][16][128 B]
    bf16 *s_q = reinterpret_cast<bf16 *>(s_new + NEW_BYTES);      // [G][128]: scaled q, bf16
    uint64_t *full = reinterpret_cast<uint64_t *>(s_q + MAX_G * D);  // [STAGES]
    // after the key loop the ring is free: the cross-warp and cross-split merges reuse it
    float(*red_o)[G][D] = reinterpret_cast<float(*)[G][D]>(ring);                         // [NW]
    float(*red_ml)[G][2] = reinterpret_cast<float(*)[G][2]>(ring + NW * G * D * 4);       // [NW]
    float(*sp_w)[ATTN_DECODE_MAX_SPLIT] =
        reinterpret_cast<float(*)[ATTN_DECODE_MAX_SPLIT]>(ring + NW * G * (D + 2) * 4);  // [G]
    __shared__ float s_lsum[G];
    __shared__ int s_last;
    // paged cache: the block-table entries of this CTA's key range, read once before the first
    // copy (a lookup per copy would put an L2 round trip in front of every refill of the ring)
    constexpr int MAX_BLK = PAGED ? 1024 : 1;
    __shared__ int32_t s_blk[MAX_BLK];

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int n_split = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane & 7, kg = lane >> 3;
    // Written by kernels that have completed (see above), so they may be read before the
    // dependency wait -- but only from L2 (ld.global.cg): this SM's L1 may still hold the
    // previous step's lines, and only the wait would invalidate them.
    const int slot = __ldcg(r.row_slot + b);
    const int pos = __ldcg(r.row_pos + b);
    const bool pos_ok = pos < max_ctx;
    const int per = ((pos + n_split) / n_split + CHUNK - 1) / CHUNK * CHUNK;  // ceil((pos+1)/n) in chunks
    const int k_begin = split * per;
    const int k_end = pos_ok ? min(pos + 1, k_begin + per) : k_begin;
    const int cache_end = max(k_begin, min(k_end, pos));  // cached keys [k_begin, cache_end)
    const int n_chunks = (cache_end - k_begin + CHUNK - 1) / CHUNK;
    KvMap kv = r.kv;
    if (!PAGED) kv.table = nullptr;  // the contiguous form compiles to plain slot-major offsets
    const int blk0 = PAGED ? k_begin / kv.bs : 0;
    const bool blk_cached = PAGED && cache_end > k_begin && (cache_end - 1) / kv.bs - blk0 < MAX_BLK;
    if (blk_cached) {
        for (int i = blk0 + threadIdx.x; i <= (cache_end - 1) / kv.bs; i += blockDim.x)
            s_blk[i - blk0] = __ldcg(kv.table + (size_t)slot * kv.max_blocks + i);
        __syncthreads();
    }
    auto cache_row = [&](int p) -> size_t {  // row of position p (< cache_end) of (slot, g)
        if (blk_cached) return ((size_t)s_blk[p / kv.bs - blk0] * Hkv + g) * kv.bs + p % kv.bs;
        return kv_row(kv, slot, Hkv, g, max_ctx, p);
    };
    auto issue = [&](int c) {  // chunk c of this split (keys k_begin + 64c ..) into stage c % STAGES
        const int st = c % STAGES;
        const int y = (int)cache_row(k_begin + c * CHUNK);  // a chunk never crosses a paged block
        uint8_t *dst = ring + (size_t)st * STAGE_BYTES;
        mbar_expect_tx(&full[st], STAGE_BYTES);
        tma2d(dst, &tmK, 0, y, &full[st]);
        tma2d(dst + BOX_BYTES, &tmK, 64, y, &full[st]);
        tma2d(dst + 2 * BOX_BYTES, &tmV, 0, y, &full[st]);
        tma2d(dst + 3 * BOX_BYTES, &tmV, 64, y, &full[st]);
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < STAGES; ++st) mbar_init(&full[st], 1);
        for (int c = 0; c < min(STAGES, n_chunks); ++c) issue(c);
    }
    for (int i = threadIdx.x; i < NEW_BYTES / 16; i += NW * 32)  // rows 1..15 of the new row's tile stay zero
        reinterpret_cast<uint4 *>(s_new)[i] = make_uint4(0, 0, 0, 0);
    const long long lim = wait_limit(err);
    float gq[16], gk[16];
    float2 cs[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        gq[e] = q_gain[sub * 16 + e];
        gk[e] = k_gain[sub * 16 + e];
        cs[e] = pos_ok ? rope[(size_t)pos * (D / 2) + (sub & 3) * 16 + e] : make_float2(1.0f, 0.0f);
    }
    __syncthreads();  // the barriers are initialised before anyone waits on them

    pdl_wait();
    pdl_trigger();
    if (!pos_ok) {
        if (threadIdx.x == 0 && split == 0 && err) atomicOr(err, ERR_POSITION);
        return;  // no copy was issued
    }
    const int heads = Hq + 2 * Hkv;
    const float *row = qkv + (size_t)b * heads * D;
    // per-head RMSNorm + rotate-half RoPE of the G query heads (into s_q, scaled, bf16) and of
    // the new key (into the new row's tile and the cache); warp 0's first 8-lane group writes
    for (int hh = 0; hh < G + 2; ++hh) {
        const int head = hh < G ? g * G + hh : (hh == G ? Hq + g : Hq + Hkv + g);
        float x[16];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(row + (size_t)head * D + sub * 16 + e);
            x[e] = t.x; x[e + 1] = t.y; x[e + 2] = t.z; x[e + 3] = t.w;
        }
        if (hh <= G) {
            float ss = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) ss += x[e] * x[e];
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            ss += __shfl_xor_sync(0xffffffffu, ss, 4);
            const float inv = rsqrtf(ss * (1.0f / D) + eps);
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] *= inv * (hh < G ? gq[e] : gk[e]);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float partner = __shfl_xor_sync(0xffffffffu, x[e], 4);
                x[e] = sub < 4 ? x[e] * cs[e].x - partner * cs[e].y   // x_i cos - x_{i+64} sin
                               : x[e] * cs[e].x + partner * cs[e].y;  // x_{i+64} cos + x_i sin
            }
        }
        if (warp == 0 && kg == 0) {
            const float sc = hh < G ? scale_log2 : 1.0f;
            uint4 pk[2];
            uint32_t *a = reinterpret_cast<uint32_t *>(pk);
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] = pack_bf16x2(x[2 * e] * sc, x[2 * e + 1] * sc);
            if (hh < G) {
                uint4 *dq = reinterpret_cast<uint4 *>(s_q + hh * D + sub * 16);
                dq[0] = pk[0];
                dq[1] = pk[1];
            } else {
                // row 0 of the tile (no swizzle offset in row 0): dims sub*16.. in half sub / 4
                uint4 *dn = reinterpret_cast<uint4 *>(s_new + (hh - G) * 2 * NEW_HALF + (sub >> 2) * NEW_HALF +
                                                      (sub & 3) * 32);
                dn[0] = pk[0];
                dn[1] = pk[1];
                if (split == 0) {
                    const size_t crow = kv_row(kv, slot, Hkv, g, max_ctx, pos);
                    uint4 *dc = reinterpret_cast<uint4 *>((hh == G ? k_layer : v_layer) + crow * D + sub * 16);
                    dc[0] = pk[0];
                    dc[1] = pk[1];
                }
            }
        }
    }
    __syncthreads();  // s_q and the new row's tile are written

    // the B operand Q^T of S^T = K Q^T: column (head) gq = lane / 4, rows (dims) 2t, 2t+1, +8, +9
    const int gr = lane >> 2, t = lane & 3;
    uint32_t qb[8][2];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(s_q + gr * D);
        qb[kk][0] = gr < G ? qw[8 * kk + t] : 0u;
        qb[kk][1] = gr < G ? qw[8 * kk + t + 4] : 0u;
    }
    // this lane's running state for heads 2t, 2t+1 (columns of the fragments): m and l over the
    // keys it holds (l is summed over the warp's lanes at the end), O^T rows (dims) of 8 tiles
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;

    // ldmatrix row addresses of this lane: K as the A operand (matrix q: keys + 8 (q & 1), dims
    // + 8 (q >> 1)), V^T as the A operand through .trans (matrix q: keys + 8 (q >> 1), dims
    // + 8 (q & 1))
    const int lq = lane >> 3, li = lane & 7;
    const int k_row = li + 8 * (lq & 1), k_dh = lq >> 1;
    const int v_row = li + 8 * (lq >> 1), v_dh = lq & 1;
    // one 16-key tile of this warp: rows row0 .. row0+15 of boxes of `half` bytes per 64-dim
    // half (K at kb, V at vb); keys row0 + g with g < n_valid are real
    auto tile = [&](uint32_t kb, uint32_t vb, uint32_t half, int row0, int n_valid) {
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const int kr = row0 + k_row;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a[4];
            ldsm_x4(a, kb + (kk >> 2) * half + swz(kr, (2 * kk + k_dh) & 7));
            mma16816(s, a, qb[kk][0], qb[kk][1]);
        }
        // s[0], s[1]: key row0 + gr, heads 2t, 2t+1; s[2], s[3]: key row0 + gr + 8
        const bool v0 = gr < n_valid, v1 = gr + 8 < n_valid;
        float pl[2], ph[2], corr[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(v0 ? s[j] : -INFINITY, v1 ? s[2 + j] : -INFINITY);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m_run[j], mx);
            corr[j] = m_run[j] == mn ? 1.0f : exp2f(m_run[j] - mn);  // -inf -> finite: 0
            pl[j] = v0 ? exp2f(s[j] - mn) : 0.0f;
            ph[j] = v1 ? exp2f(s[2 + j] - mn) : 0.0f;
            l_run[j] = l_run[j] * corr[j] + pl[j] + ph[j];
            m_run[j] = mn;
        }
        if (__any_sync(0xffffffffu, corr[0] != 1.0f || corr[1] != 1.0f)) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                o[mt][0] *= corr[0];
                o[mt][1] *= corr[1];
                o[mt][2] *= corr[0];
                o[mt][3] *= corr[1];
            }
        }
        // P^T as the B operand: this lane needs P[keys 2t, 2t+1, 2t+8, 2t+9][head gr], held as
        // element gr & 1 by lanes 4 (2t) + gr/2 and 4 (2t+1) + gr/2
        const int sa = 8 * t + (gr >> 1), sb = sa + 4;
        const float a0 = __shfl_sync(0xffffffffu, pl[0], sa), a1 = __shfl_sync(0xffffffffu, pl[1], sa);
        const float a2 = __shfl_sync(0xffffffffu, ph[0], sa), a3 = __shfl_sync(0xffffffffu, ph[1], sa);
        const float b0 = __shfl_sync(0xffffffffu, pl[0], sb), b1 = __shfl_sync(0xffffffffu, pl[1], sb);
        const float b2 = __shfl_sync(0xffffffffu, ph[0], sb), b3 = __shfl_sync(0xffffffffu, ph[1], sb);
        const bool odd = gr & 1, real = gr < G;
        const uint32_t pb0 = real ? pack_bf16x2(odd ? a1 : a0, odd ? b1 : b0) : 0u;
        const uint32_t pb1 = real ? pack_bf16x2(odd ? a3 : a2, odd ? b3 : b2) : 0u;
        const int vr = row0 + v_row;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t a[4];
            ldsm_x4_t(a, vb + (mt >> 2) * half + swz(vr, (2 * mt + v_dh) & 7));
            mma16816(o[mt], a, pb0, pb1);
        }
    };

    bool ok = true;
    int stop = 0;  // first chunk not consumed: chunks stop .. stop + STAGES - 1 may be in flight
    const uint32_t ring_a = smem_addr(ring);
    for (int c = 0; c < n_chunks; ++c) {
        const int st = c % STAGES;
        stop = c;
        const bool late = !mbar_wait_ctx(&full[st], (c / STAGES) & 1, err, lim);
        if (__syncthreads_or(late)) {  // the whole CTA gives up together
            ok = false;
            break;
        }
        const int n = min(CHUNK, cache_end - (k_begin + c * CHUNK));
        const uint32_t kb = ring_a + st * STAGE_BYTES;
        tile(kb, kb + 2 * BOX_BYTES, BOX_BYTES, 16 * warp, n - 16 * warp);
        __syncthreads();  // every warp is done with stage st
        if (threadIdx.x == 0 && c + STAGES < n_chunks) issue(c + STAGES);
    }
    if (!ok) {
        // Let the copies in flight land (the latest issued phase of each stage), then take part
        // in the split count as usual, so the counter is left zero; the output stays unwritten
        // and the error word says why.
        if (threadIdx.x == 0)
            for (int c = stop; c < min(stop + STAGES, n_chunks); ++c)
                mbar_wait_bounded(&full[c % STAGES], (c / STAGES) & 1, nullptr);
        if (n_split > 1 && threadIdx.x == 0 && atomicAdd(&counters[b * Hkv + g], 1) == n_split - 1)
            counters[b * Hkv + g] = 0;
        return;
    }
    if (warp == 0 && k_begin <= pos && pos < k_end) {  // the new key: row 0 of its own tile
        const uint32_t nb = smem_addr(s_new);
        tile(nb, nb + 2 * NEW_HALF, NEW_HALF, 0, 1);
    }

    // l over the warp's keys; the warps' partials through shared memory (the ring is free)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int h = 2 * t + j;
        if (h < G) {
            if (gr == 0) {
                red_ml[warp][h][0] = m_run[j];
                red_ml[warp][h][1] = l_run[j];
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                red_o[warp][h][16 * mt + gr] = o[mt][j];
                red_o[warp][h][16 * mt + gr + 8] = o[mt][2 + j];
            }
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int gi = idx / D, d = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) mx = fmaxf(mx, red_ml[w][gi][0]);
        float lsum = 0.0f, ov = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float c = mx == -INFINITY ? 0.0f : exp2f(red_ml[w][gi][0] - mx);
            lsum += red_ml[w][gi][1] * c;
            ov += red_o[w][gi][d] * c;
        }
        const int h = g * G + gi;
        if (n_split == 1) {
            out[((size_t)b * Hq + h) * D + d] = __float2bfloat16(ov / lsum);
        } else {
            const size_t part = ((size_t)b * Hq + h) * n_split + split;
            ws_o[part * D + d] = ov;
            if (d == 0) {
                ws_ml[part * 2] = mx;
                ws_ml[part * 2 + 1] = lsum;
            }
        }
    }
    if (n_split == 1) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&counters[b * Hkv + g], 1) == n_split - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // weights of the splits: exp2(m_s - max) per query head, and the merged denominator
    if (threadIdx.x < G) {
        const int gi = threadIdx.x;
        const size_t base = ((size_t)b * Hq + g * G + gi) * n_split;
        float mx = -INFINITY;
        for (int sp = 0; sp < n_split; ++sp) mx = fmaxf(mx, __ldcg(ws_ml + (base + sp) * 2));
        float lsum = 0.0f;
        for (int sp = 0; sp < n_split; ++sp) {
            const float ms = __ldcg(ws_ml + (base + sp) * 2);
            const float w = ms == -INFINITY ? 0.0f : exp2f(ms - mx);
            sp_w[gi][sp] = w;
            lsum += __ldcg(ws_ml + (base + sp) * 2 + 1) * w;
        }
        s_lsum[gi] = lsum;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int gi = idx / D, d = idx % D;
        const int h = g * G + gi;
        const float *po = ws_o + ((size_t)b * Hq + h) * n_split * D + d;
        float ov = 0.0f;
#pragma unroll 8
        for (int sp = 0; sp < n_split; ++sp) ov = fmaf(__ldcg(po + (size_t)sp * D), sp_w[gi][sp], ov);
        out[((size_t)b * Hq + h) * D + d] = __float2bfloat16(ov / s_lsum[gi]);
    }
    if (threadIdx.x == 0) counters[b * Hkv + g] = 0;
}

// 1024 bytes of alignment slack, the ring, the new row's tile, q, the barriers
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + NEW_BYTES + MAX_G * D * 2 + 64;

template <int G>
cudaError_t run_fused(const Launch &lc, const float *qkv, const Rows &r, const float *q_gain,
                      const float *k_gain, const float2 *rope, bf16 *k_layer, bf16 *v_layer, size_t kv_rows,
                      int n_split, float *ws_ml, float *ws_o, int *counters, bf16 *out, int Hq, int Hkv,
                      int max_ctx, float eps, uint32_t *err) {
    static_assert(NW * G * (D + 2) * 4 + G * ATTN_DECODE_MAX_SPLIT * 4 <= STAGES * STAGE_BYTES,
                  "merge scratch fits in the ring");
    if (n_split < 1 || n_split > ATTN_DECODE_MAX_SPLIT || (r.kv.table && r.kv.bs % CHUNK)) return cudaErrorInvalidValue;
    CUtensorMap mk, mv;
    if (!kv_tile_map(&mk, k_layer, kv_rows) || !kv_tile_map(&mv, v_layer, kv_rows)) return cudaErrorInvalidValue;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    auto kern = r.kv.table ? k_attn_decode_fused<G, true> : k_attn_decode_fused<G, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch(lc, kern, dim3(n_split, Hkv, r.B), dim3(NW * 32), SMEM_BYTES, mk, mv, qkv, r, q_gain, k_gain, rope,
                  k_layer, v_layer, ws_ml, ws_o, counters, out, Hq, Hkv, max_ctx, eps, scale_log2, err);
}

template <int G>
int ctas_per_sm() {
    int n = 0;
    if (cudaFuncSetAttribute(k_attn_decode_fused<G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_attn_decode_fused<G, false>, NW * 32, SMEM_BYTES) !=
            cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

}  // namespace

cudaError_t launch_attn_decode_fused(const Launch &lc, const float *qkv, const Rows &r,
                                     const float *q_gain, const float *k_gain, const float2 *rope,
                                     bf16 *k_layer, bf16 *v_layer, size_t kv_rows, int n_split,
                                     float *ws_ml, float *ws_o, int *counters, bf16 *out, int Hq,
                                     int Hkv, int max_ctx, float eps, uint32_t *err) {
#define Q3_ATTN(GG) run_fused<GG>(lc, qkv, r, q_gain, k_gain, rope, k_layer, v_layer, kv_rows, n_split, ws_ml, ws_o, \
                                  counters, out, Hq, Hkv, max_ctx, eps, err)
    switch (Hq / Hkv) {
        case 1: return Q3_ATTN(1);
        case 2: return Q3_ATTN(2);
        case 4: return Q3_ATTN(4);
        case 8: return Q3_ATTN(8);
    }
#undef Q3_ATTN
    return cudaErrorInvalidValue;
}

int attn_decode_ctas_per_sm(int Hq, int Hkv) {
    switch (Hq / Hkv) {
        case 1: return ctas_per_sm<1>();
        case 2: return ctas_per_sm<2>();
        case 4: return ctas_per_sm<4>();
        case 8: return ctas_per_sm<8>();
    }
    return 1;
}

}  // namespace q3
