// Split-KV decode attention: one new query row per sequence against its cached keys 0..p.
//
// A decode query at absolute position p sees every cached key 0..p, its own included
// ("从零开始写Qwen3", Attn: no causal flag for a length-1 query; "古法手撕简易LLM推理器",
// 核心计算函数与Transformer层: no mask once offset > 0, the new key appended first).  The
// Hq/Hkv query heads of one KV head are served by the same CTA so each K/V row is read
// from HBM once ("手写Qwen3-0.6B推理", Attention: K/V shared by a group of query heads).
//
// Grid (split, kv head, sequence): 8 lanes per key (16 dims each), 4 keys per warp and step;
// dot products reduced with 3 warp shuffles; an online softmax (m, l, acc) per 8-lane group,
// merged across groups with shuffles and across the warps in shared memory.  Each split
// writes (m, l) and the unnormalised acc of its key range to a workspace and the last CTA of
// a (sequence, KV head) takes the log-sum-exp merge of the splits.  Scores are pre-scaled by
// log2(e)/sqrt(128) so exp2 is used throughout.

#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
// QK-norm + RoPE + KV write in the prologue, split merge by the last CTA.
//
// Reads the new row's q/k/v straight from the QKV projection (fp32 [B, (Hq+2Hkv)*128]).
// Each CTA normalises and rotates its query heads and the new key in registers (lane `sub`
// of each 8-lane group holds elements sub*16 .. sub*16+15, so the RoPE partner i+64 of
// element i sits in lane sub^4).  The new K (rounded to bf16, as the cache stores it) and V
// are written to the cache by split 0 and taken from shared memory by the split that covers
// the new position; every other key comes from the cache.
//
// Cached keys stream through a ring of shared-memory stages filled by bulk asynchronous
// copies.  Every kernel of the decode chain passes its own dependency wait before it lets
// the next kernel launch, so when this kernel starts, every kernel before the QKV projection
// has completed: the cached rows 0..pos-1, the row positions, the gains and the RoPE table
// are final, and the first stages are requested before the wait.  Only q/k/v of the new
// row come from the immediately preceding kernel.
//
// Split s of n covers keys [s*per, min((s+1)*per, p+1)) with per = ceil((p+1)/n), taken from
// the sequence's own position on the device: the ranges stay balanced for every length that
// a recorded launch (a fixed n) serves.
//
// The CTA that finishes last for a (sequence, KV head) merges all splits (a counter per
// pair, incremented after a memory fence and reset by that CTA): no second kernel and no
// waiting on other CTAs.

constexpr int STAGES = 3;
constexpr int NW = 4;                        // warps per CTA
constexpr int KPG = 4;                       // keys per 8-lane group and step
constexpr int CHUNK = NW * 4 * KPG;          // keys per ring stage: one step of the CTA
constexpr int STAGE_BYTES = CHUNK * D * 2 * 2;  // K and V rows of one chunk

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16(x)); }

template <int G, bool PAGED>
__global__ void __launch_bounds__(NW * 32, 2) k_attn_decode_fused(
    const float *__restrict__ qkv, Rows r, const float *__restrict__ q_gain,
    const float *__restrict__ k_gain, const float2 *__restrict__ rope, bf16 *__restrict__ k_layer,
    bf16 *__restrict__ v_layer, float *__restrict__ ws_ml, float *__restrict__ ws_o,
    int *__restrict__ counters, bf16 *__restrict__ out, int Hq, int Hkv, int max_ctx, float eps,
    float scale_log2, uint32_t *err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);              // [STAGES]
    uint8_t *ring = smem + 128;                                        // [STAGES][K | V]
    float *s_new = reinterpret_cast<float *>(ring + STAGES * STAGE_BYTES);  // new K, new V [2][D]
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
    const int per = (pos + n_split) / n_split;  // ceil((pos + 1) / n_split)
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
    auto issue = [&](int c) {  // chunk c of this split into stage c % STAGES
        const int st = c % STAGES;
        const int j0 = k_begin + c * CHUNK;
        const int n = min(CHUNK, cache_end - j0);
        mbar_expect_tx(&full[st], 2 * (uint32_t)n * D * 2);
        // keys j0 .. j0+n-1 as runs of consecutive cache rows: one run, or two where a paged
        // cache's block ends inside the chunk (blocks hold at least CHUNK keys)
        for (int done = 0; done < n;) {
            const int p = j0 + done;
            const int run = PAGED ? min(n - done, kv.bs - p % kv.bs) : n - done;
            const size_t row = cache_row(p);
            const uint32_t bytes = (uint32_t)run * D * 2;
            bulk_g2s(ring + st * STAGE_BYTES + (size_t)done * D * 2, k_layer + row * D, bytes, &full[st]);
            bulk_g2s(ring + st * STAGE_BYTES + CHUNK * D * 2 + (size_t)done * D * 2, v_layer + row * D, bytes,
                     &full[st]);
            done += run;
        }
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < STAGES; ++st) mbar_init(&full[st], 1);
        for (int c = 0; c < min(STAGES, n_chunks); ++c) issue(c);
    }
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
    // one round trip: every q/k/v value this lane needs
    float x[G + 2][16];
#pragma unroll
    for (int hh = 0; hh < G + 2; ++hh) {
        const int head = hh < G ? g * G + hh : (hh == G ? Hq + g : Hq + Hkv + g);
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(row + (size_t)head * D + sub * 16 + e);
            x[hh][e] = t.x; x[hh][e + 1] = t.y; x[hh][e + 2] = t.z; x[hh][e + 3] = t.w;
        }
    }
    // per-head RMSNorm + rotate-half RoPE of the G query heads and the new key
    float qv[G][16];
#pragma unroll
    for (int hh = 0; hh < G + 1; ++hh) {
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) ss += x[hh][e] * x[hh][e];
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        const float inv = rsqrtf(ss * (1.0f / D) + eps);
        const float *gn = hh < G ? gq : gk;
#pragma unroll
        for (int e = 0; e < 16; ++e) x[hh][e] *= inv * gn[e];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float partner = __shfl_xor_sync(0xffffffffu, x[hh][e], 4);
            const float rot = sub < 4 ? x[hh][e] * cs[e].x - partner * cs[e].y   // x_i cos - x_{i+64} sin
                                      : x[hh][e] * cs[e].x + partner * cs[e].y;  // x_{i+64} cos + x_i sin
            if (hh < G) qv[hh < G ? hh : 0][e] = rot * scale_log2;
            else x[G][e] = round_bf16(rot);
        }
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) x[G + 1][e] = round_bf16(x[G + 1][e]);
    if (warp == 0 && kg == 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            s_new[sub * 16 + e] = x[G][e];
            s_new[D + sub * 16 + e] = x[G + 1][e];
        }
        if (split == 0) {
            uint4 pk[2], pv[2];
            uint32_t *a = reinterpret_cast<uint32_t *>(pk), *c = reinterpret_cast<uint32_t *>(pv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                a[e] = pack_bf16x2(x[G][2 * e], x[G][2 * e + 1]);
                c[e] = pack_bf16x2(x[G + 1][2 * e], x[G + 1][2 * e + 1]);
            }
            const size_t row = kv_row(kv, slot, Hkv, g, max_ctx, pos);
            uint4 *kd = reinterpret_cast<uint4 *>(k_layer + row * D + sub * 16);
            uint4 *vd = reinterpret_cast<uint4 *>(v_layer + row * D + sub * 16);
            kd[0] = pk[0]; kd[1] = pk[1];
            vd[0] = pv[0]; vd[1] = pv[1];
        }
    }

    float m[G], l[G], acc[G][16];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        m[gi] = -INFINITY;
        l[gi] = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[gi][e] = 0.0f;
    }
    // KPG keys of this 8-lane group: scores, one max and one rescale for all of them
    auto update = [&](const float (*kf)[16], const float (*vf)[16], const bool *valid) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            float sc[KPG];
#pragma unroll
            for (int kk = 0; kk < KPG; ++kk) {
                float t = 0.0f;
#pragma unroll
                for (int e = 0; e < 16; ++e) t = fmaf(qv[gi][e], kf[kk][e], t);
                sc[kk] = t;
            }
#pragma unroll
            for (int kk = 0; kk < KPG; ++kk) sc[kk] += __shfl_xor_sync(0xffffffffu, sc[kk], 1);
#pragma unroll
            for (int kk = 0; kk < KPG; ++kk) sc[kk] += __shfl_xor_sync(0xffffffffu, sc[kk], 2);
#pragma unroll
            for (int kk = 0; kk < KPG; ++kk) sc[kk] += __shfl_xor_sync(0xffffffffu, sc[kk], 4);
            float mn = m[gi];
#pragma unroll
            for (int kk = 0; kk < KPG; ++kk)
                if (valid[kk]) mn = fmaxf(mn, sc[kk]);
            if (mn != -INFINITY) {  // some key of the group seen so far
                const float c = exp2f(m[gi] - mn);
                float p[KPG];
                float ps = 0.0f;
#pragma unroll
                for (int kk = 0; kk < KPG; ++kk) {
                    p[kk] = valid[kk] ? exp2f(sc[kk] - mn) : 0.0f;
                    ps += p[kk];
                }
                l[gi] = l[gi] * c + ps;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float a = acc[gi][e] * c;
#pragma unroll
                    for (int kk = 0; kk < KPG; ++kk) a = fmaf(p[kk], vf[kk][e], a);
                    acc[gi][e] = a;
                }
                m[gi] = mn;
            }
        }
    };

    bool ok = true;
    int stop = 0;  // first chunk not consumed: chunks stop .. stop + STAGES - 1 may be in flight
    const int j0 = (warp * 4 + kg) * KPG;  // this group's first key in each chunk
    for (int c = 0; c < n_chunks; ++c) {
        const int st = c % STAGES;
        stop = c;
        const bool late = !mbar_wait_ctx(&full[st], (c / STAGES) & 1, err, lim);
        if (__syncthreads_or(late)) {  // the whole CTA gives up together
            ok = false;
            break;
        }
        const uint8_t *ks = ring + st * STAGE_BYTES;
        const uint8_t *vs = ks + CHUNK * D * 2;
        const int n = min(CHUNK, cache_end - (k_begin + c * CHUNK));
        float kf[KPG][16], vf[KPG][16];
        bool valid[KPG];
#pragma unroll
        for (int kk = 0; kk < KPG; ++kk) {
            valid[kk] = j0 + kk < n;
            const int js = valid[kk] ? j0 + kk : 0;
            const uint4 *kp = reinterpret_cast<const uint4 *>(ks + (size_t)js * D * 2 + sub * 32);
            const uint4 *vp = reinterpret_cast<const uint4 *>(vs + (size_t)js * D * 2 + sub * 32);
            unpack8(kp[0], kf[kk]);
            unpack8(kp[1], kf[kk] + 8);
            unpack8(vp[0], vf[kk]);
            unpack8(vp[1], vf[kk] + 8);
        }
        update(kf, vf, valid);
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
    __syncthreads();  // s_new is visible
    if (warp == 0 && k_begin <= pos && pos < k_end) {  // the new key, from shared memory
        float kf[KPG][16], vf[KPG][16];
        bool valid[KPG];
#pragma unroll
        for (int kk = 0; kk < KPG; ++kk) {
            valid[kk] = kk == 0 && kg == 0;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                kf[kk][e] = s_new[sub * 16 + e];
                vf[kk][e] = s_new[D + sub * 16 + e];
            }
        }
        update(kf, vf, valid);
    }

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
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int gi = idx / D, d = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) mx = fmaxf(mx, red_ml[w][gi][0]);
        float lsum = 0.0f, o = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float c = mx == -INFINITY ? 0.0f : exp2f(red_ml[w][gi][0] - mx);
            lsum += red_ml[w][gi][1] * c;
            o += red_o[w][gi][d] * c;
        }
        const int h = g * G + gi;
        if (n_split == 1) {
            out[((size_t)b * Hq + h) * D + d] = __float2bfloat16(o / lsum);
        } else {
            const size_t part = ((size_t)b * Hq + h) * n_split + split;
            ws_o[part * D + d] = o;
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
        float o = 0.0f;
#pragma unroll 8
        for (int sp = 0; sp < n_split; ++sp) o = fmaf(__ldcg(po + (size_t)sp * D), sp_w[gi][sp], o);
        out[((size_t)b * Hq + h) * D + d] = __float2bfloat16(o / s_lsum[gi]);
    }
    if (threadIdx.x == 0) counters[b * Hkv + g] = 0;
}

constexpr size_t SMEM_BYTES = 128 + (size_t)STAGES * STAGE_BYTES + 2 * D * sizeof(float);

template <int G>
cudaError_t run_fused(const Launch &lc, const float *qkv, const Rows &r, const float *q_gain,
                      const float *k_gain, const float2 *rope, bf16 *k_layer, bf16 *v_layer, int n_split,
                      float *ws_ml, float *ws_o, int *counters, bf16 *out, int Hq, int Hkv,
                      int max_ctx, float eps, uint32_t *err) {
    static_assert(NW * G * (D + 2) * 4 + G * ATTN_DECODE_MAX_SPLIT * 4 <= STAGES * STAGE_BYTES,
                  "merge scratch fits in the ring");
    if (n_split < 1 || n_split > ATTN_DECODE_MAX_SPLIT) return cudaErrorInvalidValue;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    auto kern = r.kv.table ? k_attn_decode_fused<G, true> : k_attn_decode_fused<G, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch(lc, kern, dim3(n_split, Hkv, r.B), dim3(NW * 32), SMEM_BYTES, qkv, r, q_gain, k_gain, rope,
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
                                     bf16 *k_layer, bf16 *v_layer, int n_split,
                                     float *ws_ml, float *ws_o, int *counters, bf16 *out, int Hq,
                                     int Hkv, int max_ctx, float eps, uint32_t *err) {
#define Q3_ATTN(GG) run_fused<GG>(lc, qkv, r, q_gain, k_gain, rope, k_layer, v_layer, n_split, ws_ml, ws_o, \
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
