// Split-KV decode attention over equal shares of all keys of a step.
//
// The same computation as k_attn_decode_fused ("从零开始写Qwen3", Attn: a one-row query sees
// every cached key; "古法手撕简易LLM推理器", 核心计算函数与Transformer层: the new key appended
// first; "手写Qwen3-0.6B推理", Attention: the K/V of a KV head shared by its query heads), with
// another division of the work.  That kernel gives every (sequence, KV head) pair the same
// number of key ranges, so when the pairs do not divide the CTA slots of one wave (256 pairs
// on 304 slots) some SMs run two ranges and some one, and the kernel lasts as long as the
// busiest.  Here the keys of all pairs are laid end to end -- pair (b, g) = KV head g of
// sequence b holds keys 0..p_b, pairs in (b, g) order -- and CTA s of S takes the keys
// [s W / S, (s+1) W / S) of the W in all: every CTA streams the same number of K/V rows.
// A CTA's range covers the end of one pair and the start of the next (rarely more); it runs
// them one after another as segments: the pair's QK-norm + RoPE of the new row (and the KV
// write, by the CTA holding position p_b), its keys through the same bulk-copy ring and
// online softmax, then the segment's partial (max, sum, unnormalised output) to the
// workspace.  A pair's segments are the CTAs its keys fall in; the last of them to finish
// (a counter per pair) merges the partials, or a pair held by one CTA writes its output
// directly.  Scores are pre-scaled by log2(e)/sqrt(128) so exp2 is used throughout.
//
// Position, slot and the cached rows are final before the dependency wait (every kernel of
// the step passes its own wait before the next may launch), so the prefix sums of the key
// counts, the segment boundaries and the first copies are done before it; only q/k/v of the
// new rows come from the kernel just before.

#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int STAGES = 3;
constexpr int NW = 4;                           // warps per CTA
constexpr int KPG = 4;                          // keys per 8-lane group and step
constexpr int CHUNK = NW * 4 * KPG;             // keys per ring stage: 64
constexpr int STAGE_BYTES = CHUNK * D * 2 * 2;  // K and V rows of one chunk
constexpr int FLAT_MAX_B = 1024;                // rows of one launch

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16(x)); }

// CTA of S (S <= W) that flattened key x falls in: the largest s with floor(s W / S) <= x.
__device__ __forceinline__ int cta_of(long long x, long long W, int S) { return (int)(((x + 1) * S - 1) / W); }

template <int G, bool PAGED>
__global__ void __launch_bounds__(NW * 32, 2) k_attn_decode_flat(
    const float *__restrict__ qkv, Rows r, const float *__restrict__ q_gain, const float *__restrict__ k_gain,
    const float2 *__restrict__ rope, bf16 *__restrict__ k_layer, bf16 *__restrict__ v_layer,
    float *__restrict__ ws_ml, float *__restrict__ ws_o, int *__restrict__ counters, bf16 *__restrict__ out,
    int Hq, int Hkv, int max_ctx, float eps, float scale_log2, uint32_t *err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);                     // [STAGES]
    uint8_t *ring = smem + 128;                                               // [STAGES][K | V]
    float *s_new = reinterpret_cast<float *>(ring + STAGES * STAGE_BYTES);   // new K, new V [2][D]
    int *s_cum = reinterpret_cast<int *>(s_new + 2 * D);                     // [B + 1] keys of rows < b
    // after a segment's keys the ring is free: its cross-warp and cross-segment merges reuse it
    float(*red_o)[G][D] = reinterpret_cast<float(*)[G][D]>(ring);
    float(*red_ml)[G][2] = reinterpret_cast<float(*)[G][2]>(ring + NW * G * D * 4);
    float(*sp_w)[ATTN_DECODE_MAX_SPLIT] =
        reinterpret_cast<float(*)[ATTN_DECODE_MAX_SPLIT]>(ring + NW * G * (D + 2) * 4);
    __shared__ float s_lsum[G];
    __shared__ int s_last;
    __shared__ int s_warp_sum[NW];
    // paged cache: the block-table entries of the current segment's keys, read once per segment
    // (a lookup per copy would put an L2 round trip in front of every refill of the ring)
    constexpr int MAX_BLK = PAGED ? 1024 : 1;
    __shared__ int32_t s_blk[MAX_BLK];

    const int S = gridDim.x, s = blockIdx.x, B = r.B;  // S CTAs; the first Se of them take keys
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane & 7, kg = lane >> 3;
    const long long lim = wait_limit(err);

    // keys per row: p_b + 1 (0 for a row whose position is out of range: nothing is done for it)
    // and their exclusive prefix sums, read before the dependency wait from L2 (see above)
    {
        constexpr int PER = (FLAT_MAX_B + NW * 32 - 1) / (NW * 32);
        int v[PER], run = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int b = threadIdx.x * PER + i;
            int n = 0;
            if (b < B) {
                const int p = __ldcg(r.row_pos + b);
                n = p < max_ctx ? p + 1 : 0;
            }
            v[i] = run;
            run += n;
        }
        int incl = run;  // inclusive scan of the per-thread totals over the CTA
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) s_warp_sum[warp] = incl;
        __syncthreads();
        int base = incl - run;
        for (int w = 0; w < warp; ++w) base += s_warp_sum[w];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int b = threadIdx.x * PER + i;
            if (b < B) s_cum[b] = base + v[i];
        }
        if (threadIdx.x == NW * 32 - 1) s_cum[B] = base + run;  // all keys
        if (threadIdx.x == 0) {
            for (int st = 0; st < STAGES; ++st) mbar_init(&full[st], 1);
        }
        __syncthreads();
    }
    // With fewer keys than CTAs only the first W CTAs take keys (one or more each): a pair's
    // segments must be exactly the CTAs of the consecutive range its keys fall in, so no CTA
    // may be left with an empty range inside it.
    const long long W = (long long)Hkv * s_cum[B];
    const int Se = (int)(W < S ? W : S);
    const long long r0 = s < Se ? W * s / Se : 0, r1 = s < Se ? W * (s + 1) / Se : 0;

    // the pair holding flattened key x: row b (largest with Hkv * cum[b] <= x), head g, key j
    auto locate = [&](long long x, int &b, int &g, int &j) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)Hkv * s_cum[mid] <= x) lo = mid; else hi = mid - 1;
        }
        b = lo;
        const int n = s_cum[b + 1] - s_cum[b];
        const long long off = x - (long long)Hkv * s_cum[b];
        g = (int)(off / n);
        j = (int)(off % n);
    };

    KvMap kv = r.kv;
    if (!PAGED) kv.table = nullptr;
    // The ring's chunks are counted across segments: chunk gc of the CTA uses stage gc % STAGES
    // in its phase gc / STAGES.  The current segment: (slot, KV head), cached rows [c0, c1),
    // its first chunk gbase.
    int seg_slot = 0, seg_g = 0, seg_c0 = 0, seg_c1 = 0, gbase = 0, blk0 = 0;
    bool blk_cached = false;
    auto cache_row = [&](int p) -> size_t {  // row of cached position p of the segment's pair
        if (blk_cached) return ((size_t)s_blk[p / kv.bs - blk0] * Hkv + seg_g) * kv.bs + p % kv.bs;
        return kv_row(kv, seg_slot, Hkv, seg_g, max_ctx, p);
    };
    auto issue = [&](int c) {  // chunk c of the segment (thread 0)
        const int gc = gbase + c, st = gc % STAGES;
        const int j0 = seg_c0 + c * CHUNK;
        const int n = min(CHUNK, seg_c1 - j0);
        mbar_expect_tx(&full[st], 2 * (uint32_t)n * D * 2);
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
    if (s == 0 && threadIdx.x == 0 && err) {  // rows whose position is out of range are skipped
        for (int b = 0; b < B; ++b)
            if (s_cum[b + 1] == s_cum[b]) {
                atomicOr(err, ERR_POSITION);
                break;
            }
    }

    bool waited = false, ok = true;
    for (long long x = r0; x < r1;) {
        int b, g, j0;
        locate(x, b, g, j0);
        const int n_keys = s_cum[b + 1] - s_cum[b];
        const int j1 = (int)min((long long)n_keys, j0 + (r1 - x));  // this segment: keys [j0, j1)
        const int pos = n_keys - 1;
        const long long off = (long long)Hkv * s_cum[b] + (long long)g * n_keys;
        const int first = cta_of(off, W, Se), n_seg = cta_of(off + n_keys - 1, W, Se) - first + 1;
        const int seg = s - first;
        x += j1 - j0;
        seg_slot = __ldcg(r.row_slot + b);
        seg_g = g;
        seg_c0 = j0;
        seg_c1 = max(j0, min(j1, pos));  // cached keys (the new one, at pos, comes from registers)
        const int n_chunks = ok ? (seg_c1 - seg_c0 + CHUNK - 1) / CHUNK : 0;
        if (PAGED) {
            blk0 = seg_c0 / kv.bs;
            blk_cached = n_chunks > 0 && (seg_c1 - 1) / kv.bs - blk0 < MAX_BLK;
            if (blk_cached)
                for (int i = blk0 + threadIdx.x; i <= (seg_c1 - 1) / kv.bs; i += blockDim.x)
                    s_blk[i - blk0] = __ldcg(kv.table + (size_t)seg_slot * kv.max_blocks + i);
            __syncthreads();
        }
        if (threadIdx.x == 0)
            for (int c = 0; c < min(STAGES, n_chunks); ++c) issue(c);

        float gq[16], gk[16];
        float2 cs[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            gq[e] = q_gain[sub * 16 + e];
            gk[e] = k_gain[sub * 16 + e];
            cs[e] = rope[(size_t)pos * (D / 2) + (sub & 3) * 16 + e];
        }
        if (!waited) {
            pdl_wait();
            pdl_trigger();
            waited = true;
        }
        const int heads = Hq + 2 * Hkv;
        const float *row = qkv + (size_t)b * heads * D;
        float xv[G + 2][16];
#pragma unroll
        for (int hh = 0; hh < G + 2; ++hh) {
            const int head = hh < G ? g * G + hh : (hh == G ? Hq + g : Hq + Hkv + g);
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 t = *reinterpret_cast<const float4 *>(row + (size_t)head * D + sub * 16 + e);
                xv[hh][e] = t.x; xv[hh][e + 1] = t.y; xv[hh][e + 2] = t.z; xv[hh][e + 3] = t.w;
            }
        }
        float qv[G][16];
#pragma unroll
        for (int hh = 0; hh < G + 1; ++hh) {  // per-head RMSNorm + rotate-half RoPE
            float ss = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) ss += xv[hh][e] * xv[hh][e];
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            ss += __shfl_xor_sync(0xffffffffu, ss, 4);
            const float inv = rsqrtf(ss * (1.0f / D) + eps);
            const float *gn = hh < G ? gq : gk;
#pragma unroll
            for (int e = 0; e < 16; ++e) xv[hh][e] *= inv * gn[e];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float partner = __shfl_xor_sync(0xffffffffu, xv[hh][e], 4);
                const float rot = sub < 4 ? xv[hh][e] * cs[e].x - partner * cs[e].y   // x_i cos - x_{i+64} sin
                                          : xv[hh][e] * cs[e].x + partner * cs[e].y;  // x_{i+64} cos + x_i sin
                if (hh < G) qv[hh < G ? hh : 0][e] = rot * scale_log2;
                else xv[G][e] = round_bf16(rot);
            }
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) xv[G + 1][e] = round_bf16(xv[G + 1][e]);
        const bool has_new = j0 <= pos && pos < j1;
        if (warp == 0 && kg == 0 && has_new) {  // the new row: kept for this segment, written to the cache
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                s_new[sub * 16 + e] = xv[G][e];
                s_new[D + sub * 16 + e] = xv[G + 1][e];
            }
            if (ok) {
                uint4 pk[2], pv[2];
                uint32_t *a = reinterpret_cast<uint32_t *>(pk), *c = reinterpret_cast<uint32_t *>(pv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    a[e] = pack_bf16x2(xv[G][2 * e], xv[G][2 * e + 1]);
                    c[e] = pack_bf16x2(xv[G + 1][2 * e], xv[G + 1][2 * e + 1]);
                }
                const size_t crow = kv_row(kv, seg_slot, Hkv, g, max_ctx, pos);
                uint4 *kd = reinterpret_cast<uint4 *>(k_layer + crow * D + sub * 16);
                uint4 *vd = reinterpret_cast<uint4 *>(v_layer + crow * D + sub * 16);
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
                if (mn != -INFINITY) {
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

        int stop = 0;  // first chunk not consumed: chunks stop .. stop + STAGES - 1 may be in flight
        const int jg = (warp * 4 + kg) * KPG;  // this group's first key in each chunk
        for (int c = 0; c < n_chunks; ++c) {
            const int gc = gbase + c, st = gc % STAGES;
            stop = c;
            const bool late = !mbar_wait_ctx(&full[st], (gc / STAGES) & 1, err, lim);
            if (__syncthreads_or(late)) {  // the whole CTA gives up together
                ok = false;
                break;
            }
            const uint8_t *ks = ring + st * STAGE_BYTES;
            const uint8_t *vs = ks + CHUNK * D * 2;
            const int n = min(CHUNK, seg_c1 - (seg_c0 + c * CHUNK));
            float kf[KPG][16], vf[KPG][16];
            bool valid[KPG];
#pragma unroll
            for (int kk = 0; kk < KPG; ++kk) {
                valid[kk] = jg + kk < n;
                const int js = valid[kk] ? jg + kk : 0;
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
        if (!ok && threadIdx.x == 0) {  // let the copies in flight land before the ring is reused
            for (int c = stop; c < min(stop + STAGES, n_chunks); ++c)
                mbar_wait_bounded(&full[(gbase + c) % STAGES], ((gbase + c) / STAGES) & 1, nullptr);
        }
        gbase += n_chunks;
        __syncthreads();  // s_new is visible; the ring is free
        if (ok && warp == 0 && has_new) {  // the new key, from shared memory
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
        // the four 8-lane groups of a warp, then the warps through shared memory
#pragma unroll
        for (int o = 8; o <= 16; o <<= 1) {
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                const float mo = __shfl_xor_sync(0xffffffffu, m[gi], o);
                const float lo = __shfl_xor_sync(0xffffffffu, l[gi], o);
                const float mn = fmaxf(m[gi], mo);
                const float c1 = mn == -INFINITY ? 0.0f : exp2f(m[gi] - mn);
                const float c2 = mn == -INFINITY ? 0.0f : exp2f(mo - mn);
                l[gi] = l[gi] * c1 + lo * c2;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float ao = __shfl_xor_sync(0xffffffffu, acc[gi][e], o);
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
        if (ok) {
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
                if (n_seg == 1) {
                    out[((size_t)b * Hq + h) * D + d] = __float2bfloat16(o / lsum);
                } else {
                    const size_t part = ((size_t)b * Hq + h) * ATTN_DECODE_MAX_SPLIT + seg;
                    ws_o[part * D + d] = o;
                    if (d == 0) {
                        ws_ml[part * 2] = mx;
                        ws_ml[part * 2 + 1] = lsum;
                    }
                }
            }
        }
        if (n_seg > 1) {  // the pair's last segment to finish merges them (a timed-out one still counts)
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_last = atomicAdd(&counters[b * Hkv + g], 1) == n_seg - 1;
            __syncthreads();
            if (s_last) {
                __threadfence();
                if (threadIdx.x < G) {
                    const int gi = threadIdx.x;
                    const size_t base = ((size_t)b * Hq + g * G + gi) * ATTN_DECODE_MAX_SPLIT;
                    float mx = -INFINITY;
                    for (int sp = 0; sp < n_seg; ++sp) mx = fmaxf(mx, __ldcg(ws_ml + (base + sp) * 2));
                    float lsum = 0.0f;
                    for (int sp = 0; sp < n_seg; ++sp) {
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
                    const float *po = ws_o + ((size_t)b * Hq + h) * ATTN_DECODE_MAX_SPLIT * D + d;
                    float o = 0.0f;
#pragma unroll 8
                    for (int sp = 0; sp < n_seg; ++sp) o = fmaf(__ldcg(po + (size_t)sp * D), sp_w[gi][sp], o);
                    out[((size_t)b * Hq + h) * D + d] = __float2bfloat16(o / s_lsum[gi]);
                }
                if (threadIdx.x == 0) counters[b * Hkv + g] = 0;
            }
        }
        __syncthreads();  // the merge scratch (the ring) is read; the next segment may fill it
    }
}

// ring + new row + prefix sums of up to FLAT_MAX_B rows
constexpr size_t FLAT_SMEM = 128 + (size_t)STAGES * STAGE_BYTES + 2 * D * sizeof(float) + (FLAT_MAX_B + 1) * 4;

}  // namespace

int attn_decode_flat_ctas_per_sm() {
    int n = 0;
    if (cudaFuncSetAttribute(k_attn_decode_flat<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)FLAT_SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_attn_decode_flat<2, false>, NW * 32, FLAT_SMEM) !=
            cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

bool attn_decode_flat_supported(int B, int Hq, int Hkv) { return B >= 1 && B <= FLAT_MAX_B && Hq == 2 * Hkv; }

cudaError_t launch_attn_decode_flat(const Launch &lc, const float *qkv, const Rows &r, const float *q_gain,
                                    const float *k_gain, const float2 *rope, bf16 *k_layer, bf16 *v_layer,
                                    int n_ctas, float *ws_ml, float *ws_o, int *counters, bf16 *out, int Hq,
                                    int Hkv, int max_ctx, float eps, uint32_t *err) {
    static_assert(NW * 2 * (D + 2) * 4 + 2 * ATTN_DECODE_MAX_SPLIT * 4 <= STAGES * STAGE_BYTES,
                  "merge scratch fits in the ring");
    if (!attn_decode_flat_supported(r.B, Hq, Hkv) || n_ctas < 1 || n_ctas > (ATTN_DECODE_MAX_SPLIT - 2) * Hkv)
        return cudaErrorInvalidValue;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    auto kern = r.kv.table ? k_attn_decode_flat<2, true> : k_attn_decode_flat<2, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FLAT_SMEM);
    if (e != cudaSuccess) return e;
    return launch(lc, kern, dim3(n_ctas), dim3(NW * 32), FLAT_SMEM, qkv, r, q_gain, k_gain, rope, k_layer, v_layer,
                  ws_ml, ws_o, counters, out, Hq, Hkv, max_ctx, eps, scale_log2, err);
}

}  // namespace q3
