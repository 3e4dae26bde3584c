// Decode of one row as two kernels per layer: the attention block and the MLP block.
//
// A decoder layer is h' = h + o_proj(attn(RMSNorm(h))), then out = h' + MLP(RMSNorm(h'))
// ("手写Qwen3-0.6B推理", Qwen3DecoderLayer; "第 3 章 前向与生成（代码走读）", 3.2-3.4).  Each RMSNorm
// needs the whole residual row, so a layer has two grid-wide dependencies and no fewer:
// these two kernels, chained with programmatic dependent launch, are the layer.  Everything
// between the two norms runs inside one kernel, with the KV-head groups as thread-block
// clusters:
//
//   k_attn_block   grid (8, Hkv), cluster (8, 1, 1): cluster g = KV head g and its two query
//                  heads ("手写Qwen3-0.6B推理", Attention: the K/V of a group shared by its query
//                  heads).  CTA i of the cluster owns 64 of the group's 512 q/k/v weight rows (32
//                  in shared memory, 32 in registers), the keys [i*per, (i+1)*per) of the row's
//                  sequence, and 128 of the 1024 o_proj output rows.  Norm of h -> its q/k/v
//                  rows -> exchanged through distributed shared memory -> per-head RMSNorm +
//                  rotate-half RoPE (+ the KV-cache write) -> online softmax over its keys -> the
//                  8 partial softmaxes merged through distributed shared memory -> its o_proj
//                  rows, added into the next residual.
//   k_mlp_block    grid of CTA pairs (clusters of 2): CTA c owns act indices [c*NA, c*NA + NA):
//                  the norm of h', its gate/up rows, SwiGLU, and its rows of the transposed down
//                  weight (a split of the down projection over its reduction dimension); a pair
//                  adds its two partial sums through distributed shared memory, then each CTA
//                  adds half of the row into the next residual with vector atomics.
//
// Sized for one CTA of each kernel on an SM together (about 88 + 131 KB of shared memory,
// 168 + 88 registers a thread): each kernel lets the next one launch at its start, the next
// one's CTAs take their place on the SMs as soon as the kernel before the current one leaves,
// bulk-copy their weight rows (and the attention block its cached K/V rows) into shared memory
// and ask L2 for the other kernel's weights of the layer -- all before their dependency wait --
// so HBM streams while the dependency chain runs.  Clusters of 8 (and pairs) because this
// GPU's GPCs hold 15 clusters of 8 but only 7 of 16 at one CTA per SM: all CTAs run in one wave.
//
// Residual buffers: three, rotating.  Layer l's attention block reads R[2l % 3] and adds into
// R[(2l+1) % 3]; its MLP block reads that and adds into R[(2l+2) % 3].  A buffer something adds
// into is zeroed by the kernel before (whose dependency wait guarantees its last reader is
// done): the attention block zeroes the MLP block's output, the MLP block the next attention
// block's, and the embedding kernel the first attention block's.
//
// Every wait on a copy is bounded (mbar_wait_ctx); a CTA whose wait gives up skips its
// arithmetic but still takes part in every cluster barrier, so no CTA of its cluster waits
// forever, and lets its copies land before it exits.

#include <cooperative_groups.h>

#include <algorithm>

#include "kernels.h"

namespace cg = cooperative_groups;

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int AB_CL = 8;        // CTAs per KV-head group (cluster size of the attention block)
constexpr int AB_C = 1024;      // hidden size this path is built for
constexpr int AB_G = 2;         // query heads per KV head
constexpr int AB_ROWS = (AB_G + 2) * D / AB_CL;  // q/k/v weight rows per CTA: 64, in two halves
constexpr int AB_HALF = AB_ROWS / 2;             // rows per pass through the weight buffer: 32
constexpr int AB_OROWS = AB_C / AB_CL;           // o_proj output rows per CTA: 128
constexpr int AB_WARPS = 8;
constexpr int KV_KEYS = 16;     // keys per K/V stage
constexpr int KV_STAGES = 2;
constexpr int MLP_WARPS = 8;

// Shared-memory layout of the attention block for nb rows (byte offsets).
struct AbLayout {
    size_t w, kv, xs, qkvx, qv, knew, vnew, wpart, part, obuf, total;
    __host__ __device__ explicit AbLayout(int nb) {
        w = 128;                                               // 32 q/k/v rows at a time, then o_proj rows
        kv = w + (size_t)AB_HALF * AB_C * 2;                   // [stage][K | V][KV_KEYS][D] bf16
        // once every key is consumed, the stages' space takes the partial softmaxes:
        wpart = kv;                                            // [warps][nb][G][D + 2] per warp
        part = wpart + (size_t)AB_WARPS * nb * AB_G * (D + 2) * 4;  // [nb][G][D + 2] this CTA's
        obuf = part + (size_t)nb * AB_G * (D + 2) * 4;         // [nb][G D] merged attention output
        const size_t stages = (size_t)KV_STAGES * 2 * KV_KEYS * D * 2;
        const size_t partials = obuf + (size_t)nb * AB_G * D * 4 - kv;
        xs = kv + (stages > partials ? stages : partials);    // [nb][C] bf16: RMSNorm(h) * g
        qkvx = xs + (size_t)nb * AB_C * 2;                     // [nb][(G+2) D] fp32: the group's q|k|v
        qv = qkvx + (size_t)nb * (AB_G + 2) * D * 4;           // [nb][G][D] normed, rotated, scaled q
        knew = qv + (size_t)nb * AB_G * D * 4;                 // [nb][D] the new key (bf16-rounded)
        vnew = knew + (size_t)nb * D * 4;                      // [nb][D] the new value (bf16-rounded)
        total = vnew + (size_t)nb * D * 4;
    }
};

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16(x)); }

// A contiguous block of `bytes` (a multiple of 16) as `parts` bulk copies of about equal size,
// issued by lanes 0 .. parts-1 of one warp, completing on `bar` (armed by the caller for the
// total).  A few large copies: each copy takes the issuing lane tens of cycles, so one copy per
// 2 KB row would spend microseconds just issuing.
__device__ __forceinline__ void copy_split(void *dst, const void *src, uint32_t bytes, int parts, uint64_t *bar,
                                           int lane) {
    const uint32_t per = ((bytes / parts) + 15) & ~15u;
    if (lane < parts) {
        const uint32_t off = per * lane;
        if (off < bytes)
            bulk_g2s(static_cast<uint8_t *>(dst) + off, static_cast<const uint8_t *>(src) + off, min(per, bytes - off),
                     bar);
    }
}

__device__ __forceinline__ float exp2_or_zero(float x) { return x == -INFINITY ? 0.0f : exp2f(x); }

// At most 168 registers a thread: with the MLP block's 80, one CTA of each fits an SM's 64 K.
template <int NB>
__global__ void __maxnreg__(168) k_attn_block(AttnBlockParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const AbLayout L(NB);
    cg::cluster_group cluster = cg::this_cluster();
    uint64_t *wbar = reinterpret_cast<uint64_t *>(smem);
    uint64_t *obar = wbar + 1;
    uint64_t *kvfull = wbar + 2;  // [KV_STAGES]
    uint4 *w4 = reinterpret_cast<uint4 *>(smem + L.w);
    bf16 *kvs = reinterpret_cast<bf16 *>(smem + L.kv);
    uint4 *xs4 = reinterpret_cast<uint4 *>(smem + L.xs);
    float *qkvx = reinterpret_cast<float *>(smem + L.qkvx);
    float *qv = reinterpret_cast<float *>(smem + L.qv);
    float *knew = reinterpret_cast<float *>(smem + L.knew);
    float *vnew = reinterpret_cast<float *>(smem + L.vnew);
    float *wpart = reinterpret_cast<float *>(smem + L.wpart);
    float *part = reinterpret_cast<float *>(smem + L.part);
    float *obuf = reinterpret_cast<float *>(smem + L.obuf);

    const int rank = (int)cluster.block_rank();  // == blockIdx.x
    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = p.Hq, Hkv = p.Hkv;
    const int cta = g * AB_CL + rank, n_cta = Hkv * AB_CL;
    const long long lim = wait_limit(p.err);

    // Positions: each row appends at its slot's length, final since the previous step's head
    // (this kernel starts after the kernel before it has passed its own dependency wait).
    int slot[NB], pos[NB], k0[NB], k1[NB], cend[NB], nch[NB];
    int n_chunks = 0;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        slot[b] = __ldcg(p.slots + b);
        pos[b] = __ldcg(p.ctx_len + slot[b]);
        const int per = (pos[b] + AB_CL) / AB_CL;  // ceil((pos + 1) / AB_CL)
        k0[b] = rank * per;
        k1[b] = min(pos[b] + 1, k0[b] + per);
        cend[b] = max(k0[b], min(k1[b], pos[b]));  // cached keys [k0, cend)
        nch[b] = (cend[b] - k0[b] + KV_KEYS - 1) / KV_KEYS;
        n_chunks += nch[b];
    }
    KvMap kv = p.kv;
    // chunk c of the flattened list of every row's chunks: (row b, first key j0, keys n, slot)
    auto chunk = [&](int c, int &b, int &j0, int &n, int &sl) {
        b = 0;
        if (NB > 1 && c >= nch[0]) {
            c -= nch[0];
            b = 1;
        }
        const int kb = b ? k0[NB - 1] : k0[0], ce = b ? cend[NB - 1] : cend[0];
        sl = b ? slot[NB - 1] : slot[0];
        j0 = kb + c * KV_KEYS;
        n = min(KV_KEYS, ce - j0);
    };
    auto issue = [&](int c) {  // chunk c into stage c % KV_STAGES (thread 0)
        int b, j0, n, sl;
        chunk(c, b, j0, n, sl);
        const int st = c % KV_STAGES;
        bf16 *kd = kvs + (size_t)st * 2 * KV_KEYS * D, *vd = kd + KV_KEYS * D;
        mbar_expect_tx(&kvfull[st], 2u * n * D * 2);
        for (int done = 0; done < n;) {  // runs of consecutive rows (a paged block may end inside)
            const int pp = j0 + done;
            const int run = kv.table ? min(n - done, kv.bs - pp % kv.bs) : n - done;
            const size_t row = kv_row(kv, sl, Hkv, g, p.max_ctx, pp);
            bulk_g2s(kd + (size_t)done * D, p.k_layer + row * D, (uint32_t)run * D * 2, &kvfull[st]);
            bulk_g2s(vd + (size_t)done * D, p.v_layer + row * D, (uint32_t)run * D * 2, &kvfull[st]);
            done += run;
        }
    };
    // this CTA's q/k/v rows: the group's rows are [q_2g | q_2g+1 | k_g | v_g], 128 each; local
    // row lr of the group is weight row wrow(lr)
    const int lr0 = rank * AB_ROWS;
    auto wrow = [&](int lr) {
        return lr < AB_G * D ? g * AB_G * D + lr
                             : (lr < (AB_G + 1) * D ? Hq * D + g * D + (lr - AB_G * D)
                                                    : (Hq + Hkv) * D + g * D + (lr - (AB_G + 1) * D));
    };
    if (threadIdx.x == 0) {
        mbar_init(wbar, 1);
        mbar_init(obar, 1);
        for (int s = 0; s < KV_STAGES; ++s) mbar_init(&kvfull[s], 1);
    }
    __syncthreads();
    // The next kernel may launch now: it only reads, before its own dependency wait, what is
    // final already (weights, cached K/V rows, slot lengths), and waits for this grid to
    // complete before it touches anything this kernel writes.
    pdl_trigger();
    if (warp == 0) {
        if (lane == 0) mbar_expect_tx(wbar, AB_HALF * AB_C * 2);
        __syncwarp();
        copy_split(w4, p.wqkv + (size_t)wrow(lr0) * AB_C, AB_HALF * AB_C * 2, 4, wbar, lane);
    } else if (warp == 1 && lane == 0) {
        for (int c = 0; c < min(KV_STAGES, n_chunks); ++c) issue(c);
    } else if (warp == 2 && lane == 0 && p.ahead_gu) {
        // this CTA's share of the layer's MLP weights into L2, for the kernel after this one
        const size_t gu = (size_t)2 * p.I * AB_C * 2, dt = (size_t)p.I * AB_C * 2;
        const size_t s_gu = (gu / n_cta + 15) & ~(size_t)15, s_dt = (dt / n_cta + 15) & ~(size_t)15;
        if ((size_t)cta * s_gu < gu)
            prefetch_l2(reinterpret_cast<const uint8_t *>(p.ahead_gu) + (size_t)cta * s_gu,
                        (uint32_t)min(s_gu, gu - (size_t)cta * s_gu));
        if ((size_t)cta * s_dt < dt)
            prefetch_l2(reinterpret_cast<const uint8_t *>(p.ahead_dt) + (size_t)cta * s_dt,
                        (uint32_t)min(s_dt, dt - (size_t)cta * s_dt));
    }
    // the second half of this CTA's q/k/v rows goes to registers: warp w, rows 4w .. 4w+3 of it,
    // the lane's four 16-byte pieces of each (64 registers)
    uint4 wreg[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const bf16 *src = p.wqkv + (size_t)wrow(lr0 + AB_HALF + warp * 4 + r) * AB_C;
#pragma unroll
        for (int i = 0; i < 4; ++i) wreg[r][i] = ld_stream(src + (i * 32 + lane) * 8);
    }
    // constants: the input norm's gains (warps 0 .. NB-1, the lane's 32 elements) and those of
    // the per-head norm + RoPE phase (warp (b, h), lane's dims lane + 32 k)
    float4 gin[8];
    if (warp < NB) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            gin[2 * i] = __ldg(reinterpret_cast<const float4 *>(p.g_in) + i * 64 + lane * 2);
            gin[2 * i + 1] = __ldg(reinterpret_cast<const float4 *>(p.g_in) + i * 64 + lane * 2 + 1);
        }
    }
    float gain4[4] = {1.0f, 1.0f, 1.0f, 1.0f};
    float2 cs0 = make_float2(1.0f, 0.0f), cs1 = make_float2(1.0f, 0.0f);
    if (warp < NB * (AB_G + 2)) {
        const int b = warp / (AB_G + 2), h = warp % (AB_G + 2);
        const int ps = b ? pos[NB - 1] : pos[0];
        if (h <= AB_G) {
            const float *gn = h < AB_G ? p.g_q : p.g_k;
#pragma unroll
            for (int k = 0; k < 4; ++k) gain4[k] = __ldg(gn + lane + 32 * k);
            cs0 = __ldg(p.rope + (size_t)ps * (D / 2) + lane);
            cs1 = __ldg(p.rope + (size_t)ps * (D / 2) + lane + 32);
        }
    }
    // every CTA of the cluster must be running before any writes into another's memory: arrive
    // now, wait right before the first such write
    cluster.barrier_arrive();
    pdl_wait();

    // residual: this CTA's share of h into the output row (other CTAs add their o_proj rows);
    // the MLP block's output buffer cleared
    if (warp == AB_WARPS - 1) {  // the last warp, so that it overlaps the norm of warps 0 .. NB-1
        const int per = (NB * AB_C + n_cta - 1) / n_cta;
        for (int i = lane; i < per; i += 32) {
            const int e = cta * per + i;
            if (e < NB * AB_C) {
                atomicAdd(p.h_out + e, __ldcg(p.h_in + e));
                p.zero_next[e] = 0.0f;
            }
        }
    }
    // RMSNorm of each row into shared memory (bf16 operand): warp b, lane holds 32 elements
    // (8 consecutive at lane*8 + 256 i)
    if (warp < NB) {
        const float4 *hr = reinterpret_cast<const float4 *>(p.h_in + (size_t)warp * AB_C);
        float4 v[8];
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __ldcg(hr + i * 64 + lane * 2);
            v[2 * i + 1] = __ldcg(hr + i * 64 + lane * 2 + 1);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        const float inv = rsqrtf(warp_sum(ss) / (float)AB_C + p.eps);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 ga = gin[2 * i], gb = gin[2 * i + 1];
            const float4 a = v[2 * i], c = v[2 * i + 1];
            uint4 o;
            o.x = pack_bf16x2(a.x * inv * ga.x, a.y * inv * ga.y);
            o.y = pack_bf16x2(a.z * inv * ga.z, a.w * inv * ga.w);
            o.z = pack_bf16x2(c.x * inv * gb.x, c.y * inv * gb.y);
            o.w = pack_bf16x2(c.z * inv * gb.z, c.w * inv * gb.w);
            xs4[warp * (AB_C / 8) + i * 32 + lane] = o;
        }
    }
    __syncthreads();
    cluster.barrier_wait();  // (0) every CTA of the cluster runs
    bool ok = __syncthreads_and(mbar_wait_ctx(wbar, 0, p.err, lim));
    // q/k/v rows: warp w takes rows 4w .. 4w+3 of each half (the first half from shared memory,
    // the second from registers); every lane ends with the sums, and lanes 0..7 store them into
    // the exchange buffer of CTA `lane` of the cluster
    auto qkv_rows = [&](int half, auto wget) {
        float acc[4][NB];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[r][b] = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 xv[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) xv[b] = xs4[b * (AB_C / 8) + i * 32 + lane];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint4 wv = wget(r, i);
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[r][b] = dot8(wv, xv[b], acc[r][b]);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[r][b] = warp_sum(acc[r][b]);
        if (lane < AB_CL) {
            float *dst = cluster.map_shared_rank(qkvx, lane);
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int r = 0; r < 4; ++r) dst[b * (AB_G + 2) * D + lr0 + half * AB_HALF + warp * 4 + r] = acc[r][b];
        }
    };
    if (ok) qkv_rows(0, [&](int r, int i) { return w4[(size_t)(warp * 4 + r) * (AB_C / 8) + i * 32 + lane]; });
    __syncthreads();  // every warp is done with the buffer: this CTA's o_proj rows go in
    if (warp == 0) {
        if (lane == 0) mbar_expect_tx(obar, AB_OROWS * AB_G * D * 2);
        __syncwarp();
        copy_split(w4, p.wog + ((size_t)g * AB_C + (size_t)rank * AB_OROWS) * AB_G * D, AB_OROWS * AB_G * D * 2, 4,
                   obar, lane);
    }
    if (ok) qkv_rows(1, [&](int r, int i) { return wreg[r][i]; });
    cluster.sync();  // (1) every CTA's q/k/v rows have landed in every CTA

    // per-head RMSNorm + rotate-half RoPE: warp (b, h) for h in q_0, q_1, k, v; lane holds
    // dims lane, lane+32, lane+64, lane+96, so both RoPE pairs (i, i+64) are in-lane
    if (warp < NB * (AB_G + 2)) {
        const int b = warp / (AB_G + 2), h = warp % (AB_G + 2);
        const int sl = b ? slot[NB - 1] : slot[0], ps = b ? pos[NB - 1] : pos[0];
        const float *src = qkvx + b * (AB_G + 2) * D + h * D;
        float x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = src[lane + 32 * k];
        if (h <= AB_G) {  // q heads and k: RMSNorm, then rotate
            float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
            const float inv = rsqrtf(warp_sum(ss) * (1.0f / D) + p.eps);
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] *= inv * gain4[k];
            const float2 c0 = cs0, c1 = cs1;
            const float r0 = x[0] * c0.x - x[2] * c0.y, r2 = x[2] * c0.x + x[0] * c0.y;
            const float r1 = x[1] * c1.x - x[3] * c1.y, r3 = x[3] * c1.x + x[1] * c1.y;
            x[0] = r0; x[1] = r1; x[2] = r2; x[3] = r3;
        }
        if (h < AB_G) {
#pragma unroll
            for (int k = 0; k < 4; ++k) qv[(b * AB_G + h) * D + lane + 32 * k] = x[k] * p.scale_log2;
        } else {
            float *dst = h == AB_G ? knew : vnew;
            const size_t row = kv_row(kv, sl, Hkv, g, p.max_ctx, ps);
            bf16 *cache = h == AB_G ? p.k_layer : p.v_layer;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bf16 r = __float2bfloat16(x[k]);
                dst[b * D + lane + 32 * k] = __bfloat162float(r);
                if (rank == 0 && ok) cache[row * D + lane + 32 * k] = r;
            }
        }
    }
    __syncthreads();

    // online softmax over this CTA's keys: warp w takes keys w, w + 8 of each 16-key chunk
    float m[NB][AB_G], l[NB][AB_G], acc[NB][AB_G][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int gi = 0; gi < AB_G; ++gi) {
            m[b][gi] = -INFINITY;
            l[b][gi] = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[b][gi][k] = 0.0f;
        }
    auto attend = [&](int b, const float *kf, const float *vf) {  // one key, lane's 4 dims
#pragma unroll
        for (int gi = 0; gi < AB_G; ++gi) {
            const float *q = qv + (b * AB_G + gi) * D;
            float s = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) s = fmaf(q[lane + 32 * k], kf[k], s);
            s = warp_sum(s);
            const float mn = fmaxf(m[b][gi], s);
            const float c = exp2_or_zero(m[b][gi] - mn), e = exp2f(s - mn);
            l[b][gi] = l[b][gi] * c + e;
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[b][gi][k] = fmaf(e, vf[k], acc[b][gi][k] * c);
            m[b][gi] = mn;
        }
    };
    int stop = 0;
    for (int c = 0; c < n_chunks; ++c) {
        const int st = c % KV_STAGES;
        stop = c;
        const bool late = !mbar_wait_ctx(&kvfull[st], (c / KV_STAGES) & 1, p.err, lim);
        if (__syncthreads_or(late)) {
            ok = false;
            break;
        }
        int b, j0, n, sl;
        chunk(c, b, j0, n, sl);
        const bf16 *ks = kvs + (size_t)st * 2 * KV_KEYS * D, *vs = ks + KV_KEYS * D;
        // NB is at most 2: select the row's registers with a uniform branch
        for (int j = warp; j < n; j += AB_WARPS) {
            float kf[4], vf[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                kf[k] = __bfloat162float(ks[j * D + lane + 32 * k]);
                vf[k] = __bfloat162float(vs[j * D + lane + 32 * k]);
            }
#pragma unroll
            for (int bb = 0; bb < NB; ++bb)
                if (bb == b) attend(bb, kf, vf);
        }
        __syncthreads();  // stage st is free
        if (threadIdx.x == 0 && c + KV_STAGES < n_chunks) issue(c + KV_STAGES);
    }
    if (ok && warp == 0) {  // the new key, for the CTA whose range holds it
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (k0[b] <= pos[b] && pos[b] < k1[b]) {
                float kf[4], vf[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    kf[k] = knew[b * D + lane + 32 * k];
                    vf[k] = vnew[b * D + lane + 32 * k];
                }
                attend(b, kf, vf);
            }
        }
    }
    // the 8 warps' partials -> this CTA's partial (m, l, acc[D]) per (row, head)
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int gi = 0; gi < AB_G; ++gi) {
            float *wp = wpart + ((size_t)(warp * NB + b) * AB_G + gi) * (D + 2);
            if (lane == 0) {
                wp[D] = m[b][gi];
                wp[D + 1] = l[b][gi];
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) wp[lane + 32 * k] = acc[b][gi][k];
        }
    __syncthreads();
    for (int o = threadIdx.x; o < NB * AB_G * D; o += blockDim.x) {
        const int bg = o / D, d = o % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < AB_WARPS; ++w) mx = fmaxf(mx, wpart[((size_t)w * NB * AB_G + bg) * (D + 2) + D]);
        float ls = 0.0f, a = 0.0f;
#pragma unroll
        for (int w = 0; w < AB_WARPS; ++w) {
            const float *wp = wpart + ((size_t)w * NB * AB_G + bg) * (D + 2);
            const float c = wp[D] == -INFINITY ? 0.0f : exp2f(wp[D] - mx);  // a warp without keys adds nothing
            ls += wp[D + 1] * c;
            a += wp[d] * c;
        }
        part[bg * (D + 2) + d] = a;
        if (d == 0) {
            part[bg * (D + 2) + D] = mx;
            part[bg * (D + 2) + D + 1] = ls;
        }
    }
    cluster.sync();  // (2) every CTA's partial is ready

    // merge the 16 partials: o = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i
    for (int o = threadIdx.x; o < NB * AB_G * D; o += blockDim.x) {
        const int bg = o / D, d = o % D;
        float mi[AB_CL], li[AB_CL], ai[AB_CL];
#pragma unroll
        for (int r = 0; r < AB_CL; ++r) {
            const float *rp = cluster.map_shared_rank(part, r) + bg * (D + 2);
            mi[r] = rp[D];
            li[r] = rp[D + 1];
            ai[r] = rp[d];
        }
        float mx = -INFINITY;
#pragma unroll
        for (int r = 0; r < AB_CL; ++r) mx = fmaxf(mx, mi[r]);
        float ls = 0.0f, a = 0.0f;
#pragma unroll
        for (int r = 0; r < AB_CL; ++r) {
            const float c = mi[r] == -INFINITY ? 0.0f : exp2f(mi[r] - mx);  // a CTA without keys adds nothing
            ls += li[r] * c;
            a += ai[r] * c;
        }
        obuf[o] = a / ls;
    }
    cluster.barrier_arrive();  // (3) this CTA reads no other CTA's memory any more
    __syncthreads();
    ok = __syncthreads_and(ok && mbar_wait_ctx(obar, 0, p.err, lim));

    // o_proj: warp w takes output rows 16w .. 16w+15 of this CTA's 128; lane holds 8 of the 256
    // columns of the group (its two heads' outputs)
    if (ok) {
        float4 o0[NB], o1[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            o0[b] = reinterpret_cast<const float4 *>(obuf + b * AB_G * D)[lane * 2];
            o1[b] = reinterpret_cast<const float4 *>(obuf + b * AB_G * D)[lane * 2 + 1];
        }
        float acc2[16][NB];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const uint4 wv = w4[(size_t)(warp * 16 + r) * (AB_G * D / 8) + lane];
            const __nv_bfloat162 *pw = reinterpret_cast<const __nv_bfloat162 *>(&wv);
            const float2 w0 = __bfloat1622float2(pw[0]), w1 = __bfloat1622float2(pw[1]);
            const float2 w2 = __bfloat1622float2(pw[2]), w3 = __bfloat1622float2(pw[3]);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float s = o0[b].x * w0.x;
                s = fmaf(o0[b].y, w0.y, s);
                s = fmaf(o0[b].z, w1.x, s);
                s = fmaf(o0[b].w, w1.y, s);
                s = fmaf(o1[b].x, w2.x, s);
                s = fmaf(o1[b].y, w2.y, s);
                s = fmaf(o1[b].z, w3.x, s);
                s = fmaf(o1[b].w, w3.y, s);
                acc2[r][b] = s;
            }
        }
#pragma unroll
        for (int r = 0; r < 16; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc2[r][b] = warp_sum(acc2[r][b]);
        if (lane < 16 * NB) {
            const int r = lane % 16, b = lane / 16;
            float v = 0.0f;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
#pragma unroll
                for (int bb = 0; bb < NB; ++bb)
                    if (rr == r && bb == b) v = acc2[rr][bb];
            atomicAdd(p.h_out + (size_t)b * AB_C + rank * AB_OROWS + warp * 16 + r, v);
        }
    }
    if (!ok && threadIdx.x == 0) {  // let every copy this CTA issued land before it exits
        mbar_wait_bounded(wbar, 0, nullptr);
        mbar_wait_bounded(obar, 0, nullptr);
        for (int c = stop; c < min(stop + KV_STAGES, n_chunks); ++c)
            mbar_wait_bounded(&kvfull[c % KV_STAGES], (c / KV_STAGES) & 1, nullptr);
    }
    cluster.barrier_wait();  // (3) no CTA leaves while another may read its partial
}

template <int NB>
__global__ void __launch_bounds__(MLP_WARPS * 32, 1) k_mlp_block(MlpBlockParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int KV = 4;
    constexpr int C = KV * 256;
    constexpr int M = NB;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int NA = p.NA;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint4 *wgu = reinterpret_cast<uint4 *>(smem + 128);     // [2*NA][C/8]; later the partial sums
    float *part = reinterpret_cast<float *>(wgu);           // [M][C], once the gate/up rows are done
    uint4 *wd = wgu + (size_t)2 * NA * (C / 8);             // [NA][C/8]
    uint4 *xs = wd + (size_t)NA * (C / 8);                  // [M][C/8]
    float *act = reinterpret_cast<float *>(xs + (size_t)M * (C / 8));  // [M][NA]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int a0 = blockIdx.x * NA;
    const int na = max(0, min(NA, p.I - a0));
    const long long lim = wait_limit(p.err);
    if (threadIdx.x == 0) mbar_init(bar, 1);
    __syncthreads();
    pdl_trigger();  // the next attention block may launch (its early reads are final already)
    if (warp == 0) {
        if (lane == 0) mbar_expect_tx(bar, (uint32_t)na * 3 * C * 2);
        __syncwarp();
        if (na > 0) {
            copy_split(wgu, p.wgu + (size_t)2 * a0 * C, (uint32_t)na * 2 * C * 2, 4, bar, lane);
            if (lane >= 4) copy_split(wd, p.wdt + (size_t)a0 * C, (uint32_t)na * C * 2, 2, bar, lane - 4);
        }
    } else if (warp == 1 && lane == 0 && p.ahead_qkv) {
        // this CTA's share of the next layer's attention weights into L2
        const size_t qkv = (size_t)p.qkv_rows * C * 2, og = (size_t)p.og_cols * C * 2;
        const size_t s_q = (qkv / gridDim.x + 15) & ~(size_t)15, s_o = (og / gridDim.x + 15) & ~(size_t)15;
        if ((size_t)blockIdx.x * s_q < qkv)
            prefetch_l2(reinterpret_cast<const uint8_t *>(p.ahead_qkv) + (size_t)blockIdx.x * s_q,
                        (uint32_t)min(s_q, qkv - (size_t)blockIdx.x * s_q));
        if ((size_t)blockIdx.x * s_o < og)
            prefetch_l2(reinterpret_cast<const uint8_t *>(p.ahead_og) + (size_t)blockIdx.x * s_o,
                        (uint32_t)min(s_o, og - (size_t)blockIdx.x * s_o));
    }
    float4 gpost[2 * KV];  // the post-attention norm's gains (warps 0 .. M-1), read before the wait
    if (warp < M) {
#pragma unroll
        for (int i = 0; i < 2 * KV; ++i) gpost[i] = __ldg(reinterpret_cast<const float4 *>(p.gain) + i * 32 + lane);
    }
    pdl_wait();
    if (warp == MLP_WARPS - 1) {  // residual share into the output; the next attention block's output cleared
        const int per = (M * C + gridDim.x - 1) / gridDim.x;
        for (int i = lane; i < per; i += 32) {
            const int e = blockIdx.x * per + i;
            if (e < M * C) {
                atomicAdd(p.h_out + e, __ldcg(p.h_in + e));
                p.zero_next[e] = 0.0f;
            }
        }
    }
    if (warp < M) {  // m = RMSNorm(h') * g_post, bf16
        const float4 *hr = reinterpret_cast<const float4 *>(p.h_in + (size_t)warp * C);
        float4 v[2 * KV];
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < 2 * KV; ++i) {
            v[i] = __ldcg(hr + i * 32 + lane);
            ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        }
        const float inv = rsqrtf(warp_sum(ss) / (float)C + p.eps);
        uint2 *dst = reinterpret_cast<uint2 *>(xs + (size_t)warp * (C / 8));
#pragma unroll
        for (int i = 0; i < 2 * KV; ++i) {
            const float4 gv = gpost[i];
            uint2 o;
            o.x = pack_bf16x2(v[i].x * inv * gv.x, v[i].y * inv * gv.y);
            o.y = pack_bf16x2(v[i].z * inv * gv.z, v[i].w * inv * gv.w);
            dst[i * 32 + lane] = o;
        }
    }
    __syncthreads();
    const bool ok = __syncthreads_and(mbar_wait_ctx(bar, 0, p.err, lim));
    if (ok) {
        for (int j = warp; j < na; j += MLP_WARPS) {  // gate/up pairs -> act (bf16-rounded)
            float gs[M], us[M];
#pragma unroll
            for (int b = 0; b < M; ++b) gs[b] = us[b] = 0.0f;
#pragma unroll
            for (int i = 0; i < KV; ++i) {
                const uint4 wg = wgu[(size_t)(2 * j) * (C / 8) + i * 32 + lane];
                const uint4 wu = wgu[(size_t)(2 * j + 1) * (C / 8) + i * 32 + lane];
#pragma unroll
                for (int b = 0; b < M; ++b) {
                    const uint4 x = xs[b * (C / 8) + i * 32 + lane];
                    gs[b] = dot8(wg, x, gs[b]);
                    us[b] = dot8(wu, x, us[b]);
                }
            }
#pragma unroll
            for (int b = 0; b < M; ++b) {
                const float gg = warp_sum(gs[b]), uu = warp_sum(us[b]);
                if (lane == 0) act[b * NA + j] = round_bf16(silu(gg) * uu);
            }
        }
    }
    __syncthreads();  // the gate/up rows are done: their space takes the partial sums
    // this CTA's share of the down projection (its act indices), 4 outputs per thread; the two
    // CTAs of a cluster add their partial sums through distributed shared memory and each adds
    // half of the row into the next residual with vector atomics (half the atomics)
#pragma unroll
    for (int b = 0; b < M; ++b) {
        const int n0 = threadIdx.x * 4;
        float4 a4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (ok) {
            for (int j = 0; j < na; ++j) {
                const float a = act[b * NA + j];
                const uint2 w = *reinterpret_cast<const uint2 *>(reinterpret_cast<const bf16 *>(wd) + (size_t)j * C + n0);
                const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
                const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
                a4.x = fmaf(a, w01.x, a4.x);
                a4.y = fmaf(a, w01.y, a4.y);
                a4.z = fmaf(a, w23.x, a4.z);
                a4.w = fmaf(a, w23.y, a4.w);
            }
        }
        reinterpret_cast<float4 *>(part + (size_t)b * C)[threadIdx.x] = a4;
    }
    cluster.sync();  // both partials are in place
    {
        const float *peer = cluster.map_shared_rank(part, rank ^ 1);
        for (int i = threadIdx.x; i < M * (C / 2) / 4; i += blockDim.x) {
            const int b = i / ((C / 2) / 4), n = rank * (C / 2) + (i % ((C / 2) / 4)) * 4;
            const float4 u = *reinterpret_cast<const float4 *>(part + (size_t)b * C + n);
            const float4 v = *reinterpret_cast<const float4 *>(peer + (size_t)b * C + n);
            atomicAdd(reinterpret_cast<float4 *>(p.h_out + (size_t)b * C + n),
                      make_float4(u.x + v.x, u.y + v.y, u.z + v.z, u.w + v.w));
        }
    }
    cluster.barrier_arrive();  // done reading the peer's partial sums
    if (!ok) mbar_wait_bounded(bar, 0, nullptr);  // let the copies land before the CTA exits
    cluster.barrier_wait();    // the peer is done reading ours
}

template <int NB>
cudaError_t run_attn_block(const Launch &lc, const AttnBlockParams &p) {
    const size_t smem = attn_block_smem(NB);
    auto kern = k_attn_block<NB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    return launch_cluster(lc, kern, dim3(AB_CL, p.Hkv), dim3(AB_WARPS * 32), smem, dim3(AB_CL, 1, 1), p);
}

}  // namespace

size_t attn_block_smem(int B) { return AbLayout(B).total; }

int mlp_block_na(int I, int num_sms) { return (I + num_sms - 1) / num_sms; }

// barrier, gate/up rows, down rows, m [B][C] bf16, act [B][NA]
size_t mlp_block_smem(int B, int C, int I, int num_sms) {
    const int NA = mlp_block_na(I, num_sms);
    return 128 + (size_t)NA * 3 * C * 2 + (size_t)B * C * 2 + (size_t)B * NA * 4;
}

// How many 16-CTA clusters of the attention block the device can hold at once (0 if none).
template <int NB>
int attn_block_max_clusters(int Hkv) {
    static int cached = -1;
    if (cached >= 0) return cached;
    auto kern = k_attn_block<NB>;
    const size_t smem = attn_block_smem(NB);
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(AB_CL, Hkv);
        cfg.blockDim = dim3(AB_WARPS * 32);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = AB_CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();  // a refused query leaves no error behind
    cached = n;
    return n;
}

bool decode_block_supported(int B, int C, int Hq, int Hkv, int head_dim, int I, int num_sms) {
    if (B < 1 || B > 2 || C != AB_C || head_dim != D || Hq != AB_G * Hkv || Hkv < 1 || Hkv > 64) return false;
    if (I % 256 || I > 4096) return false;

    // one CTA of each kernel fits an SM together: shared memory (228 KB, 1 KB reserved per CTA)
    // and registers (64 K)
    if (attn_block_smem(B) + mlp_block_smem(B, C, I, num_sms) + 2048 > 228 * 1024) return false;
    cudaFuncAttributes fa, fm;
    if (cudaFuncGetAttributes(&fa, B == 1 ? k_attn_block<1> : k_attn_block<2>) != cudaSuccess ||
        cudaFuncGetAttributes(&fm, B == 1 ? k_mlp_block<1> : k_mlp_block<2>) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    auto regs = [](int per_thread, int threads) { return ((per_thread + 7) / 8 * 8) * threads; };
    if (regs(fa.numRegs, AB_WARPS * 32) + regs(fm.numRegs, MLP_WARPS * 32) > 65536) return false;
    // and the device holds a cluster per KV head at once
    return (B == 1 ? attn_block_max_clusters<1>(Hkv) : attn_block_max_clusters<2>(Hkv)) >= Hkv;
}

cudaError_t launch_attn_block(const Launch &lc, const AttnBlockParams &p) {
    if (p.B == 1) return run_attn_block<1>(lc, p);
    if (p.B == 2) return run_attn_block<2>(lc, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_mlp_block(const Launch &lc, const MlpBlockParams &p0) {
    MlpBlockParams p = p0;
    p.NA = mlp_block_na(p.I, lc.num_sms);
    if (p.C != 1024 || p.B < 1 || p.B > 2) return cudaErrorInvalidValue;
    const int grid = ((p.I + p.NA - 1) / p.NA + 1) & ~1;  // pairs of CTAs
    const size_t smem = mlp_block_smem(p.B, p.C, p.I, lc.num_sms);
    auto kern = p.B == 1 ? k_mlp_block<1> : k_mlp_block<2>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_cluster(lc, kern, dim3(grid), dim3(MLP_WARPS * 32), smem, dim3(2, 1, 1), p);
}

}  // namespace q3
