// One decode step of the whole model in a single persistent kernel, for up to 8 sequences.
//
// The step computes what the per-kernel decode chain computes ("手写Qwen3-0.6B推理",
// Qwen3DecoderLayer / Qwen3Model: embedding, per layer RMSNorm -> q/k/v -> per-head q/k
// RMSNorm -> RoPE -> attention over the cache -> o_proj + residual -> RMSNorm -> SwiGLU MLP
// + residual, final RMSNorm, tied lm_head; "第 3 章", 4.3: greedy argmax), with the same
// roundings: bf16 GEMV operands, fp32 accumulation and residual stream.
//
// Layout of the work: one CTA per SM, launched cooperatively so that all CTAs are resident.
// The CTAs form HKV groups of gsz = grid / HKV (19 on a 152-SM GB300), one per KV head g.
// A layer has three stages:
//   A  group g computes the 512 rows of q/k/v that belong to KV head g (its two query heads,
//      the key and the value head), gsz-way split by rows;
//   B  after a wait on its own group only, every CTA of group g computes the attention of KV
//      head g (both query heads, every sequence) itself -- the K/V rows come from L2 after the
//      first CTA has read them -- and applies its block of output rows of o_proj restricted to
//      the group's 256 attention columns; the partial sums of the HKV groups are added into
//      the residual with atomics, so o_proj needs no stage of its own;
//   C  after a wait on all CTAs: RMSNorm, gate/up and SwiGLU of this CTA's block of the
//      intermediate activations, then its slice of the down projection (split along the
//      reduction dimension) added into the next residual with vector atomics.
// The final stage is the RMSNorm of the last residual and the tied lm_head over this CTA's
// block of the vocabulary, then a partial argmax per sequence.
//
// The residual stream rotates through three fp32 buffers: h (input of the layer), P (h plus
// the attention output; zero before stage B) and Q (P plus the MLP output, zero before stage
// C; the next layer's h).  Each CTA zeroes its slice of the buffer that a later stage
// accumulates into at a point where every earlier reader has finished.
//
// Weights do not depend on the activations, so one producer warp streams every weight row
// (and every cached K/V chunk) this CTA will use, in the order it will use them, through a
// ring of 16 KB shared-memory slots filled by bulk asynchronous copies.  It runs ahead across
// stage and layer boundaries, limited only by free slots, so HBM keeps streaming while the
// eight consumer warps wait on a dependency.
//
// Dependencies between CTAs are arrival counters, added to with release semantics after a
// CTA barrier and polled (acquire) by one thread per CTA: one counter for the stages that
// wait on every CTA (no CTA can finish such a stage before all CTAs have arrived at the
// previous one, so the count is exact) and one per group for stage B.  The CTA that finishes
// the step last resets them to zero.  Data written by other CTAs is read with ld.global.cg
// (L2), never from a possibly stale L1 line.
//
// Every wait is bounded (about a second of SM clocks); a wait that gives up sets ERR_TIMEOUT
// in the error word, which every other wait also watches and then returns at once.  A CTA
// that saw a failed wait still runs the rest of its step (on whatever its buffers hold) so
// that its warps pass the same barriers, then skips the step's final bookkeeping.  After a
// timeout the context's step state (counters) is not consistent any more.

#include <algorithm>

#include "kernels.h"

namespace q3 {

namespace {

constexpr int C = 1024, D = 128, HQ = 16, HKV = 8, G = HQ / HKV, GD = G * D, QD = HQ * D;
constexpr int NQKV = (HQ + 2 * HKV) * D;
constexpr int NW = 8;                    // consumer warps
constexpr int THREADS = (NW + 1) * 32;   // + the producer warp
constexpr int SLOT = 16384, NSLOT = 10;
constexpr int PIECE = SLOT;              // bytes per bulk copy (a slot may be filled by several copies)
constexpr int CHUNK = 32;                // keys per attention slot: K rows at 0, V rows at SLOT/2
constexpr int B_MAX = 8, NA_MAX = 32, OROWS_MAX = 64;
constexpr long long WAIT_LIMIT = 1ll << 31;

struct __align__(128) Smem {
    uint8_t ring[NSLOT][SLOT];
    bf16 x[B_MAX * C];                  // stage input (normed residual or attention of the group), bf16
    float gu[B_MAX][2 * NA_MAX];        // gate/up dot products of this CTA's rows
    float act[B_MAX][NA_MAX];           // silu(gate) * up, rounded to bf16
    float red_o[NW][G][D];              // attention: cross-warp merge
    float red_ml[NW][G][2];
    float s_new[2][D];                  // new key (bf16-rounded) and value of the sequence
    float gqk[2][D];                    // q_norm and k_norm gains of the layer
    float2 cs[B_MAX][D / 2];            // RoPE (cos, sin) at each sequence's position
    float hres[B_MAX][OROWS_MAX];       // group 0: the residual at this CTA's o_proj rows
    float best_v[NW][B_MAX];
    int best_i[NW][B_MAX];
    uint64_t full[NSLOT], empty[NSLOT];
    int pos[B_MAX], slot[B_MAX], tok[B_MAX];
    int last, dead;
};

struct Args {
    int L, I, V, max_ctx, B;
    float eps, scale_log2;
    const uint8_t *layers;
    size_t layer_bytes, o_wqkv, o_wog, o_wgu, o_wdownT, o_gin, o_gpost, o_gq, o_gk;
    const bf16 *embed;
    const float *g_final;
    const float2 *rope;
    bf16 *kcache, *vcache;
    size_t kv_layer_elems;              // elements of one layer's K (or V) cache
    const int32_t *tokens, *slots;
    int32_t *ctx_len, *next_tok;
    float *logits, *dump;
    float *res[3], *qkv, *part_val;
    int32_t *part_idx;
    uint32_t *arrive, *grp, *counter, *err;
};

__device__ __forceinline__ int rb(int c, int n, int parts) { return (int)(((long long)c * n) / parts); }

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ bool timed_out(const uint32_t *err) {
    return (*reinterpret_cast<const volatile uint32_t *>(err) & ERR_TIMEOUT) != 0;
}
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void red_add(float *p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_v4(float *p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16(x)); }
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// Bounded mbarrier wait that also gives up once another CTA has timed out.
__device__ bool ring_wait(uint64_t *bar, uint32_t phase, uint32_t *err) {
    const long long t0 = clock64();
    for (int it = 0;; ++it) {
        if (mbar_try_wait(bar, phase)) return true;
        if ((it & 63) == 63 && (clock64() - t0 > WAIT_LIMIT || timed_out(err))) {
            atomicOr(err, ERR_TIMEOUT);
            return false;
        }
    }
}

// One thread: until *counter >= target.  False (and ERR_TIMEOUT) if it gives up.
__device__ bool wait_count(const uint32_t *counter, uint32_t target, uint32_t *err) {
    const long long t0 = clock64();
    while (ld_acquire(counter) < target) {
        if (clock64() - t0 > WAIT_LIMIT || timed_out(err)) {
            atomicOr(err, ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// The work of one CTA.
struct Part {
    int g, gi, gsz;        // KV head group, index in the group, group size (g < 0: no group work)
    int qa, qb;            // this CTA's rows of its group's 512 q/k/v rows ("virtual" rows)
    int oa, ob;            // o_proj output rows of this CTA within its group
    int ja, jb;            // intermediate activations (MLP)
    int ra, rb_;           // slice of the residual rows this CTA zeroes / adds
    int va, vb;            // vocabulary rows
};

__device__ __forceinline__ Part make_part(const Args &a, int cta, int grid) {
    Part p;
    p.gsz = grid / HKV;
    p.g = p.gsz > 0 && cta < HKV * p.gsz ? cta / p.gsz : -1;
    p.gi = p.g >= 0 ? cta % p.gsz : 0;
    p.qa = p.g >= 0 ? rb(p.gi, 2 * GD, p.gsz) : 0;
    p.qb = p.g >= 0 ? rb(p.gi + 1, 2 * GD, p.gsz) : 0;
    p.oa = p.g >= 0 ? rb(p.gi, C, p.gsz) : 0;
    p.ob = p.g >= 0 ? rb(p.gi + 1, C, p.gsz) : 0;
    p.ja = rb(cta, a.I, grid);
    p.jb = rb(cta + 1, a.I, grid);
    p.ra = rb(cta, C, grid);
    p.rb_ = rb(cta + 1, C, grid);
    p.va = rb(cta, a.V, grid);
    p.vb = rb(cta + 1, a.V, grid);
    return p;
}

// Row of W_qkv behind virtual row v of group g: its two query heads, then its key and value.
__device__ __forceinline__ int qkv_row(int g, int v) {
    return v < GD ? g * GD + v : (v < GD + D ? QD + g * D + (v - GD) : QD + HKV * D + g * D + (v - GD - D));
}
// End (exclusive) of the run of consecutive W_qkv rows that starts at virtual row v.
__device__ __forceinline__ int qkv_run_end(int v, int vb) { return min(vb, v < GD ? GD : (v < GD + D ? GD + D : 2 * GD)); }

// residual buffers of layer l: h (input), P (after attention), Q (after the MLP = next h)
__device__ __forceinline__ float *res_h(const Args &a, int l) { return a.res[(3 - l % 3) % 3]; }
__device__ __forceinline__ float *res_p(const Args &a, int l) { return a.res[(4 - l % 3) % 3]; }

// ---- producer: the step's slots in consumption order ----------------------------------------

struct Producer {
    Smem &s;
    uint32_t *err;
    uint32_t k = 0;  // slots issued
    bool ok = true;

    __device__ Producer(Smem &sm, uint32_t *e) : s(sm), err(e) {}

    __device__ uint8_t *acquire(uint32_t bytes) {
        const int p = k % NSLOT;
        const uint32_t n = k / NSLOT;
        // (no check of the error word per slot: a global load each time would throttle the
        // stream; a wait that runs long watches it)
        if (n > 0 && !ring_wait(&s.empty[p], (n - 1) & 1, err)) {
            ok = false;
            return nullptr;
        }
        mbar_expect_tx(&s.full[p], bytes);
        return s.ring[p];
    }
    // bytes [0, n) of src into dst as copies of at most PIECE bytes
    __device__ void copy(uint8_t *dst, const uint8_t *src, uint32_t n) {
        for (uint32_t o = 0; o < n; o += PIECE) bulk_g2s(dst + o, src + o, min((uint32_t)PIECE, n - o), &s.full[k % NSLOT]);
    }
    // rows [r0, r1) of a row-major matrix with `row_bytes` per row, SLOT / row_bytes per slot
    __device__ void rows(const void *W, int r0, int r1, int row_bytes) {
        const int per = SLOT / row_bytes;
        for (int r = r0; r < r1 && ok; r += per) {
            const int n = min(per, r1 - r);
            uint8_t *dst = acquire((uint32_t)n * row_bytes);
            if (!dst) return;
            copy(dst, static_cast<const uint8_t *>(W) + (size_t)r * row_bytes, (uint32_t)n * row_bytes);
            ++k;
        }
    }
    // cached keys [j0, j1) of one (slot, head): K rows then V rows per slot
    __device__ void kv(const bf16 *kc, const bf16 *vc, int j0, int j1) {
        for (int j = j0; j < j1 && ok; j += CHUNK) {
            const int n = min(CHUNK, j1 - j);
            uint8_t *dst = acquire((uint32_t)n * D * 2 * 2);
            if (!dst) return;
            copy(dst, reinterpret_cast<const uint8_t *>(kc + (size_t)j * D), (uint32_t)n * D * 2);
            copy(dst + SLOT / 2, reinterpret_cast<const uint8_t *>(vc + (size_t)j * D), (uint32_t)n * D * 2);
            ++k;
        }
    }
    // before leaving: every copy issued has landed (bounded)
    __device__ void drain() {
        for (uint32_t q = (k > NSLOT ? k - NSLOT : 0); q < k; ++q) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&s.full[q % NSLOT], (q / NSLOT) & 1))
                if (clock64() - t0 > WAIT_LIMIT) break;
        }
    }
};

__device__ void producer(const Args &a, Smem &s, const Part &pt) {
    Producer P(s, a.err);
    for (int l = 0; l < a.L && P.ok; ++l) {
        const uint8_t *lw = a.layers + (size_t)l * a.layer_bytes;
        if (pt.g >= 0) {
            for (int v = pt.qa; v < pt.qb;) {  // stage A
                const int ve = qkv_run_end(v, pt.qb);
                P.rows(lw + a.o_wqkv, qkv_row(pt.g, v), qkv_row(pt.g, v) + (ve - v), C * 2);
                v = ve;
            }
            for (int b = 0; b < a.B; ++b) {  // stage B
                if (s.pos[b] >= a.max_ctx) continue;
                const size_t head = (size_t)l * a.kv_layer_elems + ((size_t)s.slot[b] * HKV + pt.g) * a.max_ctx * D;
                P.kv(a.kcache + head, a.vcache + head, 0, s.pos[b]);
            }
            P.rows(lw + a.o_wog + (size_t)pt.g * C * GD * 2, pt.oa, pt.ob, GD * 2);
        }
        P.rows(lw + a.o_wgu, 2 * pt.ja, 2 * pt.jb, C * 2);  // stage C
        P.rows(lw + a.o_wdownT, pt.ja, pt.jb, C * 2);
    }
    if (P.ok) P.rows(a.embed, pt.va, pt.vb, C * 2);
    if (!P.ok) s.dead = 1;
    P.drain();
}

// ---- consumers --------------------------------------------------------------------------

struct Ring {
    Smem &s;
    uint32_t *err;
    uint32_t k = 0;
    __device__ Ring(Smem &sm, uint32_t *e) : s(sm), err(e) {}
    __device__ const uint8_t *take() { return peek(0); }
    // slot k + q (q < NSLOT), waited for; on a failed wait the CTA is marked dead and control
    // flow goes on
    __device__ const uint8_t *peek(int q) {
        const uint32_t kk = k + q;
        const int p = kk % NSLOT;
        if (!ring_wait(&s.full[p], (kk / NSLOT) & 1, err)) s.dead = 1;
        return s.ring[p];
    }
    __device__ void release() {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&s.empty[k % NSLOT]);
        ++k;
    }
};

// x[b] = RMSNorm(v[b]; gain) as bf16, one warp per sequence.  v from L2 (fp32 [B][C]) or, for
// the first layer, the embedding rows of the tokens.
// When add_to is given, the elements [ra, rb) of v[b] are also added into add_to[b] (atomics).
__device__ void norm_rows(const Args &a, Smem &s, const float *v, bool from_embed, const float *gain,
                          float *add_to = nullptr, int ra = 0, int rb_ = 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int b = warp; b < a.B; b += NW) {
        float4 x[C / 128];
#pragma unroll
        for (int i = 0; i < C / 128; ++i) {
            if (from_embed) {
                const uint2 e = reinterpret_cast<const uint2 *>(a.embed + (size_t)s.tok[b] * C)[i * 32 + lane];
                const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&e.x));
                const float2 q = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&e.y));
                x[i] = make_float4(p.x, p.y, q.x, q.y);
            } else {
                x[i] = __ldcg(reinterpret_cast<const float4 *>(v + (size_t)b * C) + i * 32 + lane);
            }
        }
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < C / 128; ++i) ss += x[i].x * x[i].x + x[i].y * x[i].y + x[i].z * x[i].z + x[i].w * x[i].w;
        if (add_to) {
#pragma unroll
            for (int i = 0; i < C / 128; ++i) {
                const int e0 = (i * 32 + lane) * 4;
                const float xe[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (e0 + q >= ra && e0 + q < rb_) red_add(add_to + (size_t)b * C + e0 + q, xe[q]);
            }
        }
        const float inv = rsqrtf(warp_sum(ss) / (float)C + a.eps);
        uint2 *dst = reinterpret_cast<uint2 *>(s.x + (size_t)b * C);
#pragma unroll
        for (int i = 0; i < C / 128; ++i) {
            const float4 g = reinterpret_cast<const float4 *>(gain)[i * 32 + lane];
            uint2 o;
            o.x = pack_bf16x2(x[i].x * inv * g.x, x[i].y * inv * g.y);
            o.y = pack_bf16x2(x[i].z * inv * g.z, x[i].w * inv * g.w);
            dst[i * 32 + lane] = o;
        }
    }
}

// Dot products of the n rows in one slot (K elements each; rows warp, warp + NW, ...) with
// every x[b] (x rows K apart).  fn(row_in_slot, b, value) is called by lane 0.
template <int NB, int K, typename Fn>
__device__ __forceinline__ void slot_dots(const Args &a, const Smem &s, const uint8_t *slot, int n, Fn fn) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int row = warp; row < n; row += NW) {
        const uint4 *w = reinterpret_cast<const uint4 *>(slot + (size_t)row * K * 2);
        uint4 wr[K / 256];
#pragma unroll
        for (int i = 0; i < K / 256; ++i) wr[i] = w[i * 32 + lane];
        float acc[NB][2];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = 0.0f;
#pragma unroll
        for (int i = 0; i < K / 256; ++i) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b < a.B) {
                    const uint4 x = reinterpret_cast<const uint4 *>(s.x + (size_t)b * K)[i * 32 + lane];
                    acc[b][i & 1] = dot8(wr[i], x, acc[b][i & 1]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b < a.B) {
                const float v = warp_sum(acc[b][0] + acc[b][1]);
                if (lane == 0) fn(row, b, v);
            }
        }
    }
}

// Attention of KV head g for sequence b (both query heads): keys 0..pos, the new key and value
// from this step's q/k/v rows; the normalised output goes to x[b][gi*D + d] as bf16.
__device__ void attend(const Args &a, Smem &s, Ring &R, int l, int b, int g, bool write_kv) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int sub = lane & 7, kg = lane >> 3;
    const int pos = s.pos[b];
    const float *row = a.qkv + (size_t)b * NQKV;
    float x[G + 2][16];
#pragma unroll
    for (int hh = 0; hh < G + 2; ++hh) {
        const int head = hh < G ? g * G + hh : (hh == G ? HQ + g : HQ + HKV + g);
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            const float4 t = __ldcg(reinterpret_cast<const float4 *>(row + (size_t)head * D + sub * 16 + e));
            x[hh][e] = t.x; x[hh][e + 1] = t.y; x[hh][e + 2] = t.z; x[hh][e + 3] = t.w;
        }
    }
    float qv[G][16];
#pragma unroll
    for (int hh = 0; hh < G + 1; ++hh) {  // per-head RMSNorm + rotate-half RoPE of q and the new k
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) ss += x[hh][e] * x[hh][e];
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        const float inv = rsqrtf(ss * (1.0f / D) + a.eps);
        const float *gn = s.gqk[hh < G ? 0 : 1];
#pragma unroll
        for (int e = 0; e < 16; ++e) x[hh][e] *= inv * gn[sub * 16 + e];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float2 cs = s.cs[b][(sub & 3) * 16 + e];
            const float partner = __shfl_xor_sync(0xffffffffu, x[hh][e], 4);
            const float rot = sub < 4 ? x[hh][e] * cs.x - partner * cs.y   // x_i cos - x_{i+64} sin
                                      : x[hh][e] * cs.x + partner * cs.y;  // x_{i+64} cos + x_i sin
            if (hh < G) qv[hh < G ? hh : 0][e] = rot * a.scale_log2;
            else x[G][e] = round_bf16(rot);
        }
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) x[G + 1][e] = round_bf16(x[G + 1][e]);
    if (warp == 0 && kg == 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            s.s_new[0][sub * 16 + e] = x[G][e];
            s.s_new[1][sub * 16 + e] = x[G + 1][e];
        }
        if (write_kv) {  // the new row into the cache
            const size_t at = (size_t)l * a.kv_layer_elems + (((size_t)s.slot[b] * HKV + g) * a.max_ctx + pos) * D + sub * 16;
            uint4 pk[2], pv[2];
            uint32_t *pa = reinterpret_cast<uint32_t *>(pk), *pb = reinterpret_cast<uint32_t *>(pv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                pa[e] = pack_bf16x2(x[G][2 * e], x[G][2 * e + 1]);
                pb[e] = pack_bf16x2(x[G + 1][2 * e], x[G + 1][2 * e + 1]);
            }
            uint4 *kd = reinterpret_cast<uint4 *>(a.kcache + at), *vd = reinterpret_cast<uint4 *>(a.vcache + at);
            kd[0] = pk[0]; kd[1] = pk[1];
            vd[0] = pv[0]; vd[1] = pv[1];
        }
    }
    float m[G], lsum[G], acc[G][16];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        m[gi] = -INFINITY;
        lsum[gi] = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[gi][e] = 0.0f;
    }
    // KPG keys of this 8-lane group at once: scores, one max and one rescale for all of them
    constexpr int KPG = 2;
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
            for (int o = 1; o <= 4; o <<= 1)
#pragma unroll
                for (int kk = 0; kk < KPG; ++kk) sc[kk] += __shfl_xor_sync(0xffffffffu, sc[kk], o);
            float mn = m[gi];
#pragma unroll
            for (int kk = 0; kk < KPG; ++kk)
                if (valid[kk]) mn = fmaxf(mn, sc[kk]);
            if (mn != -INFINITY) {
                const float c = exp2f(m[gi] - mn);
                float ps = 0.0f, p[KPG];
#pragma unroll
                for (int kk = 0; kk < KPG; ++kk) {
                    p[kk] = valid[kk] ? exp2f(sc[kk] - mn) : 0.0f;
                    ps += p[kk];
                }
                lsum[gi] = lsum[gi] * c + ps;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float t = acc[gi][e] * c;
#pragma unroll
                    for (int kk = 0; kk < KPG; ++kk) t = fmaf(p[kk], vf[kk][e], t);
                    acc[gi][e] = t;
                }
                m[gi] = mn;
            }
        }
    };
    const int jj = warp * 4 + kg;  // this group's key in every slot
    for (int j = 0; j < pos; j += KPG * CHUNK) {  // cached keys 0..pos-1, KPG slots at a time
        const int nsl = min(KPG, (pos - j + CHUNK - 1) / CHUNK);
        float kf[KPG][16], vf[KPG][16];
        bool valid[KPG];
#pragma unroll
        for (int q = 0; q < KPG; ++q) {
            const uint8_t *sl = q < nsl ? R.peek(q) : s.ring[0];
            valid[q] = q < nsl && j + q * CHUNK + jj < pos;
            const int js = valid[q] ? jj : 0;
            const uint4 *kp = reinterpret_cast<const uint4 *>(sl + (size_t)js * D * 2 + sub * 32);
            const uint4 *vp = reinterpret_cast<const uint4 *>(sl + SLOT / 2 + (size_t)js * D * 2 + sub * 32);
            unpack8(kp[0], kf[q]);
            unpack8(kp[1], kf[q] + 8);
            unpack8(vp[0], vf[q]);
            unpack8(vp[1], vf[q] + 8);
        }
        update(kf, vf, valid);
        for (int q = 0; q < nsl; ++q) R.release();
    }
    consumers_sync();  // s_new is visible
    if (warp == 0) {   // the new key at pos
        float kf[KPG][16], vf[KPG][16];
        bool valid[KPG];
#pragma unroll
        for (int q = 0; q < KPG; ++q) {
            valid[q] = q == 0 && kg == 0;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                kf[q][e] = s.s_new[0][sub * 16 + e];
                vf[q][e] = s.s_new[1][sub * 16 + e];
            }
        }
        update(kf, vf, valid);
    }
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {  // merge the four 8-lane groups of the warp
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[gi], off);
            const float lo = __shfl_xor_sync(0xffffffffu, lsum[gi], off);
            const float mn = fmaxf(m[gi], mo);
            const float c1 = mn == -INFINITY ? 0.0f : exp2f(m[gi] - mn);
            const float c2 = mn == -INFINITY ? 0.0f : exp2f(mo - mn);
            lsum[gi] = lsum[gi] * c1 + lo * c2;
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
                s.red_ml[warp][gi][0] = m[gi];
                s.red_ml[warp][gi][1] = lsum[gi];
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) s.red_o[warp][gi][sub * 16 + e] = acc[gi][e];
        }
    }
    consumers_sync();
    for (int idx = tid; idx < G * D; idx += NW * 32) {  // merge the warps
        const int gi = idx / D, d = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) mx = fmaxf(mx, s.red_ml[w][gi][0]);
        float ls = 0.0f, o = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float c = mx == -INFINITY ? 0.0f : exp2f(s.red_ml[w][gi][0] - mx);
            ls += s.red_ml[w][gi][1] * c;
            o += s.red_o[w][gi][d] * c;
        }
        s.x[(size_t)b * GD + gi * D + d] = __float2bfloat16(o / ls);
    }
    consumers_sync();  // red_* and s_new are free again
}

template <int NB>
__device__ void consumer(const Args &a, Smem &s, const Part &pt, int cta, int grid) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    Ring R(s, a.err);
    auto arrive = [&](uint32_t *counter) {  // the CTA barrier orders every consumer's writes before the release
        consumers_sync();
        if (tid == 0) red_release_add(counter, 1);
    };
    auto wait = [&](const uint32_t *counter, uint32_t target) {
        if (tid == 0 && !wait_count(counter, target, a.err)) s.dead = 1;
        consumers_sync();
    };
    auto dump_rows = [&](int idx, const float *src, bool from_embed) {
        if (!a.dump) return;
        for (int i = tid; i < a.B * (pt.rb_ - pt.ra); i += NW * 32) {
            const int b = i / (pt.rb_ - pt.ra), r = pt.ra + i % (pt.rb_ - pt.ra);
            a.dump[((size_t)idx * a.B + b) * C + r] =
                from_embed ? __bfloat162float(a.embed[(size_t)s.tok[b] * C + r]) : __ldcg(src + (size_t)b * C + r);
        }
    };
    const uint32_t all = (uint32_t)grid;

    for (int l = 0; l < a.L; ++l) {
        const uint8_t *lw = a.layers + (size_t)l * a.layer_bytes;
        float *h = res_h(a, l), *P = res_p(a, l), *Q = res_h(a, l + 1);

        // ---- A: this CTA's q/k/v rows of RMSNorm(h; input gain) ----
        if (l > 0) wait(a.arrive, 2 * l * all);  // h complete
        dump_rows(l, h, l == 0);
        for (int i = tid; i < a.B * (pt.rb_ - pt.ra); i += NW * 32) {  // Q accumulates in stage C
            const int b = i / (pt.rb_ - pt.ra), r = pt.ra + i % (pt.rb_ - pt.ra);
            Q[(size_t)b * C + r] = 0.0f;
        }
        if (pt.g >= 0) {
            // inputs of stage B that are already final: gains, RoPE rows, group 0's residual rows
            for (int i = tid; i < 2 * D; i += NW * 32)
                s.gqk[i / D][i % D] = reinterpret_cast<const float *>(lw + (i < D ? a.o_gq : a.o_gk))[i % D];
            for (int i = tid; i < a.B * (D / 2); i += NW * 32) {
                const int b = i / (D / 2), pos = min(s.pos[b], a.max_ctx - 1);
                s.cs[b][i % (D / 2)] = a.rope[(size_t)pos * (D / 2) + i % (D / 2)];
            }
            if (pt.g == 0) {
                const int no = pt.ob - pt.oa;
                for (int i = tid; i < a.B * no; i += NW * 32) {
                    const int b = i / no, r = pt.oa + i % no;
                    s.hres[b][i % no] = l == 0 ? __bfloat162float(a.embed[(size_t)s.tok[b] * C + r])
                                               : __ldcg(h + (size_t)b * C + r);
                }
            }
            norm_rows(a, s, h, l == 0, reinterpret_cast<const float *>(lw + a.o_gin));
            consumers_sync();
            for (int v = pt.qa; v < pt.qb;) {
                const int ve = qkv_run_end(v, pt.qb), r0 = qkv_row(pt.g, v);
                for (int r = 0; r < ve - v; r += SLOT / (C * 2)) {
                    const uint8_t *sl = R.take();
                    const int n = min(SLOT / (C * 2), ve - v - r);
                    slot_dots<NB, C>(a, s, sl, n, [&](int i, int b, float val) {
                        a.qkv[(size_t)b * NQKV + r0 + r + i] = val;
                    });
                    R.release();
                }
                v = ve;
            }
            arrive(a.grp + pt.g);

            // ---- B: attention of KV head g, then this CTA's o_proj rows over its 256 columns ----
            wait(a.grp + pt.g, (uint32_t)((l + 1) * pt.gsz));
            for (int b = 0; b < a.B; ++b)
                if (s.pos[b] < a.max_ctx) attend(a, s, R, l, b, pt.g, pt.gi == 0);
            for (int r = pt.oa; r < pt.ob; r += SLOT / (GD * 2)) {
                const uint8_t *sl = R.take();
                const int n = min(SLOT / (GD * 2), pt.ob - r);
                slot_dots<NB, GD>(a, s, sl, n, [&](int i, int b, float val) {
                    if (pt.g == 0) val += s.hres[b][r + i - pt.oa];  // the residual, once per row
                    red_add(P + (size_t)b * C + r + i, val);
                });
                R.release();
            }
        }
        arrive(a.arrive);

        // ---- C: RMSNorm(P), SwiGLU of this CTA's activations, their slice of the down projection ----
        wait(a.arrive, (2 * l + 1) * all);  // P complete
        // RMSNorm of P; this CTA's slice of P also goes into Q (the residual of the MLP)
        norm_rows(a, s, P, false, reinterpret_cast<const float *>(lw + a.o_gpost), Q, pt.ra, pt.rb_);
        consumers_sync();
        {
            const int na = pt.jb - pt.ja;
            for (int r = 0; r < 2 * na; r += SLOT / (C * 2)) {
                const uint8_t *sl = R.take();
                const int n = min(SLOT / (C * 2), 2 * na - r);
                slot_dots<NB, C>(a, s, sl, n, [&](int i, int b, float v) { s.gu[b][r + i] = v; });
                R.release();
            }
            consumers_sync();
            for (int i = tid; i < a.B * na; i += NW * 32) {
                const int b = i / na, j = i % na;
                s.act[b][j] = round_bf16(silu(s.gu[b][2 * j]) * s.gu[b][2 * j + 1]);
            }
            consumers_sync();
            float4 acc[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            const int c0 = tid * 4;  // this thread's 4 output columns
            for (int r = 0; r < na; r += SLOT / (C * 2)) {
                const uint8_t *sl = R.take();
                const int n = min(SLOT / (C * 2), na - r);
                for (int i = 0; i < n; ++i) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(sl + (size_t)i * C * 2 + c0 * 2);
                    const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
                    const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        if (b < a.B) {
                            const float av = s.act[b][r + i];
                            acc[b].x = fmaf(av, w01.x, acc[b].x);
                            acc[b].y = fmaf(av, w01.y, acc[b].y);
                            acc[b].z = fmaf(av, w23.x, acc[b].z);
                            acc[b].w = fmaf(av, w23.y, acc[b].w);
                        }
                    }
                }
                R.release();
            }
            if (na > 0) {
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    if (b < a.B) red_add_v4(Q + (size_t)b * C + c0, acc[b]);
            }
            // the next layer's P slice starts at zero
            float *Pn = res_p(a, l + 1);
            for (int i = tid; i < a.B * (pt.rb_ - pt.ra); i += NW * 32) {
                const int b = i / (pt.rb_ - pt.ra), r = pt.ra + i % (pt.rb_ - pt.ra);
                Pn[(size_t)b * C + r] = 0.0f;
            }
        }
        arrive(a.arrive);
    }

    // ---- final RMSNorm, tied lm_head, this CTA's best (value, index) per sequence ----
    const float *fin = res_h(a, a.L);
    wait(a.arrive, 2 * a.L * all);
    dump_rows(a.L, fin, false);
    norm_rows(a, s, fin, false, a.g_final);
    consumers_sync();
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int r = pt.va; r < pt.vb; r += SLOT / (C * 2)) {
        const uint8_t *sl = R.take();
        const int n = min(SLOT / (C * 2), pt.vb - r);
        // lane 0 of each warp gets every b; lane b keeps sequence b's best
        float vals[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) vals[b] = 0.0f;
        slot_dots<NB, C>(a, s, sl, n, [&](int i, int b, float v) {
            vals[b] = v;
            if (a.logits) a.logits[(size_t)b * a.V + r + i] = v;
        });
        if (warp < n) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float v = __shfl_sync(0xffffffffu, vals[b], 0);
                if (b < a.B && lane == b && better(v, r + warp, bv, bi)) {
                    bv = v;
                    bi = r + warp;
                }
            }
        }
        R.release();
    }
    if (lane < a.B) {
        s.best_v[warp][lane] = bv;
        s.best_i[warp][lane] = bi;
    }
    consumers_sync();
    if (tid < a.B) {
        float v = s.best_v[0][tid];
        int i = s.best_i[0][tid];
        for (int w = 1; w < NW; ++w)
            if (better(s.best_v[w][tid], s.best_i[w][tid], v, i)) {
                v = s.best_v[w][tid];
                i = s.best_i[w][tid];
            }
        a.part_val[(size_t)tid * grid + cta] = v;
        a.part_idx[(size_t)tid * grid + cta] = i;
    }
}

template <int NB>
__global__ void __launch_bounds__(THREADS, 1) k_decode_persistent(const __grid_constant__ Args a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, grid = gridDim.x;
    if (threadIdx.x == 0) {
        for (int p = 0; p < NSLOT; ++p) {
            mbar_init(&s.full[p], 1);
            mbar_init(&s.empty[p], NW);
        }
        s.dead = 0;
    }
    if (threadIdx.x < a.B) {
        const int b = threadIdx.x;
        int id = a.tokens[b];
        if (id < 0 || id >= a.V) {
            if (cta == 0) atomicOr(a.err, ERR_TOKEN_RANGE);
            id = id < 0 ? 0 : a.V - 1;
        }
        const int sl = a.slots[b];
        const int pos = __ldcg(a.ctx_len + sl);
        if (pos >= a.max_ctx && cta == 0) atomicOr(a.err, ERR_POSITION);
        s.tok[b] = id;
        s.slot[b] = sl;
        s.pos[b] = pos;
    }
    __syncthreads();
    const Part pt = make_part(a, cta, grid);
    if (warp == NW) {
        if (lane == 0) producer(a, s, pt);
    } else {
        consumer<NB>(a, s, pt, cta, grid);
    }
    __syncthreads();
    if (s.dead) return;  // error already recorded; the step's outputs are not valid

    // the CTA that finishes last reduces the partial argmaxes and closes the step
    if (threadIdx.x == 0) {
        __threadfence();
        s.last = atomicAdd(a.counter, 1) == grid - 1;
    }
    __syncthreads();
    if (!s.last) return;
    __threadfence();
    if (warp < a.B) {
        const int b = warp;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int p = lane; p < grid; p += 32) {
            const float v = __ldcg(a.part_val + (size_t)b * grid + p);
            const int i = __ldcg(a.part_idx + (size_t)b * grid + p);
            if (better(v, i, bv, bi)) {
                bv = v;
                bi = i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v = __shfl_xor_sync(0xffffffffu, bv, o);
            const int i = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(v, i, bv, bi)) {
                bv = v;
                bi = i;
            }
        }
        if (lane == 0) {
            a.next_tok[b] = bi;
            if (s.pos[b] < a.max_ctx) a.ctx_len[s.slot[b]] = s.pos[b] + 1;
        }
    }
    // the next step starts from zero counters and a zero P of its first layer
    float *P0 = res_p(a, 0);
    for (int i = threadIdx.x; i < a.B * C; i += THREADS) P0[i] = 0.0f;
    if (threadIdx.x < HKV) a.grp[threadIdx.x] = 0;
    if (threadIdx.x == 0) {
        *a.arrive = 0;
        *a.counter = 0;
    }
}

template <int NB>
cudaError_t run(const Launch &lc, const Args &a) {
    const size_t smem = sizeof(Smem);
    cudaError_t e = cudaFuncSetAttribute(k_decode_persistent<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(lc.num_sms);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (lc.counter) ++*lc.counter;
    return cudaLaunchKernelEx(&cfg, k_decode_persistent<NB>, a);
}

}  // namespace

bool decode_persistent_supported(int C_, int Hq, int Hkv, int head_dim, int I, int B, int num_sms) {
    return C_ == C && Hq == HQ && Hkv == HKV && head_dim == D && B >= 1 && B <= B_MAX && num_sms >= HKV &&
           (I + num_sms - 1) / num_sms <= NA_MAX && (C + num_sms / HKV - 1) / (num_sms / HKV) <= OROWS_MAX &&
           sizeof(Smem) <= 227 * 1024;
}

cudaError_t launch_decode_persistent(const Launch &lc, const DecodePersistentArgs &p) {
    if (!decode_persistent_supported(p.C, p.Hq, p.Hkv, p.head_dim, p.I, p.B, lc.num_sms))
        return cudaErrorInvalidValue;
    Args a;
    a.L = p.L; a.I = p.I; a.V = p.V; a.max_ctx = p.max_ctx; a.B = p.B;
    a.eps = p.eps;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    a.layers = p.layers; a.layer_bytes = p.layer_bytes;
    a.o_wqkv = p.o_wqkv; a.o_wog = p.o_wog; a.o_wgu = p.o_wgu; a.o_wdownT = p.o_wdownT;
    a.o_gin = p.o_gin; a.o_gpost = p.o_gpost; a.o_gq = p.o_gq; a.o_gk = p.o_gk;
    a.embed = p.embed; a.g_final = p.g_final; a.rope = p.rope;
    a.kcache = p.kcache; a.vcache = p.vcache; a.kv_layer_elems = p.kv_layer_elems;
    a.tokens = p.tokens; a.slots = p.slots; a.ctx_len = p.ctx_len; a.next_tok = p.next_tok;
    a.logits = p.logits; a.dump = p.dump;
    for (int i = 0; i < 3; ++i) a.res[i] = p.res[i];
    a.qkv = p.qkv;
    a.part_val = p.part_val; a.part_idx = p.part_idx;
    a.arrive = p.arrive; a.grp = p.grp; a.counter = p.counter; a.err = p.err;
    if (p.B <= 1) return run<1>(lc, a);
    if (p.B <= 2) return run<2>(lc, a);
    if (p.B <= 4) return run<4>(lc, a);
    return run<8>(lc, a);
}

}  // namespace q3
