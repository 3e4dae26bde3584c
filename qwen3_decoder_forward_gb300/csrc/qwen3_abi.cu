// C ABI of the Qwen3 decoder forward: arena layout, weight packing, argument checks and the
// per-call kernel chains (prefill over a packed ragged batch; one decode step, recorded as a
// CUDA graph and replayed).  See include/qwen3_gb300.h for the contract of every call.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "kernels.h"
#include "qwen3_gb300.h"

using namespace q3;

namespace {

constexpr size_t ALIGN = 1024;
constexpr int MAX_SPLIT = ATTN_DECODE_MAX_SPLIT;  // decode attention: key ranges per (sequence, head)
constexpr int MAX_PARTS = 1024; // lm_head partial results per row

size_t align_up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

struct Layout {
    // per-layer strides (bytes) and offsets within layer 0
    size_t layer_bytes = 0, o_wqkv = 0, o_wo = 0, o_wog = 0, o_wgu = 0, o_wdown = 0, o_wdownT = 0, o_gin = 0,
           o_gpost = 0, o_gq = 0, o_gk = 0;
    size_t o_layers = 0, o_embed = 0, o_gfinal = 0, o_rope = 0, o_rope_t = 0, o_kcache = 0, o_vcache = 0,
           kv_layer_bytes = 0, o_ctxlen = 0, o_err = 0, o_kvtable = 0;
    int32_t kv_max_blocks = 0;  // paged cache: table entries per slot
    size_t o_resid = 0, o_xn = 0, o_qkv = 0, o_q = 0, o_attn = 0, o_act = 0, o_rowslot = 0,
           o_rowpos = 0, o_last = 0, o_pval = 0, o_pidx = 0, o_wsml = 0, o_wso = 0, o_counters = 0, o_pres = 0,
           o_resid2 = 0, o_ssp = 0;
    size_t total = 0;
};

bool config_supported(const qwen3_config &c, std::string *why) {
    auto fail = [&](const char *m) {
        if (why) *why = m;
        return false;
    };
    if (c.n_layers < 1 || c.hidden < 1 || c.n_q_heads < 1 || c.n_kv_heads < 1 || c.vocab < 1 ||
        c.intermediate < 1 || c.max_seqs < 1 || c.max_ctx < 1 || c.max_prefill_tokens < 1)
        return fail("config: every size must be >= 1");
    if (!(c.rms_eps >= 0.0f) || !(c.rope_theta > 0.0)) return fail("config: bad rms_eps or rope_theta");
    if (c.head_dim != 128) return fail("config: head_dim must be 128");
    if (c.n_q_heads % c.n_kv_heads != 0) return fail("config: n_q_heads must be a multiple of n_kv_heads");
    const int g = c.n_q_heads / c.n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return fail("config: n_q_heads/n_kv_heads must be 1, 2, 4 or 8");
    const int qd = c.n_q_heads * c.head_dim;
    if (c.hidden % 256 || c.hidden > 3072) return fail("config: hidden must be a multiple of 256, at most 3072");
    if (qd % 256 || qd > 4096) return fail("config: n_q_heads*head_dim must be a multiple of 256, at most 4096");
    if (c.intermediate % 256 || c.intermediate > 4096) return fail("config: intermediate must be a multiple of 256, at most 4096");
    if (c.hidden % 128 || qd % 128 || ((c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim) % 128 ||
        (2 * c.intermediate) % 128)
        return fail("config: projection widths must be multiples of 128");
    if (c.max_seqs > 1024) return fail("config: max_seqs must be at most 1024");
    if (c.flags & ~(QWEN3_FLAG_NO_GRAPH | QWEN3_FLAG_NO_PDL | QWEN3_FLAG_DECODE_CHAIN))
        return fail("config: unknown flag bits");
    if (c.kv_block_tokens < 0 || (c.kv_block_tokens > 0 && (c.kv_block_tokens % 128 || c.kv_pool_blocks < 1)))
        return fail("config: kv_block_tokens must be 0 or a multiple of 128, with kv_pool_blocks >= 1");
    if (c.kv_block_tokens > 0) {
        if (c.n_q_heads != 2 * c.n_kv_heads) return fail("config: a paged KV cache needs n_q_heads == 2 * n_kv_heads");
        if (((c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim) % 256 || c.hidden % 64)
            return fail("config: a paged KV cache needs the tensor-core QKV projection shape");
        if ((size_t)c.kv_pool_blocks * c.n_kv_heads * c.kv_block_tokens > (size_t)INT32_MAX)
            return fail("config: kv_pool_blocks too large");
    }
    return true;
}

Layout make_layout(const qwen3_config &c) {
    Layout L;
    const size_t C = c.hidden, D = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, I = c.intermediate;
    const size_t qkv_n = (Hq + 2 * Hkv) * D;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    // one layer's block
    L.o_wqkv = take(qkv_n * C * 2);
    L.o_wo = take(C * Hq * D * 2);
    L.o_wog = take(C * Hq * D * 2);  // o_proj regrouped by KV head [Hkv][C][Hq/Hkv*D] (one-row decode layer)
    L.o_wgu = take(2 * I * C * 2);
    L.o_wdown = take(C * I * 2);
    L.o_wdownT = take(C * I * 2);  // down weight transposed [I, C] for the split-K decode MLP
    L.o_gin = take(C * 4);
    L.o_gpost = take(C * 4);
    L.o_gq = take(D * 4);
    L.o_gk = take(D * 4);
    L.layer_bytes = off;
    off = 0;
    L.o_layers = take(L.layer_bytes * c.n_layers);
    L.o_embed = take((size_t)c.vocab * C * 2);
    L.o_gfinal = take(C * 4);
    L.o_rope = take((size_t)c.max_ctx * (D / 2) * 8);
    L.o_rope_t = take((size_t)c.max_ctx * (D / 2) * 8);  // the same table, by pairs of frequencies
    if (c.kv_block_tokens > 0) {  // paged: a pool of blocks [block][Hkv][bs][D] and a block table
        L.kv_layer_bytes = (size_t)c.kv_pool_blocks * Hkv * c.kv_block_tokens * D * 2;
        L.kv_max_blocks = (c.max_ctx + c.kv_block_tokens - 1) / c.kv_block_tokens;
        L.o_kvtable = take((size_t)c.max_seqs * L.kv_max_blocks * 4);
    } else {
        L.kv_layer_bytes = (size_t)c.max_seqs * Hkv * c.max_ctx * D * 2;
    }
    L.o_kcache = take(L.kv_layer_bytes * c.n_layers);
    L.o_vcache = take(L.kv_layer_bytes * c.n_layers);
    L.o_ctxlen = take((size_t)c.max_seqs * 4);
    L.o_err = take(16);
    const size_t R = std::max(c.max_prefill_tokens, c.max_seqs);
    L.o_resid = take(R * C * 4);
    L.o_xn = take(R * C * 2);
    L.o_qkv = take(R * qkv_n * 4);
    L.o_q = take(R * Hq * D * 2);
    L.o_attn = take(R * Hq * D * 2);
    L.o_act = take(R * I * 2);
    L.o_rowslot = take(R * 4);
    L.o_rowpos = take(R * 4);
    L.o_last = take((size_t)c.max_seqs * C * 2);
    L.o_pval = take((size_t)c.max_seqs * MAX_PARTS * 4);
    L.o_pidx = take((size_t)c.max_seqs * MAX_PARTS * 4);
    L.o_wsml = take((size_t)c.max_seqs * Hq * MAX_SPLIT * 2 * 4);
    L.o_wso = take((size_t)c.max_seqs * Hq * MAX_SPLIT * D * 4);
    L.o_counters = take((size_t)c.max_seqs * Hkv * 4);
    L.o_resid2 = take((size_t)c.max_seqs * C * 4);  // second residual buffer of the decode ping-pong
    L.o_pres = take((size_t)3 * c.max_seqs * C * 4);  // one-row decode layer: three residual buffers
    L.o_ssp = take(2 * R * (C / 128) * 4);  // prefill: per-128-column sums of squares of h, two norms
    L.total = off;
    return L;
}

thread_local std::string g_create_error;

}  // namespace

namespace q3 {
void set_last_error(const std::string &msg) { g_create_error = msg; }
}  // namespace q3

struct GraphEntry {
    int B, n_split;
    const void *tokens, *slots;
    void *logits, *next;
    qwen3_sampling sampling;
    cudaGraphExec_t exec;
    int64_t kernels;
};

struct qwen3_ctx {
    qwen3_config cfg;
    Layout lay;
    uint8_t *arena = nullptr;
    std::vector<int32_t> len_host;
    int num_sms = 0, n_parts = 0, attn_ctas_per_sm = 1;
    float *dump = nullptr;
    size_t dump_bytes = 0;
    cudaStream_t cap_stream = nullptr;
    std::vector<GraphEntry> graphs;
    int64_t launches = 0;
    qwen3_sampling sampling = {};  // all NULL: greedy next tokens
    std::string err;
    // paged KV cache: host copy of the block table [max_seqs][max_blocks], blocks held per
    // slot, and the free blocks (a stack)
    std::vector<int32_t> kv_table, kv_nblk, kv_free;

    template <typename T>
    T *at(size_t off) const { return reinterpret_cast<T *>(arena + off); }
    uint8_t *layer(int l) const { return arena + lay.o_layers + (size_t)l * lay.layer_bytes; }
    bf16 *kcache(int l) const { return at<bf16>(lay.o_kcache + (size_t)l * lay.kv_layer_bytes); }
    bf16 *vcache(int l) const { return at<bf16>(lay.o_vcache + (size_t)l * lay.kv_layer_bytes); }
    int fail(int code, const std::string &m) {
        err = m;
        return code;
    }
    int cuda_fail(cudaError_t e, const char *where) {
        err = std::string(where) + ": " + cudaGetErrorString(e);
        return QWEN3_E_CUDA;
    }
};

namespace {

#define Q3_TRY(x)                               \
    do {                                        \
        cudaError_t e_ = (x);                   \
        if (e_ != cudaSuccess) return e_;       \
    } while (0)

bool sampling_on(const qwen3_ctx *c) { return c->sampling.temperature != nullptr; }

// With sampling set, the next tokens are drawn from the logits the lm_head just wrote
// (replacing its argmax); otherwise nothing to do.
cudaError_t draw_next(qwen3_ctx *c, const Launch &lc, const float *logits, int B, int32_t *next) {
    if (!sampling_on(c)) return cudaSuccess;
    Launch ls = lc;
    ls.pdl = false;
    const qwen3_sampling &sp = c->sampling;
    return launch_sample(ls, logits, B, c->cfg.vocab, sp.temperature, sp.top_k, sp.top_p, sp.uniform, next);
}

// Plan of the decode attention for B rows whose longest context is max_len: from a
// power-of-two bucket of it, so a recorded graph stays valid while contexts grow inside the
// bucket; the key ranges per (sequence, KV head) of one wave: as many as the SMs hold CTAs for
// all pairs at once, ranges of at least 64 keys (the kernel divides the actual keys 0..pos of
// each sequence evenly over them, in whole 64-key chunks).
int plan_decode_attention(int num_sms, int ctas_per_sm, int B, int Hkv, int max_len, int max_ctx) {
    int bucket = 64;
    while (bucket < max_len) bucket <<= 1;
    bucket = std::min(bucket, max_ctx);
    const long long pairs = (long long)B * Hkv;
    const long long slots = (long long)num_sms * ctas_per_sm;
    return (int)std::max(1ll, std::min({slots / pairs, (long long)MAX_SPLIT, (long long)(bucket + 63) / 64}));
}

// The decode attention of layer l: n_split key ranges per (sequence, KV head).
cudaError_t decode_attention(qwen3_ctx *c, const Launch &lc, const float *qkv, const Rows &rows, const float *g_q,
                             const float *g_k, const float2 *rope, int l, int n_split, bf16 *attn, uint32_t *err) {
    const qwen3_config &k = c->cfg;
    const Layout &L = c->lay;
    return launch_attn_decode_fused(lc, qkv, rows, g_q, g_k, rope, c->kcache(l), c->vcache(l),
                                    L.kv_layer_bytes / (k.head_dim * 2), n_split, c->at<float>(L.o_wsml),
                                    c->at<float>(L.o_wso), c->at<int>(L.o_counters), attn, k.n_q_heads,
                                    k.n_kv_heads, k.max_ctx, k.rms_eps, err);
}

// Everything one call runs, in stream order.  `decode` selects the GEMV projections and the
// split-KV attention; prefill uses the tiled GEMM and the flash prefill attention.
cudaError_t run_forward(qwen3_ctx *c, const Launch &lc, const int32_t *tokens, const Rows &rows,
                        bool decode, int max_len, int n_split, float *logits,
                        int32_t *next) {
    const qwen3_config &k = c->cfg;
    const Layout &L = c->lay;
    const int C = k.hidden, D = k.head_dim, Hq = k.n_q_heads, Hkv = k.n_kv_heads, I = k.intermediate;
    const int qkv_n = (Hq + 2 * Hkv) * D, R = rows.rows;
    float *resid = c->at<float>(L.o_resid);
    bf16 *xn = c->at<bf16>(L.o_xn);
    float *qkv = c->at<float>(L.o_qkv);
    bf16 *q = c->at<bf16>(L.o_q), *attn = c->at<bf16>(L.o_attn), *act = c->at<bf16>(L.o_act);
    uint32_t *err = c->at<uint32_t>(L.o_err);
    const bf16 *embed = c->at<bf16>(L.o_embed);
    const float2 *rope = c->at<float2>(L.o_rope);
    const float4 *rope_t = c->at<float4>(L.o_rope_t);
    auto dump = [&](int l, const float *src) -> cudaError_t {
        if (!c->dump) return cudaSuccess;
        return cudaMemcpyAsync(c->dump + (size_t)l * R * C, src, (size_t)R * C * 4,
                               cudaMemcpyDeviceToDevice, lc.stream);
    };

    // decode of one row: two kernels per layer over three rotating residual buffers
    const bool block = decode && !(k.flags & QWEN3_FLAG_DECODE_CHAIN) &&
                       decode_block_supported(R, C, Hq, Hkv, D, I, lc.num_sms);
    if (block) {
        float *rb[3];
        for (int i = 0; i < 3; ++i) rb[i] = c->at<float>(L.o_pres) + (size_t)i * k.max_seqs * C;
        Q3_TRY(launch_embed_rmsnorm(lc, tokens, rows, embed, (const float *)(c->layer(0) + L.o_gin), rb[0], xn, C,
                                    k.vocab, k.rms_eps, err, rb[1]));
        Q3_TRY(dump(0, rb[0]));
        const float scale_log2 = 1.4426950408889634f / std::sqrt((float)D);
        for (int l = 0; l < k.n_layers; ++l) {
            const uint8_t *lw = c->layer(l);
            const uint8_t *nw = c->layer((l + 1) % k.n_layers);  // the next layer (the next step's first)
            AttnBlockParams a;
            a.h_in = rb[(2 * l) % 3];
            a.h_out = rb[(2 * l + 1) % 3];
            a.zero_next = rb[(2 * l + 2) % 3];
            a.g_in = (const float *)(lw + L.o_gin);
            a.wqkv = (const bf16 *)(lw + L.o_wqkv);
            a.wog = (const bf16 *)(lw + L.o_wog);
            a.g_q = (const float *)(lw + L.o_gq);
            a.g_k = (const float *)(lw + L.o_gk);
            a.rope = rope;
            a.k_layer = c->kcache(l);
            a.v_layer = c->vcache(l);
            a.slots = rows.slots;
            a.ctx_len = rows.ctx_len;
            a.kv = rows.kv;
            a.ahead_gu = (const bf16 *)(lw + L.o_wgu);
            a.ahead_dt = (const bf16 *)(lw + L.o_wdownT);
            a.B = R;
            a.Hq = Hq;
            a.Hkv = Hkv;
            a.max_ctx = k.max_ctx;
            a.I = I;
            a.eps = k.rms_eps;
            a.scale_log2 = scale_log2;
            a.err = err;
            Q3_TRY(launch_attn_block(lc, a));
            MlpBlockParams m;
            m.h_in = a.h_out;
            m.h_out = rb[(2 * l + 2) % 3];
            m.zero_next = rb[(2 * l + 3) % 3];
            m.gain = (const float *)(lw + L.o_gpost);
            m.wgu = (const bf16 *)(lw + L.o_wgu);
            m.wdt = (const bf16 *)(lw + L.o_wdownT);
            m.ahead_qkv = (const bf16 *)(nw + L.o_wqkv);
            m.ahead_og = (const bf16 *)(nw + L.o_wog);
            m.qkv_rows = qkv_n;
            m.og_cols = Hq * D;
            m.B = R;
            m.C = C;
            m.I = I;
            m.NA = 0;
            m.eps = k.rms_eps;
            m.err = err;
            Q3_TRY(launch_mlp_block(lc, m));
            Q3_TRY(dump(l + 1, m.h_out));
        }
        bf16 *last = c->at<bf16>(L.o_last);
        Q3_TRY(launch_final_norm(lc, rb[(2 * k.n_layers) % 3], nullptr, rows.B, c->at<float>(L.o_gfinal), last, C,
                                 k.rms_eps));
        Q3_TRY(launch_lmhead_argmax(lc, last, rows.B, C, embed, k.vocab, logits, c->at<float>(L.o_pval),
                                    c->at<int32_t>(L.o_pidx), c->n_parts, next, rows, err));
        return draw_next(c, lc, logits, rows.B, next);
    }
    Q3_TRY(launch_embed_rmsnorm(lc, tokens, rows, embed, (const float *)(c->layer(0) + L.o_gin),
                                resid, xn, C, k.vocab, k.rms_eps, err));
    Q3_TRY(dump(0, resid));
    const bool fused = decode && gemv_fused_supported(R, C) && gemv_fused_supported(R, Hq * D) &&
                       gemv_fused_supported(R, I);
    // residual ping-pong of the fused decode MLP: layer l reads res[l & 1] and leaves res[(l+1) & 1]
    const bool mlp = fused && mlp_fused_supported(R, C, I, lc.num_sms);
    float *res[2] = {resid, mlp ? c->at<float>(L.o_resid2) : resid};
    for (int l = 0; l < k.n_layers; ++l) {
        const uint8_t *lw = c->layer(l);
        const float *g_in = (const float *)(lw + L.o_gin), *g_post = (const float *)(lw + L.o_gpost);
        const float *g_q = (const float *)(lw + L.o_gq), *g_k = (const float *)(lw + L.o_gk);
        const bf16 *w_qkv = (const bf16 *)(lw + L.o_wqkv), *w_o = (const bf16 *)(lw + L.o_wo);
        const bf16 *w_gu = (const bf16 *)(lw + L.o_wgu), *w_down = (const bf16 *)(lw + L.o_wdown);
        if (fused) {
            // decode, few rows: the norms folded into the GEMV prologues; each projection also asks
            // L2 for its block of the next layer's weights (the next step's layer 0 after the
            // last layer), so HBM streams ahead of the kernel chain.
            const uint8_t *ahead = c->layer((l + 1) % k.n_layers);
            float *r_cur = res[l & 1], *r_next = res[(l + 1) & 1];
            Q3_TRY(launch_gemv_fused(lc, r_cur, R, C, w_qkv, qkv_n, EPI_F32, qkv, g_in, k.rms_eps, err,
                                     (const bf16 *)(ahead + L.o_wqkv), mlp ? r_next : nullptr, R * C));
            Q3_TRY(decode_attention(c, lc, qkv, rows, g_q, g_k, rope, l, n_split, attn, err));
            Q3_TRY(launch_gemv_fused(lc, attn, R, Hq * D, w_o, C, EPI_RESID_ADD, r_cur, nullptr, 0.0f, err,
                                     (const bf16 *)(ahead + L.o_wo)));
            if (mlp) {  // gate_up + SwiGLU + down in one kernel, residual into the other buffer
                Q3_TRY(launch_mlp_fused(lc, r_cur, R, C, g_post, k.rms_eps, w_gu, (const bf16 *)(lw + L.o_wdownT), I,
                                        r_next, err, (const bf16 *)(ahead + L.o_wgu),
                                        (const bf16 *)(ahead + L.o_wdownT)));
            } else {
                Q3_TRY(launch_gemv_fused(lc, r_cur, R, C, w_gu, 2 * I, EPI_SWIGLU, act, g_post, k.rms_eps, err,
                                         (const bf16 *)(ahead + L.o_wgu)));
                Q3_TRY(launch_gemv_fused(lc, act, R, I, w_down, C, EPI_RESID_ADD, r_cur, nullptr, 0.0f, err,
                                         (const bf16 *)(ahead + L.o_wdown)));
            }
        } else if (decode) {
            // larger batches: RMSNorm kernels + tensor-core projections (32 rows at a time)
            auto proj = [&](const bf16 *X, int Kd, const bf16 *W, int N, int epi, void *out) -> cudaError_t {
                for (int m0 = 0; m0 < R; m0 += 32) {
                    const int mc = std::min(32, R - m0);
                    const bf16 *Xc = X + (size_t)m0 * Kd;
                    void *oc = epi == EPI_SWIGLU ? (void *)((bf16 *)out + (size_t)m0 * (N / 2))
                                                 : (void *)((float *)out + (size_t)m0 * N);
                    cudaError_t e = gemv_mma_supported(mc, Kd, N) ? launch_gemv_mma(lc, Xc, mc, Kd, W, N, epi, oc, err)
                                                                  : launch_gemv(lc, Xc, mc, Kd, W, N, epi, oc);
                    if (e != cudaSuccess) return e;
                }
                return cudaSuccess;
            };
            if (l > 0) Q3_TRY(launch_rmsnorm(lc, resid, R, g_in, xn, C, k.rms_eps));
            Q3_TRY(proj(xn, C, w_qkv, qkv_n, EPI_F32, qkv));
            Q3_TRY(decode_attention(c, lc, qkv, rows, g_q, g_k, rope, l, n_split, attn, err));
            Q3_TRY(proj(attn, Hq * D, w_o, C, EPI_RESID_ADD, resid));
            Q3_TRY(launch_rmsnorm(lc, resid, R, g_post, xn, C, k.rms_eps));
            Q3_TRY(proj(xn, C, w_gu, 2 * I, EPI_SWIGLU, act));
            Q3_TRY(proj(act, I, w_down, C, EPI_RESID_ADD, resid));
        } else {
            // prefill: tensor-core GEMMs (tcgen05, TMA) where the shape allows, else mma.sync
            auto gemm = [&](const bf16 *X, int Kd, const bf16 *W, int N, int epi, void *out) {
                return gemm_tc_supported(R, Kd, N) ? launch_gemm_tc(lc, X, R, Kd, W, N, epi, out, err)
                                                   : launch_gemm(lc, X, R, Kd, W, N, epi, out);
            };
            // All four projections on the tensor cores: both RMSNorms ride in the GEMM epilogues.
            // The residual-add GEMM before a norm leaves bf16(h * gamma) in xn and the sums of
            // squares of h in ss_*; the GEMM after it scales its rows by rsqrt(mean + eps).
            const bool tc_norm = gemm_tc_supported(R, C, qkv_n) && gemm_tc_supported(R, Hq * D, C) &&
                                 gemm_tc_supported(R, C, 2 * I) && gemm_tc_supported(R, I, C) && C % 128 == 0;
            float *ss_in = c->at<float>(L.o_ssp);
            float *ss_post = ss_in + (size_t)std::max(k.max_prefill_tokens, k.max_seqs) * (C / 128);
            if (tc_norm) {
                // layer 0's operand comes normalised from the embedding kernel
                Q3_TRY(launch_gemm_tc_qkv(lc, xn, R, C, w_qkv, qkv_n, rows, g_q, g_k, rope_t, q, c->kcache(l),
                                          c->vcache(l), Hq, Hkv, k.max_ctx, k.rms_eps, err,
                                          l > 0 ? ss_in : nullptr));
                if (attn_prefill_tc_supported(Hq, Hkv))
                    Q3_TRY(launch_attn_prefill_tc(lc, q, R, c->kcache(l), c->vcache(l), rows.cu_seqlens, rows.slots,
                                                  rows.row_pos, rows.B, max_len, k.max_seqs, attn, Hq, Hkv,
                                                  k.max_ctx, err, rows.kv, L.kv_layer_bytes / (D * 2)));
                else
                    Q3_TRY(rows.kv.table ? cudaErrorNotSupported :  // the mma.sync kernel reads a contiguous cache
                           launch_attn_prefill(lc, q, c->kcache(l), c->vcache(l), rows.cu_seqlens, rows.slots,
                                               rows.B, max_len, attn, Hq, Hkv, k.max_ctx));
                RowNorm post;
                post.ss_out = ss_post;
                post.xn_out = xn;
                post.gamma_out = g_post;
                post.norm_c = C;
                post.eps = k.rms_eps;
                Q3_TRY(launch_gemm_tc(lc, attn, R, Hq * D, w_o, C, EPI_RESID_ADD, resid, err, post));
                RowNorm mlp_in;
                mlp_in.ss_in = ss_post;
                mlp_in.norm_c = C;
                mlp_in.eps = k.rms_eps;
                Q3_TRY(launch_gemm_tc(lc, xn, R, C, w_gu, 2 * I, EPI_SWIGLU, act, err, mlp_in));
                RowNorm next;  // the next layer's input norm (none after the last layer)
                if (l + 1 < k.n_layers) {
                    next.ss_out = ss_in;
                    next.xn_out = xn;
                    next.gamma_out = (const float *)(c->layer(l + 1) + L.o_gin);
                    next.norm_c = C;
                    next.eps = k.rms_eps;
                }
                Q3_TRY(launch_gemm_tc(lc, act, R, I, w_down, C, EPI_RESID_ADD, resid, err, next));
                Q3_TRY(dump(l + 1, resid));
                continue;
            }
            if (l > 0) Q3_TRY(launch_rmsnorm(lc, resid, R, g_in, xn, C, k.rms_eps));
            if (gemm_tc_supported(R, C, qkv_n)) {  // QK-norm, RoPE and the KV write in the GEMM epilogue
                Q3_TRY(launch_gemm_tc_qkv(lc, xn, R, C, w_qkv, qkv_n, rows, g_q, g_k, rope_t, q, c->kcache(l),
                                          c->vcache(l), Hq, Hkv, k.max_ctx, k.rms_eps, err));
            } else {
                Q3_TRY(gemm(xn, C, w_qkv, qkv_n, EPI_F32, qkv));
                Q3_TRY(rows.kv.table ? cudaErrorNotSupported :  // writes a contiguous cache
                       launch_qknorm_rope_kv(lc, qkv, rows, g_q, g_k, rope, q, c->kcache(l), c->vcache(l), Hq,
                                             Hkv, k.max_ctx, k.rms_eps, err));
            }
            if (attn_prefill_tc_supported(Hq, Hkv))
                Q3_TRY(launch_attn_prefill_tc(lc, q, R, c->kcache(l), c->vcache(l), rows.cu_seqlens, rows.slots,
                                              rows.row_pos, rows.B, max_len, k.max_seqs, attn, Hq, Hkv, k.max_ctx,
                                              err, rows.kv, L.kv_layer_bytes / (D * 2)));
            else
                Q3_TRY(rows.kv.table ? cudaErrorNotSupported :
                       launch_attn_prefill(lc, q, c->kcache(l), c->vcache(l), rows.cu_seqlens, rows.slots, rows.B,
                                           max_len, attn, Hq, Hkv, k.max_ctx));
            Q3_TRY(gemm(attn, Hq * D, w_o, C, EPI_RESID_ADD, resid));
            Q3_TRY(launch_rmsnorm(lc, resid, R, g_post, xn, C, k.rms_eps));
            Q3_TRY(gemm(xn, C, w_gu, 2 * I, EPI_SWIGLU, act));
            Q3_TRY(gemm(act, I, w_down, C, EPI_RESID_ADD, resid));
        }
        Q3_TRY(dump(l + 1, mlp ? res[(l + 1) & 1] : resid));
    }
    bf16 *last = c->at<bf16>(L.o_last);
    Q3_TRY(launch_final_norm(lc, mlp ? res[k.n_layers & 1] : resid, rows.cu_seqlens, rows.B,
                             c->at<float>(L.o_gfinal), last, C, k.rms_eps));
    Q3_TRY(launch_lmhead_argmax(lc, last, rows.B, C, embed, k.vocab, logits, c->at<float>(L.o_pval),
                                c->at<int32_t>(L.o_pidx), c->n_parts, next, rows, err));
    return draw_next(c, lc, logits, rows.B, next);
}

Rows make_rows(qwen3_ctx *c, const int32_t *cu, const int32_t *slots, int B, int rows) {
    Rows r;
    r.cu_seqlens = cu;
    r.slots = slots;
    r.row_slot = c->at<int32_t>(c->lay.o_rowslot);
    r.row_pos = c->at<int32_t>(c->lay.o_rowpos);
    r.ctx_len = c->at<int32_t>(c->lay.o_ctxlen);
    r.B = B;
    r.rows = rows;
    if (c->cfg.kv_block_tokens > 0) {
        r.kv.table = c->at<int32_t>(c->lay.o_kvtable);
        r.kv.max_blocks = c->lay.kv_max_blocks;
        r.kv.bs = c->cfg.kv_block_tokens;
    }
    return r;
}

bool kv_paged(const qwen3_ctx *c) { return c->cfg.kv_block_tokens > 0; }

// Gives back every block of `slot` (paged cache; host bookkeeping only).
void kv_release(qwen3_ctx *c, int slot) {
    const int mb = c->lay.kv_max_blocks;
    for (int i = c->kv_nblk[slot] - 1; i >= 0; --i) c->kv_free.push_back(c->kv_table[(size_t)slot * mb + i]);
    c->kv_nblk[slot] = 0;
}

// Makes each slots[b] hold blocks for positions 0 .. new_len[b]-1 (restart: its old blocks
// are given back first), then copies the changed table rows to the device in stream order.
// Nothing changes when the free blocks do not suffice.
int kv_reserve(qwen3_ctx *c, const int32_t *slots, const int *new_len, int B, bool restart, cudaStream_t st) {
    if (!kv_paged(c)) return QWEN3_OK;
    const int bs = c->cfg.kv_block_tokens, mb = c->lay.kv_max_blocks;
    long need = 0, avail = (long)c->kv_free.size();
    for (int b = 0; b < B; ++b) {
        const int have = c->kv_nblk[slots[b]];
        const int want = (new_len[b] + bs - 1) / bs;
        if (restart) {
            avail += have;
            need += want;
        } else {
            need += std::max(0, want - have);
        }
    }
    if (need > avail) return c->fail(QWEN3_E_CAPACITY, "paged KV cache: not enough free blocks");
    for (int b = 0; b < B; ++b) {
        const int slot = slots[b];
        if (restart) kv_release(c, slot);
        const int have = c->kv_nblk[slot];
        const int want = (new_len[b] + bs - 1) / bs;
        if (want <= have) continue;
        for (int i = have; i < want; ++i) {
            c->kv_table[(size_t)slot * mb + i] = c->kv_free.back();
            c->kv_free.pop_back();
        }
        c->kv_nblk[slot] = want;
        // pageable source: the copy is staged before the call returns
        const cudaError_t e = cudaMemcpyAsync(c->at<int32_t>(c->lay.o_kvtable) + (size_t)slot * mb + have,
                                              c->kv_table.data() + (size_t)slot * mb + have,
                                              (size_t)(want - have) * 4, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return c->cuda_fail(e, "paged KV cache: block table upload");
    }
    return QWEN3_OK;
}

int check_slots(qwen3_ctx *c, const int32_t *slots_host, int B) {
    std::vector<char> seen(c->cfg.max_seqs, 0);
    for (int b = 0; b < B; ++b) {
        const int s = slots_host[b];
        if (s < 0 || s >= c->cfg.max_seqs) return c->fail(QWEN3_E_INVALID, "slot out of range");
        if (seen[s]) return c->fail(QWEN3_E_INVALID, "slot repeated within one call");
        seen[s] = 1;
    }
    return QWEN3_OK;
}

}  // namespace

extern "C" {

size_t qwen3_arena_bytes(const qwen3_config *cfg) {
    if (!cfg || !config_supported(*cfg, nullptr)) return 0;
    return make_layout(*cfg).total;
}

int qwen3_create(const qwen3_config *cfg, const qwen3_weights *w, void *arena_dev,
                 size_t arena_bytes, void *stream_v, qwen3_ctx **out) {
    g_create_error.clear();
    auto fail = [](int code, const std::string &m) {
        g_create_error = m;
        return code;
    };
    if (!cfg || !w || !arena_dev || !out) return fail(QWEN3_E_INVALID, "NULL argument");
    *out = nullptr;
    std::string why;
    if (!config_supported(*cfg, &why)) return fail(QWEN3_E_UNSUPPORTED, why);
    const Layout lay = make_layout(*cfg);
    if (arena_bytes < lay.total) return fail(QWEN3_E_INVALID, "arena smaller than qwen3_arena_bytes()");
    if (reinterpret_cast<uintptr_t>(arena_dev) % 256) return fail(QWEN3_E_INVALID, "arena not 256-byte aligned");
    if (!w->embed || !w->final_norm || !w->in_norm || !w->post_norm || !w->q_norm || !w->k_norm ||
        !w->wq || !w->wk || !w->wv || !w->wo || !w->wgate || !w->wup || !w->wdown)
        return fail(QWEN3_E_INVALID, "NULL weight pointer");
    for (int l = 0; l < cfg->n_layers; ++l)
        if (!w->in_norm[l] || !w->post_norm[l] || !w->q_norm[l] || !w->k_norm[l] || !w->wq[l] ||
            !w->wk[l] || !w->wv[l] || !w->wo[l] || !w->wgate[l] || !w->wup[l] || !w->wdown[l])
            return fail(QWEN3_E_INVALID, "NULL per-layer weight pointer");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(QWEN3_E_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return fail(QWEN3_E_CUDA, std::string("cudaGetDeviceProperties: ") + cudaGetErrorString(e));
    if (prop.major != 10 || prop.minor != 3)
        return fail(QWEN3_E_UNSUPPORTED, "this build targets compute capability 10.3 (sm_103a)");

    qwen3_ctx *c = new qwen3_ctx();
    c->cfg = *cfg;
    c->lay = lay;
    c->arena = static_cast<uint8_t *>(arena_dev);
    c->len_host.assign(cfg->max_seqs, 0);
    if (cfg->kv_block_tokens > 0) {
        c->kv_table.assign((size_t)cfg->max_seqs * lay.kv_max_blocks, 0);
        c->kv_nblk.assign(cfg->max_seqs, 0);
        for (int i = 0; i < cfg->kv_pool_blocks; ++i) c->kv_free.push_back(i);  // the highest block goes first
    }
    c->num_sms = prop.multiProcessorCount;
    c->n_parts = std::min(lmhead_parts(c->num_sms), MAX_PARTS);
    c->attn_ctas_per_sm = attn_decode_ctas_per_sm(cfg->n_q_heads, cfg->n_kv_heads);
    cudaStream_t st = static_cast<cudaStream_t>(stream_v);
    Launch lc;
    lc.stream = st;
    lc.pdl = false;
    lc.num_sms = c->num_sms;
    lc.counter = &c->launches;

    const size_t C = cfg->hidden, D = cfg->head_dim, Hq = cfg->n_q_heads, Hkv = cfg->n_kv_heads,
                 I = cfg->intermediate;
    auto d2d = [&](void *dst, const void *src, size_t bytes) {
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
    };
    auto body = [&]() -> cudaError_t {
        for (int l = 0; l < cfg->n_layers; ++l) {
            uint8_t *lw = c->layer(l);
            // QKV rows stacked [q; k; v]
            Q3_TRY(d2d(lw + lay.o_wqkv, w->wq[l], Hq * D * C * 2));
            Q3_TRY(d2d(lw + lay.o_wqkv + Hq * D * C * 2, w->wk[l], Hkv * D * C * 2));
            Q3_TRY(d2d(lw + lay.o_wqkv + (Hq + Hkv) * D * C * 2, w->wv[l], Hkv * D * C * 2));
            Q3_TRY(d2d(lw + lay.o_wo, w->wo[l], C * Hq * D * 2));
            // the same o_proj with the columns of each KV head's query heads stored together
            const size_t gcols = Hq / Hkv * D;
            for (size_t g = 0; g < Hkv; ++g)
                Q3_TRY(cudaMemcpy2DAsync(lw + lay.o_wog + g * C * gcols * 2, gcols * 2,
                                         (const bf16 *)w->wo[l] + g * gcols, Hq * D * 2, gcols * 2, C,
                                         cudaMemcpyDeviceToDevice, st));
            // gate/up interleaved row by row: row 2j = gate_j, row 2j+1 = up_j
            Q3_TRY(cudaMemcpy2DAsync(lw + lay.o_wgu, 2 * C * 2, w->wgate[l], C * 2, C * 2, I,
                                     cudaMemcpyDeviceToDevice, st));
            Q3_TRY(cudaMemcpy2DAsync(lw + lay.o_wgu + C * 2, 2 * C * 2, w->wup[l], C * 2, C * 2, I,
                                     cudaMemcpyDeviceToDevice, st));
            Q3_TRY(d2d(lw + lay.o_wdown, w->wdown[l], C * I * 2));
            Q3_TRY(launch_transpose_bf16(lc, (const bf16 *)w->wdown[l], (bf16 *)(lw + lay.o_wdownT), (int)C, (int)I));
            Q3_TRY(launch_bf16_to_f32(lc, (const bf16 *)w->in_norm[l], (float *)(lw + lay.o_gin), (int)C));
            Q3_TRY(launch_bf16_to_f32(lc, (const bf16 *)w->post_norm[l], (float *)(lw + lay.o_gpost), (int)C));
            Q3_TRY(launch_bf16_to_f32(lc, (const bf16 *)w->q_norm[l], (float *)(lw + lay.o_gq), (int)D));
            Q3_TRY(launch_bf16_to_f32(lc, (const bf16 *)w->k_norm[l], (float *)(lw + lay.o_gk), (int)D));
        }
        Q3_TRY(d2d(c->arena + lay.o_embed, w->embed, (size_t)cfg->vocab * C * 2));
        Q3_TRY(launch_bf16_to_f32(lc, (const bf16 *)w->final_norm, c->at<float>(lay.o_gfinal), (int)C));
        // RoPE table: (cos, sin) of p * theta^(-2i/D), i < D/2, computed in double precision
        std::vector<float2> tab((size_t)cfg->max_ctx * (D / 2));
        for (int p = 0; p < cfg->max_ctx; ++p)
            for (size_t i = 0; i < D / 2; ++i) {
                const double inv_freq = std::pow(cfg->rope_theta, -2.0 * (double)i / (double)D);
                const double a = (double)p * inv_freq;
                tab[(size_t)p * (D / 2) + i] = make_float2((float)std::cos(a), (float)std::sin(a));
            }
        Q3_TRY(cudaMemcpyAsync(c->arena + lay.o_rope, tab.data(), tab.size() * sizeof(float2),
                               cudaMemcpyHostToDevice, st));
        // [D/4][max_ctx] of (cos, sin) of frequencies 2k, 2k+1: rows at consecutive positions read
        // neighbouring 16-byte entries
        std::vector<float4> tab_t(tab.size() / 2);
        for (int p = 0; p < cfg->max_ctx; ++p)
            for (size_t k = 0; k < D / 4; ++k) {
                const float2 a = tab[(size_t)p * (D / 2) + 2 * k], b = tab[(size_t)p * (D / 2) + 2 * k + 1];
                tab_t[k * cfg->max_ctx + p] = make_float4(a.x, a.y, b.x, b.y);
            }
        Q3_TRY(cudaMemcpyAsync(c->arena + lay.o_rope_t, tab_t.data(), tab_t.size() * sizeof(float4),
                               cudaMemcpyHostToDevice, st));
        // The KV cache starts at zero: the tensor-core prefill attention multiplies whole
        // 128-key tiles, so rows past a sequence's end (weight 0) must hold finite values --
        // zeros, or an earlier sequence's keys and values.
        Q3_TRY(cudaMemsetAsync(c->arena + lay.o_kcache, 0, lay.kv_layer_bytes * cfg->n_layers, st));
        Q3_TRY(cudaMemsetAsync(c->arena + lay.o_vcache, 0, lay.kv_layer_bytes * cfg->n_layers, st));
        Q3_TRY(cudaMemsetAsync(c->arena + lay.o_ctxlen, 0, (size_t)cfg->max_seqs * 4, st));
        if (cfg->kv_block_tokens > 0)  // unused entries name block 0: never read for a position a slot lacks
            Q3_TRY(cudaMemsetAsync(c->arena + lay.o_kvtable, 0, (size_t)cfg->max_seqs * lay.kv_max_blocks * 4, st));
        Q3_TRY(cudaMemsetAsync(c->arena + lay.o_err, 0, 16, st));
        Q3_TRY(cudaMemsetAsync(c->arena + lay.o_counters, 0, (size_t)cfg->max_seqs * cfg->n_kv_heads * 4, st));
        Q3_TRY(cudaMemsetAsync(c->arena + lay.o_pres, 0, (size_t)3 * cfg->max_seqs * C * 4, st));
        Q3_TRY(cudaStreamSynchronize(st));
        return cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking);
    };
    e = body();
    if (e != cudaSuccess) {
        delete c;
        return fail(QWEN3_E_CUDA, std::string("qwen3_create: ") + cudaGetErrorString(e));
    }
    *out = c;
    return QWEN3_OK;
}

namespace {

// qwen3_prefill (append = false: every slot restarts at position 0) and qwen3_prefill_append
// (the rows continue each slot after the tokens it holds).
int prefill_impl(qwen3_ctx *c, const int32_t *tokens_dev, const int32_t *cu_dev, const int32_t *cu_host,
                 const int32_t *slots_dev, const int32_t *slots_host, int32_t B, float *logits_dev,
                 int32_t *next_tok_dev, void *stream_v, bool append) {
    if (!c) return QWEN3_E_INVALID;
    if (!tokens_dev || !cu_dev || !cu_host || !slots_dev || !slots_host || !next_tok_dev)
        return c->fail(QWEN3_E_INVALID, "NULL argument");
    if (B < 1) return c->fail(QWEN3_E_INVALID, "B must be >= 1");
    if (B > c->cfg.max_seqs) return c->fail(QWEN3_E_CAPACITY, "B exceeds max_seqs");
    if (sampling_on(c) && !logits_dev) return c->fail(QWEN3_E_INVALID, "sampling needs the logits buffer");
    if (cu_host[0] != 0) return c->fail(QWEN3_E_INVALID, "cu_seqlens[0] must be 0");
    if (int rc = check_slots(c, slots_host, B)) return rc;
    int max_len = 0;
    for (int b = 0; b < B; ++b) {
        const int n = cu_host[b + 1] - cu_host[b];
        if (n < 1) return c->fail(QWEN3_E_INVALID, "cu_seqlens must be strictly increasing");
        const int held = append ? c->len_host[slots_host[b]] : 0;
        if (held + n > c->cfg.max_ctx) return c->fail(QWEN3_E_CAPACITY, "sequence longer than max_ctx");
        max_len = std::max(max_len, n);
    }
    const int N = cu_host[B];
    if (N > c->cfg.max_prefill_tokens) return c->fail(QWEN3_E_CAPACITY, "N exceeds max_prefill_tokens");
    if (append && !attn_prefill_tc_supported(c->cfg.n_q_heads, c->cfg.n_kv_heads))
        return c->fail(QWEN3_E_UNSUPPORTED, "appending to a slot needs the tensor-core prefill attention");
    if (c->dump && c->dump_bytes < (size_t)(c->cfg.n_layers + 1) * N * c->cfg.hidden * 4)
        return c->fail(QWEN3_E_CAPACITY, "debug dump buffer too small for this call");

    Launch lc;
    lc.stream = static_cast<cudaStream_t>(stream_v);
    lc.pdl = !(c->cfg.flags & QWEN3_FLAG_NO_PDL);
    lc.num_sms = c->num_sms;
    lc.counter = &c->launches;
    if (kv_paged(c)) {
        std::vector<int> new_len(B);
        for (int b = 0; b < B; ++b)
            new_len[b] = (append ? c->len_host[slots_host[b]] : 0) + cu_host[b + 1] - cu_host[b];
        if (int rc = kv_reserve(c, slots_host, new_len.data(), B, !append, lc.stream)) return rc;
    }
    Rows rows = make_rows(c, cu_dev, slots_dev, B, N);
    rows.append = append;
    cudaError_t e = run_forward(c, lc, tokens_dev, rows, false, max_len, 0, logits_dev, next_tok_dev);
    if (e != cudaSuccess) return c->cuda_fail(e, append ? "qwen3_prefill_append" : "qwen3_prefill");
    for (int b = 0; b < B; ++b)
        c->len_host[slots_host[b]] = (append ? c->len_host[slots_host[b]] : 0) + cu_host[b + 1] - cu_host[b];
    return QWEN3_OK;
}

}  // namespace

int qwen3_prefill(qwen3_ctx *c, const int32_t *tokens_dev, const int32_t *cu_dev,
                  const int32_t *cu_host, const int32_t *slots_dev, const int32_t *slots_host,
                  int32_t B, float *logits_dev, int32_t *next_tok_dev, void *stream_v) {
    return prefill_impl(c, tokens_dev, cu_dev, cu_host, slots_dev, slots_host, B, logits_dev, next_tok_dev, stream_v,
                        false);
}

int qwen3_prefill_append(qwen3_ctx *c, const int32_t *tokens_dev, const int32_t *cu_dev,
                         const int32_t *cu_host, const int32_t *slots_dev, const int32_t *slots_host,
                         int32_t B, float *logits_dev, int32_t *next_tok_dev, void *stream_v) {
    return prefill_impl(c, tokens_dev, cu_dev, cu_host, slots_dev, slots_host, B, logits_dev, next_tok_dev, stream_v,
                        true);
}

int qwen3_decode_step(qwen3_ctx *c, const int32_t *tokens_dev, const int32_t *slots_dev,
                      const int32_t *slots_host, int32_t B, float *logits_dev,
                      int32_t *next_tok_dev, void *stream_v) {
    if (!c) return QWEN3_E_INVALID;
    if (!tokens_dev || !slots_dev || !slots_host || !next_tok_dev)
        return c->fail(QWEN3_E_INVALID, "NULL argument");
    if (B < 1) return c->fail(QWEN3_E_INVALID, "B must be >= 1");
    if (B > c->cfg.max_seqs) return c->fail(QWEN3_E_CAPACITY, "B exceeds max_seqs");
    if (sampling_on(c) && !logits_dev) return c->fail(QWEN3_E_INVALID, "sampling needs the logits buffer");
    if (int rc = check_slots(c, slots_host, B)) return rc;
    int max_len = 0;
    for (int b = 0; b < B; ++b) {
        const int n = c->len_host[slots_host[b]];
        if (n < 1) return c->fail(QWEN3_E_INVALID, "slot has not been prefilled");
        if (n + 1 > c->cfg.max_ctx) return c->fail(QWEN3_E_CAPACITY, "slot already holds max_ctx tokens");
        max_len = std::max(max_len, n + 1);
    }
    if (c->dump && c->dump_bytes < (size_t)(c->cfg.n_layers + 1) * B * c->cfg.hidden * 4)
        return c->fail(QWEN3_E_CAPACITY, "debug dump buffer too small for this call");

    const int n_split =
        plan_decode_attention(c->num_sms, c->attn_ctas_per_sm, B, c->cfg.n_kv_heads, max_len, c->cfg.max_ctx);

    cudaStream_t st = static_cast<cudaStream_t>(stream_v);
    if (kv_paged(c)) {  // a block for the appended position where a slot's last block is full
        std::vector<int> new_len(B);
        for (int b = 0; b < B; ++b) new_len[b] = c->len_host[slots_host[b]] + 1;
        if (int rc = kv_reserve(c, slots_host, new_len.data(), B, false, st)) return rc;
    }
    const Rows rows = make_rows(c, nullptr, slots_dev, B, B);
    const bool use_graph = !(c->cfg.flags & QWEN3_FLAG_NO_GRAPH) && !c->dump;
    if (!use_graph) {
        Launch lc;
        lc.stream = st;
        lc.pdl = !(c->cfg.flags & QWEN3_FLAG_NO_PDL);
        lc.num_sms = c->num_sms;
        lc.counter = &c->launches;
        cudaError_t e = run_forward(c, lc, tokens_dev, rows, true, 0, n_split, logits_dev, next_tok_dev);
        if (e != cudaSuccess) return c->cuda_fail(e, "qwen3_decode_step");
    } else {
        GraphEntry *g = nullptr;
        for (auto &x : c->graphs)
            if (x.B == B && x.n_split == n_split && x.tokens == tokens_dev &&
                x.slots == slots_dev && x.logits == logits_dev && x.next == next_tok_dev &&
                !memcmp(&x.sampling, &c->sampling, sizeof(qwen3_sampling)))
                g = &x;
        if (!g) {
            Launch lc;
            lc.stream = c->cap_stream;
            lc.pdl = !(c->cfg.flags & QWEN3_FLAG_NO_PDL);
            lc.num_sms = c->num_sms;
            cudaError_t e = cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal);
            if (e != cudaSuccess) return c->cuda_fail(e, "cudaStreamBeginCapture");
            e = run_forward(c, lc, tokens_dev, rows, true, 0, n_split, logits_dev, next_tok_dev);
            cudaGraph_t graph = nullptr;
            const cudaError_t e2 = cudaStreamEndCapture(c->cap_stream, &graph);
            if (e != cudaSuccess || e2 != cudaSuccess) {
                if (graph) cudaGraphDestroy(graph);
                return c->cuda_fail(e != cudaSuccess ? e : e2, "decode graph capture");
            }
            cudaGraphExec_t exec = nullptr;
            e = cudaGraphInstantiate(&exec, graph, 0);
            size_t n_nodes = 0;
            if (e == cudaSuccess) e = cudaGraphGetNodes(graph, nullptr, &n_nodes);
            std::vector<cudaGraphNode_t> nodes(n_nodes);
            int64_t kernels = 0;
            if (e == cudaSuccess && n_nodes) e = cudaGraphGetNodes(graph, nodes.data(), &n_nodes);
            for (size_t i = 0; e == cudaSuccess && i < n_nodes; ++i) {
                cudaGraphNodeType t;
                e = cudaGraphNodeGetType(nodes[i], &t);
                if (t == cudaGraphNodeTypeKernel) ++kernels;
            }
            cudaGraphDestroy(graph);
            if (e != cudaSuccess) {
                if (exec) cudaGraphExecDestroy(exec);
                return c->cuda_fail(e, "decode graph instantiate");
            }
            c->graphs.push_back(GraphEntry{B, n_split, tokens_dev, slots_dev, logits_dev,
                                           next_tok_dev, c->sampling, exec, kernels});
            g = &c->graphs.back();
        }
        cudaError_t e = cudaGraphLaunch(g->exec, st);
        if (e != cudaSuccess) return c->cuda_fail(e, "cudaGraphLaunch");
        c->launches += g->kernels;
    }
    for (int b = 0; b < B; ++b) c->len_host[slots_host[b]] += 1;
    return QWEN3_OK;
}

int qwen3_set_sampling(qwen3_ctx *c, const qwen3_sampling *sp) {
    if (!c) return QWEN3_E_INVALID;
    if (!sp || !sp->temperature) {
        c->sampling = qwen3_sampling{};
        return QWEN3_OK;
    }
    if (!sp->top_k || !sp->top_p || !sp->uniform)
        return c->fail(QWEN3_E_INVALID, "qwen3_set_sampling: NULL array");
    if (!sample_supported(c->cfg.vocab))
        return c->fail(QWEN3_E_UNSUPPORTED, "qwen3_set_sampling: vocabulary too large for the sampler");
    c->sampling = *sp;
    return QWEN3_OK;
}

int qwen3_set_debug_dump(qwen3_ctx *c, float *hidden_dev, size_t bytes) {
    if (!c) return QWEN3_E_INVALID;
    c->dump = hidden_dev;
    c->dump_bytes = hidden_dev ? bytes : 0;
    return QWEN3_OK;
}

int qwen3_get_status(qwen3_ctx *c) {
    if (!c) return QWEN3_E_INVALID;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return c->cuda_fail(e, "qwen3_get_status");
    uint32_t word = 0;
    e = cudaMemcpy(&word, c->arena + c->lay.o_err, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return c->cuda_fail(e, "qwen3_get_status");
    if (word) {
        cudaMemset(c->arena + c->lay.o_err, 0, 4);
        std::string m = "device error word set:";
        if (word & ERR_TOKEN_RANGE) m += " token id out of range (clamped);";
        if (word & ERR_POSITION) m += " position beyond max_ctx (KV write skipped);";
        if (word & ERR_TIMEOUT) {
            m += " a bounded wait in a kernel gave up (outputs of that call are not valid);";
            // the decode attention's merge counters may be left mid-count
            cudaMemset(c->arena + c->lay.o_counters, 0, (size_t)c->cfg.max_seqs * c->cfg.n_kv_heads * 4);
        }
        return c->fail(QWEN3_E_DEVICE, m);
    }
    return QWEN3_OK;
}

const char *qwen3_last_error(const qwen3_ctx *c) {
    return c ? c->err.c_str() : g_create_error.c_str();
}

int32_t qwen3_slot_length(const qwen3_ctx *c, int32_t slot) {
    if (!c || slot < 0 || slot >= c->cfg.max_seqs) return -1;
    return c->len_host[slot];
}

int qwen3_kv_view(const qwen3_ctx *c, int32_t layer, int32_t slot, const void **k_dev,
                  const void **v_dev) {
    if (!c || !k_dev || !v_dev) return QWEN3_E_INVALID;
    if (layer < 0 || layer >= c->cfg.n_layers || slot < 0 || slot >= c->cfg.max_seqs)
        return QWEN3_E_INVALID;
    if (kv_paged(c)) return QWEN3_E_UNSUPPORTED;
    const size_t per_slot = (size_t)c->cfg.n_kv_heads * c->cfg.max_ctx * c->cfg.head_dim;
    *k_dev = c->kcache(layer) + (size_t)slot * per_slot;
    *v_dev = c->vcache(layer) + (size_t)slot * per_slot;
    return QWEN3_OK;
}

int64_t qwen3_launch_count(const qwen3_ctx *c) { return c ? c->launches : 0; }

int qwen3_get_config(const qwen3_ctx *c, qwen3_config *cfg) {
    if (!c || !cfg) return QWEN3_E_INVALID;
    *cfg = c->cfg;
    return QWEN3_OK;
}

int qwen3_release_slot(qwen3_ctx *c, int32_t slot, void *stream) {
    if (!c) return QWEN3_E_INVALID;
    if (slot < 0 || slot >= c->cfg.max_seqs) return c->fail(QWEN3_E_INVALID, "qwen3_release_slot: slot out of range");
    const cudaError_t e = cudaMemsetAsync(c->at<int32_t>(c->lay.o_ctxlen) + slot, 0, sizeof(int32_t),
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return c->cuda_fail(e, "qwen3_release_slot");
    c->len_host[slot] = 0;
    if (kv_paged(c)) kv_release(c, slot);
    return QWEN3_OK;
}

int qwen3_kv_copy_rows(const qwen3_ctx *c, int32_t layer, int32_t slot, int32_t pos0, int32_t n, void *k_out,
                       void *v_out, void *stream) {
    if (!c || !k_out || !v_out) return QWEN3_E_INVALID;
    if (layer < 0 || layer >= c->cfg.n_layers || slot < 0 || slot >= c->cfg.max_seqs || pos0 < 0 || n < 1 ||
        pos0 + n > c->len_host[slot])
        return QWEN3_E_INVALID;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int Hkv = c->cfg.n_kv_heads, D = c->cfg.head_dim, mb = c->lay.kv_max_blocks;
    const int bs = kv_paged(c) ? c->cfg.kv_block_tokens : c->cfg.max_ctx;
    for (int g = 0; g < Hkv; ++g)
        for (int p = pos0; p < pos0 + n;) {  // runs of rows inside one block (one run when contiguous)
            const int run = std::min(pos0 + n - p, bs - p % bs);
            const size_t row = kv_paged(c)
                                   ? ((size_t)c->kv_table[(size_t)slot * mb + p / bs] * Hkv + g) * bs + p % bs
                                   : ((size_t)slot * Hkv + g) * c->cfg.max_ctx + p;
            const size_t dst = ((size_t)g * n + (p - pos0)) * D;
            for (int kv = 0; kv < 2; ++kv) {
                const bf16 *src = (kv ? c->vcache(layer) : c->kcache(layer)) + row * D;
                bf16 *out = static_cast<bf16 *>(kv ? v_out : k_out) + dst;
                const cudaError_t e = cudaMemcpyAsync(out, src, (size_t)run * D * 2, cudaMemcpyDeviceToDevice, st);
                if (e != cudaSuccess) return QWEN3_E_CUDA;
            }
            p += run;
        }
    return QWEN3_OK;
}

int32_t qwen3_kv_free_blocks(const qwen3_ctx *c) {
    if (!c || !kv_paged(c)) return -1;
    return (int32_t)c->kv_free.size();
}

static bool gemv_k_ok(int K) {
    return K == 256 || K == 512 || K == 768 || K == 1024 || K == 1536 || K == 2048 || K == 2560 ||
           K == 3072 || K == 4096;
}

static Launch op_launch(void *stream) {
    Launch lc;
    lc.stream = static_cast<cudaStream_t>(stream);
    lc.pdl = false;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&lc.num_sms, cudaDevAttrMultiProcessorCount, dev);
    return lc;
}

int qwen3_op_gemv(const void *x, int32_t M, int32_t K, const void *w, int32_t N, int32_t epi,
                  void *out, void *stream) {
    g_create_error.clear();
    if (!x || !w || !out || M < 1 || N < 2 || N % 2 || !gemv_k_ok(K) || epi < 0 || epi > 2) {
        g_create_error = "qwen3_op_gemv: bad argument";
        return QWEN3_E_INVALID;
    }
    const Launch lc = op_launch(stream);
    cudaError_t e;
    if (gemv_fused_supported(M, K))
        e = launch_gemv_fused(lc, x, M, K, (const bf16 *)w, N, epi, out, nullptr, 0.0f, nullptr);
    else if (gemv_mma_supported(M, K, N) && (K <= 2048 || epi == EPI_RESID_ADD))
        e = launch_gemv_mma(lc, (const bf16 *)x, M, K, (const bf16 *)w, N, epi, out, nullptr);
    else
        e = launch_gemv(lc, (const bf16 *)x, M, K, (const bf16 *)w, N, epi, out);
    if (e != cudaSuccess) {
        g_create_error = std::string("qwen3_op_gemv: ") + cudaGetErrorString(e);
        return QWEN3_E_CUDA;
    }
    return QWEN3_OK;
}

int qwen3_op_mlp_decode(const float *h, int32_t M, int32_t C, const float *gain, float eps, const void *w_gu,
                        const void *w_dt, int32_t I, float *out, void *stream) {
    g_create_error.clear();
    if (!h || !gain || !w_gu || !w_dt || !out || M < 1 || C < 1 || I < 1 || I % 256 || !(eps >= 0.0f)) {
        g_create_error = "qwen3_op_mlp_decode: bad argument";
        return QWEN3_E_INVALID;
    }
    const Launch lc = op_launch(stream);
    if (!mlp_fused_supported(M, C, I, lc.num_sms)) {
        g_create_error = "qwen3_op_mlp_decode: unsupported size (M <= 4, C == 1024)";
        return QWEN3_E_UNSUPPORTED;
    }
    const cudaError_t e = launch_mlp_fused(lc, h, M, C, gain, eps, (const bf16 *)w_gu, (const bf16 *)w_dt, I, out,
                                           nullptr, nullptr, nullptr);
    if (e != cudaSuccess) {
        g_create_error = std::string("qwen3_op_mlp_decode: ") + cudaGetErrorString(e);
        return QWEN3_E_CUDA;
    }
    return QWEN3_OK;
}

int qwen3_op_gemm(const void *x, int32_t M, int32_t K, const void *w, int32_t N, int32_t epi,
                  void *out, void *stream) {
    g_create_error.clear();
    if (!x || !w || !out || M < 1 || N < 128 || N % 128 || K < 32 || K % 32 || epi < 0 || epi > 2) {
        g_create_error = "qwen3_op_gemm: bad argument";
        return QWEN3_E_INVALID;
    }
    // operands and output move by TMA / 16-byte vector accesses
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(out)) & 15) {
        g_create_error = "qwen3_op_gemm: x, w and out must be 16-byte aligned";
        return QWEN3_E_INVALID;
    }
    const Launch lc = op_launch(stream);
    cudaError_t e = gemm_tc_supported(M, K, N)
                        ? launch_gemm_tc(lc, (const bf16 *)x, M, K, (const bf16 *)w, N, epi, out, nullptr)
                        : launch_gemm(lc, (const bf16 *)x, M, K, (const bf16 *)w, N, epi, out);
    if (e != cudaSuccess) {
        g_create_error = std::string("qwen3_op_gemm: ") + cudaGetErrorString(e);
        return QWEN3_E_CUDA;
    }
    return QWEN3_OK;
}

size_t qwen3_op_lmhead_workspace_bytes(int32_t B) {
    if (B < 1 || B > 1024) return 0;
    return (size_t)B * MAX_PARTS * 8;
}

int qwen3_op_lmhead_argmax(const void *x, int32_t B, int32_t C, const void *embed, int32_t V,
                           float *logits, int32_t *next_tok, void *ws, size_t ws_bytes,
                           void *stream) {
    g_create_error.clear();
    if (!x || !embed || !next_tok || !ws || B < 1 || B > 1024 || V < 1 || !gemv_k_ok(C) ||
        C > 3072 || reinterpret_cast<uintptr_t>(ws) % 16 || ws_bytes < qwen3_op_lmhead_workspace_bytes(B)) {
        g_create_error = "qwen3_op_lmhead_argmax: bad argument";
        return QWEN3_E_INVALID;
    }
    const Launch lc = op_launch(stream);
    const int n_parts = std::min(lmhead_parts(lc.num_sms), MAX_PARTS);
    float *pval = static_cast<float *>(ws);
    int32_t *pidx = reinterpret_cast<int32_t *>(pval + (size_t)B * MAX_PARTS);
    Rows r;  // no KV bookkeeping for a bare call
    r.B = B;
    r.rows = B;
    cudaError_t e = launch_lmhead_argmax(lc, (const bf16 *)x, B, C, (const bf16 *)embed, V, logits,
                                         pval, pidx, n_parts, next_tok, r);
    if (e != cudaSuccess) {
        g_create_error = std::string("qwen3_op_lmhead_argmax: ") + cudaGetErrorString(e);
        return QWEN3_E_CUDA;
    }
    return QWEN3_OK;
}

int qwen3_set_wait_limit(qwen3_ctx *c, uint32_t cycles) {
    if (!c) return QWEN3_E_INVALID;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(c->arena + c->lay.o_err + 4, &cycles, 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return c->cuda_fail(e, "qwen3_set_wait_limit");
    return QWEN3_OK;
}

int qwen3_truncate_slot(qwen3_ctx *c, int32_t slot, int32_t length, void *stream) {
    if (!c) return QWEN3_E_INVALID;
    if (slot < 0 || slot >= c->cfg.max_seqs) return c->fail(QWEN3_E_INVALID, "qwen3_truncate_slot: slot out of range");
    if (length < 0 || length > c->len_host[slot])
        return c->fail(QWEN3_E_INVALID, "qwen3_truncate_slot: length outside [0, the slot's length]");
    // pageable source: the copy is staged before the call returns
    const cudaError_t e = cudaMemcpyAsync(c->at<int32_t>(c->lay.o_ctxlen) + slot, &length, sizeof(int32_t),
                                          cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return c->cuda_fail(e, "qwen3_truncate_slot");
    c->len_host[slot] = length;
    if (kv_paged(c)) {  // give back the blocks past the kept positions, last block first
        const int bs = c->cfg.kv_block_tokens, mb = c->lay.kv_max_blocks;
        const int keep = (length + bs - 1) / bs;
        for (int i = c->kv_nblk[slot] - 1; i >= keep; --i) c->kv_free.push_back(c->kv_table[(size_t)slot * mb + i]);
        c->kv_nblk[slot] = std::min(c->kv_nblk[slot], keep);
    }
    return QWEN3_OK;
}

size_t qwen3_op_attn_decode_workspace_bytes(int32_t B, int32_t n_q_heads, int32_t n_kv_heads) {
    if (B < 1 || B > 1024 || n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads) return 0;
    const size_t D = 128;
    return align_up((size_t)B * n_q_heads * MAX_SPLIT * 2 * 4) + align_up((size_t)B * n_q_heads * MAX_SPLIT * D * 4) +
           align_up((size_t)B * n_kv_heads * 4);
}

int32_t qwen3_op_attn_decode_plan(int32_t B, int32_t n_q_heads, int32_t n_kv_heads, int32_t max_len,
                                  int32_t max_ctx) {
    g_create_error.clear();
    if (B < 1 || B > 1024 || n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads || max_len < 1 ||
        max_ctx < max_len) {
        g_create_error = "qwen3_op_attn_decode_plan: bad argument";
        return QWEN3_E_INVALID;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        g_create_error = std::string("qwen3_op_attn_decode_plan: ") + cudaGetErrorString(e);
        return QWEN3_E_CUDA;
    }
    return plan_decode_attention(sms, attn_decode_ctas_per_sm(n_q_heads, n_kv_heads), B, n_kv_heads, max_len,
                                 max_ctx);
}

int qwen3_op_attn_decode(const float *qkv, int32_t B, const int32_t *slots, const int32_t *slots_host,
                         const int32_t *positions, const int32_t *positions_host, const float *q_gain,
                         const float *k_gain, const float *rope, void *k_cache, void *v_cache, int32_t n_slots,
                         int32_t max_ctx, int32_t n_q_heads, int32_t n_kv_heads, float eps, int32_t n_split, void *out,
                         void *ws, size_t ws_bytes, void *stream) {
    g_create_error.clear();
    const int g = n_kv_heads > 0 ? n_q_heads / n_kv_heads : 0;
    if (!qkv || !slots || !slots_host || !positions || !positions_host || !q_gain || !k_gain || !rope || !k_cache ||
        !v_cache || !out || !ws ||
        B < 1 || n_slots < 1 || max_ctx < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads ||
        (g != 1 && g != 2 && g != 4 && g != 8) || n_split < 0 || n_split > MAX_SPLIT || !(eps >= 0.0f) ||
        reinterpret_cast<uintptr_t>(ws) % 256 || ws_bytes < qwen3_op_attn_decode_workspace_bytes(B, n_q_heads, n_kv_heads)) {
        g_create_error = "qwen3_op_attn_decode: bad argument";
        return QWEN3_E_INVALID;
    }
    for (int b = 0; b < B; ++b)
        if (slots_host[b] < 0 || slots_host[b] >= n_slots || positions_host[b] < 0 || positions_host[b] >= max_ctx) {
            g_create_error = "qwen3_op_attn_decode: slot or position out of range";
            return QWEN3_E_INVALID;
        }
    const Launch lc = op_launch(stream);
    if (n_split == 0)  // as a decode step plans it for rows whose longest context is the largest position + 1
        n_split = plan_decode_attention(lc.num_sms, attn_decode_ctas_per_sm(n_q_heads, n_kv_heads), B, n_kv_heads,
                                        *std::max_element(positions_host, positions_host + B) + 1, max_ctx);
    const size_t D = 128;
    float *ws_ml = static_cast<float *>(ws);
    float *ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + align_up((size_t)B * n_q_heads * MAX_SPLIT * 2 * 4));
    int *counters = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(ws_o) + align_up((size_t)B * n_q_heads * MAX_SPLIT * D * 4));
    Rows r;
    r.slots = slots;
    r.row_slot = const_cast<int32_t *>(slots);
    r.row_pos = const_cast<int32_t *>(positions);
    r.B = B;
    r.rows = B;
    const cudaError_t e = launch_attn_decode_fused(
        lc, qkv, r, q_gain, k_gain, reinterpret_cast<const float2 *>(rope), static_cast<bf16 *>(k_cache),
        static_cast<bf16 *>(v_cache), (size_t)n_slots * n_kv_heads * max_ctx, n_split, ws_ml, ws_o, counters,
        static_cast<bf16 *>(out), n_q_heads, n_kv_heads, max_ctx, eps, nullptr);
    if (e != cudaSuccess) {
        g_create_error = std::string("qwen3_op_attn_decode: ") + cudaGetErrorString(e);
        return QWEN3_E_CUDA;
    }
    return QWEN3_OK;
}

void qwen3_free(qwen3_ctx *c) {
    if (!c) return;
    for (auto &g : c->graphs) cudaGraphExecDestroy(g.exec);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    delete c;
}

}  // extern "C"
