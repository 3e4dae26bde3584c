// Host-side launchers of the Qwen3 decoder-forward kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <unordered_set>
#include <utility>

#include "common.cuh"

namespace q3 {

struct Launch {
    cudaStream_t stream = nullptr;
    bool pdl = true;          // programmatic dependent launch on every kernel
    int num_sms = 148;
    int64_t *counter = nullptr;
};

// Every kernel asks for the largest shared-memory carveout, so that the L1/shared split is the
// same for all of them and a kernel launched early under programmatic dependent launch can
// be resident on an SM next to its predecessor.
inline cudaError_t prefer_max_shared(const void *kern) {
    static std::mutex mu;
    static std::unordered_set<const void *> done;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(kern)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) done.insert(kern);
    return e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch(const Launch &lc, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   Args &&...args) {
    cudaError_t pe = prefer_max_shared(reinterpret_cast<const void *>(kern));
    if (pe != cudaSuccess) return pe;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    if (lc.counter) ++*lc.counter;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The same, for a kernel launched as clusters of `cluster` CTAs (grid a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(const Launch &lc, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           dim3 cluster, Args &&...args) {
    cudaError_t pe = prefer_max_shared(reinterpret_cast<const void *>(kern));
    if (pe != cudaSuccess) return pe;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster.x;
    attr[0].val.clusterDim.y = cluster.y;
    attr[0].val.clusterDim.z = cluster.z;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = lc.pdl ? 2 : 1;
    if (lc.counter) ++*lc.counter;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Where the cached K (or V) row of (slot, KV head g, position p) lives, in rows of D elements
// from the layer's base.  Contiguous (table == nullptr): [slot][Hkv][max_ctx][D].  Paged:
// blocks of bs positions, [block][Hkv][bs][D], the block of position p of a slot being
// table[slot * max_blocks + p / bs]; the host fills the table for every position a call can
// touch before launching it.
struct KvMap {
    const int32_t *table = nullptr;
    int32_t max_blocks = 0;
    int32_t bs = 0;
};

// The table is read through L2 (ld.global.cg): kernels may read it before their dependency
// wait, when this SM's L1 could still hold an older copy of the line.
__device__ __forceinline__ size_t kv_row(const KvMap &m, int slot, int Hkv, int g, int max_ctx, int p) {
    if (!m.table) return ((size_t)slot * Hkv + g) * max_ctx + p;
    const int blk = __ldcg(m.table + (size_t)slot * m.max_blocks + p / m.bs);
    return ((size_t)blk * Hkv + g) * m.bs + p % m.bs;
}

// Row bookkeeping of one call: row r of the packed batch belongs to KV slot row_slot[r]
// at absolute position row_pos[r].
struct Rows {
    const int32_t *cu_seqlens = nullptr;  // [B+1] for prefill, nullptr for decode (one row per sequence)
    const int32_t *slots = nullptr;       // [B]
    int32_t *row_slot = nullptr;          // [rows] written by the embedding kernel
    int32_t *row_pos = nullptr;           // [rows]
    int32_t *ctx_len = nullptr;           // [max_seqs] tokens cached per slot (nullptr: no bookkeeping)
    bool append = false;                  // prefill rows continue their slot: positions start at ctx_len
    int32_t B = 0;
    int32_t rows = 0;
    KvMap kv;                             // where the cache rows of the slots live
};

// --- norm.cu ---------------------------------------------------------------------------
// zero_buf (may be null): rows [rows, C] fp32 cleared for a kernel that accumulates into them.
cudaError_t launch_embed_rmsnorm(const Launch &lc, const int32_t *tokens, const Rows &r,
                                 const bf16 *embed, const float *gamma, float *resid, bf16 *xn,
                                 int C, int V, float eps, uint32_t *err, float *zero_buf = nullptr);
cudaError_t launch_rmsnorm(const Launch &lc, const float *resid, int rows, const float *gamma,
                           bf16 *xn, int C, float eps);
// Final norm of each sequence's last row: row cu_seqlens[b+1]-1 (or b) -> out[b].
cudaError_t launch_final_norm(const Launch &lc, const float *resid, const int32_t *cu_seqlens,
                              int B, const float *gamma, bf16 *out, int C, float eps);
cudaError_t launch_bf16_to_f32(const Launch &lc, const bf16 *src, float *dst, int n);

// --- gemm.cu (prefill; out[M,N] = A[M,K] W[N,K]^T) -----------------------------------------
enum Epilogue : int {
    EPI_F32 = 0,         // out fp32 [M, N]
    EPI_RESID_ADD = 1,   // out fp32 [M, N] += result
    EPI_SWIGLU = 2,      // W rows interleaved (gate_j, up_j): out bf16 [M, N/2] = silu(g)*u
    EPI_QKV = 3,         // QKV projection straight into q (normed, rotated) and the KV cache
};
cudaError_t launch_gemm(const Launch &lc, const bf16 *A, int M, int K, const bf16 *W, int N,
                        int epi, void *out);

// --- gemm_tc.cu (prefill on tcgen05 tensor cores; K % 64 == 0, N % 256 == 0) -------------
bool gemm_tc_supported(int M, int K, int N);
// RMSNorm folded into the projections around it ("第 3 章", 3.2: the norm between the
// residual add and the next projection).  The residual-add GEMM writes, besides h, the bf16
// operand h * gamma_out (xn_out [M, N]) and the sums of squares of h over each 128 columns
// (ss_out [M, N / 128]); the next GEMM reads that operand and multiplies row r of its product
// by rsqrt(sum(ss_in[r][*]) / norm_c + eps), which equals projecting RMSNorm(h) * gamma.
struct RowNorm {
    const float *ss_in = nullptr;    // SwiGLU (and QKV): scale rows by the norm of their input
    float *ss_out = nullptr;         // residual add: per-128-column sums of squares of h
    bf16 *xn_out = nullptr;          // residual add: bf16 h * gamma_out
    const float *gamma_out = nullptr;
    int norm_c = 0;                  // the normalised width (K of the consuming GEMM)
    float eps = 0.0f;
};
cudaError_t launch_gemm_tc(const Launch &lc, const bf16 *A, int M, int K, const bf16 *W, int N, int epi,
                           void *out, uint32_t *err, const RowNorm &rn = RowNorm());
// QKV projection with the epilogue of launch_qknorm_rope_kv fused in (no fp32 qkv buffer).
// rope_t is the RoPE table by pairs of frequencies: (cos, sin) of frequencies 2k and 2k+1 at
// position p at rope_t[k * max_ctx + p], k < 64 / 2.
cudaError_t launch_gemm_tc_qkv(const Launch &lc, const bf16 *A, int M, int K, const bf16 *W, int N, const Rows &r,
                               const float *q_gain, const float *k_gain, const float4 *rope_t, bf16 *q_out,
                               bf16 *k_layer, bf16 *v_layer, int Hq, int Hkv, int max_ctx, float eps,
                               uint32_t *err, const float *ss_in = nullptr);

// --- gemv.cu (decode; same contract as launch_gemm for small M) ---------------------------
cudaError_t launch_gemv(const Launch &lc, const bf16 *X, int M, int K, const bf16 *W, int N,
                        int epi, void *out);
// M <= 8 rows: the weight block of each CTA is bulk-copied before the dependency wait.  With
// norm_gain, X is fp32 residual rows [M, K] normalised (RMSNorm, eps) on the way in; else X is
// bf16 [M, K].  W_ahead (same shape as W, may be null): weights of a later launch whose
// matching block each CTA asks L2 to fetch now.
bool gemv_fused_supported(int M, int K);
cudaError_t launch_gemv_fused(const Launch &lc, const void *X, int M, int K, const bf16 *W, int N,
                              int epi, void *out, const float *norm_gain, float eps, uint32_t *err,
                              const bf16 *W_ahead = nullptr, float *zero_buf = nullptr, int zero_n = 0);
// The decode MLP in one kernel (M <= 4 rows, C == 1024): out += h + down(silu(gate m) * up m),
// m = RMSNorm(h), with the down projection split over CTAs and added with fp32 atomics; out
// must be zero on entry.  WdT is the down weight transposed ([I, C]).
bool mlp_fused_supported(int M, int C, int I, int num_sms);
cudaError_t launch_mlp_fused(const Launch &lc, const float *h, int M, int C, const float *gain, float eps,
                             const bf16 *Wgu, const bf16 *WdT, int I, float *out, uint32_t *err,
                             const bf16 *Wgu_ahead, const bf16 *WdT_ahead);
cudaError_t launch_transpose_bf16(const Launch &lc, const bf16 *src, bf16 *dst, int rows, int cols);
// Tensor-core (mma.sync) decode projection for up to 32 rows.  With EPI_RESID_ADD the K range is
// split over 2 or 4 CTAs whose partial sums add into the output with fp32 atomics (order
// unspecified); the other epilogues keep K in one slice (K <= 2048).
bool gemv_mma_supported(int M, int K, int N);
// lm_head + argmax pass 1 on the tensor cores for 1..32 rows (C == 1024): one partial (best
// value, index) per CTA and row, as launch_lmhead_argmax's pass 1 writes them.
cudaError_t launch_lmhead_mma(const Launch &lc, const bf16 *X, int M, int C, const bf16 *E, int V, float *logits,
                              float *part_val, int32_t *part_idx, int n_parts, uint32_t *err);
// CTAs (and partials per row) of launch_lmhead_mma: one per SM.
int lmhead_mma_parts(int num_sms);
cudaError_t launch_gemv_mma(const Launch &lc, const bf16 *X, int M, int K, const bf16 *W, int N, int epi,
                            void *out, uint32_t *err);

// --- rope_kv.cu --------------------------------------------------------------------------
// qkv fp32 [rows, (Hq+2Hkv)*D] -> q bf16 [rows, Hq, D] (normed + rotated), K (normed +
// rotated) and V into the layer's cache [slot][Hkv][max_ctx][D].
cudaError_t launch_qknorm_rope_kv(const Launch &lc, const float *qkv, const Rows &r,
                                  const float *q_gain, const float *k_gain, const float2 *rope,
                                  bf16 *q_out, bf16 *k_layer, bf16 *v_layer, int Hq, int Hkv,
                                  int max_ctx, float eps, uint32_t *err);

// --- attn_prefill.cu ---------------------------------------------------------------------
cudaError_t launch_attn_prefill(const Launch &lc, const bf16 *q, const bf16 *k_layer,
                                const bf16 *v_layer, const int32_t *cu_seqlens,
                                const int32_t *slots, int B, int max_len, bf16 *out, int Hq,
                                int Hkv, int max_ctx);

// --- attn_prefill_tc.cu (tcgen05 flash attention; q has N rows) ----------------------------
// Tensor map of a layer's K or V rows ([rows][128] bf16): boxes of 64 rows x 64 columns with
// the 128-byte swizzle (the decode attention's chunks).
bool kv_tile_map(CUtensorMap *m, const bf16 *base, uint64_t rows);
bool attn_prefill_tc_supported(int Hq, int Hkv);
// Rows of sequence b are positions row_pos[cu[b]] .. of its slot (non-zero when a call
// continues a slot); keys come from the cache, causal mask aligned bottom-right.
// kv_rows: rows of the layer's K (and V) array (tensor-map extent); a paged kv needs bs % 128 == 0.
cudaError_t launch_attn_prefill_tc(const Launch &lc, const bf16 *q, int N, const bf16 *k_layer,
                                   const bf16 *v_layer, const int32_t *cu_seqlens, const int32_t *slots,
                                   const int32_t *row_pos, int B, int max_len, int max_seqs, bf16 *out, int Hq,
                                   int Hkv, int max_ctx, uint32_t *err, const KvMap &kv = KvMap(),
                                   size_t kv_rows = 0);

// --- attn_decode.cu ----------------------------------------------------------------------
// Most key ranges per (sequence, KV head) of the decode attention.
constexpr int ATTN_DECODE_MAX_SPLIT = 64;
// CTAs of the decode attention that one SM holds at once.
int attn_decode_ctas_per_sm(int Hq, int Hkv);

// Decode attention fed directly by the QKV projection (fp32 [B, (Hq+2Hkv)*D]): per-head
// QK-norm + RoPE + KV-cache write of the new row, attention over keys 0..pos, and the
// merge of the n_split key ranges (balanced over keys 0..pos on the device) by the last CTA
// of each (sequence, KV head).  counters
// [max_seqs * Hkv] must be zero on entry and are left zero.
// kv_rows: rows ([128] bf16) of the layer's K and V arrays, the extent of their tensor maps.
cudaError_t launch_attn_decode_fused(const Launch &lc, const float *qkv, const Rows &r,
                                     const float *q_gain, const float *k_gain, const float2 *rope,
                                     bf16 *k_layer, bf16 *v_layer, size_t kv_rows, int n_split,
                                     float *ws_ml, float *ws_o, int *counters, bf16 *out, int Hq,
                                     int Hkv, int max_ctx, float eps, uint32_t *err);

// --- decode_block.cu (decode of 1-2 rows: one attention-block and one MLP-block kernel per layer)
// Hidden 1024, head_dim 128, two query heads per KV head.  Row b appends to slot slots[b] at
// position ctx_len[slots[b]].
struct AttnBlockParams {
    const float *h_in;      // [B, C] residual entering the layer
    float *h_out;           // [B, C] += h_in + o_proj(attention); zero on entry
    float *zero_next;       // [B, C] cleared here (the MLP block's output)
    const float *g_in;      // [C] input_layernorm gain
    const bf16 *wqkv;       // [(Hq + 2 Hkv) D, C]
    const bf16 *wog;        // [Hkv][C][2 D]: o_proj, the columns of each KV head's query heads together
    const float *g_q, *g_k; // [D]
    const float2 *rope;     // [max_ctx][D/2] (cos, sin)
    bf16 *k_layer, *v_layer;
    const int32_t *slots;   // [B]
    const int32_t *ctx_len; // [max_seqs]
    KvMap kv;
    const bf16 *ahead_gu, *ahead_dt;  // this layer's MLP weights, asked of L2 (may be null)
    int B, Hq, Hkv, max_ctx, I;
    float eps, scale_log2;
    uint32_t *err;
};
struct MlpBlockParams {
    const float *h_in;      // [B, C] residual after attention
    float *h_out;           // [B, C] += h_in + MLP(h_in); zero on entry
    float *zero_next;       // [B, C] cleared here (the next attention block's output)
    const float *gain;      // [C] post_attention_layernorm gain
    const bf16 *wgu;        // [2I, C] gate/up rows interleaved
    const bf16 *wdt;        // [I, C] down weight transposed
    const bf16 *ahead_qkv, *ahead_og;  // the next layer's attention weights, asked of L2 (may be null)
    int qkv_rows, og_cols;  // their sizes: rows of C elements
    int B, C, I, NA;        // NA set by the launcher
    float eps;
    uint32_t *err;
};
bool decode_block_supported(int B, int C, int Hq, int Hkv, int head_dim, int I, int num_sms);
size_t attn_block_smem(int B);
cudaError_t launch_attn_block(const Launch &lc, const AttnBlockParams &p);
cudaError_t launch_mlp_block(const Launch &lc, const MlpBlockParams &p);

// --- sample.cu ---------------------------------------------------------------------------
// Temperature / top-k / top-p draw of next_tok[b] from logits fp32 [B, V] (the rule of
// qwen3_sample); launched without programmatic dependent launch, after the lm_head.
bool sample_supported(int V);
cudaError_t launch_sample(const Launch &lc, const float *logits, int B, int V, const float *temperature,
                          const int32_t *top_k, const float *top_p, const float *uniform, int32_t *next_tok);

// --- lmhead.cu ---------------------------------------------------------------------------
// next_tok[b] = argmax_v X[b] . E[v] (lowest index on ties); logits[B, V] if not null.
// Also sets ctx_len[slot] = position + 1 of each sequence's last row.
cudaError_t launch_lmhead_argmax(const Launch &lc, const bf16 *X, int B, int C, const bf16 *E,
                                 int V, float *logits, float *part_val, int32_t *part_idx,
                                 int n_parts, int32_t *next_tok, const Rows &r, uint32_t *err = nullptr);
int lmhead_parts(int num_sms);

}  // namespace q3
