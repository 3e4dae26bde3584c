/*
 * qwen3_gb300.h -- C ABI of a single-GPU (sm_103a) Qwen3-0.6B-style decoder forward.
 *
 * The forward computed here is the one hand-written in PyTorch by the pages
 *   "手写Qwen3-0.6B推理"                 (Qwen3Model, Qwen3DecoderLayer, Qwen3RMSNorm,
 *                                         Attention, Rope, MLP, 推理),
 *   "第 3 章 前向与生成（代码走读）"      (3.1 packed [N,C] tokens, 3.2 fused residual +
 *                                         RMSNorm, 3.3 QKV/RoPE/causal attention, 3.4 gated
 *                                         MLP, 4.1 last-position lm_head, 4.3 greedy sampler),
 *   "从零开始写Qwen3"                     (Attn: the decode-time causal alignment; rope),
 *   "古法手撕简易LLM推理器"               (核心计算函数与Transformer层: the KV cache;
 *                                         prefill与predict: prefill then one-token steps):
 *
 *   h_0 = E[id]                                     (no scaling)
 *   per layer:  u = RMSNorm(h; g_in)
 *               q,k,v = u Wq^T, u Wk^T, u Wv^T      (no bias)
 *               q,k  <- per-head RMSNorm (g_q, g_k), then rotate-half RoPE at the
 *                       absolute position p (pair (i, i+64), angle p * theta^(-2i/128))
 *               cache <- (k, v) at p;  o_h = softmax(q_h K_g^T / sqrt(128)) V_g over keys
 *                       0..p of the same sequence, g = h / (Hq/Hkv)
 *               h <- h + o Wo^T;  h <- h + Wdown(silu(Wgate m) * Wup m), m = RMSNorm(h; g_post)
 *   next token = argmax_v E_v . RMSNorm(h_L; g_final)   (tied head, lowest index on ties)
 *
 * Conventions common to every call
 *  - All pointers named *_dev are device pointers on the current CUDA device; *_host are
 *    host pointers.  The library never allocates device memory: the caller passes one
 *    arena (qwen3_arena_bytes) that holds packed weights, the RoPE table, the KV cache
 *    and all scratch, and must keep it alive until qwen3_free.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Calls that take a stream are asynchronous and stream-ordered; outputs are valid once
 *    the stream has been synchronised.  Calls on one context must not overlap.
 *  - Every call returns QWEN3_OK (0) or a negative QWEN3_E_* code; the message of the last
 *    failure is returned by qwen3_last_error.  No call aborts, throws or traps.
 *  - Token ids outside [0, vocab) are clamped on the device and flagged in the device
 *    error word, which qwen3_get_status reports.
 */
#ifndef QWEN3_GB300_H
#define QWEN3_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QWEN3_OK 0
#define QWEN3_E_INVALID (-1)     /* NULL pointer, bad size, bad order, bad slot */
#define QWEN3_E_CAPACITY (-2)    /* more tokens / sequences / context than the arena was sized for */
#define QWEN3_E_UNSUPPORTED (-3) /* shape or device this build does not implement */
#define QWEN3_E_CUDA (-4)        /* a CUDA runtime call failed */
#define QWEN3_E_DEVICE (-5)      /* the device error word was set (e.g. a token id out of range) */

/* qwen3_config.flags */
#define QWEN3_FLAG_NO_GRAPH 1u   /* launch decode steps one kernel at a time instead of a CUDA graph */
#define QWEN3_FLAG_NO_PDL 2u     /* launch kernels without programmatic dependent launch (for profilers) */
#define QWEN3_FLAG_DECODE_CHAIN 8u /* decode steps of one sequence as the four-kernel-per-layer
                                      chain instead of two kernels per layer (see qwen3_decode_step) */

/* Model and capacity.  Supported: head_dim == 128; n_q_heads a multiple of n_kv_heads with
 * n_q_heads / n_kv_heads <= 8; hidden, n_q_heads*head_dim and intermediate multiples of 256;
 * vocab >= 1.  Qwen3-0.6B: 28, 1024, 16, 8, 128, 3072, 151936, 1e-6, 1e6 ("古法手撕简易LLM推理器",
 * 处理参数和超参数). */
typedef struct qwen3_config {
    int32_t n_layers;
    int32_t hidden;        /* C */
    int32_t n_q_heads;     /* Hq */
    int32_t n_kv_heads;    /* Hkv */
    int32_t head_dim;      /* D */
    int32_t intermediate;  /* I */
    int32_t vocab;         /* V */
    float rms_eps;
    double rope_theta;
    int32_t max_seqs;            /* KV-cache slots; also the largest decode batch */
    int32_t max_ctx;             /* tokens per slot (prompt + generated) */
    int32_t max_prefill_tokens;  /* largest N of one qwen3_prefill call */
    uint32_t flags;              /* QWEN3_FLAG_* (other bits: E_UNSUPPORTED) */
    /* KV cache layout.  kv_block_tokens == 0: every slot owns max_ctx positions (max_seqs *
     * max_ctx rows per layer).  kv_block_tokens > 0 (a multiple of 128): a paged cache ("第 3 章",
     * the engine's KV-cache blocks) -- a pool of kv_pool_blocks blocks of kv_block_tokens
     * positions shared by all slots; a slot takes blocks as its length grows (any block of the
     * pool, in any order) and gives them back when it restarts or is released.  A call that
     * needs more blocks than are free fails with E_CAPACITY before it launches anything.
     * Paged needs n_q_heads == 2 * n_kv_heads. */
    int32_t kv_block_tokens;
    int32_t kv_pool_blocks;
} qwen3_config;

/* Weights: device pointers to bf16 tensors in the checkpoint's layout ([out, in] row-major
 * for matrices; "手写Qwen3-0.6B推理", 打印模型结构).  Per-layer members are HOST arrays of
 * n_layers device pointers.  Read only during qwen3_create (packed into the arena). */
typedef struct qwen3_weights {
    const void *embed;       /* [V, C]; also the lm_head (tied) */
    const void *final_norm;  /* [C] */
    const void *const *in_norm;    /* [C] per layer */
    const void *const *post_norm;  /* [C] */
    const void *const *q_norm;     /* [D] */
    const void *const *k_norm;     /* [D] */
    const void *const *wq;         /* [Hq*D, C] */
    const void *const *wk;         /* [Hkv*D, C] */
    const void *const *wv;         /* [Hkv*D, C] */
    const void *const *wo;         /* [C, Hq*D] */
    const void *const *wgate;      /* [I, C] */
    const void *const *wup;        /* [I, C] */
    const void *const *wdown;      /* [C, I] */
} qwen3_weights;

typedef struct qwen3_ctx qwen3_ctx; /* opaque, owned by the library (host memory) */

/* Bytes of device memory qwen3_create needs for this configuration (0 if the configuration
 * is invalid or unsupported).  Pure host arithmetic. */
size_t qwen3_arena_bytes(const qwen3_config *cfg);

/* Builds a context: validates cfg, packs the weights into `arena_dev` (256-byte aligned,
 * at least qwen3_arena_bytes(cfg) bytes), builds the RoPE table (angles in double
 * precision) and empties every KV slot.  Synchronises `stream` before returning, so the
 * weight buffers may be freed afterwards.  On success *out owns a context to be released
 * with qwen3_free.  Errors: E_INVALID (NULL argument, small arena), E_UNSUPPORTED (shape or
 * a device other than compute capability 10.3), E_CUDA. */
int qwen3_create(const qwen3_config *cfg, const qwen3_weights *w, void *arena_dev,
                 size_t arena_bytes, void *stream, qwen3_ctx **out);

/* Prefill ("第 3 章", 3.1 packed tokens; "古法手撕简易LLM推理器", prefill与predict):
 * B sequences packed in tokens_dev[N] (int32), sequence b being rows
 * cu_seqlens[b] .. cu_seqlens[b+1]-1 at positions 0 .. len_b-1.  Sequence b (re)starts KV
 * slot slots[b] and leaves it holding len_b tokens.  Writes next_tok_dev[b] (int32), the
 * greedy token after each sequence's last row ("第 3 章", 4.1), and, if logits_dev is not
 * NULL, the fp32 logits of those rows to logits_dev[B, V].  cu_seqlens and slots are given
 * twice, on the device and on the host (same values).  Errors: E_INVALID (NULL, B < 1,
 * cu_seqlens not starting at 0 or not increasing, repeated or out-of-range slot),
 * E_CAPACITY (B > max_seqs, N > max_prefill_tokens, len_b > max_ctx, a paged cache without
 * the free blocks the call needs), E_CUDA. */
int qwen3_prefill(qwen3_ctx *ctx, const int32_t *tokens_dev, const int32_t *cu_seqlens_dev,
                  const int32_t *cu_seqlens_host, const int32_t *slots_dev,
                  const int32_t *slots_host, int32_t B, float *logits_dev,
                  int32_t *next_tok_dev, void *stream);

/* Prefill that continues its slots ("从零开始写Qwen3", Attn: the causal mask of a query block
 * that follows cached keys; "古法手撕简易LLM推理器", prefill与predict: offset = the cache length):
 * the len_b tokens of sequence b are appended to slot slots[b] after the n_b tokens it holds
 * (n_b = 0 is allowed), at positions n_b .. n_b+len_b-1, each attending to keys 0 .. its own
 * position -- the cached prefix included -- and the slot then holds n_b + len_b tokens.
 * Chunked prefill: one long prompt can be fed in several calls, and prompts can be extended
 * after decode steps.  Arguments, outputs and errors as qwen3_prefill; E_CAPACITY when
 * n_b + len_b > max_ctx, E_UNSUPPORTED for head ratios other than Hq = 2 Hkv. */
int qwen3_prefill_append(qwen3_ctx *ctx, const int32_t *tokens_dev, const int32_t *cu_seqlens_dev,
                         const int32_t *cu_seqlens_host, const int32_t *slots_dev,
                         const int32_t *slots_host, int32_t B, float *logits_dev,
                         int32_t *next_tok_dev, void *stream);

/* One decode step ("古法手撕简易LLM推理器", predict): token tokens_dev[b] is appended to slot
 * slots[b] at position = the slot's current length, attends to keys 0..position, and
 * next_tok_dev[b] receives the greedy next token (logits_dev[B, V] too if not NULL).  Each
 * slot's length grows by one.  next_tok_dev may be passed as the next step's tokens_dev.
 * A step of one sequence at hidden 1024, head_dim 128 and two query heads per KV head runs each
 * layer as two kernels (the attention block as clusters of 8 CTAs per KV head, then the MLP
 * block), unless QWEN3_FLAG_DECODE_CHAIN is set; other steps run four or more kernels per
 * layer.  Unless QWEN3_FLAG_NO_GRAPH is set, the step's kernels are recorded once per (B,
 * pointers, split plan) as a CUDA graph and replayed.  Errors: E_INVALID (NULL, B < 1,
 * repeated slot, slot never prefilled), E_CAPACITY (B > max_seqs, a slot already holding
 * max_ctx tokens, a paged cache without a free block for a slot whose last block is full),
 * E_CUDA. */
int qwen3_decode_step(qwen3_ctx *ctx, const int32_t *tokens_dev, const int32_t *slots_dev,
                      const int32_t *slots_host, int32_t B, float *logits_dev,
                      int32_t *next_tok_dev, void *stream);

/* Debug dump of the residual stream: while hidden_dev is not NULL, every prefill and decode
 * call writes h_0 (the embedding rows) and h_l after each layer l, fp32, to
 * hidden_dev[(L+1), rows, C] where rows = N (prefill) or B (decode).  Needs
 * bytes >= (L+1)*rows*C*4 for the calls made, else those calls fail with E_CAPACITY.
 * Decode steps run without a graph while the dump is on.  NULL turns it off. */
int qwen3_set_debug_dump(qwen3_ctx *ctx, float *hidden_dev, size_t bytes);

/* Per-sequence sampling settings: device arrays indexed by the row of a call (row b of a
 * decode step is the sequence in slots[b]; row b of a prefill is sequence b).  The rule is
 * qwen3_sample's (below).  The library reads them on the stream when each call runs, so the
 * caller may rewrite the values (a fresh uniform draw per step, say) between calls in
 * stream order; the pointers themselves are captured into the decode graphs. */
typedef struct qwen3_sampling {
    const float *temperature;  /* fp32 [max_seqs]; <= 0 selects the argmax for that row */
    const int32_t *top_k;      /* int32 [max_seqs] */
    const float *top_p;        /* fp32 [max_seqs] */
    const float *uniform;      /* fp32 [max_seqs], each in [0, 1) */
} qwen3_sampling;

/* Next tokens drawn by sampling ("第 3 章", 4.3 Sampler): while set, every qwen3_prefill,
 * qwen3_prefill_append and qwen3_decode_step writes its logits and then replaces the greedy
 * next_tok_dev[b] by the qwen3_sample draw from them, in the same stream (inside the decode
 * graph).  Those calls then need a logits_dev buffer (E_INVALID otherwise).  sampling == NULL, or a NULL
 * temperature, returns to greedy next tokens.  The structure is copied; the arrays are
 * borrowed until the setting is replaced.  Errors: E_INVALID (a NULL array),
 * E_UNSUPPORTED (a vocabulary the sampler cannot hold). */
int qwen3_set_sampling(qwen3_ctx *ctx, const qwen3_sampling *sampling);

/* Synchronises the device, then returns QWEN3_OK, E_CUDA (a pending CUDA error) or E_DEVICE
 * (the device error word was set; the word is cleared).  The word records token ids out of
 * range (clamped), positions beyond max_ctx (KV write skipped) and bounded waits that gave up
 * (the outputs of the call they belong to are not valid; see qwen3_set_wait_limit). */
int qwen3_get_status(qwen3_ctx *ctx);

/* Failure detection.  Every wait of a kernel on an asynchronous copy or on another CTA is
 * bounded: past its limit the kernel records "a bounded wait gave up" in the device error word,
 * lets its own copies in flight land, and returns (no trap, no hang; qwen3_get_status then
 * reports E_DEVICE).  This sets the limit, in SM clock cycles, of the waits of the decode
 * kernels (the weight and KV-cache streams of qwen3_decode_step; graphs recorded earlier read
 * the new value when replayed); 0 restores the default of 2^31 cycles (about a second).  A
 * small limit makes those waits give up on purpose, to test the error path.  Synchronises the
 * device.  Errors: E_INVALID, E_CUDA. */
int qwen3_set_wait_limit(qwen3_ctx *ctx, uint32_t cycles);

/* Message of the last failed call on ctx (or of the last failed qwen3_create when ctx is NULL). */
const char *qwen3_last_error(const qwen3_ctx *ctx);

/* Host-side length of KV slot `slot` (tokens cached), or -1 for a bad slot. */
int32_t qwen3_slot_length(const qwen3_ctx *ctx, int32_t slot);

/* Device pointers to layer `layer`, slot `slot` of the KV cache: K and V are each
 * bf16 [Hkv][max_ctx][D] (rows 0..length-1 valid; K after q/k-norm and RoPE, V raw).
 * Read-only for the caller.  Errors: E_INVALID, E_UNSUPPORTED (a paged cache: the slot's
 * rows are not contiguous; use qwen3_kv_copy_rows). */
int qwen3_kv_view(const qwen3_ctx *ctx, int32_t layer, int32_t slot, const void **k_dev,
                  const void **v_dev);

/* Copies cached rows pos0 .. pos0+n-1 of (layer, slot) to k_out_dev and v_out_dev, each bf16
 * [Hkv][n][D] (K after q/k-norm and RoPE, V raw), in stream order; works for both cache
 * layouts.  Errors: E_INVALID (bad layer/slot, rows beyond the slot's length), E_CUDA. */
int qwen3_kv_copy_rows(const qwen3_ctx *ctx, int32_t layer, int32_t slot, int32_t pos0, int32_t n,
                       void *k_out_dev, void *v_out_dev, void *stream);

/* Free blocks of a paged cache (-1 for a contiguous one). */
int32_t qwen3_kv_free_blocks(const qwen3_ctx *ctx);

/* Number of kernels this context has launched so far (graph replays count every kernel
 * node of the graph). */
int64_t qwen3_launch_count(const qwen3_ctx *ctx);

/* Copies the context's configuration (as given to qwen3_create) to *cfg.  Errors: E_INVALID. */
int qwen3_get_config(const qwen3_ctx *ctx, qwen3_config *cfg);

/* Forgets the tokens KV slot `slot` holds: its length becomes 0 on the host and (in stream
 * order on `stream`) on the device, so that the next qwen3_prefill_append or qwen3_prefill
 * starts it at position 0 and decode steps reject it until then.  The cache rows keep their
 * old values (finite, never attended to).  Errors: E_INVALID (bad slot), E_CUDA. */
int qwen3_release_slot(qwen3_ctx *ctx, int32_t slot, void *stream);

/* Shortens KV slot `slot` to its first `length` tokens (0 <= length <= its current length), on
 * the host and, in stream order on `stream`, on the device: the next decode step or
 * qwen3_prefill_append continues at position `length` and overwrites the rows after it
 * ("古法手撕简易LLM推理器", prefill与predict: the position offset is the cached length).  Used
 * to rewind generated tokens (rejected drafts, a re-run of the same steps from one prompt).  A
 * paged cache gives back the blocks past the kept positions.  length 0 is qwen3_release_slot.
 * Errors: E_INVALID (bad slot or length), E_CUDA. */
int qwen3_truncate_slot(qwen3_ctx *ctx, int32_t slot, int32_t length, void *stream);

/* ---- Continuous batching ("第 3 章", the engine and its scheduler; "手写Qwen3-0.6B推理",
 * generation that stops at the end-of-sequence token) -------------------------------------
 * An engine runs requests (a prompt, a token limit, an end-of-sequence id) through one
 * context.  Each qwen3_engine_step schedules at most token_budget tokens:
 *   1. one token for every running request that has consumed its prompt (its last generated
 *      token, appended at its slot's length);
 *   2. the next chunk of every running request still in its prompt (chunked prefill);
 *   3. waiting requests, first come first served, each into a free slot, while slots and
 *      budget remain (a prompt longer than what is left is split over several steps).
 * If every scheduled row is a single generated token the step is one qwen3_decode_step;
 * otherwise it is one qwen3_prefill_append over all rows (prompt chunks and generated tokens
 * packed together).  A request whose prompt is complete takes the greedy next token of its
 * last row; it finishes on its eos_id (kept as its last token), after max_new_tokens
 * tokens, or when its slot is full, and its slot is released for the waiting requests.
 * The step synchronises `stream` once, to read the next tokens.
 * The engine owns every slot of the context, and its sampling setting, while it exists: a step
 * with a sampling request (qwen3_engine_submit_sampled) sets the per-row settings for that call
 * and clears them after it. */
typedef struct qwen3_engine qwen3_engine;

#define QWEN3_FINISH_NONE 0     /* waiting or running */
#define QWEN3_FINISH_EOS 1      /* generated its eos_id */
#define QWEN3_FINISH_LENGTH 2   /* generated max_new_tokens tokens */
#define QWEN3_FINISH_CONTEXT 3  /* its slot holds max_ctx tokens: nothing more can be appended */

typedef struct qwen3_engine_stats {
    int64_t steps;             /* steps that ran the model */
    int64_t mixed_steps;       /* of which prefill_append calls (prompt chunks, maybe generated tokens) */
    int64_t decode_steps;      /* of which decode-only calls */
    int64_t prompt_tokens;     /* prompt tokens run */
    int64_t generated_tokens;  /* tokens generated */
} qwen3_engine_stats;

/* Device workspace of an engine (token, offset, slot and next-token arrays). */
size_t qwen3_engine_workspace_bytes(const qwen3_ctx *ctx, int32_t token_budget);

/* token_budget: tokens per step, max_seqs <= token_budget <= max_prefill_tokens.  workspace_dev:
 * device memory of qwen3_engine_workspace_bytes bytes, 256-byte aligned, owned by the caller
 * and kept while the engine lives.  Errors: E_INVALID. */
int qwen3_engine_create(qwen3_ctx *ctx, int32_t token_budget, void *workspace_dev, size_t bytes,
                        qwen3_engine **out);

/* Queues a request.  prompt_host: host int32 [prompt_len] (copied), 1 <= prompt_len <= max_ctx;
 * max_new_tokens >= 1; eos_id < 0 for none.  request_id must not be queued already.
 * Errors: E_INVALID, E_CAPACITY (prompt longer than max_ctx). */
int qwen3_engine_submit(qwen3_engine *e, int64_t request_id, const int32_t *prompt_host, int32_t prompt_len,
                        int32_t max_new_tokens, int32_t eos_id);

/* One scheduling step (see above); *n_finished (if not NULL) receives how many requests
 * finished in it.  With nothing to run it returns QWEN3_OK at once.  Errors: those of the
 * context's calls (the engine's state is then undefined: free it). */
int qwen3_engine_step(qwen3_engine *e, void *stream, int32_t *n_finished);

/* Requests submitted and not finished. */
int32_t qwen3_engine_unfinished(const qwen3_engine *e);

/* qwen3_engine_submit for a request that samples ("第 3 章", 4.3 Sampler): its tokens are drawn
 * by the rule of qwen3_sample with this temperature, top_k and top_p (temperature <= 0: greedy,
 * as qwen3_engine_submit).  The uniform draw of its t-th generated token (t = 0, 1, ...) is
 * output t + 1 of the SplitMix64 generator started at state `seed` (state += 0x9E3779B97F4A7C15;
 * z = state; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB;
 * z ^= z>>31), taken as (z >> 40) / 2^24, so a request's tokens depend only on its own
 * settings and seed, not on what it was batched with.  Errors: those of qwen3_engine_submit,
 * E_INVALID for a NaN temperature or top_p. */
int qwen3_engine_submit_sampled(qwen3_engine *e, int64_t request_id, const int32_t *prompt_host,
                                int32_t prompt_len, int32_t max_new_tokens, int32_t eos_id, float temperature,
                                int32_t top_k, float top_p, uint64_t seed);

/* Tokens generated so far for request_id (up to capacity of them into tokens_host, which may
 * be NULL when capacity is 0), their count and the finish reason (QWEN3_FINISH_*).
 * Errors: E_INVALID (unknown id). */
int qwen3_engine_result(const qwen3_engine *e, int64_t request_id, int32_t *tokens_host, int32_t capacity,
                        int32_t *n_tokens, int32_t *finish_reason);

/* Drops the record of a finished request.  Errors: E_INVALID (unknown or unfinished id). */
int qwen3_engine_forget(qwen3_engine *e, int64_t request_id);

int qwen3_engine_get_stats(const qwen3_engine *e, qwen3_engine_stats *out);

/* The last step that ran the model: the request id of each of its rows (in row order; up to
 * capacity of them into ids_host, which may be NULL when capacity is 0), their count, and, if
 * a request of that step samples, *logits_dev = the fp32 logits [rows, V] its draws were taken
 * from (in the engine's workspace, valid until the next step; NULL for an all-greedy step).
 * For inspecting the distribution a token was drawn from.  Errors: E_INVALID. */
int qwen3_engine_last_step(const qwen3_engine *e, int64_t *ids_host, int32_t capacity, int32_t *n_rows,
                           const float **logits_dev);

/* Message of the engine's last failed call. */
const char *qwen3_engine_last_error(const qwen3_engine *e);

/* Frees the engine (not the workspace, not the context). */
void qwen3_engine_free(qwen3_engine *e);

/* ---- Single kernels, as the forward runs them (no context needed) ----------------------
 * These run one step of the forward on caller buffers, for per-kernel tests and timing.
 * All buffers are device memory; the calls are asynchronous on `stream`. */

#define QWEN3_EPI_F32 0        /* out fp32 [M, N] = X W^T */
#define QWEN3_EPI_RESID_ADD 1  /* out fp32 [M, N] += X W^T  (o_proj / down_proj into the residual) */
#define QWEN3_EPI_SWIGLU 2     /* W rows interleaved (gate_0, up_0, gate_1, up_1, ...):
                                  out bf16 [M, N/2] = silu(X Wg^T) * (X Wu^T)  ("手写Qwen3-0.6B推理", MLP) */

/* Decode projection (weight-streaming GEMV): X bf16 [M, K] row-major, W bf16 [N, K] row-major
 * ([out, in] as nn.Linear stores it, "手写Qwen3-0.6B推理", Attention/MLP), fp32 accumulation.
 * K must be 256, 512, 768, 1024, 1536, 2048, 2560, 3072 or 4096; N a multiple of 2; M >= 1
 * (processed in groups of 32 rows).  Errors: E_INVALID (NULL, bad size), E_CUDA. */
int qwen3_op_gemv(const void *x_dev, int32_t M, int32_t K, const void *w_dev, int32_t N,
                  int32_t epilogue, void *out_dev, void *stream);

/* The decode MLP of up to 4 rows in one kernel, as decode steps of up to 4 sequences run it
 * ("手写Qwen3-0.6B推理", MLP and Qwen3DecoderLayer's residual add; "第 3 章", 3.2/3.4):
 *   out[b] += h[b] + Wdown (silu(Wgate m[b]) * (Wup m[b])),  m[b] = RMSNorm(h[b]; gain),
 * with m and the activation rounded to bf16.  h_dev fp32 [M, C]; gain_dev fp32 [C];
 * w_gate_up_dev bf16 [2I, C] with the gate and up rows interleaved (gate_0, up_0, gate_1, ...);
 * w_down_t_dev bf16 [I, C], the down weight transposed; out_dev fp32 [M, C], accumulated into
 * (zero it for out = h + MLP(h)) with fp32 atomics in an unspecified order.  Supported:
 * 1 <= M <= 4, C == 1024, I a multiple of 256 whose per-SM share fits shared memory.
 * Errors: E_INVALID (NULL, bad size), E_UNSUPPORTED, E_CUDA. */
int qwen3_op_mlp_decode(const float *h_dev, int32_t M, int32_t C, const float *gain_dev, float eps,
                        const void *w_gate_up_dev, const void *w_down_t_dev, int32_t I, float *out_dev,
                        void *stream);

/* Prefill projection (tiled tensor-core GEMM), same operands and epilogues as qwen3_op_gemv;
 * N a multiple of 128, K a multiple of 32, any M >= 1; x_dev, w_dev and out_dev 16-byte
 * aligned (the residual of QWEN3_EPI_RESID_ADD is read and written as tiles).
 * Errors: E_INVALID (NULL, bad size, misaligned pointer), E_CUDA. */
int qwen3_op_gemm(const void *x_dev, int32_t M, int32_t K, const void *w_dev, int32_t N,
                  int32_t epilogue, void *out_dev, void *stream);

/* Bytes of workspace qwen3_op_lmhead_argmax needs for B rows. */
size_t qwen3_op_lmhead_workspace_bytes(int32_t B);

/* Tied lm_head + greedy argmax ("手写Qwen3-0.6B推理", Qwen3Model/推理; "第 3 章", 4.1 and 4.3):
 * next_tok[b] = argmax_v E[v] . x[b] (fp32 logits, lowest index on ties) for x bf16 [B, C]
 * (the final-normed last rows) and E bf16 [V, C]; logits_dev fp32 [B, V] is written when not
 * NULL.  `workspace_dev` (>= qwen3_op_lmhead_workspace_bytes(B) bytes, 16-byte aligned) holds
 * per-CTA partial maxima.  C one of 256, 512, 768, 1024, 1536, 2048, 2560, 3072; 1 <= B <= 1024.
 * A next_tok of -1 means a bounded wait of the tensor-core pass (C == 1024, 9 to 32 rows
 * per pass) gave up: that row's logits and token are not valid.
 * Errors: E_INVALID (NULL, bad size, small workspace), E_CUDA. */
int qwen3_op_lmhead_argmax(const void *x_dev, int32_t B, int32_t C, const void *embed_dev,
                           int32_t V, float *logits_dev, int32_t *next_tok_dev,
                           void *workspace_dev, size_t workspace_bytes, void *stream);

/* Allocation-free variant of qwen3_op_lmhead_argmax. The pages have no counterpart of
 * this call.
 *
 * It is for callers that cannot allocate device memory: code enqueuing work while a stream
 * is recorded into a CUDA graph (where cudaMalloc is refused or not recorded), plug-ins
 * inside a framework that owns all device allocations, and latency-critical loops that must
 * not call cudaMalloc/cudaFree (cudaFree synchronises the device).
 *
 * Scratch: the per-CTA partials live in a fixed 256 KiB array in the library's device
 * memory. Every GPU that loads the library holds it until the process exits. The array
 * limits B to at most 32 rows; a larger B fails with E_CAPACITY and a message naming the
 * limit. The call itself allocates nothing.
 *
 * Set-up: the first call on each device looks up the array's address with that device
 * current, so make that first call before any stream capture.  The address is kept for the
 * life of the process: do not call this again on a device after a cudaDeviceReset of it.
 *
 * Sharing: all calls on a device share the array, and it keeps the last call's contents.
 * Every partial a call reads is written by that same call, so nothing needs clearing.
 * Calls that overlap on the GPU (e.g. on two streams without ordering) race on the array
 * and must not be issued.  A next_tok of -1 reports a bounded wait that gave up, as for
 * qwen3_op_lmhead_argmax.
 *
 * Arguments, outputs and the other errors are those of qwen3_op_lmhead_argmax; the message
 * of a failure is returned by qwen3_last_error(NULL). */
int qwen3_op_lmhead_argmax_noalloc(const void *x_dev, int32_t B, int32_t C,
                                   const void *embed_dev, int32_t V, float *logits_dev,
                                   int32_t *next_tok_dev, void *stream);

/* Bytes of workspace qwen3_op_attn_decode needs for B rows. */
size_t qwen3_op_attn_decode_workspace_bytes(int32_t B, int32_t n_q_heads, int32_t n_kv_heads);

/* The n_split a decode step of B rows whose longest context is max_len tokens (the new one
 * included; 1 <= max_len <= max_ctx) gives its decode attention on the current device: the key
 * ranges per (row, KV head) of one wave of CTAs, 1..64 (from the context rounded up to a power
 * of two, ranges of at least 64 keys).  Passed to qwen3_op_attn_decode it runs the launch a
 * step would.  Errors (negative): E_INVALID, E_CUDA. */
int32_t qwen3_op_attn_decode_plan(int32_t B, int32_t n_q_heads, int32_t n_kv_heads, int32_t max_len,
                                  int32_t max_ctx);

/* Split-KV decode attention of B new rows, as decode steps run it ("古法手撕简易LLM推理器",
 * 核心计算函数与Transformer层: the new key appended, then attention over the whole cache;
 * "从零开始写Qwen3", Attn: a one-row query sees every cached key; "手写Qwen3-0.6B推理",
 * Attention: per-head q/k RMSNorm, rotate-half RoPE, K/V shared by Hq/Hkv query heads):
 *   for row b at position p = positions[b] of cache slot s = slots[b]:
 *     q_h, k = RMSNorm per head (q_gain, k_gain; eps), rotated at p (rope table);
 *     cache K[s][g][p] = bf16(k), V[s][g][p] = bf16(v);
 *     out[b][h] = softmax(q_h K[s][g][0..p]^T / sqrt(128)) V[s][g][0..p],  g = h / (Hq/Hkv).
 * qkv_dev fp32 [B, (Hq + 2 Hkv) * 128] (q heads, then k, then v); q_gain_dev, k_gain_dev fp32
 * [128]; rope_dev fp32 [max_ctx][64][2] = (cos, sin) of p * theta^(-2i/128); k_cache_dev,
 * v_cache_dev bf16 [n_slots][Hkv][max_ctx][128] (rows 0..p-1 of each used slot hold the
 * cached keys and values; row p is written; the last 64-key chunk of a range may read up to 63
 * rows past its keys, masked, so every row of the cache must hold finite values, e.g. zeros
 * before first use); out_dev bf16 [B, Hq, 128].  slots and positions
 * are given on the device and on the host (same values; slots distinct, 0 <= slot < n_slots,
 * 0 <= position < max_ctx).  n_split key ranges per (row, KV head), 1..64 (whole 64-key
 * chunks: ceil((p+1)/n_split) rounded up to a multiple of 64 keys each); or 0 as a decode step
 * plans it for these rows (qwen3_op_attn_decode_plan with the largest position + 1).
 * workspace_dev: qwen3_op_attn_decode_workspace_bytes bytes, 256-byte aligned, zero-filled
 * before its first use (calls leave it reusable).
 * head_dim 128; Hq/Hkv in {1, 2, 4, 8}.  Errors: E_INVALID (NULL, bad size or index), E_CUDA. */
int qwen3_op_attn_decode(const float *qkv_dev, int32_t B, const int32_t *slots_dev,
                         const int32_t *slots_host, const int32_t *positions_dev,
                         const int32_t *positions_host, const float *q_gain_dev, const float *k_gain_dev,
                         const float *rope_dev, void *k_cache_dev, void *v_cache_dev, int32_t n_slots,
                         int32_t max_ctx, int32_t n_q_heads, int32_t n_kv_heads, float eps, int32_t n_split,
                         void *out_dev, void *workspace_dev, size_t workspace_bytes, void *stream);

/* Candidates qwen3_sample draws from: the most likely tokens of a row, at most this many. */
#define QWEN3_SAMPLE_CANDIDATES 1024

/* Next-token sampling ("第 3 章", 4.3 Sampler: argmax without a temperature, otherwise
 * temperature with Top-k / Top-p; "手写Qwen3-0.6B推理", softmax with a temperature).
 *
 * logits_dev fp32 [B, V] row-major (as qwen3_decode_step / qwen3_prefill write them); per row b
 * temperature_dev[b] (fp32), top_k_dev[b] (int32), top_p_dev[b] (fp32) and uniform_dev[b]
 * (fp32, a uniform draw in [0, 1) the caller makes); next_tok_dev[b] (int32) receives the token.
 * All are device pointers; nothing is allocated; the call is asynchronous on `stream`.
 *
 * Rule per row.  temperature <= 0: the argmax (lowest index on ties), the other arguments
 * unused.  Otherwise: tokens ordered by logit descending, index ascending; the first
 * min(QWEN3_SAMPLE_CANDIDATES, V) are the candidates; top_k in [1, candidates) keeps the first
 * top_k of them (any other top_k keeps all); p_i = exp((l_i - l_max) / temperature) over the kept
 * tokens; top_p < 1 keeps the shortest prefix whose cumulative p reaches top_p times their total
 * (top_p >= 1 keeps all); the token is the first kept one whose cumulative p exceeds
 * uniform * (the total of what is left).  Arithmetic is fp32: a draw within about 1e-6
 * (relative) of a cumulative boundary may land on the neighbouring token of an fp64 evaluation.
 *
 * Errors: E_INVALID (NULL pointer, B outside [1, 65535], V < 1), E_CUDA (launch); the message
 * is returned by qwen3_last_error(NULL). */
int qwen3_sample(const float *logits_dev, int32_t B, int32_t V, const float *temperature_dev,
                 const int32_t *top_k_dev, const float *top_p_dev, const float *uniform_dev,
                 int32_t *next_tok_dev, void *stream);

/* Releases the context and its graphs.  Does not free the arena or any caller memory. */
void qwen3_free(qwen3_ctx *ctx);

#ifdef __cplusplus
}
#endif

#endif /* QWEN3_GB300_H */
