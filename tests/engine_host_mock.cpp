// Host-only stand-in for the context calls that the continuous-batching engine (engine.cu)
// makes, so that the engine's scheduling can be tested on a machine without a GPU.  The
// engine source is compiled unchanged against these definitions (test_engine_host.py builds
// both with g++ into one shared library).
//
// The stand-in "model" keeps every slot's token history on the host; the next token of a slot
// is the FNV-1a hash (64-bit offset basis and prime) of its whole history modulo the vocabulary,
// so a test can compute every expected token independently.  "Device" memory is host memory:
// the CUDA copies are memcpy.  Each prefill_append / decode_step / release_slot call is logged.
// The calls check the arguments the way the library does and also that the device-side copies
// of cu_seqlens and slots equal the host-side ones, so a wrong upload by the engine fails.

#include <cuda_runtime.h>

#include <cstring>
#include <string>
#include <vector>

#include "qwen3_gb300.h"

struct qwen3_ctx {
    qwen3_config cfg;
    qwen3_sampling sampling = {};            // as set by qwen3_set_sampling ("device" = host arrays)
    std::vector<std::vector<int32_t>> hist;  // tokens cached per slot
    std::vector<int32_t> log;                // see mock_log
    std::string err;
    int fail(int code, const char *m) {
        err = m;
        return code;
    }
};

namespace {

uint64_t fnv(const std::vector<int32_t> &h) {
    uint64_t x = 14695981039346656037ull;
    for (int32_t t : h) {
        x ^= (uint64_t)(uint32_t)t;
        x *= 1099511628211ull;
    }
    return x;
}

int32_t next_token(const std::vector<int32_t> &h, int32_t vocab) { return (int32_t)(fnv(h) % (uint64_t)vocab); }

// Row b's next token: greedy (the hash) unless the call samples and the row's temperature is
// positive; then the hash mixed with the row's uniform draw (a multiple of 2^-24) and settings,
// so a test can tell whether each row got its own draw and settings.
int32_t row_token(const qwen3_ctx *c, const std::vector<int32_t> &h, int b) {
    const qwen3_sampling &s = c->sampling;
    if (!s.temperature || !(s.temperature[b] > 0.0f)) return next_token(h, c->cfg.vocab);
    uint64_t x = fnv(h);
    x ^= (uint64_t)(s.uniform[b] * 16777216.0f) << 32;
    x ^= (uint64_t)(uint32_t)s.top_k[b] << 8;
    x ^= (uint64_t)(int64_t)(s.temperature[b] * 1000.0f + 0.5f) << 16;
    x ^= (uint64_t)(int64_t)(s.top_p[b] * 1000.0f + 0.5f) << 40;
    return (int32_t)(x % (uint64_t)c->cfg.vocab);
}

bool unique_slots(const qwen3_ctx *c, const int32_t *s, int B) {
    std::vector<char> seen(c->cfg.max_seqs, 0);
    for (int b = 0; b < B; ++b) {
        if (s[b] < 0 || s[b] >= c->cfg.max_seqs || seen[s[b]]) return false;
        seen[s[b]] = 1;
    }
    return true;
}

}  // namespace

extern "C" {

// ---- the three CUDA runtime calls the engine makes -------------------------------------
cudaError_t cudaMemcpyAsync(void *dst, const void *src, size_t count, enum cudaMemcpyKind, cudaStream_t) {
    std::memcpy(dst, src, count);
    return cudaSuccess;
}
cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }
const char *cudaGetErrorString(cudaError_t) { return "mock CUDA error"; }

// ---- the context calls -----------------------------------------------------------------
int qwen3_get_config(const qwen3_ctx *c, qwen3_config *cfg) {
    if (!c || !cfg) return QWEN3_E_INVALID;
    *cfg = c->cfg;
    return QWEN3_OK;
}

int32_t qwen3_slot_length(const qwen3_ctx *c, int32_t slot) {
    if (!c || slot < 0 || slot >= c->cfg.max_seqs) return -1;
    return (int32_t)c->hist[slot].size();
}

int qwen3_release_slot(qwen3_ctx *c, int32_t slot, void *) {
    if (!c || slot < 0 || slot >= c->cfg.max_seqs) return QWEN3_E_INVALID;
    c->hist[slot].clear();
    c->log.insert(c->log.end(), {3, slot});
    return QWEN3_OK;
}

int qwen3_prefill_append(qwen3_ctx *c, const int32_t *tokens, const int32_t *cu_dev, const int32_t *cu,
                         const int32_t *slots_dev, const int32_t *slots, int32_t B, float *logits, int32_t *next,
                         void *) {
    if (!c) return QWEN3_E_INVALID;
    if (!tokens || !cu_dev || !cu || !slots_dev || !slots || !next || (logits == nullptr) != (c->sampling.temperature == nullptr))
        return c->fail(QWEN3_E_INVALID, "args");
    if (B < 1 || B > c->cfg.max_seqs || !unique_slots(c, slots, B) || cu[0] != 0)
        return c->fail(QWEN3_E_INVALID, "rows");
    for (int b = 0; b < B; ++b) {
        if (cu_dev[b + 1] != cu[b + 1] || slots_dev[b] != slots[b]) return c->fail(QWEN3_E_INVALID, "upload");
        if (cu[b + 1] <= cu[b]) return c->fail(QWEN3_E_INVALID, "order");
        if ((int)c->hist[slots[b]].size() + cu[b + 1] - cu[b] > c->cfg.max_ctx)
            return c->fail(QWEN3_E_CAPACITY, "max_ctx");
    }
    if (cu[B] > c->cfg.max_prefill_tokens) return c->fail(QWEN3_E_CAPACITY, "max_prefill_tokens");
    c->log.insert(c->log.end(), {1, B, cu[B]});
    for (int b = 0; b < B; ++b) {
        std::vector<int32_t> &h = c->hist[slots[b]];
        h.insert(h.end(), tokens + cu[b], tokens + cu[b + 1]);
        next[b] = row_token(c, h, b);
        c->log.insert(c->log.end(), {slots[b], cu[b + 1] - cu[b]});
        c->log.insert(c->log.end(), tokens + cu[b], tokens + cu[b + 1]);
    }
    return QWEN3_OK;
}

int qwen3_decode_step(qwen3_ctx *c, const int32_t *tokens, const int32_t *slots_dev, const int32_t *slots,
                      int32_t B, float *logits, int32_t *next, void *) {
    if (!c) return QWEN3_E_INVALID;
    if (!tokens || !slots_dev || !slots || !next || (logits == nullptr) != (c->sampling.temperature == nullptr))
        return c->fail(QWEN3_E_INVALID, "args");
    if (B < 1 || B > c->cfg.max_seqs || !unique_slots(c, slots, B)) return c->fail(QWEN3_E_INVALID, "rows");
    for (int b = 0; b < B; ++b) {
        if (slots_dev[b] != slots[b]) return c->fail(QWEN3_E_INVALID, "upload");
        if (c->hist[slots[b]].empty()) return c->fail(QWEN3_E_INVALID, "slot never prefilled");
        if ((int)c->hist[slots[b]].size() + 1 > c->cfg.max_ctx) return c->fail(QWEN3_E_CAPACITY, "max_ctx");
    }
    c->log.insert(c->log.end(), {2, B, B});
    for (int b = 0; b < B; ++b) {
        std::vector<int32_t> &h = c->hist[slots[b]];
        h.push_back(tokens[b]);
        next[b] = row_token(c, h, b);
        c->log.insert(c->log.end(), {slots[b], 1, tokens[b]});
    }
    return QWEN3_OK;
}

const char *qwen3_last_error(const qwen3_ctx *c) { return c ? c->err.c_str() : ""; }

int qwen3_set_sampling(qwen3_ctx *c, const qwen3_sampling *sp) {
    if (!c) return QWEN3_E_INVALID;
    if (!sp || !sp->temperature) {
        c->sampling = qwen3_sampling{};
        return QWEN3_OK;
    }
    if (!sp->top_k || !sp->top_p || !sp->uniform) return c->fail(QWEN3_E_INVALID, "NULL sampling array");
    c->sampling = *sp;
    return QWEN3_OK;
}

// ---- test hooks ------------------------------------------------------------------------
qwen3_ctx *mock_ctx_create(int32_t max_seqs, int32_t max_ctx, int32_t max_prefill_tokens, int32_t vocab) {
    auto *c = new qwen3_ctx;
    c->cfg = qwen3_config{};
    c->cfg.max_seqs = max_seqs;
    c->cfg.max_ctx = max_ctx;
    c->cfg.max_prefill_tokens = max_prefill_tokens;
    c->cfg.vocab = vocab;
    c->hist.assign(max_seqs, {});
    return c;
}

void mock_ctx_free(qwen3_ctx *c) { delete c; }

// The call log: records of [3, slot] (release), [1, B, N, then per row: slot, n, n tokens]
// (prefill_append) and [2, B, B, then per row: slot, 1, token] (decode step).
int32_t mock_log_size(const qwen3_ctx *c) { return (int32_t)c->log.size(); }
void mock_log(const qwen3_ctx *c, int32_t *out) { std::memcpy(out, c->log.data(), c->log.size() * 4); }

}  // extern "C"
