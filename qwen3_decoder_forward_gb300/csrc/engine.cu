// Continuous batching over one context ("第 3 章", the engine and its scheduler: requests
// queue, each step runs the sequences that have work; "手写Qwen3-0.6B推理", generation ends at
// the end-of-sequence token).  Host code only: the engine is a client of the library's C ABI
// (qwen3_prefill_append, qwen3_decode_step, qwen3_release_slot) and adds no kernel.
//
// Schedule of one step (token_budget tokens at most):
//   1. every running request past its prompt contributes its last generated token;
//   2. every running request still inside its prompt contributes its next chunk;
//   3. waiting requests take free slots, first come first served, while budget remains.
// A step whose rows are all single generated tokens runs as one decode step (GEMV kernels and
// the per-batch-size CUDA graphs); any prompt chunk makes it one prefill_append call over all
// rows, where a generated token is a one-token chunk at its slot's length.
//
// A request may sample instead of taking the greedy token ("第 3 章", 4.3 Sampler: temperature
// and Top-k / Top-p): a step with such a row sets the context's per-row sampling arrays for
// that call (greedy rows get temperature 0), with the uniform draw of the request's t-th token
// taken from its seed by a counter-based generator (below), so a run is reproducible.

#include <cuda_runtime.h>

#include <algorithm>
#include <deque>
#include <map>
#include <memory>
#include <string>
#include <vector>

#include "qwen3_gb300.h"

namespace {

constexpr size_t WS_ALIGN = 256;

size_t ws_align(size_t x) { return (x + WS_ALIGN - 1) / WS_ALIGN * WS_ALIGN; }

struct WsLayout {
    size_t tokens = 0, cu = 0, slots = 0, next = 0, temp = 0, topk = 0, topp = 0, unif = 0, logits = 0, total = 0;
};

WsLayout ws_layout(const qwen3_config &cfg, int budget) {
    WsLayout w;
    size_t off = 0;
    const size_t rows = (size_t)cfg.max_seqs * 4;
    w.tokens = off;
    off = ws_align(off + (size_t)budget * 4);
    w.cu = off;
    off = ws_align(off + (size_t)(cfg.max_seqs + 1) * 4);
    w.slots = off;
    off = ws_align(off + rows);
    w.next = off;
    off = ws_align(off + rows);
    // per-row sampling settings of one call and the logits they draw from
    w.temp = off;
    off = ws_align(off + rows);
    w.topk = off;
    off = ws_align(off + rows);
    w.topp = off;
    off = ws_align(off + rows);
    w.unif = off;
    off = ws_align(off + rows);
    w.logits = off;
    off = ws_align(off + (size_t)cfg.max_seqs * cfg.vocab * 4);
    w.total = off;
    return w;
}

// The uniform draw of token t of a request with seed s: output t + 1 of the SplitMix64
// generator (Steele, Lea and Flood, "Fast splittable pseudorandom number generators", 2014)
// started at state s, its top 24 bits scaled to [0, 1) (exact in fp32).
float uniform_draw(uint64_t seed, int64_t t) {
    uint64_t z = seed + (uint64_t)(t + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return (float)(z >> 40) * (1.0f / 16777216.0f);
}

struct Request {
    int64_t id = 0;
    std::vector<int32_t> prompt;
    int32_t max_new = 0, eos = -1;
    float temperature = 0.0f, top_p = 1.0f;  // temperature <= 0: greedy
    int32_t top_k = 0;
    uint64_t seed = 0;
    int32_t slot = -1;
    int32_t consumed = 0;  // prompt tokens already run
    std::vector<int32_t> out;
    int32_t finish = QWEN3_FINISH_NONE;
};

struct Row {
    Request *req;
    int32_t n;        // tokens this step
    bool generated;  // a generated token (else a prompt chunk)
};

}  // namespace

struct qwen3_engine {
    qwen3_ctx *ctx = nullptr;
    qwen3_config cfg = {};
    int32_t budget = 0;
    uint8_t *ws = nullptr;
    WsLayout lay;
    std::map<int64_t, std::unique_ptr<Request>> requests;
    std::deque<Request *> waiting;
    std::vector<Request *> running;  // in admission order
    std::vector<int32_t> free_slots;
    qwen3_engine_stats stats = {};
    std::string err;
    // host staging of one step
    std::vector<int32_t> h_tokens, h_cu, h_slots, h_next, h_topk;
    std::vector<float> h_temp, h_topp, h_unif;
    // the last step that ran the model: the request of each row, and whether it sampled
    std::vector<int64_t> last_ids;
    bool last_sampled = false;

    int fail(int code, const std::string &m) {
        err = m;
        return code;
    }
    int ctx_fail(int code, const char *what) {
        err = std::string(what) + ": " + qwen3_last_error(ctx);
        return code;
    }
    int cuda_fail(cudaError_t e, const char *what) {
        err = std::string(what) + ": " + cudaGetErrorString(e);
        return QWEN3_E_CUDA;
    }
    void finish(Request *r, int reason) {
        r->finish = reason;
        free_slots.push_back(r->slot);
        r->slot = -1;
    }
};

extern "C" {

size_t qwen3_engine_workspace_bytes(const qwen3_ctx *ctx, int32_t token_budget) {
    qwen3_config cfg;
    if (!ctx || token_budget < 1 || qwen3_get_config(ctx, &cfg) != QWEN3_OK) return 0;
    return ws_layout(cfg, token_budget).total;
}

int qwen3_engine_create(qwen3_ctx *ctx, int32_t token_budget, void *workspace_dev, size_t bytes,
                        qwen3_engine **out) {
    if (!ctx || !workspace_dev || !out) return QWEN3_E_INVALID;
    qwen3_config cfg;
    if (qwen3_get_config(ctx, &cfg) != QWEN3_OK) return QWEN3_E_INVALID;
    if (token_budget < cfg.max_seqs || token_budget > cfg.max_prefill_tokens) return QWEN3_E_INVALID;
    if (reinterpret_cast<uintptr_t>(workspace_dev) % WS_ALIGN) return QWEN3_E_INVALID;
    const WsLayout lay = ws_layout(cfg, token_budget);
    if (bytes < lay.total) return QWEN3_E_INVALID;
    auto *e = new qwen3_engine;
    e->ctx = ctx;
    e->cfg = cfg;
    e->budget = token_budget;
    e->ws = static_cast<uint8_t *>(workspace_dev);
    e->lay = lay;
    for (int s = cfg.max_seqs - 1; s >= 0; --s) e->free_slots.push_back(s);  // slot 0 first
    *out = e;
    return QWEN3_OK;
}

int qwen3_engine_submit(qwen3_engine *e, int64_t request_id, const int32_t *prompt_host, int32_t prompt_len,
                        int32_t max_new_tokens, int32_t eos_id) {
    return qwen3_engine_submit_sampled(e, request_id, prompt_host, prompt_len, max_new_tokens, eos_id, 0.0f, 0, 1.0f,
                                       0);
}

int qwen3_engine_submit_sampled(qwen3_engine *e, int64_t request_id, const int32_t *prompt_host, int32_t prompt_len,
                                int32_t max_new_tokens, int32_t eos_id, float temperature, int32_t top_k, float top_p,
                                uint64_t seed) {
    if (!e) return QWEN3_E_INVALID;
    if (!(temperature == temperature) || !(top_p == top_p))
        return e->fail(QWEN3_E_INVALID, "qwen3_engine_submit: temperature or top_p is NaN");
    if (!prompt_host || prompt_len < 1 || max_new_tokens < 1)
        return e->fail(QWEN3_E_INVALID, "qwen3_engine_submit: empty prompt or max_new_tokens < 1");
    if (prompt_len > e->cfg.max_ctx) return e->fail(QWEN3_E_CAPACITY, "qwen3_engine_submit: prompt longer than max_ctx");
    if (e->requests.count(request_id)) return e->fail(QWEN3_E_INVALID, "qwen3_engine_submit: request id in use");
    auto r = std::make_unique<Request>();
    r->id = request_id;
    r->prompt.assign(prompt_host, prompt_host + prompt_len);
    r->max_new = max_new_tokens;
    r->eos = eos_id;
    r->temperature = temperature;
    r->top_k = top_k;
    r->top_p = top_p;
    r->seed = seed;
    e->waiting.push_back(r.get());
    e->requests.emplace(request_id, std::move(r));
    return QWEN3_OK;
}

int qwen3_engine_step(qwen3_engine *e, void *stream, int32_t *n_finished) {
    if (!e) return QWEN3_E_INVALID;
    if (n_finished) *n_finished = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::vector<Row> rows;
    int32_t left = e->budget, finished = 0;
    // 1. generated tokens of the requests past their prompt (a full slot ends the request)
    for (Request *r : e->running) {
        if (r->consumed < (int32_t)r->prompt.size()) continue;
        if (qwen3_slot_length(e->ctx, r->slot) >= e->cfg.max_ctx) {
            e->finish(r, QWEN3_FINISH_CONTEXT);
            ++finished;
            continue;
        }
        rows.push_back(Row{r, 1, true});
        --left;
    }
    // 2. the next prompt chunk of the requests still inside their prompt
    for (Request *r : e->running) {
        if (r->finish != QWEN3_FINISH_NONE || r->consumed >= (int32_t)r->prompt.size() || left <= 0) continue;
        const int32_t n = std::min<int32_t>((int32_t)r->prompt.size() - r->consumed, left);
        rows.push_back(Row{r, n, false});
        left -= n;
    }
    // 3. waiting requests into free slots
    while (!e->waiting.empty() && !e->free_slots.empty() && left > 0) {
        Request *r = e->waiting.front();
        e->waiting.pop_front();
        r->slot = e->free_slots.back();
        e->free_slots.pop_back();
        if (qwen3_release_slot(e->ctx, r->slot, stream) != QWEN3_OK) return e->ctx_fail(QWEN3_E_CUDA, "release slot");
        e->running.push_back(r);
        const int32_t n = std::min<int32_t>((int32_t)r->prompt.size(), left);
        rows.push_back(Row{r, n, false});
        left -= n;
    }
    e->running.erase(std::remove_if(e->running.begin(), e->running.end(),
                                    [](Request *r) { return r->finish != QWEN3_FINISH_NONE; }),
                     e->running.end());
    if (rows.empty()) {
        if (n_finished) *n_finished = finished;
        return QWEN3_OK;
    }

    const int32_t B = (int32_t)rows.size();
    bool mixed = false, sampled = false;
    e->h_tokens.clear();
    e->h_cu.assign(1, 0);
    e->h_slots.clear();
    e->h_temp.clear();
    e->h_topk.clear();
    e->h_topp.clear();
    e->h_unif.clear();
    e->last_ids.clear();
    for (const Row &w : rows) {
        Request *r = w.req;
        e->last_ids.push_back(r->id);
        // the draw of the token this row produces (index = tokens generated so far)
        sampled = sampled || r->temperature > 0.0f;
        e->h_temp.push_back(r->temperature);
        e->h_topk.push_back(r->top_k);
        e->h_topp.push_back(r->top_p);
        e->h_unif.push_back(uniform_draw(r->seed, (int64_t)r->out.size()));
        if (w.generated) {
            e->h_tokens.push_back(r->out.back());
        } else {
            mixed = true;
            e->h_tokens.insert(e->h_tokens.end(), r->prompt.begin() + r->consumed,
                               r->prompt.begin() + r->consumed + w.n);
        }
        e->h_cu.push_back((int32_t)e->h_tokens.size());
        e->h_slots.push_back(r->slot);
    }
    int32_t *d_tokens = reinterpret_cast<int32_t *>(e->ws + e->lay.tokens);
    int32_t *d_cu = reinterpret_cast<int32_t *>(e->ws + e->lay.cu);
    int32_t *d_slots = reinterpret_cast<int32_t *>(e->ws + e->lay.slots);
    int32_t *d_next = reinterpret_cast<int32_t *>(e->ws + e->lay.next);
    cudaError_t ce = cudaMemcpyAsync(d_tokens, e->h_tokens.data(), e->h_tokens.size() * 4, cudaMemcpyHostToDevice, st);
    if (ce == cudaSuccess) ce = cudaMemcpyAsync(d_slots, e->h_slots.data(), (size_t)B * 4, cudaMemcpyHostToDevice, st);
    if (ce == cudaSuccess && mixed)
        ce = cudaMemcpyAsync(d_cu, e->h_cu.data(), (size_t)(B + 1) * 4, cudaMemcpyHostToDevice, st);
    qwen3_sampling sp = {};
    float *d_logits = nullptr;
    if (sampled) {  // this call draws: per-row settings (greedy rows have temperature 0)
        sp.temperature = reinterpret_cast<float *>(e->ws + e->lay.temp);
        sp.top_k = reinterpret_cast<int32_t *>(e->ws + e->lay.topk);
        sp.top_p = reinterpret_cast<float *>(e->ws + e->lay.topp);
        sp.uniform = reinterpret_cast<float *>(e->ws + e->lay.unif);
        d_logits = reinterpret_cast<float *>(e->ws + e->lay.logits);
        if (ce == cudaSuccess)
            ce = cudaMemcpyAsync((void *)sp.temperature, e->h_temp.data(), (size_t)B * 4, cudaMemcpyHostToDevice, st);
        if (ce == cudaSuccess)
            ce = cudaMemcpyAsync((void *)sp.top_k, e->h_topk.data(), (size_t)B * 4, cudaMemcpyHostToDevice, st);
        if (ce == cudaSuccess)
            ce = cudaMemcpyAsync((void *)sp.top_p, e->h_topp.data(), (size_t)B * 4, cudaMemcpyHostToDevice, st);
        if (ce == cudaSuccess)
            ce = cudaMemcpyAsync((void *)sp.uniform, e->h_unif.data(), (size_t)B * 4, cudaMemcpyHostToDevice, st);
    }
    if (ce != cudaSuccess) return e->cuda_fail(ce, "qwen3_engine_step: upload");
    int rc = qwen3_set_sampling(e->ctx, sampled ? &sp : nullptr);
    if (rc != QWEN3_OK) return e->ctx_fail(rc, "qwen3_engine_step: set_sampling");
    if (mixed) {
        rc = qwen3_prefill_append(e->ctx, d_tokens, d_cu, e->h_cu.data(), d_slots, e->h_slots.data(), B, d_logits,
                                  d_next, stream);
        if (rc != QWEN3_OK) return e->ctx_fail(rc, "qwen3_engine_step: prefill_append");
        ++e->stats.mixed_steps;
    } else {
        rc = qwen3_decode_step(e->ctx, d_tokens, d_slots, e->h_slots.data(), B, d_logits, d_next, stream);
        if (rc != QWEN3_OK) return e->ctx_fail(rc, "qwen3_engine_step: decode_step");
        ++e->stats.decode_steps;
    }
    if (sampled && (rc = qwen3_set_sampling(e->ctx, nullptr)) != QWEN3_OK)
        return e->ctx_fail(rc, "qwen3_engine_step: set_sampling");
    e->last_sampled = sampled;
    ++e->stats.steps;
    e->h_next.resize(B);
    ce = cudaMemcpyAsync(e->h_next.data(), d_next, (size_t)B * 4, cudaMemcpyDeviceToHost, st);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
    if (ce != cudaSuccess) return e->cuda_fail(ce, "qwen3_engine_step: next tokens");

    for (int32_t b = 0; b < B; ++b) {
        const Row &w = rows[b];
        Request *r = w.req;
        if (!w.generated) {
            r->consumed += w.n;
            e->stats.prompt_tokens += w.n;
            if (r->consumed < (int32_t)r->prompt.size()) continue;  // the prompt goes on next step
        }
        const int32_t tok = e->h_next[b];
        r->out.push_back(tok);
        ++e->stats.generated_tokens;
        if (r->eos >= 0 && tok == r->eos)
            e->finish(r, QWEN3_FINISH_EOS);
        else if ((int32_t)r->out.size() >= r->max_new)
            e->finish(r, QWEN3_FINISH_LENGTH);
        else
            continue;
        ++finished;
    }
    e->running.erase(std::remove_if(e->running.begin(), e->running.end(),
                                    [](Request *r) { return r->finish != QWEN3_FINISH_NONE; }),
                     e->running.end());
    if (n_finished) *n_finished = finished;
    return QWEN3_OK;
}

int32_t qwen3_engine_unfinished(const qwen3_engine *e) {
    if (!e) return 0;
    return (int32_t)(e->waiting.size() + e->running.size());
}

int qwen3_engine_result(const qwen3_engine *e, int64_t request_id, int32_t *tokens_host, int32_t capacity,
                        int32_t *n_tokens, int32_t *finish_reason) {
    if (!e || capacity < 0 || (capacity > 0 && !tokens_host)) return QWEN3_E_INVALID;
    auto it = e->requests.find(request_id);
    if (it == e->requests.end()) return QWEN3_E_INVALID;
    const Request &r = *it->second;
    const int32_t n = (int32_t)r.out.size();
    std::copy(r.out.begin(), r.out.begin() + std::min(n, capacity), tokens_host);
    if (n_tokens) *n_tokens = n;
    if (finish_reason) *finish_reason = r.finish;
    return QWEN3_OK;
}

int qwen3_engine_forget(qwen3_engine *e, int64_t request_id) {
    if (!e) return QWEN3_E_INVALID;
    auto it = e->requests.find(request_id);
    if (it == e->requests.end() || it->second->finish == QWEN3_FINISH_NONE)
        return e->fail(QWEN3_E_INVALID, "qwen3_engine_forget: unknown or unfinished request");
    e->requests.erase(it);
    return QWEN3_OK;
}

int qwen3_engine_last_step(const qwen3_engine *e, int64_t *ids_host, int32_t capacity, int32_t *n_rows,
                           const float **logits_dev) {
    if (!e || capacity < 0 || (capacity > 0 && !ids_host)) return QWEN3_E_INVALID;
    const int32_t n = (int32_t)e->last_ids.size();
    std::copy(e->last_ids.begin(), e->last_ids.begin() + std::min(n, capacity), ids_host);
    if (n_rows) *n_rows = n;
    if (logits_dev) *logits_dev = e->last_sampled ? reinterpret_cast<const float *>(e->ws + e->lay.logits) : nullptr;
    return QWEN3_OK;
}

int qwen3_engine_get_stats(const qwen3_engine *e, qwen3_engine_stats *out) {
    if (!e || !out) return QWEN3_E_INVALID;
    *out = e->stats;
    return QWEN3_OK;
}

const char *qwen3_engine_last_error(const qwen3_engine *e) { return e ? e->err.c_str() : ""; }

void qwen3_engine_free(qwen3_engine *e) { delete e; }

}  // extern "C"
