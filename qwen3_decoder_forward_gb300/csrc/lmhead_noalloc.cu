// lm_head + greedy argmax for callers that cannot allocate device memory.
//
// qwen3_op_lmhead_argmax needs a caller-provided workspace for its per-CTA partial maxima.
// Some callers have no way to provide one:
//  * code that enqueues this work while a stream is being recorded into a CUDA graph,
//    where a cudaMalloc is refused (global capture mode) or not recorded at all;
//  * plug-ins running inside a host framework that owns every device allocation;
//  * latency-critical loops that must not call cudaMalloc/cudaFree, because cudaFree
//    synchronises the whole device.
// This variant keeps its scratch in a fixed array in the library's own device memory.
// It runs the same kernels as qwen3_op_lmhead_argmax, so its results are identical.

#include <algorithm>
#include <mutex>
#include <string>

#include "kernels.h"
#include "qwen3_gb300.h"

namespace q3 {
void set_last_error(const std::string &msg);  // message returned by qwen3_last_error(NULL)
}

namespace {

using namespace q3;

constexpr int NOALLOC_MAX_B = 32;      // largest batch this entry point accepts
constexpr int NOALLOC_PARTS = 1024;    // partial results per row (one per CTA of pass 1)
constexpr size_t NOALLOC_BYTES = (size_t)NOALLOC_MAX_B * NOALLOC_PARTS * 8;  // 256 KiB
constexpr int MAX_DEVICES = 256;

// The scratch itself. Every GPU that loads this library holds these 256 KiB until the
// process exits. All calls on a device share it. The host name of the array is not a
// device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

struct DeviceScratch {
    void *ptr = nullptr;
    int num_sms = 0;
    bool ready = false;
};
std::mutex g_mu;
DeviceScratch g_dev[MAX_DEVICES];

bool c_supported(int C) {
    return C == 256 || C == 512 || C == 768 || C == 1024 || C == 1536 || C == 2048 || C == 2560 ||
           C == 3072;
}

int fail(int code, const std::string &m) {
    set_last_error("qwen3_op_lmhead_argmax_noalloc: " + m);
    return code;
}

}  // namespace

extern "C" int qwen3_op_lmhead_argmax_noalloc(const void *x_dev, int32_t B, int32_t C,
                                              const void *embed_dev, int32_t V, float *logits_dev,
                                              int32_t *next_tok_dev, void *stream) {
    set_last_error("");
    if (!x_dev || !embed_dev || !next_tok_dev) return fail(QWEN3_E_INVALID, "NULL argument");
    if (B < 1 || V < 1 || !c_supported(C)) return fail(QWEN3_E_INVALID, "bad B, C or V");
    if (B > NOALLOC_MAX_B)
        return fail(QWEN3_E_CAPACITY, "B = " + std::to_string(B) + " exceeds the fixed scratch, which holds at most " +
                                          std::to_string(NOALLOC_MAX_B) + " rows");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(QWEN3_E_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= MAX_DEVICES) return fail(QWEN3_E_UNSUPPORTED, "device ordinal out of range");
    DeviceScratch s;
    {
        // First call on this device: look up the array's device address with this device
        // current. Done once per device; later calls reuse the cached address (which is why
        // the library must not outlive a cudaDeviceReset of that device: the reset unloads
        // the module the address belongs to).
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_dev[dev].ready) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return fail(QWEN3_E_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
            int sms = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return fail(QWEN3_E_CUDA, cudaGetErrorString(e));
            g_dev[dev].ptr = p;
            g_dev[dev].num_sms = sms;
            g_dev[dev].ready = true;
        }
        s = g_dev[dev];
    }
    const int n_parts = std::min(lmhead_parts(s.num_sms), NOALLOC_PARTS);
    // Pass 1 writes every (row, CTA) partial that pass 2 reads -- a CTA whose bounded wait
    // gave up writes (+inf, -1), which makes that row's token -1 -- so the previous call's
    // contents never leak into this one and nothing needs clearing first.
    float *part_val = static_cast<float *>(s.ptr);
    int32_t *part_idx = reinterpret_cast<int32_t *>(part_val + (size_t)NOALLOC_MAX_B * NOALLOC_PARTS);
    Launch lc;
    lc.stream = static_cast<cudaStream_t>(stream);
    lc.pdl = false;
    lc.num_sms = s.num_sms;
    Rows r;  // no KV-cache bookkeeping for a bare call
    r.B = B;
    r.rows = B;
    e = launch_lmhead_argmax(lc, static_cast<const bf16 *>(x_dev), B, C,
                             static_cast<const bf16 *>(embed_dev), V, logits_dev, part_val, part_idx,
                             n_parts, next_tok_dev, r);
    if (e != cudaSuccess) return fail(QWEN3_E_CUDA, cudaGetErrorString(e));
    return QWEN3_OK;
}
