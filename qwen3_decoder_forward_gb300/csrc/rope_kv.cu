// Per-head Q/K RMSNorm, rotate-half RoPE and the KV-cache write.
//
//  * q and k of each head are RMS-normalised over head_dim with their own gains, v is
//    left as projected ("手写Qwen3-0.6B推理", Attention: q_norm/k_norm; "第 3 章", 3.3).
//  * RoPE pairs element i with i+64 and rotates by p*theta^(-2i/128) at the row's absolute
//    position p ("手写Qwen3-0.6B推理", Rope: rotate_half; "古法手撕简易LLM推理器",
//    RoPE的细节: Qwen3 uses rotate_half).  cos/sin come from a table built on the host in
//    double precision.
//  * The cache keeps rotated K and raw V per slot ("古法手撕简易LLM推理器", 核心计算函数与
//    Transformer层), laid out [slot][Hkv][max_ctx][128] so one head's keys are contiguous.
//
// One warp per (row, head); lane l holds elements {2l, 2l+1} and {64+2l, 65+2l}, so both
// members of every RoPE pair sit in the same lane.

#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;

__global__ void __launch_bounds__(256) k_qknorm_rope_kv(
    const float *__restrict__ qkv, Rows r, const float *__restrict__ q_gain,
    const float *__restrict__ k_gain, const float2 *__restrict__ rope, bf16 *__restrict__ q_out,
    bf16 *__restrict__ k_layer, bf16 *__restrict__ v_layer, int Hq, int Hkv, int max_ctx,
    float eps, uint32_t *err) {
    pdl_wait();
    pdl_trigger();
    const int heads = Hq + 2 * Hkv;
    const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (item >= r.rows * heads) return;
    const int lane = threadIdx.x & 31;
    const int row = item / heads, h = item % heads;
    const float *src = qkv + (size_t)row * heads * D + h * D;
    float2 a = *reinterpret_cast<const float2 *>(src + 2 * lane);
    float2 b = *reinterpret_cast<const float2 *>(src + 64 + 2 * lane);
    const int slot = r.row_slot[row], pos = r.row_pos[row];

    if (h < Hq + Hkv) {  // q or k head: norm then rotate
        const float *gain = h < Hq ? q_gain : k_gain;
        const float ss = warp_sum(a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y);
        const float inv = rsqrtf(ss * (1.0f / D) + eps);
        const float2 ga = *reinterpret_cast<const float2 *>(gain + 2 * lane);
        const float2 gb = *reinterpret_cast<const float2 *>(gain + 64 + 2 * lane);
        a.x *= inv * ga.x; a.y *= inv * ga.y;
        b.x *= inv * gb.x; b.y *= inv * gb.y;
        if (pos < max_ctx) {
            const float2 c0 = rope[(size_t)pos * 64 + 2 * lane];      // (cos, sin) of pair 2l
            const float2 c1 = rope[(size_t)pos * 64 + 2 * lane + 1];  // pair 2l+1
            const float2 na = make_float2(a.x * c0.x - b.x * c0.y, a.y * c1.x - b.y * c1.y);
            const float2 nb = make_float2(b.x * c0.x + a.x * c0.y, b.y * c1.x + a.y * c1.y);
            a = na;
            b = nb;
        }
    }
    bf16 *dst;
    if (h < Hq) {
        dst = q_out + ((size_t)row * Hq + h) * D;
    } else {
        if (pos >= max_ctx) {
            if (lane == 0) atomicOr(err, ERR_POSITION);
            return;
        }
        const int g = h < Hq + Hkv ? h - Hq : h - Hq - Hkv;
        bf16 *base = h < Hq + Hkv ? k_layer : v_layer;
        dst = base + (((size_t)slot * Hkv + g) * max_ctx + pos) * D;
    }
    *reinterpret_cast<uint32_t *>(dst + 2 * lane) = pack_bf16x2(a.x, a.y);
    *reinterpret_cast<uint32_t *>(dst + 64 + 2 * lane) = pack_bf16x2(b.x, b.y);
}

}  // namespace

cudaError_t launch_qknorm_rope_kv(const Launch &lc, const float *qkv, const Rows &r,
                                  const float *q_gain, const float *k_gain, const float2 *rope,
                                  bf16 *q_out, bf16 *k_layer, bf16 *v_layer, int Hq, int Hkv,
                                  int max_ctx, float eps, uint32_t *err) {
    const int items = r.rows * (Hq + 2 * Hkv);
    return launch(lc, k_qknorm_rope_kv, dim3((items + 7) / 8), dim3(256), 0, qkv, r, q_gain,
                  k_gain, rope, q_out, k_layer, v_layer, Hq, Hkv, max_ctx, eps, err);
}

}  // namespace q3
