// Next-token sampling from fp32 logits: temperature, top-k and top-p ("第 3 章", 4.3 Sampler;
// "手写Qwen3-0.6B推理", softmax with a temperature).
//
// Rule (the pages name the steps, not their exact order or tie-breaking; this is the reading
// this library implements):
//   temperature <= 0: the argmax, lowest index on ties.
//   otherwise: tokens ordered by logit descending, index ascending; the first
//   min(SAMPLE_CANDIDATES, V) of them are the candidates; top_k in [1, candidates) keeps the
//   first top_k; p_i = exp((l_i - l_max) / temperature) over the kept tokens; top_p < 1 keeps
//   the shortest prefix whose cumulative p reaches top_p times the kept total; the token is
//   the first kept one whose cumulative p exceeds u times the total of what is left, with u
//   in [0, 1) a uniform draw the caller supplies.
// Dividing by a positive temperature keeps the order of the logits, so the candidates are
// chosen on the fp32 logits themselves, bit for bit.
//
// A cluster of eight CTAs per row (1024 threads each).  Each CTA reads its eighth of the row
// once, as order-preserving 32-bit keys, into shared memory; the rest of the work reads only
// shared memory.  The candidate boundary (the 1024-th largest key) is found by a three-pass
// radix select (12, 10 and 10 bits): each CTA counts its own keys and adds its non-zero bins
// into every CTA's copy of the cluster histogram (distributed shared memory atomics), so that
// after one cluster barrier per pass every CTA finds the same digit in its own shared memory.
// Each CTA then writes its keys above the boundary, and its lowest-index keys equal to it,
// straight into the candidate array of the cluster's first CTA, at offsets given by the counts
// of the CTAs before it.  That CTA sorts the candidates (bitonic: warp shuffles for strides
// below 32, shared memory above), scans the probabilities and draws.  Greedy rows reduce
// (key, index) maxima across the cluster the same way.

#include <cooperative_groups.h>
#include <string>

#include "kernels.h"
#include "qwen3_gb300.h"

namespace q3 {
void set_last_error(const std::string &msg);  // message returned by qwen3_last_error(NULL)
}

namespace {

using namespace q3;
namespace cg = cooperative_groups;

constexpr int ST = 1024;          // threads per CTA
constexpr int CL = 8;             // CTAs per row (one cluster)
constexpr int CAND = 1024;        // candidates per row (QWEN3_SAMPLE_CANDIDATES)
constexpr int HIST = 4096;        // bins of the widest radix pass (12 bits)
constexpr uint32_t FULL = 0xffffffffu;
constexpr int MAX_SMEM = 227 * 1024;

static_assert(CAND == ST, "one candidate per thread");

// Order-preserving map of an fp32 value to an unsigned key: a > b  <=>  key(a) > key(b) for
// non-NaN values.  -0 is keyed as +0, so that equal values have equal keys.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = f == 0.f ? 0u : __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Candidate entry: key in the high word, the complemented index in the low word, so that a
// larger entry comes first in (logit descending, index ascending) order.  0 is below every
// real entry (its low word would be the index 0xffffffff).
__device__ __forceinline__ uint64_t entry(uint32_t key, int idx) {
    return ((uint64_t)key << 32) | (uint32_t)(~(uint32_t)idx);
}

__device__ __forceinline__ int entry_index(uint64_t e) { return (int)(~(uint32_t)(e & 0xffffffffu)); }

constexpr int GHIST = HIST + 2 * 1024;  // cluster histograms of the three passes

// Fixed part of the shared memory; the CTA's keys follow it.
struct SampleSmem {
    uint32_t hist[HIST];    // this CTA's histogram of the current pass; later the sort's 2nd buffer
    uint32_t ghist[GHIST];  // cluster histograms, passes 0, 1, 2 at offsets 0, 4096, 5120
    uint64_t cand[CAND];    // candidates (filled in the first CTA of the cluster)
    float fscan[32];
    int iscan[32];
    int wgt[32];            // per warp: keys above the boundary, then their exclusive prefix
    int weq[32];            // per warp: keys equal to it, likewise
    int base_gt;            // keys above the boundary in the CTAs before this one (added by them)
    int base_eq;            // keys equal to it, likewise
    int digit;
    int krem;
    float total;
    uint32_t best_k[32];
    int best_i[32];
    uint32_t red_k[CL];     // per CTA of the cluster: its greedy maximum (first CTA only)
    int red_i[CL];
};

// The keys start 16-byte aligned plus up to three words, so that the 16-byte-aligned part of
// the row lands on 16-byte-aligned keys.
__host__ __device__ constexpr size_t keys_offset() { return (sizeof(SampleSmem) + 15) & ~size_t(15); }
constexpr size_t KEYS_PAD = 16;

// Exclusive prefix sum of v over the block (all threads call it).
__device__ int block_excl_scan(int v, int *ws) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = ws[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, t, o);
            if (lane >= o) t += y;
        }
        ws[lane] = t;
    }
    __syncthreads();
    const int base = w ? ws[w - 1] : 0;
    __syncthreads();
    return base + x - v;
}

// Inclusive prefix sum of fp32 p over the block, in thread order.
__device__ float block_incl_scan(float p, float *ws) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float x = p;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    if (w == 0) {
        float t = ws[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(FULL, t, o);
            if (lane >= o) t += y;
        }
        ws[lane] = t;
    }
    __syncthreads();
    const float r = (w ? ws[w - 1] : 0.f) + x;
    __syncthreads();
    return r;
}

// (key, index) order of the greedy choice: larger key, then lower index.
__device__ __forceinline__ bool better(uint32_t k, int i, uint32_t bk, int bi) {
    return k > bk || (k == bk && i < bi);
}

__device__ __forceinline__ int lanes_below(uint32_t ballot) {
    return __popc(ballot & ((1u << (threadIdx.x & 31)) - 1u));
}

// Bitonic compare-exchange partner value of this thread's element at `stride`: a warp shuffle
// below 32, otherwise through shared memory (`buf`, alternating between two arrays so that one
// barrier per exchange suffices).
__device__ __forceinline__ uint64_t partner_value(uint64_t x, int stride, uint64_t *buf) {
    if (stride < 32) {
        const uint32_t lo = __shfl_xor_sync(FULL, (uint32_t)x, stride);
        const uint32_t hi = __shfl_xor_sync(FULL, (uint32_t)(x >> 32), stride);
        return ((uint64_t)hi << 32) | lo;
    }
    buf[threadIdx.x] = x;
    __syncthreads();
    return buf[threadIdx.x ^ stride];
}

__global__ void __launch_bounds__(ST, 1)
k_sample(const float *__restrict__ logits, int V, int chunk, const float *__restrict__ temperature,
         const int32_t *__restrict__ top_k, const float *__restrict__ top_p,
         const float *__restrict__ uniform, int32_t *__restrict__ next_tok) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SampleSmem &s = *reinterpret_cast<SampleSmem *>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / CL, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const float *row = logits + (size_t)b * V;
    const int beg = rank * chunk;
    const int n_loc = max(0, min(chunk, V - beg));

    // This CTA's slice of the row, as keys: a ragged head of up to three values, 16-byte
    // vectors, a ragged tail.  keys[head] is 16-byte aligned.
    const float *src = row + beg;
    const int head = min(n_loc, (int)(((16u - ((uint32_t)(uintptr_t)src & 15u)) & 15u) >> 2));
    const int n4 = (n_loc - head) >> 2;
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw + keys_offset()) + ((4 - head) & 3);
    {
        if (tid < head) keys[tid] = order_key(src[tid]);
        const float4 *src4 = reinterpret_cast<const float4 *>(src + head);
        uint4 *keys4 = reinterpret_cast<uint4 *>(keys + head);
        int q = tid;
        for (; q + 3 * ST < n4; q += 4 * ST) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = src4[q + u * ST];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                keys4[q + u * ST] = make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w));
        }
        for (; q < n4; q += ST) {
            const float4 v = src4[q];
            keys4[q] = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
        }
        const int i = head + 4 * n4 + tid;
        if (i < n_loc) keys[i] = order_key(src[i]);
    }
    for (int j = tid; j < HIST; j += ST) s.hist[j] = 0;
    for (int j = tid; j < GHIST; j += ST) s.ghist[j] = 0;
    if (tid == 0) {
        s.base_gt = 0;
        s.base_eq = 0;
        s.digit = 0;
        s.krem = CAND;
    }
    const float T = temperature[b];
    // Every CTA of the cluster has started and cleared what the others add into.
    cluster.sync();

    if (!(T > 0.f)) {
        uint32_t bk = 0;
        int bi = 0x7fffffff;
        for (int i = tid; i < n_loc; i += ST)
            if (better(keys[i], beg + i, bk, bi)) {
                bk = keys[i];
                bi = beg + i;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint32_t ok = __shfl_xor_sync(FULL, bk, o);
            const int oi = __shfl_xor_sync(FULL, bi, o);
            if (better(ok, oi, bk, bi)) {
                bk = ok;
                bi = oi;
            }
        }
        if (lane == 0) {
            s.best_k[w] = bk;
            s.best_i[w] = bi;
        }
        __syncthreads();
        if (w == 0) {
            bk = s.best_k[lane];
            bi = s.best_i[lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint32_t ok = __shfl_xor_sync(FULL, bk, o);
                const int oi = __shfl_xor_sync(FULL, bi, o);
                if (better(ok, oi, bk, bi)) {
                    bk = ok;
                    bi = oi;
                }
            }
            if (lane == 0) {
                *cluster.map_shared_rank(&s.red_k[rank], 0) = bk;
                *cluster.map_shared_rank(&s.red_i[rank], 0) = bi;
            }
        }
        cluster.sync();
        if (rank == 0 && tid == 0) {
            bk = s.red_k[0];
            bi = s.red_i[0];
            for (int r = 1; r < CL; ++r)
                if (better(s.red_k[r], s.red_i[r], bk, bi)) {
                    bk = s.red_k[r];
                    bi = s.red_i[r];
                }
            next_tok[b] = bi == 0x7fffffff ? 0 : bi;
        }
        return;
    }

    if (V <= CAND) {
        // Every token is a candidate.
        if (rank == 0) s.cand[tid] = tid < V ? entry(order_key(row[tid]), tid) : 0ull;
    } else {
        // Radix select of the CAND-th largest key t; afterwards krem = CAND - #{key > t}.
        uint32_t prefix = 0, pmask = 0;
        int krem = CAND;
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int bits = pass == 0 ? 12 : 10;
            const int shift = pass == 0 ? 20 : (pass == 1 ? 10 : 0);
            const int nb = 1 << bits;
            uint32_t *gh = s.ghist + (pass == 0 ? 0 : (pass == 1 ? HIST : HIST + 1024));
            for (int i = tid; i < n_loc; i += ST) {
                const uint32_t k = keys[i];
                if ((k & pmask) == prefix) atomicAdd(&s.hist[(k >> shift) & (nb - 1)], 1u);
            }
            __syncthreads();
            // Add the non-zero bins into every CTA's cluster histogram; clear them for the next
            // pass (whose counting starts after the cluster barrier below).
            for (int bin = tid; bin < nb; bin += ST) {
                const uint32_t c = s.hist[bin];
                if (c) {
                    s.hist[bin] = 0;
#pragma unroll
                    for (int r = 0; r < CL; ++r) atomicAdd(cluster.map_shared_rank(gh + bin, r), c);
                }
            }
            cluster.sync();  // every CTA's bins have landed everywhere
            // Thread tid owns the bins nb-1-tid*per .. nb-per-tid*per (descending); the owner
            // of the crossing finds the digit.
            const int per = nb / ST;
            int mine = 0;
            for (int j = 0; j < per; ++j) mine += (int)gh[nb - 1 - (tid * per + j)];
            int above = block_excl_scan(mine, s.iscan);
            if (above < krem && above + mine >= krem) {
                for (int j = 0; j < per; ++j) {
                    const int bin = nb - 1 - (tid * per + j);
                    const int c = (int)gh[bin];
                    if (above + c >= krem) {
                        s.digit = bin;
                        s.krem = krem - above;
                        break;
                    }
                    above += c;
                }
            }
            __syncthreads();
            prefix |= (uint32_t)s.digit << shift;
            pmask |= (uint32_t)(nb - 1) << shift;
            krem = s.krem;
        }
        const uint32_t t = prefix;
        const int need_eq = krem;            // candidates equal to t (>= 1)
        const int n_gt = CAND - need_eq;     // keys above t: all candidates

        // Counts per warp segment of the slice, then per CTA; each CTA adds its counts into
        // the bases of the CTAs after it.
        const int seg = (((n_loc + 31) / 32) + 31) & ~31;
        const int wb = w * seg, we = min(n_loc, wb + seg);
        int g = 0, e = 0;
        for (int base = wb; base < we; base += 32) {
            const int i = base + lane;
            const uint32_t k = i < we ? keys[i] : 0u;
            g += __popc(__ballot_sync(FULL, i < we && k > t));
            e += __popc(__ballot_sync(FULL, i < we && k == t));
        }
        if (lane == 0) {
            s.wgt[w] = g;
            s.weq[w] = e;
        }
        __syncthreads();
        if (w == 0) {
            int xg = s.wgt[lane], xe = s.weq[lane];
            const int g0 = xg, e0 = xe;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yg = __shfl_up_sync(FULL, xg, o);
                const int ye = __shfl_up_sync(FULL, xe, o);
                if (lane >= o) {
                    xg += yg;
                    xe += ye;
                }
            }
            s.wgt[lane] = xg - g0;
            s.weq[lane] = xe - e0;
            const int tot_g = __shfl_sync(FULL, xg, 31), tot_e = __shfl_sync(FULL, xe, 31);
            const int r = rank + 1 + lane;
            if (r < CL) {
                atomicAdd(cluster.map_shared_rank(&s.base_gt, r), tot_g);
                atomicAdd(cluster.map_shared_rank(&s.base_eq, r), tot_e);
            }
        }
        cluster.sync();  // every CTA's counts have landed
        int gt_base = s.base_gt + s.wgt[w], eq_base = s.base_eq + s.weq[w];
        uint64_t *cand0 = cluster.map_shared_rank(s.cand, 0);
        for (int base = wb; base < we; base += 32) {
            const int i = base + lane;
            const uint32_t k = i < we ? keys[i] : 0u;
            const bool gt = i < we && k > t, eq = i < we && k == t;
            const uint32_t bg = __ballot_sync(FULL, gt), be = __ballot_sync(FULL, eq);
            if (gt) {
                const int slot = gt_base + lanes_below(bg);
                if (slot < n_gt) cand0[slot] = entry(k, beg + i);  // exactly n_gt keys are above t
            }
            if (eq) {
                const int r = eq_base + lanes_below(be);
                if (r < need_eq) cand0[n_gt + r] = entry(t, beg + i);
            }
            gt_base += __popc(bg);
            eq_base += __popc(be);
        }
    }
    cluster.sync();  // the candidates have landed in the first CTA
    if (rank != 0) return;

    // Bitonic sort, descending: entry order = (logit desc, index asc).  Each thread holds one
    // entry; of a compare-exchange pair the lower position keeps the larger entry in a
    // descending block and the smaller in an ascending one.
    uint64_t x = s.cand[tid];
    uint64_t *const other = reinterpret_cast<uint64_t *>(s.hist);
    bool to_other = true;  // s.cand was last read above; the first shared exchange writes the other
#pragma unroll
    for (int size = 2; size <= CAND; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            uint64_t *buf = to_other ? other : s.cand;
            if (stride >= 32) to_other = !to_other;
            const uint64_t y = partner_value(x, stride, buf);
            const bool desc = (tid & size) == 0, lower = (tid & stride) == 0;
            x = (lower == desc) ? (x > y ? x : y) : (x < y ? x : y);
        }
    }
    __syncthreads();  // every exchange through s.cand has been read
    s.cand[tid] = x;
    __syncthreads();

    const int K = V < CAND ? V : CAND;
    int n = K;
    const int tk = top_k[b];
    if (tk >= 1 && tk < n) n = tk;
    const float v0 = key_value((uint32_t)(s.cand[0] >> 32));
    float p = 0.f;
    if (tid < n) p = expf((key_value((uint32_t)(x >> 32)) - v0) / T);
    const float cum = block_incl_scan(p, s.fscan);
    const float tp = top_p[b];
    if (tp < 1.f) {
        if (tid == n - 1) s.total = cum;
        __syncthreads();
        const float thr = tp * s.total;
        const int below = __syncthreads_count(tid < n && cum < thr);
        n = min(below + 1, n);
    }
    if (tid == n - 1) s.total = cum;
    __syncthreads();
    const float target = uniform[b] * s.total;
    const int at = min(__syncthreads_count(tid < n && cum <= target), n - 1);
    if (tid == 0) next_tok[b] = entry_index(s.cand[at]);
}

size_t sample_smem_bytes(int V) { return keys_offset() + KEYS_PAD + (size_t)((V + CL - 1) / CL) * 4; }

int fail(int code, const std::string &m) {
    set_last_error("qwen3_sample: " + m);
    return code;
}

}  // namespace

namespace q3 {

bool sample_supported(int V) { return V >= 1 && sample_smem_bytes(V) <= (size_t)MAX_SMEM; }

cudaError_t launch_sample(const Launch &lc, const float *logits, int B, int V, const float *temperature,
                          const int32_t *top_k, const float *top_p, const float *uniform, int32_t *next_tok) {
    const size_t smem = sample_smem_bytes(V);
    cudaError_t e = cudaFuncSetAttribute(k_sample, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B * CL);
    cfg.blockDim = dim3(ST);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (lc.counter) ++*lc.counter;
    return cudaLaunchKernelEx(&cfg, k_sample, logits, V, (V + CL - 1) / CL, temperature, top_k, top_p, uniform,
                              next_tok);
}

}  // namespace q3

extern "C" int qwen3_sample(const float *logits_dev, int32_t B, int32_t V, const float *temperature_dev,
                            const int32_t *top_k_dev, const float *top_p_dev, const float *uniform_dev,
                            int32_t *next_tok_dev, void *stream) {
    set_last_error("");
    if (!logits_dev || !temperature_dev || !top_k_dev || !top_p_dev || !uniform_dev || !next_tok_dev)
        return fail(QWEN3_E_INVALID, "NULL argument");
    if (B < 1 || B > 65535 || V < 1) return fail(QWEN3_E_INVALID, "bad B or V");
    if (!sample_supported(V))
        return fail(QWEN3_E_UNSUPPORTED, "V = " + std::to_string(V) + " exceeds the shared memory of a cluster (at most " +
                                             std::to_string((MAX_SMEM - keys_offset() - KEYS_PAD) / 4 * CL) + " tokens)");
    Launch lc;
    lc.stream = static_cast<cudaStream_t>(stream);
    lc.pdl = false;
    const cudaError_t e = launch_sample(lc, logits_dev, B, V, temperature_dev, top_k_dev, top_p_dev, uniform_dev,
                                        next_tok_dev);
    if (e != cudaSuccess) return fail(QWEN3_E_CUDA, cudaGetErrorString(e));
    return QWEN3_OK;
}
