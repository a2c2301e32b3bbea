// The token sampling chain on the GPU, one CTA per logits row ("Inside the
// inference engine: model architectures and forward pass", section "Token
// sampling pipeline": temperature 0 -> argmax, else Top-K -> Temperature ->
// Softmax -> Top-P -> Min-P -> weighted random sample; "LLama.cpp — how it
// works", "Steps 14–15: logits and sampling": a repeat penalty first).
//
//   1. repeat penalty: a bitmap of the distinct recent tokens in shared memory;
//      a marked logit is divided by the penalty if positive, else multiplied;
//   2. top-K: radix select of the K-th largest value over the whole row (four
//      8-bit passes on order-preserving keys, shared-memory histograms), then
//      the candidates are gathered in token-id order with a block-wide scan
//      (ties at the threshold take the lowest ids) and sorted by (value
//      descending, id ascending) with a bitonic sort;
//   3. temperature, softmax, top-P (shortest prefix reaching p), min-P
//      (probability >= min_p * top probability) and the draw with the given
//      uniform (first candidate whose running sum exceeds u * kept total).
//      Exponentials are computed in parallel; every sum is taken by one thread
//      in candidate order, so the float32 decisions do not depend on timing.
#include "common.cuh"
#include "launch.cuh"

namespace llm {

namespace {

constexpr int STHREADS = 1024;
constexpr int MAX_K = 1024;

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// exclusive block scan of one value per thread (STHREADS threads); returns the prefix, *total the sum
__device__ int block_scan(int v, int *ws, int *total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = ws[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        ws[lane] = w;
    }
    __syncthreads();
    const int before = (warp > 0 ? ws[warp - 1] : 0) + x - v;
    *total = ws[31];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(STHREADS) sample_kernel(const float *logits, int V, SampleParams p,
                                                          const float *u, const int *history, int n_hist,
                                                          int *out) {
    extern __shared__ __align__(16) uint32_t bitmap[];          // V bits
    __shared__ unsigned hist[256];
    __shared__ unsigned long long ck[MAX_K];                    // sort keys: value key << 32 | ~id
    __shared__ float ce[MAX_K];                                 // exp / probabilities of the candidates
    __shared__ int ws[32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    __shared__ float s_best_v[32];
    __shared__ int s_best_i[32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    const float *lg = logits + (size_t)row * V;

    if (p.temperature <= 0.f) {
        // greedy: argmax, ties to the lowest id
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int v = tid; v < V; v += STHREADS) {
            const float x = lg[v];
            if (x > bv || (x == bv && v < bi)) { bv = x; bi = v; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { s_best_v[warp] = bv; s_best_i[warp] = bi; }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < STHREADS / 32; ++w)
                if (s_best_v[w] > bv || (s_best_v[w] == bv && s_best_i[w] < bi)) { bv = s_best_v[w]; bi = s_best_i[w]; }
            out[row] = bi == 0x7fffffff ? 0 : bi;
        }
        return;
    }

    // ---- 1. distinct recent tokens
    const int nb = (V + 31) / 32;
    for (int i = tid; i < nb; i += STHREADS) bitmap[i] = 0u;
    __syncthreads();
    const bool pen = p.repeat_penalty != 1.f && p.penalty_last_n > 0;
    if (pen) {
        const int h0 = n_hist > p.penalty_last_n ? n_hist - p.penalty_last_n : 0;
        for (int i = h0 + tid; i < n_hist; i += STHREADS) {
            const int t = history[i];
            if (t >= 0 && t < V) atomicOr(&bitmap[t >> 5], 1u << (t & 31));
        }
    }
    __syncthreads();
    const float rp = p.repeat_penalty;
    auto value = [&](int v) -> float {
        float x = lg[v];
        if (pen && (bitmap[v >> 5] >> (v & 31) & 1u)) x = x > 0.f ? x / rp : x * rp;
        return x;
    };

    // ---- 2. radix select of the K-th largest key
    const int K = p.top_k;
    uint32_t prefix = 0u, mask = 0u;
    int need = K;
    for (int d = 3; d >= 0; --d) {
        for (int i = tid; i < 256; i += STHREADS) hist[i] = 0u;
        __syncthreads();
        for (int v = tid; v < V; v += STHREADS) {
            const uint32_t k = order_key(value(v));
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> (8 * d)) & 255u], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            int cum = 0, b = 255;
            for (; b > 0; --b) {
                if (cum + (int)hist[b] >= need) break;
                cum += (int)hist[b];
            }
            s_prefix = prefix | ((uint32_t)b << (8 * d));
            s_need = need - cum;
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        mask |= 255u << (8 * d);
        __syncthreads();
    }
    const uint32_t thr = prefix;              // the K-th largest key; `need` of its copies are taken

    // gather in id order: each thread owns a contiguous range of ids
    const int per = (V + STHREADS - 1) / STHREADS;
    const int v0 = tid * per, v1 = min(V, v0 + per);
    int n_gt = 0, n_eq = 0;
    for (int v = v0; v < v1; ++v) {
        const uint32_t k = order_key(value(v));
        n_gt += k > thr;
        n_eq += k == thr;
    }
    int tot_gt, tot_eq;
    int pos_gt = block_scan(n_gt, ws, &tot_gt);
    int pos_eq = block_scan(n_eq, ws, &tot_eq);
    for (int v = v0; v < v1; ++v) {
        const float x = value(v);
        const uint32_t k = order_key(x);
        if (k > thr) {
            if (pos_gt < K) ck[pos_gt] = ((unsigned long long)k << 32) | (uint32_t)(~(uint32_t)v);
            ++pos_gt;
        } else if (k == thr) {
            if (pos_eq < need && tot_gt + pos_eq < K)
                ck[tot_gt + pos_eq] = ((unsigned long long)k << 32) | (uint32_t)(~(uint32_t)v);
            ++pos_eq;
        }
    }
    // pad to a power of two with the smallest key and sort descending
    int n2 = 1;
    while (n2 < K) n2 <<= 1;
    for (int i = K + tid; i < n2; i += STHREADS) ck[i] = 0ull;
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2; i += STHREADS) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const unsigned long long a = ck[i], b = ck[j];
                    if (desc ? (a < b) : (a > b)) { ck[i] = b; ck[j] = a; }
                }
            }
            __syncthreads();
        }
    }

    // ---- 3. temperature, softmax, top-P, min-P, draw
    const float T = p.temperature;
    const float s0 = key_value((uint32_t)(ck[0] >> 32)) / T;
    for (int i = tid; i < K; i += STHREADS) ce[i] = expf(key_value((uint32_t)(ck[i] >> 32)) / T - s0);
    __syncthreads();
    if (tid == 0) {
        float z = 0.f;
        for (int i = 0; i < K; ++i) z += ce[i];
        ws[0] = __float_as_int(z);
    }
    __syncthreads();
    const float z = __int_as_float(ws[0]);
    for (int i = tid; i < K; i += STHREADS) ce[i] = ce[i] / z;
    __syncthreads();
    if (tid == 0) {
        int keep = K;
        if (p.top_p < 1.f) {
            float c = 0.f;
            for (int i = 0; i < K; ++i) {
                c += ce[i];
                if (c >= p.top_p) { keep = i + 1; break; }
            }
        }
        if (p.min_p > 0.f) {
            const float t = p.min_p * ce[0];
            int m = 0;
            while (m < keep && ce[m] >= t) ++m;
            keep = m > 1 ? m : 1;
        }
        float total = 0.f;
        for (int i = 0; i < keep; ++i) total += ce[i];
        const float target = u[row] * total;
        int choice = keep - 1;
        float c = 0.f;
        for (int i = 0; i < keep; ++i) {
            c += ce[i];
            if (c > target) { choice = i; break; }
        }
        out[row] = (int)(~(uint32_t)(ck[choice] & 0xFFFFFFFFull));
    }
}

}  // namespace

size_t sample_smem_bytes(int V) { return (size_t)((V + 31) / 32) * sizeof(uint32_t); }

cudaError_t launch_sample(const float *logits, int n_rows, int V, const SampleParams &p, const float *u,
                          const int *history, int n_hist, int *out, const Launch &l) {
    if (n_rows < 1 || V < 1 || (p.temperature > 0.f && (p.top_k < 1 || p.top_k > MAX_K || p.top_k > V)))
        return cudaErrorInvalidValue;
    return launch_kernel(sample_kernel, dim3(n_rows), dim3(STHREADS), sample_smem_bytes(V), l, logits, V, p, u,
                         history, n_hist, out);
}

cudaError_t init_sample_attributes() { return allow_smem(sample_kernel, 96 * 1024); }

}  // namespace llm
