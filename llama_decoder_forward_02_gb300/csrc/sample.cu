// The token sampling chain on the GPU ("Inside the inference engine: model
// architectures and forward pass", section "Token sampling pipeline":
// temperature 0 -> argmax, else Top-K -> Temperature -> Softmax -> Top-P ->
// Min-P -> weighted random sample; "LLama.cpp — how it works", "Steps 14–15:
// logits and sampling": a repeat penalty first).
//
// One row is taken by a cluster of ROW_CLUSTER CTAs; CTA r owns the slice
// [r * S, r * S + len) of the row and holds it in shared memory as 32-bit
// order-preserving keys, so the row is read from global memory once.
//
//   1. repeat penalty: the distinct recent tokens that fall in a CTA's slice
//      are marked in a shared bitmap; the thread that sets a token's bit
//      divides its logit by the penalty if positive, else multiplies it;
//   2. top-K: radix select of the K-th largest key over the row (four 8-bit
//      passes; each CTA counts its slice into per-warp shared histograms and
//      adds the 256 totals into every CTA of the cluster through distributed
//      shared memory, so every CTA picks the same digit); then the candidates
//      are gathered in token-id order (ballots within a warp, a block scan
//      across warps, the slice counts across CTAs), ties at the threshold
//      taking the lowest ids, into rank 0, which ranks them by (value
//      descending, id ascending);
//   3. rank 0: temperature, softmax, top-P (shortest prefix reaching p), min-P
//      (probability >= min_p * top probability) and the draw with the given
//      uniform (first candidate whose running sum exceeds u * kept total).
//      Exponentials and searches are parallel; the two running sums (the
//      softmax normaliser and the cumulative probabilities) are taken by one
//      thread in candidate order, so the float32 decisions do not depend on
//      timing.
#include "common.cuh"
#include "launch.cuh"
#include "cluster.cuh"

namespace llm {

namespace {

constexpr int STHREADS = 1024;
constexpr int NWARP = STHREADS / 32;
constexpr int MAX_K = 1024;
constexpr int MAX_SLICE = SAMPLE_MAX_VOCAB / ROW_CLUSTER;   // keys per CTA

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// exclusive block scan of one value per thread; returns the prefix, *total the sum
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

// Digit of the K-th largest key from a 256-bin histogram: scanning bins from
// 255 down, the first bin b where the count through b reaches `need` (bin 0
// if none); *need_left = need minus the count of the bins above b.  Warp 0
// only: lane l holds bins 255 - 8l - j, j = 0..7.
__device__ void pick_digit(const unsigned *tot, int need, int *digit, int *need_left) {
    const int lane = threadIdx.x & 31;
    int c[8], s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) { c[j] = (int)tot[255 - 8 * lane - j]; s += c[j]; }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
    const int L = hit ? __ffs(hit) - 1 : 31;
    if (lane == L) {
        int cum = incl - s, b = 255 - 8 * lane - 7;
#pragma unroll
        for (int j = 0; j < 7; ++j) {
            if (cum + c[j] >= need) { b = 255 - 8 * lane - j; break; }
            cum += c[j];
        }
        *digit = b;
        *need_left = need - cum;
    }
}

__global__ void __launch_bounds__(STHREADS, 1) sample_kernel(const float *logits, int V, SampleParams p,
                                                          const float *u, const int *history, int n_hist,
                                                          int *out) {
    extern __shared__ __align__(16) uint32_t dsm[];
    __shared__ unsigned tot[2][256];                 // cluster-wide digit counts, by pass parity
    __shared__ unsigned cnt[ROW_CLUSTER][2];         // per-rank counts above / at the threshold
    __shared__ unsigned long long ck[MAX_K];         // rank 0: candidates, value key << 32 | ~id
    __shared__ float ce[MAX_K];                      // rank 0: exponentials, then probabilities
    __shared__ float cum[MAX_K];                     // rank 0: running sums of the probabilities
    __shared__ int ws[32];
    __shared__ int s_digit, s_need, s_first;

    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x / ROW_CLUSTER;
    const float *lg = logits + (size_t)row * V;

    if (p.temperature <= 0.f) {                      // greedy
        const int best = cluster_row_argmax(lg, V);
        if (best >= 0 && tid == 0) out[row] = best;
        return;
    }

    const uint32_t rank = cluster_rank();
    const int S = row_slice_len(V);
    const int lo = (int)rank * S, len = max(0, min(S, V - lo));
    uint32_t *key = dsm;                             // [S] keys of the slice
    uint32_t *bm = dsm + S;                          // [S / 32] penalty marks
    unsigned *hist_w = bm + S / 32;                  // [NWARP][256] per-warp histograms
    unsigned *my_hist = hist_w + warp * 256;
    const uint4 *key4 = reinterpret_cast<const uint4 *>(key);
    const int n4 = len >> 2;

    // ---- load the slice as keys; clear the marks and the first pass's totals
    for (int i = tid; i < S / 32; i += STHREADS) bm[i] = 0u;
    if (tid < 256) tot[0][tid] = 0u;
    cluster_arrive();                                // totals zeroed before any CTA adds (wait below)
    {
        const float4 *src = reinterpret_cast<const float4 *>(lg + lo);
        uint4 *dst = reinterpret_cast<uint4 *>(key);
        for (int i0 = tid; i0 < n4; i0 += 4 * STHREADS) {
            float4 q[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (i0 + j * STHREADS < n4) q[j] = __ldg(src + i0 + j * STHREADS);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (i0 + j * STHREADS < n4)
                    dst[i0 + j * STHREADS] = make_uint4(order_key(q[j].x), order_key(q[j].y), order_key(q[j].z),
                                                        order_key(q[j].w));
        }
    }
    __syncthreads();
    // ---- 1. repeat penalty on the distinct recent tokens of this slice
    if (p.repeat_penalty != 1.f && p.penalty_last_n > 0) {
        const float rp = p.repeat_penalty;
        const int h0 = n_hist > p.penalty_last_n ? n_hist - p.penalty_last_n : 0;
        for (int i = h0 + tid; i < n_hist; i += STHREADS) {
            const int t = history[i] - lo;
            if (t >= 0 && t < len) {
                const uint32_t bit = 1u << (t & 31);
                if (!(atomicOr(&bm[t >> 5], bit) & bit)) {
                    const float x = key_value(key[t]);
                    key[t] = order_key(x > 0.f ? x / rp : x * rp);
                }
            }
        }
    }
    cluster_wait();

    // ---- 2. radix select of the K-th largest key
    const int K = p.top_k;
    uint32_t prefix = 0u, mask = 0u;
    int need = K;
    for (int d = 3; d >= 0; --d) {
        const int q = (3 - d) & 1;
        for (int i = tid; i < NWARP * 256; i += STHREADS) hist_w[i] = 0u;
        if (tid < 256) tot[q ^ 1][tid] = 0u;         // next pass's totals, last read a pass ago
        __syncthreads();
        for (int i = tid; i < n4; i += STHREADS) {
            const uint4 k4 = key4[i];
            const uint32_t k[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if ((k[e] & mask) == prefix) atomicAdd(&my_hist[(k[e] >> (8 * d)) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 256) {
            unsigned t = 0u;
#pragma unroll 8
            for (int w = 0; w < NWARP; ++w) t += hist_w[w * 256 + tid];
            if (t)
                for (int r = 0; r < ROW_CLUSTER; ++r) dsmem_add_u32(dsmem(&tot[q][tid], (uint32_t)r), t);
        }
        cluster_sync();
        if (warp == 0) pick_digit(tot[q], need, &s_digit, &s_need);
        __syncthreads();
        prefix |= (uint32_t)s_digit << (8 * d);
        need = s_need;
        mask |= 255u << (8 * d);
    }
    const uint32_t thr = prefix;              // the K-th largest key; `need` of its copies are taken

    // ---- gather in id order: warp w owns [w * per, (w+1) * per) of the slice
    // (per a multiple of 128), read 128 keys at a time as one uint4 per lane;
    // the four ballots of a group rank each hit in id order (lane, then
    // element); a block scan orders the warps and the cluster counts the CTAs
    const int per = ((len + NWARP - 1) / NWARP + 127) / 128 * 128;
    const int w0 = min(len, warp * per), w1 = min(len, w0 + per);
    const unsigned below = (1u << lane) - 1u;
    int n_gt = 0, n_eq = 0;
    for (int b0 = w0; b0 < w1; b0 += 128) {
        const int i = b0 + lane * 4;
        const uint4 k4 = i < w1 ? key4[i >> 2] : make_uint4(0, 0, 0, 0);
        const uint32_t k[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            n_gt += __popc(__ballot_sync(0xffffffffu, k[e] > thr));
            n_eq += __popc(__ballot_sync(0xffffffffu, k[e] == thr && k[e] != 0u));
        }
    }
    int cta_gt, cta_eq;
    int pos_gt = block_scan(lane == 0 ? n_gt : 0, ws, &cta_gt);
    int pos_eq = block_scan(lane == 0 ? n_eq : 0, ws, &cta_eq);
    pos_gt = __shfl_sync(0xffffffffu, pos_gt, 0);
    pos_eq = __shfl_sync(0xffffffffu, pos_eq, 0);
    if (tid < ROW_CLUSTER) {                         // this CTA's counts, into every CTA's slot `rank`
        dsmem_st_u32(dsmem(&cnt[rank][0], (uint32_t)tid), (uint32_t)cta_gt);
        dsmem_st_u32(dsmem(&cnt[rank][1], (uint32_t)tid), (uint32_t)cta_eq);
    }
    cluster_sync();
    int tot_gt = 0;
    for (int r = 0; r < ROW_CLUSTER; ++r) {
        tot_gt += (int)cnt[r][0];
        if (r < (int)rank) { pos_gt += (int)cnt[r][0]; pos_eq += (int)cnt[r][1]; }
    }
    for (int b0 = w0; b0 < w1; b0 += 128) {
        const int i = b0 + lane * 4;
        const uint4 k4 = i < w1 ? key4[i >> 2] : make_uint4(0, 0, 0, 0);
        const uint32_t k[4] = {k4.x, k4.y, k4.z, k4.w};
        unsigned bg[4], be[4];
        int cg = 0, cq = 0;                          // hits of this group in lower lanes
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            bg[e] = __ballot_sync(0xffffffffu, k[e] > thr);
            be[e] = __ballot_sync(0xffffffffu, k[e] == thr && k[e] != 0u);
            cg += __popc(bg[e] & below);
            cq += __popc(be[e] & below);
        }
        int rg = pos_gt + cg, re = pos_eq + cq;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const unsigned long long kv = ((unsigned long long)k[e] << 32) | (uint32_t)(~(uint32_t)(lo + i + e));
            if (bg[e] >> lane & 1u) {
                if (rg < K) dsmem_st_u64(dsmem(&ck[rg], 0), kv);
                ++rg;
            }
            if (be[e] >> lane & 1u) {
                if (re < need && tot_gt + re < K) dsmem_st_u64(dsmem(&ck[tot_gt + re], 0), kv);
                ++re;
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            pos_gt += __popc(bg[e]);
            pos_eq += __popc(be[e]);
        }
    }
    cluster_sync();
    if (rank != 0) return;

    // ---- rank the K candidates by key, descending (keys are distinct: ids differ)
    unsigned long long *sorted = reinterpret_cast<unsigned long long *>(hist_w);
    for (int i = tid; i < K; i += STHREADS) {
        const unsigned long long mine = ck[i];
        int r = 0;
#pragma unroll 8
        for (int j = 0; j < K; ++j) r += ck[j] > mine;
        sorted[r] = mine;
    }
    __syncthreads();

    // ---- 3. temperature, softmax, top-P, min-P, draw
    const float T = p.temperature;
    const float s0 = key_value((uint32_t)(sorted[0] >> 32)) / T;
    for (int i = tid; i < K; i += STHREADS) ce[i] = expf(key_value((uint32_t)(sorted[i] >> 32)) / T - s0);
    __syncthreads();
    if (tid == 0) {
        float z = 0.f;
#pragma unroll 8
        for (int i = 0; i < K; ++i) z += ce[i];
        ws[0] = __float_as_int(z);
    }
    __syncthreads();
    const float z = __int_as_float(ws[0]);
    for (int i = tid; i < K; i += STHREADS) ce[i] = ce[i] / z;
    __syncthreads();
    if (tid == 0) {
        float c = 0.f;
#pragma unroll 8
        for (int i = 0; i < K; ++i) { c += ce[i]; cum[i] = c; }
        s_first = K;
    }
    __syncthreads();
    int keep = K;
    if (p.top_p < 1.f) {                             // shortest prefix whose sum reaches p
        for (int i = tid; i < K; i += STHREADS)
            if (cum[i] >= p.top_p) atomicMin(&s_first, i + 1);
        __syncthreads();
        keep = s_first;
        __syncthreads();
    }
    if (p.min_p > 0.f) {                             // leading run with prob >= min_p * top
        const float t = p.min_p * ce[0];
        if (tid == 0) s_first = keep;
        __syncthreads();
        for (int i = tid; i < keep; i += STHREADS)
            if (!(ce[i] >= t)) atomicMin(&s_first, i);
        __syncthreads();
        keep = max(s_first, 1);
        __syncthreads();
    }
    const float target = u[row] * cum[keep - 1];
    if (tid == 0) s_first = keep - 1;
    __syncthreads();
    for (int i = tid; i < keep; i += STHREADS)
        if (cum[i] > target) atomicMin(&s_first, i);
    __syncthreads();
    if (tid == 0) out[row] = (int)(~(uint32_t)(sorted[s_first] & 0xFFFFFFFFull));
}

}  // namespace

size_t sample_smem_bytes(int V) {
    const size_t S = (size_t)row_slice_len(V);
    return (S + S / 32 + (size_t)NWARP * 256) * sizeof(uint32_t);
}

cudaError_t launch_sample(const float *logits, int n_rows, int V, const SampleParams &p, const float *u,
                          const int *history, int n_hist, int *out, const Launch &l) {
    // rows are read as float4 (V a multiple of 4, a 16-byte aligned base) and
    // a CTA's slice of a row fits its shared memory
    if (n_rows < 1 || V < 4 || V % 4 || V > ROW_CLUSTER * MAX_SLICE ||
        (reinterpret_cast<uintptr_t>(logits) & 15u) ||
        (p.temperature > 0.f && (p.top_k < 1 || p.top_k > MAX_K || p.top_k > V)))
        return cudaErrorInvalidValue;
    return launch_cluster_kernel(sample_kernel, dim3(n_rows * ROW_CLUSTER), dim3(STHREADS), ROW_CLUSTER,
                                 p.temperature > 0.f ? sample_smem_bytes(V) : 0, l, logits, V, p, u, history,
                                 n_hist, out);
}

cudaError_t init_sample_attributes() {
    return allow_smem(sample_kernel, sample_smem_bytes(ROW_CLUSTER * MAX_SLICE));
}

}  // namespace llm
