// Small kernels of the forward pass: token embedding (with the first
// RMSNorm's input for prefill), row gather (last-layer output rows), greedy
// argmax and the on-device greedy feedback used by llm_generate.
#include "common.cuh"
#include "launch.cuh"
#include "cluster.cuh"

namespace llm {

namespace {

// "LLama.cpp — how it works", "Step 11: tokens become embeddings": row
// token[t] of the embedding table becomes input row t.  fp16 -> fp32 is exact.
// For decode-sized inputs it also leaves the per-64-column sums of squares
// that the next GEMV's fused RMSNorm reads.
__global__ void __launch_bounds__(128) embed_kernel(const f16 *E, const int *tok, int d, int n_vocab,
                                                    float *h, float *ss_part, uint32_t *err) {
    const int t = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    int id = tok[t];
    const bool ok = id >= 0 && id < n_vocab;
    if (!ok && tid == 0) raise_error(err, ERRF_BAD_TOKEN);
    const uint4 *src = reinterpret_cast<const uint4 *>(E + (size_t)(ok ? id : 0) * d);
    float4 *dst = reinterpret_cast<float4 *>(h + (size_t)t * d);
    const int nchunk = d / 8;                       // 8 bf16 per chunk, 8 chunks per 64 columns
    for (int base = 0; base < nchunk; base += 128) {
        const int c = base + tid;
        float sq = 0.f;
        if (c < nchunk) {
            uint4 v = ok ? src[c] : make_uint4(0, 0, 0, 0);
            const float4 a = make_float4(h2lo(v.x), h2hi(v.x), h2lo(v.y), h2hi(v.y));
            const float4 b = make_float4(h2lo(v.z), h2hi(v.z), h2lo(v.w), h2hi(v.w));
            dst[2 * c] = a;
            dst[2 * c + 1] = b;
            sq = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
        }
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 2);
        sq += __shfl_xor_sync(0xffffffffu, sq, 4);
        if (ss_part && c < nchunk && (c & 7) == 0) ss_part[(c >> 3) * 8 + t] = sq;
    }
}

// Prefill embedding with the first RMSNorm's input: h[t] = E[tok[t]] (fp32),
// x[t] = f16(h[t] * gain) and the per-32-column partial sums of h^2,
// ss32[t][d/32], which the first QKV GEMM turns into the row's scale.  Each
// thread takes 8 consecutive columns (16-byte loads); four lanes make a
// 32-column group.
__global__ void __launch_bounds__(128) embed_norm_kernel(const f16 *E, const int *tok, int d, int n_vocab,
                                                         float *h, const float *gain, f16 *x, float *ss32,
                                                         uint32_t *err) {
    const int t = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const int id = tok[t];
    const bool ok = id >= 0 && id < n_vocab;
    if (!ok && tid == 0) raise_error(err, ERRF_BAD_TOKEN);
    const uint4 *src = reinterpret_cast<const uint4 *>(E + (size_t)(ok ? id : 0) * d);
    float4 *hd = reinterpret_cast<float4 *>(h + (size_t)t * d);
    uint4 *xd = reinterpret_cast<uint4 *>(x + (size_t)t * d);
    const float4 *g4 = reinterpret_cast<const float4 *>(gain);
    for (int base = 0; base < d / 8; base += 128) {      // every lane runs every pass (the shuffles)
        const int c = base + tid;
        const bool in = c < d / 8;                       // d % 32 == 0: whole 4-lane groups
        const uint4 v = ok && in ? src[c] : make_uint4(0, 0, 0, 0);
        const float4 a = make_float4(h2lo(v.x), h2hi(v.x), h2lo(v.y), h2hi(v.y));
        const float4 b = make_float4(h2lo(v.z), h2hi(v.z), h2lo(v.w), h2hi(v.w));
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 ga = in ? g4[2 * c] : z, gb = in ? g4[2 * c + 1] : z;
        if (in) {
            hd[2 * c] = a;
            hd[2 * c + 1] = b;
            const float xv[8] = {a.x * ga.x, a.y * ga.y, a.z * ga.z, a.w * ga.w, b.x * gb.x, b.y * gb.y, b.z * gb.z, b.w * gb.w};
            bool bad = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) bad |= f16_bad(xv[j]);
            if (bad) raise_error(err, ERRF_F16_RANGE);
            xd[c] = make_uint4(pack_h2(xv[0], xv[1]), pack_h2(xv[2], xv[3]), pack_h2(xv[4], xv[5]), pack_h2(xv[6], xv[7]));
        }
        float sq = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 2);
        if (in && (c & 3) == 0) ss32[(size_t)t * (d / 32) + c / 4] = sq;
    }
}

__global__ void __launch_bounds__(256) gather_kernel(const float *src, const int *rows, int d, float *dst,
                                                     const float *ss_src, float *ss_dst, const f16 *x_src,
                                                     f16 *x_dst, const float *ss32_src, float *ss32_dst) {
    const int r = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const int s = rows[r];
    const float4 *a = reinterpret_cast<const float4 *>(src + (size_t)s * d);
    float4 *b = reinterpret_cast<float4 *>(dst + (size_t)r * d);
    for (int i = tid; i < d / 4; i += 256) b[i] = a[i];
    if (ss_src)
        for (int p = tid; p < d / 64; p += 256) ss_dst[p * 8 + r] = ss_src[p * 8 + s];
    if (x_src) {
        const uint4 *xa = reinterpret_cast<const uint4 *>(x_src + (size_t)s * d);
        uint4 *xb = reinterpret_cast<uint4 *>(x_dst + (size_t)r * d);
        for (int i = tid; i < d / 8; i += 256) xb[i] = xa[i];
        for (int p = tid; p < d / 32; p += 256) ss32_dst[(size_t)r * (d / 32) + p] = ss32_src[(size_t)s * (d / 32) + p];
    }
}

// Greedy choice: the row argmax by a cluster of ROW_CLUSTER CTAs, each
// reading an eighth of the row (cluster_row_argmax); rank 0 writes.
__global__ void __launch_bounds__(1024) argmax_kernel(const float *logits, int n_vocab, int *out) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x / ROW_CLUSTER;
    const int best = cluster_row_argmax(logits + (size_t)r * n_vocab, n_vocab);
    if (best >= 0 && threadIdx.x == 0) out[r] = best;
}

__global__ void __launch_bounds__(1024) argmax_feed_kernel(const float *logits, int n_vocab, int *tokens_out,
                                                           int *step, const int *n_steps, int *next_tok, int *pos,
                                                           int advance) {
    pdl_wait();
    pdl_trigger();
    const int best = cluster_row_argmax(logits, n_vocab);
    if (best >= 0 && threadIdx.x == 0) {
        const int k = *step;
        if (k < *n_steps) tokens_out[k] = best;
        *step = k + 1;
        next_tok[0] = best;
        pos[0] += advance;
    }
}

__global__ void copy_kernel(const float *src, float *dst, size_t n) {
    pdl_wait();
    pdl_trigger();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

// Model set-up: widen bf16 norm gains to fp32.
__global__ void widen_kernel(const bf16 *src, float *dst, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = bf16f(src[i]);
}

// Model set-up: bf16 -> fp16 of a row block (dst may have a longer row
// pitch; its padding is left as is).  Out-of-range values raise the flag.
__device__ __forceinline__ f16 to_f16_checked(bf16 v, uint32_t *err) {
    const float f = bf16f(v);
    if (!(fabsf(f) <= 65504.0f)) raise_error(err, ERRF_BAD_INDEX);
    return f2h(f);
}

__global__ void convert_rows_kernel(const bf16 *src, int src_ld, f16 *dst, int dst_ld, int rows, int cols,
                                    uint32_t *err) {
    const int r = blockIdx.x;
    if (r >= rows) return;
    for (int c = threadIdx.x; c < cols; c += blockDim.x)
        dst[(size_t)r * dst_ld + c] = to_f16_checked(src[(size_t)r * src_ld + c], err);
}

// Model set-up: pack gate and up [F][d] into [2*F_pad][d] with groups of
// GU_GROUP gate rows followed by the GU_GROUP up rows of the same indices;
// rows past F are zero.
__global__ void repack_gate_up_kernel(const bf16 *gate, const bf16 *up, int F, int d, f16 *dst, uint32_t *err) {
    const int p = blockIdx.x;
    const int blk = p / (2 * GU_GROUP), r = p % (2 * GU_GROUP);
    const int src_row = blk * GU_GROUP + (r % GU_GROUP);
    f16 *o = dst + (size_t)p * d;
    if (src_row >= F) {
        for (int c = threadIdx.x; c < d; c += blockDim.x) o[c] = f2h(0.f);
        return;
    }
    const bf16 *src = (r < GU_GROUP ? gate : up) + (size_t)src_row * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) o[c] = to_f16_checked(src[c], err);
}

}  // namespace

cudaError_t launch_embed(const f16 *E, const int *tok, int T, int d, int n_vocab, float *h,
                         float *ss_part, uint32_t *err, const Launch &l, const float *gain, f16 *x, float *ss32) {
    if (T < 1 || d % 64) return cudaErrorInvalidValue;
    if (gain) {
        if (d % 32) return cudaErrorInvalidValue;
        return launch_kernel(embed_norm_kernel, dim3(T), dim3(128), 0, l, E, tok, d, n_vocab, h, gain, x, ss32, err);
    }
    return launch_kernel(embed_kernel, dim3(T), dim3(128), 0, l, E, tok, d, n_vocab, h,
                         T <= 8 ? ss_part : (float *)nullptr, err);
}

cudaError_t launch_gather_rows(const float *src, const int *rows, int n_rows, int d, float *dst,
                               const float *ss_src, float *ss_dst, const Launch &l, const f16 *x_src, f16 *x_dst,
                               const float *ss32_src, float *ss32_dst) {
    if (n_rows < 1) return cudaSuccess;
    return launch_kernel(gather_kernel, dim3(n_rows), dim3(256), 0, l, src, rows, d, dst, ss_src, ss_dst, x_src,
                         x_dst, ss32_src, ss32_dst);
}

cudaError_t launch_argmax(const float *logits, int n_rows, int n_vocab, int *out, const Launch &l) {
    if (n_rows < 1) return cudaSuccess;
    if (n_vocab < 4 || n_vocab % 4 || (reinterpret_cast<uintptr_t>(logits) & 15u)) return cudaErrorInvalidValue;
    return launch_cluster_kernel(argmax_kernel, dim3(n_rows * ROW_CLUSTER), dim3(1024), ROW_CLUSTER, 0, l, logits,
                                 n_vocab, out);
}

cudaError_t launch_argmax_feed(const float *logits, int n_vocab, int *tokens_out, int *step, const int *n_steps,
                               int *next_tok, int *pos, int advance, const Launch &l) {
    if (n_vocab < 4 || n_vocab % 4 || (reinterpret_cast<uintptr_t>(logits) & 15u)) return cudaErrorInvalidValue;
    return launch_cluster_kernel(argmax_feed_kernel, dim3(ROW_CLUSTER), dim3(1024), ROW_CLUSTER, 0, l, logits,
                                 n_vocab, tokens_out, step, n_steps, next_tok, pos, advance);
}

cudaError_t launch_copy_f32(const float *src, float *dst, size_t n, const Launch &l) {
    if (!n) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    return launch_kernel(copy_kernel, dim3(blocks), dim3(256), 0, l, src, dst, n);
}

}  // namespace llm

namespace llm {

cudaError_t launch_widen_bf16(const bf16 *src, float *dst, int n, cudaStream_t st) {
    widen_kernel<<<(n + 255) / 256, 256, 0, st>>>(src, dst, n);
    return cudaGetLastError();
}

cudaError_t launch_repack_gate_up(const bf16 *gate, const bf16 *up, int F, int F_pad, int d, f16 *dst,
                                  uint32_t *err, cudaStream_t st) {
    repack_gate_up_kernel<<<2 * F_pad, 128, 0, st>>>(gate, up, F, d, dst, err);
    return cudaGetLastError();
}

cudaError_t launch_convert_rows(const bf16 *src, int src_ld, f16 *dst, int dst_ld, int rows, int cols,
                                uint32_t *err, cudaStream_t st) {
    if (rows < 1) return cudaSuccess;
    convert_rows_kernel<<<rows, 256, 0, st>>>(src, src_ld, dst, dst_ld, rows, cols, err);
    return cudaGetLastError();
}

}  // namespace llm

namespace llm {

namespace {

// Context shift of one sequence's cache ("Inside the inference engine: model
// architectures and forward pass", "KV Cache": when the cache is full the
// model's Shift function adjusts the RoPE position encoding so the window
// slides forward without discarding the whole context).  Positions
// [p0, p0 + n) are dropped; the row at position p in [p0 + n, end) moves to
// p - n, its key re-rotated by the RoPE rotation of -n (rotations compose),
// its value copied.  One CTA per (layer, kv head) walks the rows upward in
// blocks of SHIFT_ROWS: a block is read whole (into registers) before it is
// written n rows lower, and every row a block overwrites lies below the next
// block's rows, so nothing is overwritten before it is read.
constexpr int SHIFT_ROWS = 16, SHIFT_THREADS = 128;

// P: one element pair of the cache, f16x2 (uint32_t) or FP8 E4M3 x2 (uint16_t).
template <class P>
__global__ void __launch_bounds__(SHIFT_THREADS) kv_shift_kernel(P *kc, P *vc, int n_ctx, int hd, int p0, int n,
                                                                 int end, const float2 *rope) {
    const size_t base = (size_t)blockIdx.x * n_ctx * hd / 2;    // (layer, head) block of this sequence, in pairs
    P *k32 = kc + base;
    P *v32 = vc + base;
    const int half = hd / 2;                                // element pairs per row
    const float2 *cs = rope + (size_t)n * half;             // cos, sin of n * theta_i
    constexpr int PER = SHIFT_ROWS * 64 / SHIFT_THREADS;    // pairs per thread (hd <= 128)
    for (int r0 = p0 + n; r0 < end; r0 += SHIFT_ROWS) {
        const int rows = end - r0 < SHIFT_ROWS ? end - r0 : SHIFT_ROWS;
        P kk[PER], vv[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int idx = threadIdx.x + j * SHIFT_THREADS;    // pair index within the block
            if (idx < rows * half) {
                const int row = idx / half, i = idx - row * half;
                const size_t off = (size_t)(r0 + row) * half + i;
                float2 f;
                if constexpr (sizeof(P) == 2) {
                    const uint32_t h = e4m3x2_to_h2(k32[off]);
                    f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
                } else {
                    f = __half22float2(*reinterpret_cast<const __half2 *>(k32 + off));
                }
                const float2 c = cs[i];
                // R(-n): (a, b) -> (a cos + b sin, -a sin + b cos)
                const float r0v = f.x * c.x + f.y * c.y, r1v = -f.x * c.y + f.y * c.x;
                if constexpr (sizeof(P) == 2) kk[j] = pack_e4m3x2(r0v, r1v);
                else kk[j] = pack_h2(r0v, r1v);
                vv[j] = v32[off];
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int idx = threadIdx.x + j * SHIFT_THREADS;
            if (idx < rows * half) {
                const int row = idx / half, i = idx - row * half;
                const size_t off = (size_t)(r0 + row - n) * half + i;
                k32[off] = kk[j];
                v32[off] = vv[j];
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_kv_shift(const KvView &kv0, int n_layer, int seq, int p0, int n, int end, const float2 *rope,
                            const Launch &l) {
    if (n < 1 || p0 < 0 || p0 + n > end || end > kv0.n_ctx || kv0.head_dim > 128 || kv0.head_dim % 2 ||
        seq < 0 || seq >= kv0.n_seq)
        return cudaErrorInvalidValue;
    if (p0 + n == end) return cudaSuccess;                  // nothing after the dropped rows
    const size_t so = (size_t)seq * kv0.seq_stride;
    if (kv0.k8)
        return launch_kernel(kv_shift_kernel<uint16_t>, dim3(n_layer * kv0.n_kv_head), dim3(SHIFT_THREADS), 0, l,
                             reinterpret_cast<uint16_t *>(kv0.k8 + so), reinterpret_cast<uint16_t *>(kv0.v8 + so),
                             kv0.n_ctx, kv0.head_dim, p0, n, end, rope);
    return launch_kernel(kv_shift_kernel<uint32_t>, dim3(n_layer * kv0.n_kv_head), dim3(SHIFT_THREADS), 0, l,
                         reinterpret_cast<uint32_t *>(kv0.k + so), reinterpret_cast<uint32_t *>(kv0.v + so),
                         kv0.n_ctx, kv0.head_dim, p0, n, end, rope);
}

}  // namespace llm
