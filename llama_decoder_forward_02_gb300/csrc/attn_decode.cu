// Decode attention with the cache split along the sequence (flash-decoding):
// for each decode row t and query head h, o = softmax(q K^T / sqrt(hd)) V over
// the cached positions c <= pos[t] of sequence seq[t] ("Inside the inference
// engine: model architectures and forward pass", sections "Detailed
// explanation: Llama's forward pass in Go" (GQA, ScaledDotProduct with the
// cache) and "KV Cache: memory for causal attention" (full causal mask);
// "LLama.cpp — how it works", "KV-cache and the Prefill / Decode stages": the
// new token's Q meets every cached K and V).
//
// Bound by HBM reads of K and V.  One CTA per (split, kv head, row) reads its
// span of keys once for all G = H/Hkv query heads of the group (the GQA
// sharing).  Scores use one key per lane (the key row is read whole from L2
// lines shared by the warp), the value pass one group of dims per lane (fully
// coalesced rows).  The softmax runs online in base 2 with q pre-scaled by
// log2(e)/sqrt(hd).  Each CTA writes (max, sum, unnormalised output) for its
// split; the CTA that arrives last at the (row, kv head) counter merges all
// splits in split order, so the result is deterministic and nothing spins.
#include <mutex>

#include "common.cuh"
#include "launch.cuh"
#include "../../include/llm.h"

namespace llm {

namespace {

constexpr int THREADS = 128;
constexpr int NW = THREADS / 32;

constexpr int KEYS_PER_PASS = NW * 32;   // one key per lane per warp
constexpr int MAX_SPLIT = 128;

// Keys per split: at least one full pass of the CTA, and no more splits than
// the sequence needs (later splits have nothing to do and exit at once).
__device__ __forceinline__ int split_chunk(int S, int n_split) {
    int chunk = (S + n_split - 1) / n_split;
    chunk = ((chunk + KEYS_PER_PASS - 1) / KEYS_PER_PASS) * KEYS_PER_PASS;
    return chunk < KEYS_PER_PASS ? KEYS_PER_PASS : chunk;
}

template <int HD, int G>
__global__ void __launch_bounds__(THREADS) attn_decode_kernel(const AttnDecodeArgs a) {
    constexpr int D = HD / 32;                 // dims per lane in the value pass
    constexpr int CH = HD / 8;                 // 16-byte chunks per key row
    __shared__ __align__(16) float q_s[G][HD];
    __shared__ float p_s[NW][G][32];
    __shared__ float w_m[NW][G], w_l[NW][G];
    __shared__ __align__(16) float w_o[NW][G][HD];
    __shared__ float f_s[G][MAX_SPLIT], l_s[G][MAX_SPLIT];
    __shared__ float inv_l[G];
    __shared__ int s_last;

    const int sp = blockIdx.x, j = blockIdx.y, t = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, n_split = a.n_split;

    pdl_wait();
    pdl_trigger();

    const int pos = a.pos[t], seq = a.seq[t];
    const bool ok = pos >= 0 && pos < a.kv.n_ctx && seq >= 0 && seq < a.kv.n_seq;
    if (!ok && tid == 0 && sp == 0 && j == 0) raise_error(a.err, ERRF_BAD_INDEX);
    const int S = ok ? pos + 1 : 0;
    const int chunk = split_chunk(S, n_split);
    const int n_eff = S > 0 ? (S + chunk - 1) / chunk : 1;   // splits that take part
    if (sp >= n_eff) return;
    const int kb = sp * chunk, ke = min(S, kb + chunk);

    const float qscale = 1.4426950408889634f / sqrtf((float)HD);
    for (int i = tid; i < G * HD; i += THREADS) {
        const int g = i / HD, d = i - g * HD;
        q_s[g][d] = a.q[(size_t)t * H * HD + (size_t)(j * G + g) * HD + d] * qscale;
    }
    __syncthreads();

    const size_t base = ok ? (size_t)seq * a.kv.seq_stride + (size_t)j * a.kv.n_ctx * HD : 0;
    const f16 *K = a.kv.k + base;
    const f16 *V = a.kv.v + base;

    float m[G], l[G], o[G][D];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) o[g][d] = 0.f;
    }

    for (int b = kb + warp * 32; b < ke; b += KEYS_PER_PASS) {
        const int key = b + lane;
        const bool valid = key < ke;
        // scores: this lane's key row, all chunks in flight before use
        uint4 kr[CH];
        const uint4 *kp = reinterpret_cast<const uint4 *>(K + (size_t)(valid ? key : b) * HD);
#pragma unroll
        for (int c = 0; c < CH; ++c) kr[c] = __ldg(kp + c);
        float s[G];
#pragma unroll
        for (int g = 0; g < G; ++g) s[g] = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const float k0 = h2lo(kr[c].x), k1 = h2hi(kr[c].x), k2 = h2lo(kr[c].y), k3 = h2hi(kr[c].y);
            const float k4 = h2lo(kr[c].z), k5 = h2hi(kr[c].z), k6 = h2lo(kr[c].w), k7 = h2hi(kr[c].w);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float4 qa = *reinterpret_cast<const float4 *>(&q_s[g][c * 8]);
                const float4 qb = *reinterpret_cast<const float4 *>(&q_s[g][c * 8 + 4]);
                s[g] += qa.x * k0 + qa.y * k1 + qa.z * k2 + qa.w * k3 +
                        qb.x * k4 + qb.y * k5 + qb.z * k6 + qb.w * k7;
            }
        }
        const int nk = min(32, ke - b);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float sv = valid ? s[g] : -INFINITY;
            const float mx = warp_max(sv);
            const float mn = fmaxf(m[g], mx);          // finite: key b is valid
            const float corr = exp2f(m[g] - mn);       // m = -inf -> 0
            const float p = valid ? exp2f(sv - mn) : 0.f;
            l[g] = l[g] * corr + warp_sum(p);
            m[g] = mn;
#pragma unroll
            for (int d = 0; d < D; ++d) o[g][d] *= corr;
            p_s[warp][g][lane] = p;
        }
        __syncwarp();
        // values: one group of D dims per lane, 8 keys of loads in flight
        for (int k0 = 0; k0 < nk; k0 += 8) {
            float v[8][D];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int kk = min(k0 + u, nk - 1);
                const f16 *vr = V + (size_t)(b + kk) * HD + lane * D;
                if (D == 4) {
                    const uint2 w = __ldg(reinterpret_cast<const uint2 *>(vr));
                    v[u][0] = h2lo(w.x); v[u][1 % D] = h2hi(w.x); v[u][2 % D] = h2lo(w.y); v[u][3 % D] = h2hi(w.y);
                } else if (D == 2) {
                    const uint32_t w = __ldg(reinterpret_cast<const unsigned int *>(vr));
                    v[u][0] = h2lo(w); v[u][1 % D] = h2hi(w);
                } else {
                    v[u][0] = hf(vr[0]);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k0 + u >= nk) break;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float p = p_s[warp][g][k0 + u];
#pragma unroll
                    for (int d = 0; d < D; ++d) o[g][d] += p * v[u][d];
                }
            }
        }
        __syncwarp();
    }

    // ---- combine the warps of this CTA
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (lane == 0) { w_m[warp][g] = m[g]; w_l[warp][g] = l[g]; }
#pragma unroll
        for (int d = 0; d < D; ++d) w_o[warp][g][lane * D + d] = o[g][d];
    }
    __syncthreads();
    const int rec = HD + 2;
    float *mypart = a.part + ((size_t)(t * H + j * G) * n_split + sp) * rec;
    for (int i = tid; i < G * HD; i += THREADS) {
        const int g = i / HD, d = i - g * HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, w_m[w][g]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float f = exp2f(w_m[w][g] - M);
                num += f * w_o[w][g][d];
                den += f * w_l[w][g];
            }
        }
        float *rp = mypart + (size_t)g * n_split * rec;
        rp[2 + d] = num;
        if (d == 0) { rp[0] = M; rp[1] = den; }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0)
        s_last = atomicAdd(&a.counters[t * a.kv.n_kv_head + j], 1u) == (unsigned)(n_eff - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of this (row, kv head): merge the splits in split order.
    // All (max, sum) pairs are fetched at once, then scale factors per (head,
    // split), then each dim's partials with independent loads.
    for (int i = tid; i < G * n_eff; i += THREADS) {
        const int g = i / n_eff, p = i - g * n_eff;
        const float *rp = a.part + ((size_t)(t * H + j * G + g) * n_split + p) * rec;
        f_s[g][p] = __ldcg(rp);
        l_s[g][p] = __ldcg(rp + 1);
    }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int p = 0; p < n_eff; ++p) M = fmaxf(M, f_s[tid][p]);
        float den = 0.f;
        for (int p = 0; p < n_eff; ++p) {
            const float mp = f_s[tid][p];
            const float f = mp == -INFINITY ? 0.f : exp2f(mp - M);
            f_s[tid][p] = f;
            den += f * l_s[tid][p];
        }
        inv_l[tid] = den > 0.f ? 1.f / den : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < G * HD; i += THREADS) {
        const int g = i / HD, d = i - g * HD;
        const float *rp = a.part + ((size_t)(t * H + j * G + g) * n_split) * rec + 2 + d;
        float num = 0.f;
        int p = 0;
        for (; p + 4 <= n_eff; p += 4) {
            const float v0 = __ldcg(rp + (size_t)p * rec), v1 = __ldcg(rp + (size_t)(p + 1) * rec);
            const float v2 = __ldcg(rp + (size_t)(p + 2) * rec), v3 = __ldcg(rp + (size_t)(p + 3) * rec);
            num += f_s[g][p] * v0;
            num += f_s[g][p + 1] * v1;
            num += f_s[g][p + 2] * v2;
            num += f_s[g][p + 3] * v3;
        }
        for (; p < n_eff; ++p) num += f_s[g][p] * __ldcg(rp + (size_t)p * rec);
        a.o[(size_t)t * H * HD + (size_t)(j * G + g) * HD + d] = f2h(num * inv_l[g]);
    }
    if (tid == 0) a.counters[t * a.kv.n_kv_head + j] = 0u;
}

}  // namespace

size_t attn_decode_scratch_floats(int T, int H, int hd, int n_split) {
    return (size_t)T * H * n_split * (hd + 2);
}

#define ATTN_DEC_CASE(HDV, GV)                                                              \
    if (a.kv.head_dim == HDV && G == GV)                                                    \
        return launch_kernel(attn_decode_kernel<HDV, GV>, grid, dim3(THREADS), 0, l, a);

cudaError_t launch_attn_decode(const AttnDecodeArgs &a, const Launch &l) {
    if (a.T < 1 || a.T > 8 || a.n_split < 1 || a.n_split > MAX_SPLIT || a.kv.n_kv_head < 1 || a.H % a.kv.n_kv_head)
        return cudaErrorInvalidValue;
    const int G = a.H / a.kv.n_kv_head;
    const dim3 grid(a.n_split, a.kv.n_kv_head, a.T);
    ATTN_DEC_CASE(32, 1) ATTN_DEC_CASE(32, 2) ATTN_DEC_CASE(32, 4) ATTN_DEC_CASE(32, 8)
    ATTN_DEC_CASE(64, 1) ATTN_DEC_CASE(64, 2) ATTN_DEC_CASE(64, 4) ATTN_DEC_CASE(64, 8)
    ATTN_DEC_CASE(128, 1) ATTN_DEC_CASE(128, 2) ATTN_DEC_CASE(128, 4) ATTN_DEC_CASE(128, 8)
    return cudaErrorInvalidValue;
}

}  // namespace llm

// ---------------------------------------------------------------------------
// Zero-allocation variant of the decode attention entry point.
//
// Some callers cannot call cudaMalloc at all: code that runs while a CUDA
// graph is being captured (an allocation would break the capture), host code
// under an allocator that owns all device memory and forbids outside
// allocations, or real-time loops that must never block in the driver's
// allocator.  For them the split partials and split counters live in one
// file-scope device array instead of caller- or library-allocated memory.
// Every GPU that loads this library holds that array (4 MiB + 2 KiB) until
// the process exits.
// ---------------------------------------------------------------------------
namespace llm {
namespace {

constexpr size_t NOALLOC_PART_FLOATS = (size_t)1 << 20;    // 4 MiB of split partials
constexpr size_t NOALLOC_COUNTERS = 512;                    // (row, kv head) counters
// partials first, then the counters (as 32-bit words)
static __device__ __align__(256) float g_noalloc_scratch[NOALLOC_PART_FLOATS + NOALLOC_COUNTERS];

std::mutex g_noalloc_mu;
void *g_noalloc_addr[256] = {nullptr};   // per device: the array's device address

}  // namespace

// Records the message llm_last_error(NULL) reports (defined with the C ABI).
void set_global_error(const char *msg);

}  // namespace llm

extern "C" int32_t llm_op_attn_decode_noalloc(const float *q, const void *k_cache, const void *v_cache,
                                              const int32_t *pos, const int32_t *seq, void *o, int32_t T,
                                              int32_t H, int32_t Hkv, int32_t hd, int32_t n_ctx,
                                              int32_t n_split, void *stream) {
    using namespace llm;
    if (!q || !k_cache || !v_cache || !pos || !seq || !o || T < 1 || T > 8 || Hkv < 1 || H % Hkv ||
        n_ctx < 1 || n_split < 1 || (hd != 32 && hd != 64 && hd != 128)) {
        set_global_error("llm_op_attn_decode_noalloc: invalid argument");
        return LLM_ERR_INVALID;
    }
    const size_t need = attn_decode_scratch_floats(T, H, hd, n_split);
    if (need > NOALLOC_PART_FLOATS || (size_t)T * Hkv > NOALLOC_COUNTERS) {
        set_global_error("llm_op_attn_decode_noalloc: T*H*n_split*(head_dim+2) exceeds the 1048576-float "
                         "static scratch (or T*n_head_kv exceeds 512); use llm_op_attn_decode");
        return LLM_ERR_INVALID;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) {
        set_global_error("llm_op_attn_decode_noalloc: no current device");
        return LLM_ERR_COMPUTE;
    }
    void *base = nullptr;
    {
        // once per device, with that device current: the host-side name of
        // the array is not a device address, so ask the runtime for it
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) {
                set_global_error("llm_op_attn_decode_noalloc: cudaGetSymbolAddress failed");
                return LLM_ERR_COMPUTE;
            }
            g_noalloc_addr[dev] = p;
        }
        base = g_noalloc_addr[dev];
    }
    float *part = static_cast<float *>(base);
    unsigned *counters = reinterpret_cast<unsigned *>(part + NOALLOC_PART_FLOATS);
    cudaStream_t st = (cudaStream_t)stream;
    // the counters must start at zero; the array keeps whatever the last call left
    cudaError_t e = cudaMemsetAsync(counters, 0, (size_t)T * Hkv * sizeof(unsigned), st);
    AttnDecodeArgs at;
    at.q = q;
    at.kv.k = (f16 *)k_cache; at.kv.v = (f16 *)v_cache;
    at.kv.seq_stride = (long long)Hkv * n_ctx * hd;
    at.kv.n_ctx = n_ctx; at.kv.n_seq = 1 << 30; at.kv.head_dim = hd; at.kv.n_kv_head = Hkv;
    at.pos = pos; at.seq = seq; at.o = (f16 *)o; at.T = T; at.H = H; at.n_split = n_split;
    at.part = part; at.counters = counters; at.err = nullptr;
    if (!e) e = launch_attn_decode(at, Launch{st, false, nullptr});
    if (e) {
        set_global_error("llm_op_attn_decode_noalloc: launch failed");
        return LLM_ERR_COMPUTE;
    }
    return LLM_OK;
}
