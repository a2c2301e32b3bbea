// Decode GEMV: y[t][n] = sum_k W[n][k] x[t][k] for 1..8 rows t, with the
// RMSNorm fused into the prologue and RoPE + KV append, SiLU*Up or the
// residual add fused into the epilogue ("Inside the inference engine: model
// architectures and forward pass", section "Detailed explanation: Llama's
// forward pass in Go": Q/K/V = Linear(RMSNorm(h)), RoPE(Q, K), h += Output(a),
// h += Down(SiLU(Gate x) * Up x); "LLama.cpp — how it works", "KV-cache and the
// Prefill / Decode stages": decode computes K, V for the new token and appends
// them to the cache).
//
// Decode is bound by HBM: every weight byte is read once per step.  A CTA
// owns 64 output rows and one K slice; each warp streams 16 rows with 128-bit
// loads laid out directly as mma.sync A fragments (the K index is permuted
// identically on the x side, which leaves the dot product unchanged), so one
// warp-wide load pair feeds two m16n8k16 MMAs over all 8 token columns.
// Loads are double-buffered in registers and the first ones are issued before
// the programmatic-dependent-launch wait, since weights never depend on the
// preceding kernel.  K slices of the same tile are combined by the CTA that
// arrives last at a per-tile counter (no spinning), in split order, so the
// result is deterministic.
#include "common.cuh"
#include "launch.cuh"

#include <algorithm>
#include <map>
#include <mutex>

namespace llm {

namespace {

constexpr int BM = 64;          // rows per CTA
constexpr int THREADS = 128;    // 4 warps x 16 rows
constexpr int U = 8;            // 32-wide K chunks per register buffer
constexpr int XPAD = 32;        // f16 elements of padding per x row in smem

struct Frag { uint4 lo[U], hi[U]; };

// Chunks past the slice's nchunk (a slice is a multiple of 4 chunks, U may be
// larger) are zero, not loaded: they add nothing to the dot product.
__device__ __forceinline__ void load_frag(Frag &f, const f16 *wlo, const f16 *whi, int chunk, int nchunk) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (chunk + u < nchunk) {
            f.lo[u] = ldg_stream(wlo + (chunk + u) * 32);
            f.hi[u] = ldg_stream(whi + (chunk + u) * 32);
        } else {
            f.lo[u] = f.hi[u] = make_uint4(0, 0, 0, 0);
        }
    }
}

__device__ __forceinline__ void mma_frag(float (&acc)[4], const Frag &f, const f16 *xs_row,
                                         int chunk, int nchunk, bool row_valid) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (chunk + u >= nchunk) break;
        uint4 b = make_uint4(0, 0, 0, 0);
        if (row_valid) b = *reinterpret_cast<const uint4 *>(xs_row + (chunk + u) * 32);
        const uint32_t a0[4] = {f.lo[u].x, f.hi[u].x, f.lo[u].y, f.hi[u].y};
        const uint32_t b0[2] = {b.x, b.y};
        mma_f16_16816(acc, a0, b0);
        const uint32_t a1[4] = {f.lo[u].z, f.hi[u].z, f.lo[u].w, f.hi[u].w};
        const uint32_t b1[2] = {b.z, b.w};
        mma_f16_16816(acc, a1, b1);
    }
}

template <int PRO, int EPI>
__global__ void __launch_bounds__(THREADS) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ float res[BM][9];
    __shared__ float s_r[8];
    __shared__ int s_row[8];
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int tile = blockIdx.x / a.ksplit, split = blockIdx.x % a.ksplit;
    const int Ks = a.K / a.ksplit, k0 = split * Ks;
    const int m0 = tile * BM;
    const int T = a.T;
    const int ldxs = Ks + XPAD;
    f16 *xs = reinterpret_cast<f16 *>(smem_raw);

    const f16 *wlo = a.W + (size_t)(m0 + warp * 16 + g) * a.K + k0 + 8 * t4;
    const f16 *whi = wlo + 8 * (size_t)a.K;
    const int nchunk = Ks / 32;

    Frag f0, f1;
    load_frag(f0, wlo, whi, 0, nchunk);

    pdl_wait();
    pdl_trigger();

    // ---- prologue: this CTA's K slice of the T input rows, as f16 in smem
    if (PRO == PRO_NORM) {
        if (tid < T) s_row[tid] = a.row_map ? a.row_map[tid] : tid;
        __syncthreads();
        if (a.ss_part) {
            // 16 threads per row t sum the per-64-row partial sums of squares
            // (independent loads, then a shuffle tree)
            const int t = tid >> 4, sub = tid & 15;
            const int np = a.K / 64;
            float s = 0.f;
            if (t < T)
                for (int p = sub; p < np; p += 16) s += a.ss_part[p * 8 + t];
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (t < T && sub == 0) s_r[t] = 1.0f / sqrtf(s / (float)a.K + a.eps);
        } else {
            for (int t = warp; t < T; t += THREADS / 32) {
                const float4 *hr = reinterpret_cast<const float4 *>(a.h + (size_t)s_row[t] * a.ldh);
                float s = 0.f;
                for (int i = lane; i < a.K / 4; i += 32) {
                    float4 v = hr[i];
                    s += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                }
                s = warp_sum(s);
                if (lane == 0) s_r[t] = 1.0f / sqrtf(s / (float)a.K + a.eps);
            }
        }
        __syncthreads();
        const int nv = Ks / 8;
        for (int i = tid; i < T * nv; i += THREADS) {
            const int t = i / nv, kv = i - t * nv, k = k0 + kv * 8;
            const float4 *hp = reinterpret_cast<const float4 *>(a.h + (size_t)s_row[t] * a.ldh + k);
            const float4 *gp = reinterpret_cast<const float4 *>(a.gain + k);
            const float4 h0 = hp[0], h1 = hp[1], g0 = gp[0], g1 = gp[1];
            const float r = s_r[t];
            uint4 o;
            const float xv[8] = {h0.x * r * g0.x, h0.y * r * g0.y, h0.z * r * g0.z, h0.w * r * g0.w,
                                 h1.x * r * g1.x, h1.y * r * g1.y, h1.z * r * g1.z, h1.w * r * g1.w};
            bool bad = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) bad |= f16_bad(xv[j]);
            if (bad) raise_error(a.err, ERRF_F16_RANGE);
            o.x = pack_h2(xv[0], xv[1]);
            o.y = pack_h2(xv[2], xv[3]);
            o.z = pack_h2(xv[4], xv[5]);
            o.w = pack_h2(xv[6], xv[7]);
            *reinterpret_cast<uint4 *>(xs + t * ldxs + kv * 8) = o;
        }
    } else {
        const int nv = Ks / 8;
        for (int i = tid; i < T * nv; i += THREADS) {
            const int t = i / nv, kv = i - t * nv;
            *reinterpret_cast<uint4 *>(xs + t * ldxs + kv * 8) =
                *reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.ldx + k0 + kv * 8);
        }
    }
    __syncthreads();

    // ---- main loop: double-buffered register fragments
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const bool row_valid = g < T;
    const f16 *xrow = xs + (row_valid ? g : 0) * ldxs + 8 * t4;
    for (int c = 0; c < nchunk; c += 2 * U) {
        if (c + U < nchunk) load_frag(f1, wlo, whi, c + U, nchunk);
        mma_frag(acc, f0, xrow, c, nchunk, row_valid);
        if (c + U >= nchunk) break;
        if (c + 2 * U < nchunk) load_frag(f0, wlo, whi, c + 2 * U, nchunk);
        mma_frag(acc, f1, xrow, c + U, nchunk, row_valid);
    }

    // ---- gather this CTA's 64 x 8 tile of partial sums in smem
    const int r0 = warp * 16 + g;
    res[r0][2 * t4] = acc[0];
    res[r0][2 * t4 + 1] = acc[1];
    res[r0 + 8][2 * t4] = acc[2];
    res[r0 + 8][2 * t4 + 1] = acc[3];
    __syncthreads();

    if (a.ksplit > 1) {
        // partials of the T live columns only; the CTA that arrives last at
        // the tile's counter sums them in split order, every split's value in
        // flight at once
        float *mine = a.part + ((size_t)split * a.N + m0) * 8;
        for (int i = tid; i < BM * T; i += THREADS) {
            const int r = i / T, t = i - r * T;
            mine[r * 8 + t] = res[r][t];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = (atomicAdd(&a.counters[tile], 1u) == (unsigned)(a.ksplit - 1));
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        const float *pb = a.part + (size_t)m0 * 8;
        const size_t pstride = (size_t)a.N * 8;
        for (int i = tid; i < BM * T; i += THREADS) {
            const int r = i / T, t = i - r * T;
            const float *src = pb + r * 8 + t;
            float s = 0.f;
            for (int p0 = 0; p0 < a.ksplit; p0 += 16) {
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    v[u] = (p0 + u < a.ksplit) ? __ldcg(src + (size_t)(p0 + u) * pstride) : 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) s += v[u];
            }
            res[r][t] = s;
        }
        if (tid == 0) a.counters[tile] = 0u;
        __syncthreads();
    }

    // ---- epilogues
    if (EPI == EPI_STORE) {
        for (int i = tid; i < BM * T; i += THREADS) {
            const int t = i / BM, r = i - t * BM;
            a.out[(size_t)t * a.ldo + m0 + r] = res[r][t];
        }
    } else if (EPI == EPI_RESID) {
        // threads 0..63 take even tokens, 64..127 odd ones; one row each
        const int r = tid & 63, half = tid >> 6;
        __shared__ float s_part[2][2];
        for (int tb = 0; tb < T; tb += 2) {
            const int t = tb + half;
            float sq = 0.f;
            if (t < T) {
                float *hp = a.hres + (size_t)t * a.ldh_res + m0 + r;
                const float v = *hp + res[r][t];
                *hp = v;
                sq = v * v;
            }
            sq = warp_sum(sq);
            if (lane == 0) s_part[half][(tid >> 5) & 1] = sq;
            __syncthreads();
            if (a.ss_out && (tid & 63) == 0 && t < T) a.ss_out[tile * 8 + t] = s_part[half][0] + s_part[half][1];
            __syncthreads();
        }
    } else if (EPI == EPI_QKV) {
        const int hd = a.kv.head_dim, half_hd = hd / 2;
        for (int i = tid; i < (BM / 2) * T; i += THREADS) {
            const int t = i / (BM / 2), p = i - t * (BM / 2);
            const int n = m0 + 2 * p;
            const int pos = a.pos[t], seq = a.seq[t];
            if (pos < 0 || pos >= a.kv.n_ctx || seq < 0 || seq >= a.kv.n_seq) {
                raise_error(a.err, ERRF_BAD_INDEX);
                continue;
            }
            float x0 = res[2 * p][t], x1 = res[2 * p + 1][t];
            if (n < a.n_q + a.n_kv) {   // rotate q and k rows
                const int d = (n < a.n_q ? n : n - a.n_q) % hd;
                const float2 cs = a.rope[(size_t)pos * half_hd + d / 2];
                const float y0 = x0 * cs.x - x1 * cs.y, y1 = x0 * cs.y + x1 * cs.x;
                x0 = y0;
                x1 = y1;
            }
            if (n < a.n_q) {
                *reinterpret_cast<float2 *>(a.q_out + (size_t)t * a.n_q + n) = make_float2(x0, x1);
            } else {
                const bool is_k = n < a.n_q + a.n_kv;
                const int c = n - a.n_q - (is_k ? 0 : a.n_kv);
                const int head = c / hd, d = c - head * hd;
                const size_t off = (size_t)seq * a.kv.seq_stride + ((size_t)head * a.kv.n_ctx + pos) * hd + d;
                if (a.kv.k8)
                    *reinterpret_cast<uint16_t *>((is_k ? a.kv.k8 : a.kv.v8) + off) = pack_e4m3x2(x0, x1);
                else {
                    if (f16_bad(x0) || f16_bad(x1)) raise_error(a.err, ERRF_F16_RANGE);
                    *reinterpret_cast<uint32_t *>((is_k ? a.kv.k : a.kv.v) + off) = pack_h2(x0, x1);
                }
            }
        }
    } else if (EPI == EPI_SWIGLU) {
        for (int i = tid; i < (BM / 2) * T; i += THREADS) {
            const int t = i / (BM / 2), jj = i - t * (BM / 2);
            const int grp = jj / GU_GROUP, r = jj - grp * GU_GROUP;
            const float gate = res[grp * 2 * GU_GROUP + r][t];
            const float up = res[grp * 2 * GU_GROUP + GU_GROUP + r][t];
            const int j = (m0 / (2 * GU_GROUP) + grp) * GU_GROUP + r;
            const float u = silu(gate) * up;
            if (f16_bad(u)) raise_error(a.err, ERRF_F16_RANGE);
            a.u_out[(size_t)t * a.ldu + j] = f2h(u);
        }
    }
}

template <int PRO, int EPI>
const void *kernel_ptr() { return reinterpret_cast<const void *>(&gemv_kernel<PRO, EPI>); }

}  // namespace

size_t gemv_smem_bytes(int K, int ksplit, int T) {
    return (size_t)T * (K / ksplit + XPAD) * sizeof(f16);
}

namespace {

// CTAs of one GEMV launch that fit on an SM together, for a given dynamic
// shared-memory size (the smallest over the kernel variants; memoised).
int gemv_ctas_per_sm(size_t smem) {
    static std::mutex mu;
    static std::map<size_t, int> memo;
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(smem);
    if (it != memo.end()) return it->second;
    const void *ks[] = {kernel_ptr<PRO_BF16, EPI_STORE>(), kernel_ptr<PRO_NORM, EPI_STORE>(),
                        kernel_ptr<PRO_NORM, EPI_QKV>(), kernel_ptr<PRO_BF16, EPI_RESID>(),
                        kernel_ptr<PRO_NORM, EPI_SWIGLU>(), kernel_ptr<PRO_BF16, EPI_SWIGLU>()};
    int best = 1 << 30;
    for (const void *k : ks) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, THREADS, smem) != cudaSuccess) {
            cudaGetLastError();
            n = 4;
        }
        best = std::min(best, std::max(n, 1));
    }
    memo[smem] = best;
    return best;
}

}  // namespace

int gemv_pick_split(int N, int K, int T, int num_sms) {
    // Largest split whose grid fits in one wave of resident CTAs, with K
    // slices that are multiples of 128 and at least 256 wide: a CTA's time is
    // set by its memory round trips, so a second, partly filled wave costs
    // almost as much as the first.  Then grow the split until the x slice
    // fits comfortably in shared memory.
    const long long tiles = N / BM;
    int best = 1;
    for (int s = 2; s <= 64; ++s) {
        if (K % (s * 128)) continue;
        if (K / s < 256) break;
        const size_t smem = gemv_smem_bytes(K, s, T);
        if (smem > 100 * 1024) continue;
        if (tiles * s > (long long)gemv_ctas_per_sm(smem) * num_sms) continue;
        best = s;
    }
    // Many rows (no split fits one wave) and x slices of >= 32 KB: two
    // halves of K double the CTAs an SM holds, which hides more of their
    // memory latency than the extra partials cost (8-row steps of the 8B
    // shape: gate/up 448 and LM head 2004 row tiles, 5.79 -> 4.83 ms a step)
    if (best == 1 && T >= 4 && K % 256 == 0 && K / 2 >= 2048) best = 2;
    while (gemv_smem_bytes(K, best, T) > 100 * 1024) {
        int nxt = best + 1;
        while (nxt <= K / 128 && K % (nxt * 128)) ++nxt;
        if (nxt > K / 128) break;
        best = nxt;
    }
    return best;
}

#define GEMV_CASE(P, E)                                                                   \
    if (pro == P && epi == E)                                                             \
        return launch_kernel(gemv_kernel<P, E>, dim3(grid), dim3(THREADS), smem, l, a);

cudaError_t launch_gemv(int pro, int epi, const GemvArgs &a, const Launch &l) {
    if (a.T < 1 || a.T > 8 || a.N % BM || a.ksplit < 1 || a.K % (128 * a.ksplit))
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)(a.N / BM) * a.ksplit;
    const size_t smem = gemv_smem_bytes(a.K, a.ksplit, a.T);
    GEMV_CASE(PRO_BF16, EPI_STORE)
    GEMV_CASE(PRO_NORM, EPI_STORE)
    GEMV_CASE(PRO_NORM, EPI_QKV)
    GEMV_CASE(PRO_BF16, EPI_RESID)
    GEMV_CASE(PRO_NORM, EPI_SWIGLU)
    GEMV_CASE(PRO_BF16, EPI_SWIGLU)
    return cudaErrorInvalidValue;
}

cudaError_t init_gemv_attributes() {
    const size_t mx = 200 * 1024;
    cudaError_t e = cudaSuccess;
    e = allow_smem(gemv_kernel<PRO_BF16, EPI_STORE>, mx); if (e) return e;
    e = allow_smem(gemv_kernel<PRO_NORM, EPI_STORE>, mx); if (e) return e;
    e = allow_smem(gemv_kernel<PRO_NORM, EPI_QKV>, mx); if (e) return e;
    e = allow_smem(gemv_kernel<PRO_BF16, EPI_RESID>, mx); if (e) return e;
    e = allow_smem(gemv_kernel<PRO_NORM, EPI_SWIGLU>, mx); if (e) return e;
    e = allow_smem(gemv_kernel<PRO_BF16, EPI_SWIGLU>, mx);
    return e;
}

}  // namespace llm
