// Decode GEMV: y[t][n] = sum_k W[n][k] x[t][k] for 1..8 rows t, with the
// RMSNorm fused into the prologue and RoPE + KV append, SiLU*Up or the
// residual add fused into the epilogue ("Inside the inference engine: model
// architectures and forward pass", section "Detailed explanation: Llama's
// forward pass in Go": Q/K/V = Linear(RMSNorm(h)), RoPE(Q, K), h += Output(a),
// h += Down(SiLU(Gate x) * Up x); "LLama.cpp — how it works", "KV-cache and the
// Prefill / Decode stages": decode computes K, V for the new token and appends
// them to the cache).
//
// Decode is bound by HBM: every weight byte is read once per step.  The
// matrix is cut into units of 64 rows x 128 k (16 KB); a persistent grid of
// P CTAs (about four per SM, all resident) takes equal contiguous ranges of
// units in tile-major order ("stream-K"), so every SM streams the same
// number of bytes and none idles while others finish.  Each warp streams 16
// rows of a unit with 128-bit loads laid out directly as mma.sync A
// fragments (the K index is permuted identically on the x side, which leaves
// the dot product unchanged), so one warp-wide load pair feeds two m16n8k16
// MMAs over all 8 token columns; the next unit's loads are in flight while
// the current one is multiplied, and the first unit's are issued before the
// programmatic-dependent-launch wait, since weights never depend on the
// preceding kernel.  A tile whose units span several CTAs is finished by the
// CTA that arrives last at the tile's counter, summing the pieces in CTA
// order: deterministic, and nothing spins.
#include "common.cuh"
#include "launch.cuh"

namespace llm {

namespace {

constexpr int BM = 64;          // rows per tile
constexpr int THREADS = 128;    // 4 warps x 16 rows
constexpr int KU = 128;         // k per unit: 4 chunks of 32
constexpr int U = KU / 32;
constexpr int XPAD = 32;        // fp16 elements of padding per x row in smem
constexpr int CTAS_PER_SM = 4;

struct Frag { uint4 lo[U], hi[U]; };

__device__ __forceinline__ void load_frag(Frag &f, const f16 *wlo, const f16 *whi) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        f.lo[u] = ldg_stream(wlo + u * 32);
        f.hi[u] = ldg_stream(whi + u * 32);
    }
}

__device__ __forceinline__ void mma_frag(float (&acc)[4], const Frag &f, const f16 *xs_row, bool row_valid) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        uint4 b = make_uint4(0, 0, 0, 0);
        if (row_valid) b = *reinterpret_cast<const uint4 *>(xs_row + u * 32);
        const uint32_t a0[4] = {f.lo[u].x, f.hi[u].x, f.lo[u].y, f.hi[u].y};
        const uint32_t b0[2] = {b.x, b.y};
        mma_f16_16816(acc, a0, b0);
        const uint32_t a1[4] = {f.lo[u].z, f.hi[u].z, f.lo[u].w, f.hi[u].w};
        const uint32_t b1[2] = {b.z, b.w};
        mma_f16_16816(acc, a1, b1);
    }
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

// Units [u0(c), u0(c+1)) belong to CTA c; the CTA holding unit u.
__device__ __forceinline__ long long first_unit(long long c, long long total, int P) { return c * total / P; }
__device__ __forceinline__ int cta_of(long long u, long long total, int P) {
    return (int)(((u + 1) * P - 1) / total);
}

// The fused epilogue of one finished 64-row tile (sums in res[row][token]).
template <int EPI>
__device__ __forceinline__ void tile_epilogue(const GemvArgs &a, float (&res)[BM][9], int tile, int tid, int lane) {
    const int m0 = tile * BM, T = a.T;
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
                const int cc = n - a.n_q - (is_k ? 0 : a.n_kv);
                const int head = cc / hd, d = cc - head * hd;
                f16 *base = is_k ? a.kv.k : a.kv.v;
                const size_t off = (size_t)seq * a.kv.seq_stride + ((size_t)head * a.kv.n_ctx + pos) * hd + d;
                *reinterpret_cast<uint32_t *>(base + off) = pack_h2(x0, x1);
            }
        }
    } else if (EPI == EPI_SWIGLU) {
        for (int i = tid; i < (BM / 2) * T; i += THREADS) {
            const int t = i / (BM / 2), jj = i - t * (BM / 2);
            const int grp = jj / GU_GROUP, r = jj - grp * GU_GROUP;
            const float gate = res[grp * 2 * GU_GROUP + r][t];
            const float up = res[grp * 2 * GU_GROUP + GU_GROUP + r][t];
            const int j = (m0 / (2 * GU_GROUP) + grp) * GU_GROUP + r;
            a.u_out[(size_t)t * a.ldu + j] = f2h(silu(gate) * up);
        }
    }
}

template <int PRO, int EPI>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ float res[BM][9];
    __shared__ float s_r[8];
    __shared__ int s_row[8];
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int T = a.T, K = a.K, upt = K / KU;
    const long long total = (long long)(a.N / BM) * upt;
    const int P = gridDim.x, c = blockIdx.x;
    const long long u0 = first_unit(c, total, P), u1 = first_unit(c + 1, total, P);
    if (u0 >= u1) return;
    // x columns this CTA keeps: all of K, or just its units' k ranges in unit order
    const bool full_k = (u1 - u0) >= upt;
    const int xcols = full_k ? K : (int)(u1 - u0) * KU;
    const int ldxs = xcols + XPAD;
    f16 *xs = reinterpret_cast<f16 *>(smem_raw);

    auto wrow = [&](long long u) {
        const long long tile = u / upt;
        const int k = (int)(u - tile * upt) * KU;
        return a.W + (size_t)(tile * BM + warp * 16 + g) * K + k + 8 * t4;
    };

    Frag cur;
    {
        const f16 *w = wrow(u0);
        load_frag(cur, w, w + 8 * (size_t)K);
    }

    pdl_wait();
    pdl_trigger();

    // ---- prologue: the needed columns of the T input rows, fp16 in smem
    const int nv = xcols / 8;
    if (PRO == PRO_NORM) {
        if (tid < T) s_row[tid] = a.row_map ? a.row_map[tid] : tid;
        __syncthreads();
        if (a.ss_part) {
            if (tid < T) {
                float sum = 0.f;
                const int np = K / 64;
                for (int p = 0; p < np; ++p) sum += a.ss_part[p * 8 + tid];
                s_r[tid] = 1.0f / sqrtf(sum / (float)K + a.eps);
            }
        } else {
            for (int t = warp; t < T; t += THREADS / 32) {
                const float4 *hr = reinterpret_cast<const float4 *>(a.h + (size_t)s_row[t] * a.ldh);
                float sum = 0.f;
                for (int i = lane; i < K / 4; i += 32) {
                    const float4 v = hr[i];
                    sum += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                }
                sum = warp_sum(sum);
                if (lane == 0) s_r[t] = 1.0f / sqrtf(sum / (float)K + a.eps);
            }
        }
        __syncthreads();
    }
    for (int i = tid; i < T * nv; i += THREADS) {
        const int t = i / nv, col = (i - t * nv) * 8;
        const int k = full_k ? col : (int)((u0 + col / KU) % upt) * KU + (col % KU);
        uint4 o;
        if (PRO == PRO_NORM) {
            const float4 *hp = reinterpret_cast<const float4 *>(a.h + (size_t)s_row[t] * a.ldh + k);
            const float4 *gp = reinterpret_cast<const float4 *>(a.gain + k);
            const float4 h0 = hp[0], h1 = hp[1], g0 = gp[0], g1 = gp[1];
            const float r = s_r[t];
            o.x = pack_h2(h0.x * r * g0.x, h0.y * r * g0.y);
            o.y = pack_h2(h0.z * r * g0.z, h0.w * r * g0.w);
            o.z = pack_h2(h1.x * r * g1.x, h1.y * r * g1.y);
            o.w = pack_h2(h1.z * r * g1.z, h1.w * r * g1.w);
        } else {
            o = *reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.ldx + k);
        }
        *reinterpret_cast<uint4 *>(xs + t * ldxs + col) = o;
    }
    __syncthreads();

    const bool row_valid = g < T;
    const f16 *xrow = xs + (row_valid ? g : 0) * ldxs + 8 * t4;
    const long long tile_first = u0 / upt;
    long long u = u0;
    while (u < u1) {
        const long long tile = u / upt;
        const long long seg_begin = u, seg_end = min(u1, (tile + 1) * upt);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (; u < seg_end; ++u) {
            Frag nxt;
            const bool more = u + 1 < u1;
            if (more) {
                const f16 *w = wrow(u + 1);
                load_frag(nxt, w, w + 8 * (size_t)K);
            }
            const int xp = full_k ? (int)(u - tile * upt) * KU : (int)(u - u0) * KU;
            mma_frag(acc, cur, xrow + xp, row_valid);
            if (more) cur = nxt;
        }
        const int r0 = warp * 16 + g;
        res[r0][2 * t4] = acc[0];
        res[r0][2 * t4 + 1] = acc[1];
        res[r0 + 8][2 * t4] = acc[2];
        res[r0 + 8][2 * t4 + 1] = acc[3];
        __syncthreads();
        const bool whole = seg_begin == tile * upt && seg_end == (tile + 1) * upt;
        bool finish = whole;
        if (!whole) {
            // one piece of a tile shared with neighbouring CTAs: slot 0 for this
            // CTA's first tile, slot 1 for its last
            const int slot = tile == tile_first ? 0 : 1;
            float *mine = a.part + ((size_t)c * 2 + slot) * (BM * 8);
            for (int i = tid; i < BM * 8; i += THREADS) mine[i] = res[i >> 3][i & 7];
            __threadfence();
            __syncthreads();
            const int c_first = cta_of(tile * upt, total, P), c_last = cta_of((tile + 1) * upt - 1, total, P);
            if (tid == 0)
                s_last = atomicAdd(&a.counters[tile], 1u) == (unsigned)(c_last - c_first);
            __syncthreads();
            finish = s_last != 0;
            if (finish) {
                __threadfence();
                for (int i = tid; i < BM * 8; i += THREADS) {
                    float sum = 0.f;
                    for (int cc = c_first; cc <= c_last; ++cc) {
                        const int sl = (first_unit(cc, total, P) / upt) == tile ? 0 : 1;
                        sum += __ldcg(a.part + ((size_t)cc * 2 + sl) * (BM * 8) + i);
                    }
                    res[i >> 3][i & 7] = sum;
                }
                if (tid == 0) a.counters[tile] = 0u;
                __syncthreads();
            }
        }
        if (finish) tile_epilogue<EPI>(a, res, (int)tile, tid, lane);
        __syncthreads();
    }
}

}  // namespace

size_t gemv_smem_bytes(int N, int K, int T, int P) {
    const long long total = (long long)(N / BM) * (K / KU);
    const long long maxu = (total + P - 1) / P;
    const long long cols = maxu >= K / KU ? K : maxu * KU;
    return (size_t)T * (cols + XPAD) * sizeof(f16);
}

int gemv_pick_ctas(int N, int K, int T, int num_sms) {
    // about four resident CTAs per SM, fewer when the x slice is large
    const long long total = (long long)(N / BM) * (K / KU);
    int per_sm = CTAS_PER_SM;
    while (per_sm > 1 && gemv_smem_bytes(N, K, T, per_sm * num_sms) + 3 * 1024 > (size_t)(227 * 1024 / per_sm)) --per_sm;
    long long P = (long long)per_sm * num_sms;
    if (P > total) P = total;
    return (int)P;
}

size_t gemv_scratch_floats(int P) { return (size_t)P * 2 * BM * 8; }

#define GEMV_CASE(P, E)                                                                   \
    if (pro == P && epi == E)                                                             \
        return launch_kernel(gemv_kernel<P, E>, dim3(grid), dim3(THREADS), smem, l, a);

cudaError_t launch_gemv(int pro, int epi, const GemvArgs &a, const Launch &l) {
    if (a.T < 1 || a.T > 8 || a.N % BM || a.K % KU || a.ctas < 1 || (long long)a.ctas > (long long)(a.N / BM) * (a.K / KU))
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)a.ctas;
    const size_t smem = gemv_smem_bytes(a.N, a.K, a.T, a.ctas);
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
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
