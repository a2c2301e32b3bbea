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
// one CTA per SM takes equal contiguous ranges of units in tile-major order
// ("stream-K"), so every SM streams the same number of bytes.  In each CTA a
// producer warp keeps an 8-stage ring of units in flight with 2-D TMA loads
// (128 KB per SM, issued from the kernel's first instruction, since weights
// never depend on the preceding kernel), and four consumer warps multiply
// them from shared memory: each takes 16 rows, loads its mma.sync A fragments
// with one 128-bit read per row and chunk (the K index is permuted
// identically on the x side, which leaves the dot product unchanged), and
// runs two m16n8k16 MMAs per 32-wide chunk over all 8 token columns.  A tile
// whose units span several CTAs is finished by the CTA that arrives last at
// the tile's counter, summing the pieces in CTA order: deterministic, and
// nothing spins.  Every mbarrier wait is bounded (see tma.cuh).
#include "common.cuh"
#include "launch.cuh"
#include "tma.cuh"

namespace llm {

namespace {

constexpr int BM = 64;          // rows per tile
constexpr int KU = 128;         // k per unit: 4 chunks of 32
constexpr int U = KU / 32;
constexpr int XPAD = 32;        // fp16 elements of padding per x row in smem
constexpr int CWARPS = 4;       // consumer warps, 16 rows each
constexpr int THREADS = CWARPS * 32;            // consumer threads
constexpr int GTHREADS = THREADS + 32;          // + the producer warp
constexpr int STAGES = 8;
constexpr uint32_t STAGE_BYTES = BM * KU * 2;   // 16 KB

// consumer-only barrier (the producer warp runs its own loop)
__device__ __forceinline__ void csync() { named_sync(1, THREADS); }

// 4 chunks of 32 k of one unit for this lane: rows lo and lo+8, from the
// dense [64][128] stage in shared memory, against x from shared memory.
__device__ __forceinline__ void mma_unit(float (&acc)[4], const f16 *wlo, const f16 *whi, const f16 *xs_row,
                                         bool row_valid) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint4 lo = *reinterpret_cast<const uint4 *>(wlo + u * 32);
        const uint4 hi = *reinterpret_cast<const uint4 *>(whi + u * 32);
        uint4 b = make_uint4(0, 0, 0, 0);
        if (row_valid) b = *reinterpret_cast<const uint4 *>(xs_row + u * 32);
        const uint32_t a0[4] = {lo.x, hi.x, lo.y, hi.y};
        const uint32_t b0[2] = {b.x, b.y};
        mma_f16_16816(acc, a0, b0);
        const uint32_t a1[4] = {lo.z, hi.z, lo.w, hi.w};
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
            csync();
            if (a.ss_out && (tid & 63) == 0 && t < T) a.ss_out[tile * 8 + t] = s_part[half][0] + s_part[half][1];
            csync();
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
__global__ void __launch_bounds__(GTHREADS, 1)
gemv_kernel(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ float res[BM][9];
    __shared__ float s_r[8];
    __shared__ int s_row[8];
    __shared__ int s_last;
    __shared__ int s_abort;
    __shared__ __align__(8) uint64_t bars[2 * STAGES];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int T = a.T, K = a.K, upt = K / KU;
    const long long total = (long long)(a.N / BM) * upt;
    const int P = gridDim.x, c = blockIdx.x;
    const long long u0 = first_unit(c, total, P), u1 = first_unit(c + 1, total, P);
    if (u0 >= u1) return;
    const int n = (int)(u1 - u0);
    // x columns this CTA keeps: all of K, or just its units' k ranges in unit order
    const bool full_k = n >= upt;
    const int xcols = full_k ? K : n * KU;
    const int ldxs = xcols + XPAD;
    const uint32_t wbase = smem_u32(smem_raw);                       // STAGES x 16 KB
    f16 *wsm = reinterpret_cast<f16 *>(smem_raw);
    f16 *xs = reinterpret_cast<f16 *>(smem_raw + STAGES * STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    volatile int *abort = &s_abort;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), CWARPS);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == CWARPS) {
        // ---- producer: weights only, so no dependency wait
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < n; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES && !mbar_wait(empty(s), ((i / STAGES) & 1) ^ 1, abort, a.err)) break;
                const long long u = u0 + i, tile = u / upt;
                mbar_expect_tx(full(s), STAGE_BYTES);
                tma_load_2d(wbase + s * STAGE_BYTES, &tmW, full(s), (int)(u - tile * upt) * KU, (int)(tile * BM));
                issued = i + 1;
            }
            if (*abort) {
                // let every armed stage land before the CTA's shared memory goes away
                for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
                    for (uint32_t r = 0; r < WAIT_LIMIT && !mbar_try_wait(full(i % STAGES), (i / STAGES) & 1); ++r) {
                    }
            }
        }
        return;
    }

    pdl_wait();
    pdl_trigger();

    // ---- prologue: the needed columns of the T input rows, fp16 in smem
    const int nv = xcols / 8;
    if (PRO == PRO_NORM) {
        if (tid < T) s_row[tid] = a.row_map ? a.row_map[tid] : tid;
        csync();
        if (a.ss_part) {
            if (tid < T) {
                float sum = 0.f;
                const int np = K / 64;
                for (int p = 0; p < np; ++p) sum += a.ss_part[p * 8 + tid];
                s_r[tid] = 1.0f / sqrtf(sum / (float)K + a.eps);
            }
        } else {
            for (int t = warp; t < T; t += CWARPS) {
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
        csync();
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
    csync();

    const bool row_valid = g < T;
    const f16 *xrow = xs + (row_valid ? g : 0) * ldxs + 8 * t4;
    const int rlo = warp * 16 + g;
    const long long tile_first = u0 / upt;
    // After an abort every consumer warp still walks the same segments and
    // barriers (skipping the work), so no warp is left waiting at a barrier.
    int i = 0;
    while (i < n) {
        const long long tile = (u0 + i) / upt;
        const long long seg_begin = u0 + i, seg_end = min(u1, (tile + 1) * upt);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (; u0 + i < seg_end; ++i) {
            const int s = i % STAGES;
            if (!mbar_wait(full(s), (i / STAGES) & 1, abort, a.err)) continue;
            const f16 *stage = wsm + (size_t)s * (STAGE_BYTES / 2);
            const long long u = u0 + i;
            const int xp = full_k ? (int)(u - tile * upt) * KU : i * KU;
            mma_unit(acc, stage + rlo * KU + 8 * t4, stage + (rlo + 8) * KU + 8 * t4, xrow + xp, row_valid);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
        }
        res[rlo][2 * t4] = acc[0];
        res[rlo][2 * t4 + 1] = acc[1];
        res[rlo + 8][2 * t4] = acc[2];
        res[rlo + 8][2 * t4 + 1] = acc[3];
        csync();
        const bool whole = seg_begin == tile * upt && seg_end == (tile + 1) * upt;
        bool finish = whole;
        if (!whole) {
            // one piece of a tile shared with neighbouring CTAs: slot 0 for this
            // CTA's first tile, slot 1 for its last
            const int slot = tile == tile_first ? 0 : 1;
            float *mine = a.part + ((size_t)c * 2 + slot) * (BM * 8);
            for (int e = tid; e < BM * 8; e += THREADS) mine[e] = res[e >> 3][e & 7];
            __threadfence();
            csync();
            const int c_first = cta_of(tile * upt, total, P), c_last = cta_of((tile + 1) * upt - 1, total, P);
            if (tid == 0) s_last = atomicAdd(&a.counters[tile], 1u) == (unsigned)(c_last - c_first);
            csync();
            finish = s_last != 0;
            if (finish) {
                __threadfence();
                for (int e = tid; e < BM * 8; e += THREADS) {
                    float sum = 0.f;
                    for (int c0 = c_first; c0 <= c_last; c0 += 8) {
                        float v[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int cc = c0 + q;
                            v[q] = 0.f;
                            if (cc <= c_last) {
                                const int sl = (first_unit(cc, total, P) / upt) == tile ? 0 : 1;
                                v[q] = __ldcg(a.part + ((size_t)cc * 2 + sl) * (BM * 8) + e);
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q) sum += v[q];
                    }
                    res[e >> 3][e & 7] = sum;
                }
                if (tid == 0) a.counters[tile] = 0u;
                csync();
            }
        }
        if (finish) tile_epilogue<EPI>(a, res, (int)tile, tid, lane);
        csync();
    }
}

}  // namespace

size_t gemv_smem_bytes(int N, int K, int T, int P) {
    const long long total = (long long)(N / BM) * (K / KU);
    const long long maxu = (total + P - 1) / P;
    const long long cols = maxu >= K / KU ? K : maxu * KU;
    return (size_t)STAGES * STAGE_BYTES + (size_t)T * (cols + XPAD) * sizeof(f16);
}

int gemv_pick_ctas(int N, int K, int T, int num_sms) {
    // one CTA per SM (each keeps 128 KB of weights in flight)
    const long long total = (long long)(N / BM) * (K / KU);
    long long P = num_sms;
    if (P > total) P = total;
    return (int)P;
}

bool make_gemv_map(TmaMap *m, const f16 *ptr, int rows, int cols) {
    return make_plain_map(m, ptr, rows, cols, BM, KU);
}

size_t gemv_scratch_floats(int P) { return (size_t)P * 2 * BM * 8; }

#define GEMV_CASE(P, E)                                                                   \
    if (pro == P && epi == E)                                                             \
        return launch_kernel(gemv_kernel<P, E>, dim3(grid), dim3(GTHREADS), smem, l,      \
                             *reinterpret_cast<const CUtensorMap *>(&mw), a);

cudaError_t launch_gemv(int pro, int epi, const GemvArgs &a, const TmaMap &mw, const Launch &l) {
    if (a.T < 1 || a.T > 8 || a.N % BM || a.K % KU || a.ctas < 1 || (long long)a.ctas > (long long)(a.N / BM) * (a.K / KU))
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)a.ctas;
    const size_t smem = gemv_smem_bytes(a.N, a.K, a.T, a.ctas);
    if (smem > 220 * 1024) return cudaErrorInvalidValue;
    GEMV_CASE(PRO_BF16, EPI_STORE)
    GEMV_CASE(PRO_NORM, EPI_STORE)
    GEMV_CASE(PRO_NORM, EPI_QKV)
    GEMV_CASE(PRO_BF16, EPI_RESID)
    GEMV_CASE(PRO_NORM, EPI_SWIGLU)
    GEMV_CASE(PRO_BF16, EPI_SWIGLU)
    return cudaErrorInvalidValue;
}

cudaError_t init_gemv_attributes() {
    const size_t mx = 220 * 1024;
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
