// The decode-attention work item (one split of one kv head for one decode
// row), shared by the standalone decode-attention kernel and the persistent
// decode kernel.  See attn_decode.cu for the method.
#pragma once
#include "attn_tile.cuh"
#include "common.cuh"
#include "kernels.h"

namespace llm {
namespace attn_dec {

constexpr int THREADS = 128;
constexpr int NW = THREADS / 32;
constexpr int TK = 64;                   // keys per K/V tile; each warp takes 16
constexpr int MAX_SPLIT = ATTN_DECODE_MAX_SPLIT;

// Keys per split: whole tiles, and no more splits than the sequence needs
// (later splits have nothing to do and exit at once).
__device__ __forceinline__ int split_chunk(int S, int n_split) {
    int chunk = (S + n_split - 1) / n_split;
    chunk = ((chunk + TK - 1) / TK) * TK;
    return chunk < TK ? TK : chunk;
}

template <int HD>
constexpr size_t decode_smem_bytes() {
    return (size_t)(4 * TK + 16) * HD * sizeof(f16) + (size_t)NW * 8 * (HD + 2) * sizeof(float);
}

// Dependency hook of a work item that may start before the kernel producing
// q and the newest K/V rows has finished: Dep::wait() returns once that
// kernel's writes are visible.
struct NoDep {
    __device__ static __forceinline__ void wait() {}
};

// One (split sp, kv head j, row t) work item, run by THREADS threads
// (tid 0..THREADS-1) that synchronize with CtaSync::sync(); smem_raw holds
// decode_smem_bytes<HD>() bytes.  The cached keys below pos[t] - (T - 1) were
// written before the preceding kernel started (the rows of one ubatch that
// share a sequence have consecutive positions), so their K/V tiles are
// requested before Dep::wait(); q and the newest rows after it.
template <int HD, int G, class CtaSync, class Dep = NoDep, bool F8 = false>
__device__ __forceinline__ void attn_decode_unit(const AttnDecodeArgs &a, int sp, int j, int t, int tid,
                                                 uint8_t *smem_raw) {
    static_assert(G <= 8, "the query heads of a group fill the first 8 rows of an m16 tile");
    constexpr int REC = HD + 2;
    f16 *Ks = reinterpret_cast<f16 *>(smem_raw);        // [2][TK][HD]
    f16 *Vs = Ks + 2 * TK * HD;                         // [2][TK][HD]
    f16 *Qs = Vs + 2 * TK * HD;                         // [16][HD]
    float *wst = reinterpret_cast<float *>(Qs + 16 * HD);   // [NW][G][REC]: m, l, o
    __shared__ int s_last;

    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int H = a.H, n_split = a.n_split;

    const int pos = a.pos[t], seq = a.seq[t];
    const bool ok = pos >= 0 && pos < a.kv.n_ctx && seq >= 0 && seq < a.kv.n_seq;
    if (!ok && tid == 0 && sp == 0 && j == 0) raise_error(a.err, ERRF_BAD_INDEX);
    // visible keys [lo, pos]: all earlier positions, or the last `window` ones
    const int lo = (ok && a.window > 0 && pos + 1 > a.window) ? pos + 1 - a.window : 0;
    const int S = ok ? pos + 1 - lo : 0;
    const int chunk = split_chunk(S, n_split);
    const int n_eff = S > 0 ? (S + chunk - 1) / chunk : 1;   // splits that take part
    if (sp >= n_eff) return;
    const int kb = lo + sp * chunk, ke = min(lo + S, kb + chunk);
    const int n_t = ke > kb ? (ke - kb + TK - 1) / TK : 0;

    const size_t base = ok ? (size_t)seq * a.kv.seq_stride + (size_t)j * a.kv.n_ctx * HD : 0;
    const f16 *Kg = a.kv.k + base;
    const f16 *Vg = a.kv.v + base;
    // FP8 E4M3 cache: rows are staged as bytes and widened to fp16 per tile
    constexpr bool f8 = F8;                 // FP8 E4M3 cache (the caller picks the instantiation)
    const uint8_t *Kg8 = f8 ? a.kv.k8 + base : nullptr;
    const uint8_t *Vg8 = f8 ? a.kv.v8 + base : nullptr;
    auto span = [&](f16 *dK, f16 *dV, int row0, int r_lo, int r_hi, int r_zero) {
        if (f8) {
            load_rows_span8<HD, TK, THREADS>(dK, Kg8 + (size_t)row0 * HD, r_lo, r_hi, r_zero, tid);
            load_rows_span8<HD, TK, THREADS>(dV, Vg8 + (size_t)row0 * HD, r_lo, r_hi, r_zero, tid);
        } else {
            load_rows_span<HD, TK, THREADS>(dK, Kg + (size_t)row0 * HD, r_lo, r_hi, r_zero, tid);
            load_rows_span<HD, TK, THREADS>(dV, Vg + (size_t)row0 * HD, r_lo, r_hi, r_zero, tid);
        }
    };

    // first two tiles in flight before anything else: the rows that are
    // already final before the dependency wait, the newest ones after it
    const int pre_end = min(ke, max(kb, pos - a.T + 1));
    const int v0 = ke - kb, v1 = ke - kb - TK;               // valid rows of tiles 0 and 1
    const int p0 = pre_end - kb, p1 = pre_end - kb - TK;     // of which final before the wait
    if (n_t > 0) span(Ks, Vs, kb, 0, p0, v0);
    if (n_t > 1) span(Ks + TK * HD, Vs + TK * HD, kb + TK, 0, p1, v1);
    cp_async_commit();
    Dep::wait();
    if (n_t > 0 && p0 < v0 && p0 < TK) span(Ks, Vs, kb, max(p0, 0), v0, TK);
    if (n_t > 1 && p1 < v1) span(Ks + TK * HD, Vs + TK * HD, kb + TK, max(p1, 0), v1, TK);
    cp_async_commit();

    // the group's query heads as rows 0..G-1 of a 16 x HD tile (fp16, scaled)
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);
    for (int i = tid; i < 16 * HD / 2; i += THREADS) {
        const int r = i / (HD / 2), d = (i - r * (HD / 2)) * 2;
        float x0 = 0.f, x1 = 0.f;
        if (r < G) {
            const float *qp = a.q + (size_t)t * H * HD + (size_t)(j * G + r) * HD + d;
            x0 = __ldcg(qp) * qscale;        // through L2: q is rewritten between uses
            x1 = __ldcg(qp + 1) * qscale;
        }
        *reinterpret_cast<uint32_t *>(Qs + Swz<HD>::off(r, d / 8) + (d & 7)) = pack_h2(x0, x1);
    }
    CtaSync::sync();
    uint32_t qf[HD / 16][4];
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = kk * 2 + (lane >> 4);
        ldmatrix_x4(qf[kk], smem_u32(Qs + Swz<HD>::off(r, c)));
    }

    float o[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow = -INFINITY, lrow = 0.f;      // row g (rows g+8 are padding)

    cp_async_wait<0>();                 // tiles 0 and 1
    for (int it = 0; it < n_t; ++it) {
        cp_async_wait<1>();                 // tile it (tile it + 1 may still be in flight)
        CtaSync::sync();
        if (f8) {                           // widen the staged fp8 rows of tile it
            convert_tile8<HD, TK, THREADS>(Ks + (it & 1) * TK * HD, tid);
            convert_tile8<HD, TK, THREADS>(Vs + (it & 1) * TK * HD, tid);
        }
        const f16 *Kt = Ks + (it & 1) * TK * HD;
        const f16 *Vt = Vs + (it & 1) * TK * HD;
        const int key0 = kb + it * TK + warp * 16;      // this warp's 16 keys

        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            uint32_t kf[4];
            const int r = warp * 16 + (lane & 7) + (lane >> 4) * 8;
            const int c = kk * 2 + ((lane >> 3) & 1);
            ldmatrix_x4(kf, smem_u32(Kt + Swz<HD>::off(r, c)));
            const uint32_t b0[2] = {kf[0], kf[1]}, b1[2] = {kf[2], kf[3]};
            mma_f16_16816(sc[0], qf[kk], b0);
            mma_f16_16816(sc[1], qf[kk], b1);
        }
        // keys past the span are masked; online softmax on row g
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + nt * 8 + 2 * t4 + (e & 1);
                if (key >= ke) sc[nt][e] = -INFINITY;
                if (e < 2) mx = fmaxf(mx, sc[nt][e]);
            }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(mrow, mx);
        const float corr = (mn == -INFINITY) ? 1.f : exp2f(mrow - mn);
        mrow = mn;
        float rs = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p = (e < 2 && mn != -INFINITY) ? exp2f(sc[nt][e] - mn) : 0.f;
                sc[nt][e] = p;
                rs += p;
            }
        rs += __shfl_xor_sync(0xffffffffu, rs, 1);
        rs += __shfl_xor_sync(0xffffffffu, rs, 2);
        lrow = lrow * corr + rs;
#pragma unroll
        for (int dt = 0; dt < HD / 8; ++dt) { o[dt][0] *= corr; o[dt][1] *= corr; }
        const uint32_t pa[4] = {pack_h2(sc[0][0], sc[0][1]), pack_h2(sc[0][2], sc[0][3]),
                                pack_h2(sc[1][0], sc[1][1]), pack_h2(sc[1][2], sc[1][3])};
#pragma unroll
        for (int dp = 0; dp < HD / 16; ++dp) {
            uint32_t vf[4];
            const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int c = dp * 2 + (lane >> 4);
            ldmatrix_x4_trans(vf, smem_u32(Vt + Swz<HD>::off(r, c)));
            const uint32_t b0[2] = {vf[0], vf[1]}, b1[2] = {vf[2], vf[3]};
            mma_f16_16816(o[2 * dp], pa, b0);
            mma_f16_16816(o[2 * dp + 1], pa, b1);
        }
        CtaSync::sync();                                  // every warp is done with this buffer
        if (it + 2 < n_t) {
            const int nb = kb + (it + 2) * TK;
            span(Ks + (it & 1) * TK * HD, Vs + (it & 1) * TK * HD, nb, 0, ke - nb, ke - nb);
        }
        cp_async_commit();
    }
    cp_async_wait<0>();

    // ---- combine the warps: row g < G of each warp (rows live in lanes 4g..4g+3)
    if (g < G) {
        float *ws = wst + ((size_t)warp * G + g) * REC;
        if (t4 == 0) { ws[0] = mrow; ws[1] = lrow; }
#pragma unroll
        for (int dt = 0; dt < HD / 8; ++dt) {
            ws[2 + dt * 8 + 2 * t4] = o[dt][0];
            ws[2 + dt * 8 + 2 * t4 + 1] = o[dt][1];
        }
    }
    CtaSync::sync();
    float *mypart = a.part + ((size_t)(t * H + j * G) * n_split + sp) * REC;
    for (int i = tid; i < G * HD; i += THREADS) {
        const int gg = i / HD, d = i - gg * HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wst[((size_t)w * G + gg) * REC]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float *ws = wst + ((size_t)w * G + gg) * REC;
                const float f = exp2f(ws[0] - M);
                num += f * ws[2 + d];
                den += f * ws[1];
            }
        }
        float *rp = mypart + (size_t)gg * n_split * REC;
        rp[2 + d] = num;
        if (d == 0) { rp[0] = M; rp[1] = den; }
    }
    __threadfence();
    CtaSync::sync();
    if (tid == 0)
        s_last = atomicAdd(&a.counters[t * a.kv.n_kv_head + j], 1u) == (unsigned)(n_eff - 1);
    CtaSync::sync();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of this (row, kv head): merge the splits in split order.
    // Thread tid takes head gg = tid / TPG and DPT consecutive dims (DPT even,
    // G * HD / DPT <= THREADS threads take part); it fetches the (max, sum)
    // pair and its dims of MB splits at once, then folds them in split order
    // into a running max, sum and numerators, so a merge costs a few L2 round
    // trips.
    constexpr int DPT = G * HD / THREADS > 2 ? G * HD / THREADS : 2;   // dims per thread
    constexpr int TPG = HD / DPT;                                       // threads per head
    if (tid < G * TPG) {
        constexpr int MB = 8;                            // splits fetched at once
        const int gg = tid / TPG, d0 = (tid - gg * TPG) * DPT;
        const float *rp = a.part + ((size_t)(t * H + j * G + gg) * n_split) * REC;
        float m_run = -INFINITY, l_run = 0.f, num[DPT];
#pragma unroll
        for (int e = 0; e < DPT; ++e) num[e] = 0.f;
        for (int p0 = 0; p0 < n_eff; p0 += MB) {
            float2 st[MB];
            float2 v[MB][DPT / 2];
#pragma unroll
            for (int q = 0; q < MB; ++q) {
                if (p0 + q < n_eff) {
                    const float *r = rp + (size_t)(p0 + q) * REC;
                    st[q] = __ldcg(reinterpret_cast<const float2 *>(r));
#pragma unroll
                    for (int e = 0; e < DPT / 2; ++e) v[q][e] = __ldcg(reinterpret_cast<const float2 *>(r + 2 + d0) + e);
                }
            }
#pragma unroll
            for (int q = 0; q < MB; ++q) {
                if (p0 + q < n_eff && st[q].x != -INFINITY) {
                    const float mn = fmaxf(m_run, st[q].x);
                    const float fo = m_run == -INFINITY ? 0.f : exp2f(m_run - mn);
                    const float fn = exp2f(st[q].x - mn);
                    l_run = l_run * fo + st[q].y * fn;
#pragma unroll
                    for (int e = 0; e < DPT / 2; ++e) {
                        num[2 * e] = num[2 * e] * fo + v[q][e].x * fn;
                        num[2 * e + 1] = num[2 * e + 1] * fo + v[q][e].y * fn;
                    }
                    m_run = mn;
                }
            }
        }
        const float il = l_run > 0.f ? 1.f / l_run : 0.f;
        f16 *op = a.o + (size_t)t * H * HD + (size_t)(j * G + gg) * HD + d0;
#pragma unroll
        for (int e = 0; e < DPT / 2; ++e)
            *reinterpret_cast<uint32_t *>(op + 2 * e) = pack_h2(num[2 * e] * il, num[2 * e + 1] * il);
    }
    if (tid == 0) a.counters[t * a.kv.n_kv_head + j] = 0u;
}

}  // namespace attn_dec
}  // namespace llm
