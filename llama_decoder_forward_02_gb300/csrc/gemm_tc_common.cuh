// Pieces shared by the tcgen05 kernels (the CTA-pair prefill GEMMs and the
// prefill attention): tile constants, tcgen05 fences, the shared-memory
// operand descriptor, the TMEM load, and the fused epilogues of the Llama
// layer applied to 32 accumulator columns of one output row.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace llm {
namespace tcg {

constexpr int BM = 128, BK = 64, THREADS = 128;

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand in the canonical
// 128-byte-swizzle layout TMA writes: 8-row x 128-byte atoms, 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);     // start address
    d |= (uint64_t)1 << 16;                      // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;                      // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                      // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The RMSNorm scale of a row whose A operand was f16(h * gain): from the
// producer's per-32-column partial sums of h^2, summed in column order.
// Eight loads are issued together per round (n_ss is a multiple of 4).
__device__ __forceinline__ float row_norm_scale(const GemmArgs &a, int row) {
    if (!a.row_ss) return 1.f;
    const float4 *p = reinterpret_cast<const float4 *>(a.row_ss + (size_t)row * a.n_ss);
    const int n4 = a.n_ss / 4;
    float s = 0.f;
    for (int g0 = 0; g0 < n4; g0 += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = g0 + i < n4 ? __ldcg(p + g0 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            s += v[i].x; s += v[i].y; s += v[i].z; s += v[i].w;
        }
    }
    return 1.0f / sqrtf(s / (float)(32 * a.n_ss) + a.eps);
}

// The RMSNorm scales of rows row0 .. row0 + BM - 1 into s[0 .. BM - 1], by
// the warps wi = 0 .. nw - 1 of the caller together.  A warp takes RB rows at
// a time and reads each row's partial sums as consecutive float4s across its
// lanes, one coalesced request per row and RB requests in flight; one row
// per thread made every request touch 32 lines, which held up the SM's
// memory pipeline and with it the TMA ring for microseconds.  Each row's sum
// is then reduced by shuffles.  Rows past M, or no row_ss, give 1.
__device__ __forceinline__ void row_norm_scales(const GemmArgs &a, int row0, float *s, int wi, int nw, int lane) {
    constexpr int RB = 8;
    const int n4 = a.n_ss / 4;
    for (int r0 = wi * RB; r0 < BM; r0 += nw * RB) {
        float v[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) v[i] = 0.f;
        if (a.row_ss) {
            for (int g = lane; g < n4; g += 32) {
                float4 x[RB];
#pragma unroll
                for (int i = 0; i < RB; ++i)
                    x[i] = row0 + r0 + i < a.M
                               ? __ldcg(reinterpret_cast<const float4 *>(a.row_ss + (size_t)(row0 + r0 + i) * a.n_ss) + g)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < RB; ++i) v[i] += (x[i].x + x[i].y) + (x[i].z + x[i].w);
            }
        }
#pragma unroll
        for (int i = 0; i < RB; ++i) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
            if (lane == 0)
                s[r0 + i] = a.row_ss && row0 + r0 + i < a.M ? 1.0f / sqrtf(v[i] / (float)(32 * a.n_ss) + a.eps) : 1.f;
        }
    }
}

// ---------------------------------------------------------------- epilogue on 32 columns of one row
// The epilogue's inputs other than the accumulator for 32 columns of one
// row, loaded ahead of them (epi_fetch) so that their latency overlaps the
// previous 32 columns' work: the residual h (EPI_RESID) or the RoPE cos /
// sin pairs of the row's position (EPI_QKV, q and k columns).
struct EpiSide {
    float4 f[8];
};
template <int EPI>
__device__ __forceinline__ void epi_fetch(const GemmArgs &a, int row, int col, EpiSide &s) {
    if (EPI == EPI_RESID) {
        const float4 *src = reinterpret_cast<const float4 *>(a.hres + (size_t)row * a.ldh + col);
#pragma unroll
        for (int i = 0; i < 8; ++i) s.f[i] = src[i];
    } else if (EPI == EPI_QKV) {
        const int pos = a.pos[row], hd = a.kv.head_dim;
        if (col < a.n_q + a.n_kv && pos >= 0 && pos < a.kv.n_ctx) {
            // 32 columns of q or k never straddle a head: their 16 (cos, sin)
            // pairs are consecutive in the row of the table
            const int rbase = col < a.n_q ? 0 : a.n_q;
            const int p0 = ((col - rbase) % hd) / 2;
            if (a.rope_t) {
                // position-minor table: lane l reads position pos_l of pair p0 + i,
                // consecutive positions in one request
                float2 *f2 = reinterpret_cast<float2 *>(s.f);
#pragma unroll
                for (int i = 0; i < 16; ++i) f2[i] = a.rope_t[(size_t)(p0 + i) * a.rope_n + pos];
            } else {
                const float4 *cs = reinterpret_cast<const float4 *>(a.rope + (size_t)pos * (hd / 2) + p0);
#pragma unroll
                for (int i = 0; i < 8; ++i) s.f[i] = cs[i];
            }
        }
    }
}

// scale: the row's RMSNorm scale (row_norm_scale; 1 for the residual GEMMs);
// side: what epi_fetch<EPI> loaded for the same row and columns
template <int EPI>
__device__ __forceinline__ void epilogue32(const GemmArgs &a, int row, int col, const uint32_t (&r)[32],
                                           float scale, const EpiSide &side) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * scale;
    if (EPI == EPI_STORE) {
        float4 *dst = reinterpret_cast<float4 *>(a.C + (size_t)row * a.ldc + col);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else if (EPI == EPI_RESID) {
        float4 *dst = reinterpret_cast<float4 *>(a.hres + (size_t)row * a.ldh + col);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 h = side.f[i];
            h.x += v[4 * i]; h.y += v[4 * i + 1]; h.z += v[4 * i + 2]; h.w += v[4 * i + 3];
            dst[i] = h;
            v[4 * i] = h.x; v[4 * i + 1] = h.y; v[4 * i + 2] = h.z; v[4 * i + 3] = h.w;
        }
        if (a.x_next) {
            // the next RMSNorm's input, gain applied, and this 32-column share of sum(h^2)
            const float4 *g4 = reinterpret_cast<const float4 *>(a.gain_next + col);
            uint32_t pk[16];
            float ss = 0.f;
            bool bad = false;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 g = g4[i];
                const float x0 = v[4 * i] * g.x, x1 = v[4 * i + 1] * g.y, x2 = v[4 * i + 2] * g.z, x3 = v[4 * i + 3] * g.w;
                bad |= f16_bad(x0) | f16_bad(x1) | f16_bad(x2) | f16_bad(x3);
                pk[2 * i] = pack_h2(x0, x1);
                pk[2 * i + 1] = pack_h2(x2, x3);
            }
            if (bad) raise_error(a.err, ERRF_F16_RANGE);
#pragma unroll
            for (int i = 0; i < 32; ++i) ss += v[i] * v[i];
            uint4 *xd = reinterpret_cast<uint4 *>(a.x_next + (size_t)row * a.N + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) xd[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            a.ss_next[(size_t)row * (a.N / 32) + col / 32] = ss;
        }
    } else if (EPI == EPI_SWIGLU) {
        // 32 columns = two groups of (8 gate, 8 up) with the same 8 output indices
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const int j = ((col + grp * 16) / (2 * GU_GROUP)) * GU_GROUP;
            uint4 o;
            uint32_t *op = &o.x;
            bool bad = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float g0 = v[grp * 16 + 2 * i], g1 = v[grp * 16 + 2 * i + 1];
                const float u0 = v[grp * 16 + 8 + 2 * i], u1 = v[grp * 16 + 8 + 2 * i + 1];
                const float y0 = silu_fast(g0) * u0, y1 = silu_fast(g1) * u1;
                bad |= f16_bad(y0) | f16_bad(y1);
                op[i] = pack_h2(y0, y1);
            }
            if (bad) raise_error(a.err, ERRF_F16_RANGE);
            *reinterpret_cast<uint4 *>(a.u_out + (size_t)row * a.ldu + j) = o;
        }
    } else if (EPI == EPI_QKV) {
        const int pos = a.pos[row], seq = a.seq[row];
        if (pos < 0 || pos >= a.kv.n_ctx || seq < 0 || seq >= a.kv.n_seq) {
            raise_error(a.err, ERRF_BAD_INDEX);
            return;
        }
        const int hd = a.kv.head_dim;
        const bool rot = col < a.n_q + a.n_kv;           // 32 columns never straddle q/k/v
        if (rot) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float4 q4 = side.f[i / 2];
                const float cx = (i & 1) ? q4.z : q4.x, cy = (i & 1) ? q4.w : q4.y;
                const float x0 = v[2 * i], x1 = v[2 * i + 1];
                v[2 * i] = x0 * cx - x1 * cy;
                v[2 * i + 1] = x0 * cy + x1 * cx;
            }
        }
        if (col >= a.n_q && a.kv.k8) {
            // FP8 E4M3 cache: 32 columns are 32 bytes
            const bool is_k = col < a.n_q + a.n_kv;
            const int c = col - a.n_q - (is_k ? 0 : a.n_kv);
            const int head = c / hd, d = c - head * hd;
            uint32_t p8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                p8[i] = (uint32_t)pack_e4m3x2(v[4 * i], v[4 * i + 1]) |
                        ((uint32_t)pack_e4m3x2(v[4 * i + 2], v[4 * i + 3]) << 16);
            uint4 *d8 = reinterpret_cast<uint4 *>((is_k ? a.kv.k8 : a.kv.v8) + (size_t)seq * a.kv.seq_stride +
                                                  ((size_t)head * a.kv.n_ctx + pos) * hd + d);
            d8[0] = make_uint4(p8[0], p8[1], p8[2], p8[3]);
            d8[1] = make_uint4(p8[4], p8[5], p8[6], p8[7]);
            return;
        }
        uint32_t pk[16];
        bool bad = false;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            bad |= f16_bad(v[2 * i]) | f16_bad(v[2 * i + 1]);
            pk[i] = pack_h2(v[2 * i], v[2 * i + 1]);
        }
        if (bad) raise_error(a.err, ERRF_F16_RANGE);
        f16 *dst;
        if (col < a.n_q) {
            dst = a.q_out + (size_t)row * a.n_q + col;
        } else {
            const bool is_k = col < a.n_q + a.n_kv;
            const int c = col - a.n_q - (is_k ? 0 : a.n_kv);
            const int head = c / hd, d = c - head * hd;
            dst = (is_k ? a.kv.k : a.kv.v) + (size_t)seq * a.kv.seq_stride + ((size_t)head * a.kv.n_ctx + pos) * hd + d;
        }
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
}

// The epilogue of one accumulator row over the 32-column chunks [c0, c1) of
// the tile at column n0, the chunk's accumulator at tmem_row + 32 c: the
// side inputs of the next chunk are requested before this chunk's
// accumulator is read and applied, so two chunks' loads are in flight.
template <int EPI>
__device__ __forceinline__ void epilogue_chunks(const GemmArgs &a, int row, int n0, uint32_t tmem_row, int c0, int c1,
                                                float scale) {
    const bool live = row < a.M;
    EpiSide s0, s1;
    if (live && c0 < c1) epi_fetch<EPI>(a, row, n0 + c0 * 32, s0);
#pragma unroll 1
    for (int c = c0; c < c1; c += 2) {
        uint32_t r[32];
        if (live && c + 1 < c1) epi_fetch<EPI>(a, row, n0 + (c + 1) * 32, s1);
        tmem_ld32(tmem_row + (uint32_t)(c * 32), r);
        if (live) epilogue32<EPI>(a, row, n0 + c * 32, r, scale, s0);
        if (c + 1 < c1) {
            if (live && c + 2 < c1) epi_fetch<EPI>(a, row, n0 + (c + 2) * 32, s0);
            tmem_ld32(tmem_row + (uint32_t)((c + 1) * 32), r);
            if (live) epilogue32<EPI>(a, row, n0 + (c + 1) * 32, r, scale, s1);
        }
    }
}

}  // namespace tcg
}  // namespace llm
