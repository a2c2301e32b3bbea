// Prefill attention on the 5th-generation tensor cores: causal grouped-query
// attention of a ubatch's rows against their sequence's KV cache, tiled over
// keys with an online softmax ("Inside the inference engine: model
// architectures and forward pass", sections "Detailed explanation: Llama's
// forward pass in Go" (ScaledDotProduct over the cache, GQA) and "KV Cache:
// memory for causal attention" (full causal mask, optional sliding window);
// "LLama.cpp — how it works", "KV-cache and the Prefill / Decode stages").
//
// One CTA takes 128 query rows of one sequence (consecutive positions pos0 ..)
// for one query head h and walks the 128-key tiles of its kv head j = h / G.
// Both products run as tcgen05.mma (kind::f16, M = 128, fp32 accumulators in
// tensor memory):
//   S_t = Q K_t^T   A = Q (128 x hd, K-major), B = K_t (128 keys x hd,
//                   K-major), into one of two 128-column S buffers;
//   O  += P_t V_t   A = P_t (128 x 128 keys, fp16, held in tensor memory:
//                   lane = row, each 32-bit column a pair of keys; two
//                   buffers), B = V_t (keys x hd with hd contiguous: the
//                   MN-major operand form), into the hd-column O accumulator.
// Q, K_t and V_t arrive by TMA (128-byte swizzle, boxes of 128 rows x 64
// columns) straight from the cache layout [seq][layer][kv_head][pos][hd].
//
// Warps (384 threads):
//   0  TMA producer of Q (once) and K_t, 10 TMA producer of V_t, each into its
//      own ring (head_dim 128: 3 K and 3 V stages; 64: 4 and 4): a K stage is
//      free again once S_t is computed, a V stage once O += P_t V_t is.  With
//      every SM loading, a 32 KB tile takes microseconds to land, so the
//      rings are as deep as shared memory allows.  The tiles of keys written
//      by earlier ubatches are requested before the programmatic-dependent-
//      launch wait.
//   1  issuer of S_t = Q K_t^T (one lane), into S buffer t & 1 once the
//      softmax has read S_{t-2} from it;
//   11 issuer of O += P_t V_t (one lane) once the softmax has written P_t.
//      Two issuers, so that neither stream waits behind the other's
//      dependencies (one issuer doing both took ~1.35 us a key tile, two
//      ~0.96 us); the tensor pipe computes S_{t+1} while the softmax warps
//      work on S_t.
//   2-9  softmax, two threads per query row (TMEM lane 32 (w % 4) + lane),
//      warps 2-5 on keys 0-63 of each tile and warps 6-9 on keys 64-127: load
//      the half row of S, mask, tile maximum (the two halves exchange theirs
//      through spare tensor-memory columns), running max in base 2,
//      p = 2^(s c - m c) with c = log2(e) / sqrt(hd) (exponents in fp32,
//      rounded to fp16 pairs, two results a special-function op), partial
//      row sum of those fp16 values in fp32, the half row of P into tensor
//      memory (tcgen05.st).  The running max is raised (and O and the sums
//      rescaled) only when a tile's maximum exceeds it by more than 8 in base
//      2, so most tiles skip the O rescale; p stays <= 2^8, well inside fp16.
//      At the end each half divides its half of the O row by the summed row
//      sum and stores it as fp16.
// Every mbarrier wait is bounded; on a timeout the CTA raises
// ERRF_WAIT_TIMEOUT, stops, waits (bounded) for its own copies in flight,
// frees its tensor memory and returns.
#include <cuda.h>

#include "common.cuh"
#include "launch.cuh"
#include "tma.cuh"
#include "cluster.cuh"
#include "gemm_tc_common.cuh"

namespace llm {

namespace {

using tcg::sdesc;
using tcg::tc_fence_after;
using tcg::tc_fence_before;
using tcg::tmem_ld32;

constexpr int BQ = 128, BKEY = 128, FA_THREADS = 384;   // 2 + 8 + 2 warps
constexpr int SM_WARPS = 8;                                   // softmax warps (2-9)
constexpr int V_WARP = 10;                                    // the V producer
constexpr int PV_WARP = 11;                                   // the issuer of O += P V
constexpr uint32_t BOX = 128 * 128;          // bytes of one 128-row x 64-column fp16 box
constexpr uint32_t TMEM_COLS = 512;          // S0 [0, 128), S1 [128, 256), O [256, 256 + hd), P0, P1 (64 each)
constexpr float RESCALE_LOG2 = 8.f;          // raise the running max only past this margin

template <int HD>
struct FaCfg {
    static constexpr int NB = HD / 64;                          // 64-column boxes per row
    static constexpr uint32_t Q_OFF = 0;
    // ring depths: as many tiles in flight as shared memory allows
    static constexpr int KST = HD == 128 ? 3 : 4;               // K stages
    static constexpr int VST = HD == 128 ? 3 : 4;               // V stages
    static constexpr uint32_t O_COL = 256;                      // O accumulator columns [256, 256 + HD)
    static constexpr uint32_t P_COL = 256 + HD;                 // P_t (fp16 pairs): 64 columns, two buffers
    static constexpr uint32_t K_OFF = NB * BOX;                 // [KST stages][NB boxes]
    static constexpr uint32_t V_OFF = K_OFF + KST * NB * BOX;   // [VST stages][NB boxes]
    static constexpr uint32_t BAR_OFF = V_OFF + VST * NB * BOX;
    // barriers + alignment slack; at least 120 KB so that one CTA fills an SM
    // (a second CTA would only wait in tcgen05.alloc for the first's columns)
    static constexpr size_t SMEM = BAR_OFF + 256 + 1024 > 120 * 1024 ? BAR_OFF + 256 + 1024 : 120 * 1024;
    // kind::f16 instruction descriptors: D fp32 (bit 4), A and B fp16, M = 128
    // (M >> 4 at bit 24), N >> 3 at bit 17; bit 16 marks B as MN-major
    static constexpr uint32_t IDESC_S = (1u << 4) | ((uint32_t)(BKEY >> 3) << 17) | ((uint32_t)(BQ >> 4) << 24);
    static constexpr uint32_t IDESC_O =
        (1u << 4) | (1u << 16) | ((uint32_t)(HD >> 3) << 17) | ((uint32_t)(BQ >> 4) << 24);
};

__device__ __forceinline__ void mma1(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        :: "r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(accum) : "memory");
}
// The same with A in tensor memory (P: lane = row, 32-bit column j = the fp16
// pair of keys 2j, 2j + 1; a K = 16 step reads 8 columns).
__device__ __forceinline__ void mma1_ts(uint32_t tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
        :: "r"(tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum) : "memory");
}
__device__ __forceinline__ void commit1(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}
// Shared-memory descriptor of an MN-major operand (the MN dimension
// contiguous) in the 128-byte-swizzle layout: atoms of 64 MN elements x 8 K
// rows; `lbo` bytes between 64-element MN blocks, 1024 bytes between 8-row K
// groups.
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
           "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
           "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// One 32-bit value per lane to / from a TMEM column (the softmax halves
// exchange their row maxima and sums through columns of an idle S buffer).
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" :: "r"(taddr), "r"(__float_as_uint(v)) : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
    uint32_t v;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    return __uint_as_float(v);
}
// 2^x of an fp16 pair on the special-function unit (two results an op)
__device__ __forceinline__ uint32_t ex2_h2(uint32_t x) {
    uint32_t y;
    asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// acc + lo + hi of an fp16 pair, each added exactly into fp32 (fma by 1)
__device__ __forceinline__ float add_h2_f32(uint32_t p, float acc) {
    asm("{\n\t.reg .b16 lo, hi, one;\n\t"
        "mov.b32 {lo, hi}, %1;\n\tmov.b16 one, 0x3C00;\n\t"
        "fma.rn.f32.f16 %0, lo, one, %0;\n\tfma.rn.f32.f16 %0, hi, one, %0;\n\t}"
        : "+f"(acc) : "r"(p));
    return acc;
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// The softmax warps (2-9) of a query tile: two threads per row, each on 64
// keys of every 128-key tile (see the kernel comment).  s_full(b) / pv_done(pb)
// are this CTA's barriers; s_free_arrive(b) / p_full_arrive(b) report this
// warp's share to the MMA issuer's barriers.
template <int HD, bool WIN, class SFull, class SFree, class PFull, class PvDone>
__device__ __forceinline__ void softmax_warps(const AttnPrefillTcArgs &a, const AttnTile &tl, int h, int kt0, int nt,
                                              uint32_t tmem, int warp, int lane, volatile int *abort, SFull s_full,
                                              SFree s_free_arrive, PFull p_full_arrive, PvDone pv_done) {
    using C = FaCfg<HD>;
    const int W = WIN ? a.window : 0;
    // ---- softmax: thread row r of the query tile, keys [64 hf, 64 hf + 64) of each tile
    constexpr int HK = BKEY / 2;
    const int quarter = warp & 3, hf = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int qpos = tl.pos0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t o_col = C::O_COL + hf * (HD / 2);     // this half's O columns
    const float c = 1.4426950408889634f / sqrtf((float)HD);
    float m_run = -INFINITY, l_run = 0.f;
    // ok stays uniform over each warp (__all_sync), and every softmax
    // thread runs all nt iterations, so the named barriers (which have
    // no time limit) are always reached by all 256 threads; after a
    // timeout the iterations only pass the barriers
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
        const int b = t & 1, key0 = (kt0 + t) * BKEY + hf * HK;
        ok = __all_sync(0xffffffffu, ok && mbar_wait(s_full(b), (t >> 1) & 1, abort, a.err));
        float s[HK];
        float mx = -INFINITY;
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < HK / 32; ++q) {
                uint32_t v[32];
                tmem_ld32(lane_base + b * BKEY + hf * HK + q * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[q * 32 + i] = __uint_as_float(v[i]);
            }
            // causal (and window) mask: key k is visible iff k <= qpos (and qpos - k < W)
            const bool need_mask = key0 + HK - 1 > qpos || (WIN && qpos - key0 >= W);
            if (need_mask) {
#pragma unroll
                for (int i = 0; i < HK; ++i) {
                    const int k = key0 + i;
                    if (k > qpos || (WIN && qpos - k >= W)) s[i] = -INFINITY;
                }
            }
            // half-row maximum as a tree of 8 independent chains
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
            for (int i = 8; i < HK; ++i) m8[i & 7] = fmaxf(m8[i & 7], s[i]);
            mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        }
        // the halves exchange their maxima through the first column of each
        // half of this S buffer (already read by its own half); the buffer
        // is released to the next QK^T only after both have read
        if (ok) tmem_st1(lane_base + b * BKEY + hf * HK, mx);
        named_sync(1, SM_WARPS * 32);
        if (ok) {
            mx = fmaxf(mx, tmem_ld1(lane_base + b * BKEY + (hf ^ 1) * HK));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) s_free_arrive(b);
        }
        if (!ok) continue;
        // raise the running max only when this tile's max passes it by > 8 (base 2)
        float factor = 1.f;
        const bool raise = mx != -INFINITY && (m_run == -INFINITY || (mx - m_run) * c > RESCALE_LOG2);
        if (raise) {
            factor = m_run == -INFINITY ? 0.f : ex2((m_run - mx) * c);
            m_run = mx;
        }
        const float mc = m_run == -INFINITY ? 0.f : m_run * c;
        uint32_t p[HK / 2];
        float rs8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
        for (int i = 0; i < HK / 2; ++i) {
            // exponents in fp32, rounded to fp16 pairs; one special-function
            // op gives two fp16 probabilities (<= 2^8), which are the P the
            // tensor cores read; the row sum adds those same values in fp32
            const float x0 = fmaf(s[2 * i], c, -mc), x1 = fmaf(s[2 * i + 1], c, -mc);
            p[i] = ex2_h2(pack_h2(x0, x1));
            rs8[i & 7] = add_h2_f32(p[i], rs8[i & 7]);
        }
        const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        l_run = l_run * factor + rs;
        // P_t goes to TMEM buffer t & 1, last read by P_{t-2} V_{t-2}; a raised
        // maximum also rescales O, which P_{t-1} V_{t-1} must have finished
        const bool any_raise = __any_sync(0xffffffffu, raise);
        if (t >= 1 && any_raise) {
            ok = __all_sync(0xffffffffu, mbar_wait(pv_done((t - 1) & 1), ((t - 1) >> 1) & 1, abort, a.err));
            if (!ok) continue;
            tc_fence_after();
#pragma unroll 1
            for (int q = 0; q < HD / 64; ++q) {
                uint32_t v[32];
                tmem_ld32(lane_base + o_col + q * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * factor);
                tmem_st32(lane_base + o_col + q * 32, v);
            }
        }
        if (t >= 2) {
            ok = __all_sync(0xffffffffu, mbar_wait(pv_done(t & 1), ((t >> 1) - 1) & 1, abort, a.err));
            if (!ok) continue;
            tc_fence_after();
        }
        // this half of the P row: 64 keys as 32 fp16 pairs into the row's TMEM lane
        tmem_st32(lane_base + C::P_COL + (uint32_t)(t & 1) * 64 + hf * 32, p);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) p_full_arrive(t & 1);
    }
    // the row sum is the two halves' partial sums (same running max),
    // exchanged through S buffer 0, idle once the last S has been read
    if (ok) tmem_st1(lane_base + hf * HK, l_run);
    named_sync(1, SM_WARPS * 32);
    const float l_row = ok ? l_run + tmem_ld1(lane_base + (hf ^ 1) * HK) : 0.f;
    if (__all_sync(0xffffffffu, ok && mbar_wait(pv_done((nt - 1) & 1), ((nt - 1) >> 1) & 1, abort, a.err))) {
        tc_fence_after();
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
        f16 *dst = a.o + (size_t)(tl.row0 + r) * a.ldo + h * HD + hf * (HD / 2);
#pragma unroll 1
        for (int q = 0; q < HD / 64; ++q) {
            uint32_t v[32];
            tmem_ld32(lane_base + o_col + q * 32, v);
            if (r < tl.n_rows) {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + q * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    d4[i] = make_uint4(pack_h2(__uint_as_float(v[8 * i]) * inv, __uint_as_float(v[8 * i + 1]) * inv),
                                       pack_h2(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv),
                                       pack_h2(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv),
                                       pack_h2(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv));
            }
        }
    }
}

template <int HD, bool WIN>
__global__ void __launch_bounds__(FA_THREADS, 1)
attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const AttnPrefillTcArgs a) {
    using C = FaCfg<HD>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ int s_abort;
    __shared__ uint32_t s_tmem;
    __shared__ int s_issued[2];              // K and V tiles each producer armed

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t bar = base + C::BAR_OFF;
    // q_full, s_full[2], s_free[2], p_full[2] (at 5 and 24), pv_done[2] (at 6 and 23), k_full[4], k_empty[4],
    // v_full[4], v_empty[4]
    const uint32_t q_full = bar;
    auto k_full = [&](int s) { return bar + 8u * (7 + s); };
    auto k_empty = [&](int s) { return bar + 8u * (11 + s); };
    auto v_full = [&](int s) { return bar + 8u * (15 + s); };
    auto v_empty = [&](int s) { return bar + 8u * (19 + s); };
    auto s_full = [&](int b) { return bar + 8u * (1 + b); };
    auto s_free = [&](int b) { return bar + 8u * (3 + b); };
    auto p_full = [&](int pb) { return bar + 8u * (pb ? 24 : 5); };    // P of tiles with this P buffer written
    auto pv_done = [&](int pb) { return bar + 8u * (pb ? 23 : 6); };   // PV of tiles with this P buffer
    auto q_box = [&](int i) { return base + C::Q_OFF + i * BOX; };
    auto k_box = [&](int s, int i) { return base + C::K_OFF + (s * C::NB + i) * BOX; };
    auto v_box = [&](int s, int i) { return base + C::V_OFF + (s * C::NB + i) * BOX; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // longest tiles (latest positions) first
    const AttnTile tl = a.tiles[a.n_tiles - 1 - (int)blockIdx.x];
    const int h = blockIdx.y, G = a.H / a.Hkv, j = h / G;
    volatile int *abort = &s_abort;

    const bool bad = tl.seq < 0 || tl.seq >= a.n_seq || tl.pos0 < 0 || tl.n_rows < 1 || tl.n_rows > BQ ||
                     tl.pos0 + tl.n_rows > a.n_ctx;
    if (bad) {
        if (threadIdx.x == 0) raise_error(a.err, ERRF_BAD_INDEX);
        return;
    }
    const int pos_last = tl.pos0 + tl.n_rows - 1;
    const int W = WIN ? a.window : 0;
    const int kt0 = (W > 0 && tl.pos0 + 1 > W) ? (tl.pos0 + 1 - W) / BKEY : 0;
    const int kt1 = pos_last / BKEY + 1;                 // key tiles [kt0, kt1)
    const int nt = kt1 - kt0;
    // cache row of (seq, layer, kv head j, position 0)
    const int kv_row0 = ((tl.seq * a.n_layer + a.layer) * a.Hkv + j) * a.n_ctx;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < C::KST; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < C::VST; ++s) {
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(s_free(b), SM_WARPS);
        }
        mbar_init(p_full(0), SM_WARPS);
        mbar_init(p_full(1), SM_WARPS);
        s_issued[0] = s_issued[1] = 0;
        mbar_init(pv_done(0), 1);
        mbar_init(pv_done(1), 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&s_tmem)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // keys below kv_ready were written before the kernel that precedes this one
    auto load_k = [&](int t) {
        const int s = t % C::KST, key0 = (kt0 + t) * BKEY;
        mbar_expect_tx(k_full(s), C::NB * BOX);
        for (int i = 0; i < C::NB; ++i) tma_load_2d(k_box(s, i), &tmK, k_full(s), i * 64, kv_row0 + key0);
    };
    auto load_v = [&](int t) {
        const int s = t % C::VST, key0 = (kt0 + t) * BKEY;
        mbar_expect_tx(v_full(s), C::NB * BOX);
        for (int i = 0; i < C::NB; ++i) tma_load_2d(v_box(s, i), &tmV, v_full(s), i * 64, kv_row0 + key0);
    };
    const bool producer = (warp == 0 || warp == V_WARP) && lane == 0;
    int early = 0;                                       // tiles requested before the dependency wait
    if (producer) {
        const int ring = warp == 0 ? C::KST : C::VST;
        while (early < ring && early < nt && (kt0 + early + 1) * BKEY <= tl.kv_ready) {
            if (warp == 0) load_k(early); else load_v(early);
            ++early;
        }
    }
    pdl_wait();
    pdl_trigger();

    if (warp == 0 || warp == V_WARP) {
        if (lane == 0) {
            const bool is_k = warp == 0;
            if (is_k) {
                mbar_expect_tx(q_full, C::NB * BOX);
                for (int i = 0; i < C::NB; ++i) tma_load_2d(q_box(i), &tmQ, q_full, h * HD + i * 64, tl.row0);
            }
            int issued = early;
            for (int t = early; t < nt; ++t) {
                const int ns = is_k ? C::KST : C::VST;
                if (t >= ns && !mbar_wait(is_k ? k_empty(t % ns) : v_empty(t % ns), ((t / ns) - 1) & 1, abort, a.err))
                    break;
                if (is_k) load_k(t); else load_v(t);
                issued = t + 1;
            }
            s_issued[is_k ? 0 : 1] = issued;
        }
        __syncwarp();
    } else if (warp == 1) {
        // S_t = Q K_t^T into S buffer t & 1 once the softmax has read S_{t-2} from it
        if (lane == 0 && mbar_wait(q_full, 0, abort, a.err)) {
            for (int t = 0; t < nt; ++t) {
                const int b = t & 1;
                if (t >= 2 && !mbar_wait(s_free(b), ((t >> 1) - 1) & 1, abort, a.err)) break;
                const int ks = t % C::KST;
                if (!mbar_wait(k_full(ks), (t / C::KST) & 1, abort, a.err)) break;
                tc_fence_after();
                const uint32_t s_acc = tmem + b * BKEY;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t ad = sdesc(q_box(kk >> 2) + (kk & 3) * 32);
                    const uint64_t bd = sdesc(k_box(ks, kk >> 2) + (kk & 3) * 32);
                    mma1(s_acc, ad, bd, C::IDESC_S, kk != 0);
                }
                commit1(k_empty(ks));                  // the K stage is free once S_t is done
                commit1(s_full(b));
            }
        }
        __syncwarp();
    } else if (warp == PV_WARP) {
        // O (+)= P_t V_t once the softmax has written P_t (and rescaled O)
        if (lane == 0) {
            const uint32_t o_acc = tmem + C::O_COL;
            for (int t = 0; t < nt; ++t) {
                if (!mbar_wait(p_full(t & 1), (t >> 1) & 1, abort, a.err) ||
                    !mbar_wait(v_full(t % C::VST), (t / C::VST) & 1, abort, a.err))
                    break;
                tc_fence_after();
                const uint32_t p_tm = tmem + C::P_COL + (uint32_t)(t & 1) * 64;
#pragma unroll
                for (int kk = 0; kk < BKEY / 16; ++kk) {
                    const uint64_t bd = sdesc_mn(v_box(t % C::VST, 0) + kk * 2048, BOX);
                    mma1_ts(o_acc, p_tm + (uint32_t)kk * 8, bd, C::IDESC_O, (t | kk) != 0);
                }
                commit1(v_empty(t % C::VST));
                commit1(pv_done(t & 1));
            }
        }
        __syncwarp();
    } else {
        softmax_warps<HD, WIN>(a, tl, h, kt0, nt, tmem, warp, lane, abort, s_full,
                               [&](int b) { mbar_arrive(s_free(b)); }, [&](int b) { mbar_arrive(p_full(b)); },
                               pv_done);
    }
    tc_fence_before();
    __syncthreads();
    if (*abort && (warp == 0 || warp == V_WARP) && lane == 0) {
        // wait (bounded) for the copies still in flight before the memory is released
        const bool is_k = warp == 0;
        if (is_k)
            for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(q_full, 0); ++i) {
            }
        const int issued = s_issued[is_k ? 0 : 1] > early ? s_issued[is_k ? 0 : 1] : early;
        const int ns = is_k ? C::KST : C::VST;
        for (int t = (issued > ns ? issued - ns : 0); t < issued; ++t) {
            const uint32_t fb = is_k ? k_full(t % ns) : v_full(t % ns);
            for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(fb, (t / ns) & 1); ++i) {
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------- CTA pairs
// The two query heads 2i and 2i + 1 of one GQA group (same kv head, same
// rows) run on a pair of SMs as one cta_group::2 MMA stream with M = 256:
// CTA r holds head 2i + r's 128 query rows and accumulators (its S, P and O
// in its own tensor memory) and stages half of every K/V tile: keys
// [64 r, 64 r + 64) of K_t (the pair's S_t = Q K_t^T takes its N = 128 keys
// from both CTAs) and head_dim columns [64 r, 64 r + 64) of V_t (O's
// N = 128 columns likewise).  An SM thus receives 32 KB a key tile instead
// of 64 KB.  The even CTA issues every MMA; all TMA loads of both CTAs
// complete on the even CTA's barriers, the odd CTA's softmax warps arrive on
// them remotely, and every commit is multicast to both CTAs.  head_dim 128
// only (one 64-column V box per CTA), G even.  Measured on the 8B shape's
// 512-row ubatches it is slower than one CTA a head (22.4 vs 20.6 us a
// layer): with the MMA issue split over two warps both run at ~0.96 us a
// key tile, bounded by neither the loads nor the MMAs' nominal time, and the
// pair adds the lock step of two SMs; it is option "attn_prefill" 2.
template <int HD>
struct FaPairCfg {
    static constexpr int NB = HD / 64;
    static constexpr int KST = 6, VST = 6;                      // ring stages (16 KB each)
    static constexpr uint32_t KBOX = 64 * 128;                  // one 64-key x 64-column box
    static constexpr uint32_t K_STAGE = NB * KBOX;              // a CTA's half of K_t
    static constexpr uint32_t V_STAGE = BOX;                    // a CTA's 128 keys x 64 columns of V_t
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t K_OFF = NB * BOX;
    static constexpr uint32_t V_OFF = K_OFF + KST * K_STAGE;
    static constexpr uint32_t BAR_OFF = V_OFF + VST * V_STAGE;
    static constexpr size_t SMEM = BAR_OFF + 512 + 1024;
    // M = 256 (the pair's rows), N = 128 keys / HD columns
    static constexpr uint32_t IDESC_S = (1u << 4) | ((uint32_t)(BKEY >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
    static constexpr uint32_t IDESC_O =
        (1u << 4) | (1u << 16) | ((uint32_t)(HD >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
};

__device__ __forceinline__ void mma2(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}"
        :: "r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(accum) : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}"
        :: "r"(tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum) : "memory");
}
// arrive once on the mbarrier at this offset in both CTAs when the MMAs issued so far are done
__device__ __forceinline__ void commit2(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        :: "r"(bar), "h"((uint16_t)3) : "memory");
}
// a TMA load into this CTA that completes on an mbarrier of either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t cluster_bar, int x,
                                                 int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(x), "r"(y) : "memory");
}
// arrive on an mbarrier of either CTA of the pair (default semantics: a
// cluster-scope release here cost ~0.5 us an arrival, measured)
__device__ __forceinline__ void arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" :: "r"(cluster_bar) : "memory");
}
__device__ __forceinline__ uint32_t leader_addr(uint32_t local) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(0u));
    return r;
}
// After an abort: wait (bounded) until every load of a ring that either CTA
// issued has landed on the even CTA's barriers (`mine` / `peer` tiles issued;
// a tile only the odd CTA issued gets the even CTA's arrival with its bytes).
__device__ void drain_ring(uint32_t full0, int mine, int peer, int stages, uint32_t bytes) {
    const int hi = mine > peer ? mine : peer;
    for (int t = (hi > stages ? hi - stages : 0); t < hi; ++t) {
        const uint32_t b = full0 + 8u * (uint32_t)(t % stages);
        if (t >= mine) mbar_expect_tx(b, bytes);
        for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(b, (t / stages) & 1); ++i) {
        }
    }
}

template <int HD, bool WIN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FA_THREADS, 1)
attn_prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK64,
                         const __grid_constant__ CUtensorMap tmV, const AttnPrefillTcArgs a) {
    using C = FaPairCfg<HD>;
    using F = FaCfg<HD>;                      // tensor-memory columns as in the one-CTA kernel
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ int s_abort;
    __shared__ uint32_t s_tmem;
    __shared__ int s_issued[2];               // K and V tiles this CTA's producers issued
    __shared__ int s_peer[3];                 // (even CTA) the odd CTA's issued K, V tiles and abort flag

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t bar = base + C::BAR_OFF;
    // q_full 0, s_full 1-2, s_free 3-4, p_full 5 and 38, pv_done 6-7, k_full 8-13, k_empty 16-21, v_full 24-29,
    // v_empty 32-37
    const uint32_t q_full = bar;
    auto s_full = [&](int b) { return bar + 8u * (1 + b); };
    auto s_free = [&](int b) { return bar + 8u * (3 + b); };
    auto p_full = [&](int pb) { return bar + 8u * (pb ? 38 : 5); };
    auto pv_done = [&](int pb) { return bar + 8u * (6 + pb); };
    auto k_full = [&](int s) { return bar + 8u * (8 + s); };
    auto k_empty = [&](int s) { return bar + 8u * (16 + s); };
    auto v_full = [&](int s) { return bar + 8u * (24 + s); };
    auto v_empty = [&](int s) { return bar + 8u * (32 + s); };
    auto q_box = [&](int i) { return base + C::Q_OFF + i * BOX; };
    auto k_box = [&](int s, int i) { return base + C::K_OFF + s * C::K_STAGE + i * C::KBOX; };
    auto v_box = [&](int s) { return base + C::V_OFF + s * C::V_STAGE; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const AttnTile tl = a.tiles[a.n_tiles - 1 - (int)(blockIdx.x >> 1)];
    const int h = 2 * (int)blockIdx.y + (int)rank, G = a.H / a.Hkv, j = h / G;
    volatile int *abort = &s_abort;

    // both CTAs hold the same tile, so both leave here together
    const bool bad = tl.seq < 0 || tl.seq >= a.n_seq || tl.pos0 < 0 || tl.n_rows < 1 || tl.n_rows > BQ ||
                     tl.pos0 + tl.n_rows > a.n_ctx;
    if (bad) {
        if (threadIdx.x == 0) raise_error(a.err, ERRF_BAD_INDEX);
        return;
    }
    const int pos_last = tl.pos0 + tl.n_rows - 1;
    const int W = WIN ? a.window : 0;
    const int kt0 = (W > 0 && tl.pos0 + 1 > W) ? (tl.pos0 + 1 - W) / BKEY : 0;
    const int nt = pos_last / BKEY + 1 - kt0;
    const int kv_row0 = ((tl.seq * a.n_layer + a.layer) * a.Hkv + j) * a.n_ctx;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);                 // (even CTA) both CTAs' Q
        for (int s = 0; s < C::KST; ++s) {
            mbar_init(k_full(s), 1);          // (even CTA) both halves of K_t
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < C::VST; ++s) {
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(s_free(b), 2 * SM_WARPS);   // (even CTA) the softmax warps of both CTAs
            mbar_init(pv_done(b), 1);
        }
        mbar_init(p_full(0), 2 * SM_WARPS);       // (even CTA) the softmax warps of both CTAs
        mbar_init(p_full(1), 2 * SM_WARPS);
        s_issued[0] = s_issued[1] = 0;
        s_peer[0] = s_peer[1] = s_peer[2] = 0;
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmK64)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&s_tmem)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();                           // barriers and tensor memory ready in both CTAs
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    constexpr uint32_t KB = C::K_STAGE, VB = C::V_STAGE;
    auto load_k = [&](int t) {
        const int s = t % C::KST, key0 = (kt0 + t) * BKEY + 64 * (int)rank;
        if (rank == 0) mbar_expect_tx(k_full(s), 2 * KB);
        for (int i = 0; i < C::NB; ++i) tma_load_2d_pair(k_box(s, i), &tmK64, leader_addr(k_full(s)), i * 64, kv_row0 + key0);
    };
    auto load_v = [&](int t) {
        const int s = t % C::VST, key0 = (kt0 + t) * BKEY;
        if (rank == 0) mbar_expect_tx(v_full(s), 2 * VB);
        tma_load_2d_pair(v_box(s), &tmV, leader_addr(v_full(s)), 64 * (int)rank, kv_row0 + key0);
    };
    const bool producer = (warp == 0 || warp == V_WARP) && lane == 0;
    int early = 0;
    if (producer) {
        const int ring = warp == 0 ? C::KST : C::VST;
        while (early < ring && early < nt && (kt0 + early + 1) * BKEY <= tl.kv_ready) {
            if (warp == 0) load_k(early); else load_v(early);
            ++early;
        }
    }
    pdl_wait();
    pdl_trigger();

    if (warp == 0 || warp == V_WARP) {
        if (lane == 0) {
            const bool is_k = warp == 0;
            if (is_k) {
                if (rank == 0) mbar_expect_tx(q_full, 2 * C::NB * BOX);
                for (int i = 0; i < C::NB; ++i)
                    tma_load_2d_pair(q_box(i), &tmQ, leader_addr(q_full), h * HD + i * 64, tl.row0);
            }
            int issued = early;
            const int ns = is_k ? C::KST : C::VST;
            for (int t = early; t < nt; ++t) {
                if (t >= ns && !mbar_wait(is_k ? k_empty(t % ns) : v_empty(t % ns), ((t / ns) - 1) & 1, abort, a.err))
                    break;
                if (is_k) load_k(t); else load_v(t);
                issued = t + 1;
            }
            s_issued[is_k ? 0 : 1] = issued;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0 && mbar_wait(q_full, 0, abort, a.err)) {
            for (int t = 0; t < nt; ++t) {
                const int b = t & 1;
                if (t >= 2 && !mbar_wait(s_free(b), ((t >> 1) - 1) & 1, abort, a.err)) break;
                const int ks = t % C::KST;
                if (!mbar_wait(k_full(ks), (t / C::KST) & 1, abort, a.err)) break;
                tc_fence_after();
                const uint32_t s_acc = tmem + b * BKEY;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t ad = sdesc(q_box(kk >> 2) + (kk & 3) * 32);
                    const uint64_t bd = sdesc(k_box(ks, kk >> 2) + (kk & 3) * 32);
                    mma2(s_acc, ad, bd, C::IDESC_S, kk != 0);
                }
                commit2(k_empty(ks));
                commit2(s_full(b));
            }
        }
        __syncwarp();
    } else if (warp == PV_WARP) {
        if (lane == 0 && rank == 0) {
            const uint32_t o_acc = tmem + F::O_COL;
            for (int t = 0; t < nt; ++t) {
                if (!mbar_wait(p_full(t & 1), (t >> 1) & 1, abort, a.err) ||
                    !mbar_wait(v_full(t % C::VST), (t / C::VST) & 1, abort, a.err))
                    break;
                tc_fence_after();
                const uint32_t p_tm = tmem + F::P_COL + (uint32_t)(t & 1) * 64;
#pragma unroll
                for (int kk = 0; kk < BKEY / 16; ++kk) {
                    const uint64_t bd = sdesc_mn(v_box(t % C::VST) + kk * 2048, BOX);
                    mma2_ts(o_acc, p_tm + (uint32_t)kk * 8, bd, C::IDESC_O, (t | kk) != 0);
                }
                commit2(v_empty(t % C::VST));
                commit2(pv_done(t & 1));
            }
        }
        __syncwarp();
    } else {
        const uint32_t sfree0 = leader_addr(s_free(0)), pfull0 = leader_addr(p_full(0)), pfull1 = leader_addr(p_full(1));
        softmax_warps<HD, WIN>(a, tl, h, kt0, nt, tmem, warp, lane, abort, s_full,
                               [&](int b) { arrive_cluster(sfree0 + 8u * (uint32_t)b); },
                               [&](int b) { arrive_cluster(b ? pfull1 : pfull0); }, pv_done);
    }
    tc_fence_before();
    __syncthreads();
    // the odd CTA's loads complete only on the even CTA's barriers: before
    // either CTA leaves, the even CTA waits for every load still in flight
    if (rank != 0 && threadIdx.x == 0) {
        dsmem_st_u32(dsmem(&s_peer[0], 0), (uint32_t)(s_issued[0] > early ? s_issued[0] : early));
        dsmem_st_u32(dsmem(&s_peer[1], 0), (uint32_t)(s_issued[1] > early ? s_issued[1] : early));
        dsmem_st_u32(dsmem(&s_peer[2], 0), (uint32_t)*abort);
    }
    cluster_sync();
    if (rank == 0 && threadIdx.x == 0 && (*abort || s_peer[2])) {
        for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(q_full, 0); ++i) {
        }
        drain_ring(k_full(0), s_issued[0] > early ? s_issued[0] : early, s_peer[0], C::KST, KB);
        drain_ring(v_full(0), s_issued[1] > early ? s_issued[1] : early, s_peer[1], C::VST, VB);
    }
    cluster_sync();                           // neither CTA leaves while the pair still uses its memory
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace

bool attn_prefill_tc_ok(int head_dim, bool fp8_cache) { return !fp8_cache && (head_dim == 64 || head_dim == 128); }

cudaError_t launch_attn_prefill_tc(const AttnPrefillTcArgs &a, const TmaMap &mQ, const TmaMap &mK, const TmaMap &mV,
                                   const Launch &l) {
    if (a.n_tiles < 1) return cudaSuccess;
    if (a.Hkv < 1 || a.H % a.Hkv || !attn_prefill_tc_ok(a.head_dim, false)) return cudaErrorInvalidValue;
    const dim3 grid(a.n_tiles, a.H);
    const CUtensorMap &q = *reinterpret_cast<const CUtensorMap *>(&mQ);
    const CUtensorMap &k = *reinterpret_cast<const CUtensorMap *>(&mK);
    const CUtensorMap &v = *reinterpret_cast<const CUtensorMap *>(&mV);
    const bool win = a.window > 0;
    if (a.head_dim == 128)
        return launch_kernel(win ? attn_prefill_tc_kernel<128, true> : attn_prefill_tc_kernel<128, false>, grid,
                             dim3(FA_THREADS), FaCfg<128>::SMEM, l, q, k, v, a);
    return launch_kernel(win ? attn_prefill_tc_kernel<64, true> : attn_prefill_tc_kernel<64, false>, grid,
                         dim3(FA_THREADS), FaCfg<64>::SMEM, l, q, k, v, a);
}

bool attn_prefill_pair_ok(int head_dim, int H, int Hkv, bool fp8_cache) {
    return !fp8_cache && head_dim == 128 && Hkv > 0 && H % Hkv == 0 && (H / Hkv) % 2 == 0;
}

cudaError_t launch_attn_prefill_pair(const AttnPrefillTcArgs &a, const TmaMap &mQ, const TmaMap &mK64,
                                     const TmaMap &mV, const Launch &l) {
    if (a.n_tiles < 1) return cudaSuccess;
    if (!attn_prefill_pair_ok(a.head_dim, a.H, a.Hkv, false)) return cudaErrorInvalidValue;
    const dim3 grid(2 * a.n_tiles, a.H / 2);
    const CUtensorMap &q = *reinterpret_cast<const CUtensorMap *>(&mQ);
    const CUtensorMap &k = *reinterpret_cast<const CUtensorMap *>(&mK64);
    const CUtensorMap &v = *reinterpret_cast<const CUtensorMap *>(&mV);
    return launch_kernel(a.window > 0 ? attn_prefill_pair_kernel<128, true> : attn_prefill_pair_kernel<128, false>,
                         grid, dim3(FA_THREADS), FaPairCfg<128>::SMEM, l, q, k, v, a);
}

cudaError_t init_attn_prefill_tc_attributes() {
    cudaError_t e = allow_smem(attn_prefill_tc_kernel<128, false>, FaCfg<128>::SMEM);
    if (!e) e = allow_smem(attn_prefill_tc_kernel<128, true>, FaCfg<128>::SMEM);
    if (!e) e = allow_smem(attn_prefill_tc_kernel<64, false>, FaCfg<64>::SMEM);
    if (!e) e = allow_smem(attn_prefill_tc_kernel<64, true>, FaCfg<64>::SMEM);
    if (!e) e = allow_smem(attn_prefill_pair_kernel<128, false>, FaPairCfg<128>::SMEM);
    if (!e) e = allow_smem(attn_prefill_pair_kernel<128, true>, FaPairCfg<128>::SMEM);
    return e;
}

}  // namespace llm
