// Prefill GEMM on CTA pairs (tcgen05 cta_group::2): C[m][n] = sum_k A[m][k] W[n][k]
// with the same fused epilogues as the one-CTA kernel ("Inside the inference
// engine: model architectures and forward pass", section "Detailed
// explanation: Llama's forward pass in Go").
//
// A cluster of two CTAs computes a 256 x BN tile with M = 256 MMAs issued by
// the even CTA (the leader).  Each CTA stages its own 128 rows of A and its
// own BN/2 rows of W, so an SM's shared memory carries half the weight bytes
// of a one-CTA 128 x BN tile for the same accumulator: the one-CTA MMA is
// bounded by shared-memory bandwidth, the pair much less so.  Each CTA's
// tensor memory receives its 128 accumulator rows x BN columns.
//
//   warp 0, one lane, both CTAs: TMA producer into the CTA's own ring
//     (weight boxes of the first stages before the dependency wait); the odd
//     CTA's loads complete on the leader's "full" mbarrier of the stage, which
//     the leader arms with the bytes of both.
//   warp 1, one lane, leader: waits for a stage, issues its M = 256 MMAs and
//     commits the stage's "empty" mbarrier in both CTAs (multicast), finally
//     the accumulator mbarrier of both.
//   all eight warps of both CTAs: epilogue of the CTA's 128 rows.
// A residual GEMM with a long K can run with K split in two over two sets of
// pairs (blockIdx.z), which exchange their partial accumulators through L2
// (GemmArgs::split_k).
// Every wait is bounded (ERRF_WAIT_TIMEOUT, then the CTA winds down).
#include <cuda.h>

#include "common.cuh"
#include "launch.cuh"
#include "tma.cuh"
#include "cluster.cuh"
#include "gemm_tc_common.cuh"

namespace llm {

namespace {

using namespace tcg;

template <int BN, int KS_ = 2>
struct Cfg2 {
    static constexpr int BNH = BN / 2;                          // weight rows staged per CTA
    static constexpr int KS = KS_;                              // 64-deep K blocks per stage
    static constexpr uint32_t A_SUB = BM * BK * 2;              // one 128 x 64 box of A
    static constexpr uint32_t B_SUB = BNH * BK * 2;             // one BN/2 x 64 box of W
    static constexpr uint32_t STAGE_BYTES = KS * (A_SUB + B_SUB);
    // as many stages as fit beside ~1.5 KB of barriers and the static
    // variables (192-wide tiles: 4 x 56 KB, which hides the latency of weights
    // coming from DRAM: 3 stages cost the QKV GEMM ~3 us)
    static constexpr int STAGES = (224 * 1024) / STAGE_BYTES > 12 ? 12 : (224 * 1024) / STAGE_BYTES;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 512;
    static constexpr uint32_t TMEM_COLS = BN <= 128 ? 128 : 256;
    // kind::f16 instruction descriptor: D fp32, A/B fp16 K-major, N >> 3 at
    // bit 17, M >> 4 at bit 24 with M = 256 (the pair's rows)
    static constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
};

__device__ __forceinline__ void mma_pair(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}"
        :: "r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(accum) : "memory");
}
// TMA load into this CTA's shared memory that completes its bytes on an
// mbarrier of either CTA of the pair (the odd CTA's loads count on the
// leader's barrier, so the MMA issuer waits on one barrier per stage)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t cluster_bar, int x,
                                                 int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(x), "r"(y) : "memory");
}
// arrive once on the mbarrier at this shared offset in both CTAs of the pair
// when the MMAs issued so far are complete
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        :: "r"(bar), "h"((uint16_t)3) : "memory");
}
// Arrive on a barrier of the other CTA.  Waits on every barrier stay at the
// default CTA scope: cluster-scope acquire / release in the spin loops slowed
// the pair's TMA streams about fourfold.
__device__ __forceinline__ void remote_arrive(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" :: "r"(cluster_bar) : "memory");
}

constexpr int PAIR_THREADS = 256;     // warp 0 TMA, warp 1 MMA (leader); all 8 warps drain the tile

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// After an abort: wait (bounded) until every stage either CTA of the pair
// issued has landed on the leader's full barriers.  `mine` / `peer`: stages
// the leader / the odd CTA issued (each at most STAGES ahead of the MMAs).
// A stage only the odd CTA issued gets the leader's arrival with the odd
// CTA's bytes, so that its phase can complete.
template <typename Bytes>
__device__ void drain_pair_loads(uint32_t full0, int mine, int peer, int stages, Bytes bytes) {
    const int hi = mine > peer ? mine : peer;
    for (int kb = (hi > stages ? hi - stages : 0); kb < hi; ++kb) {
        const uint32_t bar = full0 + 8u * (uint32_t)(kb % stages);
        if (kb >= mine) mbar_expect_tx(bar, bytes(kb));
        for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(bar, (kb / stages) & 1); ++i) {
        }
    }
}

// The residual epilogue through shared memory (EPI_RESID with a.tma_epi): the
// CTA's 128 x BN tile of h (fp32, boxes of 32 columns, 128-byte swizzle) is
// read by TMA into the first two ring slots the last MMAs free, so it has
// landed when the accumulator is ready; h + y and f16((h + y) * gain) are
// written in place and into a third slot (boxes of 64 columns) and go back by
// TMA stores.  Rows past M are computed on whatever the workspace holds there
// and stored back into it (the workspaces have n_ubatch rows; nothing reads
// them).
constexpr uint32_t EPI_BOX = 128 * 128;      // one 128-row x 128-byte box

template <int BN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PAIR_THREADS, 1)
gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmX, const GemmArgs a) {
    using C = Cfg2<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ int s_abort;
    __shared__ uint32_t s_tmem;
    __shared__ int s_peer[2];                 // (leader) the odd CTA's issued stages and abort flag
    __shared__ float s_scale[BM];             // the RMSNorm scale of each of this CTA's rows
    __shared__ int s_h_armed;                 // the residual tile's loads were issued

    // the layout is identical in both CTAs: the leader's descriptors address
    // the same offsets in its peer
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bar0 = base + C::STAGES * C::STAGE_BYTES;    // full[S], empty[S], accum, hfull
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    const uint32_t accum = bar0 + 8u * (2 * C::STAGES);
    const uint32_t hfull = bar0 + 8u * (2 * C::STAGES + 1);
    // a stage holds KS 64-deep blocks: [A block 0][A block 1][W block 0][W block 1]
    auto a_smem = [&](int s, int j) { return base + s * C::STAGE_BYTES + j * C::A_SUB; };
    auto b_smem = [&](int s, int j) { return base + s * C::STAGE_BYTES + C::KS * C::A_SUB + j * C::B_SUB; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int m0 = (blockIdx.x >> 1) * (2 * BM) + (int)rank * BM;   // this CTA's rows
    const int n0 = blockIdx.y * BN;                                  // the pair's columns
    const int nb0 = n0 + (int)rank * C::BNH;                         // weight rows this CTA stages
    // K split in two (a.split_k): this pair's half of the whole stages
    const bool split = EPI == EPI_RESID && a.split_k;
    const int khalf = split ? (int)blockIdx.z : 0;
    const int nk64_all = a.K / BK, h64 = split ? (nk64_all / C::KS / 2) * C::KS : nk64_all;
    const int k64_0 = khalf ? h64 : 0, nk64 = khalf ? nk64_all - h64 : h64;
    const int nk = (nk64 + C::KS - 1) / C::KS;                       // stages
    auto nsub = [&](int st) { return nk64 - st * C::KS < C::KS ? nk64 - st * C::KS : C::KS; };
    auto bytes = [&](int st) { return (uint32_t)nsub(st) * (C::A_SUB + C::B_SUB); };
    volatile int *abort = &s_abort;
    const bool tma_epi = EPI == EPI_RESID && a.tma_epi;
    const int cta_idx = blockIdx.y * gridDim.x + blockIdx.x;        // this CTA's tile (both halves)
    // the 32-column chunks of the tile this CTA finishes: all of them, or with
    // K split the half khalf, [cz, cz + nch)
    constexpr int NC = BN / 32, HHALF = (NC + 1) / 2;               // residual boxes (32 columns), per ring slot
    const int nch = split ? NC / 2 : NC, cz = split ? khalf * (NC / 2) : 0;
    auto slot = [&](int s) { return base + (uint32_t)s * C::STAGE_BYTES; };
    auto h_box = [&](int b) {
        const int l = b - cz;
        return slot((nk + (l < HHALF ? 0 : 1)) % C::STAGES) + (uint32_t)(l % HHALF) * EPI_BOX;
    };
    const uint32_t x_slot = slot((nk + 2) % C::STAGES);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full(s), 1);            // (leader) both CTAs' bytes of the stage
            mbar_init(empty(s), 1);
        }
        mbar_init(accum, 1);
        mbar_init(hfull, 1);
        s_abort = 0;
        s_h_armed = 0;
        s_peer[0] = s_peer[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {                          // both CTAs allocate the pair's columns together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&s_tmem)), "r"(C::TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();                           // barriers initialised and TMEM allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // every load of both CTAs completes on the leader's full barrier of its
    // stage, which the leader arms with the bytes of both
    uint32_t full0;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(full0) : "r"(full(0)), "r"(0u));
    auto fullc = [&](int s) { return full0 + 8u * s; };
    auto load_b = [&](int kb, int s) {
        if (rank == 0) mbar_expect_tx(full(s), 2 * bytes(kb));
        for (int j = 0; j < nsub(kb); ++j) tma_load_2d_pair(b_smem(s, j), &tmB, fullc(s), (k64_0 + kb * C::KS + j) * BK, nb0);
    };
    const int pre = nk < C::STAGES ? nk : C::STAGES;
    int issued = 0;
    if (warp == 0 && lane == 0) {
        for (int kb = 0; kb < pre; ++kb) load_b(kb, kb);    // weights do not depend on the previous kernel
    }
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % C::STAGES;
                if (kb >= pre) {
                    if (!mbar_wait(empty(s), ((kb / C::STAGES) & 1) ^ 1, abort, a.err)) break;
                    load_b(kb, s);
                }
                for (int j = 0; j < nsub(kb); ++j)
                    tma_load_2d_pair(a_smem(s, j), &tmA, fullc(s), (k64_0 + kb * C::KS + j) * BK, m0);
                issued = kb + 1;
            }
            if (tma_epi && issued == nk) {
                // this CTA's residual tile (its half with K split) into the ring
                // slots of stages nk (and nk + 1), each taken once the MMAs have
                // read the stage it held
                mbar_expect_tx(hfull, nch * EPI_BOX);
                s_h_armed = 1;
                for (int v = nk; v < nk + (nch + HHALF - 1) / HHALF; ++v) {
                    const int sl = v % C::STAGES;
                    if (v >= C::STAGES && !mbar_wait(empty(sl), ((v / C::STAGES) & 1) ^ 1, abort, a.err)) break;
                    for (int l = (v - nk) * HHALF; l < nch && l < (v - nk + 1) * HHALF; ++l)
                        tma_load_2d(h_box(cz + l), &tmH, hfull, n0 + (cz + l) * 32, m0);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            if (rank == 0) {
                for (int kb = 0; kb < nk; ++kb) {
                    const int s = kb % C::STAGES;
                    const uint32_t ph = (kb / C::STAGES) & 1;
                    if (!mbar_wait(full(s), ph, abort, a.err)) break;
                    tc_fence_after();
                    for (int j = 0; j < nsub(kb); ++j) {
                        const uint64_t ad = sdesc(a_smem(s, j)), bd = sdesc(b_smem(s, j));
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_pair(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), C::IDESC, (kb | j | k) != 0);
                    }
                    commit_pair(empty(s));
                }
                commit_pair(accum);           // fires in both CTAs once the issued MMAs are complete
            }
        }
        __syncwarp();
    }

    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. (its accumulator
    // rows) and the half w / 4 of the tile's 32-column chunks
    const int q = warp & 3, hf = warp >> 2;
    const int row = m0 + q * 32 + lane;
    if (warp >= 4) row_norm_scales(a, m0, s_scale, warp - 4, 4, lane);   // during the MMAs
    mbar_wait(accum, 0, abort, a.err);
    // K split: park the partner's half of the columns of this CTA's
    // accumulator (column-major: a warp's 32 rows of one column are one
    // 128-byte run), publish it, and wait for the partner's parked half of
    // this CTA's columns
    const float *peer = split ? a.part + ((size_t)cta_idx * 2 + (1 - khalf)) * BM * (BN / 2) + q * 32 + lane : nullptr;
    if (split && !*abort) {
        float *park = a.part + ((size_t)cta_idx * 2 + khalf) * BM * (BN / 2) + q * 32 + lane;
        const int co = (1 - khalf) * (NC / 2);
        tc_fence_after();
#pragma unroll 1
        for (int l = hf * (NC / 4); l < (hf + 1) * (NC / 4); ++l) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((co + l) * 32), r);
#pragma unroll
            for (int i = 0; i < 32; ++i) __stcg(park + (size_t)(l * 32 + i) * BM, __uint_as_float(r[i]));
        }
        __threadfence();
    }
    if (tma_epi) mbar_wait(hfull, 0, abort, a.err);
    __syncthreads();
    if (split && threadIdx.x == 0 && !*abort) {
        st_release_u32(a.flags + cta_idx * 2 + khalf, a.epoch);
        uint32_t i = 0;
        while (ld_acquire_u32(a.flags + cta_idx * 2 + (1 - khalf)) != a.epoch && i < WAIT_LIMIT) ++i;
        if (i == WAIT_LIMIT) {
            raise_error(a.err, ERRF_WAIT_TIMEOUT);
            *abort = 1;
        }
    }
    __syncthreads();
    const bool ok = !*abort;
    tc_fence_after();
    if (ok && tma_epi) {
        const int rl = q * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
        for (int c = cz + hf * nch / 2; c < cz + (hf + 1) * nch / 2; ++c) {
            uint32_t r[32];
            float pv[32];
            if (split) {
#pragma unroll
                for (int i = 0; i < 32; ++i) pv[i] = __ldcg(peer + (size_t)((c - cz) * 32 + i) * BM);
            }
            tmem_ld32(trow + (uint32_t)(c * 32), r);
            if (split) {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + pv[i]);
            }
            const uint32_t hrow = h_box(c) + (uint32_t)rl * 128;
            float v[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t ad = hrow + ((uint32_t)(j ^ (rl & 7)) << 4);
                float4 hv;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(hv.x), "=f"(hv.y), "=f"(hv.z), "=f"(hv.w) : "r"(ad));
                v[4 * j] = hv.x + __uint_as_float(r[4 * j]);
                v[4 * j + 1] = hv.y + __uint_as_float(r[4 * j + 1]);
                v[4 * j + 2] = hv.z + __uint_as_float(r[4 * j + 2]);
                v[4 * j + 3] = hv.w + __uint_as_float(r[4 * j + 3]);
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                             :: "r"(ad), "f"(v[4 * j]), "f"(v[4 * j + 1]), "f"(v[4 * j + 2]), "f"(v[4 * j + 3]) : "memory");
            }
            if (a.x_next) {
                // the next RMSNorm's input, gain applied, and this 32-column share of sum(h^2)
                const float4 *g4 = reinterpret_cast<const float4 *>(a.gain_next + n0 + c * 32);
                const uint32_t xrow = x_slot + (uint32_t)((c - cz) >> 1) * EPI_BOX + (uint32_t)rl * 128;
                bool bad = false;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float4 ga = g4[2 * jj], gb = g4[2 * jj + 1];
                    float xs[8] = {v[8 * jj] * ga.x, v[8 * jj + 1] * ga.y, v[8 * jj + 2] * ga.z, v[8 * jj + 3] * ga.w,
                                   v[8 * jj + 4] * gb.x, v[8 * jj + 5] * gb.y, v[8 * jj + 6] * gb.z, v[8 * jj + 7] * gb.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) bad |= f16_bad(xs[i]);
                    const uint32_t p0 = pack_h2(xs[0], xs[1]), p1 = pack_h2(xs[2], xs[3]);
                    const uint32_t p2 = pack_h2(xs[4], xs[5]), p3 = pack_h2(xs[6], xs[7]);
                    const uint32_t ad = xrow + ((uint32_t)(((c & 1) * 4 + jj) ^ (rl & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(ad), "r"(p0), "r"(p1), "r"(p2), "r"(p3)
                                 : "memory");
                }
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) ss += v[i] * v[i];
                if (row < a.M) {
                    a.ss_next[(size_t)row * (a.N / 32) + (n0 / 32 + c)] = ss;
                    if (bad) raise_error(a.err, ERRF_F16_RANGE);
                }
            }
        }
        fence_proxy_async();                  // the tiles, visible to the TMA stores
    } else if (ok) {
        epilogue_chunks<EPI>(a, row, n0, tmem + ((uint32_t)(q * 32) << 16), hf * BN / 64, (hf + 1) * BN / 64,
                             s_scale[q * 32 + lane]);
    }
    tc_fence_before();
    __syncthreads();
    if (ok && tma_epi && threadIdx.x == 0) {
        for (int b = cz; b < cz + nch; ++b) tma_store_2d(&tmH, h_box(b), n0 + b * 32, m0);
        if (a.x_next)
            for (int b = cz / 2; b < (cz + nch) / 2; ++b)
                tma_store_2d(&tmX, x_slot + (uint32_t)(b - cz / 2) * EPI_BOX, n0 + b * 64, m0);
        bulk_commit();
        bulk_wait_all();                      // written before the CTA (and its shared memory) goes
    }
    if (!ok && s_h_armed && threadIdx.x == 0)
        for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(hfull, 0); ++i) {
        }
    // the odd CTA's loads complete only on the leader's barriers: before
    // either CTA leaves, the leader waits for every load still in flight
    if (rank != 0 && warp == 0 && lane == 0) {
        dsmem_st_u32(dsmem(&s_peer[0], 0), (uint32_t)issued);
        dsmem_st_u32(dsmem(&s_peer[1], 0), (uint32_t)*abort);
    }
    cluster_sync();
    if (rank == 0 && warp == 0 && lane == 0 && (*abort || s_peer[1])) drain_pair_loads(full(0), issued, s_peer[0], C::STAGES, [&](int kb) { return bytes(kb); });
    cluster_sync();                           // neither CTA leaves while the pair still uses its memory
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(C::TMEM_COLS) : "memory");
    }
}


// ---------------------------------------------------------------- persistent CTA pairs
// The same 256 x BN pair tiles, but a cluster loops over tiles t = pair,
// pair + n_pairs, ... (the two M tiles of one weight tile first, so that
// weight tile is read from HBM once).  The TMA ring and the MMA stream run on
// across tile boundaries; the accumulator is double-buffered in tensor memory
// (2 x BN columns) so eight dedicated epilogue warps drain tile i while the
// MMAs of tile i + 1 run.  Warps: 0 TMA producer (both CTAs), 1 MMA issuer
// (leader), 2-9 epilogue (warp w reads TMEM lanes 32 (w % 4) .. +31 and half
// (w - 2) / 4 of the columns).  Each epilogue warp of both CTAs arrives on
// the leader's "accumulator empty" barrier of the buffer it drained.
constexpr int PTHREADS = 320;         // warp 0 TMA, warp 1 MMA (leader), warps 2-9 epilogue

// 64-deep stages: twice as many in the same shared memory, so more of the
// ring is in flight while the MMAs hold one stage
constexpr int PKS = 1;

template <int BN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PTHREADS, 1)
gemm_pair_persist_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const GemmArgs a, int n_mt, int n_nt) {
    using C = Cfg2<BN, PKS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ int s_abort;
    __shared__ uint32_t s_tmem;
    __shared__ int s_peer[2];                 // (leader) the odd CTA's issued stages and abort flag
    __shared__ float s_scale[BM];             // the RMSNorm scales of this CTA's rows in the current tile

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bar0 = base + C::STAGES * C::STAGE_BYTES;    // full[S], empty[S], afull[2], aempty[2]
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto afull = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
    auto aempty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 + b); };
    auto a_smem = [&](int s, int j) { return base + s * C::STAGE_BYTES + j * C::A_SUB; };
    auto b_smem = [&](int s, int j) { return base + s * C::STAGE_BYTES + C::KS * C::A_SUB + j * C::B_SUB; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1, n_tiles = n_mt * n_nt;
    const int nk64 = a.K / BK;
    const int nk = (nk64 + C::KS - 1) / C::KS;
    auto nsub = [&](int st) { return nk64 - st * C::KS < C::KS ? nk64 - st * C::KS : C::KS; };
    auto bytes = [&](int st) { return (uint32_t)nsub(st) * (C::A_SUB + C::B_SUB); };
    volatile int *abort = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full(s), 1);                 // (leader) both CTAs' bytes of the stage
            mbar_init(empty(s), 1);
        }
        s_peer[0] = s_peer[1] = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(afull(b), 1);
            mbar_init(aempty(b), 16);              // 8 epilogue warps in each CTA of the pair
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&s_tmem)), "r"(512u) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    pdl_wait();
    pdl_trigger();
    uint32_t full0;                           // the leader's full barriers, where both CTAs' loads complete
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(full0) : "r"(full(0)), "r"(0u));
    int issued = 0;

    if (warp == 0) {
        if (lane == 0) {
            int g = 0;
            bool go = true;
            for (int t = pair; go && t < n_tiles; t += n_pairs) {
                const int m0 = (t % n_mt) * (2 * BM) + (int)rank * BM, nb0 = (t / n_mt) * BN + (int)rank * C::BNH;
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = g % C::STAGES;
                    if (g >= C::STAGES && !mbar_wait(empty(s), ((g / C::STAGES) & 1) ^ 1, abort, a.err)) {
                        go = false;
                        break;
                    }
                    if (rank == 0) mbar_expect_tx(full(s), 2 * bytes(kb));
                    for (int j = 0; j < nsub(kb); ++j) {
                        tma_load_2d_pair(b_smem(s, j), &tmB, full0 + 8u * s, (kb * C::KS + j) * BK, nb0);
                        tma_load_2d_pair(a_smem(s, j), &tmA, full0 + 8u * s, (kb * C::KS + j) * BK, m0);
                    }
                    issued = g + 1;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int g = 0, it = 0;
            bool go = true;
            for (int t = pair; go && rank == 0 && t < n_tiles; t += n_pairs, ++it) {
                const int b = it & 1;
                if (it >= 2 && !mbar_wait(aempty(b), ((it >> 1) - 1) & 1, abort, a.err)) break;
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * BN);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = g % C::STAGES;
                    const uint32_t ph = (g / C::STAGES) & 1;
                    if (!mbar_wait(full(s), ph, abort, a.err)) {
                        go = false;
                        break;
                    }
                    tc_fence_after();
                    for (int j = 0; j < nsub(kb); ++j) {
                        const uint64_t ad = sdesc(a_smem(s, j)), bd = sdesc(b_smem(s, j));
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_pair(acc, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), C::IDESC, (kb | j | k) != 0);
                    }
                    commit_pair(empty(s));
                }
                if (!go) break;
                commit_pair(afull(b));                   // fires in both CTAs when the tile's MMAs are done
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue warps: drain buffer it & 1 of each tile; warp w takes
        // TMEM lanes 32 (w % 4) .. and half (w - 2) / 4 of the 32-column chunks
        const int q = warp & 3, hf = (warp - 2) >> 2;
        uint32_t leader_empty[2];
        for (int b = 0; b < 2; ++b)
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(leader_empty[b]) : "r"(aempty(b)), "r"(0u));
        // ok stays uniform over each warp and every epilogue warp runs every
        // iteration, so the named barrier (no time limit) is always reached
        // by all eight; after a timeout the iterations only pass it
        int it = 0;
        bool ok = true;
        for (int t = pair; t < n_tiles; t += n_pairs, ++it) {
            const int b = it & 1;
            const int row0 = (t % n_mt) * (2 * BM) + (int)rank * BM;
            const int n0 = (t / n_mt) * BN;
            // the tile's RMSNorm scales, by the eight warps together while its
            // MMAs run; every warp takes its row's scale before any rewrites
            // the buffer for the next tile (static shared memory has no room
            // for a second buffer beside the 192-wide ring)
            if (ok) row_norm_scales(a, row0, s_scale, warp - 2, 8, lane);
            named_sync(1, 8 * 32);
            const float scale = s_scale[q * 32 + lane];
            named_sync(1, 8 * 32);
            ok = __all_sync(0xffffffffu, ok && mbar_wait(afull(b), (it >> 1) & 1, abort, a.err));
            if (!ok) continue;
            tc_fence_after();
            epilogue_chunks<EPI>(a, row0 + q * 32 + lane, n0, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN),
                                 hf * BN / 64, (hf + 1) * BN / 64, scale);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) remote_arrive(leader_empty[b]);     // (the leader's own address when rank 0)
        }
    }
    tc_fence_before();
    __syncthreads();
    // the odd CTA's loads complete only on the leader's barriers: before
    // either CTA leaves, the leader waits for every load still in flight
    if (rank != 0 && warp == 0 && lane == 0) {
        dsmem_st_u32(dsmem(&s_peer[0], 0), (uint32_t)issued);
        dsmem_st_u32(dsmem(&s_peer[1], 0), (uint32_t)*abort);
    }
    cluster_sync();
    if (rank == 0 && warp == 0 && lane == 0 && (*abort || s_peer[1]))
        drain_pair_loads(full(0), issued, s_peer[0], C::STAGES, [&](int g) { return bytes(g % nk); });
    cluster_sync();                           // neither CTA leaves while the pair still uses its memory
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(512u) : "memory");
    }
}

// ---------------------------------------------------------------- stream-K CTA pairs
// The persistent pairs with the work split by K stages instead of by tiles.
// The pairs form groups of n_mt (one pair per 256-row M tile); a group's
// pairs walk the same weight tiles and K stages in step, each for its own M
// tile, so every weight stage is read from HBM once and shared through L2.
// The n_nt * nk (weight tile, k-stage) units (a stage is 128 K-columns) are
// cut into one contiguous range per group, so every pair gets the same
// number of MMAs whatever the tile count (an O projection of a 512-row
// ubatch has 32 256-wide tiles for 76 pairs).  A range is a run of segments
// (weight tile, k-stages [kb0, kb1)) in unit order: at most one leading
// segment that starts inside a tile, whole tiles, and at most one trailing
// segment that starts a tile.
//   * a segment that starts inside its tile (kb0 > 0) is a partial: the
//     epilogue warps park it in the pair's workspace slot (fp32 [128][BN] per
//     CTA) and publish the slot with the launch's epoch (release);
//   * a segment with kb0 == 0 owns its tile: when the tile continues in later
//     pairs (those pairs' leading segments), it waits (acquire, bounded) for
//     their slots, adds them in K order to its accumulator and applies the
//     fused epilogue.  Such a segment is always the last of its pair, and the
//     partials it waits for are the first work of the pairs after it, so the
//     wait is short and nothing waits on a waiter.
// The sum order depends only on the number of pairs, so results are the same
// from launch to launch.
struct SkRange {
    long long U;
    int P, nk;
    __device__ __forceinline__ long long start(int p) const { return (long long)p * U / P; }
};


template <int BN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PTHREADS, 1)
gemm_pair_sk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs a, int n_mt, int n_nt, float *ws, unsigned *flags, unsigned epoch) {
    using C = Cfg2<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ int s_abort;
    __shared__ uint32_t s_tmem;
    __shared__ int s_peer[2];                 // (leader) the odd CTA's issued stages and abort flag

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bar0 = base + C::STAGES * C::STAGE_BYTES;    // full[S], empty[S], afull[2], aempty[2]
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto afull = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
    auto aempty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 + b); };
    auto a_smem = [&](int s, int j) { return base + s * C::STAGE_BYTES + j * C::A_SUB; };
    auto b_smem = [&](int s, int j) { return base + s * C::STAGE_BYTES + C::KS * C::A_SUB + j * C::B_SUB; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1;
    const int grp = pair / n_mt, mt = pair - grp * n_mt;        // this pair's group and M tile
    const int nk64 = a.K / BK;
    const int nk = (nk64 + C::KS - 1) / C::KS;
    auto nsub = [&](int st) { return nk64 - st * C::KS < C::KS ? nk64 - st * C::KS : C::KS; };
    // every stage loads KS blocks (a block past K reads zeros), so that every
    // stage has the same byte count
    constexpr uint32_t BYTES = C::KS * (C::A_SUB + C::B_SUB);
    const SkRange R{(long long)n_nt * nk, (int)(gridDim.x >> 1) / n_mt, nk};
    const long long u_begin = R.start(grp), u_end = R.start(grp + 1);
    // walk this pair's segments: f(it, tile, kb0, kb1) returns false to stop
    auto segments = [&](auto &&f) {
        int it = 0;
        for (long long u = u_begin; u < u_end; ++it) {
            const int t = (int)(u / nk), kb0 = (int)(u - (long long)t * nk);
            const int kb1 = (int)min((long long)nk, kb0 + (u_end - u));
            if (!f(it, t, kb0, kb1)) return;
            u += kb1 - kb0;
        }
    };
    volatile int *abort = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full(s), 1);                 // (leader) both CTAs' bytes of the stage
            mbar_init(empty(s), 1);
        }
        s_peer[0] = s_peer[1] = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(afull(b), 1);
            mbar_init(aempty(b), 16);              // 8 epilogue warps in each CTA of the pair
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&s_tmem)), "r"(512u) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    pdl_wait();
    pdl_trigger();
    uint32_t full0;                           // the leader's full barriers, where both CTAs' loads complete
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(full0) : "r"(full(0)), "r"(0u));
    int issued = 0;

    if (warp == 0) {
        if (lane == 0) {
            int g = 0;
            segments([&](int, int t, int kb0, int kb1) {
                const int m0 = mt * (2 * BM) + (int)rank * BM, nb0 = t * BN + (int)rank * C::BNH;
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int s = g % C::STAGES;
                    if (g >= C::STAGES && !mbar_wait(empty(s), ((g / C::STAGES) & 1) ^ 1, abort, a.err)) return false;
                    if (rank == 0) mbar_expect_tx(full(s), 2 * BYTES);
                    for (int j = 0; j < C::KS; ++j) {
                        tma_load_2d_pair(b_smem(s, j), &tmB, full0 + 8u * s, (kb * C::KS + j) * BK, nb0);
                        tma_load_2d_pair(a_smem(s, j), &tmA, full0 + 8u * s, (kb * C::KS + j) * BK, m0);
                    }
                    issued = g + 1;
                }
                return true;
            });
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int g = 0;
            if (rank == 0) segments([&](int it, int, int kb0, int kb1) {
                const int b = it & 1;
                if (it >= 2 && !mbar_wait(aempty(b), ((it >> 1) - 1) & 1, abort, a.err)) return false;
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * BN);
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int s = g % C::STAGES;
                    const uint32_t ph = (g / C::STAGES) & 1;
                    if (!mbar_wait(full(s), ph, abort, a.err)) return false;
                    tc_fence_after();
                    for (int j = 0; j < nsub(kb); ++j) {
                        const uint64_t ad = sdesc(a_smem(s, j)), bd = sdesc(b_smem(s, j));
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_pair(acc, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), C::IDESC,
                                     (kb != kb0 || j || k) ? 1u : 0u);
                    }
                    commit_pair(empty(s));
                }
                commit_pair(afull(b));                   // fires in both CTAs when the segment's MMAs are done
                return true;
            });
        }
        __syncwarp();
    } else {
        // ---- epilogue warps: TMEM lanes 32 (w % 4) .., half (w - 2) / 4 of the chunks
        const int q = warp & 3, hf = (warp - 2) >> 2;
        constexpr int NC = BN / 32;
        const int rloc = q * 32 + lane;                      // row within this CTA's 128
        uint32_t leader_empty[2];
        for (int b = 0; b < 2; ++b)
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(leader_empty[b]) : "r"(aempty(b)), "r"(0u));
        // a pair's parked partial: column-major per CTA ([BN][128 rows]) so that a
        // warp's 32 rows of one column are one coalesced 128-byte access
        auto slot = [&](int p) { return ws + (size_t)(p * 2 + (int)rank) * BM * BN + rloc; };
        segments([&](int it, int t, int kb0, int kb1) {
            const int b = it & 1;
            if (!mbar_wait(afull(b), (it >> 1) & 1, abort, a.err)) return false;
            tc_fence_after();
            const int row = mt * (2 * BM) + (int)rank * BM + rloc;
            const int n0 = t * BN;
            const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN);
            if (kb0 > 0) {
                // a partial: park it, free the accumulator, publish the slot
                float *dst = slot(pair);
#pragma unroll 1
                for (int c = hf * NC / 2; c < (hf + 1) * NC / 2; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tacc + (uint32_t)(c * 32), r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) __stcg(dst + (size_t)(c * 32 + i) * BM, __uint_as_float(r[i]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) remote_arrive(leader_empty[b]);
                __threadfence();
                named_sync(1, 256);
                if (warp == 2 && lane == 0) st_release_u32(flags + pair * 2 + (int)rank, epoch);
                return true;
            }
            // owner of tile (mt, t): the groups after this one that hold the rest
            // of its K stages, each through its pair for the same M tile
            const long long t_end = (long long)(t + 1) * nk;
            int g_last = grp;
            if (kb1 < nk) {
                for (int gg = grp + 1; gg < R.P && R.start(gg) < t_end; ++gg) {
                    if (R.start(gg + 1) == R.start(gg)) continue;          // an empty range
                    g_last = gg;
                    const int p = gg * n_mt + mt;
                    uint32_t i = 0;
                    while (ld_acquire_u32(flags + p * 2 + (int)rank) != epoch && i < WAIT_LIMIT) ++i;
                    if (i == WAIT_LIMIT) {
                        raise_error(a.err, ERRF_WAIT_TIMEOUT);
                        *abort = 1;
                        return false;
                    }
                }
            }
            const float scale = row < a.M ? row_norm_scale(a, row) : 1.f;
#pragma unroll 1
            for (int c = hf * NC / 2; c < (hf + 1) * NC / 2; ++c) {
                uint32_t r[32];
                EpiSide sd;
                if (row < a.M) epi_fetch<EPI>(a, row, n0 + c * 32, sd);
                tmem_ld32(tacc + (uint32_t)(c * 32), r);
                for (int gg = grp + 1; gg <= g_last; ++gg) {
                    if (R.start(gg + 1) == R.start(gg)) continue;
                    const float *sp = slot(gg * n_mt + mt) + (size_t)c * 32 * BM;
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __ldcg(sp + (size_t)i * BM);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + v[i]);
                }
                if (row < a.M) epilogue32<EPI>(a, row, n0 + c * 32, r, scale, sd);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) remote_arrive(leader_empty[b]);
            return true;
        });
    }
    tc_fence_before();
    __syncthreads();
    // the odd CTA's loads complete only on the leader's barriers: before
    // either CTA leaves, the leader waits for every load still in flight
    if (rank != 0 && warp == 0 && lane == 0) {
        dsmem_st_u32(dsmem(&s_peer[0], 0), (uint32_t)issued);
        dsmem_st_u32(dsmem(&s_peer[1], 0), (uint32_t)*abort);
    }
    cluster_sync();
    if (rank == 0 && warp == 0 && lane == 0 && (*abort || s_peer[1]))
        drain_pair_loads(full(0), issued, s_peer[0], C::STAGES, [&](int) { return BYTES; });
    cluster_sync();                           // neither CTA leaves while the pair still uses its memory
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(512u) : "memory");
    }
}

}  // namespace

int gemm_pair_pick_bn(int M, int N, int max_clusters) {
    // Each SM's shared memory carries A (128 x 64) plus BN/2 x 64 of W per
    // stage, written once by TMA and read once by the MMA: per 16-deep K step
    // 8 KB + 32 * BN bytes against a BN-wide MMA, ~1.4x an SM's bandwidth at
    // BN 128 and ~0.9x at 256.  Pick the width with the smaller
    // waves x width / efficiency.
    static const int widths[3] = {128, 192, 256};
    static const double eff[3] = {0.70, 0.85, 0.90};
    const long long mp = (M + 2 * BM - 1) / (2 * BM);
    int best = 0;
    double best_cost = 0.0;
    for (int i = 0; i < 3; ++i) {
        if (N % widths[i]) continue;
        const long long tiles = mp * (N / widths[i]);
        const long long waves = (tiles + max_clusters - 1) / max_clusters;
        const double cost = (double)waves * widths[i] / eff[i];
        if (!best || cost < best_cost) { best = widths[i]; best_cost = cost; }
    }
    return best;
}

#define PAIR_CASE(BNV, E)                                                                             \
    if (bn == BNV && epi == E)                                                                        \
        return launch_kernel(gemm_pair_kernel<BNV, E>, grid, dim3(PAIR_THREADS), Cfg2<BNV>::SMEM, l2, \
                             *reinterpret_cast<const CUtensorMap *>(&mA), *reinterpret_cast<const CUtensorMap *>(&mB), \
                             *reinterpret_cast<const CUtensorMap *>(mh), *reinterpret_cast<const CUtensorMap *>(mx), g);

cudaError_t launch_gemm_pair(int epi, const GemmArgs &a, const TmaMap &mA, const TmaMap &mB, int bn,
                             const Launch &l, const TmaMap *mH, const TmaMap *mX) {
    // mA: boxes of 128 rows of A; mB: boxes of bn / 2 rows of W; mH, mX (EPI_RESID
    // through shared memory): hres fp32 in 128 x 32 boxes, x_next as an operand map
    if (a.M < 1 || a.K % BK || (bn != 128 && bn != 192 && bn != 256) || a.N % bn)
        return cudaErrorInvalidValue;
    GemmArgs g = a;
    g.tma_epi = epi == EPI_RESID && a.tma_epi && mH && (mX || !a.x_next) ? 1 : 0;
    const TmaMap *mh = g.tma_epi ? mH : &mA, *mx = g.tma_epi && mX ? mX : &mA;
    // split K: 256-wide residual tiles through shared memory only, with a
    // workspace and whole stages for both halves
    if (a.split_k && (epi != EPI_RESID || bn != 256 || !g.tma_epi || !a.part || !a.flags || a.K / BK < 8))
        return cudaErrorInvalidValue;
    const dim3 grid(2 * ((a.M + 2 * BM - 1) / (2 * BM)), a.N / bn, a.split_k ? 2 : 1);
    // the halves of a split wait on each other: a cooperative launch makes
    // every CTA resident at once even beside other streams' kernels
    Launch lc = l;
    if (a.split_k) lc.cooperative = true;
    const Launch &l2 = lc;
    PAIR_CASE(128, EPI_STORE) PAIR_CASE(128, EPI_RESID) PAIR_CASE(128, EPI_QKV) PAIR_CASE(128, EPI_SWIGLU)
    PAIR_CASE(192, EPI_STORE) PAIR_CASE(192, EPI_RESID) PAIR_CASE(192, EPI_QKV) PAIR_CASE(192, EPI_SWIGLU)
    PAIR_CASE(256, EPI_STORE) PAIR_CASE(256, EPI_RESID) PAIR_CASE(256, EPI_QKV) PAIR_CASE(256, EPI_SWIGLU)
    return cudaErrorInvalidValue;
}

int gemm_pair_max_clusters() {
    // pairs of this kernel that can be resident at once (clusters need both
    // SMs in one GPC), queried once per device
    constexpr int MAX_DEV = 64;
    static int n[MAX_DEV] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) {
        cudaGetLastError();
        dev = 0;
    }
    if (n[dev] <= 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(PAIR_THREADS);
        cfg.dynamicSmemBytes = Cfg2<256>::SMEM;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, gemm_pair_kernel<256, EPI_STORE>, &cfg) != cudaSuccess || c < 1) {
            cudaGetLastError();
            int sms = 0;
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            c = sms / 2;
        }
        n[dev] = c;
    }
    return n[dev];
}

#define PERSIST_CASE(BNV, E)                                                                          \
    if (bn == BNV && epi == E)                                                                        \
        return launch_kernel(gemm_pair_persist_kernel<BNV, E>, grid, dim3(PTHREADS), Cfg2<BNV, PKS>::SMEM, l, \
                             *reinterpret_cast<const CUtensorMap *>(&mA), *reinterpret_cast<const CUtensorMap *>(&mB), \
                             a, n_mt, n_nt);

cudaError_t launch_gemm_pair_persist(int epi, const GemmArgs &a, const TmaMap &mA, const TmaMap &mB, int bn,
                                     const Launch &l) {
    if (a.M < 1 || a.K % BK || (bn != 128 && bn != 192 && bn != 256) || a.N % bn)
        return cudaErrorInvalidValue;
    const int n_mt = (a.M + 2 * BM - 1) / (2 * BM), n_nt = a.N / bn;
    const int tiles = n_mt * n_nt, mc = gemm_pair_max_clusters();
    const dim3 grid(2 * (tiles < mc ? tiles : mc), 1, 1);
    PERSIST_CASE(128, EPI_STORE) PERSIST_CASE(128, EPI_RESID) PERSIST_CASE(128, EPI_QKV) PERSIST_CASE(128, EPI_SWIGLU)
    PERSIST_CASE(192, EPI_STORE) PERSIST_CASE(192, EPI_RESID) PERSIST_CASE(192, EPI_QKV) PERSIST_CASE(192, EPI_SWIGLU)
    PERSIST_CASE(256, EPI_STORE) PERSIST_CASE(256, EPI_RESID) PERSIST_CASE(256, EPI_QKV) PERSIST_CASE(256, EPI_SWIGLU)
    return cudaErrorInvalidValue;
}

int gemm_pair_sk_clusters(int M, int N, int K) {
    // groups of n_mt pairs (one per 256-row M tile), as many as fit at once
    // and no more than there are (weight tile, k-stage) units
    const int n_mt = (M + 2 * BM - 1) / (2 * BM);
    const long long units = (long long)(N / 256) * ((K / BK + 1) / 2);
    const int mc = gemm_pair_max_clusters();
    long long groups = mc / n_mt;
    if (groups > units) groups = units;
    return (int)(groups * n_mt);
}

size_t gemm_pair_sk_ws_floats(int max_clusters) { return (size_t)max_clusters * 2 * BM * 256; }

#define SK_CASE(E)                                                                                     \
    if (epi == E)                                                                                      \
        return launch_kernel(gemm_pair_sk_kernel<256, E>, grid, dim3(PTHREADS), Cfg2<256>::SMEM, l,       \
                             *reinterpret_cast<const CUtensorMap *>(&mA), *reinterpret_cast<const CUtensorMap *>(&mB), \
                             a, n_mt, n_nt, ws, flags, epoch);

cudaError_t launch_gemm_pair_sk(int epi, const GemmArgs &a, const TmaMap &mA, const TmaMap &mB, float *ws,
                                unsigned *flags, unsigned epoch, const Launch &l) {
    if (a.M < 1 || a.K % BK || a.N % 256 || !ws || !flags || epoch == 0) return cudaErrorInvalidValue;
    if (gemm_pair_sk_clusters(a.M, a.N, a.K) < 1) return cudaErrorInvalidValue;       // more M tiles than pairs
    const int n_mt = (a.M + 2 * BM - 1) / (2 * BM), n_nt = a.N / 256;
    const dim3 grid(2 * gemm_pair_sk_clusters(a.M, a.N, a.K), 1, 1);
    SK_CASE(EPI_STORE) SK_CASE(EPI_RESID) SK_CASE(EPI_QKV) SK_CASE(EPI_SWIGLU)
    return cudaErrorInvalidValue;
}

cudaError_t init_gemm_pair_attributes() {
    cudaError_t e = cudaSuccess;
#define PAIR_ATTR(BNV, E) if (!e) e = allow_smem(gemm_pair_kernel<BNV, E>, Cfg2<BNV>::SMEM);
    PAIR_ATTR(128, EPI_STORE) PAIR_ATTR(128, EPI_RESID) PAIR_ATTR(128, EPI_QKV) PAIR_ATTR(128, EPI_SWIGLU)
    PAIR_ATTR(192, EPI_STORE) PAIR_ATTR(192, EPI_RESID) PAIR_ATTR(192, EPI_QKV) PAIR_ATTR(192, EPI_SWIGLU)
    PAIR_ATTR(256, EPI_STORE) PAIR_ATTR(256, EPI_RESID) PAIR_ATTR(256, EPI_QKV) PAIR_ATTR(256, EPI_SWIGLU)
#undef PAIR_ATTR
#define PERSIST_ATTR(BNV, E) if (!e) e = allow_smem(gemm_pair_persist_kernel<BNV, E>, Cfg2<BNV, PKS>::SMEM);
    PERSIST_ATTR(128, EPI_STORE) PERSIST_ATTR(128, EPI_RESID) PERSIST_ATTR(128, EPI_QKV) PERSIST_ATTR(128, EPI_SWIGLU)
    PERSIST_ATTR(192, EPI_STORE) PERSIST_ATTR(192, EPI_RESID) PERSIST_ATTR(192, EPI_QKV) PERSIST_ATTR(192, EPI_SWIGLU)
    PERSIST_ATTR(256, EPI_STORE) PERSIST_ATTR(256, EPI_RESID) PERSIST_ATTR(256, EPI_QKV) PERSIST_ATTR(256, EPI_SWIGLU)
#undef PERSIST_ATTR
    if (!e) e = allow_smem(gemm_pair_sk_kernel<256, EPI_STORE>, Cfg2<256>::SMEM);
    if (!e) e = allow_smem(gemm_pair_sk_kernel<256, EPI_RESID>, Cfg2<256>::SMEM);
    if (!e) e = allow_smem(gemm_pair_sk_kernel<256, EPI_QKV>, Cfg2<256>::SMEM);
    if (!e) e = allow_smem(gemm_pair_sk_kernel<256, EPI_SWIGLU>, Cfg2<256>::SMEM);
    return e;
}

}  // namespace llm
