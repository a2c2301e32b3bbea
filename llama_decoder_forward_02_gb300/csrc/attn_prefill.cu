// Prefill attention: causal grouped-query attention of a ubatch's rows
// against their sequences' KV cache, tiled over keys with an online softmax
// ("Inside the inference engine: model architectures and forward pass",
// sections "Detailed explanation: Llama's forward pass in Go" and "KV Cache:
// memory for causal attention"; "LLama.cpp — how it works", "KV-cache and the
// Prefill / Decode stages": prefill writes K, V of every prompt position and
// each position attends to those at or before it).
//
// A CTA takes 64 query rows of one sequence (consecutive positions pos0 ..)
// and one query head; 4 warps own 16 rows each.  K and V tiles of 64 keys are
// double-buffered in XOR-swizzled shared memory with cp.async; S = Q K^T and
// O += P V run on mma.sync m16n8k16 (f16 in, fp32 accumulate).  The mask
// keeps key c for the row at position p iff c <= p; K/V of the ubatch itself
// were appended to the cache by the QKV epilogue beforehand.
#include "attn_tile.cuh"
#include "common.cuh"
#include "launch.cuh"

namespace llm {

namespace {

constexpr int BQ = 64, BKEY = 64, THREADS = 128;

template <int HD>
__device__ __forceinline__ void load_tile(f16 *dst, const f16 *src, int rows_valid, int tid) {
    load_rows<HD, BKEY, THREADS>(dst, src, rows_valid, tid);
}

template <int HD, bool F8, bool WIN>
__global__ void __launch_bounds__(THREADS) attn_prefill_kernel(const AttnPrefillArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    f16 *Qs = reinterpret_cast<f16 *>(smem_raw);
    f16 *Ks = Qs + BQ * HD;            // [2][BKEY][HD]
    f16 *Vs = Ks + 2 * BKEY * HD;      // [2][BKEY][HD]

    const AttnTile tl = a.tiles[blockIdx.x];
    const int h = blockIdx.y;
    const int H = a.H, Hkv = a.kv.n_kv_head, group = H / Hkv, j = h / group;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;

    pdl_wait();
    pdl_trigger();

    if (tl.seq < 0 || tl.seq >= a.kv.n_seq || tl.pos0 < 0 || tl.pos0 + tl.n_rows > a.kv.n_ctx) {
        if (tid == 0) raise_error(a.err, ERRF_BAD_INDEX);
        return;
    }
    const size_t cbase = (size_t)tl.seq * a.kv.seq_stride + (size_t)j * a.kv.n_ctx * HD;
    const f16 *Kg = a.kv.k + cbase;
    const f16 *Vg = a.kv.v + cbase;
    // FP8 E4M3 cache: rows are staged as bytes and widened to fp16 per tile
    constexpr bool f8 = F8;                 // the cache's element type is fixed per launch
    const uint8_t *Kg8 = f8 ? a.kv.k8 + cbase : nullptr;
    const uint8_t *Vg8 = f8 ? a.kv.v8 + cbase : nullptr;
    auto tile = [&](f16 *dK, f16 *dV, int row0, int rows_valid) {
        if (f8) {
            load_rows8<HD, BKEY, THREADS>(dK, Kg8 + (size_t)row0 * HD, rows_valid, tid);
            load_rows8<HD, BKEY, THREADS>(dV, Vg8 + (size_t)row0 * HD, rows_valid, tid);
        } else {
            load_tile<HD>(dK, Kg + (size_t)row0 * HD, rows_valid, tid);
            load_tile<HD>(dV, Vg + (size_t)row0 * HD, rows_valid, tid);
        }
    };
    const int n_keys = tl.pos0 + tl.n_rows;
    const int n_kt = (n_keys + BKEY - 1) / BKEY;
    // sliding window: the tiles before the first row's oldest visible key hold nothing visible
    const int W = WIN ? a.window : 0;       // the windowed variant is compiled apart
    const int kt0 = (W > 0 && tl.pos0 + 1 > W) ? (tl.pos0 + 1 - W) / BKEY : 0;

    // Q tile (rows past n_rows are zero)
    {
        constexpr int CH = HD / 8;
        const size_t ldq = (size_t)H * HD;
        for (int i = tid; i < BQ * CH; i += THREADS) {
            const int r = i / CH, c = i - r * CH;
            const bool pv = r < tl.n_rows;
            cp_async16(Qs + Swz<HD>::off(r, c), a.q + (size_t)(tl.row0 + (pv ? r : 0)) * ldq + h * HD + c * 8, pv);
        }
    }
    tile(Ks, Vs, kt0 * BKEY, n_keys - kt0 * BKEY);
    cp_async_commit();

    float o[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    const float sl2 = 1.4426950408889634f / sqrtf((float)HD);
    const int qp0 = tl.pos0 + warp * 16 + g;       // position of this thread's first row
    uint32_t qf[HD / 16][4];

    for (int kt = kt0; kt < n_kt; ++kt) {
        const int cur = (kt - kt0) & 1;
        if (kt + 1 < n_kt) {
            const int nb = (kt + 1) * BKEY;
            tile(Ks + (cur ^ 1) * BKEY * HD, Vs + (cur ^ 1) * BKEY * HD, nb, n_keys - nb);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (f8) {                           // widen the staged fp8 rows of tile kt
            convert_tile8<HD, BKEY, THREADS>(Ks + cur * BKEY * HD, tid);
            convert_tile8<HD, BKEY, THREADS>(Vs + cur * BKEY * HD, tid);
        }
        if (kt == kt0) {
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = kk * 2 + (lane >> 4);
                ldmatrix_x4(qf[kk], smem_u32(Qs + Swz<HD>::off(r, c)));
            }
        }
        const f16 *Kt = Ks + cur * BKEY * HD;
        const f16 *Vt = Vs + cur * BKEY * HD;

        // S = Q K^T for 16 rows x 64 keys
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {   // pairs of 8-key tiles
                uint32_t kf[4];
                const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = kk * 2 + ((lane >> 3) & 1);
                ldmatrix_x4(kf, smem_u32(Kt + Swz<HD>::off(r, c)));
                const uint32_t b0[2] = {kf[0], kf[1]}, b1[2] = {kf[2], kf[3]};
                mma_f16_16816(s[2 * np], qf[kk], b0);
                mma_f16_16816(s[2 * np + 1], qf[kk], b1);
            }
        }
        // mask + online softmax (rows qp0 and qp0 + 8)
        const int key0 = kt * BKEY;
        const bool need_mask = key0 + BKEY - 1 > tl.pos0 + warp * 16 || WIN;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + nt * 8 + 2 * t4 + (e & 1);
                const int qp = qp0 + (e >> 1) * 8;
                float v = s[nt][e] * sl2;
                if (need_mask && (key > qp || (WIN && qp - key >= W))) v = -INFINITY;
                s[nt][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
        }
        float corr[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            const float mn = fmaxf(mrow[r], mx[r]);
            corr[r] = (mn == -INFINITY) ? 1.f : exp2f(mrow[r] - mn);
            mrow[r] = mn;
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mr = mrow[e >> 1];
                const float p = (mr == -INFINITY) ? 0.f : exp2f(s[nt][e] - mr);
                s[nt][e] = p;
                rs[e >> 1] += p;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
            rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
            lrow[r] = lrow[r] * corr[r] + rs[r];
        }
#pragma unroll
        for (int dt = 0; dt < HD / 8; ++dt) {
            o[dt][0] *= corr[0]; o[dt][1] *= corr[0];
            o[dt][2] *= corr[1]; o[dt][3] *= corr[1];
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < BKEY / 16; ++kk) {
            const uint32_t pa[4] = {pack_h2(s[2 * kk][0], s[2 * kk][1]), pack_h2(s[2 * kk][2], s[2 * kk][3]),
                                    pack_h2(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                                    pack_h2(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
            for (int dp = 0; dp < HD / 16; ++dp) {
                uint32_t vf[4];
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = dp * 2 + (lane >> 4);
                ldmatrix_x4_trans(vf, smem_u32(Vt + Swz<HD>::off(r, c)));
                const uint32_t b0[2] = {vf[0], vf[1]}, b1[2] = {vf[2], vf[3]};
                mma_f16_16816(o[2 * dp], pa, b0);
                mma_f16_16816(o[2 * dp + 1], pa, b1);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // normalise and store
    const size_t ldo = (size_t)H * HD;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = warp * 16 + g + r * 8;
        if (row >= tl.n_rows) continue;
        const float inv = lrow[r] > 0.f ? 1.f / lrow[r] : 0.f;
        f16 *dst = a.o + (size_t)(tl.row0 + row) * ldo + h * HD;
#pragma unroll
        for (int dt = 0; dt < HD / 8; ++dt) {
            const int d = dt * 8 + 2 * t4;
            *reinterpret_cast<uint32_t *>(dst + d) = pack_h2(o[dt][2 * r] * inv, o[dt][2 * r + 1] * inv);
        }
    }
}

template <int HD>
constexpr size_t smem_bytes() { return (size_t)(BQ + 4 * BKEY) * HD * sizeof(f16); }

}  // namespace

cudaError_t launch_attn_prefill(const AttnPrefillArgs &a, const Launch &l) {
    if (a.n_tiles < 1) return cudaSuccess;
    const dim3 grid(a.n_tiles, a.H);
    const bool f8 = a.kv.k8 != nullptr, win = a.window > 0;
#define PRE_CASE(HDV)                                                                                   \
    if (a.kv.head_dim == HDV) {                                                                         \
        auto k = f8 ? (win ? attn_prefill_kernel<HDV, true, true> : attn_prefill_kernel<HDV, true, false>) \
                    : (win ? attn_prefill_kernel<HDV, false, true> : attn_prefill_kernel<HDV, false, false>); \
        return launch_kernel(k, grid, dim3(THREADS), smem_bytes<HDV>(), l, a);                           \
    }
    PRE_CASE(32) PRE_CASE(64) PRE_CASE(128)
#undef PRE_CASE
    return cudaErrorInvalidValue;
}

cudaError_t init_attn_prefill_attributes() {
    cudaError_t e = cudaSuccess;
#define PRE_ATTR(HDV)                                                                       \
    if (!e) e = allow_smem(attn_prefill_kernel<HDV, false, false>, smem_bytes<HDV>());       \
    if (!e) e = allow_smem(attn_prefill_kernel<HDV, false, true>, smem_bytes<HDV>());        \
    if (!e) e = allow_smem(attn_prefill_kernel<HDV, true, false>, smem_bytes<HDV>());        \
    if (!e) e = allow_smem(attn_prefill_kernel<HDV, true, true>, smem_bytes<HDV>());
    PRE_ATTR(32) PRE_ATTR(64) PRE_ATTR(128)
#undef PRE_ATTR
    return e;
}

}  // namespace llm
