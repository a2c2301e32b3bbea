// One decode token at batch 1 as a single persistent kernel: embedding, every
// layer (RMSNorm -> QKV + RoPE + KV append -> attention over the cache -> O +
// residual -> RMSNorm -> gate/up + SiLU*up -> down + residual), final RMSNorm,
// output projection and greedy argmax ("Inside the inference engine: model
// architectures and forward pass", section "Detailed explanation: Llama's
// forward pass in Go"; "LLama.cpp — how it works", "KV-cache and the Prefill /
// Decode stages": one new token's Q, K, V, K and V appended, attention over
// the cache; "Token sampling pipeline": temperature 0 is argmax).
//
// Decode at batch 1 streams ~15 GB of weights per token; as ~160 separate
// kernels it loses several microseconds at every kernel boundary.  Here one
// CTA per SM (cooperative launch, so all are resident) runs the whole token:
//   - the producer warp walks a fixed schedule of every weight row this CTA
//     owns, in phase order, and streams it with 1-KB bulk copies into a
//     multi-stage shared-memory ring.  It never waits for the phase barriers,
//     so HBM keeps streaming the next matrix while the consumers synchronize;
//   - four consumer warps run the phases.  In a matrix phase the CTA owns a
//     contiguous, equal range of output rows (whole interleaved gate/up
//     groups, whole RoPE pairs), processes them 16 at a time with the K range
//     split across the warps (mma.sync, rows as the A operand, the input
//     vector as column 0 of B), reduces the warps in shared memory and applies
//     the fused epilogue itself: no cross-CTA reduction.  The attention phase
//     gives each CTA one (kv head, sequence split) item of the decode-attention
//     kernel's work;
//   - phases are separated by grid barriers (one counter, bounded spin); a
//     timeout anywhere raises ERRF_WAIT_TIMEOUT and a shared abort flag that
//     makes every CTA skip to the end.
// Norms: each residual phase leaves one partial sum of squares per CTA; the
// next phase sums the P partials in CTA order, so results are deterministic.
#include "attn_decode_unit.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "tma.cuh"

namespace llm {

namespace {

constexpr int MW = 4;                       // consumer warps
constexpr int CT = MW * 32;                 // consumer threads
constexpr int MTHREADS = CT + 32;           // + the producer warp
constexpr int KS = 512;                     // k per ring stage
constexpr int RSTRIDE = KS * 2 + 64;        // bytes per stage row (conflict-free A fragments)
constexpr int STAGE = 16 * RSTRIDE;         // 16 rows x 512 k
constexpr uint32_t BAR_LIMIT = 1u << 24;    // grid-barrier polls before giving up

__device__ __forceinline__ void csync() { named_sync(1, CT); }
struct ConsumerSync {
    __device__ static __forceinline__ void sync() { csync(); }
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Rows [r0, r1) of an N-row matrix owned by CTA c of P, in multiples of gran.
__device__ __forceinline__ void row_range(int N, int gran, int c, int P, int &r0, int &r1) {
    const long long units = N / gran;
    r0 = (int)((long long)c * units / P) * gran;
    r1 = (int)((long long)(c + 1) * units / P) * gran;
}

enum { ME_QKV = 0, ME_RESID = 1, ME_SWIGLU = 2, ME_LOGITS = 3 };

struct Mega {
    const MegaArgs &a;
    uint8_t *ring;                 // NST stages
    uint8_t *area;                 // x vector or attention tiles
    float (*red)[16];              // [MW][16]
    float *scal;                   // small per-CTA scalars (norm factor, sums)
    int c, P, tid, warp, lane, nst;
    uint32_t bar0;
    unsigned epoch;
    int it;                        // ring stage counter (same sequence as the producer)

    __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar0 + 8u * (nst + s); }
    __device__ bool aborted() const { return *reinterpret_cast<volatile int *>(a.abort_flag) != 0; }

    // ---- grid barrier over the consumer threads of every CTA
    __device__ void grid_sync() {
        csync();
        if (tid == 0) {
            __threadfence();
            atomicAdd(a.bar, 1u);
            const unsigned target = (epoch + 1) * (unsigned)P;
            bool ok = false;
            for (uint32_t i = 0; i < BAR_LIMIT; ++i) {
                if (ld_acquire(a.bar) >= target) { ok = true; break; }
                if (aborted()) break;
            }
            if (!ok && !aborted()) {
                raise_error(a.err, ERRF_WAIT_TIMEOUT);
                atomicExch(a.abort_flag, 1);
            }
            __threadfence();
        }
        ++epoch;
        csync();
    }

    // ---- the normalised input vector x = fp16(h * r * gain), r from the P partial sums
    __device__ void norm_x(const float *gain, int K) {
        f16 *xs = reinterpret_cast<f16 *>(area);
        float v = 0.f;
        for (int i = tid; i < P; i += CT) v += __ldcg(a.ss + i);
        v = warp_sum(v);
        if (lane == 0) scal[warp] = v;
        csync();
        if (tid == 0) {
            float s = 0.f;
            for (int w = 0; w < MW; ++w) s += scal[w];
            scal[MW] = 1.0f / sqrtf(s / (float)K + a.eps);
        }
        csync();
        const float r = scal[MW];
        for (int i = tid; i < K / 8; i += CT) {
            const float4 *hp = reinterpret_cast<const float4 *>(a.h + i * 8);
            const float4 *gp = reinterpret_cast<const float4 *>(gain + i * 8);
            const float4 h0 = __ldcg(hp), h1 = __ldcg(hp + 1), g0 = gp[0], g1 = gp[1];
            uint4 o;
            o.x = pack_h2(h0.x * r * g0.x, h0.y * r * g0.y);
            o.y = pack_h2(h0.z * r * g0.z, h0.w * r * g0.w);
            o.z = pack_h2(h1.x * r * g1.x, h1.y * r * g1.y);
            o.w = pack_h2(h1.z * r * g1.z, h1.w * r * g1.w);
            *reinterpret_cast<uint4 *>(xs + i * 8) = o;
        }
        csync();
    }
    __device__ void copy_x(const f16 *src, int K) {
        f16 *xs = reinterpret_cast<f16 *>(area);
        for (int i = tid; i < K / 8; i += CT)
            *reinterpret_cast<uint4 *>(xs + i * 8) = __ldcg(reinterpret_cast<const uint4 *>(src + i * 8));
        csync();
    }

    // ---- one matrix phase: y = W x over this CTA's rows, fused epilogue
    template <int EPI>
    __device__ void matrix(const f16 *W, int N, int K, int gran, const KvView *kv) {
        const f16 *xs = reinterpret_cast<const f16 *>(area);
        const int g = lane >> 2, t4 = lane & 3;
        int r0, r1;
        row_range(N, gran, c, P, r0, r1);
        const int nks = K / KS;
        float ss_local = 0.f, best_v = -INFINITY;
        int best_i = 0x7fffffff;
        for (int g0 = r0; g0 < r1; g0 += 16) {
            const int rows = min(16, r1 - g0);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int s = 0; s < nks; ++s, ++it) {
                if (s % MW != warp) continue;
                const int slot = it % nst;
                if (!mbar_wait(full(slot), (it / nst) & 1, a.abort_flag, a.err)) continue;
                const uint8_t *st = ring + (size_t)slot * STAGE;
                const f16 *wlo = reinterpret_cast<const f16 *>(st + g * RSTRIDE) + 8 * t4;
                const f16 *whi = reinterpret_cast<const f16 *>(st + (g + 8) * RSTRIDE) + 8 * t4;
                const f16 *xp = xs + s * KS + 8 * t4;
#pragma unroll 4
                for (int ch = 0; ch < KS / 32; ++ch) {
                    const uint4 lo = *reinterpret_cast<const uint4 *>(wlo + ch * 32);
                    const uint4 hi = *reinterpret_cast<const uint4 *>(whi + ch * 32);
                    uint4 b = make_uint4(0, 0, 0, 0);
                    if (g == 0) b = *reinterpret_cast<const uint4 *>(xp + ch * 32);
                    const uint32_t a0[4] = {lo.x, hi.x, lo.y, hi.y};
                    const uint32_t b0[2] = {b.x, b.y};
                    mma_f16_16816(acc, a0, b0);
                    const uint32_t a1[4] = {lo.z, hi.z, lo.w, hi.w};
                    const uint32_t b1[2] = {b.z, b.w};
                    mma_f16_16816(acc, a1, b1);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(slot));
            }
            if (t4 == 0) {            // column 0 = the one token
                red[warp][g] = acc[0];
                red[warp][g + 8] = acc[2];
            }
            csync();
            if (EPI == ME_SWIGLU) {
                if (tid < GU_GROUP) {     // a whole group: 8 gate rows then the 8 up rows
                    float gt = 0.f, up = 0.f;
#pragma unroll
                    for (int w = 0; w < MW; ++w) { gt += red[w][tid]; up += red[w][tid + GU_GROUP]; }
                    const int j = (g0 / (2 * GU_GROUP)) * GU_GROUP + tid;
                    a.u[j] = f2h(gt / (1.0f + expf(-gt)) * up);
                }
            } else if (EPI == ME_QKV) {
                if (tid < 8 && 2 * tid < rows) {
                    const int n = g0 + 2 * tid;
                    float x0 = 0.f, x1 = 0.f;
#pragma unroll
                    for (int w = 0; w < MW; ++w) { x0 += red[w][2 * tid]; x1 += red[w][2 * tid + 1]; }
                    const int pos = a.pos[0], seq = a.seq[0];
                    if (pos < 0 || pos >= kv->n_ctx || seq < 0 || seq >= kv->n_seq) {
                        raise_error(a.err, ERRF_BAD_INDEX);
                    } else {
                        const int hd = kv->head_dim;
                        if (n < a.n_q + a.n_kv) {
                            const int d = (n < a.n_q ? n : n - a.n_q) % hd;
                            const float2 cs = a.rope[(size_t)pos * (hd / 2) + d / 2];
                            const float y0 = x0 * cs.x - x1 * cs.y, y1 = x0 * cs.y + x1 * cs.x;
                            x0 = y0;
                            x1 = y1;
                        }
                        if (n < a.n_q) {
                            a.qf[n] = x0;
                            a.qf[n + 1] = x1;
                        } else {
                            const bool is_k = n < a.n_q + a.n_kv;
                            const int cc = n - a.n_q - (is_k ? 0 : a.n_kv);
                            const int head = cc / hd, d = cc - head * hd;
                            f16 *base = is_k ? kv->k : kv->v;
                            const size_t off = (size_t)seq * kv->seq_stride + ((size_t)head * kv->n_ctx + pos) * hd + d;
                            *reinterpret_cast<uint32_t *>(base + off) = pack_h2(x0, x1);
                        }
                    }
                }
            } else if (tid < 16) {
                // one row per lane of warp 0; fixed shuffle trees keep it deterministic
                const bool ok = tid < rows;
                float y = 0.f;
#pragma unroll
                for (int w = 0; w < MW; ++w) y += red[w][tid];
                if (EPI == ME_RESID) {
                    float sq = 0.f;
                    if (ok) {
                        const float v = a.h[g0 + tid] + y;
                        a.h[g0 + tid] = v;
                        sq = v * v;
                    }
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffu, sq, o);
                    if (tid == 0) ss_local += sq;
                } else {
                    if (ok) a.logits[g0 + tid] = y;
                    float bv = ok ? y : -INFINITY;
                    int bi = ok ? g0 + tid : 0x7fffffff;
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffu, bv, o);
                        const int oi = __shfl_xor_sync(0xffffu, bi, o);
                        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
                    }
                    if (tid == 0 && bv > best_v) { best_v = bv; best_i = bi; }
                }
            }
            csync();
        }
        if (tid == 0) {
            if (EPI == ME_RESID) a.ss[c] = ss_local;
            if (EPI == ME_LOGITS) { a.amax_v[c] = best_v; a.amax_i[c] = best_i; }
        }
    }
};

// The producer's schedule: the same matrices and row ranges, in phase order.
__device__ __forceinline__ bool stream_matrix(const MegaArgs &a, const f16 *W, int N, int K, int gran, int c, int P,
                                              int lane, uint8_t *ring, uint32_t bar0, int nst, int &it) {
    int r0, r1;
    row_range(N, gran, c, P, r0, r1);
    for (int g0 = r0; g0 < r1; g0 += 16) {
        const int rows = min(16, r1 - g0);
        for (int k = 0; k < K; k += KS, ++it) {
            const int slot = it % nst;
            int ok = 1;
            if (lane == 0) {
                if (it >= nst) ok = mbar_wait(bar0 + 8u * (nst + slot), ((it / nst) & 1) ^ 1, a.abort_flag, a.err);
                if (ok) mbar_expect_tx(bar0 + 8u * slot, (uint32_t)rows * KS * 2);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) return false;
            if (lane < rows)
                bulk_load(smem_u32(ring + (size_t)slot * STAGE + lane * RSTRIDE), W + (size_t)(g0 + lane) * K + k,
                          KS * 2, bar0 + 8u * slot);
        }
    }
    return true;
}

template <int HD, int G>
__global__ void __launch_bounds__(MTHREADS, 1) decode_mega_kernel(const MegaArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ float red[MW][16];
    __shared__ float scal[8];
    __shared__ __align__(8) uint64_t bars[2 * 16];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, c = blockIdx.x, nst = a.n_stages;
    uint8_t *ring = smem_raw;
    uint8_t *area = smem_raw + (size_t)nst * STAGE;
    const uint32_t bar0 = smem_u32(bars);

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(bar0 + 8u * s, 1);
            mbar_init(bar0 + 8u * (nst + s), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int L = a.L;
    if (warp == MW) {
        // ---- producer: weights only, in the consumers' order
        int it = 0;
        bool ok = true;
        for (int l = 0; l < L && ok; ++l) {
            const MegaLayer &w = a.layers[l];
            ok = stream_matrix(a, w.wqkv, a.n_qkv, a.d, 2, c, P, lane, ring, bar0, nst, it) &&
                 stream_matrix(a, w.wo, a.d, a.n_q, 1, c, P, lane, ring, bar0, nst, it) &&
                 stream_matrix(a, w.wgu, 2 * a.F_pad, a.d, 2 * GU_GROUP, c, P, lane, ring, bar0, nst, it) &&
                 stream_matrix(a, w.wdown, a.d, a.F_pad, 1, c, P, lane, ring, bar0, nst, it);
        }
        if (ok) stream_matrix(a, a.w_out, a.V, a.d, 1, c, P, lane, ring, bar0, nst, it);
        if (lane == 0) {
            // every armed stage lands before the CTA's shared memory goes away
            for (int i = it > nst ? it - nst : 0; i < it; ++i)
                for (uint32_t r = 0; r < WAIT_LIMIT && !mbar_try_wait(bar0 + 8u * (i % nst), (i / nst) & 1); ++r) {
                }
        }
        return;
    }

    Mega m{a, ring, area, red, scal, c, P, tid, warp, lane, nst, bar0, 0u, 0};

    // ---- embedding: this CTA's rows of h, and their sum of squares
    {
        int r0, r1;
        row_range(a.d, 1, c, P, r0, r1);
        const int tok = a.tok[0];
        const bool ok = tok >= 0 && tok < a.V;
        if (!ok && tid == 0) raise_error(a.err, ERRF_BAD_TOKEN);
        float sq = 0.f;
        for (int r = r0 + tid; r < r1; r += CT) {
            const float v = ok ? hf(a.token_embd[(size_t)tok * a.d + r]) : 0.f;
            a.h[r] = v;
            sq += v * v;
        }
        sq = warp_sum(sq);
        if (lane == 0) scal[warp] = sq;
        csync();
        if (tid == 0) a.ss[c] = scal[0] + scal[1] + scal[2] + scal[3];
        m.grid_sync();
    }

    const long long per_layer = (long long)a.Hkv * a.n_ctx * HD;
    for (int l = 0; l < L; ++l) {
        const MegaLayer &w = a.layers[l];
        KvView kv;
        kv.k = a.kc + l * per_layer;
        kv.v = a.vc + l * per_layer;
        kv.seq_stride = per_layer * L;
        kv.n_ctx = a.n_ctx; kv.n_seq = a.n_seq; kv.head_dim = HD; kv.n_kv_head = a.Hkv;

        m.norm_x(w.attn_norm, a.d);
        m.matrix<ME_QKV>(w.wqkv, a.n_qkv, a.d, 2, &kv);
        m.grid_sync();

        // attention: one (kv head, split) item per CTA
        if (c < a.Hkv * a.n_split) {
            AttnDecodeArgs at;
            at.q = a.qf; at.kv = kv; at.pos = a.pos; at.seq = a.seq; at.o = a.o; at.T = 1; at.H = a.H;
            at.n_split = a.n_split; at.part = a.attn_part; at.counters = a.attn_cnt; at.err = a.err;
            attn_dec::attn_decode_unit<HD, G, ConsumerSync>(at, c % a.n_split, c / a.n_split, 0, tid, area);
        }
        m.grid_sync();

        m.copy_x(a.o, a.n_q);
        m.matrix<ME_RESID>(w.wo, a.d, a.n_q, 1, nullptr);
        m.grid_sync();

        m.norm_x(w.ffn_norm, a.d);
        m.matrix<ME_SWIGLU>(w.wgu, 2 * a.F_pad, a.d, 2 * GU_GROUP, nullptr);
        m.grid_sync();

        m.copy_x(a.u, a.F_pad);
        m.matrix<ME_RESID>(w.wdown, a.d, a.F_pad, 1, nullptr);
        m.grid_sync();
    }

    m.norm_x(a.out_norm, a.d);
    m.matrix<ME_LOGITS>(a.w_out, a.V, a.d, 1, nullptr);
    m.grid_sync();

    // ---- greedy choice over the CTAs' candidates (ties: lowest index)
    if (c == 0 && tid == 0) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = 0; i < P; ++i) {
            const float v = __ldcg(a.amax_v + i);
            const int ix = __ldcg(a.amax_i + i);
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
        if (bi == 0x7fffffff) bi = 0;
        a.argmax_out[0] = bi;
        if (a.feed) {
            const int k = *a.gen_step;
            if (k < *a.gen_nsteps) a.gen_tokens[k] = bi;
            *a.gen_step = k + 1;
            a.tok_next[0] = bi;
            a.pos_next[0] += 1;
        }
    }
}

}  // namespace

size_t mega_smem_bytes(int n_stages, int head_dim, int max_k) {
    size_t area = (size_t)max_k * sizeof(f16);
    size_t attn = head_dim == 128 ? attn_dec::decode_smem_bytes<128>() : attn_dec::decode_smem_bytes<64>();
    if (attn > area) area = attn;
    return (size_t)n_stages * STAGE + area;
}

bool mega_supported(int T, int d, int n_q, int F_pad, int head_dim, int group) {
    return T == 1 && d % KS == 0 && n_q % KS == 0 && F_pad % KS == 0 && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

#define MEGA_CASE(HDV, GV)                                                                        \
    if (hd == HDV && group == GV)                                                                 \
        return launch_kernel(decode_mega_kernel<HDV, GV>, grid, dim3(MTHREADS), smem, l2, a);

cudaError_t launch_decode_mega(const MegaArgs &a, int group, int grid_ctas, const Launch &l) {
    const int hd = a.head_dim;
    const size_t smem = mega_smem_bytes(a.n_stages, hd, a.F_pad > a.d ? a.F_pad : a.d);
    const dim3 grid(grid_ctas);
    // cooperative: every CTA is resident, which the grid barriers need
    Launch l2 = l;
    l2.cooperative = true;
    MEGA_CASE(64, 1) MEGA_CASE(64, 2) MEGA_CASE(64, 4) MEGA_CASE(64, 8)
    MEGA_CASE(128, 1) MEGA_CASE(128, 2) MEGA_CASE(128, 4) MEGA_CASE(128, 8)
    return cudaErrorInvalidValue;
}

cudaError_t init_mega_attributes() {
    cudaError_t e = cudaSuccess;
#define MEGA_ATTR(HDV, GV) if (!e) e = allow_smem_max(decode_mega_kernel<HDV, GV>);
    MEGA_ATTR(64, 1) MEGA_ATTR(64, 2) MEGA_ATTR(64, 4) MEGA_ATTR(64, 8)
    MEGA_ATTR(128, 1) MEGA_ATTR(128, 2) MEGA_ATTR(128, 4) MEGA_ATTR(128, 8)
#undef MEGA_ATTR
    return e;
}

int mega_pick_stages(int head_dim, int max_k) {
    // as many ring stages as fit next to the largest phase area (at most 16)
    const size_t budget = 227 * 1024 - 12 * 1024;   // dynamic; leaves room for static smem
    int n = 16;
    while (n > 2 && mega_smem_bytes(n, head_dim, max_k) > budget) --n;
    return n;
}

}  // namespace llm
