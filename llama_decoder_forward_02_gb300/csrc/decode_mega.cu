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
//   - in a matrix phase the CTA owns a contiguous, equal range of output rows
//     (whole interleaved gate/up groups, whole RoPE pairs).  Its work is cut
//     into units of 16 rows x 512 k, dealt round-robin to 8 warps; each warp
//     streams its units with 128-bit loads laid out directly as mma.sync A
//     fragments (the input vector is column 0 of B), double-buffered in
//     registers so ~16 KB per warp are always in flight.  Unit results meet in
//     shared memory and are summed in k order; the CTA applies the fused
//     epilogue itself: no cross-CTA reduction;
//   - the attention phase gives each CTA one (kv head, sequence split) item of
//     the decode-attention kernel's work (warps 0-3);
//   - phases are separated by grid barriers (one counter, bounded spin).
//     Weights never depend on a barrier, so before waiting every warp asks L2
//     for its first unit of the next matrix and HBM keeps streaming; a timeout
//     anywhere raises ERRF_WAIT_TIMEOUT and a shared abort flag that makes
//     every CTA skip to the end.
// Norms: each residual phase leaves one partial sum of squares per CTA; the
// next phase sums the P partials in CTA order, so results are deterministic.
#include "attn_decode_unit.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "tma.cuh"

#include <algorithm>

namespace llm {

namespace {

constexpr int NWARP = 8;                    // warps per CTA
constexpr int MTHREADS = NWARP * 32;
constexpr int AW = 4;                       // warps that run the attention item
constexpr int KC = 512;                     // k per unit
constexpr int NCH = KC / 32;                // 32-wide chunks per unit
constexpr int UB = NCH / 2;                 // chunks per register buffer (half a unit)
constexpr int MAX_PART = 8192;              // floats of unit results in smem
constexpr uint32_t BAR_LIMIT = 1u << 24;    // grid-barrier polls before giving up

__device__ __forceinline__ void csync() { __syncthreads(); }
struct AttnSync {
    __device__ static __forceinline__ void sync() { named_sync(2, AW * 32); }
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

struct Frag { uint4 lo[UB], hi[UB]; };

struct Mega {
    const MegaArgs &a;
    uint8_t *area;                 // x vector or attention tiles
    float *part;                   // unit results [MAX_PART]
    float *scal;                   // small per-CTA scalars
    int c, P, tid, warp, lane;
    unsigned epoch;

    __device__ bool aborted() const { return *reinterpret_cast<volatile int *>(a.abort_flag) != 0; }

    // ---- grid barrier over every thread of every CTA
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

    // ---- ask L2 for this warp's first unit of a coming matrix (weights only)
    __device__ void prefetch(const f16 *W, int N, int K, int gran) {
        int r0, r1;
        row_range(N, gran, c, P, r0, r1);
        const int nkc = K / KC;
        const int n_groups = (r1 - r0 + 15) / 16;
        const int u = warp;
        if (u >= n_groups * nkc) return;
        const int g0 = r0 + (u / nkc) * 16, kc = u % nkc;
        const int rows = min(16, r1 - g0);
        // 16 rows x 1 KB = 128 lines of 128 bytes: 4 per lane
        for (int i = lane; i < rows * 8; i += 32) {
            const int r = i >> 3, ln = i & 7;
            asm volatile("prefetch.global.L2 [%0];" :: "l"(W + (size_t)(g0 + r) * K + kc * KC + ln * 64));
        }
    }

    // ---- the normalised input vector x = fp16(h * r * gain), r from the P partial sums
    __device__ void norm_x(const float *gain, int K) {
        f16 *xs = reinterpret_cast<f16 *>(area);
        float v = 0.f;
        for (int i = tid; i < P; i += MTHREADS) v += __ldcg(a.ss + i);
        v = warp_sum(v);
        if (lane == 0) scal[warp] = v;
        csync();
        if (tid == 0) {
            float s = 0.f;
            for (int w = 0; w < NWARP; ++w) s += scal[w];
            scal[NWARP] = 1.0f / sqrtf(s / (float)K + a.eps);
        }
        csync();
        const float r = scal[NWARP];
        for (int i = tid; i < K / 8; i += MTHREADS) {
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
        for (int i = tid; i < K / 8; i += MTHREADS)
            *reinterpret_cast<uint4 *>(xs + i * 8) = __ldcg(reinterpret_cast<const uint4 *>(src + i * 8));
        csync();
    }

    // ---- one matrix phase: y = W x over this CTA's rows, fused epilogue
    template <int EPI>
    __device__ __forceinline__ void matrix(const f16 *W, int N, int K, int gran, const KvView *kv) {
        const f16 *xs = reinterpret_cast<const f16 *>(area);
        const int g = lane >> 2, t4 = lane & 3;
        int r0, r1;
        row_range(N, gran, c, P, r0, r1);
        const int nkc = K / KC;
        const int n_groups = (r1 - r0 + 15) / 16;
        const int units = n_groups * nkc;
        // this warp's stream: units warp, warp + NWARP, ...; each unit is two
        // batches of UB chunks (NCH = 2 * UB), so a batch never leaves its unit
        const int my_units = units > warp ? (units - warp + NWARP - 1) / NWARP : 0;
        const int n_batches = my_units * 2;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        auto load = [&](Frag &f, int bq) {
            if (bq >= n_batches) return;
            const int u = warp + (bq >> 1) * NWARP;
            const int grp = u / nkc, kc = u - grp * nkc;
            const int g0 = r0 + grp * 16;
            int rl = g0 + g, rh = rl + 8;
            if (rl >= r1) rl = g0;                   // padding lanes reread a valid row
            if (rh >= r1) rh = g0;
            const int k = kc * KC + (bq & 1) * (UB * 32) + 8 * t4;
            const f16 *plo = W + (size_t)rl * K + k, *phi = W + (size_t)rh * K + k;
#pragma unroll
            for (int i = 0; i < UB; ++i) {
                f.lo[i] = ldg_stream(plo + i * 32);
                f.hi[i] = ldg_stream(phi + i * 32);
            }
        };
        auto consume = [&](const Frag &f, int bq) {
            if (bq >= n_batches) return;
            const int u = warp + (bq >> 1) * NWARP;
            const int kc = u % nkc;
            const f16 *xp = xs + kc * KC + (bq & 1) * (UB * 32) + 8 * t4;
#pragma unroll
            for (int i = 0; i < UB; ++i) {
                uint4 b = make_uint4(0, 0, 0, 0);
                if (g == 0) b = *reinterpret_cast<const uint4 *>(xp + i * 32);
                const uint32_t a0[4] = {f.lo[i].x, f.hi[i].x, f.lo[i].y, f.hi[i].y};
                const uint32_t b0[2] = {b.x, b.y};
                mma_f16_16816(acc, a0, b0);
                const uint32_t a1[4] = {f.lo[i].z, f.hi[i].z, f.lo[i].w, f.hi[i].w};
                const uint32_t b1[2] = {b.z, b.w};
                mma_f16_16816(acc, a1, b1);
            }
            if (bq & 1) {                            // unit done: park its 16 sums
                if (t4 == 0) {
                    float *pp = part + (size_t)u * 16;
                    pp[g] = acc[0];
                    pp[g + 8] = acc[2];
                }
                acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            }
        };
        Frag f0, f1;
        load(f0, 0);
        for (int bq = 0; bq < n_batches; bq += 2) {
            load(f1, bq + 1);
            consume(f0, bq);
            load(f0, bq + 2);
            consume(f1, bq + 1);
        }
        csync();

        // ---- epilogues, one 16-row group per warp at a time
        float ss_local = 0.f, best_v = -INFINITY;
        int best_i = 0x7fffffff;
        for (int grp = warp; grp < n_groups; grp += NWARP) {
            const int g0 = r0 + grp * 16, rows = min(16, r1 - g0);
            float y = 0.f;                  // lane < 16: row lane of the group, summed in k order
            if (lane < 16)
                for (int kc = 0; kc < nkc; ++kc) y += part[(size_t)(grp * nkc + kc) * 16 + lane];
            if (EPI == ME_SWIGLU) {
                const float up = __shfl_down_sync(0xffffffffu, y, GU_GROUP);
                if (lane < GU_GROUP) {
                    const int j = (g0 / (2 * GU_GROUP)) * GU_GROUP + lane;
                    a.u[j] = f2h(y / (1.0f + expf(-y)) * up);
                }
            } else if (EPI == ME_QKV) {
                const float y1 = __shfl_down_sync(0xffffffffu, y, 1);
                if (lane < 16 && (lane & 1) == 0 && lane < rows) {
                    const int n = g0 + lane;
                    float x0 = y, x1 = y1;
                    const int pos = a.pos[0], seq = a.seq[0];
                    if (pos < 0 || pos >= kv->n_ctx || seq < 0 || seq >= kv->n_seq) {
                        raise_error(a.err, ERRF_BAD_INDEX);
                    } else {
                        const int hd = kv->head_dim;
                        if (n < a.n_q + a.n_kv) {
                            const int d = (n < a.n_q ? n : n - a.n_q) % hd;
                            const float2 cs = a.rope[(size_t)pos * (hd / 2) + d / 2];
                            const float z0 = x0 * cs.x - x1 * cs.y, z1 = x0 * cs.y + x1 * cs.x;
                            x0 = z0;
                            x1 = z1;
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
            } else if (EPI == ME_RESID) {
                float sq = 0.f;
                if (lane < rows) {
                    const float v = a.h[g0 + lane] + y;
                    a.h[g0 + lane] = v;
                    sq = v * v;
                }
                sq = warp_sum(sq);
                if (lane == 0) part[MAX_PART - 1 - grp] = sq;     // per-group sums, tail of the buffer
            } else {   // ME_LOGITS
                const bool ok = lane < rows;
                if (ok) a.logits[g0 + lane] = y;
                float bv = ok ? y : -INFINITY;
                int bi = ok ? g0 + lane : 0x7fffffff;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
                }
                if (lane == 0 && (bv > best_v || (bv == best_v && bi < best_i))) { best_v = bv; best_i = bi; }
            }
        }
        if (EPI == ME_LOGITS && lane == 0) {
            scal[16 + warp] = best_v;
            reinterpret_cast<int *>(scal)[24 + warp] = best_i;
        }
        csync();
        if (tid == 0) {
            if (EPI == ME_RESID) {
                for (int grp = 0; grp < n_groups; ++grp) ss_local += part[MAX_PART - 1 - grp];
                a.ss[c] = ss_local;
            }
            if (EPI == ME_LOGITS) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
                for (int w = 0; w < NWARP; ++w) {
                    const float v = scal[16 + w];
                    const int ix = reinterpret_cast<int *>(scal)[24 + w];
                    if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
                }
                a.amax_v[c] = bv;
                a.amax_i[c] = bi;
            }
        }
        csync();
    }
};

template <int HD, int G>
__device__ __noinline__ void attention_item(const MegaArgs &a, const KvView &kv, int c, int tid, uint8_t *area) {
    AttnDecodeArgs at;
    at.q = a.qf; at.kv = kv; at.pos = a.pos; at.seq = a.seq; at.o = a.o; at.T = 1; at.H = a.H;
    at.n_split = a.n_split; at.part = a.attn_part; at.counters = a.attn_cnt; at.err = a.err;
    attn_dec::attn_decode_unit<HD, G, AttnSync>(at, c % a.n_split, c / a.n_split, 0, tid, area);
}

template <int HD, int G>
__global__ void __launch_bounds__(MTHREADS, 1) decode_mega_kernel(const MegaArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ float scal[32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, c = blockIdx.x;
    float *part = reinterpret_cast<float *>(smem_raw);
    uint8_t *area = smem_raw + MAX_PART * sizeof(float);
    const int L = a.L;

    Mega m{a, area, part, scal, c, P, tid, warp, lane, 0u};

    // ---- embedding: this CTA's rows of h, and their sum of squares
    {
        const MegaLayer &w0 = a.layers[0];
        if (L > 0) m.prefetch(w0.wqkv, a.n_qkv, a.d, 2);
        int r0, r1;
        row_range(a.d, 1, c, P, r0, r1);
        const int tok = a.tok[0];
        const bool ok = tok >= 0 && tok < a.V;
        if (!ok && tid == 0) raise_error(a.err, ERRF_BAD_TOKEN);
        float sq = 0.f;
        for (int r = r0 + tid; r < r1; r += MTHREADS) {
            const float v = ok ? hf(a.token_embd[(size_t)tok * a.d + r]) : 0.f;
            a.h[r] = v;
            sq += v * v;
        }
        sq = warp_sum(sq);
        if (lane == 0) scal[warp] = sq;
        csync();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < NWARP; ++w) t += scal[w];
            a.ss[c] = t;
        }
        m.grid_sync();
    }

    const long long per_layer = (long long)a.Hkv * a.n_ctx * HD;
    for (int l = 0; l < L && !m.aborted(); ++l) {
        const MegaLayer &w = a.layers[l];
        KvView kv;
        kv.k = a.kc + l * per_layer;
        kv.v = a.vc + l * per_layer;
        kv.seq_stride = per_layer * L;
        kv.n_ctx = a.n_ctx; kv.n_seq = a.n_seq; kv.head_dim = HD; kv.n_kv_head = a.Hkv;

        m.norm_x(w.attn_norm, a.d);
        m.matrix<ME_QKV>(w.wqkv, a.n_qkv, a.d, 2, &kv);
        m.prefetch(w.wo, a.d, a.n_q, 1);
        m.grid_sync();

        // attention: one (kv head, split) item per CTA, on warps 0..AW-1
        if (c < a.Hkv * a.n_split && warp < AW) attention_item<HD, G>(a, kv, c, tid, area);
        m.grid_sync();

        m.copy_x(a.o, a.n_q);
        m.matrix<ME_RESID>(w.wo, a.d, a.n_q, 1, nullptr);
        m.prefetch(w.wgu, 2 * a.F_pad, a.d, 2 * GU_GROUP);
        m.grid_sync();

        m.norm_x(w.ffn_norm, a.d);
        m.matrix<ME_SWIGLU>(w.wgu, 2 * a.F_pad, a.d, 2 * GU_GROUP, nullptr);
        m.prefetch(w.wdown, a.d, a.F_pad, 1);
        m.grid_sync();

        m.copy_x(a.u, a.F_pad);
        m.matrix<ME_RESID>(w.wdown, a.d, a.F_pad, 1, nullptr);
        if (l + 1 < L) m.prefetch(a.layers[l + 1].wqkv, a.n_qkv, a.d, 2);
        else m.prefetch(a.w_out, a.V, a.d, 1);
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
    (void)n_stages;
    size_t area = (size_t)max_k * sizeof(f16);
    size_t attn = head_dim == 128 ? attn_dec::decode_smem_bytes<128>() : attn_dec::decode_smem_bytes<64>();
    if (attn > area) area = attn;
    return MAX_PART * sizeof(float) + area;
}

bool mega_supported(int T, int d, int n_q, int F_pad, int head_dim, int group) {
    return T == 1 && d % KC == 0 && n_q % KC == 0 && F_pad % KC == 0 && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

// Whether every CTA's unit results fit the shared buffer for these shapes.
bool mega_fits(int grid, int d, int n_qkv, int n_q, int F_pad, int V) {
    auto units = [&](int N, int K, int gran) {
        const long long per = ((long long)(N / gran) + grid - 1) / grid * gran;
        return ((per + 15) / 16) * (K / KC) * 16 + 64;
    };
    const long long need = std::max(std::max(units(n_qkv, d, 2), units(d, n_q, 1)),
                                    std::max(std::max(units(2 * F_pad, d, 16), units(d, F_pad, 1)), units(V, d, 1)));
    return need <= MAX_PART;
}

#define MEGA_CASE(HDV, GV)                                                                        \
    if (hd == HDV && group == GV)                                                                 \
        return launch_kernel(decode_mega_kernel<HDV, GV>, grid, dim3(MTHREADS), smem, l2, a);

cudaError_t launch_decode_mega(const MegaArgs &a, int group, int grid_ctas, const Launch &l) {
    const int hd = a.head_dim;
    const size_t smem = mega_smem_bytes(0, hd, a.F_pad > a.d ? a.F_pad : a.d);
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

int mega_pick_stages(int head_dim, int max_k) { (void)head_dim; (void)max_k; return 0; }

}  // namespace llm
