// One decode token at batch 1 as a single persistent kernel: embedding, every
// layer (RMSNorm -> QKV + RoPE + KV append -> attention over the cache -> O +
// residual -> RMSNorm -> gate/up + SiLU*up -> down + residual), final RMSNorm,
// output projection and greedy argmax ("Inside the inference engine: model
// architectures and forward pass", section "Detailed explanation: Llama's
// forward pass in Go"; "LLama.cpp — how it works", "KV-cache and the Prefill /
// Decode stages": one new token's Q, K, V, K and V appended, attention over
// the cache; "Token sampling pipeline": temperature 0 is argmax).
//
// Decode at batch 1 is a stream of ~15 GB of weights per token through a
// chain of tiny dependent computations.  Weights never depend on activations,
// so the stream is decoupled from the chain:
//   - one CTA per SM (cooperative launch, so all are resident).  In every
//     matrix phase the CTA owns a contiguous range of output rows, which is one
//     contiguous byte range of the row-major weight matrix;
//   - warp 0 (one lane) is the producer.  It walks the CTA's whole schedule for
//     the token -- each layer's QKV rows, the K/V rows of its attention item,
//     O rows, gate/up rows, down rows, then the output-projection rows -- and
//     copies it in chunks of whole rows (up to 32 KB) into a ring of shared-memory stages with
//     cp.async.bulk, each stage completing an mbarrier by transaction bytes.
//     It waits only for free stages, never for activations, so HBM keeps
//     streaming across the phase boundaries while the chain resolves;
//   - warps 1..8 are consumers.  A phase starts when a grid-wide counter says
//     its input is complete; the consumers then build the phase's input vector
//     in shared memory and take the stages (whole rows) in ring order, each
//     warp a fixed 1/8 of the columns of every row, whose input values it
//     keeps in registers.  At batch 1 a weight takes one multiply-add, which
//     the CUDA cores do with ample headroom (the legacy mma.sync path would
//     waste most of each instruction here).  Per-warp row sums meet in a small
//     shared buffer and the fused epilogue (RoPE + KV append, residual,
//     SiLU*up, logits + argmax) runs in blocks of rows;
//   - attention gives each CTA one (kv head, sequence split) item; the producer
//     streams the item's cached K/V rows (all final before the kernel starts),
//     the consumers add the newest row, which this token's QKV phase wrote, and
//     the CTA arriving last at the head's counter merges the splits.
// Every wait is bounded: a timeout raises ERRF_WAIT_TIMEOUT and a shared abort
// flag that makes every CTA skip to the end; the producer then waits (bounded)
// for its own copies in flight before the CTA exits.  Sums run in a fixed
// order, so results do not depend on timing.
#include "common.cuh"
#include "launch.cuh"
#include "tma.cuh"

#include <algorithm>

namespace llm {

namespace {

constexpr int NCW = 8;                      // consumer warps
constexpr int CTHREADS = NCW * 32;
constexpr int MTHREADS = CTHREADS + 32;     // + the producer warp
constexpr int STAGE = 32768;                // bytes per ring stage
constexpr int NST = 5;                      // ring stages
constexpr int SEG = 256;                    // fp16 weights per warp segment (512 bytes)
constexpr int RB = 128;                     // row slots of the row-sum buffer
constexpr int EPI_ROWS = 64;                // rows per epilogue block (at least)
constexpr uint32_t SPIN_LIMIT = 1u << 23;   // polls of a grid counter before giving up
constexpr int MAX_SPLIT = 128;
constexpr int MAX_G = 8;
constexpr int JD = 2;                       // K / 2048 of the d-wide inputs (n_embd, n_head * head_dim) at most
constexpr int JF = 7;                       // K / 2048 of the FFN input (padded n_ff) at most

enum { ME_QKV = 0, ME_RESID = 1, ME_SWIGLU = 2, ME_LOGITS = 3 };

// Rows [r0, r1) of an N-row matrix owned by CTA c of P, in multiples of gran.
__device__ __forceinline__ void row_range(int N, int gran, int c, int P, int &r0, int &r1) {
    const long long units = N / gran;
    r0 = (int)((long long)c * units / P) * gran;
    r1 = (int)((long long)(c + 1) * units / P) * gran;
}

// The CTA's rows of one matrix, streamed as chunks of whole rows (as many as
// fit a stage; K * 2 <= STAGE).
struct Slice {
    const f16 *w;   // first byte of the CTA's rows
    int r0, rows, K;
    __device__ int rows_per_chunk() const { return STAGE / (K * 2); }
    __device__ int chunks() const { return (rows + rows_per_chunk() - 1) / rows_per_chunk(); }
};

__device__ __forceinline__ Slice make_slice(const f16 *W, int N, int K, int gran, int c, int P) {
    int r0, r1;
    row_range(N, gran, c, P, r0, r1);
    return Slice{W + (size_t)r0 * K, r0, r1 - r0, K};
}

// The CTA's attention item: keys [kb, ke) of kv head j; keys below pre_end are
// streamed through the ring in tiles of tk keys (a K chunk, then a V chunk).
struct Item {
    int active, j, sp, kb, ke, pre_end, n_eff, tk;
    const f16 *kg, *vg;      // head j of the row's sequence, key 0
    __device__ int tiles() const { return active ? (pre_end - kb + tk - 1) / tk : 0; }
};

__device__ __forceinline__ Item make_item(const MegaArgs &a, const f16 *kc, const f16 *vc, int c, int pos,
                                          int seq, bool ok) {
    Item it;
    it.tk = STAGE / (a.head_dim * 2);
    it.j = c / a.n_split;
    it.sp = c - it.j * a.n_split;
    const int S = ok ? pos + 1 : 0;
    int chunk = (S + a.n_split - 1) / a.n_split;
    chunk = ((chunk + it.tk - 1) / it.tk) * it.tk;
    if (chunk < it.tk) chunk = it.tk;
    it.n_eff = S > 0 ? (S + chunk - 1) / chunk : 0;
    it.active = ok && it.j < a.Hkv && it.sp < it.n_eff;
    it.kb = it.sp * chunk;
    it.ke = min(S, it.kb + chunk);
    it.pre_end = min(it.ke, max(it.kb, pos));       // the newest key (pos) is written this token
    const size_t base = ok ? (size_t)seq * ((size_t)a.L * a.Hkv * a.n_ctx * a.head_dim) +
                                 (size_t)it.j * a.n_ctx * a.head_dim
                           : 0;
    it.kg = kc + base;
    it.vg = vc + base;
    return it;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

// ====================================================================== shared state of one CTA
struct Cta {
    const MegaArgs &a;
    uint8_t *ring;            // NST x STAGE
    uint8_t *area;            // input vector (fp16) or attention scratch
    float *part;              // [RB][NCW] per-warp row sums
    float *red;               // [2 * NCW] reduction scratch
    uint32_t bar_full, bar_empty;
    int c, P, tid, warp, lane;
    int *s_abort;             // shared copy of the abort state

    __device__ uint32_t full(int s) const { return bar_full + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar_empty + 8u * s; }
    __device__ bool aborted() const { return *reinterpret_cast<volatile int *>(s_abort) != 0; }
    __device__ void abort_all() const {
        *reinterpret_cast<volatile int *>(s_abort) = 1;
        atomicExch(a.abort_flag, 1);
    }
    __device__ bool global_abort() const { return *reinterpret_cast<volatile int *>(a.abort_flag) != 0; }
};

// Bounded mbarrier wait that also gives up once the grid aborts; a failure
// marks the CTA aborted (so its other warps end the phase too).
__device__ __forceinline__ bool ring_wait(const Cta &m, uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        // the shared flag is cheap; the grid-wide one costs an L2 round trip
        if (((i & 63) == 63 && m.aborted()) || ((i & 8191) == 8191 && m.global_abort())) {
            m.abort_all();
            return false;
        }
    }
    raise_error(m.a.err, ERRF_WAIT_TIMEOUT);
    m.abort_all();
    return false;
}

// ====================================================================== producer
struct Producer {
    Cta &m;
    int st = 0, ph = 0;
    long long issued = 0;     // chunks armed so far
    uint64_t pol;

    __device__ bool put(const void *src, uint32_t bytes) {
        if (m.aborted()) return false;
        if (issued >= NST && !ring_wait(m, m.empty(st), ph ^ 1)) return false;
        mbar_expect_tx(m.full(st), bytes);
        bulk_load_hint(smem_u32(m.ring + (size_t)st * STAGE), src, bytes, m.full(st), pol);
        ++issued;
        if (++st == NST) { st = 0; ph ^= 1; }
        return true;
    }
    __device__ bool slice(const Slice &s) {
        const int rpc = s.rows_per_chunk();
        for (int r = 0; r < s.rows; r += rpc)
            if (!put(s.w + (size_t)r * s.K, (uint32_t)(min(rpc, s.rows - r) * s.K * 2))) return false;
        return true;
    }
    __device__ bool item(const Item &it, int hd) {
        for (int t = 0, k0 = it.kb; t < it.tiles(); ++t, k0 += it.tk) {
            const int nk = min(it.tk, it.pre_end - k0);
            const uint32_t bytes = (uint32_t)nk * hd * 2;
            if (!put(it.kg + (size_t)k0 * hd, bytes)) return false;
            if (!put(it.vg + (size_t)k0 * hd, bytes)) return false;
        }
        return true;
    }
    // wait (bounded) for every copy still in flight before shared memory goes away
    __device__ void drain() {
        for (long long q = issued > NST ? issued - NST : 0; q < issued; ++q) {
            const int s = (int)(q % NST);
            const uint32_t parity = (uint32_t)((q / NST) & 1);
            for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(m.full(s), parity); ++i) {
            }
        }
    }
};

// ====================================================================== consumers
struct Consumer {
    Cta &m;
    int ctid, cw, lane;
    int st = 0, ph = 0;
    float ssq = 0.f;            // per-thread sum of squares of residual rows
    float best_v = -INFINITY;   // per-thread logits candidate
    int best_i = 0x7fffffff;

    __device__ void csync() const { named_sync(1, CTHREADS); }

    // Wait until *ctr >= target (one thread polls), then release all consumers.
    __device__ bool wait_count(const unsigned *ctr, unsigned target) {
        if (ctid == 0) {
            bool ok = false;
            for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
                if (ld_acquire(ctr) >= target) { ok = true; break; }
                if ((i & 15) == 15 && m.global_abort()) break;
            }
            if (!ok) {
                if (!m.global_abort()) raise_error(m.a.err, ERRF_WAIT_TIMEOUT);
                m.abort_all();
            }
        }
        csync();
        return !m.aborted();
    }
    // Make this CTA's phase outputs visible, then count the CTA in.
    __device__ void signal(unsigned *ctr) {
        __threadfence();
        csync();
        if (ctid == 0) {
            __threadfence();
            atomicAdd(ctr, 1u);
        }
    }
    // Lane 0 waits (bounded) and the warp follows its decision; the other
    // lanes then observe the completed phase themselves, which makes the bulk
    // copy's bytes visible to them (the stage cannot be re-armed before this
    // warp releases it, so the phase cannot move on meanwhile).
    __device__ bool next_stage(uint8_t *&stg) {
        int okv = 0;
        if (lane == 0) okv = ring_wait(m, m.full(st), ph) ? 1 : 0;
        okv = __shfl_sync(0xffffffffu, okv, 0);
        if (!okv) return false;
        for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(m.full(st), ph); ++i) {
        }
        __syncwarp();
        stg = m.ring + (size_t)st * STAGE;
        return true;
    }
    __device__ void release_stage() {
        __syncwarp();
        if (lane == 0) mbar_arrive(m.empty(st));
        advance();
    }
    // step to the next stage without releasing the current one
    __device__ void advance() {
        if (++st == NST) { st = 0; ph ^= 1; }
    }
    // release an earlier stage (by index) that was skipped by advance()
    __device__ void release_at(int s_idx) {
        __syncwarp();
        if (lane == 0) mbar_arrive(m.empty(s_idx));
    }

    // ---- input vectors (fp16 in m.area).  x = fp16(h * r * gain) with r from
    // the P per-CTA sums of squares (summed in CTA order); the h and gain loads
    // are issued together with the partial sums.
    __device__ void norm_x(const float *gain, int K) {
        const MegaArgs &a = m.a;
        f16 *xs = reinterpret_cast<f16 *>(m.area);
        const int n = K / 8;
        constexpr int U = 2;
        float v = 0.f;
        for (int i = ctid; i < m.P; i += CTHREADS) v += __ldcg(a.ss + i);
        float r = 0.f;
        for (int i0 = ctid, pass = 0; i0 < n || pass == 0; i0 += U * CTHREADS, ++pass) {
            float4 h0[U], h1[U], g0[U], g1[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * CTHREADS;
                if (i < n) {
                    const float4 *hp = reinterpret_cast<const float4 *>(a.h + i * 8);
                    const float4 *gp = reinterpret_cast<const float4 *>(gain + i * 8);
                    h0[u] = __ldcg(hp); h1[u] = __ldcg(hp + 1); g0[u] = gp[0]; g1[u] = gp[1];
                }
            }
            if (pass == 0) {
                v = warp_sum(v);
                if (lane == 0) m.red[cw] = v;
                csync();
                float t = 0.f;
#pragma unroll
                for (int w = 0; w < NCW; ++w) t += m.red[w];
                r = 1.0f / sqrtf(t / (float)K + a.eps);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * CTHREADS;
                if (i < n) {
                    uint4 o;
                    o.x = pack_h2(h0[u].x * r * g0[u].x, h0[u].y * r * g0[u].y);
                    o.y = pack_h2(h0[u].z * r * g0[u].z, h0[u].w * r * g0[u].w);
                    o.z = pack_h2(h1[u].x * r * g1[u].x, h1[u].y * r * g1[u].y);
                    o.w = pack_h2(h1[u].z * r * g1[u].z, h1[u].w * r * g1[u].w);
                    *reinterpret_cast<uint4 *>(xs + i * 8) = o;
                }
            }
        }
        csync();
    }
    __device__ void copy_x(const f16 *src, int K) {
        f16 *xs = reinterpret_cast<f16 *>(m.area);
        const int n = K / 8;
        for (int i0 = ctid; i0 < n; i0 += 8 * CTHREADS) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * CTHREADS;
                if (i < n) v[u] = __ldcg(reinterpret_cast<const uint4 *>(src + i * 8));
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * CTHREADS;
                if (i < n) *reinterpret_cast<uint4 *>(xs + i * 8) = v[u];
            }
        }
        csync();
    }

    // Row sums on the CUDA cores.  At batch 1 a weight takes one multiply-add,
    // which the CUDA cores do with ample headroom.  Warp cw owns columns
    // [cw K/8, (cw+1) K/8) of every row: its slice of the input vector stays in
    // registers (fp32) for the whole phase, and each lane reads 16 contiguous
    // bytes per 256 columns of a row (J = K / 2048 reads per row), so shared
    // memory carries only the weights.  The warp's partial sum of a row goes
    // to the row-sum buffer; the epilogue adds the 8 partials in warp order.
    template <int EPI, int JMAX>
    __device__ bool matrix(const Slice &s, int gran, const KvView *kv, int pos, int seq) {
        const int J = s.K / 2048;                           // 16-byte reads per lane per row (<= JMAX)
        const int col0 = cw * (s.K / NCW) + lane * 8;       // first column of this lane
        // the lane's inputs: fp32 for short slices, packed fp16 pairs (widened at
        // use) for the long FFN slice, to stay within the register budget
        constexpr bool XH = JMAX > 4;
        float xr[XH ? 1 : JMAX][8];
        __half2 xh[XH ? JMAX : 1][4];
        {
            const f16 *xs = reinterpret_cast<const f16 *>(m.area);
#pragma unroll
            for (int j = 0; j < JMAX; ++j) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (j < J) v = *reinterpret_cast<const uint4 *>(xs + col0 + j * 256);
                const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (XH) {
                        xh[XH ? j : 0][e] = h[e];
                    } else {
                        const float2 f = __half22float2(h[e]);
                        xr[XH ? 0 : j][2 * e] = f.x;
                        xr[XH ? 0 : j][2 * e + 1] = f.y;
                    }
                }
            }
        }
        const int rpc = s.rows_per_chunk();
        const int nch = s.chunks();
        int epi_done = 0;
        bool bad = false;           // this warp's ring wait failed: no more stages
        for (int i = 0; i < nch; ++i) {
            const int r0 = i * rpc, nr = min(rpc, s.rows - r0);
            uint8_t *stg = nullptr;
            if (!bad && !next_stage(stg)) bad = true;
            if (!bad) {
                // four rows at a time: independent loads, sums and reductions
                const uint8_t *base = stg + (size_t)col0 * 2;
                for (int r = 0; r < nr; r += 4) {
                    float acc[4][2];
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) {
                        acc[rr][0] = acc[rr][1] = 0.f;
                        if (r + rr < nr) {
                            const uint8_t *rowp = base + (size_t)(r + rr) * s.K * 2;
#pragma unroll
                            for (int j = 0; j < JMAX; ++j) {
                                if (j < J) {
                                    const uint4 v = *reinterpret_cast<const uint4 *>(rowp + j * 512);
                                    const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float2 f = __half22float2(h[e]);
                                        float2 x;
                                        if (XH) x = __half22float2(xh[XH ? j : 0][e]);
                                        else x = make_float2(xr[XH ? 0 : j][2 * e], xr[XH ? 0 : j][2 * e + 1]);
                                        acc[rr][0] = fmaf(f.x, x.x, acc[rr][0]);
                                        acc[rr][1] = fmaf(f.y, x.y, acc[rr][1]);
                                    }
                                }
                            }
                        }
                    }
                    // reduce the four rows across the warp by halving: after the
                    // xor-16 and xor-8 exchanges each lane holds one row's partial
                    // (row (lane >> 3) & 3), which three more exchanges complete
                    const float v0 = acc[0][0] + acc[0][1], v1 = acc[1][0] + acc[1][1];
                    const float v2 = acc[2][0] + acc[2][1], v3 = acc[3][0] + acc[3][1];
                    const bool hi16 = lane & 16, hi8 = lane & 8;
                    // lanes < 16 keep rows 0,1 and send rows 2,3; lanes >= 16 the reverse
                    const float s0 = hi16 ? v0 : v2, s1 = hi16 ? v1 : v3;
                    float k0 = (hi16 ? v2 : v0) + __shfl_xor_sync(0xffffffffu, s0, 16);
                    float k1 = (hi16 ? v3 : v1) + __shfl_xor_sync(0xffffffffu, s1, 16);
                    // now rows {0,1} (lanes < 16) or {2,3}; keep one by bit 3
                    float t = (hi8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, hi8 ? k0 : k1, 8);
                    t += __shfl_xor_sync(0xffffffffu, t, 4);
                    t += __shfl_xor_sync(0xffffffffu, t, 2);
                    t += __shfl_xor_sync(0xffffffffu, t, 1);
                    const int rr = (hi16 ? 2 : 0) + (hi8 ? 1 : 0);
                    if ((lane & 7) == 0 && r + rr < nr) m.part[((r0 + r + rr) % RB) * NCW + cw] = t;
                }
                release_stage();
            }
            const int done_rows = r0 + nr;
            const int upto = (i == nch - 1) ? s.rows : done_rows - done_rows % gran;
            if (upto - epi_done >= EPI_ROWS || (i == nch - 1 && upto > epi_done)) {
                csync();
                epilogue<EPI>(s, epi_done, upto, kv, pos, seq);
                csync();
                epi_done = upto;
            }
        }
        csync();
        return !m.aborted();
    }

    // Sum of row r's per-warp partials (in warp order); the slot is cleared by
    // the same thread for the row that reuses it.
    __device__ float row_sum(int r) {
        float y = 0.f;
        float *p = m.part + (r % RB) * NCW;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            y += p[w];
            p[w] = 0.f;
        }
        return y;
    }

    template <int EPI>
    __device__ void epilogue(const Slice &s, int ra, int rb, const KvView *kv, int pos, int seq) {
        const MegaArgs &a = m.a;
        if (EPI == ME_RESID) {
            for (int r = ra + ctid; r < rb; r += CTHREADS) {
                const int n = s.r0 + r;
                const float v = __ldcg(a.h + n) + row_sum(r);
                a.h[n] = v;
                ssq += v * v;
            }
        } else if (EPI == ME_LOGITS) {
            for (int r = ra + ctid; r < rb; r += CTHREADS) {
                const int n = s.r0 + r;
                const float y = row_sum(r);
                a.logits[n] = y;
                if (y > best_v || (y == best_v && n < best_i)) { best_v = y; best_i = n; }
            }
        } else if (EPI == ME_SWIGLU) {
            // groups of 16 rows: 8 gate rows, then the 8 up rows of the same outputs
            for (int i = ctid; i < (rb - ra) / 2; i += CTHREADS) {
                const int grp = i / GU_GROUP, jj = i - grp * GU_GROUP;
                const int rg = ra + grp * 2 * GU_GROUP + jj;
                const float g = row_sum(rg), up = row_sum(rg + GU_GROUP);
                const int j = ((s.r0 + ra) / (2 * GU_GROUP) + grp) * GU_GROUP + jj;
                a.u[j] = f2h(silu(g) * up);
            }
        } else {   // ME_QKV: rows come in RoPE pairs (2i, 2i+1)
            const int hd = a.head_dim;
            for (int i = ctid; i < (rb - ra) / 2; i += CTHREADS) {
                const int r = ra + 2 * i, n = s.r0 + r;
                float x0 = row_sum(r), x1 = row_sum(r + 1);
                if (n < a.n_q + a.n_kv) {
                    const int d = (n < a.n_q ? n : n - a.n_q) % hd;
                    const float2 cs = a.rope[(size_t)pos * (hd / 2) + d / 2];
                    const float z0 = x0 * cs.x - x1 * cs.y, z1 = x0 * cs.y + x1 * cs.x;
                    x0 = z0;
                    x1 = z1;
                }
                if (n < a.n_q) {
                    *reinterpret_cast<float2 *>(a.qf + n) = make_float2(x0, x1);
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
    }

    // Fixed-order CTA sums of the per-thread residual / argmax state.
    __device__ void finish_resid() {
        float v = warp_sum(ssq);
        ssq = 0.f;
        if (lane == 0) m.red[NCW + cw] = v;
        csync();
        if (ctid == 0) {
            float s = 0.f;
            for (int w = 0; w < NCW; ++w) s += m.red[NCW + w];
            m.a.ss[m.c] = s;
        }
    }
    __device__ void finish_logits() {
        float bv = best_v;
        int bi = best_i;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) {
            m.red[cw] = bv;
            reinterpret_cast<int *>(m.red)[NCW + cw] = bi;
        }
        csync();
        if (ctid == 0) {
            float v = -INFINITY;
            int ix = 0x7fffffff;
            for (int w = 0; w < NCW; ++w) {
                const float ov = m.red[w];
                const int oi = reinterpret_cast<int *>(m.red)[NCW + w];
                if (ov > v || (ov == v && oi < ix)) { v = ov; ix = oi; }
            }
            m.a.amax_v[m.c] = v;
            m.a.amax_i[m.c] = ix;
        }
    }

    // ---- the attention item: this split of kv head j, merged by the last split.
    // Warp cw takes keys cw, cw + 8, ... of each K/V tile (the tile's K chunk
    // and V chunk are two consecutive stages); lane l holds dims
    // [l DPL, (l+1) DPL) of q, K, V and o for the G query heads of the group.
    // Each key updates the warp's online softmax at once (the G partial dot
    // products are reduced together), so no score arrays are kept.
    template <int HD, int G>
    __device__ __noinline__ bool attention(const Item &it, const KvView &kv, int l) {
        const MegaArgs &a = m.a;
        constexpr int DPL = HD / 32;                 // dims per lane
        constexpr int REC = HD + 2;
        const float qscale = 1.4426950408889634f / sqrtf((float)HD);
        float q[G][DPL], o[G][DPL], mrow[G], lrow[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                q[g][e] = __ldcg(a.qf + (size_t)(it.j * G + g) * HD + lane * DPL + e) * qscale;
                o[g][e] = 0.f;
            }
            mrow[g] = -INFINITY;
            lrow[g] = 0.f;
        }
        // one key: k and v are this lane's DPL dims of the key's K and V rows
        auto key = [&](const float (&k)[DPL], const float (&v)[DPL]) {
            float sc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float p = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) p = fmaf(q[g][e], k[e], p);
                sc[g] = p;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int g = 0; g < G; ++g) sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], off);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mn = fmaxf(mrow[g], sc[g]);
                const float corr = exp2f(mrow[g] - mn);     // 0 when mrow is -inf
                const float p = exp2f(sc[g] - mn);
                mrow[g] = mn;
                lrow[g] = lrow[g] * corr + p;
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[g][e] = fmaf(o[g][e], corr, p * v[e]);
            }
        };
        auto load_row = [&](const f16 *row, float (&out)[DPL], bool global) {
#pragma unroll
            for (int e = 0; e < DPL; e += 2) {
                uint32_t w;
                if (global) w = __ldcg(reinterpret_cast<const unsigned *>(row + lane * DPL + e));
                else w = *reinterpret_cast<const unsigned *>(row + lane * DPL + e);
                out[e] = h2lo(w);
                out[e + 1] = h2hi(w);
            }
        };

        const int tk = it.tk;
        for (int t = 0, k0 = it.kb; t < it.tiles(); ++t, k0 += tk) {
            const int nk = min(tk, it.pre_end - k0);
            uint8_t *kst = nullptr, *vst = nullptr;
            if (!next_stage(kst)) break;
            const int kst_i = st;                    // remember the K stage; take the V stage next
            advance();
            if (!next_stage(vst)) { release_at(kst_i); break; }
            const f16 *Kt = reinterpret_cast<const f16 *>(kst), *Vt = reinterpret_cast<const f16 *>(vst);
            for (int kk = cw; kk < nk; kk += NCW) {
                float kr[DPL], vr[DPL];
                load_row(Kt + (size_t)kk * HD, kr, false);
                load_row(Vt + (size_t)kk * HD, vr, false);
                key(kr, vr);
            }
            release_at(kst_i);
            release_stage();
        }
        // the newest keys [pre_end, ke), written by this token's QKV phase (through L2)
        for (int k = it.pre_end + cw; k < it.ke; k += NCW) {
            float kr[DPL], vr[DPL];
            load_row(it.kg + (size_t)k * HD, kr, true);
            load_row(it.vg + (size_t)k * HD, vr, true);
            key(kr, vr);
        }

        // ---- combine the 8 warps, write this split's record
        float *wst = reinterpret_cast<float *>(m.area);    // [NCW][G][REC]
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float *ws = wst + ((size_t)cw * G + g) * REC;
            if (lane == 0) { ws[0] = mrow[g]; ws[1] = lrow[g]; }
#pragma unroll
            for (int e = 0; e < DPL; ++e) ws[2 + lane * DPL + e] = o[g][e];
        }
        csync();
        if (m.aborted()) return false;
        const int H = a.H, n_split = a.n_split;
        float *recs = a.attn_part;                           // [H][n_split][REC] (row 0)
        for (int i = ctid; i < G * HD; i += CTHREADS) {
            const int g = i / HD, d = i - g * HD;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NCW; ++w) M = fmaxf(M, wst[((size_t)w * G + g) * REC]);
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < NCW; ++w) {
                    const float *ws = wst + ((size_t)w * G + g) * REC;
                    const float f = exp2f(ws[0] - M);
                    num += f * ws[2 + d];
                    den += f * ws[1];
                }
            }
            float *rp = recs + ((size_t)(it.j * G + g) * n_split + it.sp) * REC;
            rp[2 + d] = num;
            if (d == 0) { rp[0] = M; rp[1] = den; }
        }
        __threadfence();
        csync();
        __shared__ int s_last;
        if (ctid == 0) s_last = atomicAdd(&a.attn_cnt[it.j], 1u) == (unsigned)(it.n_eff - 1);
        csync();
        if (!s_last) return true;
        __threadfence();

        // ---- last split of head j: merge in split order, write o (fp16)
        __shared__ float f_s[MAX_G][MAX_SPLIT], l_s[MAX_G][MAX_SPLIT], inv_l[MAX_G];
        const int ne = it.n_eff;
        for (int i = ctid; i < G * ne; i += CTHREADS) {
            const int g = i / ne, p = i - g * ne;
            const float *rp = recs + ((size_t)(it.j * G + g) * n_split + p) * REC;
            f_s[g][p] = __ldcg(rp);
            l_s[g][p] = __ldcg(rp + 1);
        }
        csync();
        if (ctid < G) {
            float M = -INFINITY;
            for (int p = 0; p < ne; ++p) M = fmaxf(M, f_s[ctid][p]);
            float den = 0.f;
            for (int p = 0; p < ne; ++p) {
                const float mp = f_s[ctid][p];
                const float f = mp == -INFINITY ? 0.f : exp2f(mp - M);
                f_s[ctid][p] = f;
                den += f * l_s[ctid][p];
            }
            inv_l[ctid] = den > 0.f ? 1.f / den : 0.f;
        }
        csync();
        for (int i = ctid; i < G * HD; i += CTHREADS) {
            const int g = i / HD, d = i - g * HD;
            const float *rp = recs + ((size_t)(it.j * G + g) * n_split) * REC + 2 + d;
            float num = 0.f;
            int p = 0;
            for (; p + 4 <= ne; p += 4) {
                const float v0 = __ldcg(rp + (size_t)p * REC), v1 = __ldcg(rp + (size_t)(p + 1) * REC);
                const float v2 = __ldcg(rp + (size_t)(p + 2) * REC), v3 = __ldcg(rp + (size_t)(p + 3) * REC);
                num += f_s[g][p] * v0;
                num += f_s[g][p + 1] * v1;
                num += f_s[g][p + 2] * v2;
                num += f_s[g][p + 3] * v3;
            }
            for (; p < ne; ++p) num += f_s[g][p] * __ldcg(rp + (size_t)p * REC);
            a.o[(size_t)(it.j * G + g) * HD + d] = f2h(num * inv_l[g]);
        }
        if (ctid == 0) a.attn_cnt[it.j] = 0u;
        signal(a.bar + 1);          // one merged head
        (void)kv;
        (void)l;
        return true;
    }
};

template <int HD, int G>
__global__ void __launch_bounds__(MTHREADS, 1) decode_mega_kernel(const MegaArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t s_bars[2 * NST];
    __shared__ float s_red[2 * NCW];
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, c = blockIdx.x;
    const int d = a.d, L = a.L;
    const size_t area_bytes = (size_t)max(max(d, a.n_q), a.F_pad) * 2 > (size_t)NCW * G * (HD + 2) * 4
                                  ? (size_t)max(max(d, a.n_q), a.F_pad) * 2
                                  : (size_t)NCW * G * (HD + 2) * 4;
    Cta m{a, smem_raw, smem_raw + (size_t)NST * STAGE,
          reinterpret_cast<float *>(smem_raw + (size_t)NST * STAGE + ((area_bytes + 127) / 128) * 128), s_red,
          smem_u32(&s_bars[0]), smem_u32(&s_bars[NST]), c, P, tid, warp, lane, &s_abort};

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(m.full(s), 1);
            mbar_init(m.empty(s), NCW);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < RB * NCW; i += MTHREADS) m.part[i] = 0.f;
    __syncthreads();

    // the row's metadata is final before the launch
    const int tok = a.tok[0], pos = a.pos[0], seq = a.seq[0];
    const bool ok = pos >= 0 && pos < a.n_ctx && seq >= 0 && seq < a.n_seq;
    const long long per_layer = (long long)a.Hkv * a.n_ctx * HD;
    auto kv_of = [&](int l) {
        KvView kv;
        kv.k = a.kc + l * per_layer;
        kv.v = a.vc + l * per_layer;
        kv.seq_stride = per_layer * L;
        kv.n_ctx = a.n_ctx; kv.n_seq = a.n_seq; kv.head_dim = HD; kv.n_kv_head = a.Hkv;
        return kv;
    };

    if (warp == 0) {
        // ================================================ producer
        if (lane == 0) {
            Producer pr{m};
            pr.pol = evict_first_policy();
            bool go = true;
            for (int l = 0; l < L && go; ++l) {
                const MegaLayer &w = a.layers[l];
                const KvView kv = kv_of(l);
                go = go && pr.slice(make_slice(w.wqkv, a.n_qkv, d, 2, c, P));
                go = go && pr.item(make_item(a, kv.k, kv.v, c, pos, seq, ok), HD);
                go = go && pr.slice(make_slice(w.wo, d, a.n_q, 1, c, P));
                go = go && pr.slice(make_slice(w.wgu, 2 * a.F_pad, d, 2 * GU_GROUP, c, P));
                go = go && pr.slice(make_slice(w.wdown, d, a.F_pad, 1, c, P));
            }
            if (go) pr.slice(make_slice(a.w_out, a.V, d, 1, c, P));
            pr.drain();
        }
    } else {
        // ================================================ consumers
        Consumer cs{m, tid - 32, warp - 1, lane};
        if (!ok && cs.ctid == 0 && c == 0) raise_error(a.err, ERRF_BAD_INDEX);
        unsigned *ctr = a.bar;
        // embedding: this CTA's rows of h and their sum of squares
        {
            int r0, r1;
            row_range(d, 1, c, P, r0, r1);
            const bool tok_ok = tok >= 0 && tok < a.V;
            if (!tok_ok && cs.ctid == 0 && c == 0) raise_error(a.err, ERRF_BAD_TOKEN);
            for (int r = r0 + cs.ctid; r < r1; r += CTHREADS) {
                const float v = tok_ok ? hf(a.token_embd[(size_t)tok * d + r]) : 0.f;
                a.h[r] = v;
                cs.ssq += v * v;
            }
            cs.finish_resid();
            cs.signal(ctr);
        }
        bool go = true;
        for (int l = 0; l < L && go; ++l) {
            const MegaLayer &w = a.layers[l];
            const KvView kv = kv_of(l);
            const unsigned base = (unsigned)P * (1u + 4u * (unsigned)l);
            // QKV + RoPE + KV append
            go = go && cs.wait_count(ctr, base);
            if (go) cs.norm_x(w.attn_norm, d);
            go = go && cs.matrix<ME_QKV, JD>(make_slice(w.wqkv, a.n_qkv, d, 2, c, P), 2, &kv, ok ? pos : 0, ok ? seq : 0);
            if (go) cs.signal(ctr);
            // attention
            go = go && cs.wait_count(ctr, base + P);
            const Item it = make_item(a, kv.k, kv.v, c, pos, seq, ok);
            if (go && it.active) go = cs.attention<HD, G>(it, kv, l);
            if (ok) go = go && cs.wait_count(a.bar + 1, (unsigned)a.Hkv * (unsigned)(l + 1));
            // O + residual
            if (go) cs.copy_x(a.o, a.n_q);
            go = go && cs.matrix<ME_RESID, JD>(make_slice(w.wo, d, a.n_q, 1, c, P), 1, nullptr, 0, 0);
            if (go) { cs.finish_resid(); cs.signal(ctr); }
            // gate/up + SiLU * up
            go = go && cs.wait_count(ctr, base + 2 * P);
            if (go) cs.norm_x(w.ffn_norm, d);
            go = go && cs.matrix<ME_SWIGLU, JD>(make_slice(w.wgu, 2 * a.F_pad, d, 2 * GU_GROUP, c, P), 2 * GU_GROUP,
                                            nullptr, 0, 0);
            if (go) cs.signal(ctr);
            // down + residual
            go = go && cs.wait_count(ctr, base + 3 * P);
            if (go) cs.copy_x(a.u, a.F_pad);
            go = go && cs.matrix<ME_RESID, JF>(make_slice(w.wdown, d, a.F_pad, 1, c, P), 1, nullptr, 0, 0);
            if (go) { cs.finish_resid(); cs.signal(ctr); }
        }
        // final norm, output projection, greedy choice
        go = go && cs.wait_count(ctr, (unsigned)P * (1u + 4u * (unsigned)L));
        if (go) cs.norm_x(a.out_norm, d);
        go = go && cs.matrix<ME_LOGITS, JD>(make_slice(a.w_out, a.V, d, 1, c, P), 1, nullptr, 0, 0);
        if (go) {
            cs.finish_logits();
            if (cs.ctid == 0) {
                // the CTA whose ticket completes the count picks the token; every
                // candidate was written and fenced before its CTA took a ticket
                __threadfence();
                if (atomicAdd(a.bar + 2, 1u) == (unsigned)P - 1) {
                    __threadfence();
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
        }
    }
    __syncthreads();
}

size_t area_bytes_for(int d, int n_q, int F_pad, int hd, int group) {
    const size_t x = (size_t)std::max(std::max(d, n_q), F_pad) * 2;
    const size_t at = (size_t)NCW * group * (hd + 2) * 4;
    return std::max(x, at);
}

}  // namespace

size_t mega_smem_bytes(int d, int n_q, int F_pad, int hd, int group) {
    return (size_t)NST * STAGE + (area_bytes_for(d, n_q, F_pad, hd, group) + 127) / 128 * 128 +
           (size_t)RB * NCW * sizeof(float);
}

bool mega_supported(int T, int d, int n_q, int F_pad, int head_dim, int group) {
    // every K a multiple of 2048 columns (a warp's 1/8 of a row is whole
    // 256-column runs) and at most JMAX * 2048 (its slice of the input stays in
    // registers: up to JD * 2048 for the d-wide inputs, JF * 2048 for the FFN
    // input); head_dim 64 or 128 (whole lanes)
    auto k_ok = [](int K, int jmax) { return K % 2048 == 0 && K / 2048 <= jmax; };
    return T == 1 && k_ok(d, JD) && k_ok(n_q, JD) && k_ok(F_pad, JF) && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

bool mega_fits(int d, int n_q, int F_pad, int hd, int group, int optin_smem) {
    // static shared memory: barriers, reductions, merge tables (< 10 KB)
    return mega_smem_bytes(d, n_q, F_pad, hd, group) + 10 * 1024 <= (size_t)optin_smem;
}

int mega_keys_per_stage(int head_dim) { return STAGE / (head_dim * 2); }

#define MEGA_CASE(HDV, GV)                                                                        \
    if (hd == HDV && group == GV)                                                                 \
        return launch_kernel(decode_mega_kernel<HDV, GV>, grid, dim3(MTHREADS), smem, l2, a);

cudaError_t launch_decode_mega(const MegaArgs &a, int group, int grid_ctas, const Launch &l) {
    const int hd = a.head_dim;
    const size_t smem = mega_smem_bytes(a.d, a.n_q, a.F_pad, hd, group);
    const dim3 grid(grid_ctas);
    // cooperative: every CTA is resident, which the grid counters need
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

}  // namespace llm
