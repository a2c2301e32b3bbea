// Batch-1 decode GEMV streamed through shared memory, one CTA per SM
// ("Inside the inference engine: model architectures and forward pass",
// section "Detailed explanation: Llama's forward pass in Go": every linear
// layer of a one-token step; the fused prologues and epilogues are those of
// the register-fragment GEMV: RMSNorm in, RoPE + KV append, SiLU*Up or the
// residual add out).
//
// A one-token step reads every weight byte once, so it is bound by HBM, and
// at one-token sizes the cost of a kernel boundary (the previous kernel's
// tail, the launch, the first round trip) is a large share of each GEMV.
// This kernel is built to overlap those boundaries under programmatic
// dependent launch:
//   * the grid is one CTA per SM and the CTA takes more than half of an SM's
//     shared memory (up to ~200 KB, or a smaller cap that leaves room for a
//     decode-attention CTA beside it), so exactly one CTA of each GEMV fits on
//     an SM, and the next GEMV's CTA lands on an SM as soon as this one leaves
//     it, evenly over the SMs;
//   * CTA b owns whole output rows [r0, r1) (balanced in units of 1, 2 or 16
//     rows: the RoPE pairs and the gate/up interleave stay inside a CTA), so
//     its weights are one contiguous slab and no K-split fixup is needed;
//   * a producer warp streams the slab through a ring of up to eight stages
//     with cp.async.bulk as soon as the CTA starts, before the dependency
//     wait (weights never depend on the previous kernel);
//   * eight consumer warps wait for the previous kernel, load their fixed
//     column slice of x into registers (x = h * gain for the RMSNorm
//     prologue; the 1/rms factor is applied to the finished dot products),
//     and reduce each stage's rows on the CUDA cores in fp32.  R rows of a
//     stage (R = 32 KB / row bytes, a power of two <= 8) go to distinct
//     warps: warp w takes segment w % (8/R) of row w / (8/R); a stage may hold
//     RW such row groups, which the same warps take in turn with the x slice
//     they hold.  Segment partials are summed in segment order, so the result
//     is deterministic and does not depend on RW.
// Q8 instantiations read Q8_0 rows instead of fp16 ones (K one-byte codes,
// then K/32 fp16 block scales; the layout is set out where the rows are
// encoded): half the bytes a weight, stages of several row groups, and each
// lane's 8-element group, which lies inside one 32-element block, is one dot
// product of the codes with x times that block's scale.
// Every mbarrier wait is bounded (ERRF_WAIT_TIMEOUT, then the CTA winds down).
#include "common.cuh"
#include "launch.cuh"
#include "tma.cuh"

namespace llm {

namespace {

constexpr int SW = 8;                     // consumer warps
constexpr int STHREADS = (SW + 1) * 32;   // + one producer warp
constexpr int STAGE_MAX = 32768;          // bytes of one ring stage of one row a warp
constexpr size_t Q8_STAGE_MAX = 98304;    // ... of the stages of Q8_0 rows (several rows a warp)
constexpr int XMAX = 8;                   // 8-element groups of x per lane
constexpr size_t SMEM_MIN = 120 * 1024;   // more than half an SM: one CTA per SM
constexpr size_t SMEM_CAP = 224 * 1024;

struct Plan {
    int unit;          // rows kept together in one CTA
    int R;             // rows per stage taken by distinct warps
    int RW;            // rows each warp takes per stage (same x slice)
    int SR;            // rows per stage, R * RW
    int segs;          // warps per row (8 / R)
    int nx;            // 8-element groups of x per lane (segment = 256 * nx)
    int nst;           // ring stages
    int rows_max;      // largest row count of a CTA
    uint32_t row_bytes;   // 2K (fp16) or K + K/16 (Q8_0)
    uint32_t stage_bytes;
    size_t smem;
    size_t gain_off;   // byte offset of the gain slice in shared memory
};

}  // namespace

int gemv_stream_unit(int epi) { return epi == EPI_QKV ? 2 : epi == EPI_SWIGLU ? 2 * GU_GROUP : 1; }

namespace {

// stage_max: 0 keeps one row per warp and stage; otherwise each warp takes
// RW rows of a stage (a power of two up to 8, all against the x slice it
// holds) while a stage stays within stage_max bytes and at least three stages
// fit.  Wider stages carry more bytes per copy and per barrier round trip:
// they speed up the Q8_0 rows and leave the fp16 rows as they are.
bool make_plan(int epi, int N, int K, int nsm, size_t cap, bool q8, size_t stage_max, Plan *p) {
    const int unit = gemv_stream_unit(epi);
    if (N < 1 || K < 256 || N % unit || nsm < 1) return false;
    const long long row_bytes = q8 ? (long long)K + K / 16 : 2LL * K;
    if (row_bytes > STAGE_MAX) return false;
    // R doubles while two stage rows fit and a lane's share of x stays in
    // XMAX groups (which binds only for Q8_0 rows, half as wide in bytes)
    int R = 1;
    while (2 * R <= SW && 2 * R * row_bytes <= STAGE_MAX && (long long)K * 2 * R <= 256LL * SW * XMAX) R *= 2;
    const int segs = SW / R;
    if (K % (256 * segs)) return false;
    const int nx = K / segs / 256;
    if (nx < 1 || nx > XMAX) return false;
    const long long units = N / unit;
    const int rows_max = (int)((units + nsm - 1) / nsm) * unit;
    const size_t part = (size_t)rows_max * segs * sizeof(float);
    const size_t gsl = ((size_t)rows_max * sizeof(float) + 15) / 16 * 16;
    if (cap < part + gsl + 512) return false;
    const long long room = (long long)(cap - part - gsl - 512);
    int RW = 1;
    while (stage_max && RW < 8 && 2LL * RW * R * row_bytes <= (long long)stage_max &&
           room / (2LL * RW * R * row_bytes) >= 3)
        RW *= 2;
    const uint32_t stage = (uint32_t)(R * RW * row_bytes);
    long long nst = room / stage;
    if (nst > 8) nst = 8;
    if (nst < 3 || (size_t)nst * stage + part + gsl + 512 > cap) return false;
    p->unit = unit; p->R = R; p->RW = RW; p->SR = R * RW; p->segs = segs; p->nx = nx; p->nst = (int)nst; p->rows_max = rows_max;
    p->row_bytes = (uint32_t)row_bytes;
    p->stage_bytes = stage;
    size_t smem = (size_t)nst * stage + part + gsl + 512;
    p->smem = smem < SMEM_MIN ? SMEM_MIN : smem;
    p->gain_off = (size_t)nst * stage + part;           // the rows' next-norm gains (EPI_RESID)
    return true;
}

// Two products of fp16 pairs added to an fp32 sum, one rounding each
// (mixed-precision FMA: fp16 operands, fp32 accumulator).
__device__ __forceinline__ float fma2_f16(uint32_t w, uint32_t x, float s) {
    asm("{\n\t.reg .b16 w0, w1, x0, x1;\n\t"
        "mov.b32 {w0, w1}, %1;\n\tmov.b32 {x0, x1}, %2;\n\t"
        "fma.rn.f32.f16 %0, w0, x0, %0;\n\tfma.rn.f32.f16 %0, w1, x1, %0;\n\t}"
        : "+f"(s) : "r"(w), "r"(x));
    return s;
}

__device__ __forceinline__ float dot8(const uint4 w, const uint4 x) {
    float s = 0.f;
    s = fma2_f16(w.x, x.x, s);
    s = fma2_f16(w.y, x.y, s);
    s = fma2_f16(w.z, x.z, s);
    s = fma2_f16(w.w, x.w, s);
    return s;
}

// Eight Q8_0 codes (little-endian bytes of w) against x.  A code b is flipped
// to the unsigned byte b + 128 and placed by a byte permute in the low
// mantissa of the fp16 1024 (bits 0x6400), which then reads 1024 + b + 128
// exactly; subtracting 1152 in fp16 leaves b, exactly.
__device__ __forceinline__ float dot8_q8(const uint2 w, const uint4 x) {
    const uint32_t lo = w.x ^ 0x80808080u, hi = w.y ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    auto q2 = [&](uint32_t u, uint32_t sel) {
        const uint32_t b = __byte_perm(u, 0x64646464u, sel);
        const __half2 v = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
        return *reinterpret_cast<const uint32_t *>(&v);
    };
    float s = 0.f;
    s = fma2_f16(q2(lo, 0x5140), x.x, s);
    s = fma2_f16(q2(lo, 0x5342), x.y, s);
    s = fma2_f16(q2(hi, 0x5140), x.z, s);
    s = fma2_f16(q2(hi, 0x5342), x.w, s);
    return s;
}

template <int PRO, int EPI, bool Q8>
__global__ void __launch_bounds__(STHREADS, 1) gemv_stream_kernel(const GemvArgs a, const Plan p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t bars[16];                 // full[8], empty[8]
    __shared__ float s_red[SW];
    __shared__ float s_red2[STHREADS / 32];
    __shared__ float s_r;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = a.K;
    const long long units = a.N / p.unit;
    const int u0 = (int)((long long)blockIdx.x * units / gridDim.x);
    const int u1 = (int)((long long)(blockIdx.x + 1) * units / gridDim.x);
    const int r0 = u0 * p.unit, nrows = (u1 - u0) * p.unit;
    const int nstages = (nrows + p.SR - 1) / p.SR;
    uint8_t *ring = smem_raw;
    float *part = reinterpret_cast<float *>(smem_raw + (size_t)p.nst * p.stage_bytes);
    const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[8]);
    volatile int *abort = &s_abort;

    if (tid == 0) {
        for (int s = 0; s < p.nst; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, SW);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_trigger();

    if (warp == SW) {
        // ---- producer: the CTA's weight slab, R rows per stage
        int issued = 0;
        if (lane == 0) {
            const uint8_t *src = (Q8 ? a.W8 : reinterpret_cast<const uint8_t *>(a.W)) + (size_t)r0 * p.row_bytes;
            for (int j = 0; j < nstages; ++j) {
                const int s = j % p.nst;
                if (j >= p.nst && !mbar_wait(empty0 + 8u * s, ((j / p.nst) & 1) ^ 1, abort, a.err)) break;
                const int rows = nrows - j * p.SR < p.SR ? nrows - j * p.SR : p.SR;
                const uint32_t bytes = (uint32_t)rows * p.row_bytes;
                mbar_expect_tx(full0 + 8u * s, bytes);
                bulk_load(smem_u32(ring + (size_t)s * p.stage_bytes), src + (size_t)j * p.stage_bytes, bytes,
                          full0 + 8u * s);
                issued = j + 1;
            }
            // the next GEMVs' first stages for this CTA index, into L2
            auto prefetch = [&](const f16 *W, const uint8_t *W8, int pN, int pK, int unit, long long bytes) {
                if ((!W && !W8) || *abort) return;
                const long long pu = pN / unit;
                const long long q0 = (long long)blockIdx.x * pu / gridDim.x;
                const long long q1 = (long long)(blockIdx.x + 1) * pu / gridDim.x;
                const long long prb = W8 ? (long long)pK + pK / 16 : 2LL * pK;
                const long long slab = (q1 - q0) * unit * prb;
                const long long want = slab < bytes ? slab : bytes;
                const uint8_t *pf = (W8 ? W8 : reinterpret_cast<const uint8_t *>(W)) + (size_t)q0 * unit * prb;
                for (long long off = 0; off < want; off += STAGE_MAX) {
                    const uint32_t n = (uint32_t)(want - off < STAGE_MAX ? want - off : STAGE_MAX);
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(pf + off), "r"(n) : "memory");
                }
            };
            prefetch(a.pf_W, a.pf_W8, a.pf_N, a.pf_K, a.pf_unit, a.pf_bytes);
            prefetch(a.pf2_W, a.pf2_W8, a.pf2_N, a.pf2_K, a.pf2_unit, a.pf2_bytes);
            if (*abort) {
                // let every issued copy land before the shared memory goes away
                for (int j = issued > p.nst ? issued - p.nst : 0; j < issued; ++j) {
                    const int s = j % p.nst;
                    for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(full0 + 8u * s, (j / p.nst) & 1); ++i) {
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ---- consumers
        float *gsl = reinterpret_cast<float *>(smem_raw + p.gain_off);
        if (EPI == EPI_RESID && a.xg_out) {
            // the next norm's gains of this CTA's rows: constant, fetched before the wait
            for (int i = tid; i < nrows; i += SW * 32)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_u32(gsl + i)), "l"(a.gain_next + r0 + i)
                             : "memory");
            cp_async_commit();
        }
        pdl_wait();
        const int seg = warp % p.segs, rin = warp / p.segs;
        const int L = p.nx * 256;
        const int kb = seg * L + lane * 8;             // first element of this lane's x groups
        uint4 xh[XMAX];
        if (PRO == PRO_NORM && a.xg) {
            // x * gain in fp16 and the sum of squares as per-CTA partials, both
            // written by the previous kernel.  Warp 0 alone reads the partials
            // (as float4: every CTA reading them thread by thread made a hot
            // spot of those few L2 lines) and sums them in a fixed order; the
            // factor is needed only by the epilogue
#pragma unroll
            for (int i = 0; i < XMAX; ++i) {
                xh[i] = i < p.nx ? *reinterpret_cast<const uint4 *>(a.xg + kb + i * 256) : make_uint4(0, 0, 0, 0);
            }
            if (warp == 0) {
                // two float4 loads a lane at most (<= 256 partials), issued together
                const int n4 = a.n_ss_in >> 2;
                const float4 *s4 = reinterpret_cast<const float4 *>(a.ss_in);
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 q0 = lane < n4 ? s4[lane] : z;
                const float4 q1 = lane + 32 < n4 ? s4[lane + 32] : z;
                float sp = ((q0.x + q0.y) + (q0.z + q0.w)) + ((q1.x + q1.y) + (q1.z + q1.w));
                if (lane < (a.n_ss_in & 3)) sp += a.ss_in[4 * n4 + lane];
                sp = warp_sum(sp);
                if (lane == 0) s_r = 1.0f / sqrtf(sp / (float)K + a.eps);
            }
        } else if (PRO == PRO_NORM) {
            const int row = a.row_map ? a.row_map[0] : 0;
            const float *hp = a.h + (size_t)row * a.ldh;
            const float *gp = a.gain;
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < XMAX; ++i) {
                if (i < p.nx) {
                    const int k = kb + i * 256;
                    const float4 h0 = *reinterpret_cast<const float4 *>(hp + k);
                    const float4 h1 = *reinterpret_cast<const float4 *>(hp + k + 4);
                    const float4 g0 = *reinterpret_cast<const float4 *>(gp + k);
                    const float4 g1 = *reinterpret_cast<const float4 *>(gp + k + 4);
                    ss += h0.x * h0.x + h0.y * h0.y + h0.z * h0.z + h0.w * h0.w;
                    ss += h1.x * h1.x + h1.y * h1.y + h1.z * h1.z + h1.w * h1.w;
                    xh[i] = make_uint4(pack_h2(h0.x * g0.x, h0.y * g0.y), pack_h2(h0.z * g0.z, h0.w * g0.w),
                                       pack_h2(h1.x * g1.x, h1.y * g1.y), pack_h2(h1.z * g1.z, h1.w * g1.w));
                    if (f16_bad(h0.x * g0.x) | f16_bad(h0.y * g0.y) | f16_bad(h0.z * g0.z) | f16_bad(h0.w * g0.w) |
                        f16_bad(h1.x * g1.x) | f16_bad(h1.y * g1.y) | f16_bad(h1.z * g1.z) | f16_bad(h1.w * g1.w))
                        raise_error(a.err, ERRF_F16_RANGE);
                } else {
                    xh[i] = make_uint4(0, 0, 0, 0);
                }
            }
            // the warps of stage row 0 cover every column once
            ss = warp_sum(ss);
            if (lane == 0 && rin == 0) s_red[seg] = ss;
            named_sync(1, SW * 32);
            if (tid == 0) {
                float t = 0.f;
                for (int s = 0; s < p.segs; ++s) t += s_red[s];
                s_r = 1.0f / sqrtf(t / (float)K + a.eps);
            }
        } else {
#pragma unroll
            for (int i = 0; i < XMAX; ++i) {
                xh[i] = i < p.nx ? *reinterpret_cast<const uint4 *>(a.x + kb + i * 256) : make_uint4(0, 0, 0, 0);
            }
        }
        for (int j = 0; j < nstages; ++j) {
            const int s = j % p.nst;
            if (!mbar_wait(full0 + 8u * s, (j / p.nst) & 1, abort, a.err)) break;
            const int rows = nrows - j * p.SR < p.SR ? nrows - j * p.SR : p.SR;
            // one row's lane partial: independent 8-element dot products summed as a tree
            auto lane_part = [&](int rr) {
                const uint8_t *rowp = ring + (size_t)s * p.stage_bytes + (size_t)rr * p.row_bytes;
                float d[XMAX];
                if (Q8) {
                    // group i starts at element kb + 256 i, in block (kb >> 5) + 8 i
                    const __half *sc = reinterpret_cast<const __half *>(rowp + K) + (kb >> 5);
                    uint2 w[XMAX];
#pragma unroll
                    for (int i = 0; i < XMAX; ++i)
                        if (i < p.nx) w[i] = *reinterpret_cast<const uint2 *>(rowp + kb + i * 256);
#pragma unroll
                    for (int i = 0; i < XMAX; ++i) d[i] = i < p.nx ? dot8_q8(w[i], xh[i]) * __half2float(sc[8 * i]) : 0.f;
                } else {
                    const uint4 *wp = reinterpret_cast<const uint4 *>(rowp) + (kb >> 3);
                    uint4 w[XMAX];
#pragma unroll
                    for (int i = 0; i < XMAX; ++i)
                        if (i < p.nx) w[i] = wp[i * 32];
#pragma unroll
                    for (int i = 0; i < XMAX; ++i) d[i] = i < p.nx ? dot8(w[i], xh[i]) : 0.f;
                }
#pragma unroll
                for (int h = XMAX / 2; h > 0; h >>= 1)
#pragma unroll
                    for (int i = 0; i < h; ++i) d[i] += d[i + h];
                return d[0];
            };
            if (Q8) {
                // Q8_0 stages hold several rows a warp: two rows in flight (the
                // second repeats the first when the stage has no other row for
                // this warp; its result is dropped)
                for (int rr = rin; rr < rows; rr += 2 * p.R) {
                    const bool two = rr + p.R < rows;
                    float a0 = lane_part(rr);
                    float a1 = lane_part(two ? rr + p.R : rr);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        a0 += __shfl_xor_sync(0xffffffffu, a0, o);
                        a1 += __shfl_xor_sync(0xffffffffu, a1, o);
                    }
                    if (lane == 0) {
                        part[(j * p.SR + rr) * p.segs + seg] = a0;
                        if (two) part[(j * p.SR + rr + p.R) * p.segs + seg] = a1;
                    }
                }
            } else {
                for (int rr = rin; rr < rows; rr += p.R) {
                    const float acc = warp_sum(lane_part(rr));
                    if (lane == 0) part[(j * p.SR + rr) * p.segs + seg] = acc;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8u * s);
        }
        if (EPI == EPI_RESID && a.xg_out) cp_async_wait<0>();
    }
    __syncthreads();
    if (*abort) return;

    // ---- epilogue over the CTA's rows (segment partials in segment order)
    const float r = PRO == PRO_NORM ? s_r : 1.0f;
    auto y = [&](int i) {
        float v = 0.f;
        for (int s = 0; s < p.segs; ++s) v += part[i * p.segs + s];
        return v * r;
    };
    if (EPI == EPI_STORE) {
        for (int i = tid; i < nrows; i += STHREADS) a.out[r0 + i] = y(i);
    } else if (EPI == EPI_RESID) {
        const float *gsl = reinterpret_cast<const float *>(smem_raw + p.gain_off);
        float sq = 0.f;
        for (int i = tid; i < nrows; i += STHREADS) {
            const float v = a.hres[r0 + i] + y(i);
            a.hres[r0 + i] = v;
            if (a.xg_out) {
                const float xg = v * gsl[i];
                if (f16_bad(xg)) raise_error(a.err, ERRF_F16_RANGE);
                a.xg_out[r0 + i] = f2h(xg);
                sq += v * v;
            }
        }
        if (a.xg_out) {
            // this CTA's sum of squares of the new h, reduced in a fixed order
            sq = warp_sum(sq);
            if (lane == 0) s_red2[warp] = sq;
            __syncthreads();
            if (tid == 0) {
                float t = 0.f;
                for (int w = 0; w < STHREADS / 32; ++w) t += s_red2[w];
                a.ss_cta[blockIdx.x] = t;
            }
        }
    } else if (EPI == EPI_QKV) {
        const int hd = a.kv.head_dim, half_hd = hd / 2;
        const int pos = a.pos[0], seq = a.seq[0];
        if (pos < 0 || pos >= a.kv.n_ctx || seq < 0 || seq >= a.kv.n_seq) {
            if (tid == 0) raise_error(a.err, ERRF_BAD_INDEX);
            return;
        }
        for (int pi = tid; pi < nrows / 2; pi += STHREADS) {
            const int n = r0 + 2 * pi;
            float x0 = y(2 * pi), x1 = y(2 * pi + 1);
            if (n < a.n_q + a.n_kv) {              // rotate q and k rows
                const int d = (n < a.n_q ? n : n - a.n_q) % hd;
                const float2 cs = a.rope[(size_t)pos * half_hd + d / 2];
                const float y0 = x0 * cs.x - x1 * cs.y, y1 = x0 * cs.y + x1 * cs.x;
                x0 = y0;
                x1 = y1;
            }
            if (n < a.n_q) {
                *reinterpret_cast<float2 *>(a.q_out + n) = make_float2(x0, x1);
            } else {
                const bool is_k = n < a.n_q + a.n_kv;
                const int c = n - a.n_q - (is_k ? 0 : a.n_kv);
                const int head = c / hd, d = c - head * hd;
                const size_t off = (size_t)seq * a.kv.seq_stride + ((size_t)head * a.kv.n_ctx + pos) * hd + d;
                if (a.kv.k8)
                    *reinterpret_cast<uint16_t *>((is_k ? a.kv.k8 : a.kv.v8) + off) = pack_e4m3x2(x0, x1);
                else {
                    if (f16_bad(x0) || f16_bad(x1)) raise_error(a.err, ERRF_F16_RANGE);
                    *reinterpret_cast<uint32_t *>((is_k ? a.kv.k : a.kv.v) + off) = pack_h2(x0, x1);
                }
            }
        }
    } else if (EPI == EPI_SWIGLU) {
        for (int i = tid; i < nrows / 2; i += STHREADS) {
            const int grp = i / GU_GROUP, rr = i - grp * GU_GROUP;
            const float gate = y(grp * 2 * GU_GROUP + rr), up = y(grp * 2 * GU_GROUP + GU_GROUP + rr);
            const int j = (r0 / (2 * GU_GROUP) + grp) * GU_GROUP + rr;
            const float u = silu(gate) * up;
            if (f16_bad(u)) raise_error(a.err, ERRF_F16_RANGE);
            a.u_out[j] = f2h(u);
        }
    }
}

}  // namespace

bool gemv_stream_ok(int epi, int N, int K, int num_sms, int smem_kb, bool q8) {
    Plan p;
    return make_plan(epi, N, K, num_sms, smem_kb > 0 ? (size_t)smem_kb * 1024 : SMEM_CAP, q8, 0, &p);
}

#define GS_CASE(P, E)                                                                                     \
    if (pro == P && epi == E)                                                                             \
        return q8 ? launch_kernel(gemv_stream_kernel<P, E, true>, dim3(num_sms), dim3(STHREADS), p.smem, l, a, p) \
                  : launch_kernel(gemv_stream_kernel<P, E, false>, dim3(num_sms), dim3(STHREADS), p.smem, l, a, p);

cudaError_t launch_gemv_stream(int pro, int epi, const GemvArgs &a, int num_sms, int smem_kb, const Launch &l,
                               int stage_kb) {
    Plan p;
    const size_t cap = smem_kb > 0 ? (size_t)smem_kb * 1024 : SMEM_CAP;
    const bool q8 = a.W8 != nullptr;
    // Q8_0 rows are half as wide: their stages take several rows a warp
    const size_t smax = stage_kb > 0 ? (size_t)stage_kb * 1024 : q8 ? Q8_STAGE_MAX : 0;
    if (a.T != 1 || cap > SMEM_CAP || !make_plan(epi, a.N, a.K, num_sms, cap, q8, smax, &p))
        return cudaErrorInvalidValue;
    GS_CASE(PRO_NORM, EPI_QKV)
    GS_CASE(PRO_BF16, EPI_RESID)
    GS_CASE(PRO_NORM, EPI_SWIGLU)
    GS_CASE(PRO_NORM, EPI_STORE)
    GS_CASE(PRO_BF16, EPI_STORE)
    return cudaErrorInvalidValue;
}

cudaError_t init_gemv_stream_attributes() {
    cudaError_t e = cudaSuccess;
    // every SM keeps its largest shared-memory carveout, so a GEMV CTA and a
    // decode-attention CTA can share an SM without reconfiguring it
#define GS_ATTR1(P, E, Q)                                                                                   \
    if (!e) e = allow_smem(gemv_stream_kernel<P, E, Q>, SMEM_CAP);                                          \
    if (!e) e = cudaFuncSetAttribute(gemv_stream_kernel<P, E, Q>, cudaFuncAttributePreferredSharedMemoryCarveout, \
                                     cudaSharedmemCarveoutMaxShared);
#define GS_ATTR(P, E) GS_ATTR1(P, E, false) GS_ATTR1(P, E, true)
    GS_ATTR(PRO_NORM, EPI_QKV) GS_ATTR(PRO_BF16, EPI_RESID) GS_ATTR(PRO_NORM, EPI_SWIGLU)
    GS_ATTR(PRO_NORM, EPI_STORE) GS_ATTR(PRO_BF16, EPI_STORE)
#undef GS_ATTR
#undef GS_ATTR1
    return e;
}

}  // namespace llm
