// Prefill GEMM on the 5th-generation tensor cores: C[m][n] = sum_k A[m][k] W[n][k]
// (activations [M][K], weights [N][K], both K-contiguous fp16, fp32 accumulate),
// with the epilogues of the Llama layer fused in ("Inside the inference engine:
// model architectures and forward pass", section "Detailed explanation: Llama's
// forward pass in Go": Q/K/V + RoPE + KV append, output projection + residual,
// SiLU(Gate)*Up, Down + residual, the output projection).
//
// One CTA computes a 128 x BN tile (BN = 128 or 256), or one K split of it
// (gridDim.z splits, residual epilogue only: the last split to finish adds
// them in split order), with four warps:
//   warp 0, one lane: TMA producer.  Each stage is a 128 x 64 A box and a
//     BN x 64 W box in 128-byte-swizzled shared memory, completing a "full"
//     mbarrier by transaction bytes.  Weight boxes of the first stages are
//     issued before the programmatic-dependent-launch wait.
//   warp 1, one lane: tcgen05.mma issuer (kind::f16, M = 128, N = BN, K = 16,
//     four per stage) into a BN-column fp32 accumulator in tensor memory;
//     tcgen05.commit frees each stage's "empty" mbarrier and finally signals
//     the accumulator barrier.  Warp 1 also allocates and frees the TMEM.
//   all four warps: epilogue.  Warp w reads TMEM lanes 32w..32w+31 (its
//     accumulator rows) 32 columns at a time with tcgen05.ld and applies the
//     fused epilogue in registers.
// Every mbarrier wait is bounded: on timeout the kernel raises
// ERRF_WAIT_TIMEOUT, stops issuing, waits (bounded) for what it issued, frees
// its TMEM and returns.  No multicast, no clusters.
#include <cuda.h>

#include "common.cuh"
#include "launch.cuh"
#include "tma.cuh"
#include "gemm_tc_common.cuh"

namespace llm {

namespace {

using namespace tcg;

template <int BN>
struct Cfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BYTES = BN * BK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 256;
    // instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
    // (formats 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24
    static constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
};

__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        :: "r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(accum) : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

template <int BN, int EPI>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
    using C = Cfg<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ int s_abort;
    __shared__ uint32_t s_tmem;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bar0 = base + C::STAGES * C::STAGE_BYTES;    // full[S], empty[S], accum
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    const uint32_t accum = bar0 + 8u * (2 * C::STAGES);
    auto a_smem = [&](int s) { return base + s * C::STAGE_BYTES; };
    auto b_smem = [&](int s) { return base + s * C::STAGE_BYTES + C::A_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    // split-K: CTA z of gridDim.z takes k-blocks [kb0, kb0 + nk)
    const int nk_all = a.K / BK, z = blockIdx.z, nz = gridDim.z;
    const int kb0 = (int)((long long)z * nk_all / nz);
    const int nk = (int)((long long)(z + 1) * nk_all / nz) - kb0;
    volatile int *abort = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(accum, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&s_tmem)), "r"((uint32_t)BN) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    const int pre = nk < C::STAGES ? nk : C::STAGES;
    int issued = 0;                          // stages the producer armed
    if (warp == 0 && lane == 0) {
        // weights do not depend on the previous kernel: start their boxes now
        for (int kb = 0; kb < pre; ++kb) {
            mbar_expect_tx(full(kb), C::STAGE_BYTES);
            tma_load_2d(b_smem(kb), &tmB, full(kb), (kb0 + kb) * BK, n0);
        }
    }
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % C::STAGES;
                if (kb >= pre) {
                    if (!mbar_wait(empty(s), ((kb / C::STAGES) & 1) ^ 1, abort, a.err)) break;
                    mbar_expect_tx(full(s), C::STAGE_BYTES);
                    tma_load_2d(b_smem(s), &tmB, full(s), (kb0 + kb) * BK, n0);
                }
                tma_load_2d(a_smem(s), &tmA, full(s), (kb0 + kb) * BK, m0);
                issued = kb + 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int done = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % C::STAGES;
                if (!mbar_wait(full(s), (kb / C::STAGES) & 1, abort, a.err)) break;
                tc_fence_after();
                const uint64_t ad = sdesc(a_smem(s)), bd = sdesc(b_smem(s));
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)   // advance 16 elements = 32 bytes inside the swizzle atom
                    tc_mma(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), C::IDESC, (kb | k) != 0);
                tc_commit(empty(s));
                done = kb + 1;
            }
            tc_commit(accum);                    // fires once the issued MMAs are complete
            (void)done;
        }
        __syncwarp();
    }

    // ---- epilogue: warp w owns accumulator rows (TMEM lanes) 32w .. 32w+31
    mbar_wait(accum, 0, abort, a.err);       // a timeout marks the CTA aborted
    __syncthreads();
    const bool ok = !*abort;                 // the same for every thread of the CTA
    tc_fence_after();
    if (ok && nz == 1) {
        const int row = m0 + warp * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c * 32), r);
            if (row < a.M) epilogue32<EPI>(a, row, n0 + c * 32, r);
        }
    } else if (ok && EPI == EPI_RESID) {
        // split-K: each split parks its fp32 tile in the workspace; the CTA that
        // arrives last at the tile's counter adds the splits in split order to
        // the residual, so the result does not depend on arrival order
        const int row = m0 + warp * 32 + lane;
        const size_t ld = (size_t)a.N;
        float *mine = a.ws + (size_t)z * a.M * ld;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c * 32), r);
            if (row < a.M) {
                float4 *dst = reinterpret_cast<float4 *>(mine + (size_t)row * ld + n0 + c * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                         __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
            }
        }
        __threadfence();
        __syncthreads();
        __shared__ int s_last;
        const int tile = blockIdx.x * gridDim.y + blockIdx.y;
        if (threadIdx.x == 0) s_last = atomicAdd(&a.tile_cnt[tile], 1u) == (unsigned)(nz - 1);
        __syncthreads();
        if (s_last) {
            __threadfence();
            if (row < a.M) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; c += 2) {
                    float v[64];
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = 0.f;
                    for (int p = 0; p < nz; ++p) {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            a.ws + ((size_t)p * a.M + row) * ld + n0 + c * 32);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float4 q = __ldcg(src + i);
                            v[4 * i] += q.x; v[4 * i + 1] += q.y; v[4 * i + 2] += q.z; v[4 * i + 3] += q.w;
                        }
                    }
                    float4 *h = reinterpret_cast<float4 *>(a.hres + (size_t)row * a.ldh + n0 + c * 32);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float4 x = h[i];
                        x.x += v[4 * i]; x.y += v[4 * i + 1]; x.z += v[4 * i + 2]; x.w += v[4 * i + 3];
                        h[i] = x;
                    }
                }
            }
            if (threadIdx.x == 0) a.tile_cnt[tile] = 0u;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort && warp == 0 && lane == 0) {
        // let every armed stage land before the CTA's shared memory goes away
        for (int kb = (issued > C::STAGES ? issued - C::STAGES : 0); kb < issued; ++kb) {
            const int s = kb % C::STAGES;
            for (uint32_t i = 0; i < WAIT_LIMIT && !mbar_try_wait(full(s), (kb / C::STAGES) & 1); ++i) {
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"((uint32_t)BN) : "memory");
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace

int gemm_tc_pick_bn(int M, int N, int num_sms) {
    // Per-SM throughput is set by shared memory: the MMA's operand reads plus
    // the TMA writes need ~2x an SM's shared-memory bandwidth with 128 x 128
    // tiles (tensor pipe <= ~50% busy) and ~1.5x with 128 x 256 tiles (~68%).
    // Wider tiles halve the CTA count, so pick the width with the smaller
    // waves x width / efficiency.
    if (N % 256) return 128;
    const long long mt = (M + BM - 1) / BM;
    const long long w128 = (mt * (N / 128) + num_sms - 1) / num_sms;
    const long long w256 = (mt * (N / 256) + num_sms - 1) / num_sms;
    return (double)w256 * 256 / 0.68 < (double)w128 * 128 / 0.50 ? 256 : 128;
}

int gemm_tc_pick_split(int M, int N, int K, int bn, int num_sms) {
    // split K when the tiles fill less than half of the SMs (at most 4 ways,
    // keeping at least 16 k-blocks per split)
    const int tiles = ((M + BM - 1) / BM) * (N / bn);
    int ks = 1;
    while (ks < 4 && tiles * (ks + 1) <= num_sms && K / BK / (ks + 1) >= 16) ++ks;
    return ks;
}

bool make_operand_map(TmaMap *m, const f16 *ptr, int rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !ptr || cols % 64 || rows < 1 || (reinterpret_cast<uintptr_t>(ptr) & 15)) return false;
    static_assert(sizeof(TmaMap) == sizeof(CUtensorMap), "TmaMap must hold a CUtensorMap");
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(reinterpret_cast<CUtensorMap *>(m), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void *)ptr, dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#define TC_CASE(BNV, E)                                                                              \
    if (bn == BNV && epi == E)                                                                       \
        return launch_kernel(gemm_tc_kernel<BNV, E>, grid, dim3(THREADS), Cfg<BNV>::SMEM, l,         \
                             *reinterpret_cast<const CUtensorMap *>(&mA), *reinterpret_cast<const CUtensorMap *>(&mB), a);

cudaError_t launch_gemm_tc(int epi, const GemmArgs &a, const TmaMap &mA, const TmaMap &mB, int bn,
                           const Launch &l) {
    if (a.M < 1 || a.K % BK || a.N % bn || (bn != 128 && bn != 256)) return cudaErrorInvalidValue;
    const int ks = a.ksplit > 1 ? a.ksplit : 1;
    if (ks > 1 && (epi != EPI_RESID || !a.ws || !a.tile_cnt || a.K / BK < ks)) return cudaErrorInvalidValue;
    const dim3 grid((a.M + BM - 1) / BM, a.N / bn, ks);
    TC_CASE(128, EPI_STORE) TC_CASE(128, EPI_RESID) TC_CASE(128, EPI_QKV) TC_CASE(128, EPI_SWIGLU)
    TC_CASE(256, EPI_STORE) TC_CASE(256, EPI_RESID) TC_CASE(256, EPI_QKV) TC_CASE(256, EPI_SWIGLU)
    return cudaErrorInvalidValue;
}

cudaError_t init_gemm_tc_attributes() {
    cudaError_t e = cudaSuccess;
#define TC_ATTR(BNV, E) if (!e) e = allow_smem(gemm_tc_kernel<BNV, E>, Cfg<BNV>::SMEM);
    TC_ATTR(128, EPI_STORE) TC_ATTR(128, EPI_RESID) TC_ATTR(128, EPI_QKV) TC_ATTR(128, EPI_SWIGLU)
    TC_ATTR(256, EPI_STORE) TC_ATTR(256, EPI_RESID) TC_ATTR(256, EPI_QKV) TC_ATTR(256, EPI_SWIGLU)
#undef TC_ATTR
    return e;
}

}  // namespace llm
