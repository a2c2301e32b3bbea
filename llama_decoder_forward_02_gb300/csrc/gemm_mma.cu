// Prefill GEMM on the legacy tensor-core path (mma.sync m16n8k16, f16 in,
// fp32 accumulate): C[m][n] = sum_k A[m][k] W[n][k], with the epilogues of the
// Llama layer fused in ("Inside the inference engine: model architectures
// and forward pass", section "Detailed explanation: Llama's forward pass in
// Go": Q/K/V projections + RoPE, output projection + residual, SiLU(Gate)*Up,
// Down + residual; the KV append of "KV Cache: memory for causal attention").
//
// 128 x 128 x 32 CTA tiles, 8 warps of 64 x 32, a 4-stage cp.async ring in
// XOR-swizzled shared memory and ldmatrix fragment loads.  The grid walks M
// fastest so the CTAs that share a weight tile run together and the tile is
// fetched from HBM once.  This is the baseline the tcgen05 kernel replaces.
#include "common.cuh"
#include "launch.cuh"

namespace llm {

namespace {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 4, THREADS = 256;
constexpr int TILE_ELEMS = BM * BK;   // == BN * BK

// rows of 32 f16 = four 16-byte chunks; swizzle by row pairs
__device__ __forceinline__ int sw(int r, int c) { return r * BK + ((c ^ ((r >> 1) & 3)) * 8); }

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

template <int EPI>
__global__ void __launch_bounds__(THREADS) gemm_mma_kernel(const GemmArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    f16 *As = reinterpret_cast<f16 *>(smem_raw);
    f16 *Bs = As + STAGES * TILE_ELEMS;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int wm = warp >> 2, wn = warp & 3;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int nk = a.K / BK;

    // weights do not depend on the previous kernel: start the first stages'
    // B loads before the dependency wait, A loads after it
    auto load_b = [&](int stage, int kt) {
        f16 *dst = Bs + stage * TILE_ELEMS;
        const f16 *src = a.W + (size_t)n0 * a.K + kt * BK;
        for (int i = tid; i < BN * 4; i += THREADS) {
            const int r = i >> 2, c = i & 3;
            cp_async16(dst + sw(r, c), src + (size_t)r * a.K + c * 8, true);
        }
    };
    auto load_a = [&](int stage, int kt) {
        f16 *dst = As + stage * TILE_ELEMS;
        for (int i = tid; i < BM * 4; i += THREADS) {
            const int r = i >> 2, c = i & 3;
            const int m = m0 + r;
            const bool pv = m < a.M;
            cp_async16(dst + sw(r, c), a.A + (size_t)(pv ? m : 0) * a.K + kt * BK + c * 8, pv);
        }
    };

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s)
        if (s < nk) load_b(s, s);
    pdl_wait();
    pdl_trigger();
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nk) load_a(s, s);
        cp_async_commit();
    }

    float acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jn = 0; jn < 4; ++jn) acc[i][jn][0] = acc[i][jn][1] = acc[i][jn][2] = acc[i][jn][3] = 0.f;

    for (int kt = 0; kt < nk; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        const int pf = kt + STAGES - 1;
        if (pf < nk) { load_b(pf % STAGES, pf); load_a(pf % STAGES, pf); }
        cp_async_commit();

        const f16 *At = As + (kt % STAGES) * TILE_ELEMS;
        const f16 *Bt = Bs + (kt % STAGES) * TILE_ELEMS;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            uint32_t af[4][4], bfr[4][2];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi) {
                const int r = wm * 64 + mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = ks * 2 + (lane >> 4);
                ldmatrix_x4(af[mi], smem_u32(At + sw(r, c)));
            }
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t t[4];
                const int r = wn * 32 + np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = ks * 2 + ((lane >> 3) & 1);
                ldmatrix_x4(t, smem_u32(Bt + sw(r, c)));
                bfr[2 * np][0] = t[0]; bfr[2 * np][1] = t[1];
                bfr[2 * np + 1][0] = t[2]; bfr[2 * np + 1][1] = t[3];
            }
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) mma_f16_16816(acc[mi][ni], af[mi], bfr[ni]);
        }
    }
    cp_async_wait<0>();

    // ---- epilogue: element pairs (row, col), (row, col+1) with col even
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int row = m0 + wm * 64 + mi * 16 + g + hr * 8;
            if (row >= a.M) continue;
            if (EPI == EPI_SWIGLU) {
#pragma unroll
                for (int gp = 0; gp < 2; ++gp) {   // n8 tiles (gate, up) = (2gp, 2gp+1)
                    const int colg = n0 + wn * 32 + gp * 16;
                    const int jbase = (colg / (2 * GU_GROUP)) * GU_GROUP + 2 * t4;
                    const float g0 = acc[mi][2 * gp][2 * hr], g1 = acc[mi][2 * gp][2 * hr + 1];
                    const float u0 = acc[mi][2 * gp + 1][2 * hr], u1 = acc[mi][2 * gp + 1][2 * hr + 1];
                    *reinterpret_cast<uint32_t *>(a.u_out + (size_t)row * a.ldu + jbase) =
                        pack_h2(silu(g0) * u0, silu(g1) * u1);
                }
                continue;
            }
            int pos = 0, seq = 0;
            bool meta_ok = true;
            if (EPI == EPI_QKV) {
                pos = a.pos[row];
                seq = a.seq[row];
                meta_ok = pos >= 0 && pos < a.kv.n_ctx && seq >= 0 && seq < a.kv.n_seq;
                if (!meta_ok) raise_error(a.err, ERRF_BAD_INDEX);
            }
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int col = n0 + wn * 32 + ni * 8 + 2 * t4;
                float x0 = acc[mi][ni][2 * hr], x1 = acc[mi][ni][2 * hr + 1];
                if (EPI == EPI_STORE) {
                    *reinterpret_cast<float2 *>(a.C + (size_t)row * a.ldc + col) = make_float2(x0, x1);
                } else if (EPI == EPI_RESID) {
                    float2 *hp = reinterpret_cast<float2 *>(a.hres + (size_t)row * a.ldh + col);
                    float2 v = *hp;
                    v.x += x0;
                    v.y += x1;
                    *hp = v;
                } else if (EPI == EPI_QKV && meta_ok) {
                    const int hd = a.kv.head_dim;
                    if (col < a.n_q + a.n_kv) {
                        const int d = (col < a.n_q ? col : col - a.n_q) % hd;
                        const float2 cs = a.rope[(size_t)pos * (hd / 2) + d / 2];
                        const float y0 = x0 * cs.x - x1 * cs.y, y1 = x0 * cs.y + x1 * cs.x;
                        x0 = y0;
                        x1 = y1;
                    }
                    if (col < a.n_q) {
                        *reinterpret_cast<uint32_t *>(a.q_out + (size_t)row * a.n_q + col) = pack_h2(x0, x1);
                    } else {
                        const bool is_k = col < a.n_q + a.n_kv;
                        const int c = col - a.n_q - (is_k ? 0 : a.n_kv);
                        const int head = c / hd, d = c - head * hd;
                        const size_t off = (size_t)seq * a.kv.seq_stride + ((size_t)head * a.kv.n_ctx + pos) * hd + d;
                        if (a.kv.k8)
                            *reinterpret_cast<uint16_t *>((is_k ? a.kv.k8 : a.kv.v8) + off) = pack_e4m3x2(x0, x1);
                        else
                            *reinterpret_cast<uint32_t *>((is_k ? a.kv.k : a.kv.v) + off) = pack_h2(x0, x1);
                    }
                }
            }
        }
    }
}

constexpr size_t SMEM = (size_t)2 * STAGES * TILE_ELEMS * sizeof(f16);

}  // namespace

cudaError_t launch_gemm_mma(int epi, const GemmArgs &a, const Launch &l) {
    if (a.M < 1 || a.N % BN || a.K % BK) return cudaErrorInvalidValue;
    const dim3 grid((a.M + BM - 1) / BM, a.N / BN);
    switch (epi) {
        case EPI_STORE: return launch_kernel(gemm_mma_kernel<EPI_STORE>, grid, dim3(THREADS), SMEM, l, a);
        case EPI_RESID: return launch_kernel(gemm_mma_kernel<EPI_RESID>, grid, dim3(THREADS), SMEM, l, a);
        case EPI_QKV: return launch_kernel(gemm_mma_kernel<EPI_QKV>, grid, dim3(THREADS), SMEM, l, a);
        case EPI_SWIGLU: return launch_kernel(gemm_mma_kernel<EPI_SWIGLU>, grid, dim3(THREADS), SMEM, l, a);
    }
    return cudaErrorInvalidValue;
}

cudaError_t init_gemm_mma_attributes() {
    cudaError_t e = allow_smem(gemm_mma_kernel<EPI_STORE>, SMEM);
    if (!e) e = allow_smem(gemm_mma_kernel<EPI_RESID>, SMEM);
    if (!e) e = allow_smem(gemm_mma_kernel<EPI_QKV>, SMEM);
    if (!e) e = allow_smem(gemm_mma_kernel<EPI_SWIGLU>, SMEM);
    return e;
}

}  // namespace llm
