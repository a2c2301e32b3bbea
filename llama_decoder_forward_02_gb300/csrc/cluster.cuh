// Thread-block cluster helpers: rank, cluster-wide barriers and distributed
// shared memory (a CTA's shared variable addressed in another CTA of the same
// cluster), plus the row argmax that a cluster of CTAs takes together.
#pragma once
#include "common.cuh"

namespace llm {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Split cluster barrier: arrive (release: this CTA's earlier shared-memory
// writes become visible to the cluster) and wait (acquire).  Every thread of
// every CTA of the cluster takes the same sequence of arrive / wait.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
    cluster_arrive();
    cluster_wait();
}

// Address of shared variable `p` in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t dsmem(const void *p, uint32_t rank) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void dsmem_st_u32(uint32_t a, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st_u64(uint32_t a, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ void dsmem_add_u32(uint32_t a, uint32_t v) {
    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// CTAs per row for the cluster row kernels (argmax, sampling): eight SMs
// share one vocabulary row, each reading an eighth of it.
constexpr int ROW_CLUSTER = 8;

// Slice of a row of n elements owned by cluster rank r: [lo, lo + len), with
// lo a multiple of 128 elements (512 bytes) and len a multiple of 4 when n is.
__host__ __device__ __forceinline__ int row_slice_len(int n) {
    return ((n + ROW_CLUSTER - 1) / ROW_CLUSTER + 127) / 128 * 128;
}

// Greedy choice over a row ("Inside the inference engine: model
// architectures and forward pass", "Token sampling pipeline": temperature 0
// takes the argmax), by a cluster of ROW_CLUSTER CTAs of blockDim.x threads.
// Ties go to the lowest index; NaN never wins; an all -inf / NaN row gives 0.
// The row is read as float4: n % 4 == 0 and `row` 16-byte aligned.  Must be
// called by every thread of every CTA of the cluster; the result is valid in
// cluster rank 0 only (other ranks get -1).  Takes two cluster barriers.
__device__ __forceinline__ void argmax_better(float &bv, int &bi, float v, int i) {
    if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
}

__device__ inline int cluster_row_argmax(const float *row, int n) {
    __shared__ float c_v[32];
    __shared__ int c_i[32];
    __shared__ float r_v[ROW_CLUSTER];
    __shared__ int r_i[ROW_CLUSTER];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const uint32_t rank = cluster_rank();
    cluster_arrive();                                   // every CTA has started (waited below)
    const int S = row_slice_len(n);
    const int lo = (int)rank * S, len = max(0, min(S, n - lo));
    const float4 *r4 = reinterpret_cast<const float4 *>(row + lo);
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    const int n4 = len >> 2;
    for (int i0 = tid; i0 < n4; i0 += 4 * blockDim.x) {
        float4 q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * blockDim.x;
            q[j] = i < n4 ? __ldg(r4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int v = lo + 4 * (i0 + j * blockDim.x);
            argmax_better(bv, bi, q[j].x, v);
            argmax_better(bv, bi, q[j].y, v + 1);
            argmax_better(bv, bi, q[j].z, v + 2);
            argmax_better(bv, bi, q[j].w, v + 3);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        argmax_better(bv, bi, ov, oi);
    }
    if (lane == 0) { c_v[warp] = bv; c_i[warp] = bi; }
    __syncthreads();
    cluster_wait();
    if (warp == 0) {
        bv = lane < nw ? c_v[lane] : -INFINITY;
        bi = lane < nw ? c_i[lane] : 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            argmax_better(bv, bi, ov, oi);
        }
        if (lane == 0) {                                // this CTA's best, into rank 0's slots
            dsmem_st_u32(dsmem(&r_v[rank], 0), __float_as_uint(bv));
            dsmem_st_u32(dsmem(&r_i[rank], 0), (uint32_t)bi);
        }
    }
    cluster_sync();
    if (rank != 0) return -1;
    bv = -INFINITY;
    bi = 0x7fffffff;
    for (int r = 0; r < ROW_CLUSTER; ++r) argmax_better(bv, bi, r_v[r], r_i[r]);
    return bi == 0x7fffffff ? 0 : bi;
}

}  // namespace llm
