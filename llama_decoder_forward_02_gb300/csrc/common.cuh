// Shared device helpers for the sm_103a kernels of the Llama forward pass.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <cuda_fp8.h>

namespace llm {

// Error-flag bits raised by kernels (ORed into a device word the host reads).
enum : uint32_t {
    ERRF_BAD_TOKEN = 1u,      // embedding saw a token id outside [0, n_vocab)
    ERRF_BAD_INDEX = 2u,      // a metadata index (seq, pos, row) was out of range
    ERRF_WAIT_TIMEOUT = 4u,   // a bounded wait gave up
    ERRF_F16_RANGE = 8u,      // an activation narrowed to fp16 was not finite or beyond +-65504
};

__device__ __forceinline__ void raise_error(uint32_t *err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

// Tensor-core operands, activations and the KV cache are fp16 (see the
// model set-up for why); the residual stream and accumulators are fp32.
// Widening fp16 -> fp32 is exact; narrowing rounds to nearest even.
__device__ __forceinline__ float h2lo(uint32_t packed) {
    return __low2float(*reinterpret_cast<const __half2 *>(&packed));
}
__device__ __forceinline__ float h2hi(uint32_t packed) {
    return __high2float(*reinterpret_cast<const __half2 *>(&packed));
}
__device__ __forceinline__ float hf(__half v) { return __half2float(v); }
__device__ __forceinline__ __half f2h(float v) { return __float2half_rn(v); }
// two FP8 E4M3 values (nearest, saturating at +-448), lo in the low byte
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
// two FP8 E4M3 values (low byte first) widened exactly to f16x2
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint16_t v) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// SiLU(x) = x / (1 + e^-x), the gate of the SwiGLU MLP, Down(SiLU(Gate x) * Up x)
// ("Inside the inference engine: model architectures and forward pass",
// section "Detailed explanation: Llama's forward pass in Go")
__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }
// The same through the fast exponential and division intrinsics, for the
// prefill epilogue that evaluates it on every element of a tile: a few ulp
// of fp32, far inside the fp16 rounding of its result (x / inf gives -0 for
// very negative x, as the exact form does)
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }
// true when a value cannot be stored as a finite fp16 (NaN, or |v| > 65504)
__device__ __forceinline__ bool f16_bad(float v) { return !(fabsf(v) <= 65504.f); }
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}
// bf16 bits -> fp32 (exact): the inputs handed to the library are bf16.
__device__ __forceinline__ float bf16f(__nv_bfloat16 v) { return __bfloat162float(v); }

// Programmatic dependent launch: a kernel may start before its predecessor
// in the stream finishes; it must call pdl_wait() before touching anything
// the predecessor writes (and before writing anything the predecessor
// reads).  pdl_trigger() lets the successor start launching.  Both are
// no-ops when the launch did not ask for programmatic serialization.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// 128-bit streaming load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// mma.sync m16n8k16, fp16 inputs, fp32 accumulate (row.col).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool pred) {
    int n = pred ? 16 : 0;   // zero-fill when the source row is past the end
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(smem_u32(smem)), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t (&r)[2], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}

}  // namespace llm
