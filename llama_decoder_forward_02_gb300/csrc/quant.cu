// Q8_0 weight blocks for the one-row decode GEMVs.  "LLama.cpp — how it
// works", section "The GGUF format (reference)", names Q8_0 among the tensor
// element types (quantised formats that shrink the model) without giving its
// layout; the one taken here: a row is cut into blocks of 32 consecutive
// elements; a block keeps one scale d = max|w| / 127 (stored as fp16) and 32
// signed bytes q = nearest integer to w / d (ties to even), both computed in
// float32 with one rounding per operation, and stands for the weights q * d
// with the stored d.  A block of zeros has d = 0 and q = 0.
//
// In device memory a Q8_0 matrix [N][K] is N rows of K + K/16 bytes: the K
// codes in element order, then the K/32 fp16 scales.  K % 256 == 0 keeps every
// row 16-byte aligned, as the bulk copies of the streamed GEMV need.
#include "common.cuh"
#include "kernels.h"

namespace llm {

namespace {

constexpr int QB = 32;   // elements per block

// One thread per block: thread b of the grid takes block b % (K/32) of row
// b / (K/32).  The block's 32 fp16 elements are read as four 16-byte loads.
// q8 == nullptr skips the encoded copy; write_back replaces the fp16 elements
// by the weights the block stands for, f16(q * d) (one rounding).
__global__ void quantize_q8_0_kernel(f16 *w, int N, int K, uint8_t *q8, int write_back) {
    const int nb = K / QB;
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= (long long)N * nb) return;
    const int row = (int)(b / nb), blk = (int)(b - (long long)row * nb);
    f16 *src = w + (size_t)row * K + (size_t)blk * QB;
    uint4 raw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) raw[i] = reinterpret_cast<const uint4 *>(src)[i];
    const __half2 *h = reinterpret_cast<const __half2 *>(raw);
    float v[QB];
#pragma unroll
    for (int i = 0; i < QB / 2; ++i) {
        const float2 f = __half22float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < QB; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float d = __fdiv_rn(amax, 127.0f);
    int q[QB];
#pragma unroll
    for (int i = 0; i < QB; ++i) q[i] = d > 0.f ? __float2int_rn(__fdiv_rn(v[i], d)) : 0;
    const __half dh = __float2half_rn(d);
    if (q8) {
        uint32_t word[QB / 4];
#pragma unroll
        for (int j = 0; j < QB / 4; ++j)
            word[j] = (uint32_t)(q[4 * j] & 0xff) | (uint32_t)(q[4 * j + 1] & 0xff) << 8 |
                      (uint32_t)(q[4 * j + 2] & 0xff) << 16 | (uint32_t)(q[4 * j + 3] & 0xff) << 24;
        uint8_t *rq = q8 + (size_t)row * ((size_t)K + K / 16);
        uint4 *dst = reinterpret_cast<uint4 *>(rq + (size_t)blk * QB);
        dst[0] = make_uint4(word[0], word[1], word[2], word[3]);
        dst[1] = make_uint4(word[4], word[5], word[6], word[7]);
        reinterpret_cast<__half *>(rq + K)[blk] = dh;
    }
    if (write_back) {
        const float ds = __half2float(dh);
        uint4 out[4];
        uint32_t *o = reinterpret_cast<uint32_t *>(out);
#pragma unroll
        for (int i = 0; i < QB / 2; ++i) o[i] = pack_h2((float)q[2 * i] * ds, (float)q[2 * i + 1] * ds);
#pragma unroll
        for (int i = 0; i < 4; ++i) reinterpret_cast<uint4 *>(src)[i] = out[i];
    }
}

}  // namespace

size_t q8_0_row_bytes(int K) { return (size_t)K + (size_t)K / 16; }

cudaError_t launch_quantize_q8_0(f16 *w, int N, int K, uint8_t *q8, bool write_back, cudaStream_t st) {
    if (N < 1 || K < QB || K % QB || (q8 && K % 256)) return cudaErrorInvalidValue;
    const long long nblk = (long long)N * (K / QB);
    quantize_q8_0_kernel<<<(unsigned)((nblk + 255) / 256), 256, 0, st>>>(w, N, K, q8, write_back ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace llm
