// Shared-memory tiles of K/V rows for the attention kernels: rows of head_dim
// fp16 values, 16-byte chunks XOR-swizzled so that ldmatrix over 8
// consecutive rows is free of bank conflicts, filled with cp.async.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace llm {

template <int HD>
struct Swz {
    static constexpr int CH = HD / 8;                      // 16-byte chunks per row
    __device__ static __forceinline__ int chunk(int r, int c) {
        return CH >= 8 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & (CH - 1)));
    }
    __device__ static __forceinline__ int off(int r, int c) { return r * HD + chunk(r, c) * 8; }
};

// rows [0, rows_valid) of src (row stride HD) into a ROWS x HD swizzled tile;
// the remaining rows are zero-filled.
template <int HD, int ROWS, int THREADS>
__device__ __forceinline__ void load_rows(f16 *dst, const f16 *src, int rows_valid, int tid) {
    constexpr int CH = HD / 8;
    for (int i = tid; i < ROWS * CH; i += THREADS) {
        const int r = i / CH, c = i - r * CH;
        const bool pv = r < rows_valid;
        cp_async16(dst + Swz<HD>::off(r, c), src + (size_t)(pv ? r : 0) * HD + c * 8, pv);
    }
}

// rows [r_lo, r_hi) of src (row stride HD) into a ROWS x HD swizzled tile,
// rows [r_zero, ROWS) zero-filled, every other row left untouched (so that a
// later call can fill it: two cp.async writes to one address are unordered).
template <int HD, int ROWS, int THREADS>
__device__ __forceinline__ void load_rows_span(f16 *dst, const f16 *src, int r_lo, int r_hi, int r_zero, int tid) {
    constexpr int CH = HD / 8;
    for (int i = tid; i < ROWS * CH; i += THREADS) {
        const int r = i / CH, c = i - r * CH;
        const bool copy = r >= r_lo && r < r_hi;
        if (copy || r >= r_zero)
            cp_async16(dst + Swz<HD>::off(r, c), src + (size_t)(copy ? r : 0) * HD + c * 8, copy);
    }
}

// FP8 E4M3 cache rows.  A ROWS x HD fp16 tile buffer is 2 * ROWS * HD bytes; its
// upper half stages the fp8 rows (HD bytes each, linear) that convert_tile8
// then widens in place into the swizzled fp16 layout.  Same row selection as
// load_rows_span.
template <int HD, int ROWS, int THREADS>
__device__ __forceinline__ void load_rows_span8(f16 *tile, const uint8_t *src, int r_lo, int r_hi, int r_zero,
                                                int tid) {
    constexpr int CH = HD / 16;                            // 16-byte chunks per fp8 row
    uint8_t *stage = reinterpret_cast<uint8_t *>(tile) + ROWS * HD;
    for (int i = tid; i < ROWS * CH; i += THREADS) {
        const int r = i / CH, c = i - r * CH;
        const bool copy = r >= r_lo && r < r_hi;
        if (copy || r >= r_zero)
            cp_async16(stage + r * HD + c * 16, src + (size_t)(copy ? r : 0) * HD + c * 16, copy);
    }
}
template <int HD, int ROWS, int THREADS>
__device__ __forceinline__ void load_rows8(f16 *tile, const uint8_t *src, int rows_valid, int tid) {
    load_rows_span8<HD, ROWS, THREADS>(tile, src, 0, rows_valid, rows_valid, tid);
}

// Widen the staged fp8 rows of a tile into its fp16 swizzled layout (exact).
// Every thread reads all of its chunks before any is written (the CTA-wide
// barrier in between), since the fp16 rows overlap the staging area.  Ends
// with a barrier: the tile is ready for ldmatrix.
template <int HD, int ROWS, int THREADS>
__device__ __forceinline__ void convert_tile8(f16 *tile, int tid) {
    constexpr int CH = HD / 16;
    constexpr int PER = (ROWS * CH + THREADS - 1) / THREADS;
    const uint8_t *stage = reinterpret_cast<const uint8_t *>(tile) + ROWS * HD;
    uint4 buf[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = tid + j * THREADS;
        if (i < ROWS * CH) buf[j] = *reinterpret_cast<const uint4 *>(stage + (i / CH) * HD + (i % CH) * 16);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = tid + j * THREADS;
        if (i < ROWS * CH) {
            const int r = i / CH, c = i - r * CH;
            const uint32_t w[4] = {buf[j].x, buf[j].y, buf[j].z, buf[j].w};
            uint32_t h[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                h[2 * e] = e4m3x2_to_h2((uint16_t)(w[e] & 0xFFFFu));
                h[2 * e + 1] = e4m3x2_to_h2((uint16_t)(w[e] >> 16));
            }
            *reinterpret_cast<uint4 *>(tile + Swz<HD>::off(r, 2 * c)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(tile + Swz<HD>::off(r, 2 * c + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
    __syncthreads();
}

}  // namespace llm
